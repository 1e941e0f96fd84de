// conv_gemm.cuh -- tcgen05 implicit-GEMM convolution for every tensor-core
// layer of the decoder: conv_in (k7), the polyphase ConvTranspose1d, the k7
// dilated conv1 and the k1 conv2 of each residual unit.
//
// GEMM view (channels-last activations, time on M, output columns on N):
//   D[t][n] = sum_tap sum_ci A[t + off(tap, n)][ci] * Wt[tap][n][ci]
// * regular conv: off(tap) = tap*dil - pad_left, n = output channel;
// * ConvTranspose1d of stride s, K = 2s, left crop p (polyphase form): the
//   output sample t*s + r of channel co is column n = r*C_out + co and
//     out[t*s + r][co] = sum_ci W[ci][co][k0] x[t+q][ci] + W[ci][co][k0+s] x[t+q-1][ci]
//   with q = floor((r+p)/s), k0 = (r+p) mod s, i.e. two taps at row offsets q and
//   q-1.  Row t of D is then exactly the contiguous channels-last output rows
//   t*s .. t*s+s-1, so the overlap-add of col2im happens inside the MMA and no
//   column matrix is ever written.
//
// Operands: every activation that enters an MMA is stored as a bf16 pair
// (hi, lo) with hi = bf16(x), lo = bf16(x - hi); weights are pre-split the same
// way on the host.  Each K step issues three MMAs, hi*hi + hi*lo + lo*hi, into
// one fp32 TMEM accumulator.
//
// Shared-memory layout (no swizzle, K-major): an A stage holds, for each 8-channel
// chunk, `rows` consecutive time rows of 16 bytes, so the row offset of a tap is a
// 16-byte shift of the descriptor start address and all taps reuse one staged
// halo tile (128 + span rows) loaded by TMA with zero fill outside [0, L).
//
// Roles: warp 0 lane 0 issues TMA / bulk copies, warp 1 lane 0 issues MMAs,
// warps 2..5 run the epilogue (TMEM -> registers -> bias, residual, Snake of
// the next layer, hi/lo split -> global).  The grid is persistent; two TMEM
// accumulators let the epilogue of one tile overlap the mainloop of the next.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace voc {

constexpr int kTileM = 128;
constexpr int kGemmThreads = 192;

enum : int {
  EPI_F32_SNAKE = 1,  // the fp32 output receives Snake(v) instead of v
};

// device error word bits
enum : int {
  ERR_TIMEOUT_PRODUCER = 1,
  ERR_TIMEOUT_MMA = 2,
  ERR_TIMEOUT_EPILOGUE = 4,
};

struct ConvGemmArgs {
  int B, L_in, Cp_in;      // batch, input rows per item, padded input channels
  int KB, nkb, taps;       // channels per k-block, k-blocks, taps
  int rows, off_min;       // A stage rows (multiple of 8), row offset of the stage start
  int shift0_q0, shift0_q1, tap_step;  // row shift of tap 0 (per ConvT phase group), per-tap step
  int q_split_tile;        // n-tiles >= this belong to phase group q = 1
  int N_tile, n_tiles, N_total, m_tiles;
  int na, nb;              // A / B ring slots
  int a_bytes, b_bytes;    // slot strides in bytes (b_bytes = one packed weight tile)
  int acc_cols;            // TMEM columns per accumulator (power of two >= 32)
  const uint8_t *wB;       // packed weight tiles [n_tile][tap][kb][hi|lo][chunk][n][8]
  const float *bias;       // [N_total] per-column bias
  const float *alpha;      // [N_total] Snake alpha of the next layer, or null
  const float *invb;       // [N_total] 1/(alpha + 1e-9)
  const float *skip;       // fp32 residual [B][L_in][N_total] or null
  float *out_f32;          // fp32 output [B][L_in][N_total] or null
  __nv_bfloat16 *out_hl;   // hi/lo output rows [B][L_in*s_rows][2*Cp_out] or null
  int Cp_out, s_rows;
  int flags;
  long long timeout;       // cycles a wait may take before the kernel gives up
  int *err;                // device error word
};

__device__ __forceinline__ void store_hl16(__nv_bfloat16 *dst, int Cp, const float (&s)[16]) {
  uint32_t hi[8], lo[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    __nv_bfloat16 h0 = __float2bfloat16_rn(s[2 * i]);
    __nv_bfloat16 h1 = __float2bfloat16_rn(s[2 * i + 1]);
    __nv_bfloat16 l0 = __float2bfloat16_rn(s[2 * i] - __bfloat162float(h0));
    __nv_bfloat16 l1 = __float2bfloat16_rn(s[2 * i + 1] - __bfloat162float(h1));
    hi[i] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
            (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
    lo[i] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
            (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
  }
  uint4 *dh = reinterpret_cast<uint4 *>(dst);
  uint4 *dl = reinterpret_cast<uint4 *>(dst + Cp);
  dh[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  dh[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
  dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
}

__device__ __forceinline__ void load16(const float *src, float (&v)[16]) {
  const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float4 a = __ldg(s4 + j);
    v[4 * j] = a.x, v[4 * j + 1] = a.y, v[4 * j + 2] = a.z, v[4 * j + 3] = a.w;
  }
}

__device__ __forceinline__ void store16(float *dst, const float (&v)[16]) {
  float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j) d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

// Epilogue of 16 consecutive columns n0..n0+15 of D row `drow` (= b*L_in + t).
__device__ __forceinline__ void epilogue16(const ConvGemmArgs &p, size_t drow, int n0,
                                           float (&v)[16]) {
  float tmp[16];
  load16(p.bias + n0, tmp);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] += tmp[i];
  if (p.skip) {
    load16(p.skip + drow * p.N_total + n0, tmp);  // read before the (possibly in-place) store
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] += tmp[i];
  }
  if (p.alpha) {
    float a[16], ib[16], s[16];
    load16(p.alpha + n0, a);
    load16(p.invb + n0, ib);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float sn = sinf(a[i] * v[i]);
      s[i] = fmaf(ib[i] * sn, sn, v[i]);  // Snake: v + sin^2(a v) / (a + 1e-9)
    }
    if (p.out_f32) store16(p.out_f32 + drow * p.N_total + n0, (p.flags & EPI_F32_SNAKE) ? s : v);
    if (p.out_hl) {
      const int r = n0 / p.Cp_out;
      const int co = n0 - r * p.Cp_out;
      store_hl16(p.out_hl + (drow * p.s_rows + r) * (size_t)(2 * p.Cp_out) + co, p.Cp_out, s);
    }
  } else {
    if (p.out_f32) store16(p.out_f32 + drow * p.N_total + n0, v);
    if (p.out_hl) {
      const int r = n0 / p.Cp_out;
      const int co = n0 - r * p.Cp_out;
      store_hl16(p.out_hl + (drow * p.s_rows + r) * (size_t)(2 * p.Cp_out) + co, p.Cp_out, v);
    }
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    conv_gemm_kernel(const __grid_constant__ CUtensorMap tmapA, const ConvGemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smA + (size_t)p.na * p.a_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smB + (size_t)p.nb * p.b_bytes);
  uint64_t *fullA = bars;
  uint64_t *emptyA = fullA + p.na;
  uint64_t *fullB = emptyA + p.na;
  uint64_t *emptyB = fullB + p.nb;
  uint64_t *accFull = emptyB + p.nb;
  uint64_t *accEmpty = accFull + 2;
  uint64_t *drain = accEmpty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t tmem_cols = 2u * p.acc_cols;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.na; ++i) {
      mbar_init(smem_u32(fullA + i), 1);
      mbar_init(smem_u32(emptyA + i), 1);
    }
    for (int i = 0; i < p.nb; ++i) {
      mbar_init(smem_u32(fullB + i), 1);
      mbar_init(smem_u32(emptyB + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(accFull + i), 1);
      mbar_init(smem_u32(accEmpty + i), 4 * 32);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);

  const int total_tiles = p.B * p.m_tiles * p.n_tiles;
  const int kchunks = p.KB / 8;
  const uint32_t chunkA = static_cast<uint32_t>(p.rows) * 16u;
  const uint32_t chunkB = static_cast<uint32_t>(p.N_tile) * 16u;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      prefetch_tmap(&tmapA);
      const uint32_t a_tx = 2u * kchunks * chunkA;
      int ia = 0, ib = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        const int nt = tile % p.n_tiles;
        const int rest = tile / p.n_tiles;
        const int mt = rest % p.m_tiles;
        const int b = rest / p.m_tiles;
        const int y0 = mt * kTileM + p.off_min;
        for (int kb = 0; kb < p.nkb && ok; ++kb) {
          const int sa = ia % p.na;
          const uint32_t pha = static_cast<uint32_t>(ia / p.na) & 1u;
          if (!mbar_wait(smem_u32(emptyA + sa), pha ^ 1u, p.timeout, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fa = smem_u32(fullA + sa);
          mbar_arrive_expect_tx(fa, a_tx);
          const uint32_t dstA = smem_u32(smA + (size_t)sa * p.a_bytes);
          for (int c = 0; c < kchunks; ++c) {
            const int x = kb * p.KB + c * 8;
            tma_load_3d(dstA + c * chunkA, &tmapA, fa, x, y0, b);
            tma_load_3d(dstA + (kchunks + c) * chunkA, &tmapA, fa, p.Cp_in + x, y0, b);
          }
          ++ia;
          for (int tap = 0; tap < p.taps; ++tap) {
            const int sb = ib % p.nb;
            const uint32_t phb = static_cast<uint32_t>(ib / p.nb) & 1u;
            if (!mbar_wait(smem_u32(emptyB + sb), phb ^ 1u, p.timeout, abort_flag)) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(fullB + sb);
            mbar_arrive_expect_tx(fb, static_cast<uint32_t>(p.b_bytes));
            const size_t widx = ((size_t)nt * p.taps + tap) * p.nkb + kb;
            bulk_load(smem_u32(smB + (size_t)sb * p.b_bytes), p.wB + widx * p.b_bytes,
                      static_cast<uint32_t>(p.b_bytes), fb);
            ++ib;
          }
        }
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_PRODUCER);
        *abort_flag = 1;
        // let every copy already issued land before the CTA can exit: the last
        // fill of slot s (its cnt-th) completes the phase of parity (cnt-1)&1
        const volatile int never = 0;
        for (int s = 0; s < p.na && s < ia; ++s) {
          const int cnt = (ia - s + p.na - 1) / p.na;
          mbar_wait(smem_u32(fullA + s), static_cast<uint32_t>(cnt - 1) & 1u, p.timeout, &never);
        }
        for (int s = 0; s < p.nb && s < ib; ++s) {
          const int cnt = (ib - s + p.nb - 1) / p.nb;
          mbar_wait(smem_u32(fullB + s), static_cast<uint32_t>(cnt - 1) & 1u, p.timeout, &never);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_bf16_f32(kTileM, p.N_tile);
      int ia = 0, ib = 0, it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++it) {
        const int nt = tile % p.n_tiles;
        const int shift0 = (nt >= p.q_split_tile) ? p.shift0_q1 : p.shift0_q0;
        const int acc = it & 1;
        const uint32_t phacc = static_cast<uint32_t>(it >> 1) & 1u;
        if (!mbar_wait(smem_u32(accEmpty + acc), phacc ^ 1u, p.timeout, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.acc_cols);
        for (int kb = 0; kb < p.nkb && ok; ++kb) {
          const int sa = ia % p.na;
          const uint32_t pha = static_cast<uint32_t>(ia / p.na) & 1u;
          if (!mbar_wait(smem_u32(fullA + sa), pha, p.timeout, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aBase = smem_u32(smA + (size_t)sa * p.a_bytes);
          for (int tap = 0; tap < p.taps; ++tap) {
            const int sb = ib % p.nb;
            const uint32_t phb = static_cast<uint32_t>(ib / p.nb) & 1u;
            if (!mbar_wait(smem_u32(fullB + sb), phb, p.timeout, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t bBase = smem_u32(smB + (size_t)sb * p.b_bytes);
            const uint32_t aTap = aBase + static_cast<uint32_t>(shift0 + tap * p.tap_step) * 16u;
            for (int ks = 0; ks < kchunks / 2; ++ks) {
              const uint64_t a_hi = smem_desc(aTap + (2 * ks) * chunkA, chunkA, 128);
              const uint64_t a_lo = smem_desc(aTap + (kchunks + 2 * ks) * chunkA, chunkA, 128);
              const uint64_t b_hi = smem_desc(bBase + (2 * ks) * chunkB, chunkB, 128);
              const uint64_t b_lo = smem_desc(bBase + (kchunks + 2 * ks) * chunkB, chunkB, 128);
              const uint32_t accum = (kb | tap | ks) ? 1u : 0u;
              mma_bf16(d_tmem, a_hi, b_hi, idesc, accum);
              mma_bf16(d_tmem, a_hi, b_lo, idesc, 1u);
              mma_bf16(d_tmem, a_lo, b_hi, idesc, 1u);
            }
            mma_commit(smem_u32(emptyB + sb));
            ++ib;
          }
          if (!ok) break;
          mma_commit(smem_u32(emptyA + sa));
          ++ia;
        }
        if (!ok) break;
        mma_commit(smem_u32(accFull + acc));
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_MMA);
        *abort_flag = 1;
        // wait until every MMA issued so far has finished reading shared memory
        mma_commit(smem_u32(drain));
        const volatile int never = 0;
        mbar_wait(smem_u32(drain), 0u, p.timeout, &never);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
      const int nt = tile % p.n_tiles;
      const int rest = tile / p.n_tiles;
      const int mt = rest % p.m_tiles;
      const int b = rest / p.m_tiles;
      const int acc = it & 1;
      const uint32_t phacc = static_cast<uint32_t>(it >> 1) & 1u;
      if (!mbar_wait(smem_u32(accFull + acc), phacc, p.timeout, abort_flag)) {
        atomicOr(p.err, ERR_TIMEOUT_EPILOGUE);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int t = mt * kTileM + row;
      const bool valid = t < p.L_in;
      const size_t drow = (size_t)b * p.L_in + t;
      const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * p.acc_cols) +
                             (static_cast<uint32_t>(quad * 32) << 16);
      for (int c = 0; c < p.N_tile / 16; ++c) {
        float v[16];
        tmem_ld16(tbase + c * 16, v);
        if (valid) epilogue16(p, drow, nt * p.N_tile + c * 16, v);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(accEmpty + acc));
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace voc
