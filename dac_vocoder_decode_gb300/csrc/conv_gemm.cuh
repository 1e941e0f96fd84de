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
// Roles: warp 0 lane 0 issues the A (TMA) and weight (bulk) copies, warp 1 lane 0
// issues MMAs, warps 2..9 run the epilogue (TMEM -> registers -> bias, residual,
// Snake of the next layer, hi/lo split -> global), warp 10 lane 0 prefetches the
// residual input of the epilogue by TMA.  The grid is persistent; 2 to 4 TMEM
// accumulators let the epilogue of one tile overlap the mainloop of the next.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "snake.cuh"

namespace voc {

constexpr int kTileM = 128;
constexpr int kEpiWarps = 8;                            // two per TMEM lane quadrant
constexpr int kSkipWarp = 2 + kEpiWarps;                // residual prefetch warp
constexpr int kGemmThreads = 32 * (kSkipWarp + 1);      // 352
constexpr int kMaxAcc = 4;

// bytes of per-warp epilogue staging (an fp32 tile and a hi/lo tile of 32 rows x cw columns)
__host__ __device__ constexpr int epi_stage_bytes(int cw) { return kEpiWarps * 2 * 32 * cw * 4; }
// bytes of one residual slot (128 rows x cw fp32 columns)
__host__ __device__ constexpr int skip_slot_bytes(int cw) { return kTileM * cw * 4; }

enum : int {
  EPI_F32_SNAKE = 1,  // the fp32 output receives Snake(v) instead of v
};

// device error word bits
enum : int {
  ERR_TIMEOUT_PRODUCER = 1,
  ERR_TIMEOUT_MMA = 2,
  ERR_TIMEOUT_EPILOGUE = 4,
  ERR_TIMEOUT_SKIP = 8,
};

struct ConvGemmArgs {
  int B, L_in, Cp_in;      // batch, input rows per item, padded input channels
  int KB, nkb, taps;       // channels per k-block, k-blocks, taps
  int rows, off_min;       // A stage rows (multiple of 8), row offset of the stage start
  int shift0_q0, shift0_q1, tap_step;  // row shift of tap 0 (per ConvT phase group), per-tap step
  int q_split_tile;        // n-tiles >= this belong to phase group q = 1
  int N_tile, n_tiles, N_total, m_tiles;
  int na, nb, ns;          // A / B / residual ring slots
  int a_bytes, b_bytes;    // slot strides in bytes (b_bytes = one packed weight tile)
  int acc_cols, n_acc;     // TMEM columns per accumulator (power of two >= 32), accumulators
  const uint8_t *wB;       // packed weight tiles [n_tile][tap][kb][hi|lo][chunk][n][8]
  const float *bias;       // [N_total] per-column bias
  const float *alpha;      // [N_total] Snake alpha of the next layer, or null
  const float *invb;       // [N_total] 1/(alpha + 1e-9)
  const float *skip;       // fp32 residual [B][L_in][N_total] or null (read through tmapS)
  float *out_f32;          // fp32 output [B][L_in][N_total] or null
  __nv_bfloat16 *out_hl;   // hi/lo output rows [B][L_in*s_rows][2*Cp_out] or null
  int Cp_out, s_rows;
  int flags;
  long long timeout;       // cycles a wait may take before the kernel gives up
  int *err;                // device error word
};

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

template <int N>
__device__ __forceinline__ void ldg_vec(const float *src, float (&v)[N]) {
  const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
  for (int j = 0; j < N / 4; ++j) {
    const float4 a = __ldg(s4 + j);
    v[4 * j] = a.x, v[4 * j + 1] = a.y, v[4 * j + 2] = a.z, v[4 * j + 3] = a.w;
  }
}

// Shared tiles of rows of CW fp32 (CW*4 bytes) whose 16-byte chunks are XOR-
// swizzled by the row index: the layout the TMA writes with 128-byte (CW = 32)
// or 64-byte (CW = 16) swizzling from a 1024-byte aligned base.  Row-wise and
// column-wise 16-byte accesses by a warp are then free of bank conflicts.
template <int CW>
struct Stage {
  static constexpr int NCH = CW / 4;        // 16-byte chunks per row
  static constexpr int RB = CW * 4;         // bytes per row
  static constexpr int RPI = 32 / NCH;      // rows per warp-wide 16-byte access
  __device__ static __forceinline__ uint32_t at(uint32_t base, int r, int c) {
    const int sw = (NCH == 8) ? (r & 7) : ((r >> 1) & 3);
    return base + static_cast<uint32_t>(r * RB + ((c ^ sw) << 4));
  }
};

// Epilogue of one warp for 32 rows (its TMEM lane quadrant) x CW columns.
// Global stores go through the warp's staging tiles: the thread of row r writes
// its row, then every lane moves 16-byte pieces so that one warp-wide store covers
// whole row segments (CW = 32: 4 rows x 128 B).  The residual input arrives in a
// shared slot filled by the prefetch warp (slot row r = tile row r).
template <int CW>
__device__ __forceinline__ bool epilogue_chunk(const ConvGemmArgs &p, uint32_t stf, uint32_t sth,
                                               uint32_t sslot, uint32_t sfull, uint32_t sempty,
                                               uint32_t sparity, const volatile int *abort_flag,
                                               int lane, int quad, int b, int t0w, int n0,
                                               uint32_t taddr) {
  using S = Stage<CW>;
  float v[CW];
  tmem_ld(taddr, v);
  {
    float bb[CW];
    ldg_vec(p.bias + n0, bb);
#pragma unroll
    for (int i = 0; i < CW; ++i) v[i] += bb[i];
  }
  const size_t row0 = (size_t)b * p.L_in;  // D row of t = 0 in this item
  if (p.skip) {
    if (!mbar_wait(sfull, sparity, p.timeout, abort_flag)) return false;
    const int r = quad * 32 + lane;
#pragma unroll
    for (int c = 0; c < S::NCH; ++c) {
      const uint4 x = lds128(S::at(sslot, r, c));
      v[4 * c] += __uint_as_float(x.x), v[4 * c + 1] += __uint_as_float(x.y);
      v[4 * c + 2] += __uint_as_float(x.z), v[4 * c + 3] += __uint_as_float(x.w);
    }
    mbar_arrive(sempty);
  }
  float sn[CW];
  if (p.alpha) {
    float a[CW], ib[CW];
    ldg_vec(p.alpha + n0, a);
    ldg_vec(p.invb + n0, ib);
#pragma unroll
    for (int i = 0; i < CW; ++i) sn[i] = snake(v[i], a[i], ib[i]);
  } else {
#pragma unroll
    for (int i = 0; i < CW; ++i) sn[i] = v[i];
  }
  if (p.out_f32) {
    const bool snake_out = (p.flags & EPI_F32_SNAKE) != 0;
#pragma unroll
    for (int c = 0; c < S::NCH; ++c) {
      const float *src = snake_out ? sn : v;
      sts128(S::at(stf, lane, c),
             make_uint4(__float_as_uint(src[4 * c]), __float_as_uint(src[4 * c + 1]),
                        __float_as_uint(src[4 * c + 2]), __float_as_uint(src[4 * c + 3])));
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < S::NCH; ++i) {
      const int r = i * S::RPI + lane / S::NCH, c = lane % S::NCH;
      const int t = t0w + r;
      const uint4 x = lds128(S::at(stf, r, c));
      if (t < p.L_in)
        *reinterpret_cast<uint4 *>(p.out_f32 + (row0 + t) * p.N_total + n0 + 4 * c) = x;
    }
    __syncwarp();
  }
  if (p.out_hl) {
    uint32_t hw[CW / 2], lw[CW / 2];
#pragma unroll
    for (int i = 0; i < CW / 2; ++i) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(sn[2 * i]);
      const __nv_bfloat16 h1 = __float2bfloat16_rn(sn[2 * i + 1]);
      const __nv_bfloat16 l0 = __float2bfloat16_rn(sn[2 * i] - __bfloat162float(h0));
      const __nv_bfloat16 l1 = __float2bfloat16_rn(sn[2 * i + 1] - __bfloat162float(h1));
      hw[i] = pack_bf16x2(h0, h1);
      lw[i] = pack_bf16x2(l0, l1);
    }
#pragma unroll
    for (int c = 0; c < S::NCH / 2; ++c) {
      sts128(S::at(sth, lane, c), make_uint4(hw[4 * c], hw[4 * c + 1], hw[4 * c + 2], hw[4 * c + 3]));
      sts128(S::at(sth, lane, S::NCH / 2 + c),
             make_uint4(lw[4 * c], lw[4 * c + 1], lw[4 * c + 2], lw[4 * c + 3]));
    }
    __syncwarp();
    const int ph = n0 / p.Cp_out;  // ConvT phase of these columns (0 for a conv)
    const int co0 = n0 - ph * p.Cp_out;
#pragma unroll
    for (int i = 0; i < S::NCH; ++i) {
      const int r = i * S::RPI + lane / S::NCH, c = lane % S::NCH;
      const int t = t0w + r;
      const uint4 x = lds128(S::at(sth, r, c));
      if (t < p.L_in) {
        const size_t orow = (row0 + t) * p.s_rows + ph;
        const int col = (c < S::NCH / 2) ? co0 + 8 * c : p.Cp_out + co0 + 8 * (c - S::NCH / 2);
        *reinterpret_cast<uint4 *>(p.out_hl + orow * (size_t)(2 * p.Cp_out) + col) = x;
      }
    }
    __syncwarp();
  }
  return true;
}

// Wait (bounded) until every fill issued into a ring of `slots` barriers has
// landed: the last fill of slot s (its cnt-th) completes the phase of parity (cnt-1)&1.
__device__ __forceinline__ void drain_ring(uint64_t *full, int slots, int issued, long long budget) {
  const volatile int never = 0;
  for (int s = 0; s < slots && s < issued; ++s) {
    const int cnt = (issued - s + slots - 1) / slots;
    mbar_wait(smem_u32(full + s), static_cast<uint32_t>(cnt - 1) & 1u, budget, &never);
  }
}

template <int CW>
__global__ void __launch_bounds__(kGemmThreads, 1)
    conv_gemm_kernel(const __grid_constant__ CUtensorMap tmapA,
                     const __grid_constant__ CUtensorMap tmapS, const ConvGemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smA + (size_t)p.na * p.a_bytes;
  uint8_t *smE = smB + (size_t)p.nb * p.b_bytes;   // epilogue staging
  uint8_t *smS = smE + epi_stage_bytes(CW);         // residual slots
  uint64_t *bars = reinterpret_cast<uint64_t *>(smS + (size_t)p.ns * skip_slot_bytes(CW));
  uint64_t *fullA = bars;
  uint64_t *emptyA = fullA + p.na;
  uint64_t *fullB = emptyA + p.na;
  uint64_t *emptyB = fullB + p.nb;
  uint64_t *accFull = emptyB + p.nb;
  uint64_t *accEmpty = accFull + kMaxAcc;
  uint64_t *skipFull = accEmpty + kMaxAcc;
  uint64_t *skipEmpty = skipFull + p.ns;
  uint64_t *drain = skipEmpty + p.ns;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t tmem_cols = static_cast<uint32_t>(p.n_acc * p.acc_cols);

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.na; ++i) {
      mbar_init(smem_u32(fullA + i), 1);
      mbar_init(smem_u32(emptyA + i), 1);
    }
    for (int i = 0; i < p.nb; ++i) {
      mbar_init(smem_u32(fullB + i), 1);
      mbar_init(smem_u32(emptyB + i), 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(smem_u32(accFull + i), 1);
      mbar_init(smem_u32(accEmpty + i), kEpiWarps * 32);
    }
    for (int i = 0; i < p.ns; ++i) {
      mbar_init(smem_u32(skipFull + i), 1);
      mbar_init(smem_u32(skipEmpty + i), 4 * 32);  // the four quadrant warps of one half
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
  const int n_chunks = p.N_tile / CW;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ A / weight producer
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
        drain_ring(fullA, p.na, ia, p.timeout);  // copies in flight land before the CTA exits
        drain_ring(fullB, p.nb, ib, p.timeout);
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
        const int acc = it % p.n_acc;
        const uint32_t phacc = static_cast<uint32_t>(it / p.n_acc) & 1u;
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
  } else if (warp == kSkipWarp) {
    if (lane == 0 && p.skip) {
      // ------------------------------------------------------------ residual prefetch
      prefetch_tmap(&tmapS);
      const uint32_t bytes = static_cast<uint32_t>(skip_slot_bytes(CW));
      int ks = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        const int nt = tile % p.n_tiles;
        const int rest = tile / p.n_tiles;
        const int mt = rest % p.m_tiles;
        const int b = rest / p.m_tiles;
        for (int c = 0; c < n_chunks; ++c, ++ks) {
          const int slot = ks % p.ns;
          const uint32_t ph = static_cast<uint32_t>(ks / p.ns) & 1u;
          if (!mbar_wait(smem_u32(skipEmpty + slot), ph ^ 1u, p.timeout, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fs = smem_u32(skipFull + slot);
          mbar_arrive_expect_tx(fs, bytes);
          tma_load_3d(smem_u32(smS + (size_t)slot * bytes), &tmapS, fs, nt * p.N_tile + c * CW,
                      mt * kTileM, b);
        }
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_SKIP);
        *abort_flag = 1;
        drain_ring(skipFull, p.ns, ks, p.timeout);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int e = warp - 2;     // epilogue warp 0..7
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int half = e / 4;     // the two warps of a quadrant take alternate column chunks
    const uint32_t stf = smem_u32(smE) + static_cast<uint32_t>(e * 2 * 32 * CW * 4);
    const uint32_t sth = stf + 32 * CW * 4;
    const uint32_t sbase = smem_u32(smS);
    const int ns = p.ns > 0 ? p.ns : 1;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++it) {
      const int nt = tile % p.n_tiles;
      const int rest = tile / p.n_tiles;
      const int mt = rest % p.m_tiles;
      const int b = rest / p.m_tiles;
      const int acc = it % p.n_acc;
      const uint32_t phacc = static_cast<uint32_t>(it / p.n_acc) & 1u;
      if (!mbar_wait(smem_u32(accFull + acc), phacc, p.timeout, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int t0w = mt * kTileM + quad * 32;
      const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * p.acc_cols) +
                             (static_cast<uint32_t>(quad * 32) << 16);
      for (int c = half; c < n_chunks && ok; c += 2) {
        const int kc = it * n_chunks + c;  // residual chunk counter (fill order of the slots)
        const int slot = kc % ns;
        ok = epilogue_chunk<CW>(
            p, stf, sth, sbase + static_cast<uint32_t>(slot * skip_slot_bytes(CW)),
            smem_u32(skipFull + slot), smem_u32(skipEmpty + slot),
            static_cast<uint32_t>(kc / ns) & 1u, abort_flag, lane, quad, b, t0w,
            nt * p.N_tile + c * CW, tbase + c * CW);
      }
      if (!ok) break;
      tc_fence_before();
      mbar_arrive(smem_u32(accEmpty + acc));
    }
    if (!ok) {
      atomicOr(p.err, ERR_TIMEOUT_EPILOGUE);
      *abort_flag = 1;
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
