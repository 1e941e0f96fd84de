// ru_gemm.cuh -- one residual unit of the decoder in one kernel, for units of up to 192
// channels (minimaxmusic.cpp Architecture, "Flow VAE": res_unit = skip -> snake1 -> conv1 k7
// dil d -> snake2 -> conv2 k1 -> + skip):
//
//   h = conv1(A) + b1            A = Snake1(x) as bf16 hi/lo, from HBM (TMA, halo of the taps)
//   H = Snake2(h) as bf16 hi/lo  written by the epilogue into SHARED memory, in the canonical
//                                K-major layout of an MMA operand
//   y = x + conv2(H) + b2        x (fp32) read by the epilogue warps from HBM
//
// so the conv1 result never goes to HBM: per row the unit reads 4 C bytes of A and 4 C of x
// and writes its outputs, instead of also writing and re-reading h (8 C more).
//
// Schedule (per CTA, over its 128-row tiles i = 0, 1, ...): the MMA warp issues
//   conv1(0), conv1(1), conv2(0), conv1(2), conv2(1), ...
// into one conv1 accumulator (acc1) and one conv2 accumulator (acc2) in TMEM.  When conv1(i)
// completes, the epilogue warps first copy acc1 into registers and release it -- while the
// tensor cores run the short conv2(i-1) -- so conv1(i+1) follows without a gap; then they apply
// bias and Snake2, wait until conv2(i-1) has read H, write H(i), and finish tile i-1 from acc2
// (bias, residual, Snake of the next layer, fp32 and hi/lo stores) while conv1(i+1) runs.
// Epilogue work therefore overlaps the tensor cores instead of sitting between conv1 and conv2.
//
// Roles (16 warps): warp 0 lane 0 issues the A copies (one 5-D TMA box per k-block), warp 1
// issues the MMAs (convergently; an elected lane issues), warp 2 lane 0 streams the weight
// stages (conv1's taps x k-blocks, then conv2's k-blocks, in the MMA warp's order); warps 4..15
// are the epilogue: three groups of four warps, one warp per TMEM lane quadrant, group g taking
// the 16-column chunks g, g+3, ...  The first warp group hands registers to the other three
// (setmaxnreg), which hold a tile's conv1 accumulator row in registers.
//
// B2 (units of up to 128 channels): both convolutions take the conv kernel's two-MMA K step --
// A_hi x [W_hi | W_lo] into 2N accumulator columns, then A_lo x W_hi into the first N -- and the
// epilogues add the two column halves.  The arithmetic of each epilogue is the separate conv
// kernel's, so the fused unit computes the same values as conv1 + conv2 run as two kernels.
//
// PREC: the weight form, as in the conv kernel.  The one-plane precisions (f16 or bf16 weights,
// activations as f16 / bf16 hi/lo pairs) take two MMAs per K step, A_hi x W and A_lo x W, with
// N columns each, and split their outputs into f16 parts for the F16-weight form.
#pragma once
#include "conv_gemm.cuh"

namespace voc {

// Warp group 0 (warps 0..3) issues copies and MMAs with few registers; warp groups 1..3 are the
// epilogue, with the registers the others give up (setmaxnreg): 128 x 32 + 384 x 160 = 65536,
// the 512 threads x 128 registers the block is launched with.
constexpr int kRuBWarp = 2;                          // weight copies (warp 3 idles)
constexpr int kRuEpi0 = 4;                           // first epilogue warp
constexpr int kRuEpiWarps = 4 * kEpiGroups;          // warps 4..15
constexpr int kRuThreads = 32 * (kRuEpi0 + kRuEpiWarps);  // 512
constexpr int kRuLaunchRegs = 128;                   // registers per thread at launch
constexpr int kRuCopyRegs = 32;                      // warp group 0 after the split
constexpr int kRuEpiRegs = 160;                      // epilogue warp groups after the split
static_assert(128 * kRuCopyRegs + 32 * kRuEpiWarps * kRuEpiRegs <= kRuThreads * kRuLaunchRegs,
              "the register split exceeds the launch allocation");
// 16-column chunks of one epilogue group: C <= 192 has 12 chunks (4 per group); the B2 form
// (C <= 128) at most 8 (3 per group)
template <bool B2>
__host__ __device__ constexpr int ru_max_chunks() { return B2 ? 3 : 4; }

struct RuExtra {
  const uint8_t *wB2;      // packed 1x1 weight stages [kb][...], the layout of a conv1 stage
  const float *bias_h;     // [N] conv1 bias
  const float *alpha_h;    // [N] Snake2 alpha
  const float *invb_h;     // [N] Snake2 1/(alpha + 1e-9)
  int h_bytes;             // bytes of the H tile (4 * 128 * Cp / h_parts)
  int h_parts;             // 1: H holds all Cp channels; 2: H holds half of them at a time
                           // (conv2 runs in two K halves), leaving shared memory to the
                           // weight ring of the widest units
  int skip_L;              // rows of one plane of the fp32 residual input x
  long long skip_elems;    // floats of the residual input (the self-checking build's bound)
};

// Epilogue 1, first part: this warp's 32 rows of its group's chunks of acc1, copied into
// registers (B2: the two column halves added), so that acc1 can be released at once.
template <bool B2, int MC>
__device__ __forceinline__ void ru_drain1(const ConvGemmArgs &p, int grp, int n_chunks,
                                          uint32_t t1, uint32_t (&dr)[MC][16]) {
#pragma unroll
  for (int j = 0; j < MC; ++j) {
    const int c = grp + kEpiGroups * j;
    if (c < n_chunks) {  // warp-uniform: tcgen05.ld is warp-collective
      tmem_ld_issue<16>(t1 + static_cast<uint32_t>(16 * c), dr[j]);
      if constexpr (B2) {
        uint32_t r2[16];
        tmem_ld_issue<16>(t1 + static_cast<uint32_t>(16 * c + p.N_tile), r2);
        tmem_ld_wait<16>(dr[j]);
        tmem_ld16_after_wait(r2);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          dr[j][i] = __float_as_uint(__uint_as_float(dr[j][i]) + __uint_as_float(r2[i]));
      } else {
        tmem_ld_wait<16>(dr[j]);
      }
    }
  }
}

// Epilogue 1, second part: Snake2(h + b1) split into bf16 hi/lo, in place: chunk j's 16
// values become [hi 0..7 | lo 0..7 | hi 8..15 | lo 8..15] as packed pairs (4 words each).
template <int MC, bool F16 = false>
__device__ __forceinline__ void ru_act1(const RuExtra &x, int grp, int n_chunks,
                                        uint32_t (&dr)[MC][16]) {
#pragma unroll
  for (int j = 0; j < MC; ++j) {
    const int c = grp + kEpiGroups * j;
    if (c < n_chunks) {
#pragma unroll
      for (int h = 0; h < 16; h += 8) {
        const int n0 = 16 * c + h;
        float bb[8], a[8], ib[8], v[8], sn[8];
        ldg_vec(x.bias_h + n0, bb);
        ldg_vec(x.alpha_h + n0, a);
        ldg_vec(x.invb_h + n0, ib);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(dr[j][h + i]) + bb[i];
        snake_n<8>(v, a, ib, sn);
#pragma unroll
        for (int i = 0; i < 4; ++i) split_pair<F16>(sn[2 * i], sn[2 * i + 1], dr[j][h + i], dr[j][h + 4 + i]);
      }
    }
  }
}

// Epilogue 1, last part: the packed chunks of part q (of P) into the H tile.  Part q holds the
// channels [q Cp/P, (q+1) Cp/P): its 8-channel chunk k of the hi parts at H + k * 2048, of the lo
// parts at H + (Cp/(8P) + k) * 2048, row r at + 16 r.  A warp writes 32 consecutive rows of a
// chunk: 512 contiguous bytes.
template <int MC>
__device__ __forceinline__ void ru_store_h(uint32_t hbase, int Cp, int row, int grp, int n_chunks,
                                           int q, int P, const uint32_t (&dr)[MC][16]) {
  const int cpp = n_chunks / P;  // 16-column chunks per part
  const int lo0 = Cp / (8 * P);
#pragma unroll
  for (int j = 0; j < MC; ++j) {
    const int c = grp + kEpiGroups * j;
    if (c < n_chunks && c / cpp == q) {
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {  // 8-channel chunk 2c + qq: words 8qq..8qq+3 hi, +4.. lo
        const int k = 2 * (c - q * cpp) + qq;
        sts128(hbase + static_cast<uint32_t>((k * kTileM + row) * 16),
               make_uint4(dr[j][8 * qq], dr[j][8 * qq + 1], dr[j][8 * qq + 2], dr[j][8 * qq + 3]));
        sts128(hbase + static_cast<uint32_t>(((lo0 + k) * kTileM + row) * 16),
               make_uint4(dr[j][8 * qq + 4], dr[j][8 * qq + 5], dr[j][8 * qq + 6], dr[j][8 * qq + 7]));
      }
    }
  }
}

// The residual x of this thread's row t for the 16 columns n0.. (fp32 chunk-major planes of
// skip_L rows; zeros past the plane, the last tile's tail rows, which are not results).
__device__ __forceinline__ void ru_load_skip(const ConvGemmArgs &p, const RuExtra &x, int b, int t,
                                             int n0, float (&sk)[16]) {
  if (t < x.skip_L) {
    const float4 *s = reinterpret_cast<const float4 *>(p.skip) +
                      ((size_t)b * (p.Cp_out / 4) + n0 / 4) * (size_t)x.skip_L + t;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 q = s[(size_t)j * x.skip_L];
      sk[4 * j] = q.x, sk[4 * j + 1] = q.y, sk[4 * j + 2] = q.z, sk[4 * j + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) sk[i] = 0.f;
  }
}

// The four 16-byte rows of this thread's residual x for the columns n0.. into L1 (a warp covers
// 32 rows x 16 channels: 2 KB), so that epilogue 2 finds them there two chunks later.
__device__ __forceinline__ void ru_prefetch_skip_l1(const ConvGemmArgs &p, const RuExtra &x,
                                                    int b, int t, int n0) {
  if (t >= x.skip_L) return;
  const float4 *s = reinterpret_cast<const float4 *>(p.skip) +
                    ((size_t)b * (p.Cp_out / 4) + n0 / 4) * (size_t)x.skip_L + t;
#pragma unroll
  for (int j = 0; j < 4; ++j) prefetch_l1(s + (size_t)j * x.skip_L);
}

// Epilogue 2 of one warp for its 32 rows x the 16 columns n0.. of acc2 (taddr): bias, the
// residual x (sk, loaded by the caller from global memory), Snake of the next layer, hi/lo
// split and stores -- the conv kernel's epilogue of a 1x1 conv with a residual input.  HEAD:
// the output head's partial products of this row instead of stores (see epilogue_chunk).
template <bool B2, bool HEAD, bool F16 = false>
__device__ __forceinline__ bool ru_epilogue2(const ConvGemmArgs &p, volatile int *abort_flag,
                                             int b, int t, int n0, uint32_t taddr,
                                             const float (&sk)[16], float (&hp)[kHeadFoldMaxK]) {
  float bb[16];
  ldg_vec(p.bias + n0, bb);
  uint32_t r[16], r2[16];
  tmem_ld_issue<16>(taddr, r);
  if constexpr (B2) tmem_ld_issue<16>(taddr + static_cast<uint32_t>(p.N_tile), r2);
  tmem_ld_wait<16>(r);  // the TMEM reads complete before any return
  if constexpr (B2) {
    tmem_ld16_after_wait(r2);
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
  }
  float v[16], sn[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = (__uint_as_float(r[i]) + bb[i]) + sk[i];
  if (p.alpha) {
    float a[16], ib[16];
    ldg_vec(p.alpha + n0, a);
    ldg_vec(p.invb + n0, ib);
    snake_n<16>(v, a, ib, sn);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) sn[i] = v[i];
  }
  if (t >= p.rows_pad) return true;
  if (t >= p.rows_valid) {  // padding rows: zeros
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.f, sn[i] = 0.f;
  }
  if constexpr (HEAD) {  // the folded output head: this row's partial products per tap
#pragma unroll
    for (int k = 0; k < kHeadFoldMaxK; ++k) {
      float w[16];
      ldg_vec(p.head_w + (size_t)k * p.Cp_out + n0, w);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc = fmaf(w[i], sn[i], acc);
      hp[k] = acc;
      asm volatile("" ::: "memory");  // one tap's weights in registers at a time
    }
    return true;
  }
  if (p.out_f32) {
    const size_t L_out = static_cast<size_t>(p.f32_L);
    const size_t row = static_cast<size_t>(t) + p.f32_row0;
    const float *src = (p.flags & EPI_F32_SNAKE) ? sn : v;
    VOC_CHECK((((long long)b * (p.Cp_out / 4) + n0 / 4 + 3) * (long long)L_out + row) * 4 + 4 <=
                  p.f32_elems, 52, b, n0, row);
    float *base = p.out_f32 + ((size_t)b * (p.Cp_out / 4) + n0 / 4) * L_out * 4 + row * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<float4 *>(base + (size_t)j * L_out * 4) =
          make_float4(src[4 * j], src[4 * j + 1], src[4 * j + 2], src[4 * j + 3]);
  }
  if (p.out_hl) {
    uint32_t hw[8], lw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) split_pair<F16>(sn[2 * i], sn[2 * i + 1], hw[i], lw[i]);
    const size_t L_out = static_cast<size_t>(p.hl_L);
    const size_t row = static_cast<size_t>(t) + p.hl_row0;
    const size_t item = (size_t)b * (2 * p.Cp_out / 8);
    VOC_CHECK((((long long)item + p.Cp_out / 8 + n0 / 8 + 1) * (long long)L_out + row) * 8 + 8 <=
                  p.hl_elems, 53, b, n0, row);
    __nv_bfloat16 *hbase = p.out_hl + (item + n0 / 8) * L_out * 8 + row * 8;
    __nv_bfloat16 *lbase = p.out_hl + (item + p.Cp_out / 8 + n0 / 8) * L_out * 8 + row * 8;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      *reinterpret_cast<uint4 *>(hbase + (size_t)j * L_out * 8) =
          make_uint4(hw[4 * j], hw[4 * j + 1], hw[4 * j + 2], hw[4 * j + 3]);
      *reinterpret_cast<uint4 *>(lbase + (size_t)j * L_out * 8) =
          make_uint4(lw[4 * j], lw[4 * j + 1], lw[4 * j + 2], lw[4 * j + 3]);
    }
  }
  return true;
}

// RES: resident weights (ConvGemmArgs::b_resident; the narrow units): every weight stage of both
// convolutions has a slot of its own, filled once by the first tile and kept.
template <bool B2, bool HEAD = false, bool RES = false, int PREC = kPrecBf16x3>
__global__ void __launch_bounds__(kRuThreads, 1)
    ru_gemm_kernel(const __grid_constant__ CUtensorMap tmapA, const ConvGemmArgs p,
                   const RuExtra x) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smA + (size_t)p.na * p.a_bytes;
  uint8_t *smH = smB + (size_t)p.nb * p.b_bytes;    // conv2 operand (Snake2 of conv1)
  uint64_t *bars = reinterpret_cast<uint64_t *>(smH + x.h_bytes);
  uint64_t *fullA = bars;
  uint64_t *emptyA = fullA + p.na;
  uint64_t *fullB = emptyA + p.na;
  uint64_t *emptyB = fullB + p.nb;
  uint64_t *acc1Full = emptyB + p.nb;
  uint64_t *acc1Empty = acc1Full + 1;
  uint64_t *acc2Full = acc1Empty + 1;
  uint64_t *acc2Empty = acc2Full + 1;
  uint64_t *hFull = acc2Empty + 1;
  uint64_t *hEmpty = hFull + 1;
  uint64_t *drain = hEmpty + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t tmem_cols = static_cast<uint32_t>(2 * p.acc_cols);  // acc1, acc2
#ifdef VOC_CHECKS
  if (reinterpret_cast<const volatile uint8_t *>(abort_flag + 1) > smem_raw + p.smem_bytes) {
    if (threadIdx.x == 0 && atomicCAS(p.dbg, 0, 1) == 0) {
      p.dbg[1] = static_cast<int>(reinterpret_cast<const volatile uint8_t *>(abort_flag + 1) - smem_raw);
      p.dbg[2] = p.smem_bytes;
    }
    return;  // uniform over the grid
  }
#endif

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.na; ++i) {
      mbar_init(smem_u32(fullA + i), 1);
      mbar_init(smem_u32(emptyA + i), 1);
    }
    for (int i = 0; i < p.nb; ++i) {
      mbar_init(smem_u32(fullB + i), 1);
      mbar_init(smem_u32(emptyB + i), 1);
    }
    mbar_init(smem_u32(acc1Full), 1);
    mbar_init(smem_u32(acc1Empty), kRuEpiWarps * 32);  // every epilogue thread arrives
    mbar_init(smem_u32(acc2Full), 1);
    mbar_init(smem_u32(acc2Empty), kRuEpiWarps * 32);
    mbar_init(smem_u32(hFull), kRuEpiWarps * 32);
    mbar_init(smem_u32(hEmpty), 1);
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
  pdl_launch_dependents();

  const int total_tiles = p.B * p.m_tiles;  // one column tile: N_tile = Cp
  // tiles of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ... (the grid is <= total_tiles)
  const int n_my = (total_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                   static_cast<int>(gridDim.x);
  const int kchunks = p.KB / 8;
  const int nkb2 = p.Cp_out / p.KB;
  const uint32_t chunkA = static_cast<uint32_t>(p.rows) * 16u;
  const uint32_t chunkB = static_cast<uint32_t>(p.N_tile) * 16u;
  const uint32_t chunkH = kTileM * 16u;
  const int n_chunks = p.N_tile / 16;

  // Each role changes its warp's register count first thing in its own branch (all four warps of
  // a warp group execute the same change), so that the compiler allocates each role's code
  // within its own count.
  if (warp == 0) {
    regs_dec<kRuCopyRegs>();
    if (lane == 0) {
      // ------------------------------------------------------------ A producer
      prefetch_tmap(&tmapA);
      pdl_wait();  // the previous layer's output
      const uint32_t a_tx = 2u * kchunks * chunkA;
      int ia = 0;
      bool ok = true;
      for (int it = 0; it < n_my && ok; ++it) {
        const int tile = static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
        const int mt = tile % p.m_tiles;
        const int b = tile / p.m_tiles;
        const int yg = floor_div8(p.in_row0 + mt * kTileM + p.off_min);  // 8-row group
        for (int kb = 0; kb < p.nkb; ++kb) {
          const int sa = ia % p.na;
          const uint32_t pha = static_cast<uint32_t>(ia / p.na) & 1u;
          if (!mbar_wait(smem_u32(emptyA + sa), pha ^ 1u, p.timeout, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fa = smem_u32(fullA + sa);
          const uint32_t dstA = smem_u32(smA + (size_t)sa * p.a_bytes);
#ifdef VOC_CHECKS
          if (!(dstA + a_tx <= smem_u32(smB) && (kb + 1) * kchunks <= p.chunks_a / 2 &&
                a_tx <= (uint32_t)p.a_bytes)) {
            check_fail(p, abort_flag, 54, dstA, kb, p.chunks_a);
            ok = false;
            break;
          }
#endif
          mbar_arrive_expect_tx(fa, a_tx);
          tma_load_5d(dstA, &tmapA, fa, 0, yg, kb * kchunks, 0, b);  // hi and lo chunks
          ++ia;
        }
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_PRODUCER);
        *abort_flag = 1;
        drain_ring(fullA, p.na, ia, kDrainBudget);  // copies in flight land before the CTA exits
      }
    }
  } else if (warp == 1) {
    regs_dec<kRuCopyRegs>();
    // -------------------------------------------------------------- MMA issuer (whole warp)
    // warp-uniform waits; one elected lane issues each MMA and commit
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.timeout, abort_flag));
    };
    constexpr bool F16 = PREC == kPrecF16w;   // f16 operands (else bf16)
    constexpr bool ONE = PREC != kPrecBf16x3;  // one weight plane: A_hi x W + A_lo x W
    static_assert(!(ONE && (B2 || RES)), "the one-plane forms stream their weights, three-MMA layout");
    const uint32_t idesc = F16 ? idesc_f16_f32(kTileM, p.N_tile) : idesc_bf16_f32(kTileM, p.N_tile);
    const uint32_t idesc2 = idesc_bf16_f32(kTileM, 2 * p.N_tile);  // B2: [W_hi | W_lo]
    // B2: each chunk of a weight stage holds its N hi rows, then its N lo rows
    const uint32_t chunkB_stride = B2 ? 2 * chunkB : chunkB;
    // descriptor low words, stepped in 16-byte units (see mma_bf16_warp_lo)
    const uint32_t dA_lo = (kchunks * chunkA) >> 4;
    const uint32_t dA_k = (2 * chunkA) >> 4;
    const uint32_t dB_lo = (kchunks * chunkB) >> 4;
    const uint32_t dB_k = (2 * chunkB_stride) >> 4;
    const uint32_t dH_lo = ((p.Cp_out / (8 * x.h_parts)) * chunkH) >> 4;  // lo plane of a part
    const int nkb2p = nkb2 / x.h_parts;  // k-blocks of one part
    const uint32_t dH_k = (2 * chunkH) >> 4;
    const uint32_t desc_hi = static_cast<uint32_t>(smem_desc(0u, 0u, 128) >> 32);
    const uint32_t a_desc0 = static_cast<uint32_t>(smem_desc(smem_u32(smA), chunkA, 128));
    const uint32_t b_desc0 = static_cast<uint32_t>(smem_desc(smem_u32(smB), chunkB_stride, 128));
    const uint32_t h_desc0 = static_cast<uint32_t>(smem_desc(smem_u32(smH), chunkH, 128));
    const uint32_t a_slot_step = static_cast<uint32_t>(p.a_bytes) >> 4;
    const uint32_t b_slot_step = static_cast<uint32_t>(p.b_bytes) >> 4;
    const int nks = kchunks / 2;
    const uint32_t d1 = tmem_base;
    const uint32_t d2 = tmem_base + static_cast<uint32_t>(p.acc_cols);
    int sa = 0, sb = 0;
    uint32_t pha = 0, phb = 0;
    // the K steps of one weight stage: A (hi at a_hi, lo a_lo further), B at b_hi
    auto ksteps = [&](uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t a_k, uint32_t b_hi,
                      uint32_t accum) {
      for (int ks = 0; ks < nks; ++ks, a_hi += a_k, b_hi += dB_k) {
        if constexpr (ONE) {
          mma_bf16_warp_lo<false>(d, a_hi, b_hi, desc_hi, idesc, accum);
          mma_bf16_warp_lo<false>(d, a_hi + a_lo, b_hi, desc_hi, idesc, 1u);
        } else if constexpr (B2) {
          mma_bf16_warp_lo<false>(d, a_hi, b_hi, desc_hi, idesc2, accum);
          mma_bf16_warp_lo<false>(d, a_hi + a_lo, b_hi, desc_hi, idesc, 1u);
        } else {  // A_hi x W_hi and A_hi x W_lo share A through the collector buffer
          mma_bf16_warp_lo_col<false, 1>(d, a_hi, b_hi, desc_hi, idesc, accum);
          mma_bf16_warp_lo_col<false, 2>(d, a_hi, b_hi + dB_lo, desc_hi, idesc, 1u);
          mma_bf16_warp_lo<false>(d, a_hi + a_lo, b_hi, desc_hi, idesc, 1u);
        }
        accum = 1u;
      }
    };
    bool ok = true;
    for (int it = 0; it <= n_my && ok; ++it) {
      if (it < n_my) {  // conv1 (k taps, dilated) of tile it -> acc1
        if (!wait_all(smem_u32(acc1Empty), (static_cast<uint32_t>(it) & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t accum = 0u;
        for (int kb = 0; kb < p.nkb && ok; ++kb) {
          if (!wait_all(smem_u32(fullA + sa), pha)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t a0 = a_desc0 + sa * a_slot_step + static_cast<uint32_t>(p.shift0_q0);
          for (int tap = 0; tap < p.taps; ++tap, a0 += static_cast<uint32_t>(p.tap_step)) {
            // resident weights: stage (kb, tap) has a slot of its own, filled once (phase 0)
            const int rb = RES ? kb * p.taps + tap : sb;
            if (!wait_all(smem_u32(fullB + rb), RES ? 0u : phb)) {
              ok = false;
              break;
            }
            tc_fence_after();
#ifdef VOC_CHECKS
            {
              const int sh = p.shift0_q0 + tap * p.tap_step;
              if (!__all_sync(0xffffffffu, sh >= 0 && sh + kTileM <= p.rows)) {
                if (lane == 0) check_fail(p, abort_flag, 55, sh, tap, p.rows);
                ok = false;
                break;
              }
            }
#endif
            ksteps(d1, a0, dA_lo, dA_k, b_desc0 + rb * b_slot_step, accum);
            accum = 1u;
            if constexpr (!RES) {
              mma_commit_warp(smem_u32(emptyB + sb));
              if (++sb == p.nb) sb = 0, phb ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_warp(smem_u32(emptyA + sa));
          if (++sa == p.na) sa = 0, pha ^= 1u;
        }
        if (!ok) break;
        mma_commit_warp(smem_u32(acc1Full));
      }
      if (it >= 1) {  // conv2 (1x1) of tile it - 1 on H -> acc2, in h_parts K ranges
        const int jt = it - 1;
        uint32_t accum = 0u;
        for (int q = 0; q < x.h_parts && ok; ++q) {
          const uint32_t g = static_cast<uint32_t>(jt * x.h_parts + q);  // H fill number
          if (!wait_all(smem_u32(hFull), g & 1u) ||
              (q == 0 && !wait_all(smem_u32(acc2Empty), (static_cast<uint32_t>(jt) & 1u) ^ 1u))) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < nkb2p; ++kb) {
            // resident weights: conv2's k-blocks follow conv1's stages
            const int rb = RES ? p.nkb * p.taps + q * nkb2p + kb : sb;
            if (!wait_all(smem_u32(fullB + rb), RES ? 0u : phb)) {
              ok = false;
              break;
            }
            tc_fence_after();
            ksteps(d2, h_desc0 + static_cast<uint32_t>(kb * kchunks) * (chunkH >> 4), dH_lo, dH_k,
                   b_desc0 + rb * b_slot_step, accum);
            accum = 1u;
            if constexpr (!RES) {
              mma_commit_warp(smem_u32(emptyB + sb));
              if (++sb == p.nb) sb = 0, phb ^= 1u;
            }
          }
          if (!ok) break;
          if (q == x.h_parts - 1) mma_commit_warp(smem_u32(acc2Full));
          mma_commit_warp(smem_u32(hEmpty));  // H may be rewritten once these MMAs have read it
        }
        if (!ok) break;
      }
    }
    if (!ok) {
      if (lane == 0) {
        atomicOr(p.err, ERR_TIMEOUT_MMA);
        *abort_flag = 1;
      }
      // wait until every MMA issued so far has finished reading shared memory and TMEM
      mma_commit_warp(smem_u32(drain));
      const volatile int never = 0;
      mbar_wait(smem_u32(drain), 0u, kDrainBudget, &never);
    }
  } else if (warp == kRuBWarp) {
    regs_dec<kRuCopyRegs>();
    if (lane == 0) {
      // ------------------------------------------------------------ weight producer
      // Stages in the MMA warp's order: conv1 of tile it (k-blocks x taps), then conv2 of
      // tile it - 1 (k-blocks).
      int ib = 0;
      bool ok = true;
      auto load_b = [&](const uint8_t *src) -> bool {
        const int sb = ib % p.nb;
        const uint32_t phb = static_cast<uint32_t>(ib / p.nb) & 1u;
        if (!mbar_wait(smem_u32(emptyB + sb), phb ^ 1u, p.timeout, abort_flag)) return false;
        const uint32_t fb = smem_u32(fullB + sb);
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(p.b_bytes));
        bulk_load(smem_u32(smB + (size_t)sb * p.b_bytes), src, static_cast<uint32_t>(p.b_bytes), fb);
        ++ib;
        return true;
      };
      // resident weights: every stage once, into slots 0, 1, ... in this order (conv1's k-blocks
      // x taps, then conv2's k-blocks), kept for every tile
      const int n_it = RES ? 1 : n_my;
      for (int it = 0; it <= n_it && ok; ++it) {
        if (it < n_it)
          for (int kb = 0; kb < p.nkb && ok; ++kb)
            for (int tap = 0; tap < p.taps && ok; ++tap)
              ok = load_b(p.wB + ((size_t)tap * p.nkb + kb) * p.b_bytes);
        if (it >= 1)
          for (int kb = 0; kb < nkb2 && ok; ++kb) ok = load_b(x.wB2 + (size_t)kb * p.b_bytes);
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_PRODUCER);
        *abort_flag = 1;
        drain_ring(fullB, p.nb, ib, kDrainBudget);
      }
    }
  } else if (warp < kRuEpi0) {
    regs_dec<kRuCopyRegs>();  // warp 3: no role
  } else {
    regs_inc<kRuEpiRegs>();
    // -------------------------------------------------------------- epilogue
    pdl_wait();  // the residual input is the previous layer's output; this unit's outputs
                 // overwrite buffers earlier layers read
    const int e = warp - kRuEpi0;
    const int quad = warp & 3;   // TMEM lane quadrant this warp may access
    const int grp = e / 4;       // column chunks grp, grp + 3, ...
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t t1 = tmem_base + lanes;
    const uint32_t t2 = t1 + static_cast<uint32_t>(p.acc_cols);
    const uint32_t hbase = smem_u32(smH);
    constexpr int MC = ru_max_chunks<B2>();
    uint32_t dr[MC][16];
    bool ok = true;
    for (int it = 0; it <= n_my && ok; ++it) {
      if (it < n_my && quad == 0 && lane == 0) {
        // the residual rows of tile it, used by its epilogue 2 in the next iteration: into L2
        // now (one 2 KB run of 128 rows per 4-channel plane of this group's chunks)
        const int tile = static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
        const int mt = tile % p.m_tiles;
        const int b = tile / p.m_tiles;
        const int rows = min(kTileM, x.skip_L - mt * kTileM);
        if (rows > 0)
          for (int c = grp; c < n_chunks; c += kEpiGroups)
            for (int j = 0; j < 4; ++j)
              bulk_prefetch_l2(p.skip + (((size_t)b * (p.Cp_out / 4) + 4 * c + j) * (size_t)x.skip_L +
                                         (size_t)mt * kTileM) * 4,
                               static_cast<uint32_t>(rows) * 16u);
      }
      if (it >= 1 && x.h_parts == 2) {
        // the second half of H(it - 1), from the registers of tile it - 1, once conv2 has read
        // the first half
        const uint32_t g = static_cast<uint32_t>((it - 1) * 2 + 1);  // H fill number
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(hEmpty), (g - 1u) & 1u, p.timeout, abort_flag))) {
          ok = false;
          break;
        }
        ru_store_h<MC>(hbase, p.Cp_out, row_in_tile, grp, n_chunks, 1, 2, dr);
        fence_proxy_async_smem();  // the H stores become visible to the tensor cores
        mbar_arrive(smem_u32(hFull));
      }
      if (it < n_my) {
        // epilogue 1 of tile it: acc1 -> registers (acc1 released), Snake2 -> H (the first
        // half when H holds half of the channels)
        const uint32_t ip = static_cast<uint32_t>(it) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(acc1Full), ip, p.timeout, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        ru_drain1<B2, MC>(p, grp, n_chunks, t1, dr);
        tc_fence_before();
        mbar_arrive(smem_u32(acc1Empty));
        ru_act1<MC, PREC == kPrecF16w>(x, grp, n_chunks, dr);
        // H is free once conv2 has read the previous fill
        const int g = it * x.h_parts;  // H fill number (fill -1 counts as complete)
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(hEmpty), static_cast<uint32_t>(g - 1) & 1u,
                                               p.timeout, abort_flag))) {
          ok = false;
          break;
        }
        ru_store_h<MC>(hbase, p.Cp_out, row_in_tile, grp, n_chunks, 0, x.h_parts, dr);
        fence_proxy_async_smem();  // the H stores become visible to the tensor cores
        mbar_arrive(smem_u32(hFull));
      }
      if (it >= 1) {
        // epilogue 2 of tile it - 1: acc2 -> outputs
        const int jt = it - 1;
        const int tile = static_cast<int>(blockIdx.x) + jt * static_cast<int>(gridDim.x);
        const int mt = tile % p.m_tiles;
        const int b = tile / p.m_tiles;
        const int t = mt * kTileM + row_in_tile;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(acc2Full), static_cast<uint32_t>(jt) & 1u,
                                               p.timeout, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float skn[16];  // x of the warp's next chunk, loaded one chunk ahead
        if (grp < n_chunks) ru_load_skip(p, x, b, t, 16 * grp, skn);
        for (int c = grp; c < n_chunks && ok; c += kEpiGroups) {
          float sk[16], hp[kHeadFoldMaxK] = {};
#pragma unroll
          for (int i = 0; i < 16; ++i) sk[i] = skn[i];
          if (c + kEpiGroups < n_chunks) ru_load_skip(p, x, b, t, 16 * (c + kEpiGroups), skn);
          // and the chunk after it into L1 (into L2 every chunk came one tile earlier)
          if (c + 2 * kEpiGroups < n_chunks) ru_prefetch_skip_l1(p, x, b, t, 16 * (c + 2 * kEpiGroups));
          ok = ru_epilogue2<B2, HEAD, PREC == kPrecF16w>(p, abort_flag, b, t, 16 * c,
                                                        t2 + static_cast<uint32_t>(16 * c), sk, hp);
          ok = __all_sync(0xffffffffu, ok);
          if constexpr (HEAD) {
            if (ok) ok = head_fold_store(p, hp, b, (mt * kTileM) / 32 + quad, c, lane, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
          }
        }
        tc_fence_before();
        if (!ok) break;
        mbar_arrive(smem_u32(acc2Empty));
      }
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
