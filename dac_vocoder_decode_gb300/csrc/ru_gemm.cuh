// ru_gemm.cuh -- one residual unit of the decoder in one kernel, for stages of up to
// 192 channels (minimaxmusic.cpp Architecture, "Flow VAE": res_unit = skip -> snake1
// -> conv1 k7 dil d -> snake2 -> conv2 k1 -> + skip):
//
//   h  = conv1(A) + b1                     A = Snake1(x) as bf16 hi/lo, from HBM (TMA, halo)
//   H  = Snake2(h) as bf16 hi/lo           written by the epilogue into SHARED memory, in
//                                          the canonical K-major layout of an MMA operand
//   y  = x + conv2(H) + b2                 x streamed in by the residual prefetch warp
//
// so the conv1 result never goes to HBM.  Per 128-row tile the MMA warp runs the 7-tap
// mainloop into accumulator 1, waits until the epilogue warps have turned accumulator 1
// into H, then runs the 1x1 mainloop (A = H, weights streamed through the same ring) into
// accumulator 2; the epilogue finishes the tile from accumulator 2 exactly like the
// separate conv2 kernel.  Two accumulator pairs (when they fit in TMEM) let conv1 of the
// next tile overlap the epilogue of this one.
//
// B2 (units of up to 128 channels): both mainloops take the two-MMA K step of the conv kernel's
// B2 form -- A_hi x [W_hi | W_lo] into 2N accumulator columns, then A_lo x W_hi into the first
// N -- and both epilogues add the two column halves.  A narrow layer's MMAs cost about the same
// whatever their N (the A operand is re-read for each), so this removes a third of them.
#pragma once
#include "conv_gemm.cuh"

namespace voc {

struct RuExtra {
  const uint8_t *wB2;      // packed k1 weight tiles [kb][hi|lo][chunk][n][8]
  const float *bias_h;     // [N] conv1 bias
  const float *alpha_h;    // [N] Snake2 alpha
  const float *invb_h;     // [N] Snake2 1/(alpha + 1e-9)
  int h_bytes;             // bytes of the H tile (4 * 128 * Cp)
  int n_buf;               // accumulator pairs (1 or 2)
};

// Epilogue 1 of one warp: rows quad*32.. of accumulator 1, columns n0..n0+CW-1 ->
// Snake2(acc + b1) split into hi/lo, stored into the H tile: 8-channel chunk j of the hi
// parts at H + j*2048, of the lo parts at H + (Cp/8 + j)*2048, row r at +16*r.
template <int CW, bool B2>
__device__ __forceinline__ void ru_epilogue1(const ConvGemmArgs &p, const RuExtra &x, uint32_t hbase,
                                             int row_in_tile, int n0, uint32_t taddr) {
  float v[CW];
  if constexpr (B2) {  // (CW = 16) the two column halves of the accumulator
    static_assert(CW == 16, "the B2 epilogue reads 16-column chunks");
    uint32_t r[CW], r2[CW];
    tmem_ld_issue<CW>(taddr, r);
    tmem_ld_issue<CW>(taddr + static_cast<uint32_t>(p.N_tile), r2);
    tmem_ld_wait<CW>(r);
    tmem_ld16_after_wait(r2);
#pragma unroll
    for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[i]) + __uint_as_float(r2[i]);
  } else {
    tmem_ld(taddr, v);
  }
  float bb[CW], a[CW], ib[CW];
  ldg_vec(x.bias_h + n0, bb);
  ldg_vec(x.alpha_h + n0, a);
  ldg_vec(x.invb_h + n0, ib);
#pragma unroll
  for (int i = 0; i < CW; ++i) v[i] += bb[i];
  float sn[CW];
  snake_n<CW>(v, a, ib, sn);
  uint32_t hw[CW / 2], lw[CW / 2];
#pragma unroll
  for (int i = 0; i < CW / 2; ++i) {
    const float s0 = sn[2 * i], s1 = sn[2 * i + 1];
    const __nv_bfloat16 h0 = __float2bfloat16_rn(s0), h1 = __float2bfloat16_rn(s1);
    const __nv_bfloat16 l0 = __float2bfloat16_rn(s0 - __bfloat162float(h0));
    const __nv_bfloat16 l1 = __float2bfloat16_rn(s1 - __bfloat162float(h1));  // bf16x3 only
    hw[i] = pack_bf16x2(h0, h1);
    lw[i] = pack_bf16x2(l0, l1);
  }
  const int lo0 = p.Cp_out / 8;
#pragma unroll
  for (int g = 0; g < CW / 8; ++g) {
    const int j = n0 / 8 + g;
    sts128(hbase + static_cast<uint32_t>(j * (kTileM * 16) + row_in_tile * 16),
           make_uint4(hw[4 * g], hw[4 * g + 1], hw[4 * g + 2], hw[4 * g + 3]));
    sts128(hbase + static_cast<uint32_t>((lo0 + j) * (kTileM * 16) + row_in_tile * 16),
           make_uint4(lw[4 * g], lw[4 * g + 1], lw[4 * g + 2], lw[4 * g + 3]));
  }
}

template <int CW, bool B2 = false>
__global__ void __launch_bounds__(kRuThreads, 1)
    ru_gemm_kernel(const __grid_constant__ CUtensorMap tmapA,
                   const __grid_constant__ CUtensorMap tmapS, const ConvGemmArgs p,
                   const RuExtra x) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smA + (size_t)p.na * p.a_bytes;
  uint8_t *smH = smB + (size_t)p.nb * p.b_bytes;    // conv2 operand (conv1 result)
  uint8_t *smS = smH + x.h_bytes;                   // residual slots
  uint64_t *bars = reinterpret_cast<uint64_t *>(smS + (size_t)p.ns * skip_slot_bytes(CW));
  uint64_t *fullA = bars;
  uint64_t *emptyA = fullA + p.na;
  uint64_t *fullB = emptyA + p.na;
  uint64_t *emptyB = fullB + p.nb;
  uint64_t *acc1Full = emptyB + p.nb;
  uint64_t *acc1Empty = acc1Full + 2;
  uint64_t *acc2Full = acc1Empty + 2;
  uint64_t *acc2Empty = acc2Full + 2;
  uint64_t *hFull = acc2Empty + 2;
  uint64_t *hEmpty = hFull + 1;
  uint64_t *skipFull = hEmpty + 1;
  uint64_t *skipEmpty = skipFull + p.ns;
  uint64_t *drain = skipEmpty + p.ns;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t tmem_cols = static_cast<uint32_t>(2 * x.n_buf * p.acc_cols);

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
      mbar_init(smem_u32(acc1Full + i), 1);
      mbar_init(smem_u32(acc1Empty + i), kRuEpiWarps * 32);
      mbar_init(smem_u32(acc2Full + i), 1);
      mbar_init(smem_u32(acc2Empty + i), kRuEpiWarps * 32);
    }
    mbar_init(smem_u32(hFull), kRuEpiWarps * 32);
    mbar_init(smem_u32(hEmpty), 1);
    for (int i = 0; i < p.ns; ++i) {
      mbar_init(smem_u32(skipFull + i), 1);
      mbar_init(smem_u32(skipEmpty + i), 4 * 32);
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
  pdl_launch_dependents();

  const int total_tiles = p.B * p.m_tiles;  // one column tile: N_tile = Cp
  const int kchunks = p.KB / 8;
  const int nkb2 = p.Cp_out / p.KB;
  const uint32_t chunkA = static_cast<uint32_t>(p.rows) * 16u;
  const uint32_t chunkB = static_cast<uint32_t>(p.N_tile) * 16u;
  const uint32_t chunkH = kTileM * 16u;
  const int n_chunks = p.N_tile / CW;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ A / weight producer
      prefetch_tmap(&tmapA);
      pdl_wait();  // the previous layer's output
      const uint32_t a_tx = 2u * kchunks * chunkA;
      int ia = 0, ib = 0;
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
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        const int mt = tile % p.m_tiles;
        const int b = tile / p.m_tiles;
        const int yg = floor_div8(p.in_row0 + mt * kTileM + p.off_min);  // 8-row group
        for (int kb = 0; kb < p.nkb && ok; ++kb) {
          const int sa = ia % p.na;
          const uint32_t pha = static_cast<uint32_t>(ia / p.na) & 1u;
          if (!mbar_wait(smem_u32(emptyA + sa), pha ^ 1u, p.timeout, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fa = smem_u32(fullA + sa);
          const uint32_t dstA = smem_u32(smA + (size_t)sa * p.a_bytes);
          mbar_arrive_expect_tx(fa, a_tx);
          tma_load_5d(dstA, &tmapA, fa, 0, yg, kb * kchunks, 0, b);  // hi and lo chunks
          ++ia;
          for (int tap = 0; tap < p.taps && ok; ++tap)
            ok = load_b(p.wB + ((size_t)tap * p.nkb + kb) * p.b_bytes);
        }
        for (int kb = 0; kb < nkb2 && ok; ++kb) ok = load_b(x.wB2 + (size_t)kb * p.b_bytes);
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_PRODUCER);
        *abort_flag = 1;
        drain_ring(fullA, p.na, ia, kDrainBudget);
        drain_ring(fullB, p.nb, ib, kDrainBudget);
      }
    }
  } else if (warp == 1) {
    {
      // ------------------------------------------------------------ MMA issuer (whole warp)
      // warp-uniform waits, one elected lane issues each MMA and commit
      auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.timeout, abort_flag));
      };
      const uint32_t idesc = idesc_bf16_f32(kTileM, p.N_tile);
      const uint32_t idesc2 = idesc_bf16_f32(kTileM, 2 * p.N_tile);  // B2: [W_hi | W_lo]
      // B2: each chunk of a weight stage holds its N hi rows, then its N lo rows
      const uint32_t chunkB_stride = B2 ? 2 * chunkB : chunkB;
      const uint64_t dA_lo = (uint64_t)((kchunks * chunkA) >> 4);
      const uint64_t dA_k = (uint64_t)((2 * chunkA) >> 4);
      const uint64_t dB_lo = (uint64_t)((kchunks * chunkB) >> 4);
      const uint64_t dB_k = (uint64_t)((2 * chunkB_stride) >> 4);
      const uint64_t dH_lo = (uint64_t)(((p.Cp_out / 8) * chunkH) >> 4);
      const uint64_t dH_k = (uint64_t)((2 * chunkH) >> 4);
      const uint64_t h0 = smem_desc(smem_u32(smH), chunkH, 128);
      // ring positions advance incrementally (no divisions in the issue loop)
      int sa = 0, sb = 0, j = 0;
      uint32_t pha = 0, phb = 0, ph = 0;
      int it = 0;
      bool ok = true;
      auto wait_b = [&](uint64_t &b0) -> bool {
        if (!wait_all(smem_u32(fullB + sb), phb)) return false;
        tc_fence_after();
        b0 = smem_desc(smem_u32(smB + (size_t)sb * p.b_bytes), chunkB_stride, 128);
        return true;
      };
      auto release_b = [&]() {
        mma_commit_warp(smem_u32(emptyB + sb));
        if (++sb == p.nb) sb = 0, phb ^= 1u;
      };
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++it) {
        const uint32_t d1 = tmem_base + static_cast<uint32_t>(2 * j * p.acc_cols);
        const uint32_t d2 = d1 + static_cast<uint32_t>(p.acc_cols);
        // conv1 (k taps, dilated) -> accumulator 1
        if (!wait_all(smem_u32(acc1Empty + j), ph ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < p.nkb && ok; ++kb) {
          if (!wait_all(smem_u32(fullA + sa), pha)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aBase = smem_u32(smA + (size_t)sa * p.a_bytes);
          for (int tap = 0; tap < p.taps; ++tap) {
            uint64_t b0;
            if (!wait_b(b0)) {
              ok = false;
              break;
            }
            const uint64_t a0 = smem_desc(
                aBase + static_cast<uint32_t>(p.shift0_q0 + tap * p.tap_step) * 16u, chunkA, 128);
            for (int ks = 0; ks < kchunks / 2; ++ks) {
              const uint64_t a_hi = a0 + ks * dA_k, a_lo = a_hi + dA_lo;
              const uint64_t b_hi = b0 + ks * dB_k, b_lo = b_hi + dB_lo;
              const uint32_t accum = (kb | tap | ks) ? 1u : 0u;
              if constexpr (B2) {
                mma_bf16_warp(d1, a_hi, b_hi, idesc2, accum);
                mma_bf16_warp(d1, a_lo, b_hi, idesc, 1u);
              } else {
                mma_bf16_warp(d1, a_hi, b_hi, idesc, accum);
                mma_bf16_warp(d1, a_hi, b_lo, idesc, 1u);
                mma_bf16_warp(d1, a_lo, b_hi, idesc, 1u);
              }
            }
            release_b();
          }
          if (!ok) break;
          mma_commit_warp(smem_u32(emptyA + sa));
          if (++sa == p.na) sa = 0, pha ^= 1u;
        }
        if (!ok) break;
        mma_commit_warp(smem_u32(acc1Full + j));
        // conv2 (1x1) on H -> accumulator 2, once the epilogue has written H
        if (!wait_all(smem_u32(hFull), static_cast<uint32_t>(it) & 1u) ||
            !wait_all(smem_u32(acc2Empty + j), ph ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < nkb2 && ok; ++kb) {
          uint64_t b0;
          if (!wait_b(b0)) {
            ok = false;
            break;
          }
          const uint64_t a0 = h0 + (uint64_t)((kb * kchunks * chunkH) >> 4);
          for (int ks = 0; ks < kchunks / 2; ++ks) {
            const uint64_t a_hi = a0 + ks * dH_k, a_lo = a_hi + dH_lo;
            const uint64_t b_hi = b0 + ks * dB_k, b_lo = b_hi + dB_lo;
            const uint32_t accum = (kb | ks) ? 1u : 0u;
            if constexpr (B2) {
              mma_bf16_warp(d2, a_hi, b_hi, idesc2, accum);
              mma_bf16_warp(d2, a_lo, b_hi, idesc, 1u);
            } else {
              mma_bf16_warp(d2, a_hi, b_hi, idesc, accum);
              mma_bf16_warp(d2, a_hi, b_lo, idesc, 1u);
              mma_bf16_warp(d2, a_lo, b_hi, idesc, 1u);
            }
          }
          release_b();
        }
        if (!ok) break;
        mma_commit_warp(smem_u32(acc2Full + j));
        mma_commit_warp(smem_u32(hEmpty));  // H may be rewritten once these MMAs have read it
        if (++j == x.n_buf) j = 0, ph ^= 1u;
      }
      if (!ok) {
        if (lane == 0) {
          atomicOr(p.err, ERR_TIMEOUT_MMA);
          *abort_flag = 1;
        }
        mma_commit_warp(smem_u32(drain));
        const volatile int never = 0;
        mbar_wait(smem_u32(drain), 0u, kDrainBudget, &never);
      }
    }
  } else if (warp == kRuSkipWarp) {
    if (lane == 0 && p.skip) {
      // ------------------------------------------------------------ residual prefetch
      prefetch_tmap(&tmapS);
      pdl_wait();
      const uint32_t bytes = static_cast<uint32_t>(skip_slot_bytes(CW));
      const int nsh = p.ns / 2;
      int cnt[2] = {0, 0};
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        const int mt = tile % p.m_tiles;
        const int b = tile / p.m_tiles;
        for (int c = 0; c < n_chunks; ++c) {
          const int h = c & 1;
          const int k = cnt[h]++;
          const int slot = h * nsh + k % nsh;
          const uint32_t ph = static_cast<uint32_t>(k / nsh) & 1u;
          if (!mbar_wait(smem_u32(skipEmpty + slot), ph ^ 1u, p.timeout, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fs = smem_u32(skipFull + slot);
          mbar_arrive_expect_tx(fs, bytes);
          tma_load_4d(smem_u32(smS + (size_t)slot * bytes), &tmapS, fs, 0, mt * kTileM / 8,
                      (c * CW) / 4, b);
        }
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_SKIP);
        *abort_flag = 1;
        drain_ring(skipFull, nsh, cnt[0], kDrainBudget);
        drain_ring(skipFull + nsh, nsh, cnt[1], kDrainBudget);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    pdl_wait();  // this unit's outputs overwrite buffers earlier layers read
    const int e = warp - 2;
    const int quad = warp & 3;
    const int half = e / 4;
    const int row_in_tile = quad * 32 + lane;
    const uint32_t sbase = smem_u32(smS);
    const uint32_t hbase = smem_u32(smH);
    const int nsh = p.ns > 0 ? p.ns / 2 : 1;
    int kh = 0;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++it) {
      const int mt = tile % p.m_tiles;
      const int b = tile / p.m_tiles;
      const int j = it % x.n_buf;
      const uint32_t ph = static_cast<uint32_t>(it / x.n_buf) & 1u;
      const uint32_t lanes = static_cast<uint32_t>(quad * 32) << 16;
      const uint32_t t1 = tmem_base + static_cast<uint32_t>(2 * j * p.acc_cols) + lanes;
      const uint32_t t2 = t1 + static_cast<uint32_t>(p.acc_cols);
      // epilogue 1: accumulator 1 -> H (shared), after conv2 of the previous tile read H
      if (!mbar_wait(smem_u32(acc1Full + j), ph, p.timeout, abort_flag) ||
          !mbar_wait(smem_u32(hEmpty), (static_cast<uint32_t>(it) & 1u) ^ 1u, p.timeout,
                     abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int c = half; c < n_chunks; c += 2)
        ru_epilogue1<CW, B2>(p, x, hbase, row_in_tile, c * CW, t1 + c * CW);
      fence_proxy_async_smem();  // make the H stores visible to the tensor cores
      tc_fence_before();
      mbar_arrive(smem_u32(acc1Empty + j));
      mbar_arrive(smem_u32(hFull));
      // epilogue 2: accumulator 2 -> bias, residual, Snake of the next layer, stores
      if (!mbar_wait(smem_u32(acc2Full + j), ph, p.timeout, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int t = mt * kTileM + row_in_tile;
      for (int c = half; c < n_chunks && ok; c += 2, ++kh) {
        const int slot = half * nsh + kh % nsh;
        ok = epilogue_chunk<CW, B2>(p, sbase + static_cast<uint32_t>(slot * skip_slot_bytes(CW)),
                                smem_u32(skipFull + slot), smem_u32(skipEmpty + slot),
                                static_cast<uint32_t>(kh / nsh) & 1u, abort_flag, row_in_tile, b,
                                t, c * CW, t2 + c * CW, sbase, smem_u32(bars));
      }
      if (!ok) break;
      tc_fence_before();
      mbar_arrive(smem_u32(acc2Empty + j));
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
