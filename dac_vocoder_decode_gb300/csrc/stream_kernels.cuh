// stream_kernels.cuh -- the bandwidth-bound kernels around the tensor-core convs:
//   prep_hl_kernel      channels-first fp32 -> chunk-major bf16 hi/lo (+ optional Snake)
//   out_head_kernel     Snake'd chunk-major fp32 -> k-tap conv to one channel (+bias) -> tanh
//   out_head_reg_kernel the same for 7 taps, register-blocked (the decoder's head)
//   stitch_kernel       overlap-crop stitch + clamp of windowed decodes
//   head_finish_kernel  the folded output head: partial sums of the last conv2 -> audio
//   ksplit_reduce_kernel the epilogue of a conv run with split k (the encoder's deep layers)
//   audio_conv_in_kernel the encoder's conv_in on a few audio channels, direct in fp32
//   finite_check_kernel flags a NaN / Inf in a buffer
//   rows_to_cf_kernel   chunk-major fp32 -> channels-first fp32 (single-layer ops)
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "hilo.cuh"
#include "ptx.cuh"
#include "snake.cuh"

namespace voc {

// x [B][C][T] fp32 -> hl chunk-major [B][2*Cp/8][Lp][8] at rows row0..row0+T-1: 8-channel
// chunks of the hi parts, then of the lo parts (hi = r(v), lo = r(v - hi), r the rounding to
// bf16, or to f16 when f16 != 0);
// channels C..Cp-1 are zeros, and so are rows T..T_pad-1 (the padding rows read by the
// 8-row TMA groups).  alpha == nullptr: no Snake.  One thread per (b, chunk, t):
// block 256, grid (ceil(T_pad/256), Cp/8, B).
__global__ void prep_hl_kernel(const float *__restrict__ x, int C, int T, int T_pad, int Cp,
                               const float *__restrict__ alpha, const float *__restrict__ invb,
                               __nv_bfloat16 *__restrict__ hl, int row0, long long Lp, int f16) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int c8 = blockIdx.y;
  const int b = blockIdx.z;
  if (t >= T_pad) return;
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    float v[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int c = c8 * 8 + e + u;
      v[u] = 0.f;
      if (c < C && t < T) {
        v[u] = x[((size_t)b * C + c) * T + t];
        if (alpha) v[u] = snake(v[u], alpha[c], invb[c]);
      }
    }
    if (f16)
      split_pair<true>(v[0], v[1], hw[e / 2], lw[e / 2]);
    else
      split_pair<false>(v[0], v[1], hw[e / 2], lw[e / 2]);
  }
  const size_t item = (size_t)b * (2 * Cp / 8);
  const size_t r = (size_t)row0 + t;
  *reinterpret_cast<uint4 *>(hl + ((item + c8) * Lp + r) * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4 *>(hl + ((item + Cp / 8 + c8) * Lp + r) * 8) =
      make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// audio[b][t] = tanh(bias + sum_k sum_c w[c][k] * y[b][c][t + k - pad_left]) for t in [0, L),
// y zero before row 0 and from row L on.  y is fp32 chunk-major [B][Cp/4][Ly][4] (already
// Snake'd) with y's row 0 stored at row in_row0 of its planes (the rows before it, if any,
// hold earlier samples and are read as such), w [Cp][K] (zero past the real channels).  One thread per output sample, TILE samples per block; the block stages
// its rows chunk by chunk in shared memory ([Cp/4][TILE+K-1][4]), so the global reads are
// contiguous runs and a warp's shared reads hit consecutive 16-byte words.
template <int TILE>
__global__ void __launch_bounds__(TILE) out_head_kernel(const float *__restrict__ y, int L, int Cp,
                                                        int K, int pad_left,
                                                        const float *__restrict__ w,
                                                        const float *__restrict__ bias,
                                                        float *__restrict__ audio, int in_row0,
                                                        long long Ly) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float4 sm4[];
  const int b = blockIdx.y;
  const int t0 = blockIdx.x * TILE;
  const int rows = TILE + K - 1;
  const int nch = Cp / 4;
  float4 *xs = sm4;                                            // [nch][rows]
  float *ws = reinterpret_cast<float *>(sm4 + (size_t)nch * rows);  // [Cp][K]
  for (int i = threadIdx.x; i < Cp * K; i += TILE) ws[i] = w[i];
  const float4 *yb = reinterpret_cast<const float4 *>(y) + (size_t)b * nch * Ly;
  for (int i = threadIdx.x; i < nch * rows; i += TILE) {
    const int j = i / rows, r = i - j * rows;
    const long long t = (long long)in_row0 + t0 - pad_left + r;  // stored row
    xs[i] = (t >= 0 && t < (long long)in_row0 + L) ? __ldg(yb + (size_t)j * Ly + t)
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  const int t = t0 + threadIdx.x;
  if (t >= L) return;
  float acc = 0.f;
  for (int k = 0; k < K; ++k) {
    for (int j = 0; j < nch; ++j) {
      const float4 xv = xs[(size_t)j * rows + threadIdx.x + k];
      acc = fmaf(ws[(4 * j + 0) * K + k], xv.x, acc);
      acc = fmaf(ws[(4 * j + 1) * K + k], xv.y, acc);
      acc = fmaf(ws[(4 * j + 2) * K + k], xv.z, acc);
      acc = fmaf(ws[(4 * j + 3) * K + k], xv.w, acc);
    }
  }
  audio[(size_t)b * L + t] = tanhf(bias[0] + acc);
}

// Same operation for a fixed tap count K, register-blocked: each thread computes TPT
// consecutive samples and keeps, per 4-channel chunk, the TPT + K - 1 input rows it needs in
// registers (neighbouring threads share rows through L1), two chunks at a time so that the
// loads of both are in flight together.  Weights are re-laid as w4[k][Cp/4] float4 (channel
// quadruples) and read by all lanes at once.  No shared memory and no block barrier.
// Requires Cp a multiple of 8.
template <int K, int TPT>
__global__ void __launch_bounds__(256) out_head_reg_kernel(const float *__restrict__ y, int L,
                                                            int Cp, int pad_left,
                                                            const float4 *__restrict__ w4,
                                                            const float *__restrict__ bias,
                                                            float *__restrict__ audio, int in_row0,
                                                            long long Ly) {
  constexpr int R = TPT + K - 1;  // input rows per chunk
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.y;
  const long long t0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * TPT;
  if (t0 >= L) return;
  const int nch = Cp / 4;
  const float4 *yb = reinterpret_cast<const float4 *>(y) + (size_t)b * nch * Ly;
  float acc[TPT];
#pragma unroll
  for (int i = 0; i < TPT; ++i) acc[i] = 0.f;
  const long long r0 = in_row0 + t0 - pad_left;  // stored row of the first input
  const long long rend = (long long)in_row0 + L;  // rows from here on read as zero
  const bool interior = r0 >= 0 && r0 + R <= rend;
  for (int j0 = 0; j0 < nch; j0 += 2) {
    float4 xs[2][R];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float4 *row = yb + (size_t)(j0 + u) * Ly;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const long long t = r0 + r;
        xs[u][r] = (interior || (t >= 0 && t < rend)) ? __ldg(row + t)
                                                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const float4 wk = __ldg(w4 + (size_t)k * nch + j0 + u);
#pragma unroll
        for (int i = 0; i < TPT; ++i) {
          const float4 xv = xs[u][i + k];
          acc[i] = fmaf(wk.x, xv.x, acc[i]);
          acc[i] = fmaf(wk.y, xv.y, acc[i]);
          acc[i] = fmaf(wk.z, xv.z, acc[i]);
          acc[i] = fmaf(wk.w, xv.w, acc[i]);
        }
      }
  }
  const float bb = bias[0];
#pragma unroll
  for (int i = 0; i < TPT; ++i)
    if (t0 + i < L) audio[(size_t)b * L + t0 + i] = tanhf(bb + acc[i]);
}

// Row-block copies between chunk-major buffers: job j copies `rows` rows starting at
// src_row0 + frames * src_rate of each of its `planes` planes (16-byte rows, plane lengths
// src_L and dst_L) to rows [dst_row0, ...).  Source and destination never overlap.
// grid (blocks, n_jobs), block 256.
struct RowCopyJob {
  const uint4 *src;
  uint4 *dst;
  long long src_L, dst_L;
  int src_row0, src_rate;  // first source row: src_row0 + frames * src_rate
  int dst_row0, rows, planes;
};
__global__ void row_copy_kernel(const RowCopyJob *__restrict__ jobs, int frames) {
  pdl_launch_dependents();
  const RowCopyJob j = jobs[blockIdx.y];  // written at stream creation
  pdl_wait();
  const long long n = (long long)j.planes * j.rows;
  const long long s0 = j.src_row0 + (long long)frames * j.src_rate;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long pl = i / j.rows, r = i - pl * j.rows;
    j.dst[pl * j.dst_L + j.dst_row0 + r] = j.src[pl * j.src_L + s0 + r];
  }
}

// Overlap-crop stitch (minimaxmusic.cpp Architecture, "Decode and stitch"):
// window w keeps frames [w == 0 ? 0 : cl, w == n_win-1 ? Wf : Wf - cr); pieces are
// concatenated per side and clamped to [-1, 1].  grid (ceil(len/256), n_sides).
__global__ void stitch_kernel(const float *__restrict__ dec, int n_win, int n_sides, int Wf,
                              int cl, int cr, int hop, long long len, float *__restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int side = blockIdx.y;
  if (j >= len) return;
  const long long f = j / hop;
  const int ph = static_cast<int>(j - f * hop);
  long long start = 0;
  int w = 0, lo = 0;
  for (w = 0; w < n_win; ++w) {
    lo = (w == 0) ? 0 : cl;
    const int hi = (w == n_win - 1) ? Wf : Wf - cr;
    if (f < start + (hi - lo)) break;
    start += hi - lo;
  }
  const long long src = (long long)(lo + (f - start)) * hop + ph;
  const float v = dec[(size_t)(w * n_sides + side) * (size_t)Wf * hop + src];
  out[(size_t)side * len + j] = v < -1.f ? -1.f : (v > 1.f ? 1.f : v);
}

// Output head folded into the last conv2 (the conv kernel's HEAD form): audio[b][t] =
// tanh(bias + the partial sums that the 32-row slices reaching output t stored, over all
// channel chunks).  Slice s of chunk c holds slice_len = 32 + K - 1 sums, entry j for
// output row 32 s + j - (K - 1) + pad, so output t reads the slices s with
// 0 <= t - 32 s + K - 1 - pad < slice_len (at most two).  One thread per output sample:
// block 256, grid (ceil(L / 256), B).
__global__ void head_finish_kernel(const float *__restrict__ part, int L, int slices, int nch,
                                   int K, int pad, const float *__restrict__ bias,
                                   float *__restrict__ audio) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int b = blockIdx.y;
  if (t >= L) return;
  const int slice_len = 32 + K - 1;
  const int u = t + K - 1 - pad;  // = 32 s + j
  float acc = bias[0];
  for (int s = max(0, (u - slice_len + 32) / 32); s <= u / 32 && s < slices; ++s) {
    const int j = u - 32 * s;
    if (j < 0 || j >= slice_len) continue;
    const float *src = part + ((size_t)b * slices + s) * nch * slice_len + j;
    for (int c = 0; c < nch; ++c) acc += src[(size_t)c * slice_len];
  }
  audio[(size_t)b * L + t] = tanhf(acc);
}

// Split k: y = bias + the ksplit raw sums of part ([ks][B][Cp/4][part_L][4], added in ks
// order), then the conv kernel's epilogue: fp32 output (y, or Snake(y) with f32_snake), and the
// hi/lo split of Snake(y) (or y without alpha) into chunk-major planes; rows in
// [rows_valid, rows_pad) are written as zeros.  One thread per (b, 8 channels, row): block
// 256, grid (ceil(rows_pad / 256), Cp / 8, B).
__global__ void ksplit_reduce_kernel(const float *__restrict__ part, int ksplit, int B, int Cp,
                                     long long part_L, int rows_valid, int rows_pad,
                                     const float *__restrict__ bias, const float *__restrict__ alpha,
                                     const float *__restrict__ invb, int f32_snake,
                                     float *__restrict__ out_f32, long long f32_L,
                                     __nv_bfloat16 *__restrict__ out_hl, long long hl_L, int f16) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int g = blockIdx.y;  // 8-channel group
  const int b = blockIdx.z;
  if (t >= rows_pad) return;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int ks = 0; ks < ksplit; ++ks) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float4 x = reinterpret_cast<const float4 *>(
          part)[(((size_t)ks * B + b) * (Cp / 4) + 2 * g + h) * part_L + t];
      v[4 * h] += x.x, v[4 * h + 1] += x.y, v[4 * h + 2] += x.z, v[4 * h + 3] += x.w;
    }
  }
  float sn[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = 8 * g + i;
    v[i] += bias[c];
    sn[i] = alpha ? snake(v[i], alpha[c], invb[c]) : v[i];
    if (t >= rows_valid) v[i] = 0.f, sn[i] = 0.f;
  }
  if (out_f32) {
    const float *src = f32_snake ? sn : v;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      reinterpret_cast<float4 *>(out_f32)[((size_t)b * (Cp / 4) + 2 * g + h) * f32_L + t] =
          make_float4(src[4 * h], src[4 * h + 1], src[4 * h + 2], src[4 * h + 3]);
  }
  if (out_hl) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (f16)
        split_pair<true>(sn[2 * i], sn[2 * i + 1], hw[i], lw[i]);
      else
        split_pair<false>(sn[2 * i], sn[2 * i + 1], hw[i], lw[i]);
    }
    const size_t item = (size_t)b * (2 * Cp / 8);
    *reinterpret_cast<uint4 *>(out_hl + ((item + g) * hl_L + t) * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4 *>(out_hl + ((item + Cp / 8 + g) * hl_L + t) * 8) =
        make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

// The encoder's conv_in on Cin (few) audio channels: y[c][t] = b[c] + sum_ci sum_k
// w[c][ci][k] x[ci][t + k - pad], x zero outside [0, L), in fp32 on the CUDA cores (a 1-channel
// input would fill one sixteenth of a tensor-core operand).  Writes the fp32 residual stream
// y ([B][Cp/4][Lp][4]) and the hi/lo split of Snake(y) ([B][2 Cp/8][Lp][8], f16 parts when
// f16 != 0); channels past C read zero weights, rows L..Lp-1 are zeros.  A block takes 8
// channels (blockIdx.y) and kAudioRows x 256 rows: its weights (8 x Cin x K <= 8 x 4 x 15) are
// staged in shared memory once, and each thread takes every 256th row of the block's range, so
// every store is coalesced.  Grid (ceil(Lp / (256 kAudioRows)), Cp / 8, B), block 256.
constexpr int kAudioRows = 8;
constexpr int kAudioMaxW = 8 * 4 * 15;
__global__ void audio_conv_in_kernel(const float *__restrict__ x, int Cin, int L, long long Lp,
                                     int K, int pad, const float *__restrict__ w, int C,
                                     const float *__restrict__ bias, const float *__restrict__ alpha,
                                     const float *__restrict__ invb, int Cp,
                                     float *__restrict__ out_f32, __nv_bfloat16 *__restrict__ out_hl,
                                     int f16) {
  __shared__ float ws[kAudioMaxW];  // [i][ci][k] for the block's channels 8 g + i
  pdl_launch_dependents();
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int nw = 8 * Cin * K;
  for (int e = threadIdx.x; e < nw && e < kAudioMaxW; e += blockDim.x) {
    const int i = e / (Cin * K), r = e % (Cin * K);
    const int c = 8 * g + i;
    ws[e] = c < C ? w[(size_t)c * Cin * K + r] : 0.f;
  }
  float bb[8], a[8], ib[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = 8 * g + i;
    bb[i] = bias[c];
    a[i] = alpha ? alpha[c] : 0.f;
    ib[i] = alpha ? invb[c] : 0.f;
  }
  __syncthreads();
  pdl_wait();
  const size_t item = (size_t)b * (2 * Cp / 8);
  for (int j = 0; j < kAudioRows; ++j) {
    const long long t = ((long long)blockIdx.x * kAudioRows + j) * blockDim.x + threadIdx.x;
    if (t >= Lp) break;
    float v[8], sn[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = bb[i];
    if (t < L) {
      for (int ci = 0; ci < Cin; ++ci) {
        const float *xr = x + ((size_t)b * Cin + ci) * L;
        for (int k = 0; k < K; ++k) {
          const long long u = t + k - pad;
          const float xv = (u >= 0 && u < L) ? __ldg(xr + u) : 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = fmaf(ws[(i * Cin + ci) * K + k], xv, v[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sn[i] = alpha ? snake(v[i], a[i], ib[i]) : v[i];
      if (t >= L) v[i] = 0.f, sn[i] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
      reinterpret_cast<float4 *>(out_f32)[((size_t)b * (Cp / 4) + 2 * g + h) * Lp + t] =
          make_float4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]);
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (f16)
        split_pair<true>(sn[2 * i], sn[2 * i + 1], hw[i], lw[i]);
      else
        split_pair<false>(sn[2 * i], sn[2 * i + 1], hw[i], lw[i]);
    }
    *reinterpret_cast<uint4 *>(out_hl + ((item + g) * Lp + t) * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4 *>(out_hl + ((item + Cp / 8 + g) * Lp + t) * 8) =
        make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

__global__ void finite_check_kernel(const float *__restrict__ x, long long n, int *flag) {
  pdl_launch_dependents();
  pdl_wait();
  int bad = 0;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    bad |= !isfinite(x[i]);
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(flag, 1);
}

// fp32 chunk-major [B][Cp/4][Lp][4] (planes of Lp rows) -> channels-first [B][C][L] (first
// C channels).  One thread per (b, 4-channel chunk, t): block 256, grid (ceil(L/256), Cp/4, B).
__global__ void rows_to_cf_kernel(const float *__restrict__ src, int L, long long Lp, int Cp,
                                  int C, float *__restrict__ cf) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int j = blockIdx.y;
  const int b = blockIdx.z;
  if (t >= L) return;
  const float4 v = reinterpret_cast<const float4 *>(src)[((size_t)b * (Cp / 4) + j) * Lp + t];
  const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = 4 * j + u;
    if (c < C) cf[((size_t)b * C + c) * L + t] = e[u];
  }
}

// channels-first fp32 [B][C][L] -> chunk-major fp32 [B][Cp/4][Lp][4] (zeros past C and in
// rows L..Lp-1).  One thread per (b, 4-channel chunk, row): block 256, grid (ceil(Lp/256),
// Cp/4, B).
__global__ void cf_to_rows_kernel(const float *__restrict__ cf, int L, int Lp, int Cp, int C,
                                  float *__restrict__ dst) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int j = blockIdx.y;
  const int b = blockIdx.z;
  if (t >= Lp) return;
  float e[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = 4 * j + u;
    e[u] = (c < C && t < L) ? cf[((size_t)b * C + c) * L + t] : 0.f;
  }
  reinterpret_cast<float4 *>(dst)[((size_t)b * (Cp / 4) + j) * (size_t)Lp + t] =
      make_float4(e[0], e[1], e[2], e[3]);
}

}  // namespace voc
