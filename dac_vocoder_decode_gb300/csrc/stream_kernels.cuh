// stream_kernels.cuh -- the bandwidth-bound kernels around the tensor-core convs:
//   prep_hl_kernel      channels-first fp32 -> channels-last bf16 hi/lo rows (+ optional Snake)
//   out_head_kernel     Snake'd fp32 rows -> k-tap conv to one channel (+bias) -> tanh
//   stitch_kernel       overlap-crop stitch + clamp of windowed decodes
//   finite_check_kernel flags a NaN / Inf in a buffer
//   rows_to_cf_kernel   channels-last fp32 rows -> channels-first fp32 (single-layer ops)
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "snake.cuh"

namespace voc {

// x [B][C][T] fp32 -> hl [B][T][2*Cp] bf16 (per row: Cp hi values, then Cp lo values);
// channels C..Cp-1 are written as zeros.  alpha == nullptr: no Snake.
// Block (32, 8), grid (ceil(T/32), ceil(Cp/32), B).
__global__ void prep_hl_kernel(const float *__restrict__ x, int C, int T, int Cp,
                               const float *__restrict__ alpha, const float *__restrict__ invb,
                               __nv_bfloat16 *__restrict__ hl) {
  __shared__ float tile[32][33];
  const int b = blockIdx.z;
  const int t0 = blockIdx.x * 32;
  const int c0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, t = t0 + threadIdx.x;
    float v = 0.f;
    if (c < C && t < T) {
      v = x[((size_t)b * C + c) * T + t];
      if (alpha) v = snake(v, alpha[c], invb[c]);
    }
    tile[i][threadIdx.x] = v;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int t = t0 + i, c = c0 + threadIdx.x;
    if (t < T && c < Cp) {
      const float v = tile[threadIdx.x][i];
      const __nv_bfloat16 h = __float2bfloat16_rn(v);
      const __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
      __nv_bfloat16 *row = hl + ((size_t)b * T + t) * (size_t)(2 * Cp);
      row[c] = h;
      row[Cp + c] = l;
    }
  }
}

// audio[b][t] = tanh(bias + sum_k sum_c w[c][k] * y[b][t + k - pad_left][c]), y zero outside
// [0, L).  y rows are Cp floats (already Snake'd), w [Cp][K] (zero past the real channels).
// One thread per output sample, TILE samples per block, rows staged in shared memory with a
// padded stride (Cp + 4 floats) so that float4 reads of consecutive rows hit distinct banks.
template <int TILE>
__global__ void __launch_bounds__(TILE) out_head_kernel(const float *__restrict__ y, int L, int Cp,
                                                        int K, int pad_left,
                                                        const float *__restrict__ w,
                                                        const float *__restrict__ bias,
                                                        float *__restrict__ audio) {
  extern __shared__ float4 sm4[];
  float *sm = reinterpret_cast<float *>(sm4);
  const int b = blockIdx.y;
  const int t0 = blockIdx.x * TILE;
  const int rows = TILE + K - 1;
  const int ld = Cp + 4;
  float *xs = sm;
  float *ws = sm + (size_t)rows * ld;
  for (int i = threadIdx.x; i < Cp * K; i += TILE) ws[i] = w[i];
  const int nvec = Cp / 4;
  for (int i = threadIdx.x; i < rows * nvec; i += TILE) {
    const int r = i / nvec, c4 = i - r * nvec;
    const int t = t0 - pad_left + r;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t >= 0 && t < L)
      v = __ldg(reinterpret_cast<const float4 *>(y + ((size_t)b * L + t) * Cp) + c4);
    *reinterpret_cast<float4 *>(xs + (size_t)r * ld + 4 * c4) = v;
  }
  __syncthreads();
  const int t = t0 + threadIdx.x;
  if (t >= L) return;
  float acc = 0.f;
  for (int k = 0; k < K; ++k) {
    const float *xr = xs + (size_t)(threadIdx.x + k) * ld;
    for (int c4 = 0; c4 < nvec; ++c4) {
      const float4 xv = *reinterpret_cast<const float4 *>(xr + 4 * c4);
      acc = fmaf(ws[(4 * c4 + 0) * K + k], xv.x, acc);
      acc = fmaf(ws[(4 * c4 + 1) * K + k], xv.y, acc);
      acc = fmaf(ws[(4 * c4 + 2) * K + k], xv.z, acc);
      acc = fmaf(ws[(4 * c4 + 3) * K + k], xv.w, acc);
    }
  }
  audio[(size_t)b * L + t] = tanhf(bias[0] + acc);
}

// Overlap-crop stitch (minimaxmusic.cpp Architecture, "Decode and stitch"):
// window w keeps frames [w == 0 ? 0 : cl, w == n_win-1 ? Wf : Wf - cr); pieces are
// concatenated per side and clamped to [-1, 1].  grid (ceil(len/256), n_sides).
__global__ void stitch_kernel(const float *__restrict__ dec, int n_win, int n_sides, int Wf,
                              int cl, int cr, int hop, long long len, float *__restrict__ out) {
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

__global__ void finite_check_kernel(const float *__restrict__ x, long long n, int *flag) {
  int bad = 0;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    bad |= !isfinite(x[i]);
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(flag, 1);
}

// rows [B][L][ld] fp32 (first C columns used) -> cf [B][C][L].  Block (32, 8),
// grid (ceil(L/32), ceil(C/32), B).
__global__ void rows_to_cf_kernel(const float *__restrict__ rows, int L, int ld, int C,
                                  float *__restrict__ cf) {
  __shared__ float tile[32][33];
  const int b = blockIdx.z;
  const int t0 = blockIdx.x * 32;
  const int c0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int t = t0 + i, c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (t < L && c < C) ? rows[((size_t)b * L + t) * ld + c] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, t = t0 + threadIdx.x;
    if (c < C && t < L) cf[((size_t)b * C + c) * L + t] = tile[threadIdx.x][i];
  }
}

}  // namespace voc
