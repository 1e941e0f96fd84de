// snake.cuh -- Snake activation, y = x + sin^2(a x) / (a + 1e-9), with the
// per-channel a used as stored (minimaxmusic.cpp Architecture, "Flow VAE";
// MiniMax-Music-3 -> CMF README, "What the conversion had to get right").
// inv_b = 1/(a + 1e-9) is formed on the host.
#pragma once

namespace voc {

// sin^2 has period pi, so with x = k*pi + r and |r| <= pi/2, sin^2(x) = sin^2(r).
// k*pi is removed with a two-constant (Cody & Waite) reduction: kPiHi = 201/64
// carries the leading 8 bits of pi, so k*kPiHi is exact for |k| < 2^16, and kPiLo
// holds pi - 201/64.  The hardware approximation __sinf is then evaluated on
// [-pi/2, pi/2] (within [-pi, pi], where its absolute error is about 2^-21).
// Arguments beyond 8192 in magnitude go to sinf.
constexpr float kInvPi = 0.318309886183790671538f;
constexpr float kPiHi = 3.140625f;
constexpr float kPiLo = 9.67653589793238462643e-4f;

__device__ __noinline__ float sin2_wide(float x) {
  const float s = sinf(x);
  return s * s;
}

// Reduction and __sinf for |x| <= 8192 (no branch).
__device__ __forceinline__ float sin2_fast(float x) {
  const float k = rintf(x * kInvPi);
  float r = fmaf(-k, kPiHi, x);
  r = fmaf(-k, kPiLo, r);
  const float s = __sinf(r);
  return s * s;
}

__device__ __forceinline__ float sin2(float x) {
  if (fabsf(x) > 8192.f) return sin2_wide(x);
  return sin2_fast(x);
}

__device__ __forceinline__ float snake(float v, float a, float inv_b) {
  return fmaf(inv_b, sin2(a * v), v);
}

// Snake of N values.  The common path has no branch per value, so the compiler can
// interleave the N independent computations; the values with |a v| > 8192 (if any) are
// redone with sinf afterwards, under one branch per call.
template <int N>
__device__ __forceinline__ void snake_n(const float (&v)[N], const float (&a)[N],
                                        const float (&inv_b)[N], float (&out)[N]) {
  float amax = 0.f;  // the largest |a v| of the N (one max per value instead of a compare and an or)
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float ax = a[i] * v[i];
    amax = fmaxf(amax, fabsf(ax));
    out[i] = fmaf(inv_b[i], sin2_fast(ax), v[i]);
  }
  if (!(amax <= 8192.f)) {  // unrolled too: a run-time index would put the arrays in local memory
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float ax = a[i] * v[i];
      if (fabsf(ax) > 8192.f) out[i] = fmaf(inv_b[i], sin2_wide(ax), v[i]);
    }
  }
}

}  // namespace voc
