// hilo.cuh -- the hi/lo split of fp32 activations into two 16-bit parts, the form in which
// every tensor-core layer reads its input: hi = r(x), lo = r(x - hi), with r the rounding to
// the MMA operand type, to nearest with ties to even.  bf16 parts (the bf16x3 precision) keep
// about 16 significant bits of x; f16 parts (the F16-weight precision) about 22, within the
// f16 range (|x| < 65504).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace voc {

template <bool F16>
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t &h, uint32_t &l) {
  // one packed conversion per part (cvt.rn.{f16,bf16}x2.f32: x0 in the low half), the same
  // round-to-nearest-even values as converting each element on its own
  if constexpr (F16) {
    const __half2 hh = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(hh);
    const __half2 ll = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    h = *reinterpret_cast<const uint32_t *>(&hh);
    l = *reinterpret_cast<const uint32_t *>(&ll);
  } else {
    const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(hh);
    const __nv_bfloat162 ll = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    h = *reinterpret_cast<const uint32_t *>(&hh);
    l = *reinterpret_cast<const uint32_t *>(&ll);
  }
}

}  // namespace voc
