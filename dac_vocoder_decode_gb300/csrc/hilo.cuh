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
  if constexpr (F16) {
    const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
    const __half l0 = __float2half_rn(x0 - __half2float(h0));
    const __half l1 = __float2half_rn(x1 - __half2float(h1));
    h = static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
    l = static_cast<uint32_t>(__half_as_ushort(l0)) | (static_cast<uint32_t>(__half_as_ushort(l1)) << 16);
  } else {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
    const __nv_bfloat16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
    const __nv_bfloat16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
    h = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
        (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
    l = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
        (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
  }
}

}  // namespace voc
