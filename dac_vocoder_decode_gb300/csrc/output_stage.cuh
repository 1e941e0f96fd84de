// output_stage.cuh -- the step after the stitch (minimaxmusic.cpp Architecture,
// "Post-processing"): percentile peak normalisation and WAV encoding in device memory.
//
// Level: the ceil(q * n)-th smallest |x| over all samples, q = 1 - peak_clip / 1e6
// (peak_clip = 0: the peak).  Non-negative floats order like their bit patterns, so the
// level is found exactly by a three-pass radix select over the 32-bit patterns of |x|
// (bits 31..21, 20..10, 9..0): each pass histograms, in shared memory, the values whose
// higher bits match the prefix found so far, and a one-block pass picks the bucket that
// holds the wanted rank.  Gain = 1 / level (IEEE single; 1 when the level is 0, the largest
// finite float when the reciprocal of a subnormal level overflows).
// Samples: round-half-even(clamp(x * gain, -1, 1) * (2^(bits-1) - 1)), interleaved across
// channels, little endian, after a 44-byte RIFF header; 32-bit files hold the floats as
// they are (no normalisation).
#pragma once
#include <cstdint>

namespace voc {

struct SelectState {
  unsigned long long k;  // rank still to find inside the current prefix (1-based)
  uint32_t prefix;       // bits fixed so far
  uint32_t mask;         // which bits of `prefix` are fixed
  float level, gain;
};

__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

// Histogram of bits [shift, shift + width) of |x| over the values matching st->prefix.
template <int WIDTH>
__global__ void __launch_bounds__(256) select_hist_kernel(const float *__restrict__ x, long long n,
                                                          int shift, const SelectState *__restrict__ st,
                                                          unsigned int *__restrict__ hist) {
  __shared__ unsigned int h[1 << WIDTH];
  for (int i = threadIdx.x; i < (1 << WIDTH); i += blockDim.x) h[i] = 0;
  __syncthreads();
  const uint32_t mask = st->mask, prefix = st->prefix;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const uint32_t key = abs_bits(__ldg(x + i));
    if ((key & mask) == prefix) atomicAdd(&h[(key >> shift) & ((1u << WIDTH) - 1u)], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < (1 << WIDTH); i += blockDim.x)
    if (h[i]) atomicAdd(&hist[i], h[i]);
}

// One block of 256 threads: find the bucket of the remaining rank, extend the prefix, clear
// the histogram for the next pass; after the last pass store the level and the gain.
template <int WIDTH>
__global__ void __launch_bounds__(256) select_pick_kernel(SelectState *__restrict__ st,
                                                          unsigned int *__restrict__ hist, int shift,
                                                          int last) {
  constexpr int BINS = 1 << WIDTH;
  constexpr int PER = BINS / 256;
  __shared__ unsigned long long part[256];
  const int t = threadIdx.x;
  unsigned long long sum = 0;
  for (int i = 0; i < PER; ++i) sum += hist[t * PER + i];
  part[t] = sum;
  __syncthreads();
  if (t == 0) {
    unsigned long long k = st->k, before = 0;
    int seg = 0;
    while (seg < 255 && before + part[seg] < k) before += part[seg++];
    int bin = seg * PER;
    while (bin < seg * PER + PER - 1 && before + hist[bin] < k) before += hist[bin++];
    st->k = k - before;
    st->prefix |= static_cast<uint32_t>(bin) << shift;
    st->mask |= ((1u << WIDTH) - 1u) << shift;
    if (last) {
      const float level = __uint_as_float(st->prefix);
      st->level = level;
      // IEEE division; a subnormal level whose reciprocal overflows takes the largest
      // finite gain, so that zeros stay zero
      st->gain = level > 0.f ? fminf(1.0f / level, 3.402823466e38f) : 1.0f;
    }
  }
  __syncthreads();
  for (int i = t; i < BINS; i += 256) hist[i] = 0;
}

// The 44-byte RIFF/WAVE header: eleven 32-bit little-endian words prepared on the host.
struct WavHeader {
  uint32_t w[11];
};
__global__ void wav_header_kernel(WavHeader h, uint8_t *__restrict__ out) {
  const int i = threadIdx.x;
  if (i < 11) reinterpret_cast<uint32_t *>(out)[i] = h.w[i];
}

// planar [n_ch][len] -> interleaved samples after the header; one thread per sample.
__global__ void wav_encode_kernel(const float *__restrict__ planar, int n_ch, long long len,
                                  int bytes_per_sample, const SelectState *__restrict__ st,
                                  uint8_t *__restrict__ data) {
  const long long n = (long long)n_ch * len;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // interleaved index
  if (i >= n) return;
  const long long t = i / n_ch;
  const int c = static_cast<int>(i - t * n_ch);
  const float v = __ldg(planar + (long long)c * len + t);
  if (bytes_per_sample == 4) {
    reinterpret_cast<float *>(data)[i] = v;
    return;
  }
  const float full = bytes_per_sample == 2 ? 32767.0f : 8388607.0f;
  const float y = fminf(fmaxf(v * st->gain, -1.0f), 1.0f);
  const int q = __float2int_rn(y * full);  // round half to even
  if (bytes_per_sample == 2) {
    reinterpret_cast<int16_t *>(data)[i] = static_cast<int16_t>(q);
  } else {
    uint8_t *p = data + i * 3;
    p[0] = static_cast<uint8_t>(q & 0xFF);
    p[1] = static_cast<uint8_t>((q >> 8) & 0xFF);
    p[2] = static_cast<uint8_t>((q >> 16) & 0xFF);
  }
}

}  // namespace voc
