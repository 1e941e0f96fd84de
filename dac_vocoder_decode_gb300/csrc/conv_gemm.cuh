// conv_gemm.cuh -- tcgen05 implicit-GEMM convolution for every tensor-core
// layer of the decoder: conv_in (k7), the polyphase ConvTranspose1d, the k7
// dilated conv1 and the k1 conv2 of each residual unit.
//
// GEMM view (time on M, output columns on N):
//   D[t][n] = sum_tap sum_ci A[t + off(tap, n)][ci] * Wt[tap][n][ci]
// * regular conv: off(tap) = tap*dil - pad_left, n = output channel;
// * ConvTranspose1d of stride s, K = 2s, left crop p (polyphase form): the
//   output sample t*s + r of channel co is column n = r*C_out + co and
//     out[t*s + r][co] = sum_ci W[ci][co][k0] x[t+q][ci] + W[ci][co][k0+s] x[t+q-1][ci]
//   with q = floor((r+p)/s), k0 = (r+p) mod s, i.e. two taps at row offsets q and
//   q-1.  The overlap-add of col2im happens inside the MMA accumulation and no
//   column matrix is ever written.
//
// Activation layout in global memory ("chunk-major"): a bf16 hi/lo tensor of C
// channels and length L is [B][2C/8][L][8] -- 8-channel chunks of the hi parts,
// then of the lo parts, each chunk a contiguous run of L 16-byte rows; an fp32
// tensor is [B][C/4][L][4].  hi = bf16(x), lo = bf16(x - hi).
//
// Operands: each K step issues three MMAs, hi*hi + hi*lo + lo*hi, into one fp32
// TMEM accumulator; weights are pre-split into hi/lo on the host.
//
// Shared-memory layout of an A stage (no swizzle, K-major canonical layout): for
// each 8-channel chunk, `rows` consecutive time rows of 16 bytes -- exactly the
// chunk-major global layout, so one TMA box per k-block fetches contiguous runs.
// The row offset of a tap is a 16-byte shift of the descriptor start address, so
// all taps reuse one staged halo tile (128 + span rows, zero fill outside [0, L)).
//
// Roles: warp 0 lane 0 issues the A copies (one 5-D TMA box per k-block: the hi and
// lo planes of its channel chunks), warp 1 runs the MMA loop (convergently; an elected
// lane issues), warps 2..13 run the epilogue in three groups of four warps, one warp per
// TMEM lane quadrant, group g taking column chunks g, g+3, ... (TMEM -> registers ->
// bias, residual, Snake of the next layer, hi/lo split -> global; with the chunk-major
// layout the 32 lanes of a warp store 32 consecutive rows of one chunk: 512 contiguous
// bytes), warp 14 prefetches the residual input of the three groups by TMA, warp 15
// issues the weight copies (16 warps: up to 128 registers per thread).
// The grid is persistent; 2 to 4 TMEM accumulators let the epilogue of one tile
// overlap the mainloop of the next.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include "hilo.cuh"
#include "ptx.cuh"
#include "snake.cuh"

namespace voc {

constexpr int kTileM = 128;
constexpr int kEpiGroups = 3;                           // epilogue groups of 4 warps (one per
                                                        // TMEM lane quadrant)
constexpr int kEpiWarps = 4 * kEpiGroups;               // warps 2..13
constexpr int kSkipWarp = 2 + kEpiWarps;                // residual prefetch for every group
constexpr int kBWarp = kSkipWarp + 1;                   // weight copies
constexpr int kBWarps = 1;
// 16 warps: four per SM sub-partition, so each thread may hold up to 128 registers
constexpr int kGemmThreads = 32 * (kBWarp + kBWarps);   // 512
constexpr int kMaxAcc = 4;
// Bound on the waits of a kernel that has given up (ConvGemmArgs::timeout ran out, or another
// role raised the abort flag) for its own copies and MMAs in flight: those were issued and
// complete in microseconds, so the bound is long and independent of the pipeline waits' budget
// -- a CTA must not exit (and free its shared memory and TMEM) while they can still land.
constexpr long long kDrainBudget = 4000000000LL;

// bytes of one residual slot (128 rows x cw fp32 columns, as cw/4 chunks of 128 x 16 B)
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

// Weight forms of conv_gemm_kernel (the library's VOC_PREC_* values).
constexpr int kPrecBf16x3 = 0, kPrecF16w = 1, kPrecBf16w = 2;

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
  const float *skip;       // fp32 residual (chunk-major, Cp_out channels) or null: read via TMA
  float *out_f32;          // fp32 output, chunk-major [B][Cp_out/4][f32_L][4], or null
  __nv_bfloat16 *out_hl;   // hi/lo output, chunk-major [B][2*Cp_out/8][hl_L][8], or null
  int Cp_out, s_rows;      // output channels (padded), output rows per D row
  int phase_group;         // ConvT, columns in 8-channel blocks of the G phases of a group
                           // (n = q G Cp + (co / 8) 8 G + r 8 + co % 8): G even, stored by
                           // 16-column chunks (phase pairs); G odd, by whole blocks with lane
                           // pairs (see convT_block_odd).  0: phase-major columns
                           // (n = phase * Cp_out + channel).
  int b2;                  // 1 (the kernel's B2 form): each weight chunk holds its hi rows then its lo rows, and a K
                           // step is two MMAs: A_hi x [W_hi | W_lo] into 2 N_tile accumulator
                           // columns, then A_lo x W_hi into the first N_tile; the epilogue adds
                           // the two column halves.  0: three MMAs of N_tile columns.
  // Row placement (stateful streaming keeps each layer's left context in front of its new
  // rows): A row r of D row t is input row in_row0 + t + offset; output row t*s_rows + ph
  // goes to row f32_row0 + ... of planes of f32_L rows (hl_row0 / hl_L for the hi/lo
  // output).  A plain decode has 0 offsets and planes of L_in * s_rows rows rounded up to a
  // multiple of 8.
  int in_row0, f32_row0, f32_L, hl_row0, hl_L;
  // Output rows (t * s_rows + ph) below rows_valid are results; rows in [rows_valid,
  // rows_pad) are written as zeros (the padding rows up to the next multiple of 8 that
  // the next layer's 8-row TMA groups read); rows from rows_pad on are not written.
  int rows_valid, rows_pad;
  int flags;
  int b_resident;          // 1: the nb = taps * nkb weight slots hold this CTA's whole column
                           // tile, loaded once (every CTA keeps one column tile)
  long long timeout;       // cycles a wait may take before the kernel gives up
  int *err;                // device error word
  // extents used by the self-checking build (VOC_CHECKS)
  long long f32_elems, hl_elems, w_bytes;
  int smem_bytes, L_a, chunks_a, chunks_s;
  int *dbg;                // [4]: first failed check code and three values
  // Encoder forms (kernels with ENC = true; ignored by the others):
  int split_s;             // S > 1: the hi/lo output is phase-split for a strided conv of
                           // stride S (see phase_plane)
  int kb_split;            // k-blocks kb < kb_split use taps [tap_lo0, tap_hi0), the others
  int tap_lo0, tap_hi0, tap_lo1, tap_hi1;  // [tap_lo1, tap_hi1) (a strided conv's two
                                           // phase groups each read two of its three taps)
  int ksplit;              // >= 1: the k-blocks are split into ksplit ranges of kb_per_split,
  int kb_per_split;        // one job per (range, tile); with ksplit > 1 the epilogue stores the
  float *part;             // raw sums to part[((ks * B + b) * Cp_out/4 + chunk4) * part_L + row]
  long long part_L;        // (4 floats each) and ksplit_reduce_kernel finishes the layer
  // Output head folded into this layer's epilogue (kernels with HEAD = true): the layer
  // writes no activations; each warp reduces its 32 rows x 16 channels of Snake_out(y) to
  // the 32 + head_K - 1 partial sums of the head's outputs those rows reach
  // (head_slice_len), stored at head_part[((b * head_slices + row / 32) * (Cp_out / 16)
  // + chunk) * head_slice_len + j] for output row 32 (row / 32) + j - (head_K - 1) + head_pad.
  const float *head_w;     // [head_K][Cp_out] head weights (zero past the real channels)
  float *head_part;
  int head_K, head_pad, head_slices, head_slice_len;
  // Job order: 0 -- row tiles outer, column tiles inner (each wave reads every column tile's
  // weights); band > 0 -- the row tiles in bands of `band`, and inside a band the column tiles
  // outer, so that a wave reads a part of the weights (layers whose weights outweigh L2's share).
  // Not with resident weights (each CTA keeps one column tile).
  int band;
};

// Column tile nt, row tile mt and item b of tile job jj (see ConvGemmArgs::band).
__device__ __forceinline__ void job_tile(const ConvGemmArgs &p, int jj, int &nt, int &mt, int &b) {
  if (p.band > 0) {
    const int rows = p.B * p.m_tiles;
    const int per_band = p.band * p.n_tiles;
    const int bi = jj / per_band;
    const int r0 = bi * p.band;
    const int nr = min(p.band, rows - r0);  // row tiles of this band
    const int w = jj - bi * per_band;
    nt = w / nr;
    const int rr = r0 + (w - nt * nr);
    mt = rr % p.m_tiles;
    b = rr / p.m_tiles;
  } else {
    nt = jj % p.n_tiles;
    const int rest = jj / p.n_tiles;
    mt = rest % p.m_tiles;
    b = rest / p.m_tiles;
  }
}

// Taps of the head fold (the conv kernel's HEAD form): the decoder's 7-tap head; a shorter head
// is folded with its weights zero-padded to 7 taps (head_K = 7, the same head_pad).
constexpr int kHeadFoldMaxK = 7;

// Plane (8-channel group) of channel chunk `ch`, phase `ph` in the phase-split layout of a
// strided conv's input with stride ss over cpc chunks: the phases r < R0 = ceil(ss/2) come
// first (plane ch * R0 + r), then the phases r >= R0 (plane R0 cpc + ch (ss - R0) + r - R0).
// Phases r < R0 read input row shifts {0, +1} of the conv's three taps, the others {-1, 0},
// so each group's k-blocks skip one tap.
__host__ __device__ __forceinline__ size_t phase_plane(size_t ch, size_t ph, size_t ss,
                                                       size_t cpc) {
  const size_t r0 = (ss + 1) / 2;
  return ph < r0 ? ch * r0 + ph : r0 * cpc + ch * (ss - r0) + (ph - r0);
}

#ifdef VOC_CHECKS
// Record the first failed check (code, three values), raise the abort flag; the caller skips
// the access.
__device__ __forceinline__ void check_fail(const ConvGemmArgs &p, volatile int *abort_flag,
                                           int code, long long a, long long b, long long c) {
  if (atomicCAS(p.dbg, 0, code) == 0) {
    p.dbg[1] = static_cast<int>(a);
    p.dbg[2] = static_cast<int>(b);
    p.dbg[3] = static_cast<int>(c);
  }
  atomicOr(p.err, 0x100);
  *abort_flag = 1;
}
#define VOC_CHECK(cond, code, a, b, c)                                   \
  if (!(cond)) {                                                         \
    check_fail(p, abort_flag, code, (long long)(a), (long long)(b), (long long)(c)); \
    return false;                                                        \
  }
#else
#define VOC_CHECK(cond, code, a, b, c)
#endif

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// floor(x / 8) for any sign (the row groups of the tensor maps; a negative group is
// out of range and reads as zeros)
__device__ __forceinline__ int floor_div8(int x) { return x >= 0 ? x / 8 : -((7 - x) / 8); }

template <int N>
__device__ __forceinline__ void ldg_vec(const float *src, float (&v)[N]) {
  const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
  for (int j = 0; j < N / 4; ++j) {
    const float4 a = __ldg(s4 + j);
    v[4 * j] = a.x, v[4 * j + 1] = a.y, v[4 * j + 2] = a.z, v[4 * j + 3] = a.w;
  }
}

// ConvT outputs with phase-pair columns: the 16 columns at n0 are 8 channels at two
// consecutive output rows (phases r, r+1 of input row t), written as 32-byte stores: fp32
// two planes of 4 channels, hi and lo one plane of 8 channels each.  The rows start at an
// even row (s even, r even), so every store is 32-byte aligned.
template <int CW, bool F16>
__device__ __forceinline__ bool store_phase_pair(const ConvGemmArgs &p, volatile int *abort_flag,
                                                 int b, int t, int n0, float (&v)[CW],
                                                 float (&sn)[CW]) {
  static_assert(CW == 16, "two phases of 8 channels");
  const int G = p.phase_group;
  const int gw = G * p.Cp_out;  // columns of one phase group
  const int q = n0 / gw;
  const int nn = n0 - q * gw;
  const int cg = nn / (8 * G);            // 8-channel block
  const int rl = (nn - cg * 8 * G) / 8;   // first phase within the group (even)
  const long long out_row = (long long)t * p.s_rows + q * G + rl;  // rows out_row, out_row + 1
  if (out_row >= p.rows_pad) return true;
  if (out_row >= p.rows_valid) {  // padding rows (both: rows_pad and out_row are even)
#pragma unroll
    for (int i = 0; i < CW; ++i) v[i] = 0.f, sn[i] = 0.f;
  }
  if (p.out_f32) {
    const size_t L_out = static_cast<size_t>(p.f32_L);
    const size_t row = static_cast<size_t>(out_row) + p.f32_row0;
    const float *src = (p.flags & EPI_F32_SNAKE) ? sn : v;
    VOC_CHECK((((long long)b * (p.Cp_out / 4) + 2 * cg + 1) * (long long)L_out + row + 1) * 4 + 4 <= p.f32_elems,
              16, b, cg, (int)row);
    float *base = p.out_f32 + ((size_t)b * (p.Cp_out / 4) + 2 * cg) * L_out * 4 + row * 4;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t w[8] = {__float_as_uint(src[4 * j]), __float_as_uint(src[4 * j + 1]),
                             __float_as_uint(src[4 * j + 2]), __float_as_uint(src[4 * j + 3]),
                             __float_as_uint(src[8 + 4 * j]), __float_as_uint(src[8 + 4 * j + 1]),
                             __float_as_uint(src[8 + 4 * j + 2]), __float_as_uint(src[8 + 4 * j + 3])};
      st_global_v8(base + (size_t)j * L_out * 4, w);
    }
  }
  if (p.out_hl) {
    uint32_t hw[8], lw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) split_pair<F16>(sn[2 * i], sn[2 * i + 1], hw[i], lw[i]);
    const size_t L_out = static_cast<size_t>(p.hl_L);
    const size_t row = static_cast<size_t>(out_row) + p.hl_row0;
    const size_t item = (size_t)b * (2 * p.Cp_out / 8);
    VOC_CHECK((((long long)item + p.Cp_out / 8 + cg) * (long long)L_out + row + 1) * 8 + 8 <= p.hl_elems,
              17, b, cg, (int)row);
    st_global_v8(p.out_hl + ((item + cg) * L_out + row) * 8, hw);
    st_global_v8(p.out_hl + ((item + p.Cp_out / 8 + cg) * L_out + row) * 8, lw);
  }
  return true;
}

// ConvT with an odd number G of phases per group (causal s = 3, 5): one 8-channel block of the
// G phases (8 G columns from n0, TMEM columns from taddr) for this warp's 32 rows.  Input row
// t owns output rows t G .. t G + G - 1; a lane pair (t even, t + 1) owns 2G rows starting at
// the even row t G, which split into G aligned row pairs: the even lane stores its phases
// (0, 1), (2, 3), ... and (G - 1, the odd lane's phase 0), the odd lane its phases (1, 2),
// (3, 4), ...  Each pair goes out as 32-byte stores (16-byte stores of the first row when the
// second is past the rows to write).  Two passes (fp32 output, then hi/lo output) keep at most
// three phases of 8 values live; phases are re-read from TMEM in each pass.
template <bool F16>
__device__ __forceinline__ bool convT_block_odd(const ConvGemmArgs &p, volatile int *abort_flag,
                                                int b, int t, int n0, uint32_t taddr, int lane) {
  const int G = p.phase_group;
  const bool odd_lane = (lane & 1) != 0;
  const int cg = n0 / (8 * G);               // causal: one phase group
  const long long row0 = (long long)t * p.s_rows;  // this lane's first output row
  const bool f_snake = (p.flags & EPI_F32_SNAKE) != 0;
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 0 ? !p.out_f32 : !p.out_hl) continue;
    const bool snake_it = (pass == 1 || f_snake) && p.alpha;  // hi/lo always carry the Snake
    float bb[8], a[8], ib[8];
    ldg_vec(p.bias + n0, bb);  // the same for every phase of the block
    if (snake_it) {
      ldg_vec(p.alpha + n0, a);
      ldg_vec(p.invb + n0, ib);
    }
    // this lane's value of phase r (8 channels)
    auto value = [&](int r, float (&out)[8]) {
      uint32_t q[8];
      tmem_ld8_issue(taddr + static_cast<uint32_t>(8 * r), q);
      tmem_ld8_wait(q);
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(q[i]) + bb[i];
      if (snake_it) {
        snake_n<8>(v, a, ib, out);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = v[i];
      }
    };
    float prev[8];
    value(0, prev);
    for (int k = 0; 2 * k < G; ++k) {
      float p1[8], p2[8];
      if (2 * k + 1 < G) {
        value(2 * k + 1, p1);
      } else {  // the even lane's last pair ends with the odd lane's phase 0
        float z[8];
        value(0, z);
#pragma unroll
        for (int i = 0; i < 8; ++i) p1[i] = __shfl_down_sync(0xffffffffu, z[i], 1);
      }
      const bool have2 = 2 * k + 2 < G;
      if (have2) {
        value(2 * k + 2, p2);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) p2[i] = 0.f;
      }
      // even lane: rows (2k, 2k+1) = phases (2k, 2k+1); odd lane: phases (2k+1, 2k+2)
      const long long R = row0 + 2 * k + (odd_lane ? 1 : 0);
      const bool active = !odd_lane || have2;
      if (active && R < p.rows_pad) {
        const bool two = R + 1 < p.rows_pad;
        const bool z0 = R >= p.rows_valid, z1 = R + 1 >= p.rows_valid;  // padding rows: zeros
        float A[8], B[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          A[i] = z0 ? 0.f : (odd_lane ? p1[i] : prev[i]);
          B[i] = z1 ? 0.f : (odd_lane ? p2[i] : p1[i]);
        }
        if (pass == 0) {
          const size_t L_out = static_cast<size_t>(p.f32_L);
          const size_t row = static_cast<size_t>(R) + p.f32_row0;
          VOC_CHECK((((long long)b * (p.Cp_out / 4) + 2 * cg + 1) * (long long)L_out + row + 1) * 4 + 4 <=
                        p.f32_elems, 18, b, cg, (int)row);
          float *base = p.out_f32 + ((size_t)b * (p.Cp_out / 4) + 2 * cg) * L_out * 4 + row * 4;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float *q = base + (size_t)j * L_out * 4;
            if (two) {
              const uint32_t w[8] = {__float_as_uint(A[4 * j]), __float_as_uint(A[4 * j + 1]),
                                     __float_as_uint(A[4 * j + 2]), __float_as_uint(A[4 * j + 3]),
                                     __float_as_uint(B[4 * j]), __float_as_uint(B[4 * j + 1]),
                                     __float_as_uint(B[4 * j + 2]), __float_as_uint(B[4 * j + 3])};
              st_global_v8(q, w);
            } else {
              *reinterpret_cast<float4 *>(q) = make_float4(A[4 * j], A[4 * j + 1], A[4 * j + 2], A[4 * j + 3]);
            }
          }
        } else {
          uint32_t hw[8], lw[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float x0 = i < 4 ? A[2 * i] : B[2 * i - 8];
            const float x1 = i < 4 ? A[2 * i + 1] : B[2 * i - 7];
            split_pair<F16>(x0, x1, hw[i], lw[i]);
          }
          const size_t L_out = static_cast<size_t>(p.hl_L);
          const size_t row = static_cast<size_t>(R) + p.hl_row0;
          const size_t item = (size_t)b * (2 * p.Cp_out / 8);
          VOC_CHECK((((long long)item + p.Cp_out / 8 + cg) * (long long)L_out + row + 1) * 8 + 8 <=
                        p.hl_elems, 19, b, cg, (int)row);
          __nv_bfloat16 *hq = p.out_hl + ((item + cg) * L_out + row) * 8;
          __nv_bfloat16 *lq = p.out_hl + ((item + p.Cp_out / 8 + cg) * L_out + row) * 8;
          if (two) {
            st_global_v8(hq, hw);
            st_global_v8(lq, lw);
          } else {
            *reinterpret_cast<uint4 *>(hq) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(lq) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) prev[i] = p2[i];
    }
  }
  return true;
}

// Epilogue of one warp for 32 rows (its TMEM lane quadrant) x CW columns
// n0..n0+CW-1, which lie in one ConvT phase because CW divides C_out.
// HEAD: instead of storing, hp[k] = sum over the chunk's channels c of head_w[k][c] *
// Snake_out(y)[c] for this lane's row (zero for padding rows; the caller reduces and stores).
template <int CW, bool B2 = false, bool F16 = false, bool ENC = false, bool HEAD = false>
__device__ __forceinline__ bool epilogue_chunk(const ConvGemmArgs &p, uint32_t sslot,
                                               uint32_t sfull, uint32_t sempty, uint32_t sparity,
                                               volatile int *abort_flag, int row_in_tile,
                                               int b, int t, int n0, uint32_t taddr,
                                               uint32_t smem_lo, uint32_t smem_hi,
                                               float *hp = nullptr) {
  VOC_CHECK((taddr & 0xFFFFu) + CW + (p.b2 ? p.N_tile : 0) <= (uint32_t)(p.n_acc * p.acc_cols), 11,
            taddr & 0xFFFF, CW, p.b2);
  VOC_CHECK(n0 + CW <= p.N_total, 12, n0, p.N_total, 0);
  static_assert(CW == 16, "16-column epilogue chunks");
  float v[CW];
  // Issue the independent loads first: the bias (L1-resident), the TMEM read and, once
  // its slot has landed, the residual tile; then wait for the TMEM data.
  float bb[CW];
  ldg_vec(p.bias + n0, bb);
  uint32_t r[CW], r2[CW];
  tmem_ld_issue<CW>(taddr, r);
  if constexpr (B2) tmem_ld_issue<CW>(taddr + static_cast<uint32_t>(p.N_tile), r2);
  if (p.skip) {
    VOC_CHECK(sslot >= smem_lo && sslot + skip_slot_bytes(CW) <= smem_hi, 13, sslot, smem_lo, smem_hi);
    const bool landed = mbar_wait(sfull, sparity, p.timeout, abort_flag);
    uint4 sk[CW / 4];
    if (landed) {
#pragma unroll
      for (int j = 0; j < CW / 4; ++j)
        sk[j] = lds128(sslot + static_cast<uint32_t>((j * kTileM + row_in_tile) * 16));
      mbar_arrive(sempty);
    }
    tmem_ld_wait<CW>(r);  // the TMEM reads complete before any return
    if constexpr (B2) {
      tmem_ld16_after_wait(r2);
#pragma unroll
      for (int i = 0; i < CW; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
    }
    if (!landed) return false;
#pragma unroll
    for (int j = 0; j < CW / 4; ++j) {  // (acc + bias) + skip
      v[4 * j] = (__uint_as_float(r[4 * j]) + bb[4 * j]) + __uint_as_float(sk[j].x);
      v[4 * j + 1] = (__uint_as_float(r[4 * j + 1]) + bb[4 * j + 1]) + __uint_as_float(sk[j].y);
      v[4 * j + 2] = (__uint_as_float(r[4 * j + 2]) + bb[4 * j + 2]) + __uint_as_float(sk[j].z);
      v[4 * j + 3] = (__uint_as_float(r[4 * j + 3]) + bb[4 * j + 3]) + __uint_as_float(sk[j].w);
    }
  } else {
    tmem_ld_wait<CW>(r);
    if constexpr (B2) {
      tmem_ld16_after_wait(r2);
#pragma unroll
      for (int i = 0; i < CW; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
    }
#pragma unroll
    for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[i]) + bb[i];
  }
  float sn[CW];
  if (p.alpha) {
    // 16 columns at a time keeps the register footprint of the branch-free Snake down
#pragma unroll
    for (int h = 0; h < CW; h += 16) {
      float a[16], ib[16], vv[16], out[16];
      ldg_vec(p.alpha + n0 + h, a);
      ldg_vec(p.invb + n0 + h, ib);
#pragma unroll
      for (int i = 0; i < 16; ++i) vv[i] = v[h + i];
      snake_n<16>(vv, a, ib, out);
#pragma unroll
      for (int i = 0; i < 16; ++i) sn[h + i] = out[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < CW; ++i) sn[i] = v[i];
  }
  if constexpr (CW == 16) {
    if (p.phase_group && !(p.phase_group & 1))
      return store_phase_pair<CW, F16>(p, abort_flag, b, t, n0, v, sn);
  }
  const int ph = n0 / p.Cp_out;  // ConvT phase of these columns (0 for a conv)
  const int co0 = n0 - ph * p.Cp_out;
  const long long out_row = (long long)t * p.s_rows + ph;
  if (out_row >= p.rows_pad) return true;
  if (out_row >= p.rows_valid) {  // padding rows: zeros
#pragma unroll
    for (int i = 0; i < CW; ++i) v[i] = 0.f, sn[i] = 0.f;
  }
  const size_t row_t = static_cast<size_t>(out_row);
  if constexpr (HEAD) {  // the folded output head: this row's partial products per tap
#pragma unroll
    for (int k = 0; k < kHeadFoldMaxK; ++k) {
      float w[CW];
      ldg_vec(p.head_w + (size_t)k * p.Cp_out + co0, w);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < CW; ++i) acc = fmaf(w[i], sn[i], acc);
      hp[k] = acc;
      // one tap's weights in registers at a time (the loads are L1 hits)
      asm volatile("" ::: "memory");
    }
    return true;
  }
  if (p.out_f32) {
    const size_t L_out = static_cast<size_t>(p.f32_L);
    const size_t row = row_t + p.f32_row0;
    const float *src = (p.flags & EPI_F32_SNAKE) ? sn : v;
    VOC_CHECK((((long long)b * (p.Cp_out / 4) + co0 / 4 + CW / 4 - 1) * (long long)L_out + row) * 4 + 4 <= p.f32_elems,
              14, b, co0, row);
    float *base = p.out_f32 + ((size_t)b * (p.Cp_out / 4) + co0 / 4) * L_out * 4 + row * 4;
#pragma unroll
    for (int j = 0; j < CW / 4; ++j)
      *reinterpret_cast<float4 *>(base + (size_t)j * L_out * 4) =
          make_float4(src[4 * j], src[4 * j + 1], src[4 * j + 2], src[4 * j + 3]);
  }
  if (p.out_hl) {
    uint32_t hw[CW / 2], lw[CW / 2];
#pragma unroll
    for (int i = 0; i < CW / 2; ++i) split_pair<F16>(sn[2 * i], sn[2 * i + 1], hw[i], lw[i]);
    const size_t L_out = static_cast<size_t>(p.hl_L);
    if constexpr (ENC) {
      // Phase-split output for a strided conv of stride ss = split_s (ss = 1: the plain
      // layout): row t goes to row t / ss of plane phase_plane(chunk, t % ss), so that the
      // strided conv reads its input as a 3-tap conv over ss * Cp_out channels.
      const size_t ss = static_cast<size_t>(p.split_s > 1 ? p.split_s : 1);
      const size_t ph = row_t % ss, row = row_t / ss + p.hl_row0;
      const size_t cpc = p.Cp_out / 8;
      const size_t half = ss * cpc;  // planes of the hi (and of the lo) parts
      const size_t item = (size_t)b * 2 * half;
#pragma unroll
      for (int j = 0; j < CW / 8; ++j) {
        const size_t plane = phase_plane(co0 / 8 + j, ph, ss, cpc);
        VOC_CHECK(((long long)(item + half + plane) * (long long)L_out + row) * 8 + 8 <= p.hl_elems,
                  20, b, co0, row);
        *reinterpret_cast<uint4 *>(p.out_hl + ((item + plane) * L_out + row) * 8) =
            make_uint4(hw[4 * j], hw[4 * j + 1], hw[4 * j + 2], hw[4 * j + 3]);
        *reinterpret_cast<uint4 *>(p.out_hl + ((item + half + plane) * L_out + row) * 8) =
            make_uint4(lw[4 * j], lw[4 * j + 1], lw[4 * j + 2], lw[4 * j + 3]);
      }
      return true;
    }
    const size_t row = row_t + p.hl_row0;
    const size_t item = (size_t)b * (2 * p.Cp_out / 8);
    VOC_CHECK((((long long)item + p.Cp_out / 8 + co0 / 8 + CW / 8 - 1) * (long long)L_out + row) * 8 + 8 <= p.hl_elems,
              15, b, co0, row);
    __nv_bfloat16 *hbase = p.out_hl + (item + co0 / 8) * L_out * 8 + row * 8;
    __nv_bfloat16 *lbase = p.out_hl + (item + p.Cp_out / 8 + co0 / 8) * L_out * 8 + row * 8;
#pragma unroll
    for (int j = 0; j < CW / 8; ++j) {
      *reinterpret_cast<uint4 *>(hbase + (size_t)j * L_out * 8) =
          make_uint4(hw[4 * j], hw[4 * j + 1], hw[4 * j + 2], hw[4 * j + 3]);
      *reinterpret_cast<uint4 *>(lbase + (size_t)j * L_out * 8) =
          make_uint4(lw[4 * j], lw[4 * j + 1], lw[4 * j + 2], lw[4 * j + 3]);
    }
  }
  return true;
}

// The folded output head, for one warp and one 16-channel chunk: lane l holds hp[k], the
// products of head tap k with its row (32 s + l) summed over the chunk; output row
// 32 s + j - (K - 1) + head_pad (j < 32 + K - 1) receives hp[k] of the lane j - (K - 1) + k.
// Lane l forms the sums j = l and (l < K - 1) j = 32 + l by shuffles and stores them.  Every
// lane of the warp calls this (the shuffles are warp-collective).
__device__ __forceinline__ bool head_fold_store(const ConvGemmArgs &p, const float (&hp)[kHeadFoldMaxK],
                                                int b, int slice, int chunk, int lane,
                                                volatile int *abort_flag) {
  constexpr int K = kHeadFoldMaxK;
  float y0 = 0.f, y1 = 0.f;  // j = lane, j = 32 + lane
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int up = K - 1 - k;  // j = lane reads lane - up
    const float a = __shfl_up_sync(0xffffffffu, hp[k], up);
    if (lane >= up) y0 += a;
    const int src = lane + 32 - up;  // j = 32 + lane reads lane + 32 - up (< 32 only)
    const float c = __shfl_sync(0xffffffffu, hp[k], src & 31);
    if (src < 32) y1 += c;
  }
  const long long base =
      (((long long)b * p.head_slices + slice) * (p.Cp_out / 16) + chunk) * p.head_slice_len;
  VOC_CHECK(slice < p.head_slices && chunk < p.Cp_out / 16 && p.head_K == K &&
                p.head_slice_len == 32 + K - 1,
            23, slice, chunk, p.head_slice_len);
  p.head_part[base + lane] = y0;
  if (lane < K - 1) p.head_part[base + 32 + lane] = y1;
  return true;
}

// Split k (the encoder forms): one warp's 32 rows x CW columns of a k range's raw sums (the
// two halves added in the B2 form), stored fp32 chunk-major for ksplit_reduce_kernel.  Every
// lane reads TMEM (a warp-collective read) before the row check.
template <int CW, bool B2>
__device__ __forceinline__ bool raw_chunk_store(const ConvGemmArgs &p, volatile int *abort_flag,
                                                int b, int t, int ks, int n0, uint32_t taddr) {
  static_assert(CW == 16, "split k stores 16-column chunks");
  uint32_t r[CW], r2[CW];
  tmem_ld_issue<CW>(taddr, r);
  if constexpr (B2) tmem_ld_issue<CW>(taddr + static_cast<uint32_t>(p.N_tile), r2);
  tmem_ld_wait<CW>(r);
  if constexpr (B2) {
    tmem_ld16_after_wait(r2);
#pragma unroll
    for (int i = 0; i < CW; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
  }
  if (t >= p.rows_pad) return true;
  const size_t L = static_cast<size_t>(p.part_L);
  const size_t base = (((size_t)ks * p.B + b) * (p.Cp_out / 4) + n0 / 4) * L + t;
  VOC_CHECK(t < p.part_L && n0 + CW <= p.Cp_out && ks < p.ksplit, 24, t, n0, ks);
#pragma unroll
  for (int j = 0; j < CW / 4; ++j)
    *reinterpret_cast<uint4 *>(p.part + (base + j * L) * 4) =
        make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
  return true;
}

// Taps [tap0, tap1) that k-block kb reads (the encoder's strided convs skip one of three).
__device__ __forceinline__ void tap_window(const ConvGemmArgs &p, int kb, int &tap0, int &tap1) {
  const bool second = kb >= p.kb_split;
  tap0 = second ? p.tap_lo1 : p.tap_lo0;
  tap1 = second ? p.tap_hi1 : p.tap_hi0;
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

// PAIR = false: one CTA per 128-row tile.  PAIR = true: the grid is made of 2-CTA clusters
// and each cluster computes a 256-row tile with the CTA-pair MMA (cta_group::2): each CTA
// stages its own 128-row A halo tile and half of every weight tile (columns
// [rank*N/2, (rank+1)*N/2), packed as separate column tiles), so the weights streamed
// through L2 and shared memory per output row are halved and the tensor core reads half of
// B from each SM.  The even CTA issues the MMAs; the odd CTA's MMA thread relays the
// completion of its own copies to the even CTA's `pair` barriers; the MMA commits
// multicast to both CTAs' barriers; the odd CTA's epilogue warps release an accumulator by
// arriving on the even CTA's barrier.
// drain_ring for a ring whose slots lie `stride` barriers apart.
__device__ __forceinline__ void drain_ring_strided(uint64_t *full, int slots, int stride,
                                                   int issued, long long budget) {
  const volatile int never = 0;
  for (int s = 0; s < slots && s < issued; ++s) {
    const int cnt = (issued - s + slots - 1) / slots;
    mbar_wait(smem_u32(full + s * stride), static_cast<uint32_t>(cnt - 1) & 1u, budget, &never);
  }
}

// B2: the two-MMA K step (ConvGemmArgs::b2).  ODDT: a transposed conv with an odd number of
// phases per group, stored by convT_block_odd.  PREC: the weight form -- kPrecBf16x3 (bf16
// hi/lo weight planes, three MMAs per K step, or two in the B2 form), or one weight plane and
// two MMAs per K step (A_hi x W and A_lo x W): kPrecF16w (f16 operands and f16 hi/lo outputs)
// or kPrecBf16w (bf16 operands and bf16 hi/lo outputs).  ENC: the encoder's forms -- a
// phase-split hi/lo output for a strided conv (ConvGemmArgs::split_s; the last residual unit
// of each block) and per-k-block tap windows (kb_split, tap_lo*, tap_hi*; the strided conv).
// HEAD: the decoder's output head folded into the epilogue (ConvGemmArgs::head_*).  Separate instantiations keep the common form's register budget
// and instruction stream.
template <int CW, bool PAIR, bool B2 = false, bool ODDT = false, int PREC = kPrecBf16x3,
          bool ENC = false, bool HEAD = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    conv_gemm_kernel(const __grid_constant__ CUtensorMap tmapA,
                     const __grid_constant__ CUtensorMap tmapS, const ConvGemmArgs p) {
  constexpr bool F16 = PREC == kPrecF16w;        // f16 operands (else bf16)
  constexpr bool ONE = PREC != kPrecBf16x3;      // one weight plane, two MMAs per K step
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smA + (size_t)p.na * p.a_bytes;
  uint8_t *smS = smB + (size_t)p.nb * p.b_bytes;   // residual slots
  uint64_t *bars = reinterpret_cast<uint64_t *>(smS + (size_t)p.ns * skip_slot_bytes(CW));
  uint64_t *fullA = bars;
  uint64_t *emptyA = fullA + p.na;
  uint64_t *fullB = emptyA + p.na;
  uint64_t *emptyB = fullB + p.nb;
  uint64_t *accFull = emptyB + p.nb;
  uint64_t *accEmpty = accFull + kMaxAcc;
  uint64_t *skipFull = accEmpty + kMaxAcc;
  uint64_t *skipEmpty = skipFull + p.ns;
  uint64_t *pairA = skipEmpty + p.ns;  // even CTA: the odd CTA's A stage has landed
  uint64_t *pairB = pairA + p.na;      // even CTA: the odd CTA's weight stage has landed
  uint64_t *drain = pairB + p.nb;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t tmem_cols = static_cast<uint32_t>(p.n_acc * p.acc_cols);
  constexpr int kM = PAIR ? 2 * kTileM : kTileM;  // rows of one tile job
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int job0 = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int job_step = PAIR ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  const int row0 = static_cast<int>(rank) * kTileM;  // this CTA's rows within a tile job
#ifdef VOC_CHECKS
  // the barrier block must end inside the dynamic allocation
  if (reinterpret_cast<const volatile uint8_t *>(abort_flag + 1) > smem_raw + p.smem_bytes) {
    if (threadIdx.x == 0 && atomicCAS(p.dbg, 0, 1) == 0) {
      p.dbg[1] = static_cast<int>(reinterpret_cast<const volatile uint8_t *>(abort_flag + 1) - smem_raw);
      p.dbg[2] = p.smem_bytes;
    }
    return;  // uniform over the grid: every CTA computes the same layout
  }
#endif
  // set this CTA's and (pair) the other CTA's abort flag
  auto raise_abort = [&]() {
    *abort_flag = 1;
    if (PAIR) st_cluster_u32(mapa_shared(smem_u32(const_cast<int *>(abort_flag)), rank ^ 1u), 1u);
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.na; ++i) {
      mbar_init(smem_u32(fullA + i), 1);
      mbar_init(smem_u32(emptyA + i), 1);
      mbar_init(smem_u32(pairA + i), 1);
    }
    for (int i = 0; i < p.nb; ++i) {
      mbar_init(smem_u32(fullB + i), 1);
      mbar_init(smem_u32(emptyB + i), 1);
      mbar_init(smem_u32(pairB + i), 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(smem_u32(accFull + i), 1);
      mbar_init(smem_u32(accEmpty + i), (PAIR ? 2 : 1) * kEpiWarps);  // one arrival per warp
    }
    for (int i = 0; i < p.ns; ++i) {
      mbar_init(smem_u32(skipFull + i), 1);
      mbar_init(smem_u32(skipEmpty + i), 4 * 32);  // the four quadrant warps of one group
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), tmem_cols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), tmem_cols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (PAIR)
    cluster_sync();  // the other CTA's barriers are initialised before any remote arrival
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
  pdl_launch_dependents();

  const int per_split = p.B * p.m_tiles * p.n_tiles;  // jobs of one k range
  const int total_jobs = ENC ? per_split * p.ksplit : per_split;
  // the tile index and the k-block range of a job (split k in the encoder forms)
  auto job_range = [&](int job, int &jj, int &kb0, int &kb1, int &ks) {
    if constexpr (ENC) {
      ks = job / per_split;
      jj = job - ks * per_split;
      kb0 = ks * p.kb_per_split;
      kb1 = min(p.nkb, kb0 + p.kb_per_split);
    } else {
      ks = 0, jj = job, kb0 = 0, kb1 = p.nkb;
    }
  };
  const int kchunks = p.KB / 8;
  const uint32_t chunkA = static_cast<uint32_t>(p.rows) * 16u;
  const int n_half = PAIR ? p.N_tile / 2 : p.N_tile;  // weight rows staged by this CTA
  const uint32_t chunkB = static_cast<uint32_t>(n_half) * 16u;
  const int n_chunks = p.N_tile / CW;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ A producer
      prefetch_tmap(&tmapA);
      pdl_wait();  // the previous layer's output
      const uint32_t a_tx = 2u * kchunks * chunkA;
      int ia = 0;
      bool ok = true;
      for (int job = job0; job < total_jobs && ok; job += job_step) {
        int jj, kb0, kb1, ks;
        job_range(job, jj, kb0, kb1, ks);
        int nt_, mt, b;
        job_tile(p, jj, nt_, mt, b);
        // first staged row, rounded down to the 8-row group the tensor map addresses (the
        // host adds the remainder, the same for every job, to the MMA row shift)
        const int yg = floor_div8(p.in_row0 + mt * kM + row0 + p.off_min);
        for (int kb = kb0; kb < kb1; ++kb) {
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
            check_fail(p, abort_flag, 21, dstA, kb, p.chunks_a);
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
        raise_abort();
        drain_ring(fullA, p.na, ia, kDrainBudget);  // copies in flight land before the CTA exits
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && PAIR && rank != 0) {
      // ------------------------------------------------------------ odd CTA: relay
      // Tell the even CTA that each of this CTA's stages has landed, in the order the
      // MMA thread consumes them.  A slot is refilled only after the MMAs that read it
      // completed, which needs this relay's arrival first, so no phase is ever skipped.
      const uint32_t remA = mapa_shared(smem_u32(pairA), 0u);
      const uint32_t remB = mapa_shared(smem_u32(pairB), 0u);
      int ia = 0, ib = 0;
      bool ok = true;
      for (int job = job0; job < total_jobs && ok; job += job_step) {
        const bool relay_b = !p.b_resident || job == job0;  // resident slots land once
        for (int kb = 0; kb < p.nkb && ok; ++kb) {
          const int sa = ia % p.na;
          if (!mbar_wait(smem_u32(fullA + sa), static_cast<uint32_t>(ia / p.na) & 1u, p.timeout,
                         abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(remA + static_cast<uint32_t>(sa * 8));
          ++ia;
          for (int tap = 0; tap < p.taps && relay_b; ++tap) {
            const int sb = ib % p.nb;
            if (!mbar_wait(smem_u32(fullB + sb), static_cast<uint32_t>(ib / p.nb) & 1u,
                           p.timeout, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_cluster(remB + static_cast<uint32_t>(sb * 8));
            ++ib;
          }
        }
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_MMA);
        raise_abort();
      }
    } else if (!PAIR || rank == 0) {
      // ------------------------------------------------------------ MMA issuer (whole warp)
      // Every lane runs the loop; waits are made warp-uniform; one elected lane issues
      // each MMA and commit (the same lane every time: the warp is converged).
      auto wait_all = [&](uint32_t bar, uint32_t parity, bool cluster) {
        const bool got = cluster ? mbar_wait_cluster(bar, parity, p.timeout, abort_flag)
                                 : mbar_wait(bar, parity, p.timeout, abort_flag);
        return __all_sync(0xffffffffu, got);
      };
      auto commit = [&](uint64_t *bar) {
        if (PAIR)
          mma_commit_pair_warp(smem_u32(bar), 3);
        else
          mma_commit_warp(smem_u32(bar));
      };
      const uint32_t idesc = F16 ? idesc_f16_f32(kM, p.N_tile) : idesc_bf16_f32(kM, p.N_tile);
      const uint32_t idesc2 = idesc_bf16_f32(kM, 2 * p.N_tile);  // b2: [W_hi | W_lo]
      // Descriptor low words step by 16-byte units: +1 is +16 bytes of start address.  The
      // ring positions (slot, phase) advance incrementally: this loop is issue-bound, so it
      // avoids divisions by run-time ring sizes.
      const uint32_t dA_lo = (kchunks * chunkA) >> 4;
      const uint32_t dA_k = (2 * chunkA) >> 4;
      // b2: the chunks of a weight stage hold 2 * n rows (hi, then lo), so chunks lie
      // 2 * chunkB apart
      const uint32_t chunkB_stride = B2 ? 2 * chunkB : chunkB;
      const uint32_t dB_lo = (kchunks * chunkB) >> 4;
      const uint32_t dB_k = (2 * chunkB_stride) >> 4;
      const uint32_t desc_hi = static_cast<uint32_t>(smem_desc(0u, 0u, 128) >> 32);
      const uint32_t a_desc0 = static_cast<uint32_t>(smem_desc(smem_u32(smA), chunkA, 128));
      const uint32_t b_desc0 = static_cast<uint32_t>(smem_desc(smem_u32(smB), chunkB_stride, 128));
      const uint32_t a_slot_step = static_cast<uint32_t>(p.a_bytes) >> 4;
      const uint32_t b_slot_step = static_cast<uint32_t>(p.b_bytes) >> 4;
      const int nks = kchunks / 2;
      int sa = 0, sb = 0, acc = 0;
      uint32_t pha = 0, phb = 0, phacc = 0;
      bool ok = true;
      for (int job = job0; job < total_jobs && ok; job += job_step) {
        int jj, kb0, kb1, ks;
        job_range(job, jj, kb0, kb1, ks);
        int nt, mt_, b_;
        job_tile(p, jj, nt, mt_, b_);
        const int shift0 = (nt >= p.q_split_tile) ? p.shift0_q1 : p.shift0_q0;
        if (!wait_all(smem_u32(accEmpty + acc), phacc ^ 1u, PAIR)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.acc_cols);
        uint32_t accum = 0u;  // the first MMA of a job overwrites the accumulator
        for (int kb = kb0; kb < kb1 && ok; ++kb) {
          if (!wait_all(smem_u32(fullA + sa), pha, false) ||
              (PAIR && !wait_all(smem_u32(pairA + sa), pha, true))) {
            ok = false;
            break;
          }
          tc_fence_after();
          int tap0 = 0, tap1 = p.taps;
          if constexpr (ENC) tap_window(p, kb, tap0, tap1);
          uint32_t a0 = a_desc0 + sa * a_slot_step + static_cast<uint32_t>(shift0 + tap0 * p.tap_step);
          for (int tap = tap0; tap < tap1; ++tap, a0 += static_cast<uint32_t>(p.tap_step)) {
            // a resident slot completes its first phase only, in this CTA's first job;
            // later jobs issue on it without a wait
            if (!p.b_resident || job == job0) {
              const uint32_t wph = p.b_resident ? 0u : phb;
              if (!wait_all(smem_u32(fullB + sb), wph, false) ||
                  (PAIR && !wait_all(smem_u32(pairB + sb), wph, true))) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
#ifdef VOC_CHECKS
            {
              const int sh = shift0 + tap * p.tap_step;
              if (!__all_sync(0xffffffffu, sh >= 0 && sh + kTileM <= p.rows)) {
                if (lane == 0) check_fail(p, abort_flag, 31, sh, tap, p.rows);
                ok = false;
                break;
              }
            }
#endif
            uint32_t a_hi = a0, b_hi = b_desc0 + sb * b_slot_step;
            if constexpr (ONE) {  // one weight plane
              for (int ks = 0; ks < nks; ++ks, a_hi += dA_k, b_hi += dB_k) {
                mma_bf16_warp_lo<PAIR>(d_tmem, a_hi, b_hi, desc_hi, idesc, accum);
                mma_bf16_warp_lo<PAIR>(d_tmem, a_hi + dA_lo, b_hi, desc_hi, idesc, 1u);
                accum = 1u;
              }
            } else if constexpr (B2) {
              for (int ks = 0; ks < nks; ++ks, a_hi += dA_k, b_hi += dB_k) {
                mma_bf16_warp_lo<PAIR>(d_tmem, a_hi, b_hi, desc_hi, idesc2, accum);
                mma_bf16_warp_lo<PAIR>(d_tmem, a_hi + dA_lo, b_hi, desc_hi, idesc, 1u);
                accum = 1u;
              }
            } else {  // A_hi x W_hi and A_hi x W_lo share A through the collector buffer
              for (int ks = 0; ks < nks; ++ks, a_hi += dA_k, b_hi += dB_k) {
                mma_bf16_warp_lo_col<PAIR, 1>(d_tmem, a_hi, b_hi, desc_hi, idesc, accum);
                mma_bf16_warp_lo_col<PAIR, 2>(d_tmem, a_hi, b_hi + dB_lo, desc_hi, idesc, 1u);
                mma_bf16_warp_lo<PAIR>(d_tmem, a_hi + dA_lo, b_hi, desc_hi, idesc, 1u);
                accum = 1u;
              }
            }
            if (!p.b_resident) commit(emptyB + sb);
            if (++sb == p.nb) sb = 0, phb ^= 1u;
          }
          if (!ok) break;
          commit(emptyA + sa);
          if (++sa == p.na) sa = 0, pha ^= 1u;
        }
        if (!ok) break;
        commit(accFull + acc);
        if (++acc == p.n_acc) acc = 0, phacc ^= 1u;
      }
      if (!ok) {
        if (lane == 0) {
          atomicOr(p.err, ERR_TIMEOUT_MMA);
          raise_abort();
        }
        // wait until every MMA issued so far has finished reading shared memory
        if (PAIR)
          mma_commit_pair_warp(smem_u32(drain), 1);
        else
          mma_commit_warp(smem_u32(drain));
        const volatile int never = 0;
        mbar_wait(smem_u32(drain), 0u, kDrainBudget, &never);
      }
    }
  } else if (warp >= kBWarp) {
    if (lane == 0) {
      // ------------------------------------------------------------ weight producer
      // Stage ib goes to slot ib % nb (with several producer warps, nb is a multiple of
      // their count and warp kBWarp + j fills the slots congruent to j).
      const int j = warp - kBWarp;
      int ib = 0, mine = 0;
      bool ok = true;
      // resident weights: one pass over the stages of the first job fills every slot
      const int job_end = p.b_resident ? min(total_jobs, job0 + 1) : total_jobs;
      for (int job = job0; job < job_end && ok; job += job_step) {
        int jj, kb0, kb1, ks;
        job_range(job, jj, kb0, kb1, ks);
        int nt, mt_, b_;
        job_tile(p, jj, nt, mt_, b_);
        const int wt = PAIR ? 2 * nt + static_cast<int>(rank) : nt;  // packed weight tile
        for (int kb = kb0; kb < kb1 && ok; ++kb) {
          int tap0 = 0, tap1 = p.taps;
          if constexpr (ENC) tap_window(p, kb, tap0, tap1);
          for (int tap = tap0; tap < tap1; ++tap, ++ib) {
            if (ib % kBWarps != j) continue;
            const int sb = ib % p.nb;
            const uint32_t phb = static_cast<uint32_t>(ib / p.nb) & 1u;
            if (!mbar_wait(smem_u32(emptyB + sb), phb ^ 1u, p.timeout, abort_flag)) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(fullB + sb);
            const size_t widx = ((size_t)wt * p.taps + tap) * p.nkb + kb;
#ifdef VOC_CHECKS
            if (!((long long)(widx + 1) * p.b_bytes <= p.w_bytes && (p.nb % kBWarps) == 0 &&
                  smem_u32(smB + (size_t)(sb + 1) * p.b_bytes) <= smem_u32(smS))) {
              check_fail(p, abort_flag, 22, widx, sb, p.w_bytes);
              ok = false;
              break;
            }
#endif
            mbar_arrive_expect_tx(fb, static_cast<uint32_t>(p.b_bytes));
            bulk_load(smem_u32(smB + (size_t)sb * p.b_bytes), p.wB + widx * p.b_bytes,
                      static_cast<uint32_t>(p.b_bytes), fb);
            ++mine;
          }
        }
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_PRODUCER);
        raise_abort();
        // this warp's slots j, j + kBWarps, ... form a ring of nb / kBWarps slots
        drain_ring_strided(fullB + j, p.nb / kBWarps, kBWarps, mine, kDrainBudget);
      }
    }
  } else if (warp == kSkipWarp) {
    if (lane == 0 && p.skip) {
      // ------------------------------------------------------------ residual prefetch
      prefetch_tmap(&tmapS);
      pdl_wait();
      // Chunk c of a tile is consumed by epilogue group c % kEpiGroups; each group has its
      // own ring of ns / kEpiGroups slots, filled in that group's consumption order, so a
      // slot is only ever waited on by one sequence of consumers, at most one fill ahead.
      // One thread fills the three rings, chunk by chunk in column order.
      const uint32_t bytes = static_cast<uint32_t>(skip_slot_bytes(CW));
      const int nsh = p.ns / kEpiGroups;
      int cnt[kEpiGroups] = {};  // fills issued into each group's ring
      int pos[kEpiGroups] = {};  // their ring positions and phases, advanced incrementally
      uint32_t ph[kEpiGroups] = {};
      bool ok = true;
      for (int job = job0; job < total_jobs && ok; job += job_step) {
        int nt, mt, b;
        job_tile(p, job, nt, mt, b);
        for (int c0 = 0; c0 < n_chunks && ok; c0 += kEpiGroups) {
#pragma unroll
          for (int h = 0; h < kEpiGroups; ++h) {
            const int c = c0 + h;
            if (c >= n_chunks || !ok) continue;
            const int slot = h * nsh + pos[h];
            if (!mbar_wait(smem_u32(skipEmpty + slot), ph[h] ^ 1u, p.timeout, abort_flag)) {
              ok = false;
              continue;
            }
            const uint32_t fs = smem_u32(skipFull + slot);
#ifdef VOC_CHECKS
            if (!(smem_u32(smS + (size_t)(slot + 1) * bytes) <= smem_u32(bars) &&
                  (nt * p.N_tile + c * CW) / 4 + CW / 4 <= p.chunks_s)) {
              check_fail(p, abort_flag, 41, slot, nt * p.N_tile + c * CW, p.chunks_s);
              ok = false;
              continue;
            }
#endif
            mbar_arrive_expect_tx(fs, bytes);
            tma_load_4d(smem_u32(smS + (size_t)slot * bytes), &tmapS, fs, 0, (mt * kM + row0) / 8,
                        (nt * p.N_tile + c * CW) / 4, b);
            ++cnt[h];
            if (++pos[h] == nsh) pos[h] = 0, ph[h] ^= 1u;
          }
        }
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_SKIP);
        raise_abort();
#pragma unroll
        for (int h = 0; h < kEpiGroups; ++h) drain_ring(skipFull + h * nsh, nsh, cnt[h], kDrainBudget);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    pdl_wait();  // this layer's outputs overwrite buffers earlier layers read
    const int e = warp - 2;     // epilogue warp 0..kEpiWarps-1
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int half = e / 4;     // this warp's group: column chunks half, half + kEpiGroups, ...
    const int row_in_tile = quad * 32 + lane;
    const uint32_t sbase = smem_u32(smS);
    const int nsh = p.ns > 0 ? p.ns / kEpiGroups : 1;  // residual slots of this group's ring
    constexpr bool odd_blocks = ODDT;
    // where this warp reports a free accumulator: this CTA's barrier, or the even CTA's
    const uint32_t acc_empty0 = PAIR ? mapa_shared(smem_u32(accEmpty), 0u) : smem_u32(accEmpty);
    int kslot = 0;                           // this group's residual ring position
    uint32_t kph = 0;
    int acc = 0;                             // accumulator ring position
    uint32_t phacc = 0;
    bool ok = true;
    for (int job = job0; job < total_jobs && ok; job += job_step) {
      int jj, kb0, kb1, ks;
      job_range(job, jj, kb0, kb1, ks);
      int nt, mt, b;
      job_tile(p, jj, nt, mt, b);
      // decisions stay warp-uniform: tcgen05.ld is a warp-collective instruction
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(accFull + acc), phacc, p.timeout, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int t = mt * kM + row0 + row_in_tile;
      const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * p.acc_cols) +
                             (static_cast<uint32_t>(quad * 32) << 16);
      if constexpr (odd_blocks) {  // ConvT with an odd number of phases: whole 8-channel blocks
        const int bw = 8 * p.phase_group;
        for (int blk = half; blk < p.N_tile / bw && ok; blk += kEpiGroups) {
          ok = convT_block_odd<F16>(p, abort_flag, b, t, nt * p.N_tile + blk * bw, tbase + blk * bw, lane);
          ok = __all_sync(0xffffffffu, ok);
        }
      }
      if constexpr (ENC) {
        if (p.ksplit > 1) {  // split k: this range's raw sums, finished by ksplit_reduce_kernel
          for (int c = half; c < n_chunks && ok; c += kEpiGroups) {
            ok = raw_chunk_store<CW, B2>(p, abort_flag, b, t, ks, nt * p.N_tile + c * CW,
                                         tbase + c * CW);
            ok = __all_sync(0xffffffffu, ok);
          }
          tc_fence_before();
          __syncwarp();
          if (!ok) break;
          if (lane == 0) mbar_arrive(smem_u32(accEmpty + acc));
          if (++acc == p.n_acc) acc = 0, phacc ^= 1u;
          continue;
        }
      }
      for (int c = half; c < n_chunks && ok && !odd_blocks; c += kEpiGroups) {
        const int slot = half * nsh + kslot;
        float hp[kHeadFoldMaxK] = {};
        ok = epilogue_chunk<CW, B2, F16, ENC, HEAD>(p, sbase + static_cast<uint32_t>(slot * skip_slot_bytes(CW)),
                                smem_u32(skipFull + slot), smem_u32(skipEmpty + slot), kph,
                                abort_flag, row_in_tile, b, t, nt * p.N_tile + c * CW,
                                tbase + c * CW, sbase, smem_u32(bars), hp);
        ok = __all_sync(0xffffffffu, ok);
        if constexpr (HEAD) {
          if (ok)
            ok = head_fold_store(p, hp, b, (mt * kM + row0) / 32 + quad, nt * (p.N_tile / CW) + c,
                                 lane, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
        }
        if (++kslot == nsh) kslot = 0, kph ^= 1u;
      }
      // every lane's TMEM reads of this accumulator are complete before lane 0 frees it
      tc_fence_before();
      __syncwarp();
      if (!ok) break;
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(acc_empty0 + static_cast<uint32_t>(acc * 8));
        else
          mbar_arrive(smem_u32(accEmpty + acc));
      }
      if (++acc == p.n_acc) acc = 0, phacc ^= 1u;
    }
    if (!ok) {
      atomicOr(p.err, ERR_TIMEOUT_EPILOGUE);
      raise_abort();
    }
  }

  __syncwarp();
  tc_fence_before();
  if (PAIR)
    cluster_sync();  // neither CTA leaves while the other may still reach its shared memory
  else
    __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, tmem_cols);
    else
      tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace voc
