// vocoder.cu -- C ABI of the GB300 vocoder decoder (declared in include/vocoder.h):
// validation, weight folding and packing, workspace planning, TMA descriptors and
// the launch sequence of one decode.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "vocoder.h"
#include "conv_gemm.cuh"
#include "ru_gemm.cuh"
#include "stream_kernels.cuh"
#include "output_stage.cuh"

#define VOC_API extern "C" __attribute__((visibility("default")))

namespace {

using voc::ConvGemmArgs;

constexpr int kSmemMax = 227 * 1024;         // opt-in shared memory per block
constexpr long long kWaitBudget = 4000000000LL;  // cycles (~2 s) before a wait gives up
constexpr int kHeadTile = 128;
// mbarriers (3 per A and weight slot, 2 per residual slot and accumulator, 1 drain), TMEM
// slot, flag
constexpr int kBarrierBytes = 1536;
constexpr int kMaxResidentStages = 32;  // weight slots of a resident plan
constexpr int kMaxResidentTiles = 8;    // column tiles of a resident plan (one per CTA)
constexpr int kMinAInFlight = 48 * 1024;  // A ring bytes a resident plan must keep
constexpr int kBStageMax = 36 * 1024;  // bytes of one weight stage (per CTA)
constexpr double kBandWeightBytes = 32e6;  // weights from which a layer takes the band job order
constexpr int kBandRows = 12;             // row tiles of one band

thread_local std::string g_err;  // last error without a context

// Every device allocation of the library goes through dev_alloc / dev_free, which keep a
// count of the live ones and can be told to fail one on purpose (the allocation-failure
// test hook vocoder_debug_fail_allocation).
std::atomic<long long> g_live_allocs{0};
std::atomic<int> g_fail_countdown{-1};  // >= 0: allocations to let through before one fails

cudaError_t dev_alloc(void **p, size_t bytes) {
  int n = g_fail_countdown.load();
  while (n >= 0 && !g_fail_countdown.compare_exchange_weak(n, n - 1)) {
  }
  if (n == 0) {  // this one fails, as cudaMalloc does when the device is out of memory
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  const cudaError_t e = cudaMalloc(p, bytes);
  if (e == cudaSuccess) ++g_live_allocs;
  return e;
}

void dev_free(void *p) {
  if (!p) return;
  if (cudaFree(p) == cudaSuccess) --g_live_allocs;
}

int rup(int x, int m) { return (x + m - 1) / m * m; }
// Launch with programmatic stream serialization: the kernel may be scheduled while the
// previous kernel of the stream finishes; it orders its own accesses with griddepcontrol.wait
// (pdl_wait in the kernels).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Rows of a chunk-major plane: a multiple of 8, the row group the tensor maps address.
long long pitch8(long long rows) { return (rows + 7) / 8 * 8; }
// x mod 8 in [0, 8) for any sign
int mod8(int x) { return ((x % 8) + 8) % 8; }
size_t rupz(size_t x, size_t m) { return (x + m - 1) / m * m; }

uint16_t f2bf(float f) {  // round to nearest even (finite inputs)
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}
float bf2f(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

enum Buf { BUF_H0 = 0, BUF_H1 = 1, BUF_HB = 2, BUF_FY = 3, BUF_COUNT = 4 };

struct Layer {
  std::string name;
  bool convT = false;
  int prec = VOC_PREC_BF16X3;  // VOC_PREC_*: bf16 hi/lo weights, or one f16 / bf16 plane
  // strided conv of the encoder (stride down_s, k = 2 down_s, pad down_s / 2, down_c real
  // input channels), run as a 3-tap conv over the phase-split input: Cin = down_s * Cp(down_c)
  int down_s = 0, down_c = 0;
  int Cin = 0, Cout = 0, Cp_in = 0, Cp_out = 0, K = 0, dil = 1, stride = 1;
  int level = 0;            // input rate: L_in = T * prod(strides[0..level-1])
  ConvGemmArgs g{};         // geometry; sizes and pointers filled per launch
  size_t smem = 0;
  uint8_t *w_dev = nullptr;
  float *bias_dev = nullptr, *alpha_dev = nullptr, *invb_dev = nullptr;
  int in_buf = -1, f32_buf = -1, hl_buf = -1, skip_buf = -1;
  int epi_flags = 0;
  int cw = 16;              // epilogue column chunk (16 columns in both kernels)
  bool pair = false;        // CTA-pair kernel: 256-row tiles, half of each weight tile per CTA
  int max_clusters = 0;     // pair: co-resident 2-CTA clusters of this launch shape
  // the encoder's conv_in on a few audio channels, run directly in fp32 (audio_conv_in_kernel,
  // weights wf_dev [Cout][Cin][K]) instead of as a GEMM over 16 padded channels
  bool direct = false;
  float *wf_dev = nullptr;
  // the output head folded into this layer's epilogue (the decoder's last conv2, in a
  // whole-sequence decode): partial sums go to hi/lo buffer head_buf, which it does not read
  bool head_fold = false;
  int head_buf = -1;
  // fused residual unit (conv1 k-tap + conv2 1x1 in one kernel)
  bool ru = false;
  voc::RuExtra rx{};
};

struct OutHead {
  int C = 0, Cp = 0, K = 0, pad_left = 0, level = 0;
  float *w_dev = nullptr, *b_dev = nullptr;
  float *w4_dev = nullptr;  // [K][Cp/4] channel quadruples for the register-blocked kernel
  float *wk_dev = nullptr;  // [K][Cp] for the head folded into the last conv2
};
constexpr int kHeadTpt = 2;  // samples per thread of the register-blocked head

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Conv kernel forms used for the precision PREC (voc::kPrec*): plain, odd-phase ConvT and
// phase-split output; the bf16x3 precision also has the B2 forms and the CTA-pair kernel.
template <int PREC>
cudaError_t set_conv_attrs() {
  auto set = [](auto kernel) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
  };
  cudaError_t st = set(voc::conv_gemm_kernel<16, false, false, false, PREC>);
  if (st == cudaSuccess) st = set(voc::conv_gemm_kernel<16, false, false, true, PREC>);
  if (st == cudaSuccess) st = set(voc::conv_gemm_kernel<16, false, false, false, PREC, true>);
  if (st == cudaSuccess) st = set(voc::conv_gemm_kernel<16, false, false, false, PREC, false, true>);
  if constexpr (PREC == voc::kPrecBf16x3) {
    if (st == cudaSuccess) st = set(voc::conv_gemm_kernel<16, false, true>);
    if (st == cudaSuccess) st = set(voc::conv_gemm_kernel<16, false, true, false, PREC, true>);
    if (st == cudaSuccess) st = set(voc::conv_gemm_kernel<16, false, true, false, PREC, false, true>);
    if (st == cudaSuccess) st = set(voc::conv_gemm_kernel<16, true>);
  }
  return st;
}

// The fused residual-unit kernel splits its block's registers between warp groups with
// setmaxnreg, which waits until the registers it asks for are free: it is only launched when the
// block gets the registers per thread the split assumes (set_kernel_attrs checks every form).
bool g_ru_regs_ok = false;

bool set_kernel_attrs(std::string &why) {
  static cudaError_t st = cudaErrorUnknown;
  static std::once_flag once;
  std::call_once(once, [] {
    st = set_conv_attrs<voc::kPrecBf16x3>();
    if (st == cudaSuccess) st = set_conv_attrs<voc::kPrecF16w>();
    if (st == cudaSuccess) st = set_conv_attrs<voc::kPrecBf16w>();
    auto set_ru = [](auto kernel) {
      return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    };
    if (st == cudaSuccess) st = set_ru(voc::ru_gemm_kernel<false, false>);
    if (st == cudaSuccess) st = set_ru(voc::ru_gemm_kernel<true, false>);
    if (st == cudaSuccess) st = set_ru(voc::ru_gemm_kernel<false, true>);
    if (st == cudaSuccess) st = set_ru(voc::ru_gemm_kernel<true, true>);
    if (st == cudaSuccess) st = set_ru(voc::ru_gemm_kernel<true, false, true>);
    if (st == cudaSuccess) st = set_ru(voc::ru_gemm_kernel<true, true, true>);
    if (st == cudaSuccess) st = set_ru(voc::ru_gemm_kernel<false, false, false, voc::kPrecF16w>);
    if (st == cudaSuccess) st = set_ru(voc::ru_gemm_kernel<false, true, false, voc::kPrecF16w>);
    if (st == cudaSuccess) st = set_ru(voc::ru_gemm_kernel<false, false, false, voc::kPrecBf16w>);
    if (st == cudaSuccess) st = set_ru(voc::ru_gemm_kernel<false, true, false, voc::kPrecBf16w>);
    if (st == cudaSuccess) {
      auto regs_ok = [](auto kernel) {
        cudaFuncAttributes fa{};
        return cudaFuncGetAttributes(&fa, kernel) == cudaSuccess &&
               fa.numRegs * voc::kRuThreads >=
                   128 * voc::kRuCopyRegs + 32 * voc::kRuEpiWarps * voc::kRuEpiRegs;
      };
      g_ru_regs_ok = regs_ok(voc::ru_gemm_kernel<false, false>) &&
                     regs_ok(voc::ru_gemm_kernel<true, false>) &&
                     regs_ok(voc::ru_gemm_kernel<false, true>) &&
                     regs_ok(voc::ru_gemm_kernel<true, true>) &&
                     regs_ok(voc::ru_gemm_kernel<true, false, true>) &&
                     regs_ok(voc::ru_gemm_kernel<true, true, true>) &&
                     regs_ok(voc::ru_gemm_kernel<false, false, false, voc::kPrecF16w>) &&
                     regs_ok(voc::ru_gemm_kernel<false, true, false, voc::kPrecF16w>) &&
                     regs_ok(voc::ru_gemm_kernel<false, false, false, voc::kPrecBf16w>) &&
                     regs_ok(voc::ru_gemm_kernel<false, true, false, voc::kPrecBf16w>);
    }
    if (st == cudaSuccess)
      st = cudaFuncSetAttribute(voc::out_head_kernel<kHeadTile>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
  });
  if (st != cudaSuccess) why = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(st);
  return st == cudaSuccess;
}

}  // namespace

struct vocoder {
  voc_desc desc{};
  std::vector<int> strides, widths, dils;
  int device = 0, num_sms = 0;
  int Cp_lat = 0;
  long long hop = 1;
  std::vector<Layer> layers;
  OutHead head;
  std::vector<void *> allocs;
  std::string err;
  int *err_dev = nullptr;   // device error word of the kernels (bounded waits)
  int *flag_dev = nullptr;  // finite-check flag
  long long wait_budget = kWaitBudget;
  int fuse_max_c = 0;       // residual units of up to this many (padded) channels run fused
  int fuse_min_c = 0;       // ... and of at least this many
  bool use_pair = true;     // conv layers on CTA pairs
  int prec = VOC_PREC_BF16X3;  // VOC_PREC_*: the weight form of every conv
  // TMA descriptors of the two most recent (workspace, B, T) of a decode, each set sized for
  // every layer at create time, so that a decode encodes descriptors only for a new
  // combination and never resizes them (a caller alternating two workspaces, e.g. its own
  // and the no-allocation decode's, re-encodes nothing)
  struct MapSet {
    void *ws = nullptr;
    int B = -1, T = -1;
    std::vector<CUtensorMap> maps, skip_maps;
  };
  MapSet map_sets[2];
  int map_lru = 0;  // the set a new combination replaces
  const volatile int *cancel = nullptr;  // caller's cancel flag (vocoder_set_cancel_flag)
  // profiling of the last decode with VOC_FLAG_PROFILE
  std::vector<cudaEvent_t> events;
  std::vector<std::string> prof_names;
  std::vector<double> prof_flops, prof_bytes, prof_impl;  // algorithmic / implementation bytes
  std::vector<float> prof_ms;
  int prof_n = 0;
  bool prof_ready = false;
};

namespace {

voc_status fail(vocoder *ctx, voc_status st, const std::string &msg) {
  if (ctx)
    ctx->err = msg;
  else
    g_err = msg;
  return st;
}

voc_status cuda_fail(vocoder *ctx, cudaError_t e, const char *what) {
  return fail(ctx, e == cudaErrorMemoryAllocation ? VOC_OOM : VOC_CUDA_ERROR,
              std::string(what) + ": " + cudaGetErrorString(e));
}

// ------------------------------------------------------------------ planning
// Plan the GEMM geometry of one conv (convT = false) or transposed conv layer.
bool plan_gemm(Layer &L, int padding, bool has_skip, std::string &why) {
  ConvGemmArgs &g = L.g;
  L.Cp_in = rup(L.Cin, 16);
  L.Cp_out = rup(L.Cout, 16);
  g.Cp_in = L.Cp_in;
  g.Cp_out = L.Cp_out;
  int group, off_min, off_max;
  if (L.convT) {
    const int s = L.stride;
    g.taps = 2;
    g.N_total = s * L.Cp_out;
    g.s_rows = s;
    // stride 2, symmetric: phase 0 reads rows t-1 and t, phase 1 rows t and t+1.  Both phases
    // share one column tile as a 3-shift conv over rows t-1, t, t+1 (each phase's weights are
    // zero on the shift it does not read), so a row block stages its input once and its two
    // output rows leave as row pairs, instead of two half-width tiles staging the rows twice.
    const bool shifts3 = padding == VOC_PAD_SYMMETRIC && s == 2 && L.Cp_out % 8 == 0;
    if (shifts3) {
      g.taps = 3;
      group = g.N_total;
      off_min = -1, off_max = 1;
      g.shift0_q0 = g.shift0_q1 = 0;
    } else if (padding == VOC_PAD_SYMMETRIC) {
      // phases r < s/2 read rows t and t-1 (q = 0), phases r >= s/2 rows t+1 and t (q = 1)
      group = (s / 2) * L.Cp_out;
      off_min = -1, off_max = 1;
      g.shift0_q0 = 1, g.shift0_q1 = 2;
    } else {
      group = g.N_total;  // causal: every phase reads rows t and t-1
      off_min = -1, off_max = 0;
      g.shift0_q0 = 1, g.shift0_q1 = 1;
    }
    g.tap_step = shifts3 ? 1 : -1;
    // Output columns of a phase group of G phases: with G even, each 8-channel block holds
    // its G phases consecutively (8 columns per phase), so a 16-column epilogue chunk holds
    // two consecutive output rows of 8 channels and is written with 32-byte stores; with G
    // odd, phase-major (n = r * Cp_out + co within the group).
    // With G odd (causal s = 3, 5) the columns are blocked the same way and the epilogue
    // stores whole blocks through lane pairs (the causal output rows of a lane pair are 2G
    // consecutive rows); the column tile then holds whole blocks.
    const int G = shifts3 ? 2 : (padding == VOC_PAD_SYMMETRIC) ? s / 2 : s;
    // (the CTA-pair kernel has no odd-phase epilogue)
    g.phase_group = (L.Cp_out % 8 == 0 && (G % 2 == 0 || (padding == VOC_PAD_CAUSAL && !L.pair)))
                        ? G : 0;
  } else {
    const int span = L.dil * (L.K - 1);
    const int pad_left = (padding == VOC_PAD_CAUSAL) ? span : span / 2;
    g.taps = L.K;
    g.N_total = L.Cp_out;
    g.s_rows = 1;
    group = g.N_total;
    off_min = -pad_left, off_max = span - pad_left;
    g.shift0_q0 = g.shift0_q1 = 0;
    g.tap_step = L.dil;
  }
  g.N_tile = 0;
  for (int t = 256; t >= 16; t -= 16)
    if (group % t == 0 && !(L.convT && (g.phase_group & 1) && t % (8 * g.phase_group))) {
      g.N_tile = t;
      break;
    }
  if (!g.N_tile && L.convT && (g.phase_group & 1)) {  // no tile of whole blocks: phase-major
    g.phase_group = 0;
    for (int t = 256; t >= 16; t -= 16)
      if (group % t == 0) {
        g.N_tile = t;
        break;
      }
  }
  if (!g.N_tile) {
    why = "no column tile divides " + std::to_string(group);
    return false;
  }
  g.n_tiles = g.N_total / g.N_tile;
  g.q_split_tile = (L.convT && padding == VOC_PAD_SYMMETRIC && g.taps == 2) ? group / g.N_tile
                                                                            : g.n_tiles;
  g.off_min = off_min;
  // the staged rows start at the 8-row group holding the first row (mod8(off_min) rows
  // earlier when the input rows start at a multiple of 8)
  g.rows = rup(voc::kTileM + off_max - off_min + mod8(off_min), 8);
  if (g.rows > 256) {
    why = "tap span too wide for one staged tile (" + std::to_string(off_max - off_min) + ")";
    return false;
  }
  // epilogue column chunk: 16 columns (three groups of epilogue warps take every third
  // chunk; 16-column chunks keep the register footprint within the 512-thread block)
  L.cw = 16;
  // weight columns staged per CTA: the whole tile, or (CTA pair) one half of it
  const int n_stage = L.pair ? g.N_tile / 2 : g.N_tile;
  // Channels per k-block: the largest multiple of 16 dividing Cp_in whose weight stage
  // stays within kBStageMax and A stage within 72 KB and that still leaves two weight
  // slots.  Each stage costs a copy request and a barrier round trip whatever its size,
  // so fewer, larger stages run faster.
  const int chunkA = g.rows * 16;
  const int sb = has_skip ? voc::skip_slot_bytes(L.cw) : 0;
  g.KB = 0;
  g.b_resident = 0;
  // Resident weights: when the whole column tile of a CTA (taps x Cp_in x n_stage hi/lo
  // pairs) fits beside the A ring and the residual slots, it is loaded once and kept; the
  // k-block is then the largest that leaves three A stages (else two) and at least
  // kMinAInFlight bytes of A in flight (the 1x1 convs wait on their A loads otherwise).
  // weight bytes per (channel, column): one f16 or bf16 value, or bf16 hi + lo
  const int wb = L.prec != VOC_PREC_BF16X3 ? 2 : 4;
  // a strided conv (down_s) reads two of its three taps per k-block: its k-blocks lie within
  // one phase group (ceil(s/2) Cp or floor(s/2) Cp channels)
  const int taps_eff = L.down_s ? 2 : g.taps;
  const int grp0 = L.down_s ? ((L.down_s + 1) / 2) * (L.Cin / L.down_s) : L.Cp_in;
  const int grp1 = L.down_s ? (L.down_s / 2) * (L.Cin / L.down_s) : 0;
  auto kb_ok = [&](int kb) { return L.Cp_in % kb == 0 && grp0 % kb == 0 && grp1 % kb == 0; };
  const int w_tile = wb * L.Cp_in * n_stage * taps_eff;
  for (int min_na = 3; min_na >= 2 && !g.KB && g.n_tiles <= kMaxResidentTiles; --min_na)
    for (int kb = L.Cp_in - L.Cp_in % 16; kb >= 16 && !g.KB; kb -= 16) {
      if (!kb_ok(kb) || 4 * kb * g.rows > 72 * 1024) continue;
      // a k-tap conv keeps its weights resident only when one k-block covers its channels:
      // with smaller k-blocks every tile restages its halo rows once per k-block, which costs
      // more than streaming the weights (the encoder's C = 64 dilated convs: 0.167 -> 0.122 ms)
      if (g.taps > 1 && kb != L.Cp_in) continue;
      if (taps_eff * (L.Cp_in / kb) > kMaxResidentStages) continue;
      const int a_bytes = rup(2 * (kb / 8) * chunkA, 1024);
      const int ns = has_skip ? 2 * voc::kEpiGroups : 0;
      const int avail = kSmemMax - 1024 - kBarrierBytes - w_tile - ns * sb;
      // a 1x1 conv consumes each A stage almost at once: its A ring hides the HBM latency
      const int na = std::min(g.taps == 1 ? 8 : 4, avail / a_bytes);
      if (na < min_na || na * a_bytes < kMinAInFlight) continue;
      g.KB = kb, g.a_bytes = a_bytes, g.b_bytes = wb * kb * n_stage, g.na = na, g.ns = ns;
      g.nb = taps_eff * (L.Cp_in / kb);
      g.b_resident = 1;
    }
  // streaming weights: a 1x1 conv gets up to four A stages (its A comes from HBM and is
  // consumed at once; its weight stages come from L2), a k-tap conv two
  const int na_want = g.taps == 1 ? 4 : 2;
  for (int kb = L.Cp_in - L.Cp_in % 16; kb >= 16 && !g.KB; kb -= 16) {
    if (!kb_ok(kb) || wb * kb * n_stage > kBStageMax || 4 * kb * g.rows > 72 * 1024) continue;
    const int a_bytes = rup(2 * (kb / 8) * chunkA, 1024);
    const int b_bytes = wb * kb * n_stage;
    int na = na_want;
    while (na > 2 && kSmemMax - 1024 - kBarrierBytes - na * a_bytes < 3 * b_bytes) --na;
    int avail = kSmemMax - 1024 - kBarrierBytes - na * a_bytes;
    int ns = 0;
    if (has_skip) {  // one ring per epilogue group, of 2 slots (1 when space is short)
      ns = ((avail - 2 * voc::kEpiGroups * sb) / b_bytes >= 3) ? 2 * voc::kEpiGroups
                                                                : voc::kEpiGroups;
      avail -= ns * sb;
    }
    int nb = std::min(8, avail / b_bytes);
    nb -= nb % voc::kBWarps;  // each weight-producer warp owns every kBWarps-th slot
    if (nb < 2) continue;
    g.KB = kb, g.a_bytes = a_bytes, g.b_bytes = b_bytes, g.nb = nb, g.ns = ns, g.na = na;
  }
  if (!g.KB) {
    why = "shared memory plan does not fit";
    return false;
  }
  // mbarriers: full/empty/pair per A and weight slot, full/empty per residual slot and
  // accumulator, one drain; then the TMEM address slot and the abort flag
  if ((3 * g.na + 3 * g.nb + 2 * g.ns + 2 * voc::kMaxAcc + 1) * 8 + 8 > kBarrierBytes) {
    why = "too many pipeline slots for the barrier block";
    return false;
  }
  g.nkb = L.Cp_in / g.KB;
  // taps of each k-block (the encoder kernels read these): all, or for a strided conv taps
  // 1, 2 (row shifts 0, +1) in the first phase group and 0, 1 (-1, 0) in the second
  g.ksplit = 1, g.kb_per_split = g.nkb;  // split k is chosen per encode (encoder layers)
  g.kb_split = L.down_s ? grp0 / g.KB : g.nkb;
  g.tap_lo0 = L.down_s ? 1 : 0, g.tap_hi0 = g.taps;
  g.tap_lo1 = 0, g.tap_hi1 = L.down_s ? 2 : g.taps;
  // Two MMAs per K step where the doubled column count fits one MMA (N <= 256): narrow
  // layers issue a third fewer MMA instructions, whose rate limits them.
  // (not with the odd-phase ConvT epilogue, which has its own kernel form)
  g.b2 = (!L.pair && L.prec == VOC_PREC_BF16X3 && 2 * g.N_tile <= 256 && !(L.convT && (g.phase_group & 1))) ? 1 : 0;
  int ac = 32;
  while (ac < (g.b2 ? 2 * g.N_tile : g.N_tile)) ac *= 2;
  g.acc_cols = ac;
  g.n_acc = std::min(voc::kMaxAcc, 512 / ac);
  L.smem = 1024 + (size_t)g.na * g.a_bytes + (size_t)g.nb * g.b_bytes +
           (size_t)g.ns * voc::skip_slot_bytes(L.cw) + kBarrierBytes;
  // Layers whose weights are a large share of L2 (the first transposed conv: 75 MB) take the
  // band job order: a wave covers about half of the column tiles for every row tile of a band
  // instead of every column tile, so each weight byte comes from HBM once.
  const double w_bytes = (double)g.N_total * L.Cp_in * taps_eff * wb;
  g.band = (!g.b_resident && !L.pair && w_bytes >= kBandWeightBytes) ? kBandRows : 0;
  return true;
}

// Resident 2-CTA clusters of a pair layer's launch shape (0: none fit, or the query failed).
int pair_clusters(const Layer &L) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2, attr[0].val.clusterDim.y = 1, attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(voc::kGemmThreads);
  cfg.dynamicSmemBytes = L.smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, voc::conv_gemm_kernel<16, true>, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// plan_gemm, on CTA pairs when `pair` is set and a pair launch of the layer fits the device
bool plan_layer(bool pair, Layer &L, int padding, bool has_skip, std::string &why) {
  L.pair = pair;
  if (!plan_gemm(L, padding, has_skip, why)) return false;
  if (L.pair) {
    L.max_clusters = pair_clusters(L);
    // a resident plan needs at least one cluster per column tile
    if (L.max_clusters < std::max(1, L.g.b_resident ? L.g.n_tiles : 1)) {
      L.pair = false;
      return plan_gemm(L, padding, has_skip, why);
    }
  }
  return true;
}

// Plan a fused residual unit (L.K taps at dilation L.dil, then 1x1, C -> C; ru_gemm_kernel):
// the conv1 geometry of plan_gemm, one column tile (N = Cp <= kRuMaxC), the conv1 result kept
// in a shared H tile of 128 rows x Cp hi/lo pairs, a k-block common to both convolutions,
// one conv1 and one conv2 accumulator in TMEM.
constexpr int kRuMaxC = 192;
// Residual units of up to this many (padded) channels run as one kernel by default.
constexpr int kFuseDefault = kRuMaxC;
// Smallest unit width fused by default with the one-plane precisions (F16W, BF16W).
constexpr int kRuOnePlaneMinC = 129;
// Units of at least this many channels keep half of the H tile at a time.
constexpr int kRuHalfHMinC = 160;
bool plan_ru(Layer &L, int padding, std::string &why) {
  ConvGemmArgs &g = L.g;
  L.Cp_in = L.Cp_out = rup(L.Cout, 16);
  if (L.Cp_out > kRuMaxC) {
    why = "too many channels for the fused residual unit";
    return false;
  }
  if (!g_ru_regs_ok) {
    why = "the fused residual unit's register split does not fit its launch";
    return false;
  }
  g.Cp_in = g.Cp_out = L.Cp_out;
  const int span = L.dil * (L.K - 1);
  const int pad_left = (padding == VOC_PAD_CAUSAL) ? span : span / 2;
  g.taps = L.K;
  g.N_total = g.N_tile = L.Cp_out;
  g.n_tiles = 1;
  g.q_split_tile = 1;
  g.s_rows = 1;
  g.phase_group = 0;
  g.off_min = -pad_left;
  g.shift0_q0 = g.shift0_q1 = 0;
  g.tap_step = L.dil;
  g.rows = rup(voc::kTileM + span + mod8(-pad_left), 8);
  if (g.rows > 256) {
    why = "tap span too wide for one staged tile";
    return false;
  }
  // B2 form (two MMAs per K step) when the doubled column count fits one MMA (bf16x3; the
  // one-plane precisions take two MMAs per K step of N columns)
  g.b2 = (L.prec == VOC_PREC_BF16X3 && 2 * g.N_tile <= 256) ? 1 : 0;
  const int wb = L.prec != VOC_PREC_BF16X3 ? 2 : 4;  // weight bytes per (channel, column)
  L.cw = 16;
  // The widest units keep half of H at a time (conv2 runs in two K halves): the shared memory
  // this frees goes to the weight ring, which conv1's 7 taps x C^2 weights per tile stream
  // through (with the whole H tile the ring holds three stages and conv1 waits on weights).
  L.rx.h_parts = (L.Cp_out >= kRuHalfHMinC && (L.Cp_out / 16) % 2 == 0) ? 2 : 1;
  L.rx.h_bytes = 4 * voc::kTileM * L.Cp_out / L.rx.h_parts;
  int ac = 32;
  while (ac < (g.b2 ? 2 * g.N_tile : g.N_tile)) ac *= 2;
  g.acc_cols = ac;  // acc1 at column 0, acc2 at column ac: 2 ac <= 512
  g.n_acc = 2;
  const int chunkA = g.rows * 16;
  const int avail = kSmemMax - 1024 - kBarrierBytes - L.rx.h_bytes;
  g.KB = 0;
  g.b_resident = 0;
  // Resident weights when every stage of both convolutions fits beside H and two A stages (the
  // narrow units): loaded once per CTA, so no tile streams weights.  The largest such k-block.
  for (int kb = L.Cp_in / L.rx.h_parts; kb >= 16 && !g.KB && g.b2; kb -= 16) {
    if ((L.Cp_in / L.rx.h_parts) % kb || 4 * kb * g.rows > 72 * 1024) continue;
    const int a_bytes = rup(2 * (kb / 8) * chunkA, 1024);
    const int b_bytes = wb * kb * g.N_tile;
    const int nb = (g.taps + 1) * (L.Cp_in / kb);
    if (2 * a_bytes + nb * b_bytes > avail || (4 + 2 * nb + 7) * 8 + 8 > kBarrierBytes) continue;
    g.KB = kb, g.a_bytes = a_bytes, g.b_bytes = b_bytes, g.na = 2, g.nb = nb;
    g.b_resident = 1;
  }
  // Else streamed weights: the largest k-block (a multiple of 16 dividing Cp, weight stage <=
  // kBStageMax, A stage <= 72 KB) that leaves two A stages and at least three weight stages;
  // else two.
  for (int min_nb = 3; min_nb >= 2 && !g.KB; --min_nb)
    for (int kb = L.Cp_in; kb >= 16 && !g.KB; kb -= 16) {
      if ((L.Cp_in / L.rx.h_parts) % kb || wb * kb * g.N_tile > kBStageMax ||
          4 * kb * g.rows > 72 * 1024)
        continue;
      const int a_bytes = rup(2 * (kb / 8) * chunkA, 1024);
      const int b_bytes = wb * kb * g.N_tile;
      const int na = 2;
      const int nb = std::min(8, (avail - na * a_bytes) / b_bytes);
      if (nb < min_nb) continue;
      g.KB = kb, g.a_bytes = a_bytes, g.b_bytes = b_bytes, g.na = na, g.nb = nb;
    }
  if (!g.KB) {
    why = "shared memory plan of the fused residual unit does not fit";
    return false;
  }
  g.ns = 0;  // the residual input is read by the epilogue warps directly
  g.nkb = L.Cp_in / g.KB;
  g.ksplit = 1, g.kb_per_split = g.nkb, g.kb_split = g.nkb;
  g.tap_lo0 = 0, g.tap_hi0 = g.taps, g.tap_lo1 = 0, g.tap_hi1 = g.taps;
  if ((2 * g.na + 2 * g.nb + 7) * 8 + 8 > kBarrierBytes) {
    why = "too many pipeline slots for the barrier block";
    return false;
  }
  L.smem = 1024 + (size_t)g.na * g.a_bytes + (size_t)g.nb * g.b_bytes + L.rx.h_bytes +
           kBarrierBytes;
  L.ru = true;
  return true;
}

// Value of the GEMM weight for column n, input channel ci, tap `tap`.
// ConvT column n -> (phase r, output channel co) in the column order of plan_gemm.
void convT_column(const Layer &L, int n, int &r, int &co) {
  if (L.g.phase_group) {
    const int G = L.g.phase_group;  // phases of one group
    const int gw = G * L.Cp_out;  // columns of one phase group
    const int q = n / gw, nn = n % gw;
    const int cg = nn / (8 * G), rem = nn % (8 * G);
    r = q * G + rem / 8;
    co = cg * 8 + rem % 8;
  } else {
    r = n / L.Cp_out;
    co = n % L.Cp_out;
  }
}

float weight_value(const Layer &L, int padding, const float *w, int n, int ci, int tap) {
  if (ci >= L.Cin) return 0.f;
  if (L.down_s) {
    // input channel ci = 8 * voc::phase_plane(chunk, r) + e holds channel chunk * 8 + e at
    // phase r (row u s + r of the strided conv's input); tap du + 1 (du in {-1, 0, 1}) reads
    // row u + du, i.e. original tap k = du s + r + s / 2 of the k = 2s kernel
    const int sd = L.down_s;
    const int cpc = L.Cin / (8 * sd), r0 = (sd + 1) / 2;
    const int pl = ci / 8, e = ci % 8;
    const int chunk = pl < r0 * cpc ? pl / r0 : (pl - r0 * cpc) / (sd - r0);
    const int r = pl < r0 * cpc ? pl % r0 : r0 + (pl - r0 * cpc) % (sd - r0);
    const int c = chunk * 8 + e;
    const int k = (tap - 1) * sd + r + sd / 2;
    if (n >= L.Cout || c >= L.down_c || k < 0 || k >= 2 * sd) return 0.f;
    return w[((size_t)n * L.down_c + c) * (2 * sd) + k];
  }
  if (!L.convT) {
    if (n >= L.Cout) return 0.f;
    return w[((size_t)n * L.Cin + ci) * L.K + tap];
  }
  const int s = L.stride;
  int r, co;
  convT_column(L, n, r, co);
  if (co >= L.Cout) return 0.f;
  const int p = (padding == VOC_PAD_CAUSAL) ? 0 : s / 2;
  if (L.g.taps == 3) {  // stride 2: tap u reads row t + u - 1, output row 2t + r
    const int k = r + p - s * (tap - 1);
    return (k < 0 || k >= 2 * s) ? 0.f : w[((size_t)ci * L.Cout + co) * (2 * s) + k];
  }
  const int k = (r + p) % s + tap * s;  // tap 0: k0 at row t+q, tap 1: k0+s at row t+q-1
  return w[((size_t)ci * L.Cout + co) * (2 * s) + k];
}

// Weight tiles as the kernel stages them: [tile][tap][kb][hi|lo][chunk][n][8] (b2:
// [tile][tap][kb][chunk][hi|lo][n][8]) with tiles of `pw` columns (N_tile, or N_tile / 2 for
// the CTA pair: CTA r of a pair stages tile 2 nt + r).
std::vector<uint16_t> pack_weights(const Layer &L, int padding, const float *w) {
  const ConvGemmArgs &g = L.g;
  const int pw = L.pair ? g.N_tile / 2 : g.N_tile;
  const int n_pt = g.N_total / pw;
  const size_t tile = (size_t)(L.prec != VOC_PREC_BF16X3 ? 1 : 2) * g.KB * pw;
  std::vector<uint16_t> out((size_t)n_pt * g.taps * g.nkb * tile);
  for (int nt = 0; nt < n_pt; ++nt)
    for (int tap = 0; tap < g.taps; ++tap)
      for (int kb = 0; kb < g.nkb; ++kb) {
        uint16_t *base = out.data() + (((size_t)nt * g.taps + tap) * g.nkb + kb) * tile;
        for (int c = 0; c < g.KB / 8; ++c)
          for (int n = 0; n < pw; ++n)
            for (int e = 0; e < 8; ++e) {
              const float v = weight_value(L, padding, w, nt * pw + n, kb * g.KB + c * 8 + e, tap);
              if (L.prec != VOC_PREC_BF16X3) {  // one plane of f16 / bf16 weights (nearest even)
                base[((size_t)c * pw + n) * 8 + e] = L.prec == VOC_PREC_F16W
                                                         ? __half_as_ushort(__float2half_rn(v))
                                                         : f2bf(v);
                continue;
              }
              const uint16_t hi = f2bf(v);
              const uint16_t lo = f2bf(v - bf2f(hi));
              if (g.b2) {
                base[(((size_t)c * 2 + 0) * pw + n) * 8 + e] = hi;
                base[(((size_t)c * 2 + 1) * pw + n) * 8 + e] = lo;
              } else {
                const size_t idx = ((size_t)c * pw + n) * 8 + e;
                base[idx] = hi;
                base[(size_t)g.KB * pw + idx] = lo;
              }
            }
      }
  return out;
}

template <class T>
voc_status upload(vocoder *ctx, std::vector<void *> &allocs, const std::vector<T> &host, T **dev) {
  cudaError_t e = dev_alloc(reinterpret_cast<void **>(dev), host.size() * sizeof(T));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaMalloc");
  allocs.push_back(*dev);
  e = cudaMemcpy(*dev, host.data(), host.size() * sizeof(T), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaMemcpy");
  return VOC_OK;
}

// Per-channel coefficients of one Snake: y = x + sin^2(a x) * ib.  Snake: a = alpha,
// ib = 1 / (alpha + 1e-9); SnakeBeta (log-scale parameters, p = [log alpha | log beta]):
// a = e^alpha, ib = 1 / (e^beta + 1e-9); formed in double, rounded once to fp32.  Empty:
// no Snake.
struct SnakeCoef {
  std::vector<float> a, ib;
};

SnakeCoef snake_coef(const float *p, int C, int kind) {
  SnakeCoef s;
  if (!p) return s;
  s.a.resize(C);
  s.ib.resize(C);
  for (int c = 0; c < C; ++c) {
    if (kind == VOC_SNAKE_BETA) {
      s.a[c] = static_cast<float>(std::exp(static_cast<double>(p[c])));
      s.ib[c] = static_cast<float>(1.0 / (std::exp(static_cast<double>(p[C + c])) + 1e-9));
    } else {
      s.a[c] = p[c];
      s.ib[c] = static_cast<float>(1.0 / (static_cast<double>(p[c]) + 1e-9));
    }
  }
  return s;
}

// Per-column epilogue vectors of a layer: bias, and the Snake of the layer that
// consumes this output (empty coefficients: none).
voc_status upload_columns(vocoder *ctx, std::vector<void *> &allocs, Layer &L, int padding,
                          const float *bias, const SnakeCoef &sn) {
  const int N = L.g.N_total;
  const bool has_snake = !sn.a.empty();
  std::vector<float> b(N, 0.f), a(N, 1.f), ib(N, 0.f);
  for (int n = 0; n < N; ++n) {
    int r = 0, co = n;
    if (L.convT) convT_column(L, n, r, co);
    if (co < L.Cout) {
      if (bias) b[n] = bias[co];
      if (has_snake) {
        a[n] = sn.a[co];
        ib[n] = sn.ib[co];
      }
    }
  }
  voc_status st = upload(ctx, allocs, b, &L.bias_dev);
  if (st != VOC_OK) return st;
  if (has_snake) {
    st = upload(ctx, allocs, a, &L.alpha_dev);
    if (st != VOC_OK) return st;
    st = upload(ctx, allocs, ib, &L.invb_dev);
    if (st != VOC_OK) return st;
  }
  return VOC_OK;
}

voc_status upload_layer(vocoder *ctx, std::vector<void *> &allocs, Layer &L, int padding,
                        const float *w, const float *bias, const SnakeCoef &alpha) {
  std::vector<uint16_t> packed = pack_weights(L, padding, w);
  uint16_t *wd = nullptr;
  voc_status st = upload(ctx, allocs, packed, &wd);
  if (st != VOC_OK) return st;
  L.w_dev = reinterpret_cast<uint8_t *>(wd);
  return upload_columns(ctx, allocs, L, padding, bias, alpha);
}

// Weights of a fused residual unit: conv1 (L.K taps) and conv2 (1x1) packed with the same
// k-block and column tile; epilogue 1 columns from (b1, alpha2), epilogue 2 from (b2, next).
voc_status upload_ru(vocoder *ctx, std::vector<void *> &allocs, Layer &L, int padding,
                     const float *w1, const float *b1, const SnakeCoef &a2, const float *w2,
                     const float *b2, const SnakeCoef &next_alpha) {
  voc_status st = upload_layer(ctx, allocs, L, padding, w1, b2, next_alpha);
  if (st != VOC_OK) return st;
  Layer L2 = L;
  L2.K = 1;
  L2.g.taps = 1;
  std::vector<uint16_t> packed = pack_weights(L2, padding, w2);
  uint16_t *wd = nullptr;
  if ((st = upload(ctx, allocs, packed, &wd)) != VOC_OK) return st;
  L.rx.wB2 = reinterpret_cast<const uint8_t *>(wd);
  Layer Lh = L;
  if ((st = upload_columns(ctx, allocs, Lh, padding, b1, a2)) != VOC_OK) return st;
  L.rx.bias_h = Lh.bias_dev, L.rx.alpha_h = Lh.alpha_dev, L.rx.invb_h = Lh.invb_dev;
  return VOC_OK;
}

bool check_desc(const voc_desc *d, std::string &why) {
  if (!d) return why = "desc is NULL", false;
  if (d->abi_version != VOC_ABI_VERSION)
    return why = "abi_version " + std::to_string(d->abi_version) + " != " +
                 std::to_string(VOC_ABI_VERSION),
           false;
  if (d->latent_channels < 1 || d->latent_channels > 8192) return why = "latent_channels", false;
  if (d->channels0 < 1 || d->channels0 > 8192) return why = "channels0", false;
  for (int k : {d->in_kernel, d->res_kernel, d->out_kernel})
    if (k < 1 || k > 15 || k % 2 == 0) return why = "kernel sizes must be odd in [1, 15]", false;
  if (d->n_stages < 1 || d->n_stages > 8) return why = "n_stages", false;
  if (!d->strides || !d->widths) return why = "strides / widths NULL", false;
  if (d->n_dilations < 1 || d->n_dilations > 4 || !d->dilations) return why = "dilations", false;
  if (d->out_channels != 1) return why = "out_channels must be 1", false;
  if (d->in_proj_channels < 0 || d->in_proj_channels > 8192) return why = "in_proj_channels", false;
  if (d->padding != VOC_PAD_SYMMETRIC && d->padding != VOC_PAD_CAUSAL) return why = "padding", false;
  if (d->precision != VOC_PREC_BF16X3 && d->precision != VOC_PREC_F16W &&
      d->precision != VOC_PREC_BF16W)
    return why = "precision", false;
  if (d->precision != VOC_PREC_BF16X3 && d->cta_pair > 0)
    return why = "cta_pair is available with VOC_PREC_BF16X3 only", false;
  if (d->cta_pair < -1 || d->cta_pair > 1) return why = "cta_pair must be -1, 0 or 1", false;
  if (d->snake != VOC_SNAKE && d->snake != VOC_SNAKE_BETA) return why = "snake", false;
  for (int i = 0; i < d->n_stages; ++i) {
    if (d->strides[i] < 1 || d->strides[i] > 16) return why = "stride out of [1, 16]", false;
    if (d->padding == VOC_PAD_SYMMETRIC && d->strides[i] % 2)
      return why = "odd stride needs VOC_PAD_CAUSAL (symmetric crop s/2)", false;
    if (d->widths[i] < 1 || d->widths[i] > 8192) return why = "width out of range", false;
  }
  for (int j = 0; j < d->n_dilations; ++j)
    if (d->dilations[j] < 1 || d->dilations[j] * (d->res_kernel - 1) > 120)
      return why = "dilation * (res_kernel - 1) must be in [1, 120]", false;
  if (d->in_kernel - 1 > 120 || d->out_kernel - 1 > 120) return why = "kernel too wide", false;
  return true;
}

int param_count(const voc_desc *d) {
  return (d->in_proj_channels > 0 ? 2 : 0) + 2 + d->n_stages * (3 + 6 * d->n_dilations) + 3;
}

// kind of every canonical parameter: 'w' weight, 'b' bias, 'a' Snake alpha
std::string param_kinds(const voc_desc *d) {
  std::string k = d->in_proj_channels > 0 ? "wbwb" : "wb";
  for (int i = 0; i < d->n_stages; ++i) {
    k += "awb";
    for (int j = 0; j < d->n_dilations; ++j) k += "awbawb";
  }
  return k + "awb";
}

// level lengths L_lv = T * prod(strides[0..lv-1])
long long level_len(const vocoder *ctx, int lv, int T) {
  long long L = T;
  for (int i = 0; i < lv; ++i) L *= ctx->strides[i];
  return L;
}

size_t buf_bytes(const vocoder *ctx, int B, int T) {
  size_t m = (size_t)B * (size_t)pitch8(T) *
             std::max({ctx->Cp_lat, rup(ctx->desc.channels0, 16), rup(ctx->desc.in_proj_channels, 16)});
  for (int i = 0; i < ctx->desc.n_stages; ++i)
    m = std::max(m, (size_t)B * (size_t)pitch8(level_len(ctx, i + 1, T)) *
                        (size_t)rup(ctx->widths[i], 16));
  return rupz(m * 4, 256);
}

// A operand: bf16 hi/lo chunk-major [B][2*Cp/8][L][8] with planes of L rows (L a multiple
// of 8), read in boxes of `rows` time rows x `kchunks` chunks of both planes.  The rows of
// a plane are addressed in groups of 8 (128 contiguous bytes): a box whose innermost extent
// is a single 16-byte row caps TMA reads near 4 TB/s on GB300, 128-byte rows reach the
// HBM rate.  Groups outside [0, L/8) read as zeros.
voc_status encode_map(vocoder *ctx, CUtensorMap *map, const void *base, int Cp, long long L, int B,
                      int rows, int kchunks) {
  auto enc = encode_fn();
  if (!enc) return fail(ctx, VOC_CUDA_ERROR, "cuTensorMapEncodeTiled entry point unavailable");
  if (L % 8 || rows % 8) return fail(ctx, VOC_CUDA_ERROR, "tensor map: rows not in groups of 8");
  // [B][hi|lo][Cp/8][L/8][8 rows x 8 channels]: one box covers `kchunks` chunks of both planes
  const cuuint64_t dims[5] = {64u, (cuuint64_t)(L / 8), (cuuint64_t)(Cp / 8), 2u, (cuuint64_t)B};
  const cuuint64_t strides[4] = {128u, 16u * (cuuint64_t)L, 16u * (cuuint64_t)L * (Cp / 8),
                                 16u * (cuuint64_t)L * (2 * Cp / 8)};
  const cuuint32_t box[5] = {64u, (cuuint32_t)(rows / 8), (cuuint32_t)kchunks, 2u, 1u};
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ctx, VOC_CUDA_ERROR, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
  return VOC_OK;
}

// Residual (skip) input of an epilogue: fp32 chunk-major [B][Cp/4][L][4] (L a multiple of
// 8), read in boxes of 128 rows x cw/4 chunks, rows addressed in groups of 8 (see
// encode_map).
voc_status encode_skip_map(vocoder *ctx, CUtensorMap *map, const void *base, int Cp, long long L,
                           int B, int cw) {
  auto enc = encode_fn();
  if (!enc) return fail(ctx, VOC_CUDA_ERROR, "cuTensorMapEncodeTiled entry point unavailable");
  if (L % 8) return fail(ctx, VOC_CUDA_ERROR, "residual tensor map: rows not in groups of 8");
  const cuuint64_t dims[4] = {32u, (cuuint64_t)(L / 8), (cuuint64_t)(Cp / 4), (cuuint64_t)B};
  const cuuint64_t strides[3] = {128u, 16u * (cuuint64_t)L, 16u * (cuuint64_t)L * (Cp / 4)};
  const cuuint32_t box[4] = {32u, (cuuint32_t)(voc::kTileM / 8), (cuuint32_t)(cw / 4), 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ctx, VOC_CUDA_ERROR, "cuTensorMapEncodeTiled (residual) failed (" + std::to_string((int)r) + ")");
  return VOC_OK;
}

// Input row offset of a launch: the A tensor map addresses rows in groups of 8, so the MMA
// row shift grows by the offset of the first staged row within its group.
void set_in_row0(const Layer &L, ConvGemmArgs &a, int in_row0) {
  a.in_row0 = in_row0;
  const int extra = mod8(in_row0 + L.g.off_min);
  a.shift0_q0 = L.g.shift0_q0 + extra;
  a.shift0_q1 = L.g.shift0_q1 + extra;
}

// Launch arguments of a layer whose GEMM has L_in rows per item.
void gemm_args_rows(const vocoder *ctx, const Layer &L, int B, long long L_in, void *const *bufs,
                    size_t bbytes, ConvGemmArgs &a) {
  a = L.g;
  a.B = B;
  a.L_in = static_cast<int>(L_in);
  const int kM = L.pair ? 2 * voc::kTileM : voc::kTileM;  // rows of one tile job
  a.m_tiles = static_cast<int>((L_in + kM - 1) / kM);
  a.wB = L.w_dev;
  a.bias = L.bias_dev;
  a.alpha = L.alpha_dev;
  a.invb = L.invb_dev;
  a.skip = L.skip_buf >= 0 ? static_cast<const float *>(bufs[L.skip_buf]) : nullptr;
  a.out_f32 = L.f32_buf >= 0 ? static_cast<float *>(bufs[L.f32_buf]) : nullptr;
  a.out_hl = L.hl_buf >= 0 ? static_cast<__nv_bfloat16 *>(bufs[L.hl_buf]) : nullptr;
  a.flags = L.epi_flags;
  set_in_row0(L, a, 0);
  a.f32_row0 = a.hl_row0 = 0;
  a.f32_L = a.hl_L = static_cast<int>(pitch8(L_in * L.g.s_rows));
  a.rows_valid = static_cast<int>(L_in * L.g.s_rows);
  a.rows_pad = a.f32_L;  // zero rows up to the plane's 8-row boundary
  a.timeout = ctx->wait_budget;
  a.err = ctx->err_dev;
  a.f32_elems = L.f32_buf >= 0 ? (long long)(bbytes / 4) : 0;
  a.hl_elems = L.hl_buf >= 0 ? (long long)(bbytes / 2) : 0;
  a.w_bytes = (long long)L.g.n_tiles * (L.pair ? 2 : 1) * L.g.taps * L.g.nkb * L.g.b_bytes;
  a.smem_bytes = static_cast<int>(L.smem);
  a.L_a = static_cast<int>(pitch8(L_in));
  a.chunks_a = 2 * L.Cp_in / 8;
  a.chunks_s = L.Cp_out / 4;
  a.dbg = ctx->err_dev + 4;
}

void gemm_launch_args(const vocoder *ctx, const Layer &L, int B, int T, void *const *bufs,
                      size_t bbytes, ConvGemmArgs &a) {
  gemm_args_rows(ctx, L, B, level_len(ctx, L.level, T), bufs, bbytes, a);
}

#ifdef VOC_CHECKS
// Self-checking build: wait for every launch and report the first failed check.
voc_status check_launch(vocoder *ctx, const std::string &name, cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, ("after " + name).c_str());
  int w[8] = {0};
  cudaMemcpy(w, ctx->err_dev, sizeof(w), cudaMemcpyDeviceToHost);
  if (w[0] || w[4]) {
    char buf[256];
    snprintf(buf, sizeof buf, "%s: a kernel gave up a bounded wait or failed a check: error word %d, check %d (%d, %d, %d)",
             name.c_str(), w[0], w[4], w[5], w[6], w[7]);
    cudaMemset(ctx->err_dev, 0, 8 * sizeof(int));  // reported: the next launch starts clean
    return fail(ctx, VOC_DEVICE_TIMEOUT, buf);
  }
  return VOC_OK;
}
#endif

// Partial sums per item of the head folded into layer L (L_f output rows).
double head_part_floats(const vocoder *ctx, const Layer &L, long long Lf) {
  const long long slices = 4 * ((Lf + voc::kTileM - 1) / voc::kTileM);
  return (double)slices * (L.Cp_out / 16) * (32 + voc::kHeadFoldMaxK - 1);
}

// Cost of one launch of layer L for the per-kernel rooflines.  flops: 2 per multiply-add of
// the method (a transposed conv without its zero-stuffed taps).  alg: the algorithmic HBM
// bytes -- every input of the layer read once and every output written once, as fp32 values
// of the real channels (a k-tap conv 4 Cin + 4 Cout per row; a 1x1 conv with the residual add
// also reads the skip, 4 Cout more; a transposed conv 4 Cin per input row and 4 Cout per output
// sample; a fused residual unit reads x once, for conv1 and for the skip, and writes y).  A
// launch carrying the folded output head (`folded`) writes no activations: its result leaves
// through the head, whose audio is counted on the finishing launch.  impl: the bytes the
// implementation moves by its own count -- padded channels, the weight stream, the fp32
// stream and the hi/lo operand copies of every output.
void layer_cost(const vocoder *ctx, const Layer &L, int B, int T, double &flops, double &alg,
                double &impl, bool folded = false) {
  const double L_in = (double)level_len(ctx, L.level, T);
  const double L_out = L_in * (L.convT ? L.stride : 1);
  flops = L.convT ? 4.0 * L.Cin * L.Cout * B * L_out : 2.0 * L.Cin * L.Cout * L.K * B * L_in;
  if (L.ru) flops = 2.0 * L.Cin * L.Cout * (L.K + 1) * B * L_in;
  alg = 4.0 * L.Cin * B * L_in;
  if (L.skip_buf >= 0 && !L.ru) alg += 4.0 * L.Cout * B * L_out;
  if (!folded) alg += 4.0 * L.Cout * B * L_out;
  const ConvGemmArgs &g = L.g;
  double by = 4.0 * B * L_in * L.Cp_in +
              (double)g.n_tiles * (L.pair ? 2 : 1) * (g.taps + (L.ru ? 1 : 0)) * g.nkb * g.b_bytes;
  const double out_elems = (double)B * L_out * L.Cp_out;
  if (L.skip_buf >= 0) by += 4.0 * out_elems;
  if (L.f32_buf >= 0 && !folded) by += 4.0 * out_elems;
  if (L.hl_buf >= 0) by += 4.0 * out_elems;
  if (folded) {  // the head's partial sums instead of the activations, and its products
    by += 4.0 * B * head_part_floats(ctx, L, (long long)L_out);
    flops += 2.0 * ctx->head.C * ctx->head.K * B * L_out;
  }
  impl = by;
}

// One launch of the single-CTA conv kernel of precision PREC in the form the layer needs.
template <int PREC>
cudaError_t launch_conv(const Layer &L, const ConvGemmArgs &a, int grid, const CUtensorMap &map,
                        const CUtensorMap &smap, cudaStream_t stream) {
  const dim3 g(grid), blk(voc::kGemmThreads);
  constexpr bool kB2 = PREC == voc::kPrecBf16x3;  // the B2 form exists for bf16x3 only
  if (a.head_part) {  // the output head folded into the epilogue
    if (kB2 && L.g.b2)
      return launch_pdl(voc::conv_gemm_kernel<16, false, kB2, false, PREC, false, true>, g, blk,
                        L.smem, stream, map, smap, a);
    return launch_pdl(voc::conv_gemm_kernel<16, false, false, false, PREC, false, true>, g, blk,
                      L.smem, stream, map, smap, a);
  }
  if (a.split_s > 1 || L.down_s || a.ksplit > 1) {  // encoder forms: phase split, tap windows, split k
    if (kB2 && L.g.b2)
      return launch_pdl(voc::conv_gemm_kernel<16, false, kB2, false, PREC, true>, g, blk, L.smem,
                        stream, map, smap, a);
    return launch_pdl(voc::conv_gemm_kernel<16, false, false, false, PREC, true>, g, blk, L.smem,
                      stream, map, smap, a);
  }
  if (L.convT && (L.g.phase_group & 1))
    return launch_pdl(voc::conv_gemm_kernel<16, false, false, true, PREC>, g, blk, L.smem, stream,
                      map, smap, a);
  if (kB2 && L.g.b2)
    return launch_pdl(voc::conv_gemm_kernel<16, false, kB2, false, PREC>, g, blk, L.smem, stream,
                      map, smap, a);
  return launch_pdl(voc::conv_gemm_kernel<16, false, false, false, PREC>, g, blk, L.smem, stream,
                    map, smap, a);
}

// skip_L: rows of a plane of a fused residual unit's fp32 residual input (< 0: the output
// planes', a.f32_L); skip_elems its floats (the self-checking build's bound).
voc_status launch_gemm(vocoder *ctx, const Layer &L, const CUtensorMap &map,
                       const CUtensorMap &smap, const ConvGemmArgs &a, cudaStream_t stream,
                       long long skip_L = -1, long long skip_elems = -1) {
  // jobs: tiles, times the k ranges of a split-k layer (encoder forms)
  const long long tiles = (long long)a.B * a.m_tiles * a.n_tiles * std::max(1, a.ksplit);
  // Persistent grid: one CTA (or cluster) per unit, at most one per job.  With resident
  // weights every CTA must keep one column tile, so its job stride is a multiple of n_tiles.
  auto persistent = [&](long long units) {
    if (tiles <= units) return tiles;
    return a.b_resident ? units - units % a.n_tiles : units;
  };
  if ((a.split_s > 1 || L.down_s || a.ksplit > 1) && (L.pair || L.convT || L.ru))
    return fail(ctx, VOC_UNSUPPORTED, L.name + ": the encoder forms need a plain conv kernel");
  if (L.pair) {  // persistent grid of 2-CTA clusters, at most as many as can be resident
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2, attr[0].val.clusterDim.y = 1, attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * static_cast<unsigned>(persistent(L.max_clusters)));
    cfg.blockDim = dim3(voc::kGemmThreads);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, voc::conv_gemm_kernel<16, true>, map, smap, a);
    if (e != cudaSuccess) return cuda_fail(ctx, e, ("launch " + L.name).c_str());
    return VOC_OK;
  }
  const int grid = static_cast<int>(L.ru ? std::min<long long>(tiles, ctx->num_sms)
                                         : persistent(ctx->num_sms));
  cudaError_t e;
  if (L.ru) {
    voc::RuExtra rx = L.rx;
    rx.skip_L = static_cast<int>(skip_L >= 0 ? skip_L : a.f32_L);
    rx.skip_elems = skip_elems >= 0 ? skip_elems : a.f32_elems;
    const dim3 g(grid), blk(voc::kRuThreads);
    if (L.prec == VOC_PREC_F16W)  // one weight plane: three-MMA layout, streamed weights
      e = a.head_part
              ? launch_pdl(voc::ru_gemm_kernel<false, true, false, voc::kPrecF16w>, g, blk, L.smem, stream, map, a, rx)
              : launch_pdl(voc::ru_gemm_kernel<false, false, false, voc::kPrecF16w>, g, blk, L.smem, stream, map, a, rx);
    else if (L.prec == VOC_PREC_BF16W)
      e = a.head_part
              ? launch_pdl(voc::ru_gemm_kernel<false, true, false, voc::kPrecBf16w>, g, blk, L.smem, stream, map, a, rx)
              : launch_pdl(voc::ru_gemm_kernel<false, false, false, voc::kPrecBf16w>, g, blk, L.smem, stream, map, a, rx);
    else if (L.g.b_resident)  // (resident plans are narrow: B2 form)
      e = a.head_part
              ? launch_pdl(voc::ru_gemm_kernel<true, true, true>, g, blk, L.smem, stream, map, a, rx)
              : launch_pdl(voc::ru_gemm_kernel<true, false, true>, g, blk, L.smem, stream, map, a, rx);
    else if (a.head_part)
      e = L.g.b2 ? launch_pdl(voc::ru_gemm_kernel<true, true>, g, blk, L.smem, stream, map, a, rx)
                 : launch_pdl(voc::ru_gemm_kernel<false, true>, g, blk, L.smem, stream, map, a, rx);
    else
      e = L.g.b2 ? launch_pdl(voc::ru_gemm_kernel<true, false>, g, blk, L.smem, stream, map, a, rx)
                 : launch_pdl(voc::ru_gemm_kernel<false, false>, g, blk, L.smem, stream, map, a, rx);
  } else if (L.prec == VOC_PREC_F16W) {
    e = launch_conv<voc::kPrecF16w>(L, a, grid, map, smap, stream);
  } else if (L.prec == VOC_PREC_BF16W) {
    e = launch_conv<voc::kPrecBf16w>(L, a, grid, map, smap, stream);
  } else {
    e = launch_conv<voc::kPrecBf16x3>(L, a, grid, map, smap, stream);
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, ("launch " + L.name).c_str());
  return VOC_OK;
}

// y: fp32 chunk-major with planes of Ly rows, sample 0 at row in_row0 (streaming keeps the
// head's left context in the rows before it); a plain decode passes in_row0 = 0, Ly = L.
voc_status launch_out_head(vocoder *ctx, const OutHead &h, const float *y, int B, long long L,
                           float *audio, cudaStream_t stream, int in_row0 = 0, long long Ly = -1) {
  if (Ly < 0) Ly = L;
  if (h.K == 7 && h.w4_dev) {
    const long long threads = (L + kHeadTpt - 1) / kHeadTpt;
    dim3 grid(static_cast<unsigned>((threads + 255) / 256), static_cast<unsigned>(B));
    cudaError_t e = launch_pdl(voc::out_head_reg_kernel<7, kHeadTpt>, grid, dim3(256), 0, stream,
                               y, static_cast<int>(L), h.Cp, h.pad_left,
                               reinterpret_cast<const float4 *>(h.w4_dev),
                               static_cast<const float *>(h.b_dev), audio, in_row0, Ly);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "launch out_head");
    return VOC_OK;
  }
  const size_t smem = ((size_t)(kHeadTile + h.K - 1) * h.Cp + (size_t)h.Cp * h.K) * 4;
  dim3 grid(static_cast<unsigned>((L + kHeadTile - 1) / kHeadTile), static_cast<unsigned>(B));
  cudaError_t e = launch_pdl(voc::out_head_kernel<kHeadTile>, grid, dim3(kHeadTile), smem, stream,
                             y, static_cast<int>(L), h.Cp, h.K, h.pad_left,
                             static_cast<const float *>(h.w_dev), static_cast<const float *>(h.b_dev),
                             audio, in_row0, Ly);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "launch out_head");
  return VOC_OK;
}

// Lp < 0: planes of rup8(T) rows, rows T.. zero-filled; else planes of Lp rows from row0
// (streaming: no padding rows are written).
voc_status launch_prep(vocoder *ctx, const float *x, int B, int C, int T, int Cp, const float *alpha,
                       const float *invb, __nv_bfloat16 *hl, cudaStream_t stream, int row0 = 0,
                       long long Lp = -1) {
  const int T_pad = Lp < 0 ? rup(T, 8) : T;
  dim3 grid((T_pad + 255) / 256, Cp / 8, B);
  cudaError_t e = launch_pdl(voc::prep_hl_kernel, grid, dim3(256), 0, stream, x, C, T, T_pad, Cp,
                             alpha, invb, hl, row0, Lp < 0 ? (long long)T_pad : Lp,
                             ctx->prec == VOC_PREC_F16W ? 1 : 0);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "launch prep");
  return VOC_OK;
}

}  // namespace

// =================================================================== C ABI
VOC_API int vocoder_abi_version(void) { return VOC_ABI_VERSION; }

VOC_API int vocoder_param_count(const voc_desc *desc) {
  std::string why;
  if (!check_desc(desc, why)) return -1;
  return param_count(desc);
}

VOC_API voc_status vocoder_param_shape(const voc_desc *d, int index, int dims[3], int *ndim) {
  std::string why;
  if (!check_desc(d, why)) return fail(nullptr, VOC_INVALID_ARG, why);
  if (!dims || !ndim) return fail(nullptr, VOC_INVALID_ARG, "dims / ndim NULL");
  const int n = param_count(d);
  if (index < 0 || index >= n) return fail(nullptr, VOC_INVALID_ARG, "index out of range");
  auto set = [&](int nd, int a, int b = 0, int c = 0) {
    *ndim = nd;
    dims[0] = a, dims[1] = b, dims[2] = c;
    return VOC_OK;
  };
  int c_in = d->latent_channels;
  if (d->in_proj_channels > 0) {  // in_proj.w [P][C_lat][1], in_proj.b [P]
    if (index == 0) return set(3, d->in_proj_channels, d->latent_channels, 1);
    if (index == 1) return set(1, d->in_proj_channels);
    index -= 2;
    c_in = d->in_proj_channels;
  }
  if (index == 0) return set(3, d->channels0, c_in, d->in_kernel);
  if (index == 1) return set(1, d->channels0);
  int i = index - 2;
  int C = d->channels0;
  const int per_stage = 3 + 6 * d->n_dilations;
  auto snake = [&](int c) { return d->snake == VOC_SNAKE_BETA ? set(2, 2, c) : set(1, c); };
  for (int s = 0; s < d->n_stages; ++s) {
    const int Co = d->widths[s];
    if (i < per_stage) {
      if (i == 0) return snake(C);
      if (i == 1) return set(3, C, Co, 2 * d->strides[s]);
      if (i == 2) return set(1, Co);
      const int j = (i - 3) % 6;
      if (j == 1) return set(3, Co, Co, d->res_kernel);
      if (j == 4) return set(3, Co, Co, 1);
      if (j == 0 || j == 3) return snake(Co);
      return set(1, Co);
    }
    i -= per_stage;
    C = Co;
  }
  if (i == 0) return snake(C);
  if (i == 1) return set(3, 1, C, d->out_kernel);
  return set(1, 1);
}

VOC_API voc_status vocoder_fold_weight_norm(const float *g, const float *v, int dim0,
                                            long long rest, float *w) {
  if (!g || !v || !w || dim0 <= 0 || rest <= 0)
    return fail(nullptr, VOC_INVALID_ARG, "fold: NULL pointer or non-positive size");
  for (int i = 0; i < dim0; ++i) {
    const float *row = v + (size_t)i * rest;
    double ss = 0.0;
    for (long long j = 0; j < rest; ++j) ss += (double)row[j] * (double)row[j];
    const double nrm = std::sqrt(ss);
    if (!(nrm > 0.0) || !std::isfinite(nrm))
      return fail(nullptr, VOC_INVALID_ARG, "fold: row " + std::to_string(i) + " has zero or non-finite norm");
    const double sc = (double)g[i] / nrm;
    for (long long j = 0; j < rest; ++j) {
      const float x = static_cast<float>(sc * (double)row[j]);
      if (!std::isfinite(x)) return fail(nullptr, VOC_INVALID_ARG, "fold: non-finite result");
      w[(size_t)i * rest + j] = x;
    }
  }
  return VOC_OK;
}

VOC_API void vocoder_destroy(vocoder *ctx) {
  if (!ctx) return;
  for (void *p : ctx->allocs) dev_free(p);
  for (cudaEvent_t e : ctx->events) cudaEventDestroy(e);
  delete ctx;
}

// ------------------------------------------------------------------ no-allocation workspace
// The workspace of vocoder_decode_static: one array per device, in the library's module.
static __device__ __align__(256) uint8_t g_static_ws[VOC_STATIC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ws_addr[kMaxDevices] = {};  // device address of g_static_ws, per device

// Set-up of the no-allocation decode on the current device (vocoder_create calls it with the
// context's device current): look up the device address of g_static_ws once per device.  Host
// code may not take &g_static_ws itself -- on the host that name is a stand-in, not a device
// address.
voc_status static_ws_setup(vocoder *ctx) {
  if (ctx->device < 0 || ctx->device >= kMaxDevices) return VOC_OK;  // decode_static refuses
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ws_addr[ctx->device]) return VOC_OK;
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGetSymbolAddress (no-allocation workspace)");
  g_static_ws_addr[ctx->device] = p;
  return VOC_OK;
}

void *static_ws_addr(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_mu);
  return g_static_ws_addr[device];
}

// The caller's cancel flag is set: nothing may be enqueued.
bool cancelled(const vocoder *ctx) { return ctx->cancel && *ctx->cancel != 0; }
}  // namespace

VOC_API voc_status vocoder_create(const voc_desc *desc, const float *const *params, int n_params,
                                  vocoder **out) {
  if (!out) return fail(nullptr, VOC_INVALID_ARG, "out is NULL");
  *out = nullptr;
  std::string why;
  if (!check_desc(desc, why)) return fail(nullptr, VOC_INVALID_ARG, "desc: " + why);
  if (!params) return fail(nullptr, VOC_INVALID_ARG, "params is NULL");
  if (n_params != param_count(desc))
    return fail(nullptr, VOC_INVALID_ARG, "n_params " + std::to_string(n_params) + " != " +
                                              std::to_string(param_count(desc)));
  // every entry but the biases is required; all values must be finite; alpha > 0
  const std::string kinds = param_kinds(desc);
  for (int i = 0; i < n_params; ++i) {
    if (!params[i]) {
      if (kinds[i] == 'b') continue;
      return fail(nullptr, VOC_INVALID_ARG, "params[" + std::to_string(i) + "] is NULL");
    }
    int dims[3], nd;
    vocoder_param_shape(desc, i, dims, &nd);
    size_t n = 1;
    for (int k = 0; k < nd; ++k) n *= dims[k];
    for (size_t k = 0; k < n; ++k) {
      const float x = params[i][k];
      if (!std::isfinite(x))
        return fail(nullptr, VOC_INVALID_ARG, "params[" + std::to_string(i) + "] not finite");
      if (kinds[i] == 'a' && desc->snake == VOC_SNAKE && !(x > 0.f))
        return fail(nullptr, VOC_INVALID_ARG, "Snake alpha must be positive");
      if (kinds[i] == 'a' && desc->snake == VOC_SNAKE_BETA && !(std::fabs(x) <= 80.f))
        return fail(nullptr, VOC_INVALID_ARG, "SnakeBeta log alpha / log beta must be in [-80, 80]");
    }
  }
  if (!set_kernel_attrs(why)) return fail(nullptr, VOC_CUDA_ERROR, why);

  vocoder *ctx = new vocoder();
  ctx->desc = *desc;
  ctx->strides.assign(desc->strides, desc->strides + desc->n_stages);
  ctx->widths.assign(desc->widths, desc->widths + desc->n_stages);
  ctx->dils.assign(desc->dilations, desc->dilations + desc->n_dilations);
  ctx->desc.strides = ctx->strides.data();
  ctx->desc.widths = ctx->widths.data();
  ctx->desc.dilations = ctx->dils.data();
  for (int s : ctx->strides) ctx->hop *= s;
  ctx->Cp_lat = rup(desc->latent_channels, 16);
  ctx->fuse_max_c = desc->fuse_max_channels == 0 ? kFuseDefault
                    : (desc->fuse_max_channels < 0 ? 0 : desc->fuse_max_channels);
  ctx->use_pair = desc->cta_pair > 0;
  ctx->prec = desc->precision;
  // The one-plane precisions fuse by default only the units wider than kRuOnePlaneMinC (their
  // narrower fused units ran slower than conv1 + conv2: C = 96 0.41 vs 0.36 ms, C = 48 1.04 vs
  // 1.02 ms; C = 192 0.37 vs 0.40 ms).  An explicit fuse_max_channels fuses every unit up to it.
  if (ctx->prec != VOC_PREC_BF16X3 && desc->fuse_max_channels == 0) ctx->fuse_min_c = kRuOnePlaneMinC;
  auto bail = [&](voc_status st) {
    g_err = ctx->err;
    vocoder_destroy(ctx);
    return st;
  };
  voc_status st0;
  cudaError_t e = cudaGetDevice(&ctx->device);
  if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "cudaGetDevice"));
  e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
  if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "cudaDeviceGetAttribute"));
  int cc_major = 0, cc_minor = 0;
  cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, ctx->device);
  cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, ctx->device);
  if (cc_major != 10 || cc_minor != 3)
    return bail(fail(ctx, VOC_UNSUPPORTED, "the library is compiled for sm_103 (GB300) only"));
  e = dev_alloc(reinterpret_cast<void **>(&ctx->err_dev), 8 * sizeof(int));  // [0] error word, [1] finite flag, [4..7] checks
  if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "cudaMalloc"));
  ctx->allocs.push_back(ctx->err_dev);
  ctx->flag_dev = ctx->err_dev + 1;
  cudaMemset(ctx->err_dev, 0, 8 * sizeof(int));
  if ((st0 = static_ws_setup(ctx)) != VOC_OK) return bail(st0);

  const int pad = desc->padding;
  auto plan = [&](Layer &L, bool has_skip) {
    L.prec = ctx->prec;
    return plan_layer(ctx->use_pair, L, pad, has_skip, why);
  };
  const int nd = desc->n_dilations;
  int p = 0;
  voc_status st;
  // optional 1x1 input projection (no Snake around it; its epilogue only splits hi/lo)
  int conv_in_src = BUF_H0;
  if (desc->in_proj_channels > 0) {
    Layer L;
    L.name = "in_proj";
    L.Cin = desc->latent_channels, L.Cout = desc->in_proj_channels, L.K = 1, L.dil = 1;
    L.level = 0;
    if (!plan(L, false))
      return bail(fail(ctx, VOC_UNSUPPORTED, "in_proj: " + why));
    L.in_buf = BUF_H0, L.hl_buf = BUF_HB;
    st = upload_layer(ctx, ctx->allocs, L, pad, params[0], params[1], SnakeCoef{});
    if (st != VOC_OK) return bail(st);
    ctx->layers.push_back(L);
    conv_in_src = BUF_HB;
    p = 2;
  }
  // conv_in (no Snake in front); its epilogue applies the Snake of stage 0's ConvT
  {
    Layer L;
    L.name = "conv_in";
    L.Cin = desc->in_proj_channels > 0 ? desc->in_proj_channels : desc->latent_channels;
    L.Cout = desc->channels0, L.K = desc->in_kernel, L.dil = 1;
    L.level = 0;
    if (!plan(L, false))
      return bail(fail(ctx, VOC_UNSUPPORTED, "conv_in: " + why));
    L.in_buf = conv_in_src, L.hl_buf = BUF_H1;
    st = upload_layer(ctx, ctx->allocs, L, pad, params[p], params[p + 1],
                      snake_coef(params[p + 2], L.Cout, desc->snake));
    if (st != VOC_OK) return bail(st);
    ctx->layers.push_back(L);
    p += 2;
  }
  // Three equal hi/lo buffers (H0, H1, HB) and the fp32 residual stream FY.  A layer that
  // reads a hi/lo buffer with a halo never writes that buffer in the same launch (other
  // tiles still read its halo rows); the fp32 stream is read row for row, so the residual
  // layers update it in place.
  auto other = [](int a, int b) {
    for (int c : {(int)BUF_H0, (int)BUF_H1, (int)BUF_HB})
      if (c != a && c != b) return c;
    return -1;
  };
  int x_buf = BUF_H1;  // Snake'd input of the next ConvT (written by conv_in)
  int C = desc->channels0;
  for (int i = 0; i < desc->n_stages; ++i) {
    const int Co = ctx->widths[i];
    int cur = other(x_buf, BUF_HB);  // Snake1 input of the stage's first residual unit
    {
      Layer L;
      L.name = "convT" + std::to_string(i);
      L.convT = true;
      L.Cin = C, L.Cout = Co, L.stride = ctx->strides[i], L.K = 2 * L.stride;
      L.level = i;
      if (!plan(L, false))
        return bail(fail(ctx, VOC_UNSUPPORTED, L.name + ": " + why));
      L.in_buf = x_buf, L.f32_buf = BUF_FY, L.hl_buf = cur;
      st = upload_layer(ctx, ctx->allocs, L, pad, params[p + 1], params[p + 2],
                        snake_coef(params[p + 3], L.Cout, desc->snake));
      if (st != VOC_OK) return bail(st);
      ctx->layers.push_back(L);
      p += 3;
    }
    C = Co;
    for (int j = 0; j < nd; ++j) {
      const float *w1 = params[p + 1], *b1 = params[p + 2];
      const SnakeCoef a2 = snake_coef(params[p + 3], C, desc->snake);
      const float *w2 = params[p + 4], *b2 = params[p + 5];
      p += 6;
      // next snake1 / next stage's snake / snake_out, all over this stage's C channels
      const SnakeCoef next_alpha = snake_coef(params[p], C, desc->snake);
      const bool last_stage = (i == desc->n_stages - 1);
      Layer R;  // the whole unit in one kernel when it fits and is enabled
      R.name = "s" + std::to_string(i) + "r" + std::to_string(j) + ".ru";
      R.prec = ctx->prec;
      R.Cin = C, R.Cout = C, R.K = desc->res_kernel, R.dil = ctx->dils[j];
      R.level = i + 1;
      if (rup(C, 16) <= ctx->fuse_max_c && rup(C, 16) >= ctx->fuse_min_c && plan_ru(R, pad, why)) {
        const int out = other(cur, -1);  // never the buffer this unit reads
        R.in_buf = cur, R.skip_buf = BUF_FY;
        if (j < nd - 1) {
          R.f32_buf = BUF_FY, R.hl_buf = out;
        } else if (!last_stage) {
          R.hl_buf = out;  // the next stage's ConvT input
        } else {
          R.f32_buf = BUF_FY, R.epi_flags = voc::EPI_F32_SNAKE;  // Snake_out(y) for the head
        }
        st = upload_ru(ctx, ctx->allocs, R, pad, w1, b1, a2, w2, b2, next_alpha);
        if (st != VOC_OK) return bail(st);
        ctx->layers.push_back(R);
        if (R.hl_buf >= 0) cur = out;
        continue;
      }
      const int tmp = other(cur, x_buf == cur ? -1 : x_buf);  // conv1 output, read by conv2
      Layer L1;
      L1.name = "s" + std::to_string(i) + "r" + std::to_string(j) + ".conv1";
      L1.Cin = C, L1.Cout = C, L1.K = desc->res_kernel, L1.dil = ctx->dils[j];
      L1.level = i + 1;
      if (!plan(L1, false))
        return bail(fail(ctx, VOC_UNSUPPORTED, L1.name + ": " + why));
      L1.in_buf = cur, L1.hl_buf = tmp;
      st = upload_layer(ctx, ctx->allocs, L1, pad, w1, b1, a2);
      if (st != VOC_OK) return bail(st);
      ctx->layers.push_back(L1);

      Layer L2;  // 1x1: reads `tmp` row for row, so it may write `cur`
      L2.name = "s" + std::to_string(i) + "r" + std::to_string(j) + ".conv2";
      L2.Cin = C, L2.Cout = C, L2.K = 1, L2.dil = 1;
      L2.level = i + 1;
      if (!plan(L2, true))
        return bail(fail(ctx, VOC_UNSUPPORTED, L2.name + ": " + why));
      L2.in_buf = tmp, L2.skip_buf = BUF_FY;
      if (j < nd - 1) {
        L2.f32_buf = BUF_FY, L2.hl_buf = cur;
      } else if (!last_stage) {
        L2.hl_buf = cur;
      } else {
        L2.f32_buf = BUF_FY, L2.epi_flags = voc::EPI_F32_SNAKE;
      }
      st = upload_layer(ctx, ctx->allocs, L2, pad, w2, b2, next_alpha);
      if (st != VOC_OK) return bail(st);
      ctx->layers.push_back(L2);
    }
    x_buf = cur;
  }
  // out head: Snake already applied by the last conv2 epilogue
  {
    OutHead &h = ctx->head;
    h.C = C, h.Cp = rup(C, 16), h.K = desc->out_kernel;
    h.pad_left = (pad == VOC_PAD_CAUSAL) ? h.K - 1 : (h.K - 1) / 2;
    h.level = desc->n_stages;
    const float *w_in = params[p + 1], *b = params[p + 2];
    // F16 / BF16-weight precision: the head's weights are rounded like every conv weight
    std::vector<float> w((size_t)C * h.K);
    for (size_t i = 0; i < w.size(); ++i)
      w[i] = ctx->prec == VOC_PREC_F16W    ? __half2float(__float2half_rn(w_in[i]))
             : ctx->prec == VOC_PREC_BF16W ? bf2f(f2bf(w_in[i]))
                                           : w_in[i];
    std::vector<float> wp((size_t)h.Cp * h.K, 0.f), bp(1, b ? b[0] : 0.f);
    for (int c = 0; c < C; ++c)
      for (int k = 0; k < h.K; ++k) wp[(size_t)c * h.K + k] = w[(size_t)c * h.K + k];
    st = upload(ctx, ctx->allocs, wp, &h.w_dev);
    if (st != VOC_OK) return bail(st);
    std::vector<float> w4((size_t)h.K * h.Cp, 0.f);  // [k][c/4][c%4]
    for (int c = 0; c < C; ++c)
      for (int k = 0; k < h.K; ++k) w4[((size_t)k * (h.Cp / 4) + c / 4) * 4 + c % 4] = w[(size_t)c * h.K + k];
    st = upload(ctx, ctx->allocs, w4, &h.w4_dev);
    if (st != VOC_OK) return bail(st);
    st = upload(ctx, ctx->allocs, bp, &h.b_dev);
    if (st != VOC_OK) return bail(st);
    // Fold the head into the last conv2 when that layer (a 1x1 conv of one column tile or a
    // fused residual unit, not a CTA pair) writes Snake_out(y) and the head has at most
    // kHeadFoldMaxK taps; its partial sums go to a hi/lo buffer the layer does not read.
    // Causal decoders keep the separate head: their chunk-by-chunk stream decode runs it, and
    // a streamed sequence must equal the whole-sequence decode bit for bit (the folded head
    // adds its products in another order).
    Layer &last = ctx->layers.back();
    if (pad == VOC_PAD_SYMMETRIC && !last.pair && !last.convT &&
        (last.epi_flags & voc::EPI_F32_SNAKE) &&
        last.g.n_tiles == 1 && h.K <= voc::kHeadFoldMaxK && last.Cp_out == h.Cp) {
      // [k][c], zero-padded to kHeadFoldMaxK taps (same left padding)
      std::vector<float> wk((size_t)voc::kHeadFoldMaxK * h.Cp, 0.f);
      for (int c = 0; c < C; ++c)
        for (int k = 0; k < h.K; ++k) wk[(size_t)k * h.Cp + c] = w[(size_t)c * h.K + k];
      st = upload(ctx, ctx->allocs, wk, &h.wk_dev);
      if (st != VOC_OK) return bail(st);
      last.head_fold = true;
      for (int c : {(int)BUF_H0, (int)BUF_H1, (int)BUF_HB})
        if (c != last.in_buf) {
          last.head_buf = c;
          break;
        }
    }
  }
  for (vocoder::MapSet &c : ctx->map_sets) {
    c.maps.assign(ctx->layers.size(), CUtensorMap{});
    c.skip_maps.assign(ctx->layers.size(), CUtensorMap{});
  }
  *out = ctx;
  return VOC_OK;
}

VOC_API long long vocoder_hop(const vocoder *ctx) { return ctx ? ctx->hop : -1; }

VOC_API size_t vocoder_workspace_bytes(const vocoder *ctx, int B, int T) {
  if (!ctx || B < 1 || T < 1) return 0;
  if ((long long)T * ctx->hop > 0x7FFFFFFFLL) return 0;
  return BUF_COUNT * buf_bytes(ctx, B, T);
}

VOC_API size_t vocoder_workspace_bytes_host(const vocoder *ctx, int B, int T) {
  const size_t w = vocoder_workspace_bytes(ctx, B, T);
  if (!w) return 0;
  return w + rupz((size_t)B * ctx->desc.latent_channels * T * 4, 256) +
         rupz((size_t)B * T * ctx->hop * 4, 256);
}

VOC_API int vocoder_launches_per_decode(const vocoder *ctx, int B, int T) {
  if (!ctx || B < 1 || T < 1) return -1;
  return 2 + static_cast<int>(ctx->layers.size());
}

namespace {
void head_fold_args(const vocoder *ctx, const Layer &L, void *const *bufs, ConvGemmArgs &a) {
  a.out_f32 = nullptr;  // the layer writes the head's partial sums instead
  a.head_w = ctx->head.wk_dev;
  a.head_part = static_cast<float *>(bufs[L.head_buf]);
  a.head_K = voc::kHeadFoldMaxK;  // the weights are zero-padded to this many taps
  a.head_pad = ctx->head.pad_left;
  a.head_slices = 4 * a.m_tiles;
  a.head_slice_len = 32 + voc::kHeadFoldMaxK - 1;
}

voc_status launch_head_finish(vocoder *ctx, const Layer &L, void *const *bufs, int B, long long Lf,
                              float *audio, cudaStream_t stream) {
  const OutHead &h = ctx->head;
  const int slices = static_cast<int>(4 * ((Lf + voc::kTileM - 1) / voc::kTileM));
  dim3 grid(static_cast<unsigned>((Lf + 255) / 256), static_cast<unsigned>(B));
  cudaError_t e = launch_pdl(voc::head_finish_kernel, grid, dim3(256), 0, stream,
                             static_cast<const float *>(bufs[L.head_buf]), static_cast<int>(Lf),
                             slices, L.Cp_out / 16, voc::kHeadFoldMaxK, h.pad_left,
                             static_cast<const float *>(h.b_dev), audio);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "launch head_finish");
  return VOC_OK;
}

voc_status decode_impl(vocoder *ctx, const float *latent, int B, int T, float *audio, void *ws,
                       size_t ws_bytes, cudaStream_t stream, unsigned flags) {
  const size_t need = vocoder_workspace_bytes(ctx, B, T);
  if (!need) return fail(ctx, VOC_INVALID_ARG, "invalid B / T");
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(ctx, VOC_INVALID_ARG, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < need)
    return fail(ctx, VOC_WORKSPACE_TOO_SMALL,
                "workspace " + std::to_string(ws_bytes) + " < " + std::to_string(need));
  if (reinterpret_cast<uintptr_t>(latent) & 15)
    return fail(ctx, VOC_INVALID_ARG, "latent not 16-byte aligned");
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != ctx->device) return fail(ctx, VOC_INVALID_ARG, "current device differs from the context's");

  const size_t bb = buf_bytes(ctx, B, T);
  void *bufs[BUF_COUNT];
  for (int i = 0; i < BUF_COUNT; ++i) bufs[i] = static_cast<uint8_t *>(ws) + i * bb;

  // TMA descriptors depend on the workspace address and the sizes only
  vocoder::MapSet *ms = nullptr;
  for (int k = 0; k < 2; ++k) {
    vocoder::MapSet &c = ctx->map_sets[k];
    if (c.ws == ws && c.B == B && c.T == T) {
      ms = &c;
      ctx->map_lru = 1 - k;
    }
  }
  if (!ms) {
    ms = &ctx->map_sets[ctx->map_lru];
    ctx->map_lru = 1 - ctx->map_lru;
    ms->ws = nullptr;  // invalid until every descriptor is encoded
    for (size_t i = 0; i < ctx->layers.size(); ++i) {
      const Layer &L = ctx->layers[i];
      voc_status st = encode_map(ctx, &ms->maps[i], bufs[L.in_buf], L.Cp_in,
                                 pitch8(level_len(ctx, L.level, T)), B, L.g.rows, L.g.KB / 8);
      ms->skip_maps[i] = CUtensorMap{};
      if (st == VOC_OK && L.skip_buf >= 0)
        st = encode_skip_map(ctx, &ms->skip_maps[i], bufs[L.skip_buf], L.Cp_out,
                             pitch8(level_len(ctx, L.level, T)), B, L.cw);
      if (st != VOC_OK) return st;
    }
    ms->ws = ws, ms->B = B, ms->T = T;
  }

  const bool prof = (flags & VOC_FLAG_PROFILE) != 0;
  const int n_launch = vocoder_launches_per_decode(ctx, B, T);
  if (prof) {
    while ((int)ctx->events.size() < 2 * n_launch) {
      cudaEvent_t ev;
      cudaError_t e = cudaEventCreate(&ev);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaEventCreate");
      ctx->events.push_back(ev);
    }
    ctx->prof_names.assign(n_launch, "");
    ctx->prof_flops.assign(n_launch, 0.0);
    ctx->prof_bytes.assign(n_launch, 0.0);
    ctx->prof_impl.assign(n_launch, 0.0);
    ctx->prof_ms.assign(n_launch, -1.f);
    ctx->prof_n = n_launch;
    ctx->prof_ready = false;
  }
  int li = 0;
  auto rec = [&](int which) {
    if (prof) cudaEventRecord(ctx->events[2 * li + which], stream);
  };

  // the head folded into the last conv2, when its partial sums fit the buffer they borrow
  const long long Lf_out = level_len(ctx, ctx->desc.n_stages, T);
  const bool fold = ctx->layers.back().head_fold &&
                    (double)B * head_part_floats(ctx, ctx->layers.back(), Lf_out) * 4.0 <= (double)bb;
  voc_status st;
  rec(0);
  st = launch_prep(ctx, latent, B, ctx->desc.latent_channels, T, ctx->Cp_lat, nullptr, nullptr,
                   static_cast<__nv_bfloat16 *>(bufs[BUF_H0]), stream);
  if (st != VOC_OK) return st;
#ifdef VOC_CHECKS
  if ((st = check_launch(ctx, "prep_latent", stream)) != VOC_OK) return st;
#endif
  rec(1);
  if (prof) {
    ctx->prof_names[li] = "prep_latent";  // the API layout into the kernels' operand layout
    ctx->prof_bytes[li] = (double)B * T * 8.0 * ctx->desc.latent_channels;
    ctx->prof_impl[li] = (double)B * T * (4.0 * ctx->desc.latent_channels + 4.0 * ctx->Cp_lat);
  }
  ++li;
  for (size_t i = 0; i < ctx->layers.size(); ++i, ++li) {
    const Layer &L = ctx->layers[i];
    ConvGemmArgs a;
    gemm_launch_args(ctx, L, B, T, bufs, bb, a);
    if (L.head_fold && fold) head_fold_args(ctx, L, bufs, a);
    rec(0);
    st = launch_gemm(ctx, L, ms->maps[i], ms->skip_maps[i], a, stream, -1,
                     L.skip_buf >= 0 ? (long long)(bb / 4) : -1);
    if (st != VOC_OK) return st;
#ifdef VOC_CHECKS
    if ((st = check_launch(ctx, L.name, stream)) != VOC_OK) return st;
#endif
    rec(1);
    if (prof) {
      ctx->prof_names[li] = L.name;
      layer_cost(ctx, L, B, T, ctx->prof_flops[li], ctx->prof_bytes[li], ctx->prof_impl[li],
                 L.head_fold && fold);
    }
  }
  const long long Lf = level_len(ctx, ctx->desc.n_stages, T);
  const Layer &last = ctx->layers.back();
  rec(0);
  if (fold)
    st = launch_head_finish(ctx, last, bufs, B, Lf, audio, stream);
  else
    st = launch_out_head(ctx, ctx->head, static_cast<const float *>(bufs[BUF_FY]), B, Lf, audio,
                         stream, 0, pitch8(Lf));
  if (st != VOC_OK) return st;
#ifdef VOC_CHECKS
  if ((st = check_launch(ctx, "out_head", stream)) != VOC_OK) return st;
#endif
  rec(1);
  if (prof) {
    ctx->prof_names[li] = "out_head";
    // folded: the last conv2 did the products (its launch counts them); this launch adds the
    // partial sums into the audio
    ctx->prof_flops[li] = fold ? 0.0 : 2.0 * ctx->head.C * ctx->head.K * B * (double)Lf;
    ctx->prof_bytes[li] = fold ? 4.0 * B * (double)Lf : (double)B * Lf * (4.0 * ctx->head.C + 4.0);
    ctx->prof_impl[li] = fold
                             ? (double)B * head_part_floats(ctx, last, Lf) * 4.0 + 4.0 * B * Lf
                             : (double)B * Lf * (4.0 * ctx->head.Cp + 4.0);
    ctx->prof_ready = true;
  }
  ++li;

  if (flags & VOC_FLAG_CHECK_FINITE) {
    cudaMemsetAsync(ctx->flag_dev, 0, sizeof(int), stream);
    const long long n = (long long)B * Lf;
    const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 4L * ctx->num_sms));
    voc::finite_check_kernel<<<blocks, 256, 0, stream>>>(audio, n, ctx->flag_dev);
    int flag = 0;
    cudaError_t e = cudaMemcpyAsync(&flag, ctx->flag_dev, sizeof(int), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "finite check");
    if (flag) return fail(ctx, VOC_NONFINITE, "decoded audio contains NaN or Inf");
  }
  if (flags & (VOC_FLAG_SYNC | VOC_FLAG_CHECK_FINITE)) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
    int word = 0;
    e = cudaMemcpy(&word, ctx->err_dev, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "read device error word");
    if (word) {
      cudaMemset(ctx->err_dev, 0, sizeof(int));
      return fail(ctx, VOC_DEVICE_TIMEOUT,
                  "a kernel gave up a bounded wait (code " + std::to_string(word) + ")");
    }
  }
  return VOC_OK;
}
}  // namespace

VOC_API voc_status vocoder_decode(vocoder *ctx, const float *latent_dev, int B, int T,
                                  float *audio_dev, void *ws_dev, size_t ws_bytes,
                                  voc_stream_t stream, unsigned flags) {
  if (!ctx) return fail(nullptr, VOC_INVALID_ARG, "ctx is NULL");
  if (!latent_dev || !audio_dev) return fail(ctx, VOC_INVALID_ARG, "latent / audio NULL");
  if (B < 1 || T < 1) return fail(ctx, VOC_INVALID_ARG, "B and T must be positive");
  if (cancelled(ctx)) return fail(ctx, VOC_CANCELLED, "cancelled: the caller's cancel flag is set");
  return decode_impl(ctx, latent_dev, B, T, audio_dev, ws_dev, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream), flags);
}

VOC_API voc_status vocoder_decode_host(vocoder *ctx, const float *latent_host, int B, int T,
                                       float *audio_host, void *ws_dev, size_t ws_bytes,
                                       voc_stream_t stream, unsigned flags) {
  if (!ctx) return fail(nullptr, VOC_INVALID_ARG, "ctx is NULL");
  if (!latent_host || !audio_host) return fail(ctx, VOC_INVALID_ARG, "latent / audio NULL");
  if (B < 1 || T < 1) return fail(ctx, VOC_INVALID_ARG, "B and T must be positive");
  const size_t need = vocoder_workspace_bytes_host(ctx, B, T);
  if (!need) return fail(ctx, VOC_INVALID_ARG, "invalid B / T");
  if (!ws_dev || (reinterpret_cast<uintptr_t>(ws_dev) & 255))
    return fail(ctx, VOC_INVALID_ARG, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < need)
    return fail(ctx, VOC_WORKSPACE_TOO_SMALL,
                "workspace " + std::to_string(ws_bytes) + " < " + std::to_string(need));
  if (cancelled(ctx)) return fail(ctx, VOC_CANCELLED, "cancelled: the caller's cancel flag is set");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t wdec = vocoder_workspace_bytes(ctx, B, T);
  const size_t lat_bytes = (size_t)B * ctx->desc.latent_channels * T * 4;
  const size_t aud_bytes = (size_t)B * T * ctx->hop * 4;
  uint8_t *base = static_cast<uint8_t *>(ws_dev);
  float *lat_d = reinterpret_cast<float *>(base + wdec);
  float *aud_d = reinterpret_cast<float *>(base + wdec + rupz(lat_bytes, 256));
  cudaError_t e = cudaMemcpyAsync(lat_d, latent_host, lat_bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "copy latent in");
  voc_status st = decode_impl(ctx, lat_d, B, T, aud_d, ws_dev, wdec, s, flags);
  if (st != VOC_OK) return st;
  e = cudaMemcpyAsync(audio_host, aud_d, aud_bytes, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "copy audio out");
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
  return VOC_OK;
}

VOC_API voc_status vocoder_decode_static(vocoder *ctx, const float *latent_dev, int B, int T,
                                         float *audio_dev, voc_stream_t stream, unsigned flags) {
  if (!ctx) return fail(nullptr, VOC_INVALID_ARG, "ctx is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGetDevice");
  if (dev != ctx->device) return fail(ctx, VOC_INVALID_ARG, "current device differs from the context's");
  if (!latent_dev || !audio_dev) return fail(ctx, VOC_INVALID_ARG, "latent / audio NULL");
  if (B < 1 || T < 1) return fail(ctx, VOC_INVALID_ARG, "B and T must be positive");
  if (flags & VOC_FLAG_PROFILE)
    return fail(ctx, VOC_INVALID_ARG, "VOC_FLAG_PROFILE is not available without allocation");
  const size_t need = vocoder_workspace_bytes(ctx, B, T);
  if (!need) return fail(ctx, VOC_INVALID_ARG, "invalid B / T");
  if (need > VOC_STATIC_WORKSPACE_BYTES)
    return fail(ctx, VOC_WORKSPACE_TOO_SMALL,
                "B=" + std::to_string(B) + ", T=" + std::to_string(T) + " needs " +
                    std::to_string(need) + " bytes of workspace; the built-in array holds " +
                    std::to_string(VOC_STATIC_WORKSPACE_BYTES) + " (use vocoder_decode)");
  void *ws = static_ws_addr(dev);  // looked up by vocoder_create on this device
  if (!ws) return fail(ctx, VOC_UNSUPPORTED, "no built-in workspace on this device");
  if (cancelled(ctx)) return fail(ctx, VOC_CANCELLED, "cancelled: the caller's cancel flag is set");
  return decode_impl(ctx, latent_dev, B, T, audio_dev, ws, VOC_STATIC_WORKSPACE_BYTES,
                     reinterpret_cast<cudaStream_t>(stream), flags);
}

VOC_API long long vocoder_stitched_length(int n_win, int win_frames, int crop_left, int crop_right,
                                          int hop) {
  if (n_win < 1 || win_frames < 1 || crop_left < 0 || crop_right < 0 || hop < 1) return -1;
  long long frames = 0;
  for (int w = 0; w < n_win; ++w) {
    const int lo = (w == 0) ? 0 : crop_left;
    const int hi = (w == n_win - 1) ? win_frames : win_frames - crop_right;
    if (hi < lo) return -1;
    frames += hi - lo;
  }
  return frames * hop;
}

VOC_API voc_status vocoder_stitch(const float *decoded_dev, int n_win, int n_sides, int win_frames,
                                  int crop_left, int crop_right, int hop, float *out_dev,
                                  voc_stream_t stream) {
  if (!decoded_dev || !out_dev) return fail(nullptr, VOC_INVALID_ARG, "stitch: NULL buffer");
  if (n_sides < 1 || n_sides > 65535) return fail(nullptr, VOC_INVALID_ARG, "stitch: n_sides");
  const long long len = vocoder_stitched_length(n_win, win_frames, crop_left, crop_right, hop);
  if (len < 0) return fail(nullptr, VOC_INVALID_ARG, "stitch: invalid window geometry");
  if (len == 0) return VOC_OK;
  dim3 grid(static_cast<unsigned>((len + 255) / 256), static_cast<unsigned>(n_sides));
  cudaError_t e = launch_pdl(voc::stitch_kernel, grid, dim3(256), 0,
                             reinterpret_cast<cudaStream_t>(stream), decoded_dev, n_win, n_sides,
                             win_frames, crop_left, crop_right, hop, len, out_dev);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "launch stitch");
  return VOC_OK;
}

namespace {
// Shared body of the single-layer operations.
voc_status op_layer(Layer &L, int padding, const float *x_dev, int B, int T, const float *w_host,
                    const float *b_host, const float *alpha_host, float *y_dev, cudaStream_t stream) {
  std::string why;
  if (!set_kernel_attrs(why)) return fail(nullptr, VOC_CUDA_ERROR, why);
  if (!plan_layer(false, L, padding, false, why)) return fail(nullptr, VOC_UNSUPPORTED, why);
  int dev = 0, sms = 0, major = 0, minor = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return fail(nullptr, VOC_UNSUPPORTED, "the library is compiled for sm_103 (GB300) only");
  vocoder tmp;  // carries the allocations, the error word and the launch settings
  tmp.num_sms = sms;
  tmp.device = dev;
  tmp.strides = {L.convT ? L.stride : 1};
  auto done = [&](voc_status st) {
    if (st != VOC_OK) g_err = tmp.err;
    for (void *p : tmp.allocs) dev_free(p);
    return st;
  };
  voc_status st = upload_layer(&tmp, tmp.allocs, L, padding, w_host, b_host, SnakeCoef{});
  if (st != VOC_OK) return done(st);
  cudaError_t e;
  float *alpha_d = nullptr, *invb_d = nullptr;
  if (alpha_host) {
    std::vector<float> a(alpha_host, alpha_host + L.Cin), ib(L.Cin);
    for (int c = 0; c < L.Cin; ++c) ib[c] = static_cast<float>(1.0 / ((double)a[c] + 1e-9));
    if ((st = upload(&tmp, tmp.allocs, a, &alpha_d)) != VOC_OK) return done(st);
    if ((st = upload(&tmp, tmp.allocs, ib, &invb_d)) != VOC_OK) return done(st);
  }
  const int s = L.convT ? L.stride : 1;
  const long long Tp = pitch8(T), Yp = pitch8((long long)T * s);  // plane rows
  void *hl = nullptr, *rows = nullptr;
  e = dev_alloc(reinterpret_cast<void **>(&hl), (size_t)B * Tp * L.Cp_in * 4);
  if (e != cudaSuccess) return done(cuda_fail(&tmp, e, "cudaMalloc"));
  tmp.allocs.push_back(hl);
  e = dev_alloc(reinterpret_cast<void **>(&rows), (size_t)B * Yp * L.Cp_out * 4);
  if (e != cudaSuccess) return done(cuda_fail(&tmp, e, "cudaMalloc"));
  tmp.allocs.push_back(rows);
  if ((st = launch_prep(&tmp, x_dev, B, L.Cin, T, L.Cp_in, alpha_d, invb_d,
                        static_cast<__nv_bfloat16 *>(hl), stream)) != VOC_OK)
    return done(st);
  CUtensorMap map;
  if ((st = encode_map(&tmp, &map, hl, L.Cp_in, Tp, B, L.g.rows, L.g.KB / 8)) != VOC_OK) return done(st);
  void *bufs[BUF_COUNT] = {hl, nullptr, nullptr, rows};
  L.level = 0;
  L.in_buf = 0, L.f32_buf = BUF_FY;
  ConvGemmArgs a;
  e = dev_alloc(reinterpret_cast<void **>(&tmp.err_dev), 8 * sizeof(int));
  if (e != cudaSuccess) return done(cuda_fail(&tmp, e, "cudaMalloc"));
  tmp.allocs.push_back(tmp.err_dev);
  cudaMemsetAsync(tmp.err_dev, 0, 8 * sizeof(int), stream);
  gemm_launch_args(&tmp, L, B, T, bufs, (size_t)B * Yp * L.Cp_out * 4, a);
  const CUtensorMap no_skip{};
  if ((st = launch_gemm(&tmp, L, map, no_skip, a, stream)) != VOC_OK) return done(st);
  dim3 grid((T * s + 255) / 256, L.Cp_out / 4, B);
  voc::rows_to_cf_kernel<<<grid, 256, 0, stream>>>(static_cast<const float *>(rows), T * s, Yp,
                                                   L.Cp_out, L.Cout, y_dev);
  e = cudaGetLastError();
  if (e != cudaSuccess) return done(cuda_fail(&tmp, e, "launch rows_to_cf"));
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return done(cuda_fail(&tmp, e, "cudaStreamSynchronize"));
  int word = 0;
  cudaMemcpy(&word, tmp.err_dev, sizeof(int), cudaMemcpyDeviceToHost);
  if (word) return done(fail(&tmp, VOC_DEVICE_TIMEOUT, "a kernel gave up a bounded wait"));
  return done(VOC_OK);
}
}  // namespace

VOC_API voc_status vocoder_op_conv1d(const float *x_dev, int B, int Cin, int T, const float *w_host,
                                     const float *b_host, int Cout, int K, int dil, int padding,
                                     const float *alpha_host, float *y_dev, voc_stream_t stream) {
  if (!x_dev || !w_host || !y_dev) return fail(nullptr, VOC_INVALID_ARG, "NULL pointer");
  if (B < 1 || Cin < 1 || T < 1 || Cout < 1 || K < 1 || K > 15 || K % 2 == 0 || dil < 1 ||
      dil * (K - 1) > 120 || (padding != VOC_PAD_SYMMETRIC && padding != VOC_PAD_CAUSAL))
    return fail(nullptr, VOC_INVALID_ARG, "invalid conv1d shape");
  Layer L;
  L.name = "op_conv1d";
  L.Cin = Cin, L.Cout = Cout, L.K = K, L.dil = dil;
  return op_layer(L, padding, x_dev, B, T, w_host, b_host, alpha_host, y_dev,
                  reinterpret_cast<cudaStream_t>(stream));
}

VOC_API voc_status vocoder_op_conv_transpose1d(const float *x_dev, int B, int Cin, int T,
                                               const float *w_host, const float *b_host, int Cout,
                                               int stride, int padding, const float *alpha_host,
                                               float *y_dev, voc_stream_t stream) {
  if (!x_dev || !w_host || !y_dev) return fail(nullptr, VOC_INVALID_ARG, "NULL pointer");
  if (B < 1 || Cin < 1 || T < 1 || Cout < 1 || stride < 1 || stride > 16 ||
      (padding != VOC_PAD_SYMMETRIC && padding != VOC_PAD_CAUSAL) ||
      (padding == VOC_PAD_SYMMETRIC && stride % 2))
    return fail(nullptr, VOC_INVALID_ARG, "invalid conv_transpose1d shape");
  Layer L;
  L.name = "op_convT";
  L.convT = true;
  L.Cin = Cin, L.Cout = Cout, L.stride = stride, L.K = 2 * stride;
  return op_layer(L, padding, x_dev, B, T, w_host, b_host, alpha_host, y_dev,
                  reinterpret_cast<cudaStream_t>(stream));
}

VOC_API voc_status vocoder_op_residual_unit(const float *x_dev, int B, int C, int T,
                                            const float *alpha1_host, const float *w1_host,
                                            const float *b1_host, int K, int dil,
                                            const float *alpha2_host, const float *w2_host,
                                            const float *b2_host, int padding, float *y_dev,
                                            voc_stream_t stream_) {
  if (!x_dev || !y_dev || !w1_host || !w2_host || !alpha1_host || !alpha2_host)
    return fail(nullptr, VOC_INVALID_ARG, "NULL pointer");
  if (B < 1 || C < 1 || T < 1 || K < 1 || K > 15 || K % 2 == 0 || dil < 1 ||
      dil * (K - 1) > 120 || (padding != VOC_PAD_SYMMETRIC && padding != VOC_PAD_CAUSAL))
    return fail(nullptr, VOC_INVALID_ARG, "invalid residual unit shape");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  std::string why;
  if (!set_kernel_attrs(why)) return fail(nullptr, VOC_CUDA_ERROR, why);
  int dev = 0, sms = 0, major = 0, minor = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return fail(nullptr, VOC_UNSUPPORTED, "the library is compiled for sm_103 (GB300) only");
  vocoder tmp;
  tmp.num_sms = sms;
  tmp.device = dev;
  tmp.strides = {1};
  auto done = [&](voc_status st) {
    if (st != VOC_OK) g_err = tmp.err;
    for (void *q : tmp.allocs) dev_free(q);
    return st;
  };
  const int Cp = rup(C, 16);
  const long long Tp = pitch8(T);  // plane rows
  const size_t bb = (size_t)B * Tp * Cp * 4;
  void *bufs[BUF_COUNT] = {nullptr, nullptr, nullptr, nullptr};
  for (int i : {(int)BUF_H0, (int)BUF_HB, (int)BUF_FY}) {
    cudaError_t e = dev_alloc(&bufs[i], bb);
    if (e != cudaSuccess) return done(cuda_fail(&tmp, e, "cudaMalloc"));
    tmp.allocs.push_back(bufs[i]);
  }
  cudaError_t e = dev_alloc(reinterpret_cast<void **>(&tmp.err_dev), 8 * sizeof(int));
  if (e != cudaSuccess) return done(cuda_fail(&tmp, e, "cudaMalloc"));
  tmp.allocs.push_back(tmp.err_dev);
  cudaMemsetAsync(tmp.err_dev, 0, 8 * sizeof(int), stream);
  voc_status st;
  float *alpha_d = nullptr, *invb_d = nullptr;
  {
    std::vector<float> a(alpha1_host, alpha1_host + C), ib(C);
    for (int c = 0; c < C; ++c) ib[c] = static_cast<float>(1.0 / ((double)a[c] + 1e-9));
    if ((st = upload(&tmp, tmp.allocs, a, &alpha_d)) != VOC_OK) return done(st);
    if ((st = upload(&tmp, tmp.allocs, ib, &invb_d)) != VOC_OK) return done(st);
  }
  // A = Snake1(x) as hi/lo; the residual stream x as fp32 chunk-major (updated in place)
  if ((st = launch_prep(&tmp, x_dev, B, C, T, Cp, alpha_d, invb_d,
                        static_cast<__nv_bfloat16 *>(bufs[BUF_H0]), stream)) != VOC_OK)
    return done(st);
  voc::cf_to_rows_kernel<<<dim3(static_cast<unsigned>((Tp + 255) / 256), Cp / 4, B), 256, 0, stream>>>(
      x_dev, T, static_cast<int>(Tp), Cp, C, static_cast<float *>(bufs[BUF_FY]));
  std::vector<Layer> layers;
  Layer R;
  R.name = "op_ru";
  R.Cin = C, R.Cout = C, R.K = K, R.dil = dil;
  if (plan_ru(R, padding, why)) {
    R.in_buf = BUF_H0, R.skip_buf = BUF_FY, R.f32_buf = BUF_FY;
    if ((st = upload_ru(&tmp, tmp.allocs, R, padding, w1_host, b1_host,
                        snake_coef(alpha2_host, C, VOC_SNAKE), w2_host, b2_host, SnakeCoef{})) != VOC_OK)
      return done(st);
    layers.push_back(R);
  } else {
    Layer L1, L2;
    L1.name = "op_conv1", L2.name = "op_conv2";
    L1.Cin = L1.Cout = L2.Cin = L2.Cout = C;
    L1.K = K, L1.dil = dil, L2.K = 1, L2.dil = 1;
    if (!plan_layer(false, L1, padding, false, why) || !plan_layer(false, L2, padding, true, why))
      return done(fail(&tmp, VOC_UNSUPPORTED, why));
    L1.in_buf = BUF_H0, L1.hl_buf = BUF_HB;
    L2.in_buf = BUF_HB, L2.skip_buf = BUF_FY, L2.f32_buf = BUF_FY;
    if ((st = upload_layer(&tmp, tmp.allocs, L1, padding, w1_host, b1_host,
                           snake_coef(alpha2_host, C, VOC_SNAKE))) != VOC_OK ||
        (st = upload_layer(&tmp, tmp.allocs, L2, padding, w2_host, b2_host, SnakeCoef{})) != VOC_OK)
      return done(st);
    layers.push_back(L1);
    layers.push_back(L2);
  }
  for (const Layer &L : layers) {
    CUtensorMap map, smap{};
    if ((st = encode_map(&tmp, &map, bufs[L.in_buf], L.Cp_in, Tp, B, L.g.rows, L.g.KB / 8)) != VOC_OK)
      return done(st);
    if (L.skip_buf >= 0 &&
        (st = encode_skip_map(&tmp, &smap, bufs[L.skip_buf], L.Cp_out, Tp, B, L.cw)) != VOC_OK)
      return done(st);
    ConvGemmArgs a;
    gemm_launch_args(&tmp, L, B, T, bufs, bb, a);
    if ((st = launch_gemm(&tmp, L, map, smap, a, stream)) != VOC_OK) return done(st);
  }
  voc::rows_to_cf_kernel<<<dim3((T + 255) / 256, Cp / 4, B), 256, 0, stream>>>(
      static_cast<const float *>(bufs[BUF_FY]), T, Tp, Cp, C, y_dev);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return done(cuda_fail(&tmp, e, "residual unit"));
  int word = 0;
  cudaMemcpy(&word, tmp.err_dev, sizeof(int), cudaMemcpyDeviceToHost);
  if (word) return done(fail(&tmp, VOC_DEVICE_TIMEOUT, "a kernel gave up a bounded wait"));
  return done(VOC_OK);
}

VOC_API int vocoder_profile_count(const vocoder *ctx) {
  return (ctx && ctx->prof_ready) ? ctx->prof_n : 0;
}

VOC_API voc_status vocoder_profile_entry(vocoder *ctx, int index, const char **name, double *ms,
                                         double *flops, double *bytes) {
  if (!ctx) return fail(nullptr, VOC_INVALID_ARG, "ctx is NULL");
  if (!ctx->prof_ready || index < 0 || index >= ctx->prof_n)
    return fail(ctx, VOC_INVALID_ARG, "no profile entry " + std::to_string(index));
  if (ctx->prof_ms[index] < 0.f) {
    cudaError_t e = cudaEventSynchronize(ctx->events[2 * index + 1]);
    if (e == cudaSuccess)
      e = cudaEventElapsedTime(&ctx->prof_ms[index], ctx->events[2 * index], ctx->events[2 * index + 1]);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "profile event");
  }
  if (name) *name = ctx->prof_names[index].c_str();
  if (ms) *ms = ctx->prof_ms[index];
  if (flops) *flops = ctx->prof_flops[index];
  if (bytes) *bytes = ctx->prof_bytes[index];
  return VOC_OK;
}

VOC_API voc_status vocoder_profile_impl_bytes(vocoder *ctx, int index, double *bytes) {
  if (!ctx) return fail(nullptr, VOC_INVALID_ARG, "ctx is NULL");
  if (!bytes) return fail(ctx, VOC_INVALID_ARG, "bytes is NULL");
  if (!ctx->prof_ready || index < 0 || index >= ctx->prof_n)
    return fail(ctx, VOC_INVALID_ARG, "no profile entry " + std::to_string(index));
  *bytes = ctx->prof_impl[index];
  return VOC_OK;
}

VOC_API const char *vocoder_last_error(const vocoder *ctx) {
  return ctx ? ctx->err.c_str() : g_err.c_str();
}

VOC_API voc_status vocoder_set_wait_budget(vocoder *ctx, long long cycles) {
  if (!ctx) return fail(nullptr, VOC_INVALID_ARG, "ctx is NULL");
  if (cycles < 0) return fail(ctx, VOC_INVALID_ARG, "wait budget must be >= 0");
  ctx->wait_budget = cycles == 0 ? kWaitBudget : cycles;
  return VOC_OK;
}

VOC_API voc_status vocoder_set_cancel_flag(vocoder *ctx, const volatile int *flag) {
  if (!ctx) return fail(nullptr, VOC_INVALID_ARG, "ctx is NULL");
  ctx->cancel = flag;
  return VOC_OK;
}

VOC_API void vocoder_debug_fail_allocation(int n) { g_fail_countdown.store(n < 0 ? -1 : n); }

VOC_API long long vocoder_debug_live_allocations(void) { return g_live_allocs.load(); }

// ------------------------------------------------------------------ stateful streaming
// Causal decoders only (VOC_PAD_CAUSAL): every layer looks left only, so decoding a
// sequence chunk by chunk, with each layer's last input rows carried from one chunk to the
// next, reproduces the whole-sequence decode exactly (qwentts.cpp Architecture,
// "Streaming decode (stateful path)").  Each layer reads a dedicated hi/lo input buffer
// whose planes hold `ctx` rows of left context (the layer's halo, (K-1)*dilation rows for
// a k-tap conv, one row for a transposed conv) followed by the chunk's new rows; the
// output head's fp32 input likewise.  The contexts are saved after each chunk and restored
// before the next; all of them start at zero, which matches the zero padding of a decode
// that starts at frame 0.  Every layer runs with the plan of the context's whole-sequence
// decode, so the results are identical, bit for bit.
struct vocoder_stream {
  vocoder *ctx = nullptr;
  int B = 0, max_frames = 0;
  struct LayerIO {
    uint8_t *in = nullptr;      // hi/lo input planes: ctx rows, then up to max_frames*rate rows
    long long plane = 0;        // rows per plane
    int ctx_rows = 0;
    int rate = 1;               // input rows per latent frame
    int consumer = -1;          // layer reading this layer's hi/lo output (-1: none)
    CUtensorMap map{}, smap{};
  };
  std::vector<LayerIO> io;
  uint8_t *fy = nullptr;        // fp32 residual stream, planes of max_frames*rate rows
  size_t fy_bytes = 0;
  uint8_t *head_in = nullptr;   // Snake'd fp32 input of the head: ctx rows, then new rows
  long long head_plane = 0;
  int head_ctx = 0;
  uint8_t *state = nullptr;     // all saved contexts, one contiguous block
  size_t state_bytes = 0;
  voc::RowCopyJob *jobs = nullptr;  // device: restore jobs, then save jobs
  int n_restore = 0, n_save = 0, max_job_elems = 0;
  // CUDA-graph replay: the launches of one chunk, captured once per chunk size on `cap`
  // over the staging buffers (the caller's latent is copied in, the audio copied out)
  float *lat_stage = nullptr, *aud_stage = nullptr;
  cudaStream_t cap = nullptr;
  std::vector<cudaGraphExec_t> graphs;  // [frames], null until first used
  uint8_t *block = nullptr;     // the single device allocation holding all of the above
};

namespace {
voc_status stream_fail(voc_status st, const std::string &msg) { return fail(nullptr, st, msg); }
}  // namespace

VOC_API voc_status vocoder_stream_create(vocoder *ctx, int B, int max_frames,
                                         vocoder_stream **out) {
  if (!out) return stream_fail(VOC_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!ctx) return stream_fail(VOC_INVALID_ARG, "ctx is NULL");
  if (ctx->desc.padding != VOC_PAD_CAUSAL)
    return stream_fail(VOC_UNSUPPORTED, "streaming needs a causal decoder (VOC_PAD_CAUSAL)");
  if (B < 1 || max_frames < 1 || (long long)max_frames * ctx->hop > 0x7FFFFFFFLL)
    return stream_fail(VOC_INVALID_ARG, "invalid B / max_frames");
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != ctx->device) return stream_fail(VOC_INVALID_ARG, "current device differs from the context's");

  vocoder_stream *s = new vocoder_stream();
  s->ctx = ctx, s->B = B, s->max_frames = max_frames;
  const int nl = static_cast<int>(ctx->layers.size());
  s->io.resize(nl);
  // geometry: context rows, input rate, consumer of each hi/lo output
  for (int l = 0; l < nl; ++l) {
    const Layer &L = ctx->layers[l];
    vocoder_stream::LayerIO &io = s->io[l];
    io.ctx_rows = -L.g.off_min;
    io.rate = static_cast<int>(level_len(ctx, L.level, 1));
    io.plane = pitch8(io.ctx_rows + (long long)max_frames * io.rate);
    if (L.hl_buf >= 0)
      for (int m = l + 1; m < nl; ++m)
        if (ctx->layers[m].in_buf == L.hl_buf) {
          io.consumer = m;
          break;
        }
  }
  const OutHead &h = ctx->head;
  s->head_ctx = h.pad_left;
  s->head_plane = s->head_ctx + (long long)max_frames * ctx->hop;
  // sizes of the buffers inside one allocation (each 256-byte aligned)
  auto hl_bytes = [&](int l) {
    return rupz((size_t)B * 2 * (ctx->layers[l].Cp_in / 8) * s->io[l].plane * 16, 256);
  };
  size_t fy_rows = 0;
  for (int l = 0; l < nl; ++l) {
    const Layer &L = ctx->layers[l];
    const int lv_out = L.convT ? L.level + 1 : L.level;
    fy_rows = std::max(fy_rows, (size_t)B * (L.Cp_out / 4) *
                                    (size_t)pitch8((long long)max_frames * level_len(ctx, lv_out, 1)));
  }
  s->fy_bytes = rupz(fy_rows * 16, 256);
  const size_t head_bytes = rupz((size_t)B * (h.Cp / 4) * s->head_plane * 16, 256);
  size_t state_bytes = 0;
  std::vector<size_t> state_off(nl + 1, 0);
  for (int l = 0; l < nl; ++l) {
    state_off[l] = state_bytes;
    state_bytes += rupz((size_t)B * 2 * (ctx->layers[l].Cp_in / 8) * s->io[l].ctx_rows * 16, 256);
  }
  state_off[nl] = state_bytes;  // head context
  state_bytes += rupz((size_t)B * (h.Cp / 4) * s->head_ctx * 16, 256);
  s->state_bytes = state_bytes;
  size_t total = s->fy_bytes + head_bytes + state_bytes;
  for (int l = 0; l < nl; ++l) total += hl_bytes(l);
  const size_t jobs_bytes = rupz(sizeof(voc::RowCopyJob) * 2 * (nl + 1), 256);
  total += jobs_bytes;
  const size_t lat_bytes = rupz((size_t)B * ctx->desc.latent_channels * max_frames * 4, 256);
  const size_t aud_bytes = rupz((size_t)B * max_frames * ctx->hop * 4, 256);
  total += lat_bytes + aud_bytes;
  cudaError_t e = dev_alloc(reinterpret_cast<void **>(&s->block), total);
  if (e != cudaSuccess) {
    delete s;
    return cuda_fail(nullptr, e, "cudaMalloc (stream buffers)");
  }
  uint8_t *cur = s->block;
  for (int l = 0; l < nl; ++l) s->io[l].in = cur, cur += hl_bytes(l);
  s->fy = cur, cur += s->fy_bytes;
  s->head_in = cur, cur += head_bytes;
  s->state = cur, cur += state_bytes;
  s->lat_stage = reinterpret_cast<float *>(cur), cur += lat_bytes;
  s->aud_stage = reinterpret_cast<float *>(cur), cur += aud_bytes;
  s->jobs = reinterpret_cast<voc::RowCopyJob *>(cur);
  // copy jobs: restore (state -> context rows), then save (last ctx rows of [ctx | new] -> state)
  std::vector<voc::RowCopyJob> restore, save;
  auto add = [&](uint8_t *buf, long long plane, uint8_t *st, int ctx_rows, int rate, int planes) {
    if (ctx_rows <= 0) return;
    voc::RowCopyJob r{};
    r.src = reinterpret_cast<const uint4 *>(st), r.dst = reinterpret_cast<uint4 *>(buf);
    r.src_L = ctx_rows, r.dst_L = plane, r.src_row0 = 0, r.src_rate = 0, r.dst_row0 = 0;
    r.rows = ctx_rows, r.planes = planes;
    restore.push_back(r);
    voc::RowCopyJob w{};
    w.src = reinterpret_cast<const uint4 *>(buf), w.dst = reinterpret_cast<uint4 *>(st);
    w.src_L = plane, w.dst_L = ctx_rows, w.src_row0 = 0, w.src_rate = rate, w.dst_row0 = 0;
    w.rows = ctx_rows, w.planes = planes;
    save.push_back(w);
    s->max_job_elems = std::max(s->max_job_elems, ctx_rows * planes);
  };
  for (int l = 0; l < nl; ++l)
    add(s->io[l].in, s->io[l].plane, s->state + state_off[l], s->io[l].ctx_rows, s->io[l].rate,
        B * 2 * (ctx->layers[l].Cp_in / 8));
  add(s->head_in, s->head_plane, s->state + state_off[nl], s->head_ctx, static_cast<int>(ctx->hop),
      B * (h.Cp / 4));
  s->n_restore = static_cast<int>(restore.size());
  s->n_save = static_cast<int>(save.size());
  std::vector<voc::RowCopyJob> all(restore);
  all.insert(all.end(), save.begin(), save.end());
  voc_status st = VOC_OK;
  if (!all.empty()) {
    e = cudaMemcpy(s->jobs, all.data(), sizeof(voc::RowCopyJob) * all.size(), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) st = cuda_fail(nullptr, e, "cudaMemcpy (stream jobs)");
  }
  if (st == VOC_OK) {
    e = cudaMemset(s->state, 0, state_bytes);  // zero context = the decode's zero padding
    if (e != cudaSuccess) st = cuda_fail(nullptr, e, "cudaMemset (stream state)");
  }
  // TMA descriptors: fixed buffers and plane lengths
  for (int l = 0; l < nl && st == VOC_OK; ++l) {
    const Layer &L = ctx->layers[l];
    st = encode_map(ctx, &s->io[l].map, s->io[l].in, L.Cp_in, s->io[l].plane, B, L.g.rows, L.g.KB / 8);
    if (st == VOC_OK && L.skip_buf >= 0)
      st = encode_skip_map(ctx, &s->io[l].smap, s->fy, L.Cp_out,
                           pitch8((long long)max_frames * level_len(ctx, L.level, 1)), B, L.cw);
    if (st != VOC_OK) g_err = ctx->err;
  }
  if (st == VOC_OK) {
    e = cudaStreamCreateWithFlags(&s->cap, cudaStreamNonBlocking);
    if (e != cudaSuccess) st = cuda_fail(nullptr, e, "cudaStreamCreateWithFlags");
  }
  if (st != VOC_OK) {
    if (s->cap) cudaStreamDestroy(s->cap);
    dev_free(s->block);
    delete s;
    return st;
  }
  s->graphs.assign(max_frames + 1, nullptr);
  *out = s;
  return VOC_OK;
}

VOC_API voc_status vocoder_stream_reset(vocoder_stream *s, voc_stream_t stream) {
  if (!s) return stream_fail(VOC_INVALID_ARG, "stream is NULL");
  cudaError_t e = cudaMemsetAsync(s->state, 0, s->state_bytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(s->ctx, e, "cudaMemsetAsync (stream state)");
  return VOC_OK;
}

namespace {
// The launches of one chunk: restore the contexts, the latent's hi/lo split, every layer, the
// head, save the contexts.
voc_status stream_launches(vocoder_stream *s, const float *latent_dev, int frames,
                           float *audio_dev, cudaStream_t stream) {
  vocoder *ctx = s->ctx;
  const int B = s->B;
  const int nl = static_cast<int>(ctx->layers.size());
  auto copies = [&](int first, int n) -> voc_status {
    if (n == 0) return VOC_OK;
    const int blocks = std::max(1, std::min((s->max_job_elems + 255) / 256, 64));
    cudaError_t ce = launch_pdl(voc::row_copy_kernel, dim3(blocks, n), dim3(256), 0, stream,
                                static_cast<const voc::RowCopyJob *>(s->jobs + first), frames);
    return ce == cudaSuccess ? VOC_OK : cuda_fail(ctx, ce, "launch row_copy");
  };
  voc_status st = copies(0, s->n_restore);  // contexts of the previous chunk
  if (st != VOC_OK) return st;
  st = launch_prep(ctx, latent_dev, B, ctx->desc.latent_channels, frames, ctx->Cp_lat, nullptr,
                   nullptr, reinterpret_cast<__nv_bfloat16 *>(s->io[0].in), stream, s->io[0].ctx_rows,
                   s->io[0].plane);
  if (st != VOC_OK) return st;
  void *dummy[BUF_COUNT] = {nullptr, nullptr, nullptr, nullptr};
  for (int l = 0; l < nl; ++l) {
    const Layer &L = ctx->layers[l];
    const vocoder_stream::LayerIO &io = s->io[l];
    ConvGemmArgs a;
    gemm_launch_args(ctx, L, B, frames, dummy, 0, a);  // rows and tiles of this chunk
    set_in_row0(L, a, io.ctx_rows);
    a.rows_pad = a.rows_valid;  // causal: no layer reads past its chunk's rows
    a.skip = L.skip_buf >= 0 ? reinterpret_cast<const float *>(s->fy) : nullptr;
    a.out_hl = nullptr, a.out_f32 = nullptr;
    if (L.hl_buf >= 0) {
      if (io.consumer < 0) return fail(ctx, VOC_UNSUPPORTED, L.name + ": no consumer of its output");
      const vocoder_stream::LayerIO &c = s->io[io.consumer];
      a.out_hl = reinterpret_cast<__nv_bfloat16 *>(c.in);
      a.hl_row0 = c.ctx_rows;
      a.hl_L = static_cast<int>(c.plane);
      a.hl_elems = (long long)B * 2 * (L.Cp_out / 8) * c.plane * 8;
    }
    if (L.f32_buf >= 0) {
      if (L.epi_flags & voc::EPI_F32_SNAKE) {  // the head's input, after its context rows
        a.out_f32 = reinterpret_cast<float *>(s->head_in);
        a.f32_row0 = s->head_ctx;
        a.f32_L = static_cast<int>(s->head_plane);
        a.f32_elems = (long long)B * (L.Cp_out / 4) * s->head_plane * 4;
      } else {
        const int lv_out = L.convT ? L.level + 1 : L.level;
        a.out_f32 = reinterpret_cast<float *>(s->fy);
        a.f32_row0 = 0;
        a.f32_L = static_cast<int>(pitch8((long long)s->max_frames * level_len(ctx, lv_out, 1)));
        a.f32_elems = static_cast<long long>(s->fy_bytes / 4);
      }
    }
    a.L_a = static_cast<int>(io.plane);
    st = launch_gemm(ctx, L, io.map, io.smap, a, stream,
                     pitch8((long long)s->max_frames * level_len(ctx, L.level, 1)),
                     static_cast<long long>(s->fy_bytes / 4));
    if (st != VOC_OK) return st;
#ifdef VOC_CHECKS
    if ((st = check_launch(ctx, "stream " + L.name, stream)) != VOC_OK) return st;
#endif
  }
  const long long Lf = (long long)frames * ctx->hop;
  st = launch_out_head(ctx, ctx->head, reinterpret_cast<const float *>(s->head_in), B, Lf, audio_dev,
                       stream, s->head_ctx, s->head_plane);
  if (st != VOC_OK) return st;
  return copies(s->n_restore, s->n_save);  // this chunk's contexts for the next one
}
}  // namespace

VOC_API voc_status vocoder_stream_decode(vocoder_stream *s, const float *latent_dev, int frames,
                                         float *audio_dev, voc_stream_t stream_, unsigned flags) {
  if (!s) return stream_fail(VOC_INVALID_ARG, "stream is NULL");
  vocoder *ctx = s->ctx;
  if (!latent_dev || !audio_dev) return fail(ctx, VOC_INVALID_ARG, "latent / audio NULL");
  if (frames < 1 || frames > s->max_frames)
    return fail(ctx, VOC_INVALID_ARG, "frames out of [1, max_frames]");
  if (flags & ~static_cast<unsigned>(VOC_FLAG_SYNC))
    return fail(ctx, VOC_INVALID_ARG, "only VOC_FLAG_SYNC is accepted");
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != ctx->device) return fail(ctx, VOC_INVALID_ARG, "current device differs from the context's");
  if (cancelled(ctx)) return fail(ctx, VOC_CANCELLED, "cancelled: the caller's cancel flag is set");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaError_t e;
  voc_status st;
#ifdef VOC_CHECKS
  // the self-checking build synchronises after every launch, which a capture cannot hold
  st = stream_launches(s, latent_dev, frames, audio_dev, stream);
  if (st != VOC_OK) return st;
#else
  // A chunk is a fixed sequence of about 40 small launches: it is captured once per chunk
  // size into a CUDA graph over the staging buffers and replayed on the caller's stream.
  if (!s->graphs[frames]) {
    e = cudaStreamBeginCapture(s->cap, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamBeginCapture");
    st = stream_launches(s, s->lat_stage, frames, s->aud_stage, s->cap);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(s->cap, &g);
    if (st == VOC_OK && e != cudaSuccess) st = cuda_fail(ctx, e, "cudaStreamEndCapture");
    cudaGraphExec_t exec = nullptr;
    if (st == VOC_OK) {
      e = cudaGraphInstantiate(&exec, g, 0);
      if (e != cudaSuccess) st = cuda_fail(ctx, e, "cudaGraphInstantiate");
    }
    if (g) cudaGraphDestroy(g);
    if (st != VOC_OK) {
      (void)cudaGetLastError();
      return st;
    }
    s->graphs[frames] = exec;
  }
  const size_t lat_bytes = (size_t)s->B * ctx->desc.latent_channels * frames * 4;
  const size_t aud_bytes = (size_t)s->B * frames * ctx->hop * 4;
  e = cudaMemcpyAsync(s->lat_stage, latent_dev, lat_bytes, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess) e = cudaGraphLaunch(s->graphs[frames], stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(audio_dev, s->aud_stage, aud_bytes, cudaMemcpyDeviceToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stream chunk (graph replay)");
#endif
  if (flags & VOC_FLAG_SYNC) {
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
    int word = 0;
    cudaMemcpy(&word, ctx->err_dev, sizeof(int), cudaMemcpyDeviceToHost);
    if (word) return fail(ctx, VOC_DEVICE_TIMEOUT, "a kernel gave up a bounded wait");
  }
  return VOC_OK;
}

VOC_API void vocoder_stream_destroy(vocoder_stream *s) {
  if (!s) return;
  for (cudaGraphExec_t g : s->graphs)
    if (g) cudaGraphExecDestroy(g);
  if (s->cap) cudaStreamDestroy(s->cap);
  dev_free(s->block);
  delete s;
}

// ------------------------------------------------------------------ output stage
// minimaxmusic.cpp Architecture, "Post-processing" (see output_stage.cuh).
namespace {
constexpr size_t kWavScratch = 256 + 2048 * 4;  // select state, then one 2048-bin histogram

__global__ void select_init_kernel(voc::SelectState *st, unsigned long long k) {
  if (threadIdx.x == 0) {
    st->k = k, st->prefix = 0u, st->mask = 0u, st->level = 0.f, st->gain = 1.f;
  }
}
}  // namespace

VOC_API size_t vocoder_wav_bytes(int n_ch, long long len, int bits) {
  if (n_ch < 1 || n_ch > 65535 || len < 0 || (bits != 16 && bits != 24 && bits != 32)) return 0;
  const unsigned long long data = (unsigned long long)n_ch * (unsigned long long)len * (bits / 8);
  if (36 + data > 0xFFFFFFFFull) return 0;  // the RIFF size field is 32 bits
  return static_cast<size_t>(44 + data);
}

VOC_API size_t vocoder_wav_scratch_bytes(void) { return kWavScratch; }

VOC_API voc_status vocoder_encode_wav(const float *planar_dev, int n_ch, long long len,
                                      int sample_rate, int bits, int peak_clip, void *out_dev,
                                      size_t out_bytes, void *scratch_dev, size_t scratch_bytes,
                                      voc_stream_t stream_) {
  const size_t need = vocoder_wav_bytes(n_ch, len, bits);
  if (!need) return fail(nullptr, VOC_INVALID_ARG, "bad channel count, length or bits (16, 24, 32)");
  if (sample_rate <= 0 || peak_clip < 0 || peak_clip > 1000000)
    return fail(nullptr, VOC_INVALID_ARG, "sample_rate must be > 0 and peak_clip in [0, 1e6]");
  if ((!planar_dev && len > 0) || !out_dev || (reinterpret_cast<uintptr_t>(out_dev) & 3))
    return fail(nullptr, VOC_INVALID_ARG, "planar / out NULL, or out not 4-byte aligned");
  if (out_bytes < need) return fail(nullptr, VOC_WORKSPACE_TOO_SMALL, "out smaller than vocoder_wav_bytes");
  if (bits != 32 && (!scratch_dev || scratch_bytes < kWavScratch ||
                     (reinterpret_cast<uintptr_t>(scratch_dev) & 255)))
    return fail(nullptr, VOC_WORKSPACE_TOO_SMALL, "scratch NULL, unaligned or smaller than vocoder_wav_scratch_bytes");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const long long n = (long long)n_ch * len;
  const uint32_t bps = static_cast<uint32_t>(bits / 8);
  const uint32_t data = static_cast<uint32_t>(n * bps);
  voc::WavHeader h{};
  h.w[0] = 0x46464952u;  // "RIFF"
  h.w[1] = 36u + data;
  h.w[2] = 0x45564157u;  // "WAVE"
  h.w[3] = 0x20746d66u;  // "fmt "
  h.w[4] = 16u;
  h.w[5] = (bits == 32 ? 3u : 1u) | (static_cast<uint32_t>(n_ch) << 16);
  h.w[6] = static_cast<uint32_t>(sample_rate);
  h.w[7] = static_cast<uint32_t>(sample_rate) * static_cast<uint32_t>(n_ch) * bps;
  h.w[8] = (static_cast<uint32_t>(n_ch) * bps) | (static_cast<uint32_t>(bits) << 16);
  h.w[9] = 0x61746164u;  // "data"
  h.w[10] = data;
  uint8_t *out = static_cast<uint8_t *>(out_dev);
  voc::wav_header_kernel<<<1, 32, 0, stream>>>(h, out);
  voc::SelectState *st = static_cast<voc::SelectState *>(scratch_dev);
  if (bits != 32 && n > 0) {
    // rank of the level: ceil(q * n) with q = 1 - peak_clip / 1e6, in double (as specified)
    const double q = 1.0 - static_cast<double>(peak_clip) / 1e6;
    long long k = static_cast<long long>(std::ceil(q * static_cast<double>(n)));
    k = std::min(std::max(k, 1LL), n);
    unsigned int *hist = reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(scratch_dev) + 256);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 4LL * std::max(sms, 1)));
    cudaMemsetAsync(hist, 0, 2048 * 4, stream);
    select_init_kernel<<<1, 32, 0, stream>>>(st, static_cast<unsigned long long>(k));
    voc::select_hist_kernel<11><<<blocks, 256, 0, stream>>>(planar_dev, n, 21, st, hist);
    voc::select_pick_kernel<11><<<1, 256, 0, stream>>>(st, hist, 21, 0);
    voc::select_hist_kernel<11><<<blocks, 256, 0, stream>>>(planar_dev, n, 10, st, hist);
    voc::select_pick_kernel<11><<<1, 256, 0, stream>>>(st, hist, 10, 0);
    voc::select_hist_kernel<10><<<blocks, 256, 0, stream>>>(planar_dev, n, 0, st, hist);
    voc::select_pick_kernel<10><<<1, 256, 0, stream>>>(st, hist, 0, 1);
  }
  if (n > 0)
    voc::wav_encode_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
        planar_dev, n_ch, len, static_cast<int>(bps), st, out + 44);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "launch output stage");
  return VOC_OK;
}

// =================================================================== mirror encoder
// minimaxmusic.cpp Architecture, "Flow VAE": conv_in, blocks of residual units each followed
// by Snake and a strided conv (k = 2s, stride s, pad s/2), Snake, conv_out and the posterior
// mean projection, all non-causal, on the decoder's conv kernel.  A strided conv runs as a
// 3-tap stride-1 conv over its input split into s phases: output row u reads input rows
// u s + k - s/2 for k < 2s, i.e. rows u + du of phase r for du in {-1, 0, 1}; the residual
// unit before it writes its hi/lo output in that phase-split layout, so the conv reads
// s * Cp(C) channels of L / s rows through the ordinary tensor maps.
struct vocoder_encoder {
  vocoder core;  // device, error words, precision, allocations, profile records
  voc_enc_desc desc{};
  std::vector<int> strides, widths, dils;
  long long hop = 1;
  int Cp_audio = 0, Cp_lat = 0;
  std::vector<Layer> layers;
  std::vector<long long> div;  // per layer: GEMM rows per item = L / div
  std::vector<int> split;      // per layer: 0, or the stride s of its phase-split hi/lo output
  // TMA descriptors for the last (workspace, B, L)
  void *map_ws = nullptr;
  int map_B = -1;
  long long map_L = -1;
  std::vector<CUtensorMap> maps, skip_maps;
};

namespace {

long long rup_ll(long long x, long long m) { return (x + m - 1) / m * m; }

// Device of the current thread: sm_103 check, SM count, the kernels' error words.
voc_status init_device(vocoder *ctx) {
  cudaError_t e = cudaGetDevice(&ctx->device);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaDeviceGetAttribute");
  int cc_major = 0, cc_minor = 0;
  cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, ctx->device);
  cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, ctx->device);
  if (cc_major != 10 || cc_minor != 3)
    return fail(ctx, VOC_UNSUPPORTED, "the library is compiled for sm_103 (GB300) only");
  e = dev_alloc(reinterpret_cast<void **>(&ctx->err_dev), 8 * sizeof(int));  // [0] error word, [1] finite flag, [4..7] checks
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaMalloc");
  ctx->allocs.push_back(ctx->err_dev);
  ctx->flag_dev = ctx->err_dev + 1;
  e = cudaMemset(ctx->err_dev, 0, 8 * sizeof(int));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaMemset");
  return VOC_OK;
}

bool check_enc_desc(const voc_enc_desc *d, std::string &why) {
  if (!d) return why = "desc is NULL", false;
  if (d->abi_version != VOC_ABI_VERSION)
    return why = "abi_version " + std::to_string(d->abi_version) + " != " +
                 std::to_string(VOC_ABI_VERSION),
           false;
  if (d->in_channels < 1 || d->in_channels > 16) return why = "in_channels must be in [1, 16]", false;
  if (d->channels0 < 1 || d->channels0 > 8192) return why = "channels0", false;
  if (d->latent_channels < 1 || d->latent_channels > 8192) return why = "latent_channels", false;
  for (int k : {d->in_kernel, d->res_kernel, d->out_kernel})
    if (k < 1 || k > 15 || k % 2 == 0) return why = "kernel sizes must be odd in [1, 15]", false;
  if (d->n_stages < 1 || d->n_stages > 8) return why = "n_stages", false;
  if (!d->strides || !d->widths) return why = "strides / widths NULL", false;
  if (d->n_dilations < 1 || d->n_dilations > 4 || !d->dilations) return why = "dilations", false;
  if (d->precision != VOC_PREC_BF16X3 && d->precision != VOC_PREC_F16W &&
      d->precision != VOC_PREC_BF16W)
    return why = "precision", false;
  if (d->snake != VOC_SNAKE && d->snake != VOC_SNAKE_BETA) return why = "snake", false;
  for (int i = 0; i < d->n_stages; ++i) {
    if (d->strides[i] < 1 || d->strides[i] > 16) return why = "stride out of [1, 16]", false;
    if (d->widths[i] < 1 || d->widths[i] > 8192) return why = "width out of range", false;
  }
  for (int j = 0; j < d->n_dilations; ++j)
    if (d->dilations[j] < 1 || d->dilations[j] * (d->res_kernel - 1) > 120)
      return why = "dilation * (res_kernel - 1) must be in [1, 120]", false;
  return true;
}

int enc_param_count(const voc_enc_desc *d) {
  return 2 + d->n_stages * (6 * d->n_dilations + 3) + 5;
}

// kind of every canonical encoder parameter: 'w' weight, 'b' bias, 'a' Snake parameters
std::string enc_param_kinds(const voc_enc_desc *d) {
  std::string k = "wb";
  for (int i = 0; i < d->n_stages; ++i) {
    for (int j = 0; j < d->n_dilations; ++j) k += "awbawb";
    k += "awb";
  }
  return k + "awbwb";
}

// Largest hi/lo or fp32 plane set of one encode, in bytes: B items of max over the
// levels of Cp(C) x rows (the phase-split outputs fill whole groups of 8 s rows).
size_t enc_buf_bytes(const vocoder_encoder *enc, int B, long long L) {
  long long Li = L;
  int C = enc->desc.channels0;
  size_t m = (size_t)pitch8(L) * (size_t)std::max(enc->Cp_audio, rup(C, 16));
  for (int i = 0; i < enc->desc.n_stages; ++i) {
    const int s = enc->strides[i];
    m = std::max(m, (size_t)rup_ll(Li, 8LL * s) * (size_t)rup(C, 16));
    Li /= s;
    C = enc->widths[i];
    m = std::max(m, (size_t)pitch8(Li) * (size_t)rup(C, 16));
  }
  m = std::max(m, (size_t)pitch8(Li) * (size_t)enc->Cp_lat);
  return rupz(m * (size_t)B * 4, 256);
}

// Split k for an encoder layer with `rows` GEMM rows per item: the number of k ranges (1..4)
// that fills the SMs best when its tiles alone would leave many idle (the deep layers of the
// low-rate blocks).  Only for layers without a residual input or phase-split output and with
// streamed weights; each range holds at least one k-block and the raw sums of all ranges stay
// within 64 MB (L2-sized) and the workspace slot that holds them.
constexpr size_t kSplitPartMax = 64ull << 20;
// audio channels up to which the encoder's conv_in runs directly (audio_conv_in_kernel)
constexpr int kAudioDirectMaxC = 4;
int enc_ksplit(const vocoder_encoder *enc, size_t i, int B, long long rows, size_t slot_bytes) {
  const Layer &L = enc->layers[i];
  if (L.direct || L.skip_buf >= 0 || enc->split[i] || L.g.b_resident || L.g.nkb < 2) return 1;
  const long long jobs = (long long)B * ((rows + voc::kTileM - 1) / voc::kTileM) * L.g.n_tiles;
  const long long sms = std::max(1, enc->core.num_sms);
  auto eff = [&](long long S) {
    const long long n = S * jobs;
    return (double)n / (double)(((n + sms - 1) / sms) * sms);
  };
  const size_t part1 = (size_t)B * L.Cp_out * (size_t)pitch8(rows) * 4;
  int best = 1;
  for (int S = 2; S <= std::min(4, L.g.nkb); ++S) {
    if ((size_t)S * part1 > std::min(kSplitPartMax, slot_bytes)) break;
    if (eff(S) > eff(best) + 1e-9) best = S;
  }
  return eff(best) >= 1.25 * eff(1) ? best : 1;  // at least a quarter more SMs busy
}

// Cost of an encoder layer with L_in GEMM rows per item, as layer_cost for the decoder: a
// strided conv counts its 2s taps over the C real channels (not the zero taps of its 3-tap
// form) and reads its s L_in input rows once; `alg` counts the real channels' inputs read
// once and outputs written once (the output of a split-k layer is its reduce launch's).
void enc_layer_cost(const Layer &L, int B, long long L_in, bool split_k, double &flops,
                    double &alg, double &impl) {
  const double rows = (double)B * (double)L_in;
  const double k = L.down_s ? 2.0 * L.down_s : (double)L.K + (L.ru ? 1.0 : 0.0);
  const double cin = L.down_s ? (double)L.down_c : (double)L.Cin;
  flops = 2.0 * cin * L.Cout * k * rows;
  alg = 4.0 * cin * rows * (L.down_s ? L.down_s : 1);
  if (L.skip_buf >= 0 && !L.ru) alg += 4.0 * L.Cout * rows;  // a fused unit's skip is its input
  if (!split_k) alg += 4.0 * L.Cout * rows;
  const ConvGemmArgs &g = L.g;
  double by = 4.0 * rows * L.Cp_in + (double)g.n_tiles * (g.taps + (L.ru ? 1 : 0)) * g.nkb * g.b_bytes;
  const double out_elems = rows * L.Cp_out;
  if (L.skip_buf >= 0) by += 4.0 * out_elems;
  if (L.f32_buf >= 0) by += 4.0 * out_elems;
  if (L.hl_buf >= 0) by += 4.0 * out_elems;
  impl = by;
}

}  // namespace

VOC_API int vocoder_encoder_param_count(const voc_enc_desc *desc) {
  std::string why;
  if (!check_enc_desc(desc, why)) return -1;
  return enc_param_count(desc);
}

VOC_API voc_status vocoder_encoder_param_shape(const voc_enc_desc *d, int index, int dims[3],
                                               int *ndim) {
  std::string why;
  if (!check_enc_desc(d, why)) return fail(nullptr, VOC_INVALID_ARG, why);
  if (!dims || !ndim) return fail(nullptr, VOC_INVALID_ARG, "dims / ndim NULL");
  if (index < 0 || index >= enc_param_count(d)) return fail(nullptr, VOC_INVALID_ARG, "index out of range");
  auto set = [&](int nd, int a, int b = 0, int c = 0) {
    *ndim = nd;
    dims[0] = a, dims[1] = b, dims[2] = c;
    return VOC_OK;
  };
  auto snake = [&](int c) { return d->snake == VOC_SNAKE_BETA ? set(2, 2, c) : set(1, c); };
  if (index == 0) return set(3, d->channels0, d->in_channels, d->in_kernel);
  if (index == 1) return set(1, d->channels0);
  int i = index - 2, C = d->channels0;
  const int units = 6 * d->n_dilations;
  for (int s = 0; s < d->n_stages; ++s) {
    const int Co = d->widths[s];
    if (i < units + 3) {
      if (i < units) {
        const int j = i % 6;
        if (j == 0 || j == 3) return snake(C);
        if (j == 1) return set(3, C, C, d->res_kernel);
        if (j == 4) return set(3, C, C, 1);
        return set(1, C);
      }
      if (i == units) return snake(C);
      if (i == units + 1) return set(3, Co, C, 2 * d->strides[s]);
      return set(1, Co);
    }
    i -= units + 3;
    C = Co;
  }
  if (i == 0) return snake(C);
  if (i == 1) return set(3, C, C, d->out_kernel);
  if (i == 2) return set(1, C);
  if (i == 3) return set(3, d->latent_channels, C, 1);
  return set(1, d->latent_channels);
}

VOC_API void vocoder_encoder_destroy(vocoder_encoder *enc) {
  if (!enc) return;
  for (void *p : enc->core.allocs) dev_free(p);
  for (cudaEvent_t e : enc->core.events) cudaEventDestroy(e);
  delete enc;
}

VOC_API voc_status vocoder_encoder_create(const voc_enc_desc *desc, const float *const *params,
                                          int n_params, vocoder_encoder **out) {
  if (!out) return fail(nullptr, VOC_INVALID_ARG, "out is NULL");
  *out = nullptr;
  std::string why;
  if (!check_enc_desc(desc, why)) return fail(nullptr, VOC_INVALID_ARG, "desc: " + why);
  if (!params) return fail(nullptr, VOC_INVALID_ARG, "params is NULL");
  if (n_params != enc_param_count(desc))
    return fail(nullptr, VOC_INVALID_ARG, "n_params " + std::to_string(n_params) + " != " +
                                              std::to_string(enc_param_count(desc)));
  const std::string kinds = enc_param_kinds(desc);
  for (int i = 0; i < n_params; ++i) {
    if (!params[i]) {
      if (kinds[i] == 'b') continue;
      return fail(nullptr, VOC_INVALID_ARG, "params[" + std::to_string(i) + "] is NULL");
    }
    int dims[3], nd;
    vocoder_encoder_param_shape(desc, i, dims, &nd);
    size_t n = 1;
    for (int k = 0; k < nd; ++k) n *= dims[k];
    for (size_t k = 0; k < n; ++k) {
      const float x = params[i][k];
      if (!std::isfinite(x))
        return fail(nullptr, VOC_INVALID_ARG, "params[" + std::to_string(i) + "] not finite");
      if (kinds[i] == 'a' && desc->snake == VOC_SNAKE && !(x > 0.f))
        return fail(nullptr, VOC_INVALID_ARG, "Snake alpha must be positive");
      if (kinds[i] == 'a' && desc->snake == VOC_SNAKE_BETA && !(std::fabs(x) <= 80.f))
        return fail(nullptr, VOC_INVALID_ARG, "SnakeBeta log alpha / log beta must be in [-80, 80]");
    }
  }
  if (!set_kernel_attrs(why)) return fail(nullptr, VOC_CUDA_ERROR, why);

  vocoder_encoder *enc = new vocoder_encoder();
  vocoder *ctx = &enc->core;
  enc->desc = *desc;
  enc->strides.assign(desc->strides, desc->strides + desc->n_stages);
  enc->widths.assign(desc->widths, desc->widths + desc->n_stages);
  enc->dils.assign(desc->dilations, desc->dilations + desc->n_dilations);
  enc->desc.strides = enc->strides.data();
  enc->desc.widths = enc->widths.data();
  enc->desc.dilations = enc->dils.data();
  for (int s : enc->strides) enc->hop *= s;
  enc->Cp_audio = rup(desc->in_channels, 16);
  enc->Cp_lat = rup(desc->latent_channels, 16);
  ctx->prec = desc->precision;
  ctx->use_pair = false;
  // residual units before a block's last one run as one fused kernel, as in the decoder (the
  // decoder's default: with the one-plane precisions the units wider than kRuOnePlaneMinC)
  ctx->fuse_max_c = kFuseDefault;
  if (ctx->prec != VOC_PREC_BF16X3) ctx->fuse_min_c = kRuOnePlaneMinC;
  auto bail = [&](voc_status st) {
    g_err = ctx->err;
    vocoder_encoder_destroy(enc);
    return st;
  };
  voc_status st = init_device(ctx);
  if (st != VOC_OK) return bail(st);

  const int pad = VOC_PAD_SYMMETRIC;
  auto add = [&](Layer &L, bool has_skip, const float *w, const float *b, const SnakeCoef &sn,
                 long long div, int split) {
    L.prec = ctx->prec;
    if (!plan_layer(false, L, pad, has_skip, why))
      return fail(ctx, VOC_UNSUPPORTED, L.name + ": " + why);
    const voc_status s = upload_layer(ctx, ctx->allocs, L, pad, w, b, sn);
    if (s != VOC_OK) return s;
    enc->layers.push_back(L);
    enc->div.push_back(div);
    enc->split.push_back(split > 1 ? split : 0);
    return VOC_OK;
  };
  // hi/lo buffers H0, H1, HB and the fp32 residual stream FY, used as in the decoder: a
  // layer never writes the hi/lo buffer it reads with a halo
  auto other = [](int a) { return a == BUF_H0 ? (int)BUF_H1 : (int)BUF_H0; };
  const int nd = desc->n_dilations;
  int C = desc->channels0;
  long long div = 1;
  int cur = BUF_H1;
  {  // conv_in (no Snake in front); its epilogue applies the first residual unit's Snake1
    Layer L;
    L.name = "conv_in";
    L.Cin = desc->in_channels, L.Cout = C, L.K = desc->in_kernel, L.dil = 1;
    L.in_buf = BUF_H0, L.f32_buf = BUF_FY, L.hl_buf = cur;
    if (desc->in_channels <= kAudioDirectMaxC && desc->in_kernel <= 15) {  // weights fit kAudioMaxW
      // direct fp32 kernel on the audio: weights as given (rounded like every conv weight in
      // the one-plane precisions), the epilogue vectors of a plain conv
      L.direct = true;
      L.prec = ctx->prec;
      L.Cp_in = rup(L.Cin, 16), L.Cp_out = rup(L.Cout, 16);
      L.g.N_total = L.Cp_out, L.g.Cp_out = L.Cp_out;
      std::vector<float> wf((size_t)L.Cout * L.Cin * L.K);
      for (size_t k = 0; k < wf.size(); ++k) {
        const float x = params[0][k];
        wf[k] = ctx->prec == VOC_PREC_F16W    ? __half2float(__float2half_rn(x))
                : ctx->prec == VOC_PREC_BF16W ? bf2f(f2bf(x))
                                              : x;
      }
      if ((st = upload(ctx, ctx->allocs, wf, &L.wf_dev)) != VOC_OK) return bail(st);
      if ((st = upload_columns(ctx, ctx->allocs, L, pad, params[1],
                               snake_coef(params[2], C, desc->snake))) != VOC_OK)
        return bail(st);
      enc->layers.push_back(L);
      enc->div.push_back(div);
      enc->split.push_back(0);
    } else if ((st = add(L, false, params[0], params[1], snake_coef(params[2], C, desc->snake), div,
                         0)) != VOC_OK) {
      return bail(st);
    }
  }
  int p = 2;
  for (int i = 0; i < desc->n_stages; ++i) {
    const int s = enc->strides[i], Co = enc->widths[i];
    const std::string blk = "b" + std::to_string(i);
    for (int j = 0; j < nd; ++j) {
      const float *w1 = params[p + 1], *b1 = params[p + 2];
      const SnakeCoef a2 = snake_coef(params[p + 3], C, desc->snake);
      const float *w2 = params[p + 4], *b2 = params[p + 5];
      p += 6;
      // the next unit's Snake1, or (last unit) the Snake in front of the strided conv
      const SnakeCoef next = snake_coef(params[p], C, desc->snake);
      const int tmp = other(cur);
      Layer R;  // the whole unit in one kernel; the last unit of a block writes the phase-split
                // input of the strided conv, an epilogue form of the conv kernel only
      R.name = blk + "r" + std::to_string(j) + ".ru";
      R.Cin = C, R.Cout = C, R.K = desc->res_kernel, R.dil = enc->dils[j];
      R.prec = ctx->prec;
      if (j < nd - 1 && rup(C, 16) <= ctx->fuse_max_c && rup(C, 16) >= ctx->fuse_min_c &&
          plan_ru(R, pad, why)) {
        R.in_buf = cur, R.skip_buf = BUF_FY, R.f32_buf = BUF_FY, R.hl_buf = tmp;
        if ((st = upload_ru(ctx, ctx->allocs, R, pad, w1, b1, a2, w2, b2, next)) != VOC_OK)
          return bail(st);
        enc->layers.push_back(R);
        enc->div.push_back(div);
        enc->split.push_back(0);
        cur = tmp;  // the fused unit reads `cur` with a halo: its output goes to the other buffer
        continue;
      }
      Layer L1;
      L1.name = blk + "r" + std::to_string(j) + ".conv1";
      L1.Cin = C, L1.Cout = C, L1.K = desc->res_kernel, L1.dil = enc->dils[j];
      L1.in_buf = cur, L1.hl_buf = tmp;
      if ((st = add(L1, false, w1, b1, a2, div, 0)) != VOC_OK) return bail(st);
      Layer L2;  // 1x1: reads `tmp` row for row, so it may write `cur`
      L2.name = blk + "r" + std::to_string(j) + ".conv2";
      L2.Cin = C, L2.Cout = C, L2.K = 1, L2.dil = 1;
      L2.in_buf = tmp, L2.skip_buf = BUF_FY, L2.hl_buf = cur;
      if (j < nd - 1) L2.f32_buf = BUF_FY;  // the last unit's sum is only read through its Snake
      if ((st = add(L2, true, w2, b2, next, div, j == nd - 1 ? s : 0)) != VOC_OK) return bail(st);
    }
    {  // strided conv over the phase-split Snake'd input
      const float *w = params[p + 1], *b = params[p + 2];
      p += 3;
      const bool last = i == desc->n_stages - 1;
      // the next block's first Snake1, or Snake_out
      const SnakeCoef next = snake_coef(params[p], Co, desc->snake);
      const int o = other(cur);
      Layer L;
      L.name = blk + ".down";
      L.down_s = s, L.down_c = C;
      L.Cin = s * rup(C, 16), L.Cout = Co, L.K = 3, L.dil = 1;
      L.in_buf = cur, L.hl_buf = o;
      if (!last) L.f32_buf = BUF_FY;
      div *= s;
      if ((st = add(L, false, w, b, next, div, 0)) != VOC_OK) return bail(st);
      cur = o;
      C = Co;
    }
  }
  {  // conv_out (its input already Snake'd), then the 1x1 posterior mean projection
    const int o = other(cur);
    Layer L;
    L.name = "conv_out";
    L.Cin = C, L.Cout = C, L.K = desc->out_kernel, L.dil = 1;
    L.in_buf = cur, L.hl_buf = o;
    if ((st = add(L, false, params[p + 1], params[p + 2], SnakeCoef{}, div, 0)) != VOC_OK)
      return bail(st);
    Layer P;
    P.name = "proj";
    P.Cin = C, P.Cout = desc->latent_channels, P.K = 1, P.dil = 1;
    P.in_buf = o, P.f32_buf = BUF_FY;
    if ((st = add(P, false, params[p + 3], params[p + 4], SnakeCoef{}, div, 0)) != VOC_OK)
      return bail(st);
  }
  *out = enc;
  return VOC_OK;
}

VOC_API long long vocoder_encoder_hop(const vocoder_encoder *enc) { return enc ? enc->hop : -1; }

VOC_API size_t vocoder_encoder_workspace_bytes(const vocoder_encoder *enc, int B, long long L) {
  if (!enc || B < 1 || B > 65535 || L < 1 || L % enc->hop) return 0;
  if (L > (1LL << 30)) return 0;  // GEMM rows of one item stay in the kernels' int range
  return 4 * enc_buf_bytes(enc, B, L);  // H0, H1, FY and the split-k raw sums
}

VOC_API int vocoder_encoder_launches(const vocoder_encoder *enc, int B, long long L) {
  if (!vocoder_encoder_workspace_bytes(enc, B, L)) return -1;
  const size_t bb = enc_buf_bytes(enc, B, L);
  int n = 2 + static_cast<int>(enc->layers.size()) - (enc->layers[0].direct ? 1 : 0);
  for (size_t i = 0; i < enc->layers.size(); ++i)
    if (enc_ksplit(enc, i, B, L / enc->div[i], bb) > 1) ++n;  // its reduce kernel
  return n;
}

VOC_API voc_status vocoder_encode(vocoder_encoder *enc, const float *audio_dev, int B, long long L,
                                  float *latent_dev, void *ws, size_t ws_bytes,
                                  voc_stream_t stream_h, unsigned flags) {
  if (!enc) return fail(nullptr, VOC_INVALID_ARG, "encoder is NULL");
  vocoder *ctx = &enc->core;
  if (!audio_dev || !latent_dev) return fail(ctx, VOC_INVALID_ARG, "audio / latent NULL");
  if (flags & ~(unsigned)(VOC_FLAG_SYNC | VOC_FLAG_PROFILE))
    return fail(ctx, VOC_INVALID_ARG, "flags: only VOC_FLAG_SYNC and VOC_FLAG_PROFILE apply");
  const size_t need = vocoder_encoder_workspace_bytes(enc, B, L);
  if (!need)
    return fail(ctx, VOC_INVALID_ARG, "B must be in [1, 65535] and L a positive multiple of the hop (" +
                                          std::to_string(enc->hop) + ") up to 2^30");
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(ctx, VOC_INVALID_ARG, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < need)
    return fail(ctx, VOC_WORKSPACE_TOO_SMALL,
                "workspace " + std::to_string(ws_bytes) + " < " + std::to_string(need));
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != ctx->device) return fail(ctx, VOC_INVALID_ARG, "current device differs from the encoder's");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);

  const size_t bb = enc_buf_bytes(enc, B, L);
  void *bufs[BUF_COUNT];
  uint8_t *base = static_cast<uint8_t *>(ws);
  // H0, H1, FY and (in the HB slot) the raw sums of split-k layers
  bufs[BUF_H0] = base, bufs[BUF_H1] = base + bb, bufs[BUF_FY] = base + 2 * bb;
  bufs[BUF_HB] = base + 3 * bb;
  const size_t n_layers = enc->layers.size();
  if (enc->map_ws != ws || enc->map_B != B || enc->map_L != L) {
    enc->maps.resize(n_layers);
    enc->skip_maps.assign(n_layers, CUtensorMap{});
    for (size_t i = 0; i < n_layers; ++i) {
      const Layer &Ly = enc->layers[i];
      if (Ly.direct) continue;  // reads the audio itself
      const long long rows = pitch8(L / enc->div[i]);
      voc_status st = encode_map(ctx, &enc->maps[i], bufs[Ly.in_buf], Ly.Cp_in, rows, B, Ly.g.rows,
                                 Ly.g.KB / 8);
      if (st == VOC_OK && Ly.skip_buf >= 0)
        st = encode_skip_map(ctx, &enc->skip_maps[i], bufs[Ly.skip_buf], Ly.Cp_out, rows, B, Ly.cw);
      if (st != VOC_OK) {
        enc->map_ws = nullptr;
        return st;
      }
    }
    enc->map_ws = ws, enc->map_B = B, enc->map_L = L;
  }

  const bool prof = (flags & VOC_FLAG_PROFILE) != 0;
  const int n_launch = vocoder_encoder_launches(enc, B, L);
  if (prof) {
    while ((int)ctx->events.size() < 2 * n_launch) {
      cudaEvent_t ev;
      cudaError_t e = cudaEventCreate(&ev);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaEventCreate");
      ctx->events.push_back(ev);
    }
    ctx->prof_names.assign(n_launch, "");
    ctx->prof_flops.assign(n_launch, 0.0);
    ctx->prof_bytes.assign(n_launch, 0.0);
    ctx->prof_impl.assign(n_launch, 0.0);
    ctx->prof_ms.assign(n_launch, -1.f);
    ctx->prof_n = n_launch;
    ctx->prof_ready = false;
  }
  int li = 0;
  auto rec = [&](int which) {
    if (prof) cudaEventRecord(ctx->events[2 * li + which], stream);
  };
  const int Ci = enc->desc.in_channels;
  voc_status st = VOC_OK;
  if (!enc->layers[0].direct) {  // the audio as hi/lo planes for the conv_in GEMM
    rec(0);
    st = launch_prep(ctx, audio_dev, B, Ci, static_cast<int>(L), enc->Cp_audio, nullptr, nullptr,
                     static_cast<__nv_bfloat16 *>(bufs[BUF_H0]), stream);
    if (st != VOC_OK) return st;
#ifdef VOC_CHECKS
    if ((st = check_launch(ctx, "prep_audio", stream)) != VOC_OK) return st;
#endif
    rec(1);
    if (prof) {
      ctx->prof_names[li] = "prep_audio";
      ctx->prof_bytes[li] = (double)B * L * 8.0 * Ci;
      ctx->prof_impl[li] = (double)B * L * (4.0 * Ci + 4.0 * enc->Cp_audio);
    }
    ++li;
  }
  for (size_t i = 0; i < n_layers; ++i, ++li) {
    const Layer &Ly = enc->layers[i];
    const long long rows = L / enc->div[i];
    if (Ly.direct) {  // conv_in on the audio, fp32 on the CUDA cores
      const long long Lp = pitch8(rows);
      rec(0);
      cudaError_t ce = launch_pdl(
          voc::audio_conv_in_kernel,
          dim3(static_cast<unsigned>((Lp + 256 * voc::kAudioRows - 1) / (256 * voc::kAudioRows)),
               Ly.Cp_out / 8, B),
          dim3(256), 0, stream, audio_dev, Ci, static_cast<int>(rows), Lp, Ly.K, (Ly.K - 1) / 2,
          static_cast<const float *>(Ly.wf_dev), Ly.Cout, static_cast<const float *>(Ly.bias_dev),
          static_cast<const float *>(Ly.alpha_dev), static_cast<const float *>(Ly.invb_dev),
          Ly.Cp_out, static_cast<float *>(bufs[Ly.f32_buf]),
          static_cast<__nv_bfloat16 *>(bufs[Ly.hl_buf]), ctx->prec == VOC_PREC_F16W ? 1 : 0);
      if (ce != cudaSuccess) return cuda_fail(ctx, ce, "launch audio conv_in");
#ifdef VOC_CHECKS
      if ((st = check_launch(ctx, Ly.name, stream)) != VOC_OK) return st;
#endif
      rec(1);
      if (prof) {
        ctx->prof_names[li] = Ly.name;
        ctx->prof_flops[li] = 2.0 * Ly.Cin * Ly.Cout * Ly.K * B * (double)rows;
        ctx->prof_bytes[li] = (double)B * rows * (4.0 * Ci + 4.0 * Ly.Cout);
        ctx->prof_impl[li] = (double)B * rows * (4.0 * Ci + 8.0 * Ly.Cp_out);
      }
      continue;
    }
    ConvGemmArgs a;
    gemm_args_rows(ctx, Ly, B, rows, bufs, bb, a);
    if (enc->split[i]) {
      // Phase-split hi/lo output: planes of pitch8(L/s) rows, so rows [L, s pitch8(L/s)) of
      // the layer are written as zeros -- the strided conv reads row L/s of every phase as
      // its right padding.  With s not a power of two those rows can lie past the last
      // 128-row tile of L rows: the launch covers them (its input rows there read as zeros).
      const int s = enc->split[i];
      a.split_s = s;
      a.hl_L = static_cast<int>(pitch8(rows / s));
      a.rows_pad = static_cast<int>(rup_ll(rows, 8LL * s));
      a.m_tiles = (a.rows_pad + voc::kTileM - 1) / voc::kTileM;
    }
    const int S = enc_ksplit(enc, i, B, rows, bb);
    ConvGemmArgs fin = a;  // the layer's outputs, written by the reduce kernel when split
    if (S > 1) {
      a.ksplit = S;
      a.kb_per_split = (Ly.g.nkb + S - 1) / S;
      a.ksplit = (Ly.g.nkb + a.kb_per_split - 1) / a.kb_per_split;  // no empty range
      a.part = static_cast<float *>(bufs[BUF_HB]);
      a.part_L = pitch8(rows);
    }
    rec(0);
    st = launch_gemm(ctx, Ly, enc->maps[i], enc->skip_maps[i], a, stream);
    if (st != VOC_OK) return st;
#ifdef VOC_CHECKS
    if ((st = check_launch(ctx, Ly.name, stream)) != VOC_OK) return st;
#endif
    rec(1);
    if (prof) {
      ctx->prof_names[li] = Ly.name;
      enc_layer_cost(Ly, B, rows, S > 1, ctx->prof_flops[li], ctx->prof_bytes[li],
                     ctx->prof_impl[li]);
      if (S > 1)  // the outputs are the reduce kernel's
        ctx->prof_impl[li] += 4.0 * a.ksplit * B * (double)rows * Ly.Cp_out -
                               (Ly.f32_buf >= 0 ? 4.0 : 0.0) * B * (double)rows * Ly.Cp_out -
                               (Ly.hl_buf >= 0 ? 4.0 : 0.0) * B * (double)rows * Ly.Cp_out;
    }
    if (S > 1) {
      ++li;
      rec(0);
      dim3 grid(static_cast<unsigned>((fin.rows_pad + 255) / 256), Ly.Cp_out / 8, B);
      cudaError_t ce = launch_pdl(
          voc::ksplit_reduce_kernel, grid, dim3(256), 0, stream,
          static_cast<const float *>(a.part), a.ksplit, B, Ly.Cp_out, a.part_L, fin.rows_valid,
          fin.rows_pad, static_cast<const float *>(Ly.bias_dev),
          static_cast<const float *>(Ly.alpha_dev), static_cast<const float *>(Ly.invb_dev),
          (Ly.epi_flags & voc::EPI_F32_SNAKE) ? 1 : 0, fin.out_f32, (long long)fin.f32_L,
          fin.out_hl, (long long)fin.hl_L, ctx->prec == VOC_PREC_F16W ? 1 : 0);
      if (ce != cudaSuccess) return cuda_fail(ctx, ce, ("launch reduce " + Ly.name).c_str());
#ifdef VOC_CHECKS
      if ((st = check_launch(ctx, Ly.name + ".reduce", stream)) != VOC_OK) return st;
#endif
      rec(1);
      if (prof) {
        ctx->prof_names[li] = Ly.name + ".reduce";
        ctx->prof_flops[li] = 0.0;
        ctx->prof_bytes[li] = 4.0 * B * (double)rows * Ly.Cout;  // the layer's output
        ctx->prof_impl[li] = 4.0 * B * (double)rows * Ly.Cp_out *
                              (a.ksplit + (Ly.f32_buf >= 0 ? 1 : 0) + (Ly.hl_buf >= 0 ? 1 : 0));
      }
    }
  }
  const long long Lz = L / enc->hop;
  const int Cl = enc->desc.latent_channels;
  rec(0);
  voc::rows_to_cf_kernel<<<dim3(static_cast<unsigned>((Lz + 255) / 256), enc->Cp_lat / 4, B), 256, 0,
                           stream>>>(static_cast<const float *>(bufs[BUF_FY]), static_cast<int>(Lz),
                                     pitch8(Lz), enc->Cp_lat, Cl, latent_dev);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "launch latent layout");
  rec(1);
  if (prof) {
    ctx->prof_names[li] = "latent_out";
    ctx->prof_bytes[li] = (double)B * Lz * 8.0 * Cl;
    ctx->prof_impl[li] = (double)B * Lz * (4.0 * enc->Cp_lat + 4.0 * Cl);
    ctx->prof_ready = true;
  }
  ++li;
  if (flags & VOC_FLAG_SYNC) {
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
    int word = 0;
    e = cudaMemcpy(&word, ctx->err_dev, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "read device error word");
    if (word) {
      cudaMemset(ctx->err_dev, 0, sizeof(int));
      return fail(ctx, VOC_DEVICE_TIMEOUT,
                  "a kernel gave up a bounded wait (code " + std::to_string(word) + ")");
    }
  }
  return VOC_OK;
}

VOC_API int vocoder_encoder_profile_count(const vocoder_encoder *enc) {
  return enc ? vocoder_profile_count(&enc->core) : 0;
}

VOC_API voc_status vocoder_encoder_profile_entry(vocoder_encoder *enc, int index, const char **name,
                                                 double *ms, double *flops, double *bytes) {
  if (!enc) return fail(nullptr, VOC_INVALID_ARG, "encoder is NULL");
  return vocoder_profile_entry(&enc->core, index, name, ms, flops, bytes);
}

VOC_API voc_status vocoder_encoder_profile_impl_bytes(vocoder_encoder *enc, int index,
                                                      double *bytes) {
  if (!enc) return fail(nullptr, VOC_INVALID_ARG, "encoder is NULL");
  return vocoder_profile_impl_bytes(&enc->core, index, bytes);
}

VOC_API const char *vocoder_encoder_last_error(const vocoder_encoder *enc) {
  return enc ? enc->core.err.c_str() : g_err.c_str();
}

VOC_API size_t vocoder_encoder_workspace_bytes_host(const vocoder_encoder *enc, int B, long long L) {
  const size_t w = vocoder_encoder_workspace_bytes(enc, B, L);
  if (!w) return 0;
  return w + rupz((size_t)B * enc->desc.in_channels * (size_t)L * 4, 256) +
         rupz((size_t)B * enc->desc.latent_channels * (size_t)(L / enc->hop) * 4, 256);
}

VOC_API voc_status vocoder_encode_host(vocoder_encoder *enc, const float *audio_host, int B,
                                       long long L, float *latent_host, void *ws_dev,
                                       size_t ws_bytes, voc_stream_t stream, unsigned flags) {
  if (!enc) return fail(nullptr, VOC_INVALID_ARG, "encoder is NULL");
  vocoder *ctx = &enc->core;
  if (!audio_host || !latent_host) return fail(ctx, VOC_INVALID_ARG, "audio / latent NULL");
  const size_t need = vocoder_encoder_workspace_bytes_host(enc, B, L);
  if (!need)
    return fail(ctx, VOC_INVALID_ARG, "B must be in [1, 65535] and L a positive multiple of the hop");
  if (!ws_dev || (reinterpret_cast<uintptr_t>(ws_dev) & 255))
    return fail(ctx, VOC_INVALID_ARG, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < need)
    return fail(ctx, VOC_WORKSPACE_TOO_SMALL,
                "workspace " + std::to_string(ws_bytes) + " < " + std::to_string(need));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t wenc = vocoder_encoder_workspace_bytes(enc, B, L);
  const size_t in_bytes = (size_t)B * enc->desc.in_channels * (size_t)L * 4;
  const size_t out_bytes = (size_t)B * enc->desc.latent_channels * (size_t)(L / enc->hop) * 4;
  uint8_t *base = static_cast<uint8_t *>(ws_dev);
  float *aud_d = reinterpret_cast<float *>(base + wenc);
  float *lat_d = reinterpret_cast<float *>(base + wenc + rupz(in_bytes, 256));
  cudaError_t e = cudaMemcpyAsync(aud_d, audio_host, in_bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "copy audio in");
  voc_status st = vocoder_encode(enc, aud_d, B, L, lat_d, ws_dev, wenc, stream, flags);
  if (st != VOC_OK) return st;
  e = cudaMemcpyAsync(latent_host, lat_d, out_bytes, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "copy latent out");
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
  return VOC_OK;
}
