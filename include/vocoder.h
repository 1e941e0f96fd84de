/*
 * vocoder.h -- C ABI of the GB300 DAC-style vocoder decoder.
 *
 * The decoder turns a latent sequence into a waveform (minimaxmusic.cpp
 * Architecture, section "Flow VAE"):
 *
 *   conv_in k7 (C_lat -> C0)
 *   for every upsampling stage (stride s, C_in -> C_out):
 *       Snake -> ConvTranspose1d (k = 2s, pad s/2) -> 3 residual units,
 *       residual unit (dilation d in 1, 3, 9):
 *           y = x + conv2_k1( Snake2( conv1_k7_dil_d( Snake1(x) ) ) )
 *   Snake -> conv_out k7 (C_last -> 1, with bias) -> tanh
 *
 * with Snake(x) = x + sin^2(a x) / (a + 1e-9), the per-channel a used as stored
 * (MiniMax-Music-3 -> CMF README, "What the conversion had to get right").
 * The speech-codec variant (qwentts.cpp Architecture, "Audio tokenizer
 * decoder") runs the same stack causally: k-tap convs pad (k-1)d on the left
 * only and each transposed conv keeps the first T*s samples of its col2im output.
 *
 * Conventions (pattern of qwentts.cpp Architecture, "Public API" / "ABI
 * guarantee"): plain C99, an opaque handle, negative status codes, a last-error
 * string, an ABI version checked at create time, and every argument validated
 * before any device work.  Only vocoder_* symbols are exported.
 *
 * Devices, streams, ownership:
 *   - A context lives on the CUDA device that is current when vocoder_create is
 *     called; all later calls on it must run with that device current.
 *   - The library owns its device copy of the weights (create .. destroy).
 *   - The caller owns every latent / audio / workspace buffer.  "_dev" pointers
 *     are device memory of the context's device, "_host" pointers host memory.
 *   - Work is enqueued on the caller's stream (a cudaStream_t passed as
 *     voc_stream_t; NULL is the legacy default stream) and is asynchronous
 *     unless a flag below asks for a synchronisation.
 *   - A context is not thread-safe: use it from one thread and one stream at a
 *     time.
 * Precision: fp32 storage and accumulation; every convolution runs on the
 * tensor cores as three bf16 products of a hi/lo split of both operands
 * (hi*hi + hi*lo + lo*hi), which carries about 16 significant bits per operand.
 */
#ifndef GB300_VOCODER_H
#define GB300_VOCODER_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VOC_ABI_VERSION 5

typedef struct vocoder vocoder_t;             /* opaque context */
typedef struct CUstream_st *voc_stream_t;     /* a cudaStream_t */

typedef enum {
  VOC_OK = 0,
  VOC_INVALID_ARG = -1,         /* a pointer, size or description is invalid       */
  VOC_UNSUPPORTED = -2,         /* valid in principle, not supported by the library  */
  VOC_CUDA_ERROR = -3,          /* a CUDA runtime call or a kernel launch failed    */
  VOC_OOM = -4,                 /* device or host allocation failed                 */
  VOC_WORKSPACE_TOO_SMALL = -5, /* ws_bytes below vocoder_workspace_bytes()         */
  VOC_NONFINITE = -6,           /* VOC_FLAG_CHECK_FINITE found a NaN / Inf          */
  VOC_CANCELLED = -7,           /* the caller's cancel flag was set: nothing enqueued */
  VOC_DEVICE_TIMEOUT = -8       /* a kernel gave up a bounded wait (see VOC_FLAG_SYNC) */
} voc_status;

enum { VOC_PAD_SYMMETRIC = 0, VOC_PAD_CAUSAL = 1 };
/* precision: VOC_PREC_BF16X3 -- weights and activations as bf16 hi/lo pairs, three bf16
 * products per multiply (about 16 significant bits per operand), fp32 accumulation;
 * VOC_PREC_F16W -- every convolution weight rounded to IEEE half precision, as the pages'
 * port stores them (minimaxmusic.cpp Architecture, "Flow VAE": conv weights F16 on the
 * device with F32 activations); activations as f16 hi/lo pairs (about 22 significant bits,
 * |x| < 65504), two f16 products per multiply, fp32 accumulation.  Biases and Snake
 * parameters stay fp32.  VOC_PREC_BF16W (ABI 5, added with the encoder) -- every
 * convolution weight rounded to bfloat16 (8 significant bits), the precision checkpoints
 * are commonly distributed in; activations as bf16 hi/lo pairs, two bf16 products per
 * multiply, fp32 accumulation.  The one-plane precisions (F16W, BF16W) run neither fused
 * residual units nor CTA pairs. */
enum { VOC_PREC_BF16X3 = 0, VOC_PREC_F16W = 1, VOC_PREC_BF16W = 2 };
/* activation: Snake with alpha as stored, or SnakeBeta with log-scale alpha and beta,
 * x + sin^2(e^alpha x) / (e^beta + 1e-9) (qwentts.cpp Architecture, "Audio tokenizer
 * decoder": exp applied to both stored parameters) */
enum { VOC_SNAKE = 0, VOC_SNAKE_BETA = 1 };

/* flags of vocoder_decode / vocoder_decode_host */
enum {
  VOC_FLAG_CHECK_FINITE = 1, /* scan the audio for NaN / Inf; implies a stream sync   */
  VOC_FLAG_SYNC = 2,         /* synchronise the stream and report device timeouts     */
  VOC_FLAG_PROFILE = 4       /* record a CUDA event around every kernel of the decode */
};

/* Architecture of the decoder.  All arrays are borrowed for the duration of
 * vocoder_create only. */
typedef struct {
  int abi_version;      /* VOC_ABI_VERSION                                  */
  int latent_channels;  /* C_lat (64 music, 1024 speech)                    */
  int in_kernel;        /* conv_in taps (odd, 1..15; 7)                     */
  int channels0;        /* C0, conv_in output channels                       */
  int n_stages;         /* upsampling stages (1..8)                          */
  const int *strides;   /* [n_stages] (even unless VOC_PAD_CAUSAL)           */
  const int *widths;    /* [n_stages] output channels of each stage          */
  int n_dilations;      /* residual units per stage (1..4; 3)                */
  const int *dilations; /* [n_dilations] (1, 3, 9)                           */
  int res_kernel;       /* dilated conv taps (odd; 7)                        */
  int out_kernel;       /* conv_out taps (odd; 7)                            */
  int out_channels;     /* 1                                                 */
  int padding;          /* VOC_PAD_SYMMETRIC | VOC_PAD_CAUSAL                */
  int precision;        /* VOC_PREC_BF16X3 | VOC_PREC_F16W | VOC_PREC_BF16W  */
  int fuse_max_channels;/* residual units of up to this many channels (at most 192)
                           run as one kernel (conv1 result kept on chip); 0 = library
                           default (192: every unit that fits; with VOC_PREC_F16W or
                           VOC_PREC_BF16W only the units wider than 128 channels,
                           the narrower ones being faster as two kernels there),
                           -1 = never.  A performance choice only: results agree
                           within the decode tolerance either way.               */
  int cta_pair;         /* conv layers run on CTA pairs (2-CTA clusters sharing one
                           256-row MMA, each SM staging half of the weights):
                           0 = library default (off), 1 = on, -1 = off.  A
                           performance choice only, like fuse_max_channels.     */
  int in_proj_channels; /* 0, or P > 0: a 1x1 projection C_lat -> P with bias and no
                           weight norm runs before conv_in, which then maps P -> C0
                           (the published music model's dec_in_proj 64 -> 1024,
                           minimaxmusic.cpp Architecture, "Flow VAE")          */
  int snake;            /* VOC_SNAKE | VOC_SNAKE_BETA (ABI 5)                    */
} voc_desc;

/* ABI version of the library (VOC_ABI_VERSION of the build). */
int vocoder_abi_version(void);

/* Number of parameter tensors of the architecture, or -1 for an invalid desc.
 * Canonical order and PyTorch layouts (weights already folded):
 *   [in_proj.w [P][C_lat][1], in_proj.b [P]]   (only when in_proj_channels = P > 0)
 *   conv_in.w [C0][C_lat or P][in_kernel], conv_in.b [C0],
 *   per stage i (C_in -> C_out = widths[i], stride s):
 *     snake.alpha [C_in], convT.w [C_in][C_out][2s], convT.b [C_out],
 *     per dilation: snake1.alpha [C_out], conv1.w [C_out][C_out][res_kernel],
 *                   conv1.b [C_out], snake2.alpha [C_out], conv2.w [C_out][C_out][1],
 *                   conv2.b [C_out],
 *   snake_out.alpha [C_last], conv_out.w [1][C_last][out_kernel], conv_out.b [1].
 * With VOC_SNAKE_BETA every snake*.alpha entry is [2][C] instead: log alpha, then log
 * beta, each in [-80, 80] (plain Snake alphas must be > 0). */
int vocoder_param_count(const voc_desc *desc);

/* Shape of parameter `index`: writes up to 3 dims and their count. */
voc_status vocoder_param_shape(const voc_desc *desc, int index, int dims[3], int *ndim);

/* Weight-norm fold (minimaxmusic.cpp Architecture, "Models" / "Flow VAE"):
 *   w[i, :] = g[i] * v[i, :] / ||v[i, :]||  for i < dim0, rows of `rest` values,
 * the norm running over every axis but axis 0 of the stored tensor (Conv1d
 * [Cout][Cin][K]: rest = Cin*K; ConvTranspose1d [Cin][Cout][K]: rest = Cout*K).
 * Host memory; accumulates in double; w may not alias v.  VOC_INVALID_ARG for a
 * NULL pointer, non-positive sizes, a zero-norm row or a non-finite result. */
voc_status vocoder_fold_weight_norm(const float *g, const float *v, int dim0, long long rest,
                                    float *w);

/* Create a decoder on the current device.  params: vocoder_param_count(desc)
 * host pointers in the canonical order; a NULL bias means zero, every other
 * entry is required.  The weights are re-laid out per tap, split into bf16 hi/lo
 * and copied to the device; the host arrays are not retained.  On failure *out
 * is NULL, every device allocation made so far is freed, and
 * vocoder_last_error(NULL) describes the problem (VOC_OOM when the device ran out
 * of memory).  Create also looks up, once per device, the device address of the
 * built-in workspace of vocoder_decode_static (cudaGetSymbolAddress, with the
 * context's device current).
 * Relation to the boundary sketched for this library: its `voc_weights` struct is
 * this array of `params` pointers in the canonical order above, and its precision
 * pair 3xTF32 / TF32 is VOC_PREC_BF16X3 (three bf16 products of hi/lo splits,
 * about 16 significant bits per operand, at bf16 tensor rate) / the one-plane
 * VOC_PREC_F16W and VOC_PREC_BF16W (two products per multiply, the cost of one
 * TF32 pass on this GPU, keeping more of the activations' bits than TF32). */
voc_status vocoder_create(const voc_desc *desc, const float *const *params, int n_params,
                          vocoder_t **out);

/* Upsampling factor (product of the strides), or -1 for NULL. */
long long vocoder_hop(const vocoder_t *ctx);

/* Device workspace that vocoder_decode needs for B items of T latent frames
 * (0 for invalid sizes).  vocoder_workspace_bytes_host adds room for the
 * host-buffer entry point's staging copies. */
size_t vocoder_workspace_bytes(const vocoder_t *ctx, int B, int T);
size_t vocoder_workspace_bytes_host(const vocoder_t *ctx, int B, int T);

/* Decode B mono items (a stereo track is folded by the caller into 2 items,
 * channels 0..C_lat-1 left):
 *   latent_dev [B][C_lat][T] fp32, time contiguous  ->  audio_dev [B][1][T*hop] fp32.
 * ws_dev: device workspace of at least vocoder_workspace_bytes(ctx, B, T) bytes,
 * 256-byte aligned, not used by anything else until the decode has finished on
 * `stream`.  latent_dev must be 16-byte aligned.  Asynchronous on `stream`
 * unless flags contain VOC_FLAG_SYNC or VOC_FLAG_CHECK_FINITE. */
voc_status vocoder_decode(vocoder_t *ctx, const float *latent_dev, int B, int T, float *audio_dev,
                          void *ws_dev, size_t ws_bytes, voc_stream_t stream, unsigned flags);

/* Same decode from and to HOST buffers: copies the latent in, decodes, copies
 * the audio out and synchronises `stream` before returning.  ws_bytes >=
 * vocoder_workspace_bytes_host(ctx, B, T).  Page-locked host buffers give
 * asynchronous copies; pageable ones work but are slower. */
voc_status vocoder_decode_host(vocoder_t *ctx, const float *latent_host, int B, int T,
                               float *audio_host, void *ws_dev, size_t ws_bytes,
                               voc_stream_t stream, unsigned flags);

/* Decode without allocating any device memory.  No counterpart on the source
 * pages: this entry point exists for callers that must not call cudaMalloc
 * while they run -- a real-time audio thread, where cudaMalloc can synchronise
 * the device and stall long enough to drop an audio buffer, or a host
 * application whose own allocator has already reserved the device memory and
 * forbids allocations behind its back.  The context must still be created
 * beforehand (vocoder_create allocates the weights once, at set-up time).
 *
 * Same inputs, outputs and results (bit for bit) as vocoder_decode, but the
 * workspace is a file-scope device array of VOC_STATIC_WORKSPACE_BYTES inside
 * the library, which every GPU that loads the library holds until the process
 * exits.
 *   - Sizes whose vocoder_workspace_bytes(ctx, B, T) exceeds
 *     VOC_STATIC_WORKSPACE_BYTES are rejected with VOC_WORKSPACE_TOO_SMALL.
 *   - The array's device address is looked up by vocoder_create, once per
 *     device, with that device current; this call only reads the cached
 *     address.  A call with another device current is VOC_INVALID_ARG.
 *   - Every call shares the one array, which keeps the contents of the last
 *     call.  The decode writes each workspace byte before reading it, so
 *     nothing needs clearing, but calls that overlap on the GPU (other
 *     streams, other threads, other contexts) race on the array and corrupt
 *     each other's audio: serialise them.
 *   - VOC_FLAG_PROFILE is rejected (VOC_INVALID_ARG); the other flags behave
 *     as in vocoder_decode.
 * The function calls no cudaMalloc, cudaFree or allocating routine on the
 * device.  On the host it allocates nothing while it alternates between at
 * most two (workspace, B, T) combinations on a context (for example this one
 * and one vocoder_decode workspace): the context keeps the tensor-map
 * descriptors of the two most recent combinations in storage sized at create
 * time; an error message is the only other host allocation. */
#define VOC_STATIC_WORKSPACE_BYTES (64ull << 20)
voc_status vocoder_decode_static(vocoder_t *ctx, const float *latent_dev, int B, int T,
                                 float *audio_dev, voc_stream_t stream, unsigned flags);

/* Overlap-crop stitch (minimaxmusic.cpp Architecture, "Decode and stitch"):
 *   decoded_dev [n_win*n_sides][win_frames*hop], item index w*n_sides + side;
 * window 0 keeps its left edge, later windows drop crop_left frames on the
 * left, all but the last drop crop_right frames on the right; the kept pieces
 * are concatenated per side and clamped to [-1, 1] into
 *   out_dev [n_sides][vocoder_stitched_length(...)].
 * Asynchronous on `stream`.  Buffers must be 16-byte aligned. */
long long vocoder_stitched_length(int n_win, int win_frames, int crop_left, int crop_right,
                                  int hop);
voc_status vocoder_stitch(const float *decoded_dev, int n_win, int n_sides, int win_frames,
                          int crop_left, int crop_right, int hop, float *out_dev,
                          voc_stream_t stream);

/* Single-layer operations on the same kernels as vocoder_decode, for per-layer
 * checks.  Channels-first fp32 device tensors; they allocate and free their own
 * temporaries and synchronise `stream` before returning.
 *   vocoder_op_conv1d:   y[b][co][t] = bias[co] + sum_ci sum_k
 *                          w[co][ci][k] * S(x)[b][ci][t + k*dil - pad_left]
 *     (y [B][Cout][T]; pad_left = dil*(K-1)/2 symmetric or dil*(K-1) causal)
 *   vocoder_op_conv_transpose1d: y[b][co][t*s + k - p] += w[ci][co][k] * S(x)[b][ci][t]
 *     plus bias (y [B][Cout][T*s], K = 2s; p = s/2 symmetric, 0 causal)
 * where S is Snake with per-channel alpha_host [Cin], or the identity when
 * alpha_host is NULL.  Weights are host fp32 in PyTorch layouts; b_host may be NULL. */
voc_status vocoder_op_conv1d(const float *x_dev, int B, int Cin, int T, const float *w_host,
                             const float *b_host, int Cout, int K, int dil, int padding,
                             const float *alpha_host, float *y_dev, voc_stream_t stream);
voc_status vocoder_op_conv_transpose1d(const float *x_dev, int B, int Cin, int T,
                                       const float *w_host, const float *b_host, int Cout,
                                       int stride, int padding, const float *alpha_host,
                                       float *y_dev, voc_stream_t stream);

/* One residual unit (minimaxmusic.cpp Architecture, "Flow VAE": skip -> snake1 -> conv1
 * k-tap dilated -> snake2 -> conv2 1x1 -> + skip) on the decoder's own kernels:
 *   y = x + conv2( S2( conv1( S1(x) ) + b1 ) ) + b2
 * x_dev, y_dev [B][C][T] fp32 channels-first (may not alias); w1_host [C][C][K],
 * w2_host [C][C][1], alpha1/alpha2 [C] (required), b1/b2 [C] or NULL; padding as for
 * vocoder_op_conv1d.  Up to 192 channels the unit runs as one fused kernel (the conv1
 * result stays in shared memory), above as two.  Allocates its temporaries and
 * synchronises `stream` before returning. */
voc_status vocoder_op_residual_unit(const float *x_dev, int B, int C, int T,
                                    const float *alpha1_host, const float *w1_host,
                                    const float *b1_host, int K, int dil,
                                    const float *alpha2_host, const float *w2_host,
                                    const float *b2_host, int padding, float *y_dev,
                                    voc_stream_t stream);

/* Kernel launches that one vocoder_decode(ctx, ., B, T, ...) enqueues. */
int vocoder_launches_per_decode(const vocoder_t *ctx, int B, int T);

/* Per-kernel record of the last decode that ran with VOC_FLAG_PROFILE (valid
 * after the stream has been synchronised): name, device time (ms), algorithmic
 * FLOPs (2 per multiply-add, transposed conv counted without zero-stuffing) and
 * algorithmic bytes: each input of the launch's layers read once and each output
 * written once, as fp32 values of the real channels -- a k-tap conv 4 Cin + 4 Cout
 * bytes per row, a 1x1 conv with the residual add 4 Cin + 8 Cout (it also reads
 * the skip), a transposed conv 4 Cin per input row + 4 Cout per output sample, a
 * fused residual unit 8 C per row (x read once for conv1 and the skip, y written
 * once), the output head 4 C + 4 per sample.  A launch that carries the folded
 * output head counts its inputs only; the head's finishing launch counts the audio. */
int vocoder_profile_count(const vocoder_t *ctx);
voc_status vocoder_profile_entry(vocoder_t *ctx, int index, const char **name, double *ms,
                                 double *flops, double *bytes);

/* The bytes entry `index` of the same record moves by the implementation's own count:
 * channels padded to 16, the streamed weights, and every copy of an output (the fp32
 * residual stream and the bf16 hi/lo operand of the next layer).  Diagnostic: compare
 * it with the algorithmic bytes and with measured DRAM traffic. */
voc_status vocoder_profile_impl_bytes(vocoder_t *ctx, int index, double *bytes);

/* Message of the last failed call on ctx (ctx == NULL: of the last failure on
 * this thread without a context).  Valid until the next call on ctx. */
const char *vocoder_last_error(const vocoder_t *ctx);

/* Cancellation (the pattern of minimaxmusic.cpp Architecture, "mm-server reference",
 * "Concurrency": a cancel flag polled between VAE windows).  `flag` is a host int that
 * another thread may set to nonzero; while it is nonzero, vocoder_decode,
 * vocoder_decode_host, vocoder_decode_static and vocoder_stream_decode on ctx return
 * VOC_CANCELLED before enqueuing anything (outputs untouched, stream state unchanged).
 * A caller decoding a long track window by window (or a stream chunk by chunk)
 * therefore stops at the next window boundary; work already enqueued runs to its
 * end.  The library only reads the flag; NULL removes it.  The flag must outlive its
 * registration. */
voc_status vocoder_set_cancel_flag(vocoder_t *ctx, const volatile int *flag);

/* Bound, in SM clock cycles, on each wait inside the kernels that later calls on ctx
 * enqueue (decode and its variants): a kernel whose wait runs past it gives up, waits for
 * its own copies and tensor-core work in flight, frees its tensor memory and returns, and
 * the call reports VOC_DEVICE_TIMEOUT when made with VOC_FLAG_SYNC.  0 restores the
 * default of 4e9 cycles (about 2 s); a negative value is VOC_INVALID_ARG.  A stream
 * object's chunk graphs keep the bound they were captured with.  The bound is checked
 * between the hardware's own suspended waits (microseconds), so bounds below that act as
 * that granularity.  A bound of a few hundred cycles makes every decode of a music-sized
 * decoder give up: it exists to exercise that path. */
voc_status vocoder_set_wait_budget(vocoder_t *ctx, long long cycles);

/* Test hooks for the allocation-failure path (process-wide).  After
 * vocoder_debug_fail_allocation(n), the library's device allocations let n through and
 * make the next one fail as an out-of-memory cudaMalloc would (n < 0 disarms it; it
 * fires once).  vocoder_debug_live_allocations() counts the device allocations the
 * library currently holds, for every context, stream object and encoder. */
void vocoder_debug_fail_allocation(int n);
long long vocoder_debug_live_allocations(void);

/* Free the context and its device weights (NULL is ignored). */
void vocoder_destroy(vocoder_t *ctx);

/* ---------------------------------------------------------------- stateful streaming
 * qwentts.cpp Architecture, "Streaming decode (stateful path)": every layer of a causal
 * decoder looks left only, so decoding a sequence chunk by chunk (down to one latent frame
 * at a time) with each layer's left context carried between chunks reproduces the decode
 * of the whole sequence exactly, with no recomputed context and no seams.  Here each
 * stride-1 conv keeps its last (K-1)*dilation input rows and each transposed conv its last
 * input row (its overlap with the next chunk's first outputs); all contexts start at
 * zero, the zero padding of a decode that starts at frame 0.  The layers run with the
 * context's own plans, so a streamed sequence equals vocoder_decode of the whole
 * sequence bit for bit.  Causal decoders (VOC_PAD_CAUSAL) only. */
typedef struct vocoder_stream vocoder_stream_t;

/* Stream state for B sequences decoded in chunks of up to max_frames latent frames.
 * Allocates its own device buffers (the per-layer inputs with their context rows, the
 * saved contexts; about B * max_frames * hop * 200 bytes for the speech decoder) and zeroes
 * the contexts (synchronously).  ctx must outlive the stream.  VOC_UNSUPPORTED for a
 * non-causal decoder; VOC_INVALID_ARG for bad sizes or a different current device. */
voc_status vocoder_stream_create(vocoder_t *ctx, int B, int max_frames, vocoder_stream_t **out);

/* Decode the next `frames` (1..max_frames) latent frames of every sequence:
 * latent_dev [B][C_lat][frames] fp32 (device), audio_dev [B][1][frames*hop] fp32 (device),
 * asynchronous on `stream` like vocoder_decode.  Calls on one stream object must be
 * ordered (one stream, or synchronised); they update its contexts.  flags: 0 or
 * VOC_FLAG_SYNC (wait and report VOC_DEVICE_TIMEOUT).  Errors as vocoder_decode; the
 * message is vocoder_last_error(ctx).  The chunk's launches are captured into a CUDA graph the
 * first time a chunk size is used (on a stream of the stream object's own; that call also
 * instantiates the graph) and replayed afterwards: the call copies the latent into a staging
 * buffer, launches the graph and copies the audio out, all on `stream`.  The stream object is
 * therefore not usable from inside another stream capture. */
voc_status vocoder_stream_decode(vocoder_stream_t *s, const float *latent_dev, int frames,
                                 float *audio_dev, voc_stream_t stream, unsigned flags);

/* Zero every context (asynchronous on `stream`): the next chunk starts a new sequence. */
voc_status vocoder_stream_reset(vocoder_stream_t *s, voc_stream_t stream);

/* Free the stream's device buffers (NULL is ignored). */
void vocoder_stream_destroy(vocoder_stream_t *s);

/* ---------------------------------------------------------------- output stage
 * minimaxmusic.cpp Architecture, "Post-processing": the planar float output is peak
 * normalised to the 1 - peak_clip/1e6 percentile (peak_clip = 0: plain peak
 * normalisation) and encoded as a WAV file in memory; 32-bit float files are written raw,
 * without normalisation.  The level is the ceil(q*n)-th smallest |x| over all samples of
 * all channels (q = 1 - peak_clip/1e6, computed in double), found exactly on the device;
 * the gain is 1/level in IEEE single precision (1 for a level of 0); integer samples are
 * round-half-even(clamp(x*gain, -1, 1) * (2^(bits-1) - 1)) in single precision.  The
 * file is a 44-byte RIFF/WAVE header (PCM format 1 for 16/24 bits, IEEE float format 3
 * for 32 bits) followed by the samples interleaved across channels, little endian. */

/* Size of the WAV file of n_ch channels x len samples at `bits` (16, 24 or 32), or 0 for
 * invalid arguments or a file beyond the format's 4 GiB limit. */
size_t vocoder_wav_bytes(int n_ch, long long len, int bits);

/* Device scratch the 16/24-bit encoder needs (256-byte aligned; a few KB). */
size_t vocoder_wav_scratch_bytes(void);

/* Encode planar [n_ch][len] fp32 (device) into the WAV file at out_dev (device, at least
 * vocoder_wav_bytes, 4-byte aligned), asynchronously on `stream`.  scratch_dev (device,
 * vocoder_wav_scratch_bytes, caller-owned) is used for bits 16 and 24 and may be NULL for
 * 32.  VOC_INVALID_ARG for bad arguments, VOC_WORKSPACE_TOO_SMALL for short buffers. */
voc_status vocoder_encode_wav(const float *planar_dev, int n_ch, long long len, int sample_rate,
                              int bits, int peak_clip, void *out_dev, size_t out_bytes,
                              void *scratch_dev, size_t scratch_bytes, voc_stream_t stream);

/* ---------------------------------------------------------------- mirror encoder
 * minimaxmusic.cpp Architecture, "Flow VAE": the encoder mirrors the decoder and maps audio
 * to the latent's posterior mean:
 *
 *   conv_in k7 (C_in -> C0)
 *   for every downsampling block (stride s, C -> C' = widths[i]):
 *       3 residual units at C channels (as in the decoder), then
 *       Snake -> strided Conv1d (k = 2s, stride s, pad s/2 on both sides: L -> L/s)
 *   Snake -> conv_out k3 (C_last -> C_last) -> posterior mean projection k1 (C_last -> C_lat)
 *
 * All convolutions are non-causal (k-tap convs pad (k-1)d/2 on both sides), weights are
 * folded like the decoder's, and the precision is the decoder's (VOC_PREC_*).  On the
 * device each strided conv runs as a 3-tap conv over its input split into s phases
 * (row u s + r of channel c becomes row u of channel (c/8 s + r) 8 + c%8), the split done
 * by the epilogue of the layer that produces the input. */
typedef struct vocoder_encoder vocoder_encoder_t;  /* opaque encoder context */

/* Architecture of the encoder; arrays are borrowed for vocoder_encoder_create only. */
typedef struct {
  int abi_version;      /* VOC_ABI_VERSION                                       */
  int in_channels;      /* audio channels C_in (1..16; 1)                         */
  int channels0;        /* C0, conv_in output channels                            */
  int in_kernel;        /* conv_in taps (odd, 1..15; 7)                           */
  int n_stages;         /* downsampling blocks (1..8)                             */
  const int *strides;   /* [n_stages] strides s (1..16)                           */
  const int *widths;    /* [n_stages] output channels of each block's strided conv */
  int n_dilations;      /* residual units per block (1..4; 3)                     */
  const int *dilations; /* [n_dilations] (1, 3, 9)                                */
  int res_kernel;       /* dilated conv taps (odd; 7)                             */
  int out_kernel;       /* conv_out taps (odd; 3)                                 */
  int latent_channels;  /* C_lat, projection output channels (64)                 */
  int precision;        /* VOC_PREC_BF16X3 | VOC_PREC_F16W                        */
  int snake;            /* VOC_SNAKE | VOC_SNAKE_BETA                             */
} voc_enc_desc;

/* Number of parameter tensors, or -1 for an invalid desc.  Canonical order and PyTorch
 * layouts (weights already folded), C the input channels of a block, C' = widths[i]:
 *   conv_in.w [C0][C_in][in_kernel], conv_in.b [C0],
 *   per block i: per dilation: snake1.alpha [C], conv1.w [C][C][res_kernel], conv1.b [C],
 *                              snake2.alpha [C], conv2.w [C][C][1], conv2.b [C],
 *                snake.alpha [C], down.w [C'][C][2s], down.b [C'],
 *   snake_out.alpha [C_last], conv_out.w [C_last][C_last][out_kernel], conv_out.b [C_last],
 *   proj.w [C_lat][C_last][1], proj.b [C_lat].
 * Snake entries are [2][C] with VOC_SNAKE_BETA, as for the decoder. */
int vocoder_encoder_param_count(const voc_enc_desc *desc);
voc_status vocoder_encoder_param_shape(const voc_enc_desc *desc, int index, int dims[3],
                                       int *ndim);

/* Create an encoder on the current device (params as for vocoder_create: host pointers,
 * NULL biases mean zero, not retained).  On failure *out is NULL and
 * vocoder_encoder_last_error(NULL) describes the problem. */
voc_status vocoder_encoder_create(const voc_enc_desc *desc, const float *const *params,
                                  int n_params, vocoder_encoder_t **out);

/* Downsampling factor (product of the strides), or -1 for NULL. */
long long vocoder_encoder_hop(const vocoder_encoder_t *enc);

/* Device workspace of one encode of B items of L samples (0 for invalid sizes: L must be a
 * positive multiple of the hop, B * channels * L within the int range of the kernels). */
size_t vocoder_encoder_workspace_bytes(const vocoder_encoder_t *enc, int B, long long L);

/* Encode audio_dev [B][C_in][L] fp32 (device) into
 * latent_dev [B][C_lat][L / hop] fp32 (device), asynchronously on `stream`.  ws_dev: at
 * least vocoder_encoder_workspace_bytes, 256-byte aligned, caller-owned.  flags: 0,
 * VOC_FLAG_SYNC (wait and report VOC_DEVICE_TIMEOUT) and VOC_FLAG_PROFILE. */
voc_status vocoder_encode(vocoder_encoder_t *enc, const float *audio_dev, int B, long long L,
                          float *latent_dev, void *ws_dev, size_t ws_bytes, voc_stream_t stream,
                          unsigned flags);

/* Same encode from and to HOST buffers: copies the audio in, encodes, copies the latent
 * out and synchronises `stream` before returning.  ws_bytes >=
 * vocoder_encoder_workspace_bytes_host(enc, B, L) (the device workspace plus room for the
 * staging copies).  Page-locked host buffers give asynchronous copies. */
size_t vocoder_encoder_workspace_bytes_host(const vocoder_encoder_t *enc, int B, long long L);
voc_status vocoder_encode_host(vocoder_encoder_t *enc, const float *audio_host, int B,
                               long long L, float *latent_host, void *ws_dev, size_t ws_bytes,
                               voc_stream_t stream, unsigned flags);

/* Kernel launches of one vocoder_encode of B items of L samples (-1 for invalid sizes): the
 * deep layers of the low-rate blocks may run with split k, which adds a reduce launch each. */
int vocoder_encoder_launches(const vocoder_encoder_t *enc, int B, long long L);

/* Per-kernel records of the last encode run with VOC_FLAG_PROFILE, as vocoder_profile_*
 * for the decoder (a strided conv's FLOPs count its 2s taps over the real channels). */
int vocoder_encoder_profile_count(const vocoder_encoder_t *enc);
voc_status vocoder_encoder_profile_entry(vocoder_encoder_t *enc, int index, const char **name,
                                         double *ms, double *flops, double *bytes);
voc_status vocoder_encoder_profile_impl_bytes(vocoder_encoder_t *enc, int index,
                                              double *bytes);

/* Message of the last failed call on enc (NULL: of the last failure on this thread
 * without a context). */
const char *vocoder_encoder_last_error(const vocoder_encoder_t *enc);

/* Free the encoder (NULL is ignored). */
void vocoder_encoder_destroy(vocoder_encoder_t *enc);

#ifdef __cplusplus
}
#endif
#endif
