/*
 * oracle.h -- plain CPU reference of the DAC-style vocoder decoder.
 *
 * TEST INFRASTRUCTURE ONLY.  This library exists so that the tests, the smoke
 * check and the CPU baseline of the benchmark can compare the GPU path against
 * an obviously correct implementation.  Nothing on the product path may link,
 * load or call it, and it shares no code with the CUDA library.
 *
 * Every function works in double precision (fp32 inputs are widened once) and
 * follows the plain definition of the operation, with direct loops and no
 * blocking, fusion or algebraic rewriting:
 *
 *   Snake           minimaxmusic.cpp Architecture, section "Flow VAE":
 *                   y = x + sin^2(a*x) / (a + 1e-9), with a used as stored
 *                   (MiniMax-Music-3 -> CMF README, "What the conversion had to
 *                   get right": Snake reads alpha verbatim).
 *   weight norm     minimaxmusic.cpp Architecture, sections "Models" and "Flow
 *                   VAE": w = g * v / ||v|| along axis 0 of the stored tensor.
 *   conv1d          cross-correlation with zero padding and dilation, the
 *                   textbook definition of a 1-D convolution layer.
 *   convtranspose1d scatter-add of every input column into the output at
 *                   t*s + k - p, i.e. the col2im_1d op of qwentts.cpp
 *                   Architecture, section "Custom GGML ops", with
 *                   T_out = (T_in - 1)*s + K - 2p.
 *   decoder         minimaxmusic.cpp Architecture, section "Flow VAE" (layer
 *                   list), qwentts.cpp Architecture, section "Audio tokenizer
 *                   decoder" (causal speech variant).
 *   stitch          minimaxmusic.cpp Architecture, section "Decode and stitch".
 *
 * Parity pins: every function here is checked by tests that do not reuse its
 * code (closed forms, dense-matrix brute force, adjoint identities, library
 * routines on small cases, linearity, impulse responses, shift equivariance,
 * locality, causality).  No function is "parity unpinned".
 */
#ifndef VOCODER_ORACLE_H
#define VOCODER_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

/* padding modes of the whole stack */
#define ORACLE_PAD_SYMMETRIC 0 /* music decoder: k-tap convs pad d(k-1)/2 per side, ConvT crops s/2 */
#define ORACLE_PAD_CAUSAL 1    /* speech codec: convs pad d(k-1) on the left, ConvT keeps the first T*s */

/* test switches (used by the linearity and impulse-response pins) */
#define ORACLE_FLAG_SNAKE_IDENTITY 1 /* replace every Snake by the identity */
#define ORACLE_FLAG_NO_TANH 2        /* leave out the final tanh           */

typedef struct {
  int latent_channels; /* C_lat                                   */
  int channels0;       /* C_0, output channels of conv_in         */
  int in_kernel;       /* conv_in taps (7)                         */
  int n_stages;        /* upsampling stages                        */
  const int *strides;  /* [n_stages]                               */
  const int *widths;   /* [n_stages], output channels of stage i   */
  int n_dilations;     /* residual units per stage (3)             */
  const int *dilations;/* [n_dilations] (1, 3, 9)                  */
  int res_kernel;      /* dilated conv taps in a residual unit (7) */
  int out_kernel;      /* conv_out taps (7)                        */
  int padding;         /* ORACLE_PAD_*                             */
  int flags;           /* ORACLE_FLAG_*                            */
  int in_proj_channels;/* 0, or P: a 1x1 projection C_lat -> P (with bias, no weight norm)
                          before conv_in, which then maps P -> C_0 (the published music
                          model's dec_in_proj 64 -> 1024)                              */
  int snake_beta;      /* 0: Snake with alpha used as stored; 1: SnakeBeta, every Snake
                          parameter holds two rows [2][C] of log-scale alpha and beta
                          (qwentts.cpp Architecture, "Audio tokenizer decoder")         */
} oracle_arch;

/* number of parameter tensors of the stack, in the canonical order:
 *   [in_proj.w [P][Cl][1], in_proj.b [P]]   (only when in_proj_channels = P > 0)
 *   conv_in.w [C0][Cl or P][Kin], conv_in.b [C0],
 *   for each stage i (Cin -> Cout = widths[i], stride s):
 *     snake.alpha [Cin], convT.w [Cin][Cout][2s], convT.b [Cout],
 *     for each dilation d: snake1.alpha [Cout], conv1.w [Cout][Cout][Kres],
 *       conv1.b [Cout], snake2.alpha [Cout], conv2.w [Cout][Cout][1], conv2.b [Cout]
 *   snake_out.alpha [C_last], conv_out.w [1][C_last][Kout], conv_out.b [1]
 * With snake_beta every snake*.alpha entry is [2][C] instead: log alpha, then log beta. */
int oracle_param_count(const oracle_arch *a);

/* y[i] = x[i] rounded to single precision, then to IEEE 754 binary16 (half precision),
 * both round to nearest, ties to even: the convolution weights of the F16-weight precision
 * variant (minimaxmusic.cpp Architecture, "Flow VAE": conv weights are stored F16 on the
 * device with F32 activations).  Values at or beyond 65520 in magnitude become infinite;
 * magnitudes below 2^-14 use the subnormal quantum 2^-24. */
void oracle_round_half(const double *x, long n, double *y);

/* y[i] = x[i] rounded to single precision, then to bfloat16 (8 significant bits, binary32's
 * exponent range), both round to nearest, ties to even: the convolution weights of the
 * BF16-weight precision variant.  Results of 2^128 or more in magnitude are infinite;
 * magnitudes below 2^-126 use the subnormal quantum 2^-133. */
void oracle_round_bf16(const double *x, long n, double *y);

/* w[i, :] = g[i] * v[i, :] / ||v[i, :]||, the norm taken over everything but
 * axis 0 of the stored tensor (Conv1d [Cout][Cin][K]: per output channel;
 * ConvTranspose1d [Cin][Cout][K]: per input channel).  Returns -1 when a row of
 * v has zero norm, else 0. */
int oracle_fold_weight_norm(const float *g, const float *v, int dim0, long rest, double *w);

/* y[i] = x[i] + sin^2(alpha*x[i]) / (alpha + 1e-9) for one channel row of n values.
 * identity != 0 gives y = x. */
void oracle_snake_row(const double *x, long n, double alpha, int identity, double *y);

/* SnakeBeta with log-scale parameters: y[i] = x[i] + sin^2(e^la * x[i]) / (e^lb + 1e-9)
 * for one channel row of n values (exp applied to the stored alpha and beta). */
void oracle_snake_beta_row(const double *x, long n, double log_alpha, double log_beta, double *y);

/* y[co][t] = b[co] + sum_ci sum_k w[co][ci][k] * x[ci][t + k*dil - pad_left],
 * x taken as zero outside [0, T).  Output length T + pad_left + pad_right - dil*(K-1).
 * b may be NULL (zero bias). */
int oracle_conv1d(const double *x, int Cin, int T, const double *w, const double *b, int Cout,
                  int K, int dil, int pad_left, int pad_right, double *y);

/* y[co][t*s + k - pad_left] += w[ci][co][k] * x[ci][t] for every t, k, ci with the
 * target index in [0, T_out); then y[co][j] += b[co].  b may be NULL. */
int oracle_conv_transpose1d(const double *x, int Cin, int T, const double *w, const double *b,
                            int Cout, int K, int stride, int pad_left, int T_out, double *y);

/* total upsampling factor (product of strides) */
long oracle_hop(const oracle_arch *a);

/* Full decode.  params: oracle_param_count(a) pointers to double arrays in the
 * canonical order (weights already folded; a NULL bias means zero).
 * latent [B][Cl][T] fp32 -> audio [B][T*hop] double.  When pre_tanh is not NULL
 * it receives the conv_out result before tanh ([B][T*hop]).  0 on success. */
int oracle_decode(const oracle_arch *a, const double *const *params, const float *latent, int B,
                  int T, double *audio, double *pre_tanh);

/* Overlap-crop stitch (minimaxmusic.cpp Architecture, "Decode and stitch"):
 * decoded [n_win*n_sides][win_frames*hop] with item index 2w+side ordering
 * generalised to w*n_sides + side.  Window 0 keeps its left edge, later windows
 * drop crop_left frames on the left, all but the last drop crop_right frames on
 * the right; the kept pieces are concatenated per side and clamped to [-1, 1].
 * out [n_sides][oracle_stitched_length(...)]. */
long oracle_stitched_length(int n_win, int win_frames, int crop_left, int crop_right, int hop);
int oracle_stitch(const double *decoded, int n_win, int n_sides, int win_frames, int crop_left,
                  int crop_right, int hop, double *out);


/* ------------------------------------------------------------------ output stage
 * minimaxmusic.cpp Architecture, "Post-processing": planar float output, then percentile
 * peak normalisation targeting the 1 - peak_clip/1e6 percentile (peak_clip = 0: plain peak
 * normalisation; 32-bit float output is written raw, without normalisation), then WAV
 * encoding in memory.  Readings: the percentile is the nearest-rank order statistic of
 * |x| over every sample of every channel (the ceil(q*n)-th smallest, q = 1 - peak_clip/1e6);
 * the gain maps it to full scale 1.0 (gain 1 when it is 0); integer samples are
 * round-half-even(clamp(x*gain, -1, 1) * (2^(bits-1) - 1)) with the gain, the product and
 * the rounding in IEEE single precision; a WAV file is the 44-byte RIFF
 * header (PCM format 1 for 16 and 24 bits, IEEE float format 3 for 32 bits) followed by
 * the samples interleaved across channels, little endian. */

/* The nearest-rank percentile of |x| described above (0 for n = 0). */
double oracle_abs_percentile(const float *x, long n, int peak_clip);

/* Size in bytes of the WAV file of n_ch channels of len samples at `bits` (16, 24, 32). */
long oracle_wav_bytes(int n_ch, long len, int bits);

/* Write the WAV file: planar [n_ch][len] float -> out[oracle_wav_bytes(...)].  bits 16 or
 * 24 apply the normalisation with peak_clip; bits 32 writes the floats unchanged.
 * Returns 0, or -1 for bad arguments. */
int oracle_encode_wav(const float *planar, int n_ch, long len, int sample_rate, int bits,
                      int peak_clip, unsigned char *out);

/* ------------------------------------------------------------------ mirror encoder
 * minimaxmusic.cpp Architecture, "Flow VAE": the encoder is the decoder's mirror, per side
 *   conv_in k7 (1 -> C0)
 *   for every block (stride s, C_in -> C_out): 3 residual units at C_in (dilations 1, 3, 9),
 *       then Snake and a strided conv (k = 2s, stride s, pad s/2, C_in -> C_out),
 *   Snake -> conv_out (k3, C_last -> C_last) -> posterior mean projection (k1, C_last -> Cl).
 * Readings: the widths double block by block (64 -> 128 -> 256 -> 512 -> 1024 for the music
 * model); conv_out pads 1 on each side; no Snake between conv_out and the projection; all
 * convs have a bias; the same Snake as the decoder. */
typedef struct {
  int in_channels;     /* 1 (one side of a stereo track)                         */
  int channels0;       /* C0, conv_in output channels                             */
  int in_kernel;       /* conv_in taps (7)                                        */
  int n_stages;        /* downsampling blocks                                     */
  const int *strides;  /* [n_stages] (2, 4, 8, 8)                                 */
  const int *widths;   /* [n_stages] output channels of each block's strided conv */
  int n_dilations;     /* residual units per block (3)                            */
  const int *dilations;/* [n_dilations] (1, 3, 9)                                 */
  int res_kernel;      /* dilated conv taps (7)                                   */
  int out_kernel;      /* conv_out taps (3)                                       */
  int latent_channels; /* Cl, projection output channels (64)                     */
  int flags;           /* ORACLE_FLAG_SNAKE_IDENTITY honoured                     */
  int snake_beta;      /* as oracle_arch                                          */
} oracle_enc_arch;

/* Parameter tensors, canonical order:
 *   conv_in.w [C0][Cin][Kin], conv_in.b [C0],
 *   per block i (C = C_in of the block, C' = widths[i], stride s):
 *     per dilation: snake1.alpha [C], conv1.w [C][C][Kres], conv1.b [C], snake2.alpha [C],
 *                   conv2.w [C][C][1], conv2.b [C],
 *     snake.alpha [C], down.w [C'][C][2s], down.b [C'],
 *   snake_out.alpha [C_last], conv_out.w [C_last][C_last][Kout], conv_out.b [C_last],
 *   proj.w [Cl][C_last][1], proj.b [Cl]. */
int oracle_enc_param_count(const oracle_enc_arch *a);

/* y[co][t] = b[co] + sum_ci sum_k w[co][ci][k] * x[ci][t*stride + k - pad_left], x zero
 * outside [0, T), for t in [0, T_out).  b may be NULL. */
int oracle_conv1d_strided(const double *x, int Cin, int T, const double *w, const double *b,
                          int Cout, int K, int stride, int pad_left, int T_out, double *y);

/* Full encode: audio [B][Cin][L] fp32 (L a multiple of the product of the strides) ->
 * latent [B][Cl][L / prod(strides)] double.  0 on success. */
int oracle_encode(const oracle_enc_arch *a, const double *const *params, const float *audio,
                  int B, long L, double *latent);

#ifdef __cplusplus
}
#endif
#endif
