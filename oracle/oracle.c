/*
 * oracle.c -- plain CPU reference of the DAC-style vocoder decoder.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): used by the tests, the smoke check
 * and the CPU baseline of the benchmark; never by the product path.
 *
 * Double precision throughout.  Each layer is its textbook definition written
 * as direct loops.  The only liberty taken is the position of the independent
 * output-time loop: it is innermost so that the compiler can vectorise it,
 * which leaves the order in which each output element sums its terms exactly
 * the order of the definition (input channel, then tap).
 */
#include "oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

int oracle_param_count(const oracle_arch *a) {
  return (a->in_proj_channels > 0 ? 2 : 0) + 2 + a->n_stages * (3 + 6 * a->n_dilations) + 3;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.  A finite
   value a is a multiple of its quantum 2^(e - 10), e = floor(log2 a), and of 2^-24 below the
   normal range; rounding is to the nearest multiple, ties to the even multiple. */
static double round_half_one(double x) {
  const float f = (float)x; /* the library receives single-precision weights */
  const double a = fabs((double)f);
  if (a == 0.0 || !isfinite(a)) return (double)f;
  if (a >= 65520.0) return copysign(INFINITY, (double)f); /* halfway to 2^16 rounds up */
  int E;
  frexp(a, &E);        /* a = m 2^E, m in [0.5, 1): floor(log2 a) = E - 1 */
  int e = E - 1;
  if (e < -14) e = -14; /* subnormals share the quantum of the smallest binade */
  const double q = ldexp(1.0, e - 10);
  const double r = nearbyint(a / q); /* exact quotient; default rounding: ties to even */
  return copysign(r * q, (double)f);
}

void oracle_round_half(const double *x, long n, double *y) {
  for (long i = 0; i < n; ++i) y[i] = round_half_one(x[i]);
}

/* bfloat16: 8 significant bits (7 stored), binary32's exponent range.  Same steps as
 * round_half_one: single precision first, then the nearest multiple of the binade's quantum
 * 2^(e-7), ties to even; subnormals (below 2^-126) share the smallest binade's quantum; a
 * result of 2^128 or more is infinite. */
static double round_bf16_one(double x) {
  const float f = (float)x;
  const double a = fabs((double)f);
  if (a == 0.0 || !isfinite(a)) return (double)f;
  int E;
  frexp(a, &E);
  int e = E - 1;
  if (e < -126) e = -126;
  const double q = ldexp(1.0, e - 7);
  const double r = nearbyint(a / q) * q;
  if (r >= ldexp(1.0, 128)) return copysign(INFINITY, (double)f);
  return copysign(r, (double)f);
}

void oracle_round_bf16(const double *x, long n, double *y) {
  for (long i = 0; i < n; ++i) y[i] = round_bf16_one(x[i]);
}

long oracle_hop(const oracle_arch *a) {
  long h = 1;
  for (int i = 0; i < a->n_stages; ++i) h *= a->strides[i];
  return h;
}

/* minimaxmusic.cpp Architecture, "Models": w = g * v / ||v||, axis 0. */
int oracle_fold_weight_norm(const float *g, const float *v, int dim0, long rest, double *w) {
  for (int i = 0; i < dim0; ++i) {
    const float *row = v + (long)i * rest;
    double ss = 0.0;
    for (long j = 0; j < rest; ++j) ss += (double)row[j] * (double)row[j];
    double norm = sqrt(ss);
    if (!(norm > 0.0)) return -1;
    double scale = (double)g[i] / norm;
    for (long j = 0; j < rest; ++j) w[(long)i * rest + j] = scale * (double)row[j];
  }
  return 0;
}

/* minimaxmusic.cpp Architecture, "Flow VAE": y = x + sin^2(a x) / (a + 1e-9). */
void oracle_snake_row(const double *x, long n, double alpha, int identity, double *y) {
  if (identity) {
    if (y != x) memmove(y, x, (size_t)n * sizeof(double));
    return;
  }
  double inv_b = 1.0 / (alpha + 1e-9);
  for (long i = 0; i < n; ++i) {
    double s = sin(alpha * x[i]);
    y[i] = x[i] + s * s * inv_b;
  }
}

/* qwentts.cpp Architecture, "Audio tokenizer decoder": SnakeBeta exponentiates its stored
   alpha and beta; the divisor keeps the 1e-9 of the Snake formula. */
void oracle_snake_beta_row(const double *x, long n, double log_alpha, double log_beta, double *y) {
  const double a = exp(log_alpha);
  const double inv_b = 1.0 / (exp(log_beta) + 1e-9);
  for (long i = 0; i < n; ++i) {
    double s = sin(a * x[i]);
    y[i] = x[i] + s * s * inv_b;
  }
}

int oracle_conv1d(const double *x, int Cin, int T, const double *w, const double *b, int Cout,
                  int K, int dil, int pad_left, int pad_right, double *y) {
  long T_out = (long)T + pad_left + pad_right - (long)dil * (K - 1);
  if (T_out < 0 || Cin <= 0 || Cout <= 0 || K <= 0 || dil <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int co = 0; co < Cout; ++co) {
    double *yr = y + (long)co * T_out;
    double bias = b ? b[co] : 0.0;
    for (long t = 0; t < T_out; ++t) yr[t] = bias;
    for (int ci = 0; ci < Cin; ++ci) {
      const double *xr = x + (long)ci * T;
      for (int k = 0; k < K; ++k) {
        double wv = w[((long)co * Cin + ci) * K + k];
        long shift = (long)k * dil - pad_left; /* input index = t + shift */
        long t_lo = shift < 0 ? -shift : 0;
        long t_hi = T - shift; /* exclusive: t + shift < T */
        if (t_hi > T_out) t_hi = T_out;
        for (long t = t_lo; t < t_hi; ++t) yr[t] += wv * xr[t + shift];
      }
    }
  }
  return 0;
}

/* qwentts.cpp Architecture, "Custom GGML ops": col2im_1d scatter-add of the
 * [K*OC, T_in] column matrix into [T_out, OC] at position t*s + k - p. */
int oracle_conv_transpose1d(const double *x, int Cin, int T, const double *w, const double *b,
                            int Cout, int K, int stride, int pad_left, int T_out, double *y) {
  if (T_out < 0 || Cin <= 0 || Cout <= 0 || K <= 0 || stride <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int co = 0; co < Cout; ++co) {
    double *yr = y + (long)co * T_out;
    for (long j = 0; j < T_out; ++j) yr[j] = 0.0;
    for (int ci = 0; ci < Cin; ++ci) {
      const double *xr = x + (long)ci * T;
      const double *wr = w + ((long)ci * Cout + co) * K;
      for (long t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
          long j = t * stride + k - pad_left;
          if (j >= 0 && j < T_out) yr[j] += wr[k] * xr[t];
        }
      }
    }
    if (b)
      for (long j = 0; j < T_out; ++j) yr[j] += b[co];
  }
  return 0;
}

/* Snake applied per channel row of a [C][L] activation: alpha[c] per channel, or for
   SnakeBeta (beta != 0) log alpha in p[c] and log beta in p[C + c]. */
static void snake_rows(const double *x, int C, long L, const double *p, int identity, int beta,
                       double *y) {
#pragma omp parallel for schedule(static)
  for (int c = 0; c < C; ++c) {
    if (beta && !identity)
      oracle_snake_beta_row(x + (long)c * L, L, p[c], p[C + c], y + (long)c * L);
    else
      oracle_snake_row(x + (long)c * L, L, p[c], identity, y + (long)c * L);
  }
}

static void conv_pads(int padding, int K, int dil, int *pl, int *pr) {
  int span = dil * (K - 1);
  if (padding == ORACLE_PAD_CAUSAL) {
    *pl = span;
    *pr = 0;
  } else {
    *pl = span / 2;
    *pr = span - span / 2;
  }
}

/* minimaxmusic.cpp Architecture, "Flow VAE":
 *   conv_in k7 -> for each block: snake -> conv_t (stride s, k = 2s, pad s/2)
 *   -> 3 x res_unit (skip -> snake1 -> conv1 k7 dil d -> snake2 -> conv2 k1 -> + skip)
 *   -> snake_out -> conv_out k7 (with bias) -> tanh.
 * Causal variant (qwentts.cpp Architecture, "Audio tokenizer decoder" and
 * "Streaming decode"): every stride-1 conv pads (k-1)*d on the left only and the
 * transposed conv keeps the first T*s samples of its col2im output. */
int oracle_decode(const oracle_arch *a, const double *const *params, const float *latent, int B,
                  int T, double *audio, double *pre_tanh) {
  if (!a || !params || !latent || !audio || B <= 0 || T <= 0) return -1;
  const int ident = (a->flags & ORACLE_FLAG_SNAKE_IDENTITY) != 0;
  const long hop = oracle_hop(a);
  const long L_out = (long)T * hop;

  /* largest activation (channels x length) over the stack */
  long max_elems = (long)a->latent_channels * T;
  if ((long)a->in_proj_channels * T > max_elems) max_elems = (long)a->in_proj_channels * T;
  {
    long L = T;
    long e = (long)a->channels0 * L;
    if (e > max_elems) max_elems = e;
    for (int i = 0; i < a->n_stages; ++i) {
      L *= a->strides[i];
      e = (long)a->widths[i] * L;
      if (e > max_elems) max_elems = e;
    }
  }
  double *x = (double *)malloc((size_t)max_elems * sizeof(double));
  double *s = (double *)malloc((size_t)max_elems * sizeof(double));
  double *h = (double *)malloc((size_t)max_elems * sizeof(double));
  if (!x || !s || !h) {
    free(x), free(s), free(h);
    return -2;
  }

  for (int bi = 0; bi < B; ++bi) {
    int p = 0;
    /* latent item, widened to double */
    const float *lat = latent + (long)bi * a->latent_channels * T;
    for (long i = 0; i < (long)a->latent_channels * T; ++i) s[i] = (double)lat[i];

    /* optional 1x1 input projection (minimaxmusic.cpp Architecture, "Flow VAE": dec_in_proj,
       not weight normalised), then conv_in; no Snake in front of either */
    int c_in = a->latent_channels;
    if (a->in_proj_channels > 0) {
      oracle_conv1d(s, a->latent_channels, T, params[p], params[p + 1], a->in_proj_channels, 1, 1,
                    0, 0, h);
      memcpy(s, h, (size_t)a->in_proj_channels * T * sizeof(double));
      c_in = a->in_proj_channels;
      p += 2;
    }
    int pl, pr;
    conv_pads(a->padding, a->in_kernel, 1, &pl, &pr);
    oracle_conv1d(s, c_in, T, params[p], params[p + 1], a->channels0, a->in_kernel, 1, pl, pr, x);
    p += 2;

    int C = a->channels0;
    long L = T;
    for (int st = 0; st < a->n_stages; ++st) {
      const int stride = a->strides[st];
      const int Cout = a->widths[st];
      /* snake -> transposed conv, k = 2s */
      snake_rows(x, C, L, params[p], ident, a->snake_beta, s);
      const int Kt = 2 * stride;
      const int pad_t = (a->padding == ORACLE_PAD_CAUSAL) ? 0 : stride / 2;
      oracle_conv_transpose1d(s, C, (int)L, params[p + 1], params[p + 2], Cout, Kt, stride, pad_t,
                              (int)(L * stride), x);
      p += 3;
      C = Cout;
      L *= stride;
      /* residual units */
      for (int r = 0; r < a->n_dilations; ++r) {
        const int d = a->dilations[r];
        snake_rows(x, C, L, params[p], ident, a->snake_beta, s);
        conv_pads(a->padding, a->res_kernel, d, &pl, &pr);
        oracle_conv1d(s, C, (int)L, params[p + 1], params[p + 2], C, a->res_kernel, d, pl, pr, h);
        snake_rows(h, C, L, params[p + 3], ident, a->snake_beta, s);
        oracle_conv1d(s, C, (int)L, params[p + 4], params[p + 5], C, 1, 1, 0, 0, h);
        for (long i = 0; i < (long)C * L; ++i) x[i] += h[i];
        p += 6;
      }
    }
    /* snake_out -> conv_out (with bias) -> tanh */
    snake_rows(x, C, L, params[p], ident, a->snake_beta, s);
    conv_pads(a->padding, a->out_kernel, 1, &pl, &pr);
    double *y = audio + (long)bi * L_out;
    oracle_conv1d(s, C, (int)L, params[p + 1], params[p + 2], 1, a->out_kernel, 1, pl, pr, y);
    if (pre_tanh) memcpy(pre_tanh + (long)bi * L_out, y, (size_t)L_out * sizeof(double));
    if (!(a->flags & ORACLE_FLAG_NO_TANH))
      for (long i = 0; i < L_out; ++i) y[i] = tanh(y[i]);
  }
  free(x), free(s), free(h);
  return 0;
}

/* minimaxmusic.cpp Architecture, "Decode and stitch": the first window keeps
 * its left edge, later windows crop crop_left latents on the left, all but the
 * last crop crop_right on the right; segments are concatenated and clamped. */
/* ------------------------------------------------------------------ mirror encoder */
int oracle_enc_param_count(const oracle_enc_arch *a) {
  return 2 + a->n_stages * (6 * a->n_dilations + 3) + 3 + 2;
}

/* Conv1d with a stride: the definition, zero outside [0, T). */
int oracle_conv1d_strided(const double *x, int Cin, int T, const double *w, const double *b,
                          int Cout, int K, int stride, int pad_left, int T_out, double *y) {
  if (T_out < 0 || Cin <= 0 || Cout <= 0 || K <= 0 || stride <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int co = 0; co < Cout; ++co) {
    double *yr = y + (long)co * T_out;
    for (long t = 0; t < T_out; ++t) yr[t] = b ? b[co] : 0.0;
    for (int ci = 0; ci < Cin; ++ci) {
      const double *xr = x + (long)ci * T;
      const double *wr = w + ((long)co * Cin + ci) * K;
      for (int k = 0; k < K; ++k) {
        const double wk = wr[k];
        for (long t = 0; t < T_out; ++t) {
          const long j = t * stride + k - pad_left;
          if (j >= 0 && j < T) yr[t] += wk * xr[j];
        }
      }
    }
  }
  return 0;
}

/* minimaxmusic.cpp Architecture, "Flow VAE" (the encoder, the decoder's mirror). */
int oracle_encode(const oracle_enc_arch *a, const double *const *params, const float *audio,
                  int B, long L, double *latent) {
  if (!a || !params || !audio || !latent || B <= 0 || L <= 0) return -1;
  long hop = 1;
  for (int i = 0; i < a->n_stages; ++i) hop *= a->strides[i];
  if (L % hop) return -1;
  const int ident = (a->flags & ORACLE_FLAG_SNAKE_IDENTITY) != 0;
  long max_elems = (long)a->in_channels * L;
  {
    long Lc = L;
    int C = a->channels0;
    if ((long)C * Lc > max_elems) max_elems = (long)C * Lc;
    for (int i = 0; i < a->n_stages; ++i) {
      Lc /= a->strides[i];
      C = a->widths[i];
      if ((long)C * Lc > max_elems) max_elems = (long)C * Lc;
    }
  }
  double *x = (double *)malloc((size_t)max_elems * sizeof(double));
  double *s = (double *)malloc((size_t)max_elems * sizeof(double));
  double *h = (double *)malloc((size_t)max_elems * sizeof(double));
  if (!x || !s || !h) {
    free(x), free(s), free(h);
    return -2;
  }
  const long L_lat = L / hop;
  for (int bi = 0; bi < B; ++bi) {
    int p = 0;
    const float *au = audio + (long)bi * a->in_channels * L;
    for (long i = 0; i < (long)a->in_channels * L; ++i) s[i] = (double)au[i];
    int pl, pr;
    conv_pads(ORACLE_PAD_SYMMETRIC, a->in_kernel, 1, &pl, &pr);
    oracle_conv1d(s, a->in_channels, (int)L, params[p], params[p + 1], a->channels0, a->in_kernel, 1,
                  pl, pr, x);
    p += 2;
    int C = a->channels0;
    long Lc = L;
    for (int st = 0; st < a->n_stages; ++st) {
      for (int r = 0; r < a->n_dilations; ++r) { /* residual units, as in the decoder */
        const int d = a->dilations[r];
        snake_rows(x, C, Lc, params[p], ident, a->snake_beta, s);
        conv_pads(ORACLE_PAD_SYMMETRIC, a->res_kernel, d, &pl, &pr);
        oracle_conv1d(s, C, (int)Lc, params[p + 1], params[p + 2], C, a->res_kernel, d, pl, pr, h);
        snake_rows(h, C, Lc, params[p + 3], ident, a->snake_beta, s);
        oracle_conv1d(s, C, (int)Lc, params[p + 4], params[p + 5], C, 1, 1, 0, 0, h);
        for (long i = 0; i < (long)C * Lc; ++i) x[i] += h[i];
        p += 6;
      }
      /* snake -> strided conv, k = 2s, pad s/2 */
      const int sd = a->strides[st];
      const int Co = a->widths[st];
      snake_rows(x, C, Lc, params[p], ident, a->snake_beta, s);
      oracle_conv1d_strided(s, C, (int)Lc, params[p + 1], params[p + 2], Co, 2 * sd, sd, sd / 2,
                            (int)(Lc / sd), x);
      p += 3;
      C = Co;
      Lc /= sd;
    }
    /* snake_out -> conv_out -> posterior mean projection */
    snake_rows(x, C, Lc, params[p], ident, a->snake_beta, s);
    conv_pads(ORACLE_PAD_SYMMETRIC, a->out_kernel, 1, &pl, &pr);
    oracle_conv1d(s, C, (int)Lc, params[p + 1], params[p + 2], C, a->out_kernel, 1, pl, pr, h);
    oracle_conv1d(h, C, (int)Lc, params[p + 3], params[p + 4], a->latent_channels, 1, 1, 0, 0,
                  latent + (long)bi * a->latent_channels * L_lat);
  }
  free(x), free(s), free(h);
  return 0;
}

long oracle_stitched_length(int n_win, int win_frames, int crop_left, int crop_right, int hop) {
  if (n_win <= 0 || win_frames <= 0 || hop <= 0 || crop_left < 0 || crop_right < 0) return -1;
  long frames = 0;
  for (int w = 0; w < n_win; ++w) {
    int lo = (w == 0) ? 0 : crop_left;
    int hi = (w == n_win - 1) ? win_frames : win_frames - crop_right;
    if (hi < lo) return -1;
    frames += hi - lo;
  }
  return frames * hop;
}

int oracle_stitch(const double *decoded, int n_win, int n_sides, int win_frames, int crop_left,
                  int crop_right, int hop, double *out) {
  long len = oracle_stitched_length(n_win, win_frames, crop_left, crop_right, hop);
  if (len < 0 || n_sides <= 0) return -1;
  const long win_len = (long)win_frames * hop;
  for (int side = 0; side < n_sides; ++side) {
    long pos = 0;
    for (int w = 0; w < n_win; ++w) {
      int lo = (w == 0) ? 0 : crop_left;
      int hi = (w == n_win - 1) ? win_frames : win_frames - crop_right;
      const double *src = decoded + ((long)w * n_sides + side) * win_len;
      for (long j = (long)lo * hop; j < (long)hi * hop; ++j) {
        double v = src[j];
        out[(long)side * len + pos++] = v < -1.0 ? -1.0 : (v > 1.0 ? 1.0 : v);
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------ output stage */
/* minimaxmusic.cpp Architecture, "Post-processing" (readings in oracle.h). */
static int cmp_double(const void *a, const void *b) {
  const double x = *(const double *)a, y = *(const double *)b;
  return (x > y) - (x < y);
}

double oracle_abs_percentile(const float *x, long n, int peak_clip) {
  if (n <= 0) return 0.0;
  double *v = (double *)malloc((size_t)n * sizeof(double));
  if (!v) return -1.0;
  for (long i = 0; i < n; ++i) v[i] = fabs((double)x[i]);
  qsort(v, (size_t)n, sizeof(double), cmp_double);
  const double q = 1.0 - (double)peak_clip / 1e6;
  long k = (long)ceil(q * (double)n); /* 1-based rank */
  if (k < 1) k = 1;
  if (k > n) k = n;
  const double r = v[k - 1];
  free(v);
  return r;
}

long oracle_wav_bytes(int n_ch, long len, int bits) {
  if (n_ch < 1 || len < 0 || (bits != 16 && bits != 24 && bits != 32)) return -1;
  return 44 + (long)n_ch * len * (bits / 8);
}

static void put_le(unsigned char *p, unsigned long v, int nbytes) {
  for (int i = 0; i < nbytes; ++i) p[i] = (unsigned char)((v >> (8 * i)) & 0xFFu);
}

int oracle_encode_wav(const float *planar, int n_ch, long len, int sample_rate, int bits,
                      int peak_clip, unsigned char *out) {
  const long total = oracle_wav_bytes(n_ch, len, bits);
  if (total < 0 || !planar || !out || sample_rate <= 0 || peak_clip < 0 || peak_clip > 1000000)
    return -1;
  const int bps = bits / 8;
  const long data = (long)n_ch * len * bps;
  /* RIFF header */
  memcpy(out, "RIFF", 4);
  put_le(out + 4, (unsigned long)(36 + data), 4);
  memcpy(out + 8, "WAVEfmt ", 8);
  put_le(out + 16, 16, 4);
  put_le(out + 20, bits == 32 ? 3 : 1, 2);
  put_le(out + 22, (unsigned long)n_ch, 2);
  put_le(out + 24, (unsigned long)sample_rate, 4);
  put_le(out + 28, (unsigned long)sample_rate * n_ch * bps, 4);
  put_le(out + 32, (unsigned long)(n_ch * bps), 2);
  put_le(out + 34, (unsigned long)bits, 2);
  memcpy(out + 36, "data", 4);
  put_le(out + 40, (unsigned long)data, 4);
  unsigned char *p = out + 44;
  if (bits == 32) {
    for (long t = 0; t < len; ++t)
      for (int c = 0; c < n_ch; ++c, p += 4) memcpy(p, planar + (long)c * len + t, 4);
    return 0;
  }
  const double level = oracle_abs_percentile(planar, (long)n_ch * len, peak_clip);
  if (level < 0.0) return -1;
  /* the gain and the quantisation in IEEE single precision: the integer each sample
     rounds to is decided in the precision of the GPU path (the level is one of the
     |x| values, exact in float) */
  float gain = level > 0.0 ? 1.0f / (float)level : 1.0f;
  /* a subnormal level whose reciprocal overflows takes the largest finite gain, so that
     zeros stay zero (0 * inf would be undefined) */
  if (gain > FLT_MAX) gain = FLT_MAX;
  const float full = (float)((1L << (bits - 1)) - 1);
  for (long t = 0; t < len; ++t)
    for (int c = 0; c < n_ch; ++c, p += bps) {
      float y = planar[(long)c * len + t] * gain;
      if (y > 1.0f) y = 1.0f;
      if (y < -1.0f) y = -1.0f;
      const long q = (long)nearbyintf(y * full); /* default rounding mode: half to even */
      put_le(p, (unsigned long)q, bps);           /* two's complement, little endian */
    }
  return 0;
}
