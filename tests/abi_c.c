/* Plain C99 consumer of include/vocoder.h: includes the public header and calls
 * every entry point through its early-return (argument-validation) path, so it
 * needs no GPU and loads no model.  Built with -std=c99 -Wall -Werror -pedantic
 * (pattern of qwentts.cpp Architecture, "ABI guarantee"). */
#include <stdio.h>
#include <string.h>

#include "vocoder.h"

#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "FAILED line %d: %s\n", __LINE__, #cond); \
      return 1;                                                  \
    }                                                            \
  } while (0)

int main(void) {
  int strides[4] = {8, 8, 4, 2};
  int widths[4] = {768, 384, 192, 96};
  int dils[3] = {1, 3, 9};
  int dims[3];
  int nd = 0;
  float g = 1.0f, v[3] = {0.0f, 0.0f, 0.0f}, w[3];
  vocoder_t *ctx = (vocoder_t *)0;
  voc_desc d;
  memset(&d, 0, sizeof d);
  d.abi_version = VOC_ABI_VERSION;
  d.latent_channels = 64;
  d.in_kernel = 7;
  d.channels0 = 1536;
  d.n_stages = 4;
  d.strides = strides;
  d.widths = widths;
  d.n_dilations = 3;
  d.dilations = dils;
  d.res_kernel = 7;
  d.out_kernel = 7;
  d.out_channels = 1;
  d.padding = VOC_PAD_SYMMETRIC;
  d.precision = VOC_PREC_BF16X3;

  CHECK(vocoder_abi_version() == VOC_ABI_VERSION);
  CHECK(vocoder_param_count(&d) == 2 + 4 * (3 + 6 * 3) + 3);
  CHECK(vocoder_param_count((const voc_desc *)0) == -1);
  d.snake = VOC_SNAKE_BETA; /* SnakeBeta: every Snake parameter is [2][C] */
  CHECK(vocoder_param_shape(&d, 2, dims, &nd) == VOC_OK && nd == 2 && dims[0] == 2 && dims[1] == 1536);
  d.snake = 2;
  CHECK(vocoder_param_count(&d) == -1);
  d.snake = VOC_SNAKE;
  CHECK(vocoder_param_shape(&d, 2, dims, &nd) == VOC_OK && nd == 1 && dims[0] == 1536);
  CHECK(vocoder_param_shape(&d, 3, dims, &nd) == VOC_OK && nd == 3 && dims[0] == 1536 &&
        dims[1] == 768 && dims[2] == 16);
  CHECK(vocoder_param_shape(&d, 1000, dims, &nd) == VOC_INVALID_ARG);
  CHECK(vocoder_fold_weight_norm(&g, v, 1, 3, w) == VOC_INVALID_ARG); /* zero-norm row */
  CHECK(strlen(vocoder_last_error((const vocoder_t *)0)) > 0);
  CHECK(vocoder_fold_weight_norm((const float *)0, v, 1, 3, w) == VOC_INVALID_ARG);
  d.abi_version = VOC_ABI_VERSION + 1;
  CHECK(vocoder_create(&d, (const float *const *)0, 0, &ctx) == VOC_INVALID_ARG && ctx == 0);
  d.abi_version = VOC_ABI_VERSION;
  CHECK(vocoder_create(&d, (const float *const *)0, 0, &ctx) == VOC_INVALID_ARG);
  CHECK(vocoder_create(&d, (const float *const *)0, 0, (vocoder_t **)0) == VOC_INVALID_ARG);
  CHECK(vocoder_hop((const vocoder_t *)0) == -1);
  CHECK(vocoder_workspace_bytes((const vocoder_t *)0, 1, 1) == 0);
  CHECK(vocoder_workspace_bytes_host((const vocoder_t *)0, 1, 1) == 0);
  CHECK(vocoder_decode((vocoder_t *)0, (const float *)0, 1, 1, (float *)0, (void *)0, 0,
                       (voc_stream_t)0, 0) == VOC_INVALID_ARG);
  CHECK(vocoder_decode_host((vocoder_t *)0, (const float *)0, 1, 1, (float *)0, (void *)0, 0,
                            (voc_stream_t)0, 0) == VOC_INVALID_ARG);
  CHECK(vocoder_decode_static((vocoder_t *)0, (const float *)0, 1, 1, (float *)0, (voc_stream_t)0,
                              0) == VOC_INVALID_ARG);
  CHECK(vocoder_stitched_length(8, 689, 86, 258, 512) == 1589248LL);
  CHECK(vocoder_stitched_length(0, 689, 86, 258, 512) == -1);
  CHECK(vocoder_stitch((const float *)0, 8, 2, 689, 86, 258, 512, (float *)0, (voc_stream_t)0) ==
        VOC_INVALID_ARG);
  CHECK(vocoder_op_conv1d((const float *)0, 1, 1, 1, (const float *)0, (const float *)0, 1, 7, 1,
                          VOC_PAD_SYMMETRIC, (const float *)0, (float *)0,
                          (voc_stream_t)0) == VOC_INVALID_ARG);
  CHECK(vocoder_op_conv_transpose1d((const float *)0, 1, 1, 1, (const float *)0, (const float *)0,
                                    1, 2, VOC_PAD_SYMMETRIC, (const float *)0, (float *)0,
                                    (voc_stream_t)0) == VOC_INVALID_ARG);
  CHECK(vocoder_op_residual_unit((const float *)0, 1, 1, 1, (const float *)0, (const float *)0,
                                 (const float *)0, 7, 1, (const float *)0, (const float *)0,
                                 (const float *)0, VOC_PAD_SYMMETRIC, (float *)0,
                                 (voc_stream_t)0) == VOC_INVALID_ARG);
  CHECK(vocoder_launches_per_decode((const vocoder_t *)0, 1, 1) == -1);
  CHECK(vocoder_profile_count((const vocoder_t *)0) == 0);
  CHECK(vocoder_profile_entry((vocoder_t *)0, 0, (const char **)0, (double *)0, (double *)0,
                              (double *)0) == VOC_INVALID_ARG);
  {
    double ib = 0.0;
    volatile int cancel = 0;
    CHECK(vocoder_profile_impl_bytes((vocoder_t *)0, 0, &ib) == VOC_INVALID_ARG);
    CHECK(vocoder_set_cancel_flag((vocoder_t *)0, &cancel) == VOC_INVALID_ARG);
    CHECK(vocoder_set_wait_budget((vocoder_t *)0, 0) == VOC_INVALID_ARG);
    vocoder_debug_fail_allocation(-1);
    CHECK(vocoder_debug_live_allocations() >= 0);
  }
  vocoder_destroy((vocoder_t *)0);
  {  /* the mirror encoder: music layout 1 -> 64, strides 2, 4, 8, 8, widths up to 1024 */
    int es[4] = {2, 4, 8, 8};
    int ew[4] = {128, 256, 512, 1024};
    vocoder_encoder_t *enc = (vocoder_encoder_t *)0;
    voc_enc_desc e;
    memset(&e, 0, sizeof e);
    e.abi_version = VOC_ABI_VERSION;
    e.in_channels = 1;
    e.channels0 = 64;
    e.in_kernel = 7;
    e.n_stages = 4;
    e.strides = es;
    e.widths = ew;
    e.n_dilations = 3;
    e.dilations = dils;
    e.res_kernel = 7;
    e.out_kernel = 3;
    e.latent_channels = 64;
    e.precision = VOC_PREC_BF16W;
    e.snake = VOC_SNAKE;
    CHECK(vocoder_encoder_param_count(&e) == 2 + 4 * 21 + 5);
    CHECK(vocoder_encoder_param_shape(&e, 2 + 18 + 1, dims, &nd) == VOC_OK);  /* block 0 down.w */
    CHECK(nd == 3 && dims[0] == 128 && dims[1] == 64 && dims[2] == 4);
    CHECK(vocoder_encoder_create(&e, (const float *const *)0, 91, &enc) == VOC_INVALID_ARG);
    CHECK(enc == (vocoder_encoder_t *)0);
    CHECK(strlen(vocoder_encoder_last_error((const vocoder_encoder_t *)0)) > 0);
    CHECK(vocoder_encoder_hop((const vocoder_encoder_t *)0) == -1);
    CHECK(vocoder_encoder_workspace_bytes((const vocoder_encoder_t *)0, 1, 512) == 0);
    CHECK(vocoder_encoder_workspace_bytes_host((const vocoder_encoder_t *)0, 1, 512) == 0);
    CHECK(vocoder_encode((vocoder_encoder_t *)0, (const float *)0, 1, 512, (float *)0, (void *)0,
                         0, (voc_stream_t)0, 0) == VOC_INVALID_ARG);
    CHECK(vocoder_encode_host((vocoder_encoder_t *)0, (const float *)0, 1, 512, (float *)0,
                              (void *)0, 0, (voc_stream_t)0, 0) == VOC_INVALID_ARG);
    CHECK(vocoder_encoder_launches((const vocoder_encoder_t *)0, 1, 512) == -1);
    CHECK(vocoder_encoder_profile_count((const vocoder_encoder_t *)0) == 0);
    CHECK(vocoder_encoder_profile_entry((vocoder_encoder_t *)0, 0, (const char **)0, (double *)0,
                                        (double *)0, (double *)0) == VOC_INVALID_ARG);
    {
      double ib = 0.0;
      CHECK(vocoder_encoder_profile_impl_bytes((vocoder_encoder_t *)0, 0, &ib) == VOC_INVALID_ARG);
    }
    e.strides = (const int *)0;
    CHECK(vocoder_encoder_param_count(&e) == -1);
    vocoder_encoder_destroy((vocoder_encoder_t *)0);
  }
  printf("abi_c ok\n");
  return 0;
}
