// ops.cuh -- internal pieces shared by the single-op entry points and the
// chain executor.
#pragma once
#include "common.cuh"

namespace vae {

// Make an NHWC copy of x with channels padded to cpad (zeros), applying
// x * alpha + beta and TF32 rounding on the way; passes x through untouched
// when it is already NHWC, unpadded and no transform is asked for.
int stage_nhwc(const float *x, int n, int c, long long spatial, int layout, float *staging,
               int cpad, float alpha, float beta, int round, const float **out, cudaStream_t s);
int unstage_nchw(const float *src_nhwc, int n, int c, long long spatial, float *dst_nchw,
                 cudaStream_t s);

struct AttnScratch {
  float *t, *qkv, *vt, *s, *o;
  void *gn;
};
size_t attn_ws_bytes(int n, int c, int L, int layout);
// exact: split-TF32 products on FP32 operands (weights packed unrounded),
// through the score-matrix path.
int attention_nhwc(const float *x, int n, int c, int L, int groups, float eps,
                   const float *gn_w, const float *gn_b, const float *wqkv, const float *bqkv,
                   const float *wo, const float *bo, float *y, const AttnScratch &sc,
                   cudaStream_t s, bool exact = false);

}  // namespace vae
