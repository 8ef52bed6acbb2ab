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
  float *rs;  // attn_rs_floats(L): the score rows' softmax statistics
};
size_t attn_ws_bytes(int n, int c, int L, int layout);
// Room for the per-column-tile softmax statistics of L score rows and the
// merged per-row max and reciprocal sum.
size_t attn_rs_floats(int L);
// exact: split-TF32 products on FP32 operands (weights packed unrounded),
// through the score-matrix path.
int attention_nhwc(const float *x, int n, int c, int L, int groups, float eps,
                   const float *gn_w, const float *gn_b, const float *wqkv, const float *bqkv,
                   const float *wo, const float *bo, float *y, const AttnScratch &sc,
                   cudaStream_t s, bool exact = false);

// ---------------------------------------------------------------- tiled decode
// Tile schedule of one output plane (pixels): tiles (i, j) of th x tw pixels
// starting at (ys[i], xs[j]), overlapping the next by yo[i] / xo[j]; the kept
// part of tile (i, j) lands at output (oy[i], ox[j]). Passed to the kernels
// by value.
constexpr int kMaxTilesPerAxis = 128;
struct TileSchedule {
  int ny = 0, nx = 0, th = 0, tw = 0, ratio = 1, tzh = 0, tzw = 0;
  int ys[kMaxTilesPerAxis], yo[kMaxTilesPerAxis], oy[kMaxTilesPerAxis];
  int xs[kMaxTilesPerAxis], xo[kMaxTilesPerAxis], ox[kMaxTilesPerAxis];
};
// One axis: the fewest tiles of `tile` pixels with overlaps >= min_overlap,
// the slack added to the overlaps `ratio` pixels at a time round robin (a
// single tile of the whole length when it fits).
int split_tiles(int length, int ratio, int tile, int min_overlap, int *starts, int *overlaps,
                int max_tiles, int *count, int *tile_len);
int make_tile_schedule(int height, int width, int ratio, int tile, int min_overlap,
                       TileSchedule *ts);
// Latent crops of tiles [t0, t0 + count) (tile = (image, i, j), raster order).
int gather_latent_tiles(const float *z, int c, int zh, int zw, const TileSchedule &ts,
                        long long t0, int count, float *dst, cudaStream_t s);
// Cross-fade and place every decoded tile ([n * ny * nx][co][th][tw]).
int blend_decoded_tiles(const float *tiles, int n, int co, const TileSchedule &ts, int height,
                        int width, float *out, cudaStream_t s);

}  // namespace vae
