// tiled.cu -- kernels of the tiled decode (cortiq-engine 0.8.78, vae3d.rs:
// fn split_tiles, fn crop, fn blend, VideoVae::decode_clip; a tile schedule
// and cross-fade written there for another decoder, applied here to this
// one as a memory strategy for outputs the whole-image decode cannot hold).
//
// The chain decodes the tiles' latent crops as batches (every tile has the
// same size); these kernels cut the crops out of the latent and assemble the
// decoded tiles into the output image:
//   gather  z [n][c][zh][zw] -> crops [tile][c][tzh][tzw] for a range of
//           tiles (tile = (image, tile row i, tile column j), raster order)
//   blend   decoded tiles [tile][co][th][tw] -> rgb [n][co][H][W]: a pixel of
//           tile (i, j) at (ly, lx) is the tile's value, cross-faded over the
//           first yo[i-1] rows with the tile above (as decoded, its rows
//           th - e + ly) with weights 1 - ly/e and ly/e, then over the first
//           xo[j-1] columns with the tile to the left (as decoded) likewise;
//           a tile's last yo[i] rows and xo[j] columns are left to the next
//           tile (dropped), unless it is the last of its column / row.
#include "common.cuh"
#include "ops.cuh"

namespace vae {

namespace {

__global__ void gather_tiles_kernel(const float *__restrict__ z, int c, int zh, int zw,
                                    TileSchedule ts, long long t0, int count,
                                    float *__restrict__ dst) {
  const long long per = static_cast<long long>(c) * ts.tzh * ts.tzw;
  const long long total = per * count;
  const int per_img = ts.ny * ts.nx;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long tl = t0 + e / per;
    long long r = e % per;
    const int img = static_cast<int>(tl / per_img);
    const int ij = static_cast<int>(tl % per_img);
    const int i = ij / ts.nx, j = ij % ts.nx;
    const int xx = static_cast<int>(r % ts.tzw);
    r /= ts.tzw;
    const int yy = static_cast<int>(r % ts.tzh);
    const int ch = static_cast<int>(r / ts.tzh);
    const int sy = ts.ys[i] / ts.ratio + yy, sx = ts.xs[j] / ts.ratio + xx;
    dst[e] = z[((static_cast<long long>(img) * c + ch) * zh + sy) * zw + sx];
  }
}

// One block per (output row band of a tile, tile, image): threads stride
// over the band's pixels and channels.
__global__ void blend_tiles_kernel(const float *__restrict__ tiles, int co, TileSchedule ts,
                                   int height, int width, float *__restrict__ out) {
  const int img = blockIdx.z;
  const int ij = blockIdx.y;
  const int i = ij / ts.nx, j = ij % ts.nx;
  const int th = ts.th, tw = ts.tw;
  // the part of the tile that reaches the output
  const int rows = (i + 1 < ts.ny) ? th - ts.yo[i] : th;
  const int cols = (j + 1 < ts.nx) ? tw - ts.xo[j] : tw;
  const int ey = i > 0 ? min(ts.yo[i - 1], th) : 0;
  const int ex = j > 0 ? min(ts.xo[j - 1], tw) : 0;
  const long long tstride = static_cast<long long>(co) * th * tw;
  const long long base = static_cast<long long>(img) * ts.ny * ts.nx;
  const float *t = tiles + (base + ij) * tstride;
  const float *above = i > 0 ? tiles + (base + ij - ts.nx) * tstride : nullptr;
  const float *left = j > 0 ? tiles + (base + ij - 1) * tstride : nullptr;
  const int band = (rows + gridDim.x - 1) / gridDim.x;
  const int r0 = blockIdx.x * band, r1 = min(rows, r0 + band);
  const long long n_el = static_cast<long long>(co) * (r1 - r0) * cols;
  for (long long e = threadIdx.x; e < n_el; e += blockDim.x) {
    const int lx = static_cast<int>(e % cols);
    const long long q = e / cols;
    const int ly = r0 + static_cast<int>(q % (r1 - r0));
    const int c = static_cast<int>(q / (r1 - r0));
    const long long plane = static_cast<long long>(c) * th * tw;
    float v = t[plane + static_cast<long long>(ly) * tw + lx];
    if (ly < ey) {
      const float wb = static_cast<float>(ly) / static_cast<float>(ey);
      const float a = above[plane + static_cast<long long>(th - ey + ly) * tw + lx];
      v = a * (1.0f - wb) + v * wb;
    }
    if (lx < ex) {
      const float wb = static_cast<float>(lx) / static_cast<float>(ex);
      const float a = left[plane + static_cast<long long>(ly) * tw + (tw - ex + lx)];
      v = a * (1.0f - wb) + v * wb;
    }
    out[((static_cast<long long>(img) * co + c) * height + ts.oy[i] + ly) * width + ts.ox[j] +
        lx] = v;
  }
}

}  // namespace

int split_tiles(int length, int ratio, int tile, int min_overlap, int *starts, int *overlaps,
                int max_tiles, int *count, int *tile_len) {
  if (length <= 0 || ratio <= 0 || tile <= 0 || min_overlap < 0 || min_overlap >= tile)
    return VAE_EINVAL;
  if (tile >= length) {
    *count = 1;
    starts[0] = 0;
    *tile_len = length;
    return VAE_OK;
  }
  int n = (length + tile - 1) / tile;
  while (static_cast<long long>(tile) * n < static_cast<long long>(min_overlap) * (n - 1) + length)
    ++n;
  if (n > max_tiles) return VAE_EUNSUPPORTED;
  for (int k = 0; k < n - 1; ++k) overlaps[k] = min_overlap;
  const long long slack =
      static_cast<long long>(tile) * n - static_cast<long long>(min_overlap) * (n - 1) - length;
  for (long long k = 0; k < slack / ratio; ++k) overlaps[k % (n - 1)] += ratio;
  starts[0] = 0;
  for (int k = 0; k < n - 1; ++k) starts[k + 1] = starts[k] + tile - overlaps[k];
  *count = n;
  *tile_len = tile;
  return VAE_OK;
}

int make_tile_schedule(int height, int width, int ratio, int tile, int min_overlap,
                       TileSchedule *ts) {
  *ts = TileSchedule{};
  ts->ratio = ratio;
  VAE_TRY(split_tiles(height, ratio, tile, min_overlap, ts->ys, ts->yo, kMaxTilesPerAxis, &ts->ny,
                      &ts->th));
  VAE_TRY(split_tiles(width, ratio, tile, min_overlap, ts->xs, ts->xo, kMaxTilesPerAxis, &ts->nx,
                      &ts->tw));
  ts->tzh = ts->th / ratio;
  ts->tzw = ts->tw / ratio;
  // output position of each tile's kept part: every tile but the last of an
  // axis hands its overlap to the next one
  ts->oy[0] = ts->ox[0] = 0;
  for (int i = 1; i < ts->ny; ++i) ts->oy[i] = ts->oy[i - 1] + ts->th - ts->yo[i - 1];
  for (int j = 1; j < ts->nx; ++j) ts->ox[j] = ts->ox[j - 1] + ts->tw - ts->xo[j - 1];
  return VAE_OK;
}

int gather_latent_tiles(const float *z, int c, int zh, int zw, const TileSchedule &ts,
                        long long t0, int count, float *dst, cudaStream_t s) {
  const long long total = static_cast<long long>(c) * ts.tzh * ts.tzw * count;
  const long long blocks = std::min<long long>((total + 255) / 256, 8ll * num_sms());
  gather_tiles_kernel<<<static_cast<unsigned>(std::max<long long>(blocks, 1)), 256, 0, s>>>(
      z, c, zh, zw, ts, t0, count, dst);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

int blend_decoded_tiles(const float *tiles, int n, int co, const TileSchedule &ts, int height,
                        int width, float *out, cudaStream_t s) {
  const int bands = std::max(1, std::min(ts.th, (2 * num_sms() + ts.ny * ts.nx * n - 1) /
                                                    (ts.ny * ts.nx * n)));
  const dim3 grid(static_cast<unsigned>(bands), static_cast<unsigned>(ts.ny * ts.nx),
                  static_cast<unsigned>(n));
  blend_tiles_kernel<<<grid, 256, 0, s>>>(tiles, co, ts, height, width, out);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

}  // namespace vae
