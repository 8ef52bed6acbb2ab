// layout.cu -- weight packing and layout transforms around the tensor-core
// kernels: NCHW <-> NHWC at the chain boundary, the latent de-normalisation
// (cortiq-engine "Module vae", VaeDecoder: z / scaling_factor + shift_factor)
// fused into that transpose, and V^T for the attention's second product.
#include "common.cuh"
#include "ptx.cuh"

namespace vae {

namespace {

// dst[o][tap * cin_pad + c] = tf32(w[o][c][tap]) (unrounded when !round);
// shortcut columns follow at taps * cin_pad + c; zero in every padding slot
// and padding row.
__global__ void pack_kernel(const float *__restrict__ w, int cout, int cin, int taps,
                            const float *__restrict__ wsc, int sc_cin, float *__restrict__ dst,
                            int rows, int ldb, int cin_pad, int round) {
  const long long total = static_cast<long long>(rows) * ldb;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int o = static_cast<int>(i / ldb);
    const int kidx = static_cast<int>(i % ldb);
    float v = 0.f;
    if (o < cout) {
      const int main = taps * cin_pad;
      if (kidx < main) {
        const int tap = kidx / cin_pad, c = kidx % cin_pad;
        if (c < cin) v = w[(static_cast<long long>(o) * cin + c) * taps + tap];
      } else {
        const int c = kidx - main;
        if (c < sc_cin) v = wsc[static_cast<long long>(o) * sc_cin + c];
      }
    }
    dst[i] = round ? round_tf32(v) : v;
  }
}

// Nearest-2x upsample followed by a 3x3 conv, per output parity (py, px): the
// taps ky that land on low-res row offset py - 1 + a (a = 0, 1) are those with
// floor((py + ky - 1) / 2) = py - 1 + a, and likewise for kx. Their weights
// act on the same input pixel, so they are summed into a 2x2 kernel:
// dst[par][o][(a * 2 + b) * cin_pad + c], par = py * 2 + px, TF32-rounded
// (unless !round).
__global__ void pack_upsample_kernel(const float *__restrict__ w, int cout, int cin,
                                     float *__restrict__ dst, int ldb, int cin_pad, int round) {
  const long long total = 4ll * cout * ldb;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = i / ldb;
    const int par = static_cast<int>(row / cout), o = static_cast<int>(row % cout);
    const int kidx = static_cast<int>(i % ldb);
    const int tap = kidx / cin_pad, c = kidx % cin_pad;
    const int py = par >> 1, px = par & 1, a = tap >> 1, b = tap & 1;
    float v = 0.f;
    if (c < cin) {
      const float *wc = w + (static_cast<long long>(o) * cin + c) * 9;
      for (int ky = 0; ky < 3; ++ky) {
        if (((py + ky + 1) >> 1) - py != a) continue;  // floor((py+ky-1)/2) - (py-1)
        for (int kx = 0; kx < 3; ++kx)
          if (((px + kx + 1) >> 1) - px == b) v += wc[ky * 3 + kx];
      }
    }
    dst[i] = round ? round_tf32(v) : v;
  }
}

// 32x32 tile transpose through shared memory, with an affine map and optional
// TF32 rounding on the way.
__global__ void transpose_kernel(const float *__restrict__ src, long long so, int sld,
                                 float *__restrict__ dst, long long dso, int dld, int rows,
                                 int cols, float alpha, float beta, int round) {
  __shared__ float tile[32][33];
  const int b = blockIdx.y;
  const int tiles_c = (cols + 31) / 32;
  const int r0 = static_cast<int>(blockIdx.x / tiles_c) * 32;
  const int c0 = static_cast<int>(blockIdx.x % tiles_c) * 32;
  const float *s = src + b * so;
  float *d = dst + b * dso;
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int r = r0 + dy, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[dy][threadIdx.x] = s[static_cast<long long>(r) * sld + c];
  }
  __syncthreads();
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int c = c0 + dy, r = r0 + threadIdx.x;
    if (r < rows && c < cols) {
      float v = fmaf(tile[threadIdx.x][dy], alpha, beta);
      if (round) v = round_tf32(v);
      d[static_cast<long long>(c) * dld + r] = v;
    }
  }
}

__global__ void pad_rows_kernel(const float *__restrict__ src, long long rows, int cols,
                                float *__restrict__ dst, int dcols) {
  const long long total = rows * dcols;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / dcols;
    const int c = static_cast<int>(i % dcols);
    dst[i] = c < cols ? src[r * cols + c] : 0.f;
  }
}

__global__ void add_kernel(float *dst, const float *a, const float *b, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    dst[i] = (a ? a[i] : 0.f) + (b ? b[i] : 0.f);
}

// Nearest-2x spatial upsample of NHWC images (every frame of a video on its
// own): dst[img][2y + a][2x + b][c] = src[img][y][x][c], float4 per thread.
__global__ void upsample2x_nhwc_kernel(const float4 *__restrict__ src, int h, int w, int c4,
                                       long long total, float4 *__restrict__ dst) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % c4);
    long long r = i / c4;
    const int x2 = static_cast<int>(r % (2 * w));
    r /= 2 * w;
    const int y2 = static_cast<int>(r % (2 * h));
    const long long img = r / (2 * h);
    dst[i] = src[((img * h + (y2 >> 1)) * w + (x2 >> 1)) * c4 + c];
  }
}

int grid_for(long long n, int threads) {
  long long g = (n + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  return static_cast<int>(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

int pack_conv_weights(const float *w, int cout, int cin, int taps, const float *w_sc,
                      int sc_cin, float *dst, int cout_rows, int ldb, cudaStream_t s,
                      int round) {
  if (!w || !dst || cout <= 0 || cin <= 0 || cout_rows < cout) return VAE_EINVAL;
  if (ldb != packed_ldb(cin, taps, w_sc ? sc_cin : 0)) return VAE_EINVAL;
  const long long total = static_cast<long long>(cout_rows) * ldb;
  pack_kernel<<<grid_for(total, 256), 256, 0, s>>>(w, cout, cin, taps, w_sc, w_sc ? sc_cin : 0,
                                                   dst, cout_rows, ldb, round_up32(cin), round);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

int pack_upsample_weights(const float *w, int cout, int cin, float *dst, cudaStream_t s,
                          int round) {
  if (!w || !dst || cout <= 0 || cin <= 0) return VAE_EINVAL;
  const int ldb = upsample_ldb(cin);
  pack_upsample_kernel<<<grid_for(4ll * cout * ldb, 256), 256, 0, s>>>(w, cout, cin, dst, ldb,
                                                                      round_up32(cin), round);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

int transpose(const float *src, long long src_outer_stride, int src_ld, float *dst,
              long long dst_outer_stride, int dst_ld, int outer, int rows, int cols, float alpha,
              float beta, int round, cudaStream_t s) {
  if (outer <= 0 || rows <= 0 || cols <= 0) return VAE_EINVAL;
  if (outer > 65535) return VAE_EUNSUPPORTED;
  const long long tiles = static_cast<long long>(ceil_div(cols, 32)) * ceil_div(rows, 32);
  if (tiles > 0x7fffffffll) return VAE_EUNSUPPORTED;
  dim3 grid(static_cast<unsigned>(tiles), outer);
  transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(src, src_outer_stride, src_ld, dst,
                                                 dst_outer_stride, dst_ld, rows, cols, alpha,
                                                 beta, round);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

int pad_rows(const float *src, long long rows, int cols, float *dst, int dst_cols,
             cudaStream_t s) {
  pad_rows_kernel<<<grid_for(rows * dst_cols, 256), 256, 0, s>>>(src, rows, cols, dst, dst_cols);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

int upsample_nearest2x_nhwc(const float *src, long long imgs, int h, int w, int c, float *dst,
                            cudaStream_t s) {
  if (!src || !dst || imgs <= 0 || h <= 0 || w <= 0 || c <= 0 || c % 4) return VAE_EINVAL;
  const long long total = imgs * 4ll * h * w * (c / 4);
  upsample2x_nhwc_kernel<<<grid_for(total, 256), 256, 0, s>>>(
      reinterpret_cast<const float4 *>(src), h, w, c / 4, total, reinterpret_cast<float4 *>(dst));
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

int add_bias(float *dst, const float *a, const float *b, int n, cudaStream_t s) {
  add_kernel<<<grid_for(n, 256), 256, 0, s>>>(dst, a, b, n);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

}  // namespace vae
