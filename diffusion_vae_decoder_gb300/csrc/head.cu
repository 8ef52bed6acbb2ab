// head.cu -- the decoder's last two steps fused: norm_out GroupNorm+SiLU
// followed by conv_out, a 3x3 conv down to a handful of output channels
// (cortiq-engine "Module vae", VaeDecoder: "... -> GroupNorm + SiLU ->
// conv_out").
//
// With 3 output channels the conv does 2*9*C*3 FLOP per pixel while reading
// 4*C bytes: far below the tensor cores' ridge, so it runs on the CUDA cores
// in FP32 and is bounded by reading the last activation once. Each CTA
// normalises a (TH+2) x (TW+2) halo tile of 16 channels at a time on its way
// into shared memory (zeros outside the image: the conv's padding applies
// after the normalisation); every thread accumulates four adjacent output
// pixels, reading the halo with 16-byte loads and each weight once for all
// four. The RGB result is written NCHW.
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace vae {

namespace {

// Output tile TH rows x 128 pixels (TH = 8); thread (ty, tx) computes pixels
// 4*tx .. 4*tx+3 of row ty. Channels are staged 16 at a time.
constexpr int kTW = 128, kCC = 16;
constexpr int kHW = kTW + 2;  // halo width 130
constexpr int kRow = 132;     // padded halo row (16-byte aligned rows)
constexpr int kBatch = 7;
template <int TH>
struct HeadCfg {
  static constexpr int kHH = TH + 2;                   // halo rows
  static constexpr int kChan = kHH * kRow;             // floats per staged channel
  static constexpr int kThr = TH * 32;                 // threads
  static constexpr size_t kSmem = (kCC * kChan) * sizeof(float) + 9 * kCC * sizeof(float4);
  static constexpr int kItems = kHH * kHW * (kCC / 4);  // float4 halo loads per chunk
  static constexpr int kPer = (kItems + kThr - 1) / kThr;
};

// wpk: [C/32][9 taps][32 channels] x float4 (output channels padded to 4);
// CO output channels are accumulated (CO <= 4).
template <int CO, int TH>
__global__ void __launch_bounds__(TH * 32)
    head_kernel(const float *__restrict__ x, int H, int W, int C, const float *__restrict__ scale,
                const float *__restrict__ shift, const float4 *__restrict__ wpk,
                const float *__restrict__ bias, float *__restrict__ y) {
  constexpr int cout = CO;
  using HC = HeadCfg<TH>;
  constexpr int kHH = HC::kHH, kChan = HC::kChan, kItems = HC::kItems, kPer = HC::kPer;
  constexpr int kThr = HC::kThr;
  extern __shared__ float4 head_smem[];
  float *hal = reinterpret_cast<float *>(head_smem);
  float4 *wsm = reinterpret_cast<float4 *>(hal + kCC * kChan);
  const int n = blockIdx.z;
  const int x0 = blockIdx.x * kTW, y0 = blockIdx.y * TH;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  float acc[4][4];  // [pixel][output channel]
#pragma unroll
  for (int o = 0; o < 4; ++o) {
    const float b = (o < cout && bias) ? bias[o] : 0.f;
#pragma unroll
    for (int px = 0; px < 4; ++px) acc[px][o] = b;
  }
  const float *xn = x + static_cast<size_t>(n) * H * W * C;
  const float *sc = scale + static_cast<size_t>(n) * C;
  const float *sh = shift + static_cast<size_t>(n) * C;
  for (int c0 = 0; c0 < C; c0 += kCC) {
    __syncthreads();
    // Halo: four lanes per pixel read its 16 channels (64 contiguous bytes),
    // eight pixels per warp, kBatch independent loads in flight per thread.
    // Each lane stores its four channels in an order rotated by its quad
    // index, so the transposing shared stores of a warp hit 32 distinct banks
    // (one channel plane is 8 banks from the next: kChan = 8 mod 32).
    const int q4 = threadIdx.x & 3;  // fixed: the item stride (threads) is a multiple of 4
    const int cq = c0 + q4 * 4;
    const float4 ga = __ldg(reinterpret_cast<const float4 *>(sc + cq));
    const float4 gb = __ldg(reinterpret_cast<const float4 *>(sh + cq));
    float *dq = hal + (q4 * 4) * kChan;
#pragma unroll 1
    for (int b0 = 0; b0 < kPer; b0 += kBatch) {
      float4 v[kBatch];
      bool in[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int l = threadIdx.x + (b0 + u) * kThr;
        const int pix = l >> 2;
        const int gy = y0 + pix / kHW - 1, gx = x0 + pix % kHW - 1;
        in[u] = l < kItems && gy >= 0 && gy < H && gx >= 0 && gx < W;
        v[u] = in[u] ? __ldg(reinterpret_cast<const float4 *>(
                           xn + (static_cast<size_t>(gy) * W + gx) * C + cq))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int l = threadIdx.x + (b0 + u) * kThr;
        if (l >= kItems) break;
        const int pix = l >> 2;
        float4 t = v[u];
        if (in[u]) {
          t.x = fmaf(t.x, ga.x, gb.x);
          t.y = fmaf(t.y, ga.y, gb.y);
          t.z = fmaf(t.z, ga.z, gb.z);
          t.w = fmaf(t.w, ga.w, gb.w);
          t.x = __fdividef(t.x, 1.0f + __expf(-t.x));  // SiLU, fast intrinsics
          t.y = __fdividef(t.y, 1.0f + __expf(-t.y));
          t.z = __fdividef(t.z, 1.0f + __expf(-t.z));
          t.w = __fdividef(t.w, 1.0f + __expf(-t.w));
        }
        float *d = dq + (pix / kHW) * kRow + pix % kHW;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int jj = (j + q4) & 3;
          d[jj * kChan] = jj == 0 ? t.x : jj == 1 ? t.y : jj == 2 ? t.z : t.w;
        }
      }
    }
    for (int l = threadIdx.x; l < 9 * kCC; l += kThr) {
      const int tap = l / kCC, c = l % kCC;
      const int cg = c0 + c;
      wsm[l] = wpk[(cg / 32) * 288 + tap * 32 + (cg % 32)];
    }
    __syncthreads();
#pragma unroll 2
    for (int c = 0; c < kCC; ++c) {
#pragma unroll
      for (int ky = 0; ky < 3; ++ky) {
        const float4 *rowp =
            reinterpret_cast<const float4 *>(hal + c * kChan + (ty + ky) * kRow + 4 * tx);
        const float4 a = rowp[0], b = rowp[1];
        const float xs[6] = {a.x, a.y, a.z, a.w, b.x, b.y};
#pragma unroll
        for (int kx = 0; kx < 3; ++kx) {
          const float4 w = wsm[(ky * 3 + kx) * kCC + c];
#pragma unroll
          for (int px = 0; px < 4; ++px) {
            const float xv = xs[px + kx];
            acc[px][0] = fmaf(xv, w.x, acc[px][0]);
            if (CO > 1) acc[px][1] = fmaf(xv, w.y, acc[px][1]);
            if (CO > 2) acc[px][2] = fmaf(xv, w.z, acc[px][2]);
            if (CO > 3) acc[px][3] = fmaf(xv, w.w, acc[px][3]);
          }
        }
      }
    }
  }
  const int gy = y0 + ty, gx = x0 + 4 * tx;
  if (gy >= H) return;
#pragma unroll
  for (int o = 0; o < 4; ++o) {
    if (o >= cout) break;
    float *dst = y + (static_cast<size_t>(n * cout + o) * H + gy) * W + gx;
    if (gx + 3 < W && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
      *reinterpret_cast<float4 *>(dst) = make_float4(acc[0][o], acc[1][o], acc[2][o], acc[3][o]);
    } else {
#pragma unroll
      for (int px = 0; px < 4; ++px)
        if (gx + px < W) dst[px] = acc[px][o];
    }
  }
}

// w [cout][C][3][3] -> [C/32][9][32][4], zero-padded output channels.
__global__ void head_pack_kernel(const float *__restrict__ w, int cout, int C, float *dst) {
  const int total = C * 9 * 4;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int o = i & 3;
    const int c32 = (i >> 2) & 31;
    const int tap = (i >> 7) % 9;
    const int chunk = i / (4 * 32 * 9);
    const int c = chunk * 32 + c32;
    dst[i] = (o < cout) ? w[(static_cast<size_t>(o) * C + c) * 9 + tap] : 0.f;
  }
}

}  // namespace

bool head_supported(int cin, int cout, int k) { return k == 3 && cout <= 4 && cin % 32 == 0; }

size_t head_packed_floats(int cin) { return static_cast<size_t>(cin) * 9 * 4; }

int head_pack_weights(const float *w, int cout, int cin, float *dst, cudaStream_t s) {
  if (!head_supported(cin, cout, 3)) return VAE_EUNSUPPORTED;
  const int total = cin * 9 * 4;
  head_pack_kernel<<<(total + 255) / 256, 256, 0, s>>>(w, cout, cin, dst);
  if (cudaGetLastError() != cudaSuccess) return VAE_ECUDA;
  count_launches(1);
  return VAE_OK;
}

namespace {

template <int CO, int TH>
int launch_head(const float *x, int n, int h, int w, int c, const float *scale,
                const float *shift, const float4 *wv, const float *bias, float *y,
                cudaStream_t s) {
  using HC = HeadCfg<TH>;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(head_kernel<CO, TH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(HC::kSmem));
  });
  if (attr != cudaSuccess) return VAE_ECUDA;
  if ((h + TH - 1) / TH > 65535) return VAE_EUNSUPPORTED;
  dim3 grid((w + kTW - 1) / kTW, (h + TH - 1) / TH, n);
  head_kernel<CO, TH><<<grid, HC::kThr, HC::kSmem, s>>>(x, h, w, c, scale, shift, wv, bias, y);
  return cudaGetLastError() == cudaSuccess ? VAE_OK : VAE_ECUDA;
}

template <int TH>
int launch_head_co(int cout, const float *x, int n, int h, int w, int c, const float *scale,
                   const float *shift, const float4 *wv, const float *bias, float *y,
                   cudaStream_t s) {
  switch (cout) {
    case 1: return launch_head<1, TH>(x, n, h, w, c, scale, shift, wv, bias, y, s);
    case 2: return launch_head<2, TH>(x, n, h, w, c, scale, shift, wv, bias, y, s);
    case 3: return launch_head<3, TH>(x, n, h, w, c, scale, shift, wv, bias, y, s);
    default: return launch_head<4, TH>(x, n, h, w, c, scale, shift, wv, bias, y, s);
  }
}

}  // namespace

int head_gn_silu_conv(const float *x, int n, int h, int w, int c, const float *scale,
                      const float *shift, const float *wpk, const float *bias, int cout,
                      float *y, cudaStream_t s) {
  if (!x || !scale || !shift || !wpk || !y || n <= 0 || h <= 0 || w <= 0) return VAE_EINVAL;
  if (c % 32 || cout < 1 || cout > 4 || n > 65535) return VAE_EUNSUPPORTED;
  const float4 *wv = reinterpret_cast<const float4 *>(wpk);
  // 8-row tiles (2-row tiles measured slower even on small images: the halo
  // overhead outweighs the extra CTAs)
  const int rc = launch_head_co<8>(cout, x, n, h, w, c, scale, shift, wv, bias, y, s);
  if (rc == VAE_OK) count_launches(1);
  return rc;
}

}  // namespace vae
