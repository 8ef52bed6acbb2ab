// head.cu -- the decoder's last two steps fused: norm_out GroupNorm+SiLU
// followed by conv_out, a 3x3 conv down to a handful of output channels
// (cortiq-engine "Module vae", VaeDecoder: "... -> GroupNorm + SiLU ->
// conv_out").
//
// With 3 output channels the conv does 2*9*C*3 FLOP per pixel while reading
// 4*C bytes: far below the tensor cores' ridge, so it runs on the CUDA cores
// in FP32 and is bounded by reading the last activation once. Each CTA works
// on a (TH+2) x (TW+2) halo tile, 8 channels at a time: a TMA box brings the
// raw channels of chunk i+1 into shared memory while chunk i is convolved;
// the GroupNorm affine and SiLU are applied on the way from that box into
// channel planes (zeros outside the image: the conv's padding applies after
// the normalisation). Every thread accumulates four adjacent output pixels
// of one row, reading the planes with 16-byte loads and each weight once for
// all four; a warp covers one row of the tile, so the loads of a warp are
// consecutive 16-byte words. The chunk's weights and affine are fetched
// before its box is waited for. The RGB result is written NCHW.
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace vae {

namespace {

// Output tile TH = 8 rows x TW = 128 pixels; thread (ty, tx), tx < 32,
// computes pixels 4*tx .. 4*tx+3 of row ty (256 threads: with two CTAs per
// SM, as shared memory allows, 16 warps hide the latencies).
constexpr int kTH = 8, kTW = 128, kCC = 8;  // 4-channel chunks measured slower
constexpr int kThr = kTH * 32;     // 256 threads
constexpr int kHH = kTH + 2;       // halo rows
constexpr int kHW = kTW + 2;       // halo width 130
constexpr int kRow = 132;          // padded plane row (16-byte aligned rows)
constexpr int kChan = kHH * kRow;  // floats per channel plane
constexpr int kItems = kHH * kHW;  // halo pixels per chunk
constexpr uint32_t kRawBytes = kItems * kCC * sizeof(float);  // one TMA box
constexpr size_t kSmem = 1024 + kRawBytes + kCC * kChan * sizeof(float) +
                         9 * kCC * sizeof(float4) + 16;

// wpk: [C/32][9 taps][32 channels] x float4 (output channels padded to 4);
// CO output channels are accumulated (CO <= 4). tmX: the NHWC activation,
// box (8 channels, 130 pixels, 10 rows, 1 image), no swizzle.
template <int CO>
__global__ void __launch_bounds__(kThr)
    head_kernel(const __grid_constant__ CUtensorMap tmX, int H, int W, int C,
                const float *__restrict__ scale, const float *__restrict__ shift,
                const float4 *__restrict__ wpk, const float *__restrict__ bias,
                float *__restrict__ y, int *err) {
  extern __shared__ uint8_t head_smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(head_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float *raw = reinterpret_cast<float *>(base);  // [10][130][8]
  float *hal = raw + kItems * kCC;                // [8][10][132]
  float4 *wsm = reinterpret_cast<float4 *>(hal + kCC * kChan);
  uint64_t *bar = reinterpret_cast<uint64_t *>(wsm + 9 * kCC);
  volatile uint32_t *abort = reinterpret_cast<uint32_t *>(bar + 1);
  const int n = blockIdx.z;
  const int x0 = blockIdx.x * kTW, y0 = blockIdx.y * kTH;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort = 0u;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmX);
    mbar_arrive_expect_tx(bar, kRawBytes);
    tma_load_4d(raw, &tmX, bar, 0, x0 - 1, y0 - 1, n);
  }
  float acc[4][CO];  // [pixel][output channel]
#pragma unroll
  for (int o = 0; o < CO; ++o) {
    const float b = bias ? bias[o] : 0.f;
#pragma unroll
    for (int px = 0; px < 4; ++px) acc[px][o] = b;
  }
  const float *sc = scale + static_cast<size_t>(n) * C;
  const float *sh = shift + static_cast<size_t>(n) * C;
  uint32_t phase = 0;
  for (int c0 = 0; c0 < C; c0 += kCC) {
    // this chunk's weights and affine, in flight while the box is awaited
    float4 wreg = make_float4(0.f, 0.f, 0.f, 0.f);
    if (threadIdx.x < 9 * kCC) {
      const int tap = threadIdx.x / kCC, cg = c0 + threadIdx.x % kCC;
      wreg = __ldg(wpk + (cg / 32) * 288 + tap * 32 + (cg % 32));
    }
    const float4 ga = __ldg(reinterpret_cast<const float4 *>(sc + c0));
    const float4 gb = __ldg(reinterpret_cast<const float4 *>(sc + c0 + 4));
    const float4 ha = __ldg(reinterpret_cast<const float4 *>(sh + c0));
    const float4 hb = __ldg(reinterpret_cast<const float4 *>(sh + c0 + 4));
    const bool ok = mbar_wait(bar, phase, abort);
    if (__syncthreads_or(!ok)) {  // the box never landed: report, leave
      if (threadIdx.x == 0) atomicCAS(err, 0, static_cast<int>(VAE_EDEVICE_TIMEOUT));
      return;
    }
    phase ^= 1u;
    // raw box -> normalised channel planes
    const float gs[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    const float hs[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
    const float4 *raw4 = reinterpret_cast<const float4 *>(raw);
#pragma unroll 2
    for (int l = threadIdx.x; l < kItems; l += kThr) {
      const int hy = l / kHW, hx = l % kHW;
      const int gy = y0 - 1 + hy, gx = x0 - 1 + hx;
      const bool in = gy >= 0 && gy < H && gx >= 0 && gx < W;
      const float4 v0 = raw4[2 * l], v1 = raw4[2 * l + 1];
      const float t[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      float *d = hal + hy * kRow + hx;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float r = fmaf(t[j], gs[j], hs[j]);
        r = __fdividef(r, 1.0f + __expf(-r));  // SiLU, fast intrinsics
        d[j * kChan] = in ? r : 0.f;
      }
    }
    if (threadIdx.x < 9 * kCC) wsm[threadIdx.x] = wreg;
    __syncthreads();  // box consumed; planes and weights ready
    if (threadIdx.x == 0 && c0 + kCC < C) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, kRawBytes);
      tma_load_4d(raw, &tmX, bar, c0 + kCC, x0 - 1, y0 - 1, n);
    }
#pragma unroll 2
    for (int c = 0; c < kCC; ++c) {
#pragma unroll
      for (int ky = 0; ky < 3; ++ky) {
        const float4 *rowp =
            reinterpret_cast<const float4 *>(hal + c * kChan + (ty + ky) * kRow) + tx;
        const float4 a0 = rowp[0], a1 = rowp[1];
        const float xs[6] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y};
#pragma unroll
        for (int kx = 0; kx < 3; ++kx) {
          const float4 w = wsm[(ky * 3 + kx) * kCC + c];
          const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int px = 0; px < 4; ++px)
#pragma unroll
            for (int o = 0; o < CO; ++o) acc[px][o] = fmaf(xs[px + kx], wv[o], acc[px][o]);
        }
      }
    }
    __syncthreads();  // planes read before the next chunk overwrites them
  }
  const int gy = y0 + ty;
  if (gy >= H) return;
  const int gx = x0 + 4 * tx;
#pragma unroll
  for (int o = 0; o < CO; ++o) {
    float *dst = y + (static_cast<size_t>(n * CO + o) * H + gy) * W + gx;
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
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

namespace {

template <int CO>
int launch_head(const CUtensorMap &tm, int n, int h, int w, int c, const float *scale,
                const float *shift, const float4 *wv, const float *bias, float *y, int *err,
                cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(head_kernel<CO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kSmem));
  });
  if (attr != cudaSuccess) return VAE_ECUDA;
  if ((h + kTH - 1) / kTH > 65535) return VAE_EUNSUPPORTED;
  dim3 grid((w + kTW - 1) / kTW, (h + kTH - 1) / kTH, n);
  head_kernel<CO><<<grid, kThr, kSmem, s>>>(tm, h, w, c, scale, shift, wv, bias, y, err);
  return cudaGetLastError() == cudaSuccess ? VAE_OK : VAE_ECUDA;
}

}  // namespace

int head_gn_silu_conv(const float *x, int n, int h, int w, int c, const float *scale,
                      const float *shift, const float *wpk, const float *bias, int cout,
                      float *y, cudaStream_t s) {
  if (!x || !scale || !shift || !wpk || !y || n <= 0 || h <= 0 || w <= 0) return VAE_EINVAL;
  if (c % 32 || cout < 1 || cout > 4 || n > 65535) return VAE_EUNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(x) & 15) return VAE_EINVAL;
  const float4 *wv = reinterpret_cast<const float4 *>(wpk);
  int *err = device_error_word();
  if (!err) return VAE_ECUDA;
  CUtensorMap tm{};
  const uint64_t dims[4] = {static_cast<uint64_t>(c), static_cast<uint64_t>(w),
                            static_cast<uint64_t>(h), static_cast<uint64_t>(n)};
  const uint64_t str[3] = {static_cast<uint64_t>(c) * 4, static_cast<uint64_t>(w) * c * 4,
                           static_cast<uint64_t>(h) * w * c * 4};
  const uint32_t box[4] = {kCC, kHW, kHH, 1};
  VAE_TRY(encode_tiled(&tm, x, 4, dims, str, box, false));
  int rc;
  switch (cout) {
    case 1: rc = launch_head<1>(tm, n, h, w, c, scale, shift, wv, bias, y, err, s); break;
    case 2: rc = launch_head<2>(tm, n, h, w, c, scale, shift, wv, bias, y, err, s); break;
    case 3: rc = launch_head<3>(tm, n, h, w, c, scale, shift, wv, bias, y, err, s); break;
    default: rc = launch_head<4>(tm, n, h, w, c, scale, shift, wv, bias, y, err, s); break;
  }
  if (rc == VAE_OK) count_launches(1);
  return rc;
}

}  // namespace vae
