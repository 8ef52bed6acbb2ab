// softmax.cu -- row softmax of the mid-block attention scores.
//
// cortiq-engine "Module vae", struct VaeAttnRef: softmax(q k^T / sqrt(c));
// the row softmax subtracts the row maximum, exponentiates and divides by the
// sum (vae3d.rs fn softmax_inplace). Rows are written back in place, rounded
// to TF32 because they are the A operand of the P.V tensor-core product (or
// left in FP32 for the split-TF32 product, which splits them itself); the
// padding columns [L, ld) are set to zero so that the padded reduction of P.V
// adds exact zeros.
#include "common.cuh"
#include "ptx.cuh"

namespace vae {

namespace {

constexpr int kThreads = 512;
constexpr int kPerThread = 32;  // rows up to 16384 stay in registers

__device__ __forceinline__ float block_reduce(float v, bool is_max, float *sh) {
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  v = lane < (blockDim.x >> 5) ? sh[lane] : (is_max ? -INFINITY : 0.f);
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  return v;
}

// Row length ld <= kThreads * kPerThread (ld a multiple of 4): the row lives
// in registers, read and written with 16-byte accesses. One block reduction
// of per-thread (max, sum of exp) pairs replaces separate max and sum passes:
// each thread keeps exp(v - its own max) and rescales by exp(own max - row
// max) at the end.
__global__ void __launch_bounds__(kThreads) softmax_reg(float *s, int L, int ld, float scale,
                                                        int round) {
  __shared__ float shm[32], shs[32];
  constexpr int kVec = kPerThread / 4;
  float4 *row = reinterpret_cast<float4 *>(s + static_cast<long long>(blockIdx.x) * ld);
  const int ld4 = ld >> 2;
  float v[kPerThread];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const int q = threadIdx.x + i * kThreads;
    const float4 x = q < ld4 ? row[q] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[4 * i + k] = 4 * q + k < L ? e[k] * scale : -INFINITY;
      mx = fmaxf(mx, v[4 * i + k]);
    }
  }
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    v[i] = mx == -INFINITY ? 0.f : __expf(v[i] - mx);  // exp(-inf) = 0 for the padding
    sum += v[i];
  }
  // (max, sum) merge: warp butterfly, then across warps
  float m = mx, t = sum;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float t2 = __shfl_xor_sync(0xffffffffu, t, o);
    const float mm = fmaxf(m, m2);
    t = (m == -INFINITY ? 0.f : t * __expf(m - mm)) + (m2 == -INFINITY ? 0.f : t2 * __expf(m2 - mm));
    m = mm;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    shm[warp] = m;
    shs[warp] = t;
  }
  __syncthreads();
  m = lane < (kThreads >> 5) ? shm[lane] : -INFINITY;
  t = lane < (kThreads >> 5) ? shs[lane] : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float t2 = __shfl_xor_sync(0xffffffffu, t, o);
    const float mm = fmaxf(m, m2);
    t = (m == -INFINITY ? 0.f : t * __expf(m - mm)) + (m2 == -INFINITY ? 0.f : t2 * __expf(m2 - mm));
    m = mm;
  }
  const float f = (mx == -INFINITY ? 0.f : __expf(mx - m)) / t;
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const int q = threadIdx.x + i * kThreads;
    if (q < ld4) {
      float4 o;  // padding columns: v = 0 there, so they store exact zeros
      o.x = v[4 * i] * f;
      o.y = v[4 * i + 1] * f;
      o.z = v[4 * i + 2] * f;
      o.w = v[4 * i + 3] * f;
      if (round) {
        o.x = round_tf32(o.x);
        o.y = round_tf32(o.y);
        o.z = round_tf32(o.z);
        o.w = round_tf32(o.w);
      }
      row[q] = o;
    }
  }
}

// Any row length: three sweeps over global memory.
__global__ void __launch_bounds__(kThreads) softmax_long(float *s, int L, int ld, float scale,
                                                         int round) {
  __shared__ float sh[32];
  float *row = s + static_cast<long long>(blockIdx.x) * ld;
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < L; j += kThreads) mx = fmaxf(mx, row[j] * scale);
  mx = block_reduce(mx, true, sh);
  float sum = 0.f;
  for (int j = threadIdx.x; j < L; j += kThreads) sum += expf(row[j] * scale - mx);
  sum = block_reduce(sum, false, sh);
  const float inv = 1.0f / sum;
  for (int j = threadIdx.x; j < L; j += kThreads) {
    const float v = expf(row[j] * scale - mx) * inv;
    row[j] = round ? round_tf32(v) : v;
  }
  for (int j = L + threadIdx.x; j < ld; j += kThreads) row[j] = 0.f;
}

// (max, sum of exp(v - max)) pairs merged; a pair with no value is
// (-inf, 0) and leaves the other unchanged.
__device__ __forceinline__ float2 merge_stats(float2 a, float2 b) {
  if (b.x == -INFINITY) return a;
  if (a.x == -INFINITY) return b;
  const float mx = fmaxf(a.x, b.x);
  return make_float2(mx, a.y * __expf(a.x - mx) + b.y * __expf(b.x - mx));
}

// One warp per row: the row's per-tile statistics merged into its max and
// the reciprocal of its sum of exponentials.
__global__ void __launch_bounds__(256) softmax_stats_merge(const float2 *__restrict__ part,
                                                           int rows, int tiles, int ld,
                                                           float *__restrict__ m,
                                                           float *__restrict__ inv_l) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float2 acc = make_float2(-INFINITY, 0.f);
  for (int t = lane; t < tiles; t += 32)
    acc = merge_stats(acc, part[static_cast<long long>(row) * ld + t]);
  for (int o = 16; o > 0; o >>= 1) {
    const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, acc.x, o),
                                     __shfl_xor_sync(0xffffffffu, acc.y, o));
    acc = merge_stats(acc, other);
  }
  if (lane == 0) {
    m[row] = acc.x;
    inv_l[row] = 1.0f / acc.y;
  }
}

}  // namespace

int softmax_merge_stats(const float2 *part, int rows, int tiles, int ld, float *m, float *inv_l,
                        cudaStream_t st) {
  if (!part || !m || !inv_l || rows <= 0 || tiles <= 0 || ld < tiles) return VAE_EINVAL;
  softmax_stats_merge<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(part, rows, tiles,
                                                                            ld, m, inv_l);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

int softmax_rows(float *s, long long rows, int L, int ld, float scale, cudaStream_t st,
                 int round) {
  if (!s || rows <= 0 || L <= 0 || ld < L) return VAE_EINVAL;
  if (rows > 0x7fffffffll) return VAE_EUNSUPPORTED;
  if (ld <= kThreads * kPerThread && ld % 4 == 0 &&
      (reinterpret_cast<uintptr_t>(s) & 15) == 0)
    softmax_reg<<<static_cast<unsigned>(rows), kThreads, 0, st>>>(s, L, ld, scale, round);
  else
    softmax_long<<<static_cast<unsigned>(rows), kThreads, 0, st>>>(s, L, ld, scale, round);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

}  // namespace vae
