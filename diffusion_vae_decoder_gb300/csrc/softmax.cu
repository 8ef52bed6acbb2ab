// softmax.cu -- row softmax of the mid-block attention scores.
//
// cortiq-engine "Module vae", struct VaeAttnRef: softmax(q k^T / sqrt(c));
// the row softmax subtracts the row maximum, exponentiates and divides by the
// sum (vae3d.rs fn softmax_inplace). Rows are written back in place, rounded
// to TF32 because they are the A operand of the P.V tensor-core product; the
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

// Row length L <= kThreads * kPerThread: the row lives in registers.
__global__ void __launch_bounds__(kThreads) softmax_reg(float *s, int L, int ld, float scale) {
  __shared__ float sh[32];
  float *row = s + static_cast<long long>(blockIdx.x) * ld;
  float v[kPerThread];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    const int j = threadIdx.x + i * kThreads;
    v[i] = j < L ? row[j] * scale : -INFINITY;
    mx = fmaxf(mx, v[i]);
  }
  mx = block_reduce(mx, true, sh);
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    v[i] = expf(v[i] - mx);  // exp(-inf) = 0 for the padding slots
    sum += v[i];
  }
  sum = block_reduce(sum, false, sh);
  const float inv = 1.0f / sum;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    const int j = threadIdx.x + i * kThreads;
    if (j < L)
      row[j] = round_tf32(v[i] * inv);
    else if (j < ld)
      row[j] = 0.f;
  }
}

// Any row length: three sweeps over global memory.
__global__ void __launch_bounds__(kThreads) softmax_long(float *s, int L, int ld, float scale) {
  __shared__ float sh[32];
  float *row = s + static_cast<long long>(blockIdx.x) * ld;
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < L; j += kThreads) mx = fmaxf(mx, row[j] * scale);
  mx = block_reduce(mx, true, sh);
  float sum = 0.f;
  for (int j = threadIdx.x; j < L; j += kThreads) sum += expf(row[j] * scale - mx);
  sum = block_reduce(sum, false, sh);
  const float inv = 1.0f / sum;
  for (int j = threadIdx.x; j < L; j += kThreads)
    row[j] = round_tf32(expf(row[j] * scale - mx) * inv);
  for (int j = L + threadIdx.x; j < ld; j += kThreads) row[j] = 0.f;
}

}  // namespace

int softmax_rows(float *s, long long rows, int L, int ld, float scale, cudaStream_t st) {
  if (!s || rows <= 0 || L <= 0 || ld < L) return VAE_EINVAL;
  if (rows > 0x7fffffffll) return VAE_EUNSUPPORTED;
  if (ld <= kThreads * kPerThread)
    softmax_reg<<<static_cast<unsigned>(rows), kThreads, 0, st>>>(s, L, ld, scale);
  else
    softmax_long<<<static_cast<unsigned>(rows), kThreads, 0, st>>>(s, L, ld, scale);
  if (cudaGetLastError() != cudaSuccess) return VAE_ECUDA;
  count_launches(1);
  return VAE_OK;
}

}  // namespace vae
