// peak.cu -- measured TF32 tensor-pipe rate of this GPU, the denominator the
// convolution's roofline fraction is reported against.
//
// Every SM runs one CTA whose elected thread issues back-to-back
// tcgen05.mma.cta_group::1.kind::tf32 instructions (M = 128, N = 256, K = 8,
// the conv's pixel-major tile shape) on operands that stay resident in shared
// memory, accumulating into TMEM. Nothing touches global memory inside the
// loop, so the time is the tensor pipe's alone (at whatever clock the GPU
// runs during the measurement).
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace vae {
namespace {

constexpr int kPThreads = 128;
constexpr uint32_t kPA = 128 * 128;  // A: 128 rows x 32 f32 (one K=32 chunk)
constexpr uint32_t kPB = 256 * 128;  // B: 256 rows x 32 f32
// Requested beyond what two CTAs could share, so each SM holds exactly one.
constexpr size_t kPSmem = 120 * 1024;
static_assert(1024 + kPA + kPB + 64 <= kPSmem, "operands and barrier fit");

__global__ void __launch_bounds__(kPThreads, 1) tf32_mma_loop(int iters, int *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float *ab = reinterpret_cast<float *>(smem);
  uint64_t *done = reinterpret_cast<uint64_t *>(smem + kPA + kPB);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile uint32_t *abort = tmem_slot + 1;
  // Exact small operands (sums stay exact in FP32): 0.5 and 0.25.
  for (uint32_t i = threadIdx.x; i < (kPA + kPB) / 4; i += kPThreads)
    ab[i] = i < kPA / 4 ? 0.5f : 0.25f;
  fence_proxy_async_smem();  // generic writes -> the tensor core's reads
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    *abort = 0u;
    fence_mbarrier_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = idesc_tf32(128, 256);
    const uint64_t ad = sw128_kmajor_desc(smem_u32(smem));
    const uint64_t bd = sw128_kmajor_desc(smem_u32(smem + kPA));
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int k = 0; k < 4; ++k) umma_tf32(tmem, ad + 2 * k, bd + 2 * k, idesc, (it | k) != 0);
    }
    umma_commit(done);
    if (!mbar_wait(done, 0, abort)) atomicCAS(err, 0, static_cast<int>(VAE_EDEVICE_TIMEOUT));
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace
}  // namespace vae

extern "C" int vae_measure_tf32_mma(int iters, double *flops, float *ms, vae_stream_t stream) {
  using namespace vae;
  if (iters <= 0 || !flops || !ms) return VAE_EINVAL;
  auto s = reinterpret_cast<cudaStream_t>(stream);
  int *err = device_error_word();
  if (!err) return VAE_ECUDA;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(tf32_mma_loop, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kPSmem));
  });
  if (attr != cudaSuccess) return VAE_ECUDA;
  const int sms = num_sms();
  cudaEvent_t e0, e1;
  VAE_CUDA_TRY(cudaEventCreate(&e0));
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return VAE_ECUDA;
  }
  int rc = VAE_OK;
  if (cudaEventRecord(e0, s) != cudaSuccess) rc = VAE_ECUDA;
  if (rc == VAE_OK) {
    tf32_mma_loop<<<sms, kPThreads, kPSmem, s>>>(iters, err);
    if (cudaGetLastError() != cudaSuccess) rc = VAE_ECUDA;
    else count_launches(1);
  }
  if (rc == VAE_OK && (cudaEventRecord(e1, s) != cudaSuccess ||
                       cudaEventSynchronize(e1) != cudaSuccess ||
                       cudaEventElapsedTime(ms, e0, e1) != cudaSuccess))
    rc = VAE_ECUDA;
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  *flops = static_cast<double>(sms) * iters * 4 * 2.0 * 128 * 256 * 8;
  return rc;
}
