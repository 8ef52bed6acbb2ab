// noalloc.cu -- GroupNorm(+SiLU) for callers that may not allocate device
// memory at all, not even a workspace buffer of their own.
//
// Such callers are typically plug-ins living inside a host application that
// owns the whole device-memory budget and forbids libraries to allocate, or
// latency-critical loops that cannot accept the latency (and possible
// implicit device synchronisation) of a cudaMalloc. They still pass their own
// input and output tensors; the statistics scratch that vae_groupnorm_silu
// takes from the caller's workspace comes here from one fixed array compiled
// into the library.
//
// The array lives in device global memory of every GPU that loads the
// library, for the life of the process. Host code must not hand the array's
// name to a kernel (on the host side it is only a stand-in symbol); its device
// address is fetched with cudaGetSymbolAddress, with that device current, on
// the first call made on that device, and again after the device's context
// was replaced (cudaDeviceReset gives the array a new address).
#include <mutex>

#include "common.cuh"

namespace vae {
namespace {

// Fixed scratch: per-(sample, group, block) partial statistics plus the
// per-channel scale/shift. 4 MiB holds up to 10 samples at 32 groups (any
// channel count the GroupNorm kernels accept).
constexpr size_t kNoAllocScratchBytes = 4u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};
void *g_noalloc_ctx[kMaxDevices] = {};  // context the cached address belongs to

int noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VAE_ECUDA;
  void *ctx = current_context();
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev] || g_noalloc_ctx[dev] != ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return VAE_ECUDA;
    g_noalloc_addr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *out = g_noalloc_addr[dev];
  return VAE_OK;
}

}  // namespace
}  // namespace vae

extern "C" int vae_groupnorm_silu_noalloc(const float *x, int n, int c, long long spatial,
                                          int layout, int groups, float eps, const float *gamma,
                                          const float *beta, int apply_silu, float *y,
                                          vae_stream_t stream) {
  using namespace vae;
  if (layout != VAE_NCHW && layout != VAE_NHWC) return VAE_EINVAL;
  if (!x || !y || !gamma || !beta || n <= 0 || c <= 0 || spatial <= 0 || groups <= 0)
    return VAE_EINVAL;
  if (c % groups || c % 4 || c > 1024) return VAE_EUNSUPPORTED;
  // Reject before touching the device when the fixed scratch is too small.
  if (groupnorm_ws_bytes(n, c, spatial, groups) > kNoAllocScratchBytes) return VAE_EUNSUPPORTED;
  void *ws = nullptr;
  VAE_TRY(noalloc_scratch(&ws));
  // Nothing in the scratch needs clearing: the statistics kernel writes every
  // partial before the finalize kernel reads it, and the finalize kernel
  // writes every scale/shift before the apply kernel reads it.
  return groupnorm_silu(x, n, c, spatial, layout == VAE_NHWC, groups, eps, gamma, beta,
                        apply_silu != 0, 0, y, ws, reinterpret_cast<cudaStream_t>(stream));
}
