// runtime.cu -- per-device runtime state shared by every entry point: the
// device error word kernels report into, the SM count persistent grids are
// sized from, and TMA tensor-map encoding through the driver entry point.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace vae {

namespace {
__device__ int g_vae_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_err_addr[kMaxDevices] = {};
void *g_err_ctx[kMaxDevices] = {};  // context the cached address belongs to
int g_sms[kMaxDevices] = {};
std::atomic<long long> g_launches{0};
// Test hooks (see vae_debug_*): device-wait limit, injected faults, and a
// countdown to an allocation failure inside vae_chain_prepare.
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_inject{0};
std::atomic<int> g_alloc_countdown{0};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}
}  // namespace

bool cuda_failed(cudaError_t e, const char *file, int line) {
  if (e == cudaSuccess) return false;
  static const bool verbose = [] {
    const char *v = std::getenv("VAE_VERBOSE");
    return v && v[0] == '1';
  }();
  if (verbose) std::fprintf(stderr, "vae: %s at %s:%d\n", cudaGetErrorString(e), file, line);
  return true;
}

void *current_context() {
  CUcontext ctx = nullptr;
  auto fn = ctx_get_current_fn();
  if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

int *device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void *ctx = current_context();
  std::lock_guard<std::mutex> lk(g_mu);
  // Re-resolved when the context changed (e.g. after cudaDeviceReset, the
  // symbol lives at a new address; before the first runtime call no context
  // is current yet and the lookup creates it).
  if (!g_err_addr[dev] || g_err_ctx[dev] != ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_vae_error_word) != cudaSuccess) return nullptr;
    g_err_addr[dev] = static_cast<int *>(p);
    g_err_ctx[dev] = ctx;
  }
  return g_err_addr[dev];
}

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int injected_faults() { return g_inject.load(std::memory_order_relaxed); }

bool take_alloc_failure() {
  int v = g_alloc_countdown.load();
  while (v > 0) {
    if (g_alloc_countdown.compare_exchange_weak(v, v - 1)) return v == 1;
  }
  return false;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 1;
    g_sms[dev] = v;
  }
  return g_sms[dev];
}

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
long long launch_count() { return g_launches.load(std::memory_order_relaxed); }

int encode_tiled(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return VAE_ECUDA;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, static_cast<cuuint32_t>(rank),
         const_cast<void *>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VAE_OK : VAE_EUNSUPPORTED;
}

}  // namespace vae

extern "C" {

const char *vae_status_string(int status) {
  switch (status) {
    case VAE_OK: return "ok";
    case VAE_EINVAL: return "invalid argument";
    case VAE_EUNSUPPORTED: return "unsupported shape";
    case VAE_EWORKSPACE: return "workspace too small";
    case VAE_ECUDA: return "CUDA call or launch failed";
    case VAE_ENOTPREPARED: return "chain handle not prepared";
    case VAE_EDEVICE_TIMEOUT: return "a device-side wait timed out";
    case VAE_ENOMEM: return "out of device memory";
    default: return "unknown status";
  }
}

int vae_device_error(vae_stream_t stream, int *code) {
  if (!code) return VAE_EINVAL;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VAE_ECUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, vae::g_vae_error_word, sizeof(int)) != cudaSuccess)
    return VAE_ECUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(vae::g_vae_error_word, &zero, sizeof(int)) != cudaSuccess)
    return VAE_ECUDA;
  *code = v;
  return VAE_OK;
}

int vae_num_sms(void) { return vae::num_sms(); }

int vae_debug_set_wait_limit(unsigned long long ns) {
  vae::g_wait_ns.store(ns ? ns : vae::kDefaultWaitNs);
  return VAE_OK;
}

int vae_debug_inject(int bits) {
  if (bits & ~VAE_INJECT_WITHHOLD_STREAMK_FLAG) return VAE_EINVAL;
  vae::g_inject.store(bits);
  return VAE_OK;
}

int vae_debug_fail_allocation(int nth) {
  if (nth < 0) return VAE_EINVAL;
  vae::g_alloc_countdown.store(nth);
  return VAE_OK;
}

long long vae_kernel_launch_count(void) { return vae::launch_count(); }

}  // extern "C"
