// flash.cu -- fused single-head attention on the tcgen05 tensor cores:
//   O = softmax(Q K^T * scale) V
// (cortiq-engine "Module vae", VaeAttnRef: "softmax(q k^T / sqrt(c)) v"; the
// row softmax subtracts the row maximum as vae3d.rs fn softmax_inplace does).
// The score matrix is never stored: each CTA owns 128 query rows and streams
// 128-key blocks, keeping the running row maximum m and sum l (online
// softmax) and the output accumulator in TMEM.
//
// CTA (192 threads): warp 0 issues TMA loads, warp 1 allocates TMEM and issues
// the MMAs, warps 2-5 (one query row per thread) run the softmax and the
// epilogue. Per key block j:
//   S_j = Q K_j^T          (M=128, N=128, K=d; Q and K streamed in 32-channel
//                           chunks; S double-buffered in TMEM)
//   P_j = exp(S_j - m)     (softmax warps: TF32-rounded into shared memory in
//                           the 128-byte-swizzled K-major layout)
//   O  += P_j V_j          (M=128, N=DH, K=128 keys; B = V^T key chunks)
// The maximum is updated lazily: O and l are rescaled only when a block's
// maximum exceeds the one in use by more than 8 (so exp never exceeds e^8),
// which keeps exact results while skipping most rescales.
// TMEM holds S (2 x 128 columns) and O (DH <= 256 columns); a head wider than
// 256 runs as several output slices (grid.y), each recomputing S.
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace vae {

namespace {

constexpr int kQ = 128, kBK = 128;
constexpr int kStages = 4;
constexpr uint32_t kStageBytes = 32768;
constexpr uint32_t kPBytes = 4 * 16384;  // 128 rows x 128 keys as four 32-key chunks
constexpr int kFThreads = 192;
constexpr size_t kFlashSmem = 1024 + kStages * kStageBytes + kPBytes + 16 * sizeof(uint64_t) + 16;
constexpr float kLazy = 8.0f;  // rescale threshold on the running maximum

struct FParams {
  int L;         // tokens (queries = keys)
  int d_chunks;  // head dim / 32
  int nblk;      // key blocks
  float scale;   // 1 / sqrt(head dim)
  float *out;    // [L][ldo]
  int ldo;
  int *err;
};

__device__ __forceinline__ bool all_ok(bool ok) { return __all_sync(0xffffffffu, ok); }

__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
  return true;
}

template <int DH>
__global__ void __launch_bounds__(kFThreads, 1)
    flash_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const FParams p) {
  constexpr uint32_t IDESC_S = idesc_tf32(kQ, kBK);
  constexpr uint32_t IDESC_O = idesc_tf32(kQ, DH);
  constexpr uint32_t V_BYTES = DH * 128;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *stg = smem;                        // kStages x 32 KB operand stages
  float *pbuf = reinterpret_cast<float *>(smem + kStages * kStageBytes);  // P tile
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes + kPBytes);
  uint64_t *empty = full + kStages;
  uint64_t *s_full = empty + kStages;   // [2]
  uint64_t *s_empty = s_full + 2;       // [2]
  uint64_t *p_full = s_empty + 2;
  uint64_t *pv_done = p_full + 1;
  uint64_t *drain = pv_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile uint32_t *abort = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * kQ;
  const int d_off = blockIdx.y * DH;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], 4);
    }
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
    *abort = 0u;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t o_col = 2 * kBK;  // O after the two S buffers

  auto fail = [&]() {
    *abort = 1u;
    atomicCAS(p.err, 0, static_cast<int>(VAE_EDEVICE_TIMEOUT));
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, pending = 0, pend_par = 0;
      bool ok = true;
      auto next = [&]() {
        pending |= 1u << stage;
        pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      };
      auto load_s = [&](int j) {
        for (int kc = 0; kc < p.d_chunks && ok; ++kc) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort)) {
            fail();
            ok = false;
            return;
          }
          uint8_t *dst = stg + stage * kStageBytes;
          mbar_arrive_expect_tx(&full[stage], 32768);
          tma_load_2d(dst, &tmQ, &full[stage], kc * 32, q0);
          tma_load_2d(dst + 16384, &tmK, &full[stage], kc * 32, j * kBK);
          next();
        }
      };
      auto load_v = [&](int j) {
        for (int kk = 0; kk < kBK / 32 && ok; ++kk) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort)) {
            fail();
            ok = false;
            return;
          }
          uint8_t *dst = stg + stage * kStageBytes;
          mbar_arrive_expect_tx(&full[stage], V_BYTES);
          tma_load_2d(dst, &tmV, &full[stage], j * kBK + kk * 32, d_off);
          next();
        }
      };
      load_s(0);
      for (int t = 1; t <= p.nblk && ok; ++t) {
        if (t < p.nblk) load_s(t);
        load_v(t - 1);
      }
      if (*abort)
        for (int s = 0; s < kStages; ++s)
          if (pending & (1u << s)) drain_wait(&full[s], (pend_par >> s) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true, issued = false;
      auto advance = [&]() {
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      };
      auto mma_s = [&](int j) {
        const int buf = j & 1;
        if (!mbar_wait(&s_empty[buf], ((j >> 1) & 1) ^ 1u, abort)) {
          fail();
          ok = false;
          return;
        }
        tc_fence_after();
        for (int kc = 0; kc < p.d_chunks; ++kc) {
          if (!mbar_wait(&full[stage], phase, abort)) {
            fail();
            ok = false;
            return;
          }
          tc_fence_after();
          const uint8_t *src = stg + stage * kStageBytes;
          const uint64_t ad = sw128_kmajor_desc(smem_u32(src));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(src + 16384));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_tf32(tmem + buf * kBK, ad + 2 * k, bd + 2 * k, IDESC_S, (kc | k) != 0);
          issued = true;
          umma_commit(&empty[stage]);
          advance();
        }
        umma_commit(&s_full[buf]);
      };
      auto mma_pv = [&](int j) {
        if (!mbar_wait(p_full, j & 1, abort)) {
          fail();
          ok = false;
          return;
        }
        tc_fence_after();
        for (int kk = 0; kk < kBK / 32; ++kk) {
          if (!mbar_wait(&full[stage], phase, abort)) {
            fail();
            ok = false;
            return;
          }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(smem_u32(pbuf) + kk * 16384);
          const uint64_t bd = sw128_kmajor_desc(smem_u32(stg + stage * kStageBytes));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_tf32(tmem + o_col, ad + 2 * k, bd + 2 * k, IDESC_O, (j | kk | k) != 0);
          issued = true;
          umma_commit(&empty[stage]);
          advance();
        }
        umma_commit(pv_done);
      };
      mma_s(0);
      for (int t = 1; t <= p.nblk && ok; ++t) {
        if (t < p.nblk) mma_s(t);
        if (ok) mma_pv(t - 1);
      }
      if (*abort && issued) {
        umma_commit(drain);
        drain_wait(drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;  // query row of this thread
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < p.nblk && ok; ++j) {
      const int buf = j & 1;
      if (!all_ok(mbar_wait(&s_full[buf], (j >> 1) & 1, abort))) {
        if (lane == 0) fail();
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kBK];
#pragma unroll
      for (int c = 0; c < kBK / 32; ++c) tmem_ld_32cols(tmem + lane_base + buf * kBK + c * 32, s + c * 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[buf]);
      // scale, mask keys beyond L, block maximum
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kBK; ++i) {
        const bool key_ok = j * kBK + i < p.L;
        s[i] = key_ok ? s[i] * p.scale : -INFINITY;
        mx = fmaxf(mx, s[i]);
      }
      float alpha = 1.f, m_use = m;
      if (m == -INFINITY) {
        m_use = mx;
      } else if (mx > m + kLazy) {
        m_use = mx;
        alpha = __expf(m - mx);
      }
      // P_{j-1} consumed and O holds every earlier block before we touch either.
      if (j > 0) {
        if (!all_ok(mbar_wait(pv_done, (j - 1) & 1, abort))) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < DH / 32; ++c) {
            float o[32];
            const uint32_t ta = tmem + lane_base + o_col + c * 32;
            tmem_ld_32cols(ta, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st_32cols(ta, o);
          }
        }
      }
      float sum = 0.f;
#pragma unroll
      for (int kk = 0; kk < kBK / 32; ++kk) {
        float *tile = pbuf + kk * 4096;  // 128 rows x 32 keys, 128-byte swizzle
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          float4 v;
          v.x = round_tf32(__expf(s[kk * 32 + 4 * jj] - m_use));
          v.y = round_tf32(__expf(s[kk * 32 + 4 * jj + 1] - m_use));
          v.z = round_tf32(__expf(s[kk * 32 + 4 * jj + 2] - m_use));
          v.w = round_tf32(__expf(s[kk * 32 + 4 * jj + 3] - m_use));
          sum += (v.x + v.y) + (v.z + v.w);
          *reinterpret_cast<float4 *>(tile + r * 32 + ((jj ^ (r & 7)) * 4)) = v;
        }
      }
      l = l * alpha + sum;
      m = m_use;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && all_ok(mbar_wait(pv_done, (p.nblk - 1) & 1, abort))) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      const int row = q0 + r;
#pragma unroll 1
      for (int c = 0; c < DH / 32; ++c) {
        float o[32];
        tmem_ld_32cols(tmem + lane_base + o_col + c * 32, o);
        if (row < p.L) {
          float *dst = p.out + static_cast<long long>(row) * p.ldo + d_off + c * 32;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4 *>(dst + i) =
                make_float4(round_tf32(o[i] * inv), round_tf32(o[i + 1] * inv),
                            round_tf32(o[i + 2] * inv), round_tf32(o[i + 3] * inv));
        }
      }
    } else if (ok && lane == 0) {
      fail();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DH>
int launch_flash(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                 const FParams &fp, int qtiles, int slices, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(flash_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kFlashSmem));
  });
  if (attr != cudaSuccess) return VAE_ECUDA;
  flash_kernel<DH><<<dim3(qtiles, slices), kFThreads, kFlashSmem, s>>>(tq, tk, tv, fp);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

}  // namespace

bool flash_supported(int d) { return d % 32 == 0 && (d <= 256 || d % 256 == 0) && d <= 1024; }

// q, k: token-major [L][ld] (TF32-rounded); vt: [d][ldv] (keys along rows,
// ldv >= L, zero beyond L); out: [L][ldo] (TF32-rounded on store).
int flash_attention(const float *q, const float *k, int ld, const float *vt, int ldv, int L, int d,
                    float scale, float *out, int ldo, cudaStream_t s) {
  if (!q || !k || !vt || !out || L <= 0 || !flash_supported(d) || ld % 4 || ldv % 4 || ldo % 4)
    return VAE_EINVAL;
  const int dh = d <= 256 ? d : 256;
  FParams fp{};
  fp.L = L;
  fp.d_chunks = d / 32;
  fp.nblk = ceil_div(L, kBK);
  fp.scale = scale;
  fp.out = out;
  fp.ldo = ldo;
  fp.err = device_error_word();
  if (!fp.err) return VAE_ECUDA;
  CUtensorMap tq{}, tk{}, tv{};
  const uint64_t qdims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(L)};
  const uint64_t qstr[1] = {static_cast<uint64_t>(ld) * 4};
  const uint32_t qbox[2] = {32, static_cast<uint32_t>(kQ)};
  VAE_TRY(encode_tiled(&tq, q, 2, qdims, qstr, qbox));
  VAE_TRY(encode_tiled(&tk, k, 2, qdims, qstr, qbox));
  const uint64_t vdims[2] = {static_cast<uint64_t>(ldv), static_cast<uint64_t>(d)};
  const uint64_t vstr[1] = {static_cast<uint64_t>(ldv) * 4};
  const uint32_t vbox[2] = {32, static_cast<uint32_t>(dh)};
  VAE_TRY(encode_tiled(&tv, vt, 2, vdims, vstr, vbox));
  const int qtiles = ceil_div(L, kQ), slices = d / dh;
  switch (dh) {
    case 32: return launch_flash<32>(tq, tk, tv, fp, qtiles, slices, s);
    case 64: return launch_flash<64>(tq, tk, tv, fp, qtiles, slices, s);
    case 96: return launch_flash<96>(tq, tk, tv, fp, qtiles, slices, s);
    case 128: return launch_flash<128>(tq, tk, tv, fp, qtiles, slices, s);
    case 160: return launch_flash<160>(tq, tk, tv, fp, qtiles, slices, s);
    case 192: return launch_flash<192>(tq, tk, tv, fp, qtiles, slices, s);
    case 224: return launch_flash<224>(tq, tk, tv, fp, qtiles, slices, s);
    default: return launch_flash<256>(tq, tk, tv, fp, qtiles, slices, s);
  }
}

}  // namespace vae
