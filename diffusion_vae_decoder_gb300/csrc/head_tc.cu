// head_tc.cu -- norm_out GroupNorm+SiLU and conv_out on the tensor cores
// (cortiq-engine "Module vae", VaeDecoder: "... -> GroupNorm + SiLU ->
// conv_out"; "VAE decode -> GPU handoff", "GPU plan", step 2: the conv as a
// GEMM on the tensor cores).
//
// conv_out maps C channels to a handful (CO) of output channels with a 3x3
// kernel. Written as a GEMM over the pixels of one input row,
//   Y[p][t*CO + o] = sum_c a[p][c] * w[o][c][t]        (t = ky*3 + kx)
// with a = tf32(silu(x * scale + shift)) (zero outside the image: the conv's
// padding applies after the normalisation), the conv is the sum of three
// rows' projections shifted by the tap offsets:
//   out[y][x][o] = bias[o] + sum_{ky,kx} Y_{y+ky-1}[x+kx-1][(ky*3+kx)*CO + o].
// One MMA of M = 128 pixels x N = NT (9*CO padded to a multiple of 16) x K = C
// per input row, so the MMA work per pixel is 2*NT*C FLOP (the direct conv's
// 2*9*CO*C, padded) and every input element is staged once.
//
// A CTA owns a strip of sw <= 126 output columns (its 128 MMA rows are input
// pixels x0-1 .. x0+126, of which the sw + 2 from x0-1 are normalised and
// read) and R output rows; it walks its R+2 input rows top to bottom. Warp roles (448 threads):
//   warp 0     TMA: the packed weights once, then per input row C/32 boxes of
//              128 pixels x 32 channels (128-byte swizzle) into a raw ring;
//   warp 1     TMEM allocation; one thread issues the MMAs of each row into a
//              ring of four TMEM row buffers (NT columns each);
//   warps 2-9  the GroupNorm affine + SiLU + TF32 rounding: each takes its
//              slots of a landed raw stage into registers and hands the stage
//              back to the TMA at once, then writes the results to an operand
//              stage (zero outside the image) for the MMA;
//   warps 10-13 the epilogue: output row r adds the projections of input rows
//              r, r+1, r+2 (one pixel per thread), exchanges the kx = 0 / 2
//              partial sums with the neighbouring pixels (warp shuffles; the
//              warp edges through shared memory), adds the bias and writes
//              the NCHW result; each row buffer is handed back to the MMA
//              once the last output row that reads it is done.
// Every wait is bounded: on a timeout the CTA records VAE_EDEVICE_TIMEOUT,
// waits (bounded) for its copies and MMAs in flight and returns.
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "silu.cuh"

namespace vae {

namespace {

constexpr int kHtRaw = 3;                    // 16 KB TMA stages (raw activation)
constexpr int kHtA = 2;                      // 16 KB MMA operand stages (normalised)
constexpr int kHtBufs = 4;                   // TMEM row buffers
constexpr int kHtXfWarps = 8;                // transform warps
constexpr int kHtThreads = 32 * (2 + kHtXfWarps + 4);  // 14 warps
constexpr int kHtStrip = 126;                // output columns per CTA
constexpr uint32_t kHtStageBytes = 16384;    // 128 pixels x 32 channels, either ring
constexpr uint32_t kHtMaxWeightBytes = 32768;  // C * NT * 4 resident in shared memory
constexpr int kHtMaxCo = 7;                  // NT = 16 * ceil(9 * CO / 16) <= 64

struct HtParams {
  int H, W, C, chunks;  // chunks = C / 32
  int R;                // output rows per CTA
  int sw;               // output columns per CTA (strip width, <= 126)
  const float *scale, *shift;  // [n][C]
  const float *bias;           // [CO] or null
  float *y;                    // NCHW [n][CO][H][W]
  int *err;
  uint64_t wait_ns;
};

__host__ __device__ constexpr int ht_nt(int co) { return (9 * co + 15) / 16 * 16; }
__host__ __device__ constexpr uint32_t ht_tmem_cols(int nt) {
  return kHtBufs * nt <= 64 ? 64u : kHtBufs * nt <= 128 ? 128u : 256u;
}

// Barrier `id` over `count` threads that also returns the AND of `v` over them.
__device__ __forceinline__ bool bar_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Bounded wait for a phase of `bar`, the warp parked in the barrier's
// try_wait (suspended until the phase completes, at most 20 us per try)
// rather than spinning: the waiting roles then take no issue slots from the
// transform warps. Gives up when `limit_ns` passes or another role raised
// `*abort`.
__device__ __forceinline__ bool ht_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *abort,
                                        uint64_t limit_ns) {
  auto try_wait = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
  };
  if (try_wait()) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (try_wait()) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ bool ht_drain(uint64_t *bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit) return false;
  return true;
}

template <int CO>
__global__ void __launch_bounds__(kHtThreads, 2)
    head_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const HtParams p) {
  constexpr int NT = ht_nt(CO);
  constexpr uint32_t TCOLS = ht_tmem_cols(NT);
  constexpr uint32_t IDESC = idesc_tf32(128, NT);
  constexpr uint32_t WCHUNK = NT * 128;  // bytes of one 32-channel weight chunk

  extern __shared__ uint8_t ht_smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(ht_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *raw = smem;                                  // kHtRaw x 16 KB
  uint8_t *opa = raw + kHtRaw * kHtStageBytes;          // kHtA x 16 KB
  uint8_t *wsm = opa + kHtA * kHtStageBytes;            // chunks x WCHUNK
  float *edge = reinterpret_cast<float *>(wsm + p.chunks * WCHUNK);  // [2][2][4][8]
  uint64_t *rfull = reinterpret_cast<uint64_t *>(edge + 2 * 2 * 4 * 8);
  uint64_t *rempty = rfull + kHtRaw;
  uint64_t *afull = rempty + kHtRaw;
  uint64_t *aempty = afull + kHtA;
  uint64_t *yfull = aempty + kHtA;
  uint64_t *yempty = yfull + kHtBufs;
  uint64_t *wfull = yempty + kHtBufs;
  uint64_t *drain = wfull + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile uint32_t *abort = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.z;
  const int x0 = blockIdx.x * p.sw;
  const int y0 = blockIdx.y * p.R;
  const int rows_out = min(p.R, p.H - y0);
  const int rows_in = rows_out + 2;  // input rows y0 - 1 .. y0 + rows_out

  if (threadIdx.x == 0) {
    for (int s = 0; s < kHtRaw; ++s) {
      mbar_init(&rfull[s], 1);
      mbar_init(&rempty[s], kHtXfWarps);  // one arrival per transform warp
    }
    for (int s = 0; s < kHtA; ++s) {
      mbar_init(&afull[s], kHtXfWarps);
      mbar_init(&aempty[s], 1);
    }
    for (int b = 0; b < kHtBufs; ++b) {
      mbar_init(&yfull[b], 1);
      mbar_init(&yempty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(wfull, 1);
    mbar_init(drain, 1);
    *abort = 0u;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    *abort = 1u;
    atomicCAS(p.err, 0, static_cast<int>(VAE_EDEVICE_TIMEOUT));
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(wfull, static_cast<uint32_t>(p.chunks) * WCHUNK);
      for (int k = 0; k < p.chunks; ++k) tma_load_2d(wsm + k * WCHUNK, &tmW, wfull, k * 32, 0);
      uint32_t stage = 0, phase = 0, pending = 0, pend_par = 0;
      bool ok = true;
      for (int i = 0; i < rows_in && ok; ++i) {
        const int iy = y0 - 1 + i;
        for (int k = 0; k < p.chunks; ++k) {
          if (!ht_wait(&rempty[stage], phase ^ 1u, abort, p.wait_ns)) {
            fail();
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&rfull[stage], kHtStageBytes);
          tma_load_4d(raw + stage * kHtStageBytes, &tmX, &rfull[stage], k * 32, x0 - 1, iy, n);
          pending |= 1u << stage;
          pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kHtRaw) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort) {  // copies still landing must not outlive the CTA
        ht_drain(wfull, 0, p.wait_ns);
        for (int s = 0; s < kHtRaw; ++s)
          if (pending & (1u << s)) ht_drain(&rfull[s], (pend_par >> s) & 1u, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = ht_wait(wfull, 0, abort, p.wait_ns);
      if (!ok) fail();
      bool issued = false;
      uint32_t stage = 0, phase = 0;
      for (int i = 0; i < rows_in && ok; ++i) {
        const int buf = i % kHtBufs;
        if (!ht_wait(&yempty[buf], ((i / kHtBufs) & 1) ^ 1u, abort, p.wait_ns)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * NT;
        for (int k = 0; k < p.chunks; ++k) {
          if (!ht_wait(&afull[stage], phase, abort, p.wait_ns)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(smem_u32(opa + stage * kHtStageBytes));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(wsm + k * WCHUNK));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) umma_tf32(d, ad + 2 * kk, bd + 2 * kk, IDESC, (k | kk) != 0);
          issued = true;
          umma_commit(&aempty[stage]);
          if (++stage == kHtA) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(&yfull[buf]);
      }
      if (*abort && issued) {  // MMAs in flight finish before TMEM is freed
        umma_commit(drain);
        ht_drain(drain, 0, p.wait_ns);
      }
    }
  } else if (warp < 2 + kHtXfWarps) {
    // ------------------------------------------------------------ transform
    // Thread t handles the 16-byte slot s = t & 7 of rows (t >> 3) + 32 j of
    // each stage; with the 128-byte swizzle that slot holds the channel quad
    // s ^ (row & 7), the same for all four of its rows.
    constexpr int kRowStep = kHtXfWarps * 4;  // rows between a thread's slots
    const int t = threadIdx.x - 64;
    const int s = t & 7, r0 = t >> 3;
    const int quad = s ^ (r0 & 7);
    const float *sc = p.scale + static_cast<size_t>(n) * p.C + quad * 4;
    const float *sh = p.shift + static_cast<size_t>(n) * p.C + quad * 4;
    uint32_t rs = 0, rph = 0, as = 0, aph = 0;
    bool ok = true;
    for (int i = 0; i < rows_in && ok; ++i) {
      const int iy = y0 - 1 + i;
      const bool row_in = iy >= 0 && iy < p.H;
      for (int k = 0; k < p.chunks; ++k) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(sc + k * 32));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(sh + k * 32));
        if (!__all_sync(0xffffffffu, ht_wait(&rfull[rs], rph, abort, p.wait_ns))) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        const float4 *src = reinterpret_cast<const float4 *>(raw + rs * kHtStageBytes);
        float4 v[128 / kRowStep];
#pragma unroll
        for (int j = 0; j < 128 / kRowStep; ++j) v[j] = src[(r0 + kRowStep * j) * 8 + s];
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[rs]);  // the raw stage is in registers
        if (++rs == kHtRaw) {
          rs = 0;
          rph ^= 1u;
        }
        float4 o[128 / kRowStep];
#pragma unroll
        for (int j = 0; j < 128 / kRowStep; ++j) {
          const int r = r0 + kRowStep * j;
          const int gx = x0 - 1 + r;
          o[j] = make_float4(0.f, 0.f, 0.f, 0.f);  // padding: zero after the norm
          if (r <= p.sw + 1 && row_in && gx >= 0 && gx < p.W) {
            const float2 s0 = silu2_tf32(v[j].x, v[j].y, a.x, a.y, b.x, b.y);
            const float2 s1 = silu2_tf32(v[j].z, v[j].w, a.z, a.w, b.z, b.w);
            o[j] = make_float4(s0.x, s0.y, s1.x, s1.y);
          }
        }
        if (!__all_sync(0xffffffffu, ht_wait(&aempty[as], aph ^ 1u, abort, p.wait_ns))) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        float4 *dst = reinterpret_cast<float4 *>(opa + as * kHtStageBytes);
#pragma unroll
        for (int j = 0; j < 128 / kRowStep; ++j)
          if (r0 + kRowStep * j <= p.sw + 1)  // rows beyond are read by no output
            dst[(r0 + kRowStep * j) * 8 + s] = o[j];
        fence_proxy_async_smem();  // generic writes visible to the MMA's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[as]);
        if (++as == kHtA) {
          as = 0;
          aph ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int l = q * 32 + lane;  // MMA row = input pixel x0 - 1 + l
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int gx = x0 - 1 + l;
    const bool px_out = l >= 1 && l <= p.sw && gx < p.W;
    float bias[CO];
#pragma unroll
    for (int o = 0; o < CO; ++o) bias[o] = p.bias ? __ldg(p.bias + o) : 0.f;
    for (int r = 0; r < rows_out; ++r) {
      // input rows r, r+1, r+2 of the CTA (the first two were waited for
      // by the previous output rows)
      bool good = true;
      for (int i = (r == 0 ? 0 : r + 2); i <= r + 2 && good; ++i)
        good = __all_sync(0xffffffffu,
                          ht_wait(&yfull[i % kHtBufs], (i / kHtBufs) & 1, abort, p.wait_ns));
      float z[3][CO];
#pragma unroll
      for (int kx = 0; kx < 3; ++kx)
#pragma unroll
        for (int o = 0; o < CO; ++o) z[kx][o] = 0.f;
      float *eg = edge + (r & 1) * 64;  // [0, 32): last lanes' z[0]; [32, 64): first lanes' z[2]
      if (good) {
        tc_fence_after();
        // input row r + ky contributes its columns ky*3*CO .. (ky+1)*3*CO - 1
        // (the taps of kernel row ky): only the 16-column windows holding them
        // are read
#pragma unroll
        for (int ky = 0; ky < 3; ++ky) {
          const int c0 = ky * 3 * CO, c1 = c0 + 3 * CO;
          const uint32_t ta = tmem + lane_base + ((r + ky) % kHtBufs) * NT;
#pragma unroll
          for (int w0 = 0; w0 < NT; w0 += 16) {
            if (w0 + 16 <= c0 || w0 >= c1) continue;
            float v[16];
            tmem_ld_16cols(ta + w0, v);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = w0 + jj;
              if (j >= c0 && j < c1) z[(j - c0) / CO][(j - c0) % CO] += v[jj];
            }
          }
        }
        // input row r is read for the last time: hand its buffer back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&yempty[r % kHtBufs]);
        if (lane == 31)
#pragma unroll
          for (int o = 0; o < CO; ++o) eg[q * 8 + o] = z[0][o];
        if (lane == 0)
#pragma unroll
          for (int o = 0; o < CO; ++o) eg[32 + q * 8 + o] = z[2][o];
      }
      // the four epilogue warps agree (and their edge values are visible)
      if (!bar_and(1, 128, good)) {
        if (lane == 0 && !good) fail();
        break;
      }
      // neighbours' partial sums: kx = 0 taps come from pixel l - 1, kx = 2
      // from pixel l + 1
      const int gy = y0 + r;
#pragma unroll
      for (int o = 0; o < CO; ++o) {
        float left = __shfl_up_sync(0xffffffffu, z[0][o], 1);
        float right = __shfl_down_sync(0xffffffffu, z[2][o], 1);
        if (lane == 0) left = q > 0 ? eg[(q - 1) * 8 + o] : 0.f;
        if (lane == 31) right = q < 3 ? eg[32 + (q + 1) * 8 + o] : 0.f;
        if (px_out)
          p.y[(static_cast<size_t>(n * CO + o) * p.H + gy) * p.W + gx] =
              bias[o] + ((left + z[1][o]) + right);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TCOLS);
  }
}

// w [cout][C][3][3] -> [NT][C]: row t * cout + o holds tap t of output o,
// TF32-rounded; rows 9 * cout .. NT - 1 zero.
__global__ void head_tc_pack_kernel(const float *__restrict__ w, int cout, int C, int nt,
                                    float *dst) {
  const int total = nt * C;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int j = i / C, c = i % C;
    const int t = j / cout, o = j % cout;
    dst[i] = j < 9 * cout ? round_tf32(w[(static_cast<size_t>(o) * C + c) * 9 + t]) : 0.f;
  }
}

// Dynamic shared memory for `weight_bytes` of resident packed weights.
size_t ht_smem_bytes(size_t weight_bytes) {
  return 1024 + (kHtRaw + kHtA) * kHtStageBytes + weight_bytes + 2 * 2 * 4 * 8 * sizeof(float) +
         (2 * kHtRaw + 2 * kHtA + 2 * kHtBufs + 2) * sizeof(uint64_t) + 16;
}

template <int CO>
int launch_head_tc(const CUtensorMap &tx, const CUtensorMap &tw, const HtParams &hp, dim3 grid,
                   size_t smem, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(head_tc_kernel<CO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(ht_smem_bytes(kHtMaxWeightBytes)));
  });
  if (attr != cudaSuccess) return VAE_ECUDA;
  head_tc_kernel<CO><<<grid, kHtThreads, smem, s>>>(tx, tw, hp);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

}  // namespace

bool head_tc_supported(int cin, int cout) {
  return cin > 0 && cin % 32 == 0 && cout >= 1 && cout <= kHtMaxCo &&
         static_cast<size_t>(cin) * ht_nt(cout) * 4 <= kHtMaxWeightBytes;
}

size_t head_tc_packed_floats(int cin, int cout) {
  return static_cast<size_t>(ht_nt(cout)) * cin;
}

int head_tc_pack_weights(const float *w, int cout, int cin, float *dst, cudaStream_t s) {
  if (!w || !dst) return VAE_EINVAL;
  if (!head_tc_supported(cin, cout)) return VAE_EUNSUPPORTED;
  const int total = ht_nt(cout) * cin;
  head_tc_pack_kernel<<<(total + 255) / 256, 256, 0, s>>>(w, cout, cin, ht_nt(cout), dst);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

int head_tc_gn_silu_conv(const float *x, int n, int h, int w, int c, const float *scale,
                         const float *shift, const float *wpk, const float *bias, int cout,
                         float *y, cudaStream_t s) {
  if (!x || !scale || !shift || !wpk || !y || n <= 0 || h <= 0 || w <= 0) return VAE_EINVAL;
  if (!head_tc_supported(c, cout) || n > 65535) return VAE_EUNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(wpk) |
       reinterpret_cast<uintptr_t>(scale) | reinterpret_cast<uintptr_t>(shift)) & 15)
    return VAE_EINVAL;
  const int nt = ht_nt(cout);
  HtParams hp{};
  hp.H = h;
  hp.W = w;
  hp.C = c;
  hp.chunks = c / 32;
  hp.scale = scale;
  hp.shift = shift;
  hp.bias = bias;
  hp.y = y;
  hp.err = device_error_word();
  if (!hp.err) return VAE_ECUDA;
  hp.wait_ns = wait_limit_ns();
  // Rows per CTA: as few as fill two CTAs per SM in one round.
  // Strips of equal width (at most 126 columns): the transform covers each
  // strip's columns and its two halo columns only.
  const long long strips = (w + kHtStrip - 1) / kHtStrip;
  hp.sw = static_cast<int>((w + strips - 1) / strips);
  const long long per = strips * n;
  const long long segs_max = std::max(1ll, 2ll * num_sms() / per);
  int R = static_cast<int>((h + segs_max - 1) / segs_max);
  R = std::max(R, 2);
  const long long segs = (h + R - 1) / R;
  if (strips > 0x7fffffffll || segs > 65535) return VAE_EUNSUPPORTED;
  hp.R = R;
  CUtensorMap tx{}, tw{};
  {
    const uint64_t dims[4] = {static_cast<uint64_t>(c), static_cast<uint64_t>(w),
                              static_cast<uint64_t>(h), static_cast<uint64_t>(n)};
    const uint64_t str[3] = {static_cast<uint64_t>(c) * 4, static_cast<uint64_t>(w) * c * 4,
                             static_cast<uint64_t>(h) * w * c * 4};
    const uint32_t box[4] = {32, 128, 1, 1};
    VAE_TRY(encode_tiled(&tx, x, 4, dims, str, box));
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(c), static_cast<uint64_t>(nt)};
    const uint64_t str[1] = {static_cast<uint64_t>(c) * 4};
    const uint32_t box[2] = {32, static_cast<uint32_t>(nt)};
    VAE_TRY(encode_tiled(&tw, wpk, 2, dims, str, box));
  }
  const dim3 grid(static_cast<unsigned>(strips), static_cast<unsigned>(segs), n);
  const size_t smem = ht_smem_bytes(static_cast<size_t>(c) * nt * 4);
  switch (cout) {
    case 1: return launch_head_tc<1>(tx, tw, hp, grid, smem, s);
    case 2: return launch_head_tc<2>(tx, tw, hp, grid, smem, s);
    case 3: return launch_head_tc<3>(tx, tw, hp, grid, smem, s);
    case 4: return launch_head_tc<4>(tx, tw, hp, grid, smem, s);
    case 5: return launch_head_tc<5>(tx, tw, hp, grid, smem, s);
    case 6: return launch_head_tc<6>(tx, tw, hp, grid, smem, s);
    default: return launch_head_tc<7>(tx, tw, hp, grid, smem, s);
  }
}

}  // namespace vae
