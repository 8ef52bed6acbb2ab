// splitk.cu -- the reduce step of split-K convolutions: sum the per-split
// partial accumulators in a fixed order (deterministic), then the epilogue
// (bias, residual, TF32 rounding), optionally emitting the GroupNorm
// statistics of the stored output for the next layer (cortiq-engine "Module
// vae", GroupNorm: per (sample, group) mean and biased variance; here as
// (count, mean, M2) partials per CTA, merged later with the parallel-variance
// combination).
#include "common.cuh"
#include "ptx.cuh"

namespace vae {

namespace {

constexpr int kThreads = 256;
constexpr long long kMaxReduceBlocks = 1024;  // callers size partial slots for this many CTAs

__device__ __forceinline__ void chan_merge(float &n, float &mean, float &m2, float nb, float mb,
                                           float m2b) {
  if (nb == 0.f) return;
  if (n == 0.f) {
    n = nb;
    mean = mb;
    m2 = m2b;
    return;
  }
  const float tot = n + nb;
  const float w = __fdividef(nb, tot);
  const float d = mb - mean;
  mean = fmaf(d, w, mean);
  m2 = m2 + m2b + d * d * n * w;
  n = tot;
}

// grid (blocks, samples). Each thread keeps one 4-channel quad (the float4
// stride blocks * 256 is a multiple of cout / 4).
__global__ void __launch_bounds__(kThreads)
    splitk_reduce_kernel(const float4 *__restrict__ part, int splits, long long stride4,
                         unsigned per4, int cout, const float *__restrict__ bias, float alpha,
                         const float4 *__restrict__ res, int round, float4 *__restrict__ out,
                         float *__restrict__ stat_part, int groups) {
  __shared__ float sm[kThreads * 4 * 3];
  const size_t base = static_cast<size_t>(blockIdx.y) * per4;
  const unsigned i0 = blockIdx.x * kThreads + threadIdx.x;
  const unsigned stride = gridDim.x * kThreads;
  const int quads = cout / 4;
  const int col = static_cast<int>(i0 % static_cast<unsigned>(quads)) * 4;
  float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (bias) bv = *reinterpret_cast<const float4 *>(bias + col);
  float k[4] = {0, 0, 0, 0}, s[4] = {0, 0, 0, 0}, ss[4] = {0, 0, 0, 0};
  int cnt = 0;
  for (unsigned i = i0; i < per4; i += stride) {
    const size_t g = base + i;
    float4 a = part[g];
    for (int sp = 1; sp < splits; ++sp) {
      const float4 b = part[g + sp * stride4];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    a.x = fmaf(a.x, alpha, bv.x);
    a.y = fmaf(a.y, alpha, bv.y);
    a.z = fmaf(a.z, alpha, bv.z);
    a.w = fmaf(a.w, alpha, bv.w);
    if (res) {
      const float4 r = res[g];
      a.x += r.x;
      a.y += r.y;
      a.z += r.z;
      a.w += r.w;
    }
    if (round) {
      a.x = round_tf32(a.x);
      a.y = round_tf32(a.y);
      a.z = round_tf32(a.z);
      a.w = round_tf32(a.w);
    }
    out[g] = a;
    if (stat_part) {
      const float v[4] = {a.x, a.y, a.z, a.w};
      if (cnt == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = v[j];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float d = v[j] - k[j];
        s[j] += d;
        ss[j] = fmaf(d, d, ss[j]);
      }
      ++cnt;
    }
  }
  if (!stat_part) return;
  // per-thread, per-channel (count, mean, M2), then one merge per group
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float md = cnt ? s[j] / cnt : 0.f;
    float *e = sm + (threadIdx.x * 4 + j) * 3;
    e[0] = static_cast<float>(cnt);
    e[1] = k[j] + md;
    e[2] = cnt ? fmaxf(ss[j] - s[j] * md, 0.f) : 0.f;
  }
  __syncthreads();
  const int cg = cout / groups;
  const int q_off = static_cast<int>((blockIdx.x * static_cast<unsigned>(kThreads)) % quads);
  for (int gi = threadIdx.x; gi < groups; gi += kThreads) {
    float n = 0.f, mean = 0.f, m2 = 0.f;
    // only the threads holding this group's channel quads contribute
    const int q_first = (gi * cg) / 4, q_last = ((gi + 1) * cg - 1) / 4;
    for (int qd = q_first; qd <= q_last; ++qd) {
      for (int t = (qd - q_off + quads) % quads; t < kThreads; t += quads) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if ((qd * 4 + j) / cg != gi) continue;
          const float *e = sm + (t * 4 + j) * 3;
          chan_merge(n, mean, m2, e[0], e[1], e[2]);
        }
      }
    }
    float *o = stat_part + ((static_cast<size_t>(blockIdx.y) * groups + gi) * gridDim.x +
                            blockIdx.x) * 3;
    o[0] = n;
    o[1] = mean;
    o[2] = m2;
  }
}

}  // namespace

int splitk_reduce(const float *part, int splits, long long split_stride, int samples,
                  long long rows_per_sample, int cout, const float *bias, float alpha,
                  const float *residual, int round, float *out, float *stat_part,
                  int stat_groups, long long *stat_slots, cudaStream_t s) {
  if (cout % 4 || splits < 1 || samples < 1) return VAE_EINVAL;
  const long long per4 = rows_per_sample * cout / 4;
  if (per4 > 0x7fffffffll) return VAE_EUNSUPPORTED;
  const int quads = cout / 4;
  // blocks per sample: a multiple of quads / gcd(quads, 256) so that every
  // thread keeps one channel quad
  long long gcd = quads, b = kThreads;
  while (b) {
    const long long t = gcd % b;
    gcd = b;
    b = t;
  }
  const long long unit = quads / gcd;
  long long blocks = std::min<long long>((per4 + kThreads - 1) / kThreads,
                                         std::max(1ll, 4ll * num_sms() / samples));
  blocks = std::min<long long>(blocks, kMaxReduceBlocks);
  blocks = std::max(unit, blocks / unit * unit);
  const bool stats = stat_part && stat_groups > 0 && cout % stat_groups == 0;
  splitk_reduce_kernel<<<dim3(static_cast<unsigned>(blocks), samples), kThreads, 0, s>>>(
      reinterpret_cast<const float4 *>(part), splits, split_stride / 4,
      static_cast<unsigned>(per4), cout, bias, alpha, reinterpret_cast<const float4 *>(residual),
      round, reinterpret_cast<float4 *>(out), stats ? stat_part : nullptr, stat_groups);
  VAE_LAUNCH_CHECK();
  count_launches(1);
  if (stat_slots) *stat_slots = stats ? blocks : 0;
  return VAE_OK;
}

}  // namespace vae
