// groupnorm.cu -- two-pass GroupNorm (+ SiLU), HBM-bound.
//
// Definition: cortiq-engine "Module vae", structs GroupNorm / VaeNormRef
// (eps 1e-6, affine); statistics as vae3d.rs struct GroupNorm::apply computes
// them (mean, then the biased variance, 1/sqrt(var + eps), then gamma/beta);
// SiLU as vae3d.rs fn silu.
//
// Pass 1 (stats): many CTAs per sample each reduce a contiguous slab of
// pixels. Every thread owns a fixed float4 of channels and accumulates sums
// of (x - first value it saw), which keeps f32 cancellation small; the
// per-thread (count, mean, M2) triples are merged into per-(CTA, group)
// partials with the parallel-variance (Chan et al.) combination in f64.
// Finalize: one CTA per (sample, group) merges the partials and writes the
// per-channel affine  y = x * scale[c] + shift[c].
// Pass 2 (apply): one vectorised elementwise sweep, SiLU, optional TF32
// rounding when the result feeds a tensor-core conv.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "ptx.cuh"
#include "silu.cuh"

namespace vae {

namespace {

constexpr int kStatThreads = 256;
constexpr int kMaxBlocksPerGroupSeg = 512;  // partial slots per (sample, group)
constexpr int kFinalizeThreads = 512;       // threads merging one (sample, group)

// (count, mean, M2) of a set of values; merged with the parallel-variance
// combination, which works on deviations from the means (no cancellation of
// large raw sums). FP32 arithmetic: FP64 throughput on this part is low.
struct Triple {
  float n, mean, m2;
};

__device__ __forceinline__ Triple merge(Triple a, Triple b) {
  if (a.n == 0.f) return b;
  if (b.n == 0.f) return a;
  const float n = a.n + b.n;
  const float wb = __fdividef(b.n, n);
  const float d = b.mean - a.mean;
  return {n, fmaf(d, wb, a.mean), a.m2 + b.m2 + d * d * a.n * wb};
}

// NHWC: x[n][spatial][c]. Block `blk` of `nblk` of sample n reduces its slab
// of pixels into partials [n][groups][nblk] (count, mean, M2); sm holds
// 3 * kStatThreads * 4 floats.
template <class P>
__device__ __forceinline__ void stats_slab_nhwc(const float *__restrict__ x, int c,
                                                long long spatial, int groups, int nblk, int n,
                                                int blk, float *sm, P *__restrict__ part) {
  const int tpp = c >> 2;
  const int ppi = kStatThreads / tpp;
  const int tid = threadIdx.x;
  const int lc = tid % tpp, pl = tid / tpp;
  const long long p0 = spatial * blk / nblk, p1 = spatial * (blk + 1) / nblk;
  float k[4] = {0, 0, 0, 0}, s[4] = {0, 0, 0, 0}, ss[4] = {0, 0, 0, 0};
  int cnt = 0;
  if (pl < ppi) {
    const float *base = x + (static_cast<long long>(n) * spatial) * c + 4 * lc;
    long long pix = p0 + pl;
    if (pix < p1) {  // shift every sum by the first value this thread sees
      const float4 v = __ldg(reinterpret_cast<const float4 *>(base + pix * c));
      k[0] = v.x;
      k[1] = v.y;
      k[2] = v.z;
      k[3] = v.w;
    }
    // four independent loads in flight per iteration
    for (; pix + 3 * ppi < p1; pix += 4 * ppi) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[u] = __ldg(reinterpret_cast<const float4 *>(base + (pix + u * ppi) * c));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float a[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float d = a[j] - k[j];
          s[j] += d;
          ss[j] = fmaf(d, d, ss[j]);
        }
      }
      cnt += 4;
    }
    for (; pix < p1; pix += ppi) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(base + pix * c));
      const float a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float d = a[j] - k[j];
        s[j] += d;
        ss[j] = fmaf(d, d, ss[j]);
      }
      ++cnt;
    }
    float *e = sm + (static_cast<long long>(pl) * c + 4 * lc) * 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float mean_d = cnt ? s[j] / cnt : 0.f;
      e[3 * j + 0] = static_cast<float>(cnt);
      e[3 * j + 1] = k[j] + mean_d;
      e[3 * j + 2] = cnt ? fmaxf(ss[j] - s[j] * mean_d, 0.f) : 0.f;
    }
  }
  __syncthreads();
  const int cg = c / groups;
  for (int g = tid; g < groups; g += kStatThreads) {
    Triple acc{0.f, 0.f, 0.f};
    for (int l = 0; l < ppi; ++l)
      for (int ch = g * cg; ch < (g + 1) * cg; ++ch) {
        const float *e = sm + (static_cast<long long>(l) * c + ch) * 3;
        acc = merge(acc, Triple{e[0], e[1], e[2]});
      }
    P *o = part + ((static_cast<long long>(n) * groups + g) * nblk + blk) * 3;
    o[0] = acc.n;
    o[1] = acc.mean;
    o[2] = acc.m2;
  }
}

// grid = (nblk, n). Partials [n][groups][nblk].
__global__ void __launch_bounds__(kStatThreads)
    gn_stats_nhwc(const float *__restrict__ x, int c, long long spatial, int groups, int nblk,
                  double *__restrict__ part) {
  extern __shared__ float sm[];  // [ppi][c] x 3
  stats_slab_nhwc(x, c, spatial, groups, nblk, blockIdx.y, blockIdx.x, sm, part);
}

// NCHW: group (n, g) is the contiguous segment of cg * spatial floats.
// grid = (nblk, n * groups).
__global__ void __launch_bounds__(kStatThreads)
    gn_stats_nchw(const float *__restrict__ x, int c, long long spatial, int groups, int nblk,
                  double *__restrict__ part) {
  __shared__ float red[kStatThreads][3];
  const int ng = blockIdx.y, blk = blockIdx.x;
  const int cg = c / groups;
  const long long seg = static_cast<long long>(cg) * spatial;
  const float *base = x + static_cast<long long>(ng) * seg;
  const long long e0 = seg * blk / nblk, e1 = seg * (blk + 1) / nblk;
  float k = 0.f, s = 0.f, ss = 0.f;
  int cnt = 0;
  for (long long i = e0 + threadIdx.x; i < e1; i += kStatThreads) {
    const float v = __ldg(base + i);
    if (cnt == 0) k = v;
    const float d = v - k;
    s += d;
    ss = fmaf(d, d, ss);
    ++cnt;
  }
  const float md = cnt ? s / cnt : 0.f;
  red[threadIdx.x][0] = cnt;
  red[threadIdx.x][1] = k + md;
  red[threadIdx.x][2] = cnt ? fmaxf(ss - s * md, 0.f) : 0.f;
  __syncthreads();
  for (int w = kStatThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      const Triple a{red[threadIdx.x][0], red[threadIdx.x][1], red[threadIdx.x][2]};
      const Triple b{red[threadIdx.x + w][0], red[threadIdx.x + w][1], red[threadIdx.x + w][2]};
      const Triple r = merge(a, b);
      red[threadIdx.x][0] = r.n;
      red[threadIdx.x][1] = r.mean;
      red[threadIdx.x][2] = r.m2;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    double *o = part + (static_cast<long long>(ng) * nblk + blk) * 3;
    o[0] = red[0][0];
    o[1] = red[0][1];
    o[2] = red[0][2];
  }
}

// One CTA (a power-of-two blockDim <= kFinalizeThreads) for (sample, group)
// ng: merge its nblk partials, write scale/shift per channel.
template <class P>
__device__ __forceinline__ void finalize_group(const P *__restrict__ part, long long nblk, int c,
                                               int groups, float eps,
                                               const float *__restrict__ gamma,
                                               const float *__restrict__ beta,
                                               float *__restrict__ scale,
                                               float *__restrict__ shift, int ng,
                                               float (*red)[3]) {
  const int n = ng / groups, g = ng % groups;
  Triple acc{0.f, 0.f, 0.f};
  for (long long b = threadIdx.x; b < nblk; b += blockDim.x) {
    const P *e = part + (static_cast<long long>(ng) * nblk + b) * 3;
    acc = merge(acc, Triple{static_cast<float>(e[0]), static_cast<float>(e[1]),
                            static_cast<float>(e[2])});
  }
  red[threadIdx.x][0] = acc.n;
  red[threadIdx.x][1] = acc.mean;
  red[threadIdx.x][2] = acc.m2;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      const Triple a{red[threadIdx.x][0], red[threadIdx.x][1], red[threadIdx.x][2]};
      const Triple b{red[threadIdx.x + w][0], red[threadIdx.x + w][1], red[threadIdx.x + w][2]};
      const Triple r = merge(a, b);
      red[threadIdx.x][0] = r.n;
      red[threadIdx.x][1] = r.mean;
      red[threadIdx.x][2] = r.m2;
    }
    __syncthreads();
  }
  const int cg = c / groups;
  const double cntv = red[0][0];
  const double mean = red[0][1];
  const double var = cntv > 0 ? red[0][2] / cntv : 0.0;
  const double rstd = 1.0 / sqrt(var + static_cast<double>(eps));
  for (int j = threadIdx.x; j < cg; j += blockDim.x) {
    const int ch = g * cg + j;
    const double a = rstd * gamma[ch];
    scale[n * c + ch] = static_cast<float>(a);
    shift[n * c + ch] = static_cast<float>(beta[ch] - mean * a);
  }
}

template <class P>
__global__ void gn_finalize(const P *__restrict__ part, long long nblk, int c, int groups,
                            float eps, const float *__restrict__ gamma,
                            const float *__restrict__ beta, float *__restrict__ scale,
                            float *__restrict__ shift) {
  __shared__ float red[kFinalizeThreads][3];
  finalize_group(part, nblk, c, groups, eps, gamma, beta, scale, shift, blockIdx.x, red);
}

// SiLU with the fast exponential and division: their few-ulp error sits far
// below the TF32 rounding applied to the result before the next conv.
// (v < -88: exp overflows to inf and the quotient is -0, SiLU's limit.)
__device__ __forceinline__ float act(float v, int silu) {
  return silu ? __fdividef(v, 1.0f + __expf(-v)) : v;
}

__device__ __forceinline__ float rnd(float v, int round) { return round ? round_tf32(v) : v; }

// y = [silu](x * scale + shift) (+ res), optionally TF32-rounded. Grid
// (blocks, n): blockIdx.y is the sample; the float4 stride of the loop is a
// multiple of c/4, so every thread keeps the same four channels and loads
// their scale/shift once.
__global__ void __launch_bounds__(256)
    gn_apply_nhwc(const float *__restrict__ x, unsigned per_sample4, int c,
                  const float *__restrict__ scale, const float *__restrict__ shift, int silu,
                  int round, const float *__restrict__ res, float *__restrict__ y) {
  const int n = blockIdx.y;
  const size_t base4 = static_cast<size_t>(n) * per_sample4;
  const float4 *xv = reinterpret_cast<const float4 *>(x) + base4;
  float4 *yv = reinterpret_cast<float4 *>(y) + base4;
  const float4 *rv = res ? reinterpret_cast<const float4 *>(res) + base4 : nullptr;
  const unsigned i0 = blockIdx.x * 256u + threadIdx.x;
  const unsigned stride = gridDim.x * 256u;
  const int ch = static_cast<int>((i0 * 4u) % static_cast<unsigned>(c));
  const float4 a = *reinterpret_cast<const float4 *>(scale + n * c + ch);
  const float4 b = *reinterpret_cast<const float4 *>(shift + n * c + ch);
  auto one = [&](float4 v, float4 r) {
    if (silu && round && !rv) {  // the decode's GroupNorm+SiLU: packed form
      const float2 s0 = silu2_tf32(v.x, v.y, a.x, a.y, b.x, b.y);
      const float2 s1 = silu2_tf32(v.z, v.w, a.z, a.w, b.z, b.w);
      return make_float4(s0.x, s0.y, s1.x, s1.y);
    }
    float4 o;
    o.x = act(fmaf(v.x, a.x, b.x), silu) + r.x;
    o.y = act(fmaf(v.y, a.y, b.y), silu) + r.y;
    o.z = act(fmaf(v.z, a.z, b.z), silu) + r.z;
    o.w = act(fmaf(v.w, a.w, b.w), silu) + r.w;
    o.x = rnd(o.x, round);
    o.y = rnd(o.y, round);
    o.z = rnd(o.z, round);
    o.w = rnd(o.w, round);
    return o;
  };
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  unsigned i = i0;
  for (; i + 3 * stride < per_sample4; i += 4 * stride) {
    float4 v[4], r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      v[u] = __ldg(xv + i + u * stride);
      r[u] = rv ? __ldg(rv + i + u * stride) : zero;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) yv[i + u * stride] = one(v[u], r[u]);
  }
  for (; i < per_sample4; i += stride) yv[i] = one(__ldg(xv + i), rv ? __ldg(rv + i) : zero);
}

__global__ void gn_apply_nchw(const float *__restrict__ x, long long total, int c,
                              long long spatial, const float *__restrict__ scale,
                              const float *__restrict__ shift, int silu, int round,
                              float *__restrict__ y) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long nc = i / spatial;  // n * c + ch
    y[i] = rnd(act(fmaf(x[i], scale[nc], shift[nc]), silu), round);
  }
}

// Partials per group up to which every apply block merges them itself.
constexpr int kFusedMaxSlots = 64;
constexpr int kCompactThreads = 256;

// Fixed-order merge of the 32 lanes' triples (xor butterfly: at each level a
// lane merges the lower-lane operand first); every lane returns the total,
// bit-identical to lane 0's.
__device__ __forceinline__ Triple warp_merge(Triple acc) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Triple other{__shfl_xor_sync(0xffffffffu, acc.n, o),
                       __shfl_xor_sync(0xffffffffu, acc.mean, o),
                       __shfl_xor_sync(0xffffffffu, acc.m2, o)};
    acc = (threadIdx.x & o) ? merge(other, acc) : merge(acc, other);
  }
  return acc;
}

// Compacted slots per (sample, group) in gn_compact_finalize: one block each,
// so a 32-group sample takes 512 blocks, a single wave on the SMs.
constexpr int kCompactSlots = 16;

// Merge each (sample, group)'s `slots` partials in two levels within one
// launch. Block (b, ng) merges the contiguous slot range b of kCompactSlots
// equal ranges (fixed order: thread-strided, a warp butterfly, then the
// block's warps in order) into compacted slot b, then counts itself in on
// its (sample, group)'s counter; the block that arrives last merges the
// kCompactSlots compacted slots in a fixed order (so the result does not
// depend on which block is last), writes the group's per-channel affine and
// puts the counter back to zero for the next launch. `cnt` [n * groups] must
// be zero on entry.
__global__ void __launch_bounds__(kCompactThreads)
    gn_compact_finalize(const float *__restrict__ part, long long slots, float *compact,
                        unsigned *cnt, int c, int groups, float eps,
                        const float *__restrict__ gamma, const float *__restrict__ beta,
                        float *__restrict__ scale, float *__restrict__ shift) {
  constexpr int kWarps = kCompactThreads / 32;
  __shared__ Triple red[kWarps];
  __shared__ int last;
  const int b = blockIdx.x, ng = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long per = (slots + kCompactSlots - 1) / kCompactSlots;
  const long long s0 = b * per, s1 = s0 + per < slots ? s0 + per : slots;
  const float *e = part + static_cast<long long>(ng) * slots * 3;
  Triple acc{0.f, 0.f, 0.f};
  for (long long sl = s0 + threadIdx.x; sl < s1; sl += kCompactThreads)
    acc = merge(acc, Triple{e[3 * sl], e[3 * sl + 1], e[3 * sl + 2]});
  acc = warp_merge(acc);
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  float *mine = compact + static_cast<long long>(ng) * kCompactSlots * 3;
  if (threadIdx.x == 0) {
    Triple t = red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) t = merge(t, red[w]);
    mine[3 * b] = t.n;
    mine[3 * b + 1] = t.mean;
    mine[3 * b + 2] = t.m2;
    __threadfence();  // the slot is visible device-wide before the count
    const unsigned seen = atomicAdd(cnt + ng, 1u);
    last = seen == kCompactSlots - 1;
    if (last) __threadfence();  // every other block's slot is visible to this one
  }
  __syncthreads();
  if (!last) return;
  // the last block: warp 0 merges the compacted slots
  if (warp == 0) {
    Triple t{0.f, 0.f, 0.f};
    if (lane < kCompactSlots)
      t = Triple{__ldcg(mine + 3 * lane), __ldcg(mine + 3 * lane + 1),
                 __ldcg(mine + 3 * lane + 2)};
    t = warp_merge(t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  const int cg = c / groups;
  const int n = ng / groups, g = ng % groups;
  for (int i = threadIdx.x; i < cg; i += kCompactThreads) {
    // FP64 only on the cg threads that write a channel (FP64 is slow here)
    const double cntv = red[0].n;
    const double mean = red[0].mean;
    const double var = cntv > 0 ? red[0].m2 / cntv : 0.0;
    const double rstd = 1.0 / sqrt(var + static_cast<double>(eps));
    const int ch = g * cg + i;
    const double a = rstd * gamma[ch];
    scale[n * c + ch] = static_cast<float>(a);
    shift[n * c + ch] = static_cast<float>(beta[ch] - mean * a);
  }
  if (threadIdx.x == 0) cnt[ng] = 0u;
}

__device__ __forceinline__ void apply_share(const float *__restrict__ x, unsigned per_sample4,
                                            int c, int silu, int round,
                                            const float *__restrict__ res, float *__restrict__ y,
                                            const float *ssc, const float *ssh, int n,
                                            unsigned blk, unsigned nblk);

// Merge sample n's partials ([n][groups][slots], float) into scale/shift in
// shared memory (ssc, ssh: c floats each), then the vectorised apply loop of
// gn_apply_nhwc over this block's share (block blk of nblk; nblk * 1024 a
// multiple of c).
__device__ __forceinline__ void apply_from_partials(
    const float *__restrict__ x, unsigned per_sample4, int c, const float *__restrict__ part,
    int slots, int groups, float eps, const float *__restrict__ gamma,
    const float *__restrict__ beta, int silu, int round, const float *__restrict__ res,
    float *__restrict__ y, float *ssc, float *ssh, int n, unsigned blk, unsigned nblk) {
  const int cg = c / groups;
  // tpg lanes (a power of two <= 32) merge one group's partials: strided
  // over the slots, then a butterfly over the lanes.
  int tpg = 1;
  while (tpg < 32 && tpg * 2 * groups <= 256) tpg *= 2;
  const int sub = threadIdx.x & (tpg - 1);
  for (int g0 = 0; g0 < groups; g0 += 256 / tpg) {
    const int g = g0 + threadIdx.x / tpg;  // uniform across each tpg-lane set
    Triple acc{0.f, 0.f, 0.f};
    if (g < groups) {
      const float *e = part + (static_cast<size_t>(n) * groups + g) * slots * 3;
      for (int sl = sub; sl < slots; sl += tpg)
        acc = merge(acc, Triple{e[3 * sl], e[3 * sl + 1], e[3 * sl + 2]});
    }
    for (int o = 1; o < tpg; o <<= 1) {
      const Triple other{__shfl_xor_sync(0xffffffffu, acc.n, o),
                         __shfl_xor_sync(0xffffffffu, acc.mean, o),
                         __shfl_xor_sync(0xffffffffu, acc.m2, o)};
      acc = (threadIdx.x & o) ? merge(other, acc) : merge(acc, other);
    }
    if (g < groups && sub == 0) {
      const float var = acc.n > 0.f ? acc.m2 / acc.n : 0.f;
      const float rstd = rsqrtf(var + eps);
      for (int ch = g * cg; ch < (g + 1) * cg; ++ch) {
        const float a = rstd * gamma[ch];
        ssc[ch] = a;
        ssh[ch] = beta[ch] - acc.mean * a;
      }
    }
  }
  __syncthreads();
  apply_share(x, per_sample4, c, silu, round, res, y, ssc, ssh, n, blk, nblk);
}

// The vectorised apply over block blk's share (of nblk) of sample n, with the
// affine in shared memory (ssc, ssh).
__device__ __forceinline__ void apply_share(const float *__restrict__ x, unsigned per_sample4,
                                            int c, int silu, int round,
                                            const float *__restrict__ res, float *__restrict__ y,
                                            const float *ssc, const float *ssh, int n,
                                            unsigned blk, unsigned nblk) {
  const size_t base4 = static_cast<size_t>(n) * per_sample4;
  const float4 *xv = reinterpret_cast<const float4 *>(x) + base4;
  float4 *yv = reinterpret_cast<float4 *>(y) + base4;
  const float4 *rv = res ? reinterpret_cast<const float4 *>(res) + base4 : nullptr;
  const unsigned i0 = blk * 256u + threadIdx.x;
  const unsigned stride = nblk * 256u;
  const int ch = static_cast<int>((i0 * 4u) % static_cast<unsigned>(c));
  const float4 a = *reinterpret_cast<const float4 *>(ssc + ch);
  const float4 b = *reinterpret_cast<const float4 *>(ssh + ch);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  auto one = [&](float4 v, float4 r) {
    if (silu && round && !rv) {  // the decode's GroupNorm+SiLU: packed form
      const float2 s0 = silu2_tf32(v.x, v.y, a.x, a.y, b.x, b.y);
      const float2 s1 = silu2_tf32(v.z, v.w, a.z, a.w, b.z, b.w);
      return make_float4(s0.x, s0.y, s1.x, s1.y);
    }
    float4 o;
    o.x = rnd(act(fmaf(v.x, a.x, b.x), silu) + r.x, round);
    o.y = rnd(act(fmaf(v.y, a.y, b.y), silu) + r.y, round);
    o.z = rnd(act(fmaf(v.z, a.z, b.z), silu) + r.z, round);
    o.w = rnd(act(fmaf(v.w, a.w, b.w), silu) + r.w, round);
    return o;
  };
  unsigned i = i0;
  for (; i + 3 * stride < per_sample4; i += 4 * stride) {  // four loads in flight
    float4 v[4], r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      v[u] = __ldg(xv + i + u * stride);
      r[u] = rv ? __ldg(rv + i + u * stride) : zero;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) yv[i + u * stride] = one(v[u], r[u]);
  }
  for (; i < per_sample4; i += stride) yv[i] = one(__ldg(xv + i), rv ? __ldg(rv + i) : zero);
}

// Finalize and apply in one kernel, for few partials per group: every CTA
// merges its sample's partials into shared scale/shift, then runs the same
// vectorised apply loop as gn_apply_nhwc.
__global__ void __launch_bounds__(256)
    gn_apply_fused_nhwc(const float *__restrict__ x, unsigned per_sample4, int c,
                        const float *__restrict__ part, int slots, int groups, float eps,
                        const float *__restrict__ gamma, const float *__restrict__ beta, int silu,
                        int round, const float *__restrict__ res, float *__restrict__ y) {
  __shared__ __align__(16) float ssc[1024];
  __shared__ __align__(16) float ssh[1024];
  apply_from_partials(x, per_sample4, c, part, slots, groups, eps, gamma, beta, silu, round, res,
                      y, ssc, ssh, blockIdx.y, blockIdx.x, gridDim.x);
}

// Arrive at a grid-wide barrier (counter zeroed before the launch; each
// barrier adds gridDim.x * gridDim.y) and wait for `target` arrivals; the
// wait is bounded (VAE_EDEVICE_TIMEOUT). Returns false to every thread of
// the block when it gave up.
__device__ __forceinline__ bool grid_barrier(unsigned *bar, unsigned target, int *err,
                                             unsigned long long wait_ns, int *s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    const uint64_t t0 = global_timer_ns();
    int ok = 1;
    while (static_cast<unsigned>(ld_acquire_gpu(reinterpret_cast<const int *>(bar))) < target) {
      __nanosleep(64);  // (hundreds of pollers share the counter's cache line)
      if (global_timer_ns() - t0 > wait_ns) {
        atomicCAS(err, 0, static_cast<int>(VAE_EDEVICE_TIMEOUT));
        ok = 0;
        break;
      }
    }
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// The whole GroupNorm(+SiLU) in one cooperative launch, for tensors that L2
// holds between the two reads: every block reduces its slab of pixels into
// per-(block, group) partials; after a grid barrier the first n * groups
// blocks each merge one (sample, group)'s partials into the per-channel
// affine (scale, shift); after a second barrier every block applies it to its
// share -- the second read of x comes from L2, so HBM moves each element in
// and out once.
__global__ void __launch_bounds__(256)
    gn_coop_nhwc(const float *__restrict__ x, int c, long long spatial, int groups, float eps,
                 const float *__restrict__ gamma, const float *__restrict__ beta, int silu,
                 int round, const float *__restrict__ res, float *__restrict__ y,
                 float *__restrict__ part, float *__restrict__ scale, float *__restrict__ shift,
                 unsigned *bar, int *err, unsigned long long wait_ns) {
  __shared__ __align__(16) float ssc[1024];
  __shared__ __align__(16) float ssh[1024];
  __shared__ float red[256][3];
  __shared__ int s_ok;
  extern __shared__ float sm[];  // stats scratch [ppi][c] x 3
  const int n = blockIdx.y;
  const int nblk = gridDim.x;
  const unsigned total = gridDim.x * gridDim.y;
  stats_slab_nhwc(x, c, spatial, groups, nblk, n, blockIdx.x, sm, part);
  if (!grid_barrier(bar, total, err, wait_ns, &s_ok)) return;
  const int lin = blockIdx.y * gridDim.x + blockIdx.x;
  if (lin < static_cast<int>(gridDim.y) * groups)
    finalize_group(part, nblk, c, groups, eps, gamma, beta, scale, shift, lin, red);
  if (!grid_barrier(bar, 2 * total, err, wait_ns, &s_ok)) return;
  for (int ch = threadIdx.x; ch < c; ch += blockDim.x) {
    ssc[ch] = __ldcg(scale + n * c + ch);  // (written in this launch: not through L1's
    ssh[ch] = __ldcg(shift + n * c + ch);  //  read-only path)
  }
  __syncthreads();
  apply_share(x, static_cast<unsigned>(spatial * c / 4), c, silu, round, res, y, ssc, ssh, n,
              blockIdx.x, nblk);
}

// Blocks per sample for the apply loops: a multiple of c / gcd(c, 1024) so
// the loop stride (blocks * 1024 elements) is a multiple of c.
long long apply_blocks(long long per4, int c, int n) {
  long long g = std::min<long long>((per4 + 255) / 256, std::max(1ll, 8ll * num_sms() / n));
  long long gcd = c, b2 = 1024;
  while (b2) {
    const long long t = gcd % b2;
    gcd = b2;
    b2 = t;
  }
  const long long unit = c / gcd;
  return std::max(unit, g / unit * unit);
}

int launch_apply_nhwc(const float *x, int n, int c, long long spatial, const float *scale,
                      const float *shift, int silu, int round_out, const float *residual,
                      float *y, cudaStream_t s) {
  const int threads = 256;
  const long long per4 = spatial * c / 4;
  if (per4 > 0xffffffffll / 2) return VAE_EUNSUPPORTED;
  // blocks per sample: a multiple of c / gcd(c, 1024), so the loop stride
  // (blocks * 1024 elements) is a multiple of c and channels stay fixed
  long long g = std::min<long long>((per4 + threads - 1) / threads,
                                    std::max(1ll, 8ll * num_sms() / n));
  long long gcd = c, b2 = 1024;
  while (b2) {
    const long long t = gcd % b2;
    gcd = b2;
    b2 = t;
  }
  const long long unit = c / gcd;
  g = std::max(unit, g / unit * unit);
  if ((g * 1024) % c != 0) return VAE_EUNSUPPORTED;
  gn_apply_nhwc<<<dim3(static_cast<unsigned>(g), n), threads, 0, s>>>(
      x, static_cast<unsigned>(per4), c, scale, shift, silu, round_out, residual, y);
  return cudaGetLastError() == cudaSuccess ? VAE_OK : VAE_ECUDA;
}

int nblk_for(long long elems_per_seg, int segs) {
  long long want = elems_per_seg / (kStatThreads * 16);
  const long long cap = std::max(1ll, 4ll * num_sms() / std::max(1, segs));
  want = std::min(want, cap);
  want = std::min<long long>(want, kMaxBlocksPerGroupSeg);
  return static_cast<int>(std::max(1ll, want));
}

}  // namespace

size_t groupnorm_ws_bytes(int n, int c, long long spatial, int groups) {
  (void)spatial;
  Carver cv(nullptr, 0);
  cv.take<double>(static_cast<size_t>(n) * groups * kMaxBlocksPerGroupSeg * 3);
  cv.take<float>(static_cast<size_t>(n) * c);
  cv.take<float>(static_cast<size_t>(n) * c);
  return cv.used;
}

namespace {

// VAE_GN=multipass keeps every GroupNorm on the three-launch path
// (comparisons).
bool coop_gn_enabled() {
  static const bool v = [] {
    const char *e = std::getenv("VAE_GN");
    return !(e && std::strcmp(e, "multipass") == 0);
  }();
  return v;
}

// The one-launch path (gn_coop_nhwc): NHWC tensors of at most kCoopMaxBytes
// (L2 keeps them between the two reads), the grid co-resident. Returns
// VAE_EUNSUPPORTED when it does not apply (the caller takes the three-launch
// path).
constexpr long long kCoopMaxBytes = 64ll << 20;

int groupnorm_coop(const float *x, int n, int c, long long spatial, int groups, float eps,
                   const float *gamma, const float *beta, int silu, int round_out, float *y,
                   void *ws, cudaStream_t s, const float *residual) {
  if (static_cast<long long>(n) * spatial * c * 4 > kCoopMaxBytes) return VAE_EUNSUPPORTED;
  const long long per4 = spatial * c / 4;
  if (per4 > 0xffffffffll / 2) return VAE_EUNSUPPORTED;
  const int tpp = c / 4, ppi = kStatThreads / tpp;
  const size_t sm = static_cast<size_t>(ppi) * c * 3 * sizeof(float);
  int dev = 0, coop = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
    return VAE_EUNSUPPORTED;
  // resident blocks per SM at this call's dynamic shared memory size
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gn_coop_nhwc, 256, sm) !=
      cudaSuccess || per_sm <= 0)
    return VAE_EUNSUPPORTED;
  // blocks per sample: up to four per SM in all, a multiple of c / gcd(c, 1024)
  long long gcd = c, b2 = 1024;
  while (b2) {
    const long long t = gcd % b2;
    gcd = b2;
    b2 = t;
  }
  const long long unit = c / gcd;
  const long long resident = static_cast<long long>(per_sm) * num_sms();
  long long bps = std::min<long long>(std::min(4ll * num_sms(), resident) / n,
                                      (per4 + 255) / 256);
  bps = std::min<long long>(bps, kMaxBlocksPerGroupSeg) / unit * unit;  // (fits the workspace)
  if (bps < 1 || bps * n > resident || bps > spatial) return VAE_EUNSUPPORTED;
  if (static_cast<long long>(n) * groups > bps * n) return VAE_EUNSUPPORTED;  // finalize blocks
  Carver cv(ws, ~size_t(0));
  float *part = cv.take<float>(static_cast<size_t>(n) * groups * bps * 3);
  float *scale = cv.take<float>(static_cast<size_t>(n) * c);
  float *shift = cv.take<float>(static_cast<size_t>(n) * c);
  unsigned *bar = cv.take<unsigned>(1);
  int *err = device_error_word();
  if (!err) return VAE_ECUDA;
  VAE_CUDA_TRY(cudaMemsetAsync(bar, 0, sizeof(unsigned), s));
  const unsigned long long wait_ns = wait_limit_ns();
  void *args[] = {const_cast<float **>(&x), &c, &spatial, &groups, &eps,
                  const_cast<float **>(&gamma), const_cast<float **>(&beta), &silu, &round_out,
                  const_cast<float **>(&residual), &y, &part, &scale, &shift, &bar, &err,
                  const_cast<unsigned long long *>(&wait_ns)};
  VAE_CUDA_TRY(cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(gn_coop_nhwc),
                                           dim3(static_cast<unsigned>(bps), n), dim3(256), args,
                                           sm, s));
  count_launches(1);
  return VAE_OK;
}

}  // namespace

int groupnorm_silu(const float *x, int n, int c, long long spatial, int nhwc, int groups,
                   float eps, const float *gamma, const float *beta, int silu, int round_out,
                   float *y, void *ws, cudaStream_t s, const float *residual) {
  if (!x || !y || !gamma || !beta || !ws || n <= 0 || c <= 0 || spatial <= 0 || groups <= 0)
    return VAE_EINVAL;
  if (c % groups || c % 4 || c > 1024) return VAE_EUNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
       reinterpret_cast<uintptr_t>(residual)) & 15)
    return VAE_EINVAL;
  if (residual && !nhwc) return VAE_EUNSUPPORTED;
  if (nhwc && coop_gn_enabled()) {
    const int rc = groupnorm_coop(x, n, c, spatial, groups, eps, gamma, beta, silu, round_out, y,
                                  ws, s, residual);
    if (rc != VAE_EUNSUPPORTED) return rc;
  }
  Carver cv(ws, ~size_t(0));
  double *part = cv.take<double>(static_cast<size_t>(n) * groups * kMaxBlocksPerGroupSeg * 3);
  float *scale = cv.take<float>(static_cast<size_t>(n) * c);
  float *shift = cv.take<float>(static_cast<size_t>(n) * c);
  const int cg = c / groups;
  int nblk;
  if (nhwc) {
    nblk = nblk_for(spatial * c, n);
    const int tpp = c / 4, ppi = kStatThreads / tpp;
    const size_t sm = static_cast<size_t>(ppi) * c * 3 * sizeof(float);
    gn_stats_nhwc<<<dim3(nblk, n), kStatThreads, sm, s>>>(x, c, spatial, groups, nblk, part);
  } else {
    nblk = nblk_for(spatial * cg, n * groups);
    gn_stats_nchw<<<dim3(nblk, n * groups), kStatThreads, 0, s>>>(x, c, spatial, groups, nblk,
                                                                   part);
  }
  VAE_LAUNCH_CHECK();
  gn_finalize<double><<<n * groups, kFinalizeThreads, 0, s>>>(part, nblk, c, groups, eps, gamma,
                                                               beta, scale, shift);
  VAE_LAUNCH_CHECK();
  const long long total = static_cast<long long>(n) * c * spatial;
  const int threads = 256;
  if (nhwc) {
    VAE_TRY(launch_apply_nhwc(x, n, c, spatial, scale, shift, silu, round_out, residual, y, s));
  } else {
    const long long g = std::min<long long>((total + threads - 1) / threads, 8ll * num_sms());
    gn_apply_nchw<<<static_cast<int>(g), threads, 0, s>>>(x, total, c, spatial, scale, shift,
                                                          silu, round_out, y);
  }
  VAE_LAUNCH_CHECK();
  count_launches(3);
  return VAE_OK;
}

int groupnorm_scale_shift(const float *x, int n, int c, long long spatial, int groups, float eps,
                          const float *gamma, const float *beta, const float *part,
                          long long slots, float *scale, float *shift, void *ws,
                          cudaStream_t s, unsigned *counters) {
  if (!x || !gamma || !beta || !scale || !shift || n <= 0 || c <= 0 || spatial <= 0 ||
      groups <= 0)
    return VAE_EINVAL;
  if (c % groups || c % 4 || c > 1024) return VAE_EUNSUPPORTED;
  if (part && counters && slots > kFusedMaxSlots) {
    if (!ws) return VAE_EINVAL;
    Carver cv(ws, ~size_t(0));
    float *compact = cv.take<float>(static_cast<size_t>(n) * groups * kCompactSlots * 3);
    gn_compact_finalize<<<dim3(kCompactSlots, static_cast<unsigned>(n * groups)),
                          kCompactThreads, 0, s>>>(part, slots, compact, counters, c, groups,
                                                   eps, gamma, beta, scale, shift);
    VAE_LAUNCH_CHECK();
    count_launches(1);
    return VAE_OK;
  }
  if (part) {
    gn_finalize<float><<<n * groups, kFinalizeThreads, 0, s>>>(part, slots, c, groups, eps, gamma, beta,
                                                  scale, shift);
    VAE_LAUNCH_CHECK();
    count_launches(1);
    return VAE_OK;
  }
  if (!ws) return VAE_EINVAL;
  Carver cv(ws, ~size_t(0));
  double *dpart = cv.take<double>(static_cast<size_t>(n) * groups * kMaxBlocksPerGroupSeg * 3);
  const int nblk = nblk_for(spatial * c, n);
  const int tpp = c / 4, ppi = kStatThreads / tpp;
  const size_t sm = static_cast<size_t>(ppi) * c * 3 * sizeof(float);
  gn_stats_nhwc<<<dim3(nblk, n), kStatThreads, sm, s>>>(x, c, spatial, groups, nblk, dpart);
  VAE_LAUNCH_CHECK();
  gn_finalize<double><<<n * groups, kFinalizeThreads, 0, s>>>(dpart, nblk, c, groups, eps, gamma, beta,
                                                 scale, shift);
  VAE_LAUNCH_CHECK();
  count_launches(2);
  return VAE_OK;
}

int groupnorm_apply(const float *x, int n, int c, long long spatial, const float *scale,
                    const float *shift, int silu, int round_out, float *y, cudaStream_t s) {
  if (!x || !y || !scale || !shift || n <= 0 || c <= 0 || spatial <= 0) return VAE_EINVAL;
  if (c % 4 || c > 1024) return VAE_EUNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) return VAE_EINVAL;
  VAE_TRY(launch_apply_nhwc(x, n, c, spatial, scale, shift, silu, round_out, nullptr, y, s));
  count_launches(1);
  return VAE_OK;
}

int groupnorm_from_partials(const float *x, int n, int c, long long spatial, int groups,
                            float eps, const float *gamma, const float *beta, int silu,
                            int round_out, const float *part, long long slots, float *y,
                            void *ws, cudaStream_t s, const float *residual,
                            unsigned *counters) {
  if (!x || !y || !gamma || !beta || !ws || !part || n <= 0 || c <= 0 || spatial <= 0 ||
      groups <= 0 || slots <= 0)
    return VAE_EINVAL;
  if (c % groups || c % 4 || c > 1024) return VAE_EUNSUPPORTED;
  Carver cv(ws, ~size_t(0));
  if (slots <= kFusedMaxSlots) {
    // Few partials: every apply block merges them itself (one launch).
    const long long per4 = spatial * c / 4;
    if (per4 > 0xffffffffll / 2) return VAE_EUNSUPPORTED;
    const long long g = apply_blocks(per4, c, n);
    if ((g * 1024) % c != 0) return VAE_EUNSUPPORTED;
    gn_apply_fused_nhwc<<<dim3(static_cast<unsigned>(g), n), 256, 0, s>>>(
        x, static_cast<unsigned>(per4), c, part, static_cast<int>(slots), groups, eps, gamma,
        beta, silu, round_out, residual, y);
    VAE_LAUNCH_CHECK();
    count_launches(1);
    return VAE_OK;
  }
  // Many partials: compact them with all SMs busy and merge the compacted
  // slots into scale/shift in the same launch, then the plain apply pass.
  float *scale = cv.take<float>(static_cast<size_t>(n) * c);
  float *shift = cv.take<float>(static_cast<size_t>(n) * c);
  float *compact = cv.take<float>(static_cast<size_t>(n) * groups * kCompactSlots * 3);
  if (!counters) return VAE_EINVAL;
  gn_compact_finalize<<<dim3(kCompactSlots, static_cast<unsigned>(n * groups)),
                        kCompactThreads, 0, s>>>(part, slots, compact, counters, c, groups, eps,
                                                 gamma, beta, scale, shift);
  VAE_LAUNCH_CHECK();
  VAE_TRY(launch_apply_nhwc(x, n, c, spatial, scale, shift, silu, round_out, residual, y, s));
  count_launches(2);
  return VAE_OK;
}

}  // namespace vae
