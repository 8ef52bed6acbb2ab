// igemm_kernel.cuh -- the implicit-GEMM tcgen05 kernel (igemm.cu describes
// its design): parameters, tile configurations, the kernel template and its
// launcher. Included by igemm.cu (TF32 instantiations) and igemm_split.cu
// (split-TF32 instantiations), so each kernel is instantiated in exactly one
// translation unit.
#pragma once
#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace vae {
namespace igk {


constexpr int kBM = 128;
constexpr int kThreads = 192;
constexpr uint32_t kABytes = kBM * 128;

struct KParams {
  int imgs, t, hin, win, hout, wout;
  int bh, bw;  // tile rows / cols (Conv: output pixels; Upsample: low-res pixels)
  int tiles_x, tiles_y;
  int m_tiles, n_tiles, total_tiles;
  int M;
  int k, kt, taps;
  int cin_chunks, sc_chunks, k_stages, cin_pad;
  // split-K: tile index = (split, m tile, n tile); split s covers reduction
  // steps [s * ks_per, min((s + 1) * ks_per, k_stages)) and writes its raw
  // partial sums at out + s * split_stride.
  int splits, ks_per;
  long long split_stride;
  int cout;
  float *out;
  int ldo, out_nchw;
  const float *bias;
  int bias_per_row;
  const float *residual;
  float alpha;
  int round_out;
  int epi_tma;  // 1: rows leave through shared staging + TMA stores (NHWC / GEMM)
  int has_res;  // residual present (TMA-loaded into the staging buffer when epi_tma)
  // GroupNorm statistics of the output (optional): per (sample, group, slot)
  // partial (count, mean, M2); slot = (frame, tile, sub-tile, warp).
  float *stat_part;
  int stat_cg;       // channels per group (power of two dividing 32)
  int stat_groups;   // groups over cout
  int stat_slots;    // slots per (sample, group)
  // Stream-K (when whole tiles would leave the last round of SMs mostly
  // idle): CTA c runs units [c * sk_total / G, (c + 1) * sk_total / G) of the
  // flattened (tile, reduction unit) space, sk_units units per tile (a unit
  // is one reduction step, or one 32-channel chunk in MODE 3). A tile cut
  // between two CTAs: the CTA holding its later part (the tail, at the start
  // of its range) writes the raw sums to its slot of sk_part and raises its
  // flags; the CTA holding the head (at the end of its range) adds them in
  // its epilogue. Fixed split points: deterministic. (1-SM tiles only; the
  // hand-over indexes the neighbour as blockIdx + NCTA.)
  int sk;
  int sk_units;
  long long sk_total;
  float *sk_part;
  int *sk_flag;  // [G][4]: one per epilogue warp, zeroed before the launch
  int *err;
  uint64_t wait_ns;  // limit of every device-side wait (normally kWaitTimeoutNs)
  int inject;        // test hook: VAE_INJECT_* bits (0 in normal operation)
  // XF = 1: GroupNorm (+SiLU) of the halo-staged input applied in shared
  // memory before the MMAs: v -> silu(v * gn_scale[s][c] + gn_shift[s][c]),
  // TF32-rounded, zero outside the image; s = image / t, [s][cin_pad].
  const float *gn_scale, *gn_shift;
  int gn_silu;
  // XF = 2: the A stage holds raw attention scores s; the MMA reads
  // p = exp(s * sm_scale - sm_m[row]) * sm_inv_l[row] (0 for keys >= sm_cols).
  const float *sm_m, *sm_inv_l;
  float sm_scale;
  int sm_cols;
  // GEMM epilogue (optional): per row and 256-column tile, the softmax
  // statistics (max of v * rs_scale over the valid columns, and the sum of
  // exp(v * rs_scale - max)) of the stored values, at rs_out[row * rs_ld + n tile].
  float2 *rs_out;
  float rs_scale;
  int rs_cols, rs_ld;
  // XF = 3 (GroupNorm ahead): the conv's A source ga_t (= the tensor tmA
  // reads) is the GroupNorm+SiLU of ga_x, made by four more warps of every
  // CTA while the conv runs: they take image rows (units: image * hin + row)
  // from the counter ga_next in order, write ga_t = tf32(silu(ga_x *
  // ga_scale[s][c] + ga_shift[s][c])) for the row and set ga_flags[unit] =
  // ga_epoch; the producer waits for the rows a tile reads before its copies.
  const float *ga_x, *ga_scale, *ga_shift;
  float *ga_t;
  int *ga_flags, *ga_next;
  int ga_epoch;
};

// One work item of a CTA: a tile and the range [k0, k1) of its reduction
// units (reduction steps; 32-channel chunks in MODE 3).
struct Work {
  int tile, k0, k1;
  bool head, tail;  // stream-K: the tile's first part here and the rest on the next CTA / the reverse
};

// The CTA's work items, identical in the producer, MMA and epilogue roles.
// `id` / `count`: this worker and the number of workers (a CTA, or a CTA
// pair sharing paired MMAs).
template <int MODE>
struct WorkIter {
  long long u, end;
  int tile, step;
  __device__ WorkIter(const KParams &p, int id, int count) : u(0), end(0), tile(id), step(count) {
    if (p.sk) {
      u = p.sk_total * id / count;
      end = p.sk_total * (id + 1) / count;
    }
  }
  __device__ bool next(const KParams &p, Work &w) {
    if (p.sk) {
      if (u >= end) return false;
      w.tile = static_cast<int>(u / p.sk_units);
      w.k0 = static_cast<int>(u % p.sk_units);
      const long long left = end - u;
      w.k1 = left < p.sk_units - w.k0 ? w.k0 + static_cast<int>(left) : p.sk_units;
      w.tail = w.k0 > 0;
      w.head = w.k0 == 0 && w.k1 < p.sk_units;
      u += w.k1 - w.k0;
      return true;
    }
    if (tile >= p.total_tiles) return false;
    w.tile = tile;
    if (MODE == 3) {
      w.k0 = 0;
      w.k1 = p.cin_chunks;
    } else {
      const int split = tile / (p.m_tiles * p.n_tiles);
      w.k0 = split * p.ks_per;
      w.k1 = min(w.k0 + p.ks_per, p.k_stages);
    }
    w.head = w.tail = false;
    tile += step;
    return true;
  }
};

// BN: output channels per tile (MMA N; MMA M in MODE 4). MS: 128-row M sub-tiles per tile
// sharing each B stage (1, or 2 for 128-channel convs: a 256-pixel tile keeps
// the operand bytes per FLOP of a 128 x 256 tile). MODE 3 (halo conv): the
// input tile of a 32-channel chunk is staged once, with a one-pixel halo
// ((MS + 2) rows x 130 pixels, two buffers), and serves all nine taps; the
// ring stages then carry weights only.
// PAIR: a cluster of two CTAs on paired SMs runs one tile of 256 pixel rows
// x BN channels with tcgen05.mma.cta_group::2 (M = 256): each CTA stages its
// own 128 rows of A and half of the BN weight rows, the leader CTA issues the
// MMAs, and each CTA's TMEM receives its own 128 accumulator rows. Per SM and
// reduction step half the weight bytes cross shared memory, which lifts the
// shared-memory bound of the 1-SM tile.
// SPLIT: split-TF32 products. Each stage lands in FP32; four more warps
// split it in place into TF32 parts (hi = tf32(v), lo = tf32(v - hi), lo
// stored beside hi) and the MMA issuer forms a_hi b_hi + a_lo b_hi + a_hi
// b_lo (three MMAs per step) into the FP32 accumulator.
// XF: four more warps per CTA. 1 and 2 transform each landed A buffer
// between the copy and the MMA (1: GroupNorm+SiLU of the halo buffer, MODE
// 3; 2: softmax normalisation of the GEMM A stage, MODE 2): each CTA's copy
// lands on a barrier of its own, then the transforming warps of both CTAs
// of a pair arrive on the leader's barrier the MMA issuer waits on. 3
// (MODES 3, 4) writes the conv's A operand itself, the GroupNorm+SiLU of the
// layer's input, a few rows ahead of the tiles that read it (see KParams).
template <int BN, int MS, int MODE = 0, bool PAIR = false, bool SPLIT = false, int XF = 0>
struct Cfg {
  static constexpr bool HALO = MODE == 3;
  static constexpr bool SWAP = MODE == 4;
  static_assert(!PAIR || (MS == 1 && BN == 256 && MODE <= 3),
                "paired tiles: 256 output columns, the pixel-major conv modes and GEMM");
  static_assert(!SPLIT || (!PAIR && MODE <= 2), "split products: per-step A and B stages");
  static_assert(XF == 0 || (!SPLIT && ((XF == 1 && MODE == 3) || (XF == 2 && MODE == 2 && MS == 1) ||
                                       (XF == 3 && (MODE == 3 || MODE == 4)))),
                "operand transforms: GroupNorm on halo buffers, softmax on GEMM A stages, "
                "GroupNorm ahead of the buffered-A conv modes");
  // Epilogue warps: eight (two per TMEM lane quarter, each taking half of
  // the tile's columns) on the upsample parity tiles, whose epilogue (four
  // taps of reduction per output pixel, GroupNorm statistics of a large
  // output) otherwise paces the tile: 0.74 -> 0.63 ms for the 1024^2
  // upsample conv. Four elsewhere (measured no faster with eight on the
  // channel-major and GEMM tiles).
  static constexpr int EPW = (!SPLIT && !XF && MODE == 1 && BN >= 128) ? 8 : 4;
  static constexpr int THREADS = 64 + 32 * EPW + ((SPLIT || XF) ? 128 : 0);
  static constexpr int NCTA = PAIR ? 2 : 1;
  // Separately buffered A operand (MODES 3 and 4), each buffer serving
  // several reduction steps: MODE 3 two halo buffers; MODE 4 three bands of
  // (bh + 2) rows x bw pixels with bh * bw = 256, at most 48 KB (bw <= 64),
  // so that a band's copy has two bands' MMAs to land in.
  static constexpr uint32_t HALO_BYTES =
      HALO ? ((MS + 2) * 130 * 128 + 1023) / 1024 * 1024 : SWAP ? 49152 : 0;
  static constexpr int HALO_BUFS = HALO ? 2 : SWAP ? 3 : 0;
  // MODE 4: appended-shortcut tiles (MS x 128 rows each) sharing one A buffer.
  static constexpr int SC_PER_BUF = SWAP ? static_cast<int>(HALO_BYTES / (MS * kABytes)) : 1;
  static constexpr uint32_t A_LOAD = (HALO || SWAP) ? 0 : MS * kABytes;  // TMA bytes per stage
  static constexpr uint32_t B_LOAD = (PAIR ? BN / 2 : BN) * 128;          // this CTA's weight rows
  static constexpr uint32_t A_BYTES = A_LOAD * (SPLIT ? 2 : 1);  // stage footprint (hi | lo)
  static constexpr uint32_t B_BYTES = B_LOAD * (SPLIT ? 2 : 1);
  // bytes that complete on `full` (XF = 2: the A stage lands on a barrier of
  // this CTA's own, for its transforming warps)
  static constexpr uint32_t STAGE_TX = (XF == 2 ? 0 : A_LOAD) + B_LOAD;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  // Epilogue staging: 4 warps x NSTG buffers x (32 rows x 128 bytes). Two
  // buffers let a block's store drain (and the next block's residual land)
  // while the warp works on the current one; the halo modes keep one so that
  // their shared memory holds more weight stages (measured faster on GB300).
  static constexpr int NSTG = (HALO || SWAP) ? 1 : 2;
  static constexpr uint32_t STAGING = EPW * NSTG * 4096;
  static constexpr int FIT =
      (232448 - 1024 - STAGING - 1024 - HALO_BUFS * HALO_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr uint32_t ACC_COLS = BN * MS;  // TMEM columns of one accumulator set
  static constexpr int ROWS = PAIR ? 2 : MS;  // 128-row sub-tiles of a (pair) tile
  static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS < 32 ? 32 : 2 * ACC_COLS;
  static constexpr int CH = BN < 32 ? BN : 32;  // epilogue column chunk
  static constexpr size_t SMEM = 1024 + HALO_BUFS * HALO_BYTES + STAGES * STAGE_BYTES + STAGING +
                                 (4 * STAGES + 29) * sizeof(uint64_t) + 16;
  static_assert(STAGES >= 2, "at least double-buffered stages");
  static_assert(!(HALO || SWAP) || STAGES >= 3, "buffered-A modes need a weight ring");
  static_assert(!SWAP || (BN == 128 && MS == 2), "MODE 4 tiles are 128 channels x 256 pixels");
  static_assert(TMEM_COLS <= 512, "accumulators exceed TMEM");
  static_assert(SMEM <= 232448, "shared memory budget");
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum each of NG per-lane values over the warp with a reduce-scatter
// butterfly: every step sends half of the remaining values to the partner
// lane, so NG - 1 + (5 - log2 NG) shuffles replace NG * 5. On return a[0]
// holds, in every lane, the total of group (lane >> (5 - log2 NG)).
template <int NG>
__device__ __forceinline__ void warp_reduce_scatter(float (&a)[NG], int lane) {
#pragma unroll
  for (int half = NG / 2, o = 16; half >= 1; half /= 2, o /= 2) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? a[i] : a[half + i];
      const float keep = upper ? a[half + i] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  constexpr int kLog = NG >= 32 ? 5 : NG >= 16 ? 4 : NG >= 8 ? 3 : NG >= 4 ? 2 : NG >= 2 ? 1 : 0;
#pragma unroll
  for (int o = 16 >> kLog; o >= 1; o /= 2) a[0] += __shfl_xor_sync(0xffffffffu, a[0], o);
}

// Exact two-pass (count, mean, M2) of each CG-channel group of a warp's 32
// rows x 32 channels (invalid rows excluded). The lanes holding a group's
// totals write its partial; successive groups are `gstride` floats apart.
template <int CG>
__device__ __forceinline__ void emit_group_stats(const float *v, bool valid, float nrows,
                                                 float *out, long long gstride, int lane) {
  constexpr int NG = 32 / CG;
  constexpr int kShift = NG >= 32 ? 0 : NG >= 16 ? 1 : NG >= 8 ? 2 : NG >= 4 ? 3 : NG >= 2 ? 4 : 5;
  const float cnt = nrows * CG;
  const float inv = cnt > 0.f ? __fdividef(1.0f, cnt) : 0.f;
  float a[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < CG; ++j) sum += v[g * CG + j];
    a[g] = valid ? sum : 0.f;
  }
  warp_reduce_scatter<NG>(a, lane);
  const float my_mean = a[0] * inv;  // mean of group (lane >> kShift)
  float m2[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const float mean = __shfl_sync(0xffffffffu, my_mean, g << kShift);
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < CG; ++j) {
      const float d = v[g * CG + j] - mean;
      acc = fmaf(d, d, acc);
    }
    m2[g] = valid ? acc : 0.f;
  }
  warp_reduce_scatter<NG>(m2, lane);
  if ((lane & ((1 << kShift) - 1)) == 0) {
    float *o = out + (lane >> kShift) * gstride;
    o[0] = cnt;
    o[1] = my_mean;
    o[2] = m2[0];
  }
}

__device__ __forceinline__ void raise_error(const KParams &p, volatile uint32_t *abort) {
  *abort = 1u;
  atomicCAS(p.err, 0, static_cast<int>(VAE_EDEVICE_TIMEOUT));
}

// Unbounded-by-abort wait used only while draining after an abort.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity,
                                                uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

template <int BN, int MODE, int MS, bool PAIR, bool SPLIT, int XF>
__global__ void __launch_bounds__(Cfg<BN, MS, MODE, PAIR, SPLIT, XF>::THREADS, 1)
    igemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmO,
                 const __grid_constant__ CUtensorMap tmR, const KParams p) {
  using C = Cfg<BN, MS, MODE, PAIR, SPLIT, XF>;
  constexpr int STAGES = C::STAGES;
  constexpr bool kConv = MODE == 0 || MODE == 3 || MODE == 4;  // conv tiles (epilogue geometry)
  constexpr uint32_t STAGE_TX = C::STAGE_TX;
  constexpr uint32_t IDESC = idesc_tf32(PAIR ? 2 * kBM : kBM, BN);
  constexpr uint32_t IDESC_SWAP = idesc_tf32(kBM, 256);  // MODE 4: M = channels, N = pixels

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sH = smem;  // A buffers (MODES 3 and 4)
  uint8_t *sA = smem + C::HALO_BUFS * C::HALO_BYTES;
  uint8_t *sB = sA + STAGES * C::A_BYTES;
  const uint32_t sB_u32 = smem_u32(sB);
  float *staging = reinterpret_cast<float *>(sB + STAGES * C::B_BYTES);  // 1024-aligned
  uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * C::B_BYTES + C::STAGING);
  uint64_t *empty = full + STAGES;
  uint64_t *acc_full = empty + STAGES;
  uint64_t *acc_empty = acc_full + 2;
  uint64_t *drain = acc_empty + 2;  // used only after an abort
  uint64_t *res_bar = drain + 1;    // per epilogue warp and staging buffer: residual landed
  uint64_t *a_full = res_bar + 16;  // MODES 3, 4: A buffer landed / free
  uint64_t *a_empty = a_full + 3;  // (three of each: the deepest A-buffer ring)
  uint64_t *xfull = a_empty + 3;    // SPLIT / XF 2: stage transformed, ready for the MMA
  uint64_t *xa_full = xfull + STAGES;  // XF 2: this CTA's A stage landed
  uint64_t *h_full = xa_full + STAGES;  // XF 1: this CTA's halo buffer landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(h_full + 2);
  volatile uint32_t *abort = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // PAIR: this CTA's rank in the pair; the leader (rank 0) issues the MMAs.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int wid = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int wcount = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], C::EPW * C::NCTA);  // every epilogue warp of the pair
    }
    mbar_init(drain, 1);
    for (int q = 0; q < 2 * C::EPW; ++q) mbar_init(&res_bar[q], 1);
    for (int b = 0; b < 3; ++b) {
      // XF 1: the transforming warps of every CTA of the pair arrive instead
      // of a copy completing
      mbar_init(&a_full[b], XF == 1 ? 4 * C::NCTA : 1);
      mbar_init(&a_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&h_full[b], 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&xfull[s], SPLIT ? 128 : 4 * C::NCTA);  // splitting threads / transforming warps
      mbar_init(&xa_full[s], 1);
    }
    *abort = 0u;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (kConv && p.sc_chunks > 0) prefetch_tmap(&tmS);
    if (p.epi_tma) {
      prefetch_tmap(&tmO);
      if (p.has_res) prefetch_tmap(&tmR);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Waits on barriers that the peer CTA (or the paired MMA) also arrives on
  // acquire at cluster scope.
  auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
    if constexpr (PAIR)
      return mbar_wait_cluster(bar, parity, abort, p.wait_ns);
    else
      return mbar_wait(bar, parity, abort, p.wait_ns);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t pending = 0, pend_par = 0;  // stages with a copy issued, and its parity
      uint32_t abuf = 0, aphase = 0;       // MODE 3 halo buffer ring
      uint32_t a_pending = 0, a_par = 0;  // (XF 1: copies onto h_full)
      uint32_t x_pending = 0, x_par = 0;  // XF 2: A copies onto xa_full
      bool failed = false;
      // PAIR: both CTAs' copies complete on the leader's barriers; this CTA
      // loads its own 128 A rows (tile rows from yoff) and weight rows from
      // boff. The leader expects the pair's bytes.
      const uint32_t full_c = PAIR ? mapa_rank(full, 0) : 0u;
      const uint32_t afull_c = PAIR ? mapa_rank(a_full, 0) : 0u;
      const int boff = PAIR ? static_cast<int>(rank) * (BN / 2) : 0;
      const int yoff = PAIR ? static_cast<int>(rank) * (p.bh >> 1) : 0;
      const uint32_t tx_mult = PAIR ? 2u : 1u;
      // XF 3: wait until image rows [r0, r1] (clamped to the image) are made
      // for this launch, then let the async proxy (the TMA) read them.
      auto wait_rows = [&](int img, int r0, int r1) -> bool {
        r0 = max(r0, 0);
        r1 = min(r1, p.hin - 1);
        for (int r = r0; r <= r1; ++r) {
          const int *f = p.ga_flags + static_cast<long long>(img) * p.hin + r;
          if (ld_acquire_gpu(f) == p.ga_epoch) continue;
          const uint64_t t0 = global_timer_ns();
          while (ld_acquire_gpu(f) != p.ga_epoch)
            if (*abort || global_timer_ns() - t0 > p.wait_ns) return false;
        }
        fence_proxy_async_global();
        return true;
      };
      WorkIter<MODE> it(p, wid, wcount);
      Work w;
      while (!failed && it.next(p, w)) {
        const int tile = w.tile;
        const int mn = tile % (p.m_tiles * p.n_tiles);
        const int mt = mn / p.n_tiles;
        const int n0 = (mn % p.n_tiles) * BN + boff;
        const int ks0 = w.k0, ks1 = w.k1;
        int img = 0, ty = 0, tx = 0, par = 0;
        if (MODE != 2) {
          const int per_img = p.tiles_x * p.tiles_y * (MODE == 1 ? 4 : 1);
          img = mt / per_img;
          int rem = mt % per_img;
          if (MODE == 1) {  // the four output parities of a low-res tile are adjacent tiles
            par = rem & 3;
            rem >>= 2;
          }
          ty = rem / p.tiles_x;
          tx = rem % p.tiles_x;
        }
        const int n_idx = img / p.t, t_idx = img % p.t;
        if constexpr (XF == 3) {
          // the rows this CTA's A copies of the tile read, once made
          const int r0 = MODE == 3 ? ty * p.bh + yoff - 1 : ty * p.bh - 1;
          const int r1 = MODE == 3 ? r0 + (PAIR ? (p.bh >> 1) : p.bh) + 1 : r0 + p.bh + 1;
          if (!wait_rows(img, r0, r1)) {
            raise_error(p, abort);
            failed = true;
            break;
          }
        }
        if constexpr (MODE == 3) {
          // One halo tile per 32-channel chunk, then one weight stage per tap
          // (no appended shortcut in this mode).
          for (int cc = ks0; cc < ks1 && !failed; ++cc) {
            if (!wait(&a_empty[abuf], aphase ^ 1u)) {
              raise_error(p, abort);
              failed = true;
              break;
            }
            if constexpr (XF == 1) {
              // lands on this CTA's own barrier, for its transforming warps
              mbar_arrive_expect_tx(&h_full[abuf], (MS + 2) * 130 * 128);
              tma_load_4d(sH + abuf * C::HALO_BYTES, &tmA, &h_full[abuf], cc * 32, tx * p.bw - 1,
                          ty * p.bh + yoff - 1, img);
            } else if constexpr (PAIR) {
              if (leader) mbar_arrive_expect_tx(&a_full[abuf], tx_mult * (MS + 2) * 130 * 128);
              tma_load_4d_pair(sH + abuf * C::HALO_BYTES, &tmA, afull_c + abuf * 8, cc * 32,
                               tx * p.bw - 1, ty * p.bh + yoff - 1, img);
            } else {
              mbar_arrive_expect_tx(&a_full[abuf], (MS + 2) * 130 * 128);
              tma_load_4d(sH + abuf * C::HALO_BYTES, &tmA, &a_full[abuf], cc * 32, tx * p.bw - 1,
                          ty * p.bh - 1, img);
            }
            a_pending |= 1u << abuf;
            a_par = (a_par & ~(1u << abuf)) | (aphase << abuf);
            if (++abuf == C::HALO_BUFS) {
              abuf = 0;
              aphase ^= 1u;
            }
            for (int tap = 0; tap < p.taps; ++tap) {
              if (!wait(&empty[stage], phase ^ 1u)) {
                raise_error(p, abort);
                failed = true;
                break;
              }
              if (leader) mbar_arrive_expect_tx(&full[stage], tx_mult * STAGE_TX);
              if constexpr (PAIR)
                tma_load_2d_pair(sB + stage * C::B_BYTES, &tmB, full_c + stage * 8,
                                 tap * p.cin_pad + cc * 32, n0);
              else
                tma_load_2d(sB + stage * C::B_BYTES, &tmB, &full[stage],
                            tap * p.cin_pad + cc * 32, n0);
              pending |= 1u << stage;
              pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
          continue;
        }
        if constexpr (MODE == 4) {
          // Per 32-channel chunk and kx: one band of bh + 2 rows shifted by
          // kx - 1 serves the three ky taps; then the shortcut chunks, their
          // plain tiles SC_PER_BUF to an A buffer.
          const int chunks = p.cin_chunks + (p.sc_chunks + C::SC_PER_BUF - 1) / C::SC_PER_BUF;
          for (int cc = 0; cc < chunks && !failed; ++cc) {
            const bool is_sc = cc >= p.cin_chunks;
            const int sc0 = (cc - p.cin_chunks) * C::SC_PER_BUF;
            const int nsc = is_sc ? min(C::SC_PER_BUF, p.sc_chunks - sc0) : 0;
            const int nkx = is_sc ? 1 : 3;
            for (int kx = 0; kx < nkx && !failed; ++kx) {
              if (!mbar_wait(&a_empty[abuf], aphase ^ 1u, abort, p.wait_ns)) {
                raise_error(p, abort);
                failed = true;
                break;
              }
              uint8_t *a_dst = sH + abuf * C::HALO_BYTES;
              if (!is_sc) {
                mbar_arrive_expect_tx(&a_full[abuf], (p.bh + 2) * p.bw * 128);
                tma_load_4d(a_dst, &tmA, &a_full[abuf], cc * 32, tx * p.bw + kx - 1,
                            ty * p.bh - 1, img);
              } else {
                mbar_arrive_expect_tx(&a_full[abuf], nsc * p.bh * p.bw * 128);
                for (int i = 0; i < nsc; ++i)
                  tma_load_4d(a_dst + i * p.bh * p.bw * 128, &tmS, &a_full[abuf], (sc0 + i) * 32,
                              tx * p.bw, ty * p.bh, img);
              }
              a_pending |= 1u << abuf;
              a_par = (a_par & ~(1u << abuf)) | (aphase << abuf);
              if (++abuf == C::HALO_BUFS) {
                abuf = 0;
                aphase ^= 1u;
              }
              const int nky = is_sc ? nsc : 3;
              for (int ky = 0; ky < nky; ++ky) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort, p.wait_ns)) {
                  raise_error(p, abort);
                  failed = true;
                  break;
                }
                const int kcol = is_sc ? p.taps * p.cin_pad + (sc0 + ky) * 32
                                       : (ky * 3 + kx) * p.cin_pad + cc * 32;
                mbar_arrive_expect_tx(&full[stage], STAGE_TX);
                tma_load_2d(sB + stage * C::B_BYTES, &tmB, &full[stage], kcol, n0);
                pending |= 1u << stage;
                pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) {
                  stage = 0;
                  phase ^= 1u;
                }
              }
            }
          }
          continue;
        }
        // One A box and one weight box per reduction step; under PAIR both
        // complete on the leader's barrier.
        auto load_a = [&](uint8_t *dst, const CUtensorMap *m, int stg, int c0, int c1, int c2,
                          int c3) {
          if constexpr (PAIR)
            tma_load_4d_pair(dst, m, full_c + stg * 8, c0, c1, c2, c3);
          else
            tma_load_4d(dst, m, &full[stg], c0, c1, c2, c3);
        };
        auto load_b = [&](uint8_t *dst, int stg, int c0, int c1) {
          if constexpr (PAIR)
            tma_load_2d_pair(dst, &tmB, full_c + stg * 8, c0, c1);
          else
            tma_load_2d(dst, &tmB, &full[stg], c0, c1);
        };
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!wait(&empty[stage], phase ^ 1u)) {
            raise_error(p, abort);
            failed = true;
            break;
          }
          uint8_t *a_dst = sA + stage * C::A_BYTES;
          uint8_t *b_dst = sB + stage * C::B_BYTES;
          if (leader) mbar_arrive_expect_tx(&full[stage], tx_mult * STAGE_TX);
          if (MODE == 0) {
            const int main_steps = p.taps * p.cin_chunks;
            if (ks < main_steps) {
              const int tap = ks / p.cin_chunks, cc = ks % p.cin_chunks;
              const int kk = p.k * p.k;
              const int ktap = tap / kk, sp = tap % kk;
              const int dy = sp / p.k - p.k / 2, dx = sp % p.k - p.k / 2;
              int ft = t_idx + ktap - (p.kt - 1);
              ft = ft < 0 ? 0 : ft;  // causal padding repeats the first frame
              load_a(a_dst, &tmA, stage, cc * 32, tx * p.bw + dx, ty * p.bh + yoff + dy,
                     n_idx * p.t + ft);
              load_b(b_dst, stage, tap * p.cin_pad + cc * 32, n0);
            } else {
              const int cc = ks - main_steps;
              load_a(a_dst, &tmS, stage, cc * 32, tx * p.bw, ty * p.bh + yoff, img);
              load_b(b_dst, stage, p.taps * p.cin_pad + cc * 32, n0);
            }
          } else if (MODE == 1) {
            // 2x2 tap (a, b) of parity (py, px) reads the low-res tile shifted
            // by (py - 1 + a, px - 1 + b); weights of that parity's kernel.
            const int tap = ks / p.cin_chunks, cc = ks % p.cin_chunks;
            load_a(a_dst, &tmA, stage, cc * 32, tx * p.bw + (par & 1) - 1 + (tap & 1),
                   ty * p.bh + yoff + (par >> 1) - 1 + (tap >> 1), img);
            load_b(b_dst, stage, tap * p.cin_pad + cc * 32, par * p.cout + n0);
          } else {
            // (a paired CTA loads its own 128 of the tile's rows)
            const int arow = mt * C::ROWS * kBM + static_cast<int>(rank) * kBM;
            if constexpr (XF == 2) {  // A lands on this CTA's own barrier
              mbar_arrive_expect_tx(&xa_full[stage], C::A_LOAD);
              tma_load_2d(a_dst, &tmA, &xa_full[stage], ks * 32, arow);
              x_pending |= 1u << stage;
              x_par = (x_par & ~(1u << stage)) | (phase << stage);
            } else if constexpr (PAIR) {
              tma_load_2d_pair(a_dst, &tmA, full_c + stage * 8, ks * 32, arow);
            } else {
              tma_load_2d(a_dst, &tmA, &full[stage], ks * 32, arow);
            }
            load_b(b_dst, stage, ks * 32, n0);
          }
          pending |= 1u << stage;
          pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort) {
        // Let every copy issued land before the CTA exits (under PAIR the
        // leader's barriers count both CTAs' copies; the peer leaves only
        // after the closing cluster barrier, i.e. after this drain). Copies
        // onto this CTA's own barriers (XF) are drained by each CTA.
        if (leader) {
          for (int s = 0; s < STAGES; ++s)
            if (pending & (1u << s)) mbar_wait_drain(&full[s], (pend_par >> s) & 1u, p.wait_ns);
          if (XF != 1)
            for (int b = 0; b < C::HALO_BUFS; ++b)
              if (a_pending & (1u << b))
                mbar_wait_drain(&a_full[b], (a_par >> b) & 1u, p.wait_ns);
        }
        if (XF == 1)
          for (int b = 0; b < 2; ++b)
            if (a_pending & (1u << b)) mbar_wait_drain(&h_full[b], (a_par >> b) & 1u, p.wait_ns);
        if (XF == 2)
          for (int s = 0; s < STAGES; ++s)
            if (x_pending & (1u << s)) mbar_wait_drain(&xa_full[s], (x_par >> s) & 1u, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (PAIR: the leader issues the paired MMAs; its commits arrive on the
    // barrier at the same offset in both CTAs.)
    auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
      if constexpr (PAIR)
        umma_tf32_pair(d, a, b, IDESC, acc);
      else
        umma_tf32(d, a, b, IDESC, acc);
    };
    auto commit = [&](uint64_t *bar) {
      if constexpr (PAIR)
        umma_commit_pair(bar, 0x3);
      else
        umma_commit(bar);
    };
    if (lane == 0 && leader) {
      uint32_t stage = 0, phase = 0;
      uint32_t abuf = 0, aphase = 0;
      int local = 0;
      bool failed = false, issued = false;
      WorkIter<MODE> it(p, wid, wcount);
      Work w;
      while (!failed && it.next(p, w)) {
        const int cur = local++;
        const int buf = cur & 1;
        const uint32_t aph = (cur >> 1) & 1;
        if (!wait(&acc_empty[buf], aph ^ 1u)) {
          raise_error(p, abort);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * C::ACC_COLS;
        const int ks0 = w.k0, ks1 = w.k1;
        if constexpr (MODE == 3) {
          // Tap (ky, kx) of output sub-tile `sub` reads the 128 halo pixels
          // starting at halo row sub + ky, column kx: a row offset into the
          // swizzled halo buffer.
          for (int cc = ks0; cc < ks1 && !failed; ++cc) {
            if (!wait(&a_full[abuf], aphase)) {
              raise_error(p, abort);
              failed = true;
              break;
            }
            // The nine views differ from the buffer's descriptor only in the
            // start-address field (row * 128 bytes >> 4; no carry: shared
            // addresses stay below 256 KB), so they are compile-time offsets.
            // Under PAIR each CTA's halo buffer holds its own row's halo at the
            // same offset, so one descriptor serves both.
            const uint64_t hdesc = sw128_kmajor_desc(smem_u32(sH + abuf * C::HALO_BYTES));
            const bool acc0 = cc != ks0;
            issued = true;
#pragma unroll
            for (int tap = 0; tap < 9; ++tap) {
              if (!wait(&full[stage], phase)) {
                raise_error(p, abort);
                failed = true;
                break;
              }
              tc_fence_after();
              const uint64_t bd = sw128_kmajor_desc(sB_u32 + stage * C::B_BYTES);
#pragma unroll
              for (int sub = 0; sub < MS; ++sub) {
                const uint64_t ad =
                    hdesc + static_cast<uint64_t>(((sub + tap / 3) * 130 + tap % 3) * 8);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  mma(d_tmem + sub * BN, ad + 2 * k, bd + 2 * k, acc0 || (tap != 0) || (k != 0));
              }
              commit(&empty[stage]);
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (failed) break;
            commit(&a_empty[abuf]);
            if (++abuf == C::HALO_BUFS) {
              abuf = 0;
              aphase ^= 1u;
            }
          }
          if (!failed) commit(&acc_full[buf]);
          continue;
        }
        if constexpr (MODE == 4) {
          // D[channel][pixel] += W[channel][k] . X[pixel][k]: the weight
          // stage is the 128-row M operand, the pixel band the 256-row N
          // operand, viewed from row ky * bw.
          const int chunks = p.cin_chunks + (p.sc_chunks + C::SC_PER_BUF - 1) / C::SC_PER_BUF;
          bool first = true;
          for (int cc = 0; cc < chunks && !failed; ++cc) {
            const bool is_sc = cc >= p.cin_chunks;
            const int nsc =
                is_sc ? min(C::SC_PER_BUF, p.sc_chunks - (cc - p.cin_chunks) * C::SC_PER_BUF) : 0;
            const int nkx = is_sc ? 1 : 3;
            for (int kx = 0; kx < nkx && !failed; ++kx) {
              if (!mbar_wait(&a_full[abuf], aphase, abort, p.wait_ns)) {
                raise_error(p, abort);
                failed = true;
                break;
              }
              const uint32_t abase = smem_u32(sH + abuf * C::HALO_BYTES);
              const int nky = is_sc ? nsc : 3;
              for (int ky = 0; ky < nky; ++ky) {
                if (!mbar_wait(&full[stage], phase, abort, p.wait_ns)) {
                  raise_error(p, abort);
                  failed = true;
                  break;
                }
                tc_fence_after();
                const uint64_t wd = sw128_kmajor_desc(smem_u32(sB + stage * C::B_BYTES));
                // band view from row ky * bw, or the ky-th shortcut tile
                const uint64_t xd = sw128_kmajor_desc_row(abase, ky * (is_sc ? p.bh * p.bw : p.bw));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  umma_tf32(d_tmem, wd + 2 * k, xd + 2 * k, IDESC_SWAP, !first || (k != 0));
                first = false;
                issued = true;
                umma_commit(&empty[stage]);
                if (++stage == STAGES) {
                  stage = 0;
                  phase ^= 1u;
                }
              }
              if (failed) break;
              umma_commit(&a_empty[abuf]);
              if (++abuf == C::HALO_BUFS) {
                abuf = 0;
                aphase ^= 1u;
              }
            }
          }
          if (!failed) umma_commit(&acc_full[buf]);
          continue;
        }
        for (int ks = ks0; ks < ks1; ++ks) {
          // (XF 2: the weight halves on `full`, the transformed A stages of
          // both CTAs on `xfull`)
          if (!wait(SPLIT ? &xfull[stage] : &full[stage], phase) ||
              (XF == 2 && !wait(&xfull[stage], phase))) {
            raise_error(p, abort);
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t bd = sw128_kmajor_desc(smem_u32(sB + stage * C::B_BYTES));
          // SPLIT: the lo parts sit right after the hi parts (whole swizzle atoms)
          const uint64_t bd_lo = sw128_kmajor_desc(smem_u32(sB + stage * C::B_BYTES + C::B_LOAD));
#pragma unroll
          for (int sub = 0; sub < MS; ++sub) {
            const uint64_t ad =
                sw128_kmajor_desc(smem_u32(sA + stage * C::A_BYTES + sub * kABytes));
            const uint64_t ad_lo =
                sw128_kmajor_desc(smem_u32(sA + stage * C::A_BYTES + C::A_LOAD + sub * kABytes));
#pragma unroll
            for (int k = 0; k < 4; ++k) {  // 4 x K=8 TF32 steps = 32 channels (128 bytes)
              mma(d_tmem + sub * BN, ad + 2 * k, bd + 2 * k, (ks != ks0) || (k != 0));
              if (SPLIT) {
                mma(d_tmem + sub * BN, ad_lo + 2 * k, bd + 2 * k, 1u);
                mma(d_tmem + sub * BN, ad + 2 * k, bd_lo + 2 * k, 1u);
              }
            }
          }
          issued = true;
          commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!failed) commit(&acc_full[buf]);
      }
      if (*abort && issued) {
        // Wait for the MMAs still reading shared memory / writing TMEM before
        // the CTA frees TMEM and exits.
        if constexpr (PAIR)
          umma_commit_pair(drain, 0x1);
        else
          umma_commit(drain);
        mbar_wait_drain(drain, 0, p.wait_ns);
      }
    }
  } else if (!(SPLIT || XF) || warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int ew = warp - 2;  // epilogue warp index
    // with eight epilogue warps, warp ew takes column half ew / 4 of the tile
    constexpr int kHalves = C::EPW / 4;
    const int half = ew >> 2;
    const int m = q * 32 + lane;
    float *stg = staging + ew * C::NSTG * 1024;  // this warp's 4 KB staging buffer(s)
    int sbuf = 0;
    uint32_t res_phase = 0;    // bit b: phase of this warp's residual barrier b
    uint32_t res_pending = 0;  // bit b: a residual load into buffer b not yet waited for
    bool failed = false;
    int local = 0;
    // PAIR: this CTA's accumulator rows are sub-tile `rank` of the pair's
    // tile, at TMEM column 0 of the buffer; the leader's MMA issuer waits for
    // the epilogue warps of both CTAs.
    const uint32_t acc_empty_c = PAIR ? mapa_rank(acc_empty, 0) : 0u;
    WorkIter<MODE> it(p, wid, wcount);
    Work w;
    while (!failed && it.next(p, w)) {
      const int tile = w.tile;
      const int cur = local++;
      const int buf = cur & 1;
      const uint32_t aph = (cur >> 1) & 1;
      bool ok = wait(&acc_full[buf], aph);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) raise_error(p, abort);
        break;
      }
      tc_fence_after();

      const int mn = tile % (p.m_tiles * p.n_tiles);
      const int split = tile / (p.m_tiles * p.n_tiles);
      const int mt = mn / p.n_tiles;
      const int n0 = (mn % p.n_tiles) * BN;
      float *const obase = p.out + split * p.split_stride;
      if constexpr (MODE == 4) {
        // Accumulator lanes are output channels, columns pixels: each lane
        // owns one channel and reads 32 pixels at a time, transposing into
        // the pixel-major staging block on its way to the TMA store.
        const int per_img = p.tiles_x * p.tiles_y;
        const int img = mt / per_img;
        const int rem = mt % per_img;
        const int ty = rem / p.tiles_x, tx = rem % p.tiles_x;
        const int c0 = n0 + q * 32;  // this warp's first channel (warp-uniform)
        const int ch = c0 + lane;
        const bool ch_ok = ch < p.cout;
        const float bch = (p.bias && ch_ok) ? __ldg(p.bias + ch) : 0.f;
        const int lbw = __ffs(p.bw) - 1;  // bw is a power of two
        // In-image mask of a 32-pixel chunk: lane j tests pixel j.
        auto chunk_mask = [&](int mp0) -> uint32_t {
          const int py = ty * p.bh + ((mp0 + lane) >> lbw);
          const int px = tx * p.bw + ((mp0 + lane) & (p.bw - 1));
          return __ballot_sync(0xffffffffu, py < p.hout && px < p.wout);
        };
        // Residual of a chunk: for pixel j the 32 lanes read 32 adjacent
        // channels (one 128-byte line), so plain loads are coalesced; they
        // are issued one chunk ahead of their use.
        const float *rcol = (p.has_res && ch_ok)
                                ? p.residual + static_cast<long long>(img) * p.hout * p.wout * p.ldo + ch
                                : nullptr;
        auto load_res = [&](int mp0, uint32_t mask, float(&dst)[32]) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int y = ty * p.bh + ((mp0 + j) >> lbw);
            const int x = tx * p.bw + ((mp0 + j) & (p.bw - 1));
            dst[j] = (rcol && ((mask >> j) & 1u))
                         ? __ldcg(rcol + (static_cast<long long>(y) * p.wout + x) * p.ldo)
                         : 0.f;
          }
        };
        float rnext[32], rcur[32];
        // this warp's 32-pixel chunks of the tile's 256
        const int pc0 = half * (8 / kHalves), pc1 = pc0 + 8 / kHalves;
        uint32_t mnext = chunk_mask(pc0 * 32);
        if (p.has_res) load_res(pc0 * 32, mnext, rnext);
        for (int pc = pc0; pc < pc1 && c0 < p.cout; ++pc) {
          const uint32_t vmask = mnext;
#pragma unroll
          for (int j = 0; j < 32; ++j) rcur[j] = rnext[j];
          if (pc + 1 < pc1) {
            mnext = chunk_mask((pc + 1) * 32);
            if (p.has_res) load_res((pc + 1) * 32, mnext, rnext);
          }
          float v[32];
          tmem_ld_32cols(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(buf * C::ACC_COLS + pc * 32),
                         v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = fmaf(v[j], p.alpha, bch);
          const int mp0 = pc * 32;  // first pixel of the chunk within the tile
          const int bx = tx * p.bw + (mp0 & (p.bw - 1)), by = ty * p.bh + (mp0 >> lbw);
          float *sb = stg + sbuf * 1024;
          if (lane == 0) bulk_wait_read<C::NSTG - 1>();  // the store that used sb last is done
          __syncwarp();
          // Pixel j is row j of the block, this lane's channel its column;
          // the 128-byte swizzle puts 16-byte chunk (lane / 4) at
          // (lane / 4) ^ (j % 8), so each row's 32 stores hit 32 banks.
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int idx = j * 32 + ((((lane >> 2) ^ (j & 7)) << 2) | (lane & 3));
            float val = p.has_res ? v[j] + rcur[j] : v[j];
            if (p.round_out) val = round_tf32(val);
            sb[idx] = val;
            v[j] = val;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(&tmO, sb, c0, bx, by, img);
            bulk_commit();
          }
          if (C::NSTG == 2) sbuf ^= 1;
          if (p.stat_part) {
            // (count, mean, M2) of each group (stat_cg adjacent lanes) over
            // the chunk's in-image pixels; slot = (frame, tile, chunk).
            const int nv = __popc(vmask);
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) sum += ((vmask >> j) & 1u) ? v[j] : 0.f;
            for (int o = 1; o < p.stat_cg; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            const float cnt = static_cast<float>(nv * p.stat_cg);
            const float mean = cnt > 0.f ? __fdividef(sum, cnt) : 0.f;
            float m2 = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float d = v[j] - mean;
              m2 = ((vmask >> j) & 1u) ? fmaf(d, d, m2) : m2;
            }
            for (int o = 1; o < p.stat_cg; o <<= 1) m2 += __shfl_xor_sync(0xffffffffu, m2, o);
            if (ch_ok && (lane & (p.stat_cg - 1)) == 0) {
              const long long slot =
                  (static_cast<long long>(img % p.t) * per_img + rem) * 8 + pc;
              float *o = p.stat_part +
                         ((static_cast<long long>(img / p.t) * p.stat_groups + ch / p.stat_cg) *
                              p.stat_slots + slot) * 3;
              o[0] = cnt;
              o[1] = mean;
              o[2] = m2;
            }
          }
        }
        if (failed) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        continue;
      }
      // Stream-K: this warp's rows of a tile split with the next CTA. The
      // tail's raw sums are in that CTA's slot once its flag for this warp
      // is up (set long before: the tail was its first work item).
      const size_t sk_slot_f4 = static_cast<size_t>(MS) * BN * 32;  // float4 per slot
      if (w.head) {
        bool ok = true;
        if (lane == 0) {
          const int *f = p.sk_flag + (blockIdx.x + C::NCTA) * 4 + q;
          const uint64_t t0 = global_timer_ns();
          while (ld_acquire_gpu(f) == 0) {
            if (*abort || global_timer_ns() - t0 > p.wait_ns) {
              ok = false;
              break;
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) {
          if (lane == 0) raise_error(p, abort);
          failed = true;
          break;
        }
        __syncwarp();
        __threadfence();
      }
      for (int sub = 0; sub < MS; ++sub) {
      // 128-row sub-tile of the (pair) tile this warp's rows belong to
      const int sg = PAIR ? static_cast<int>(rank) : sub;
      const int msub = sg * 128 + m;  // row of the (ROWS x 128)-row tile
      bool valid;
      long long row;          // NHWC / GEMM row index
      long long nchw0 = 0;    // NCHW: offset of channel 0 for this pixel
      long long cstride = 0;  // NCHW: distance between channels
      int bc1 = 0, bc2 = 0, bc3 = 0, bc4 = 0;  // this warp's TMA box coordinates
      if (MODE == 2) {
        row = static_cast<long long>(mt) * C::ROWS * kBM + msub;
        valid = row < p.M;
        bc1 = mt * C::ROWS * kBM + sg * kBM + q * 32;
      } else {
        const int per_img = p.tiles_x * p.tiles_y * (MODE == 1 ? 4 : 1);
        const int img = mt / per_img;
        int rem = mt % per_img;
        const int par = MODE == 1 ? (rem & 3) : 0;
        if (MODE == 1) rem >>= 2;
        const int ty = rem / p.tiles_x, tx = rem % p.tiles_x;
        int y, x;
        if (kConv) {
          y = ty * p.bh + msub / p.bw;
          x = tx * p.bw + msub % p.bw;
          valid = y < p.hout && x < p.wout;
          bc1 = tx * p.bw + (sg * 128 + q * 32) % p.bw;
          bc2 = ty * p.bh + (sg * 128 + q * 32) / p.bw;
          bc3 = img;
        } else {
          // rows are low-res pixels of the tile; all share the parity par
          const int yl = ty * p.bh + msub / p.bw, xl = tx * p.bw + msub % p.bw;
          y = 2 * yl + (par >> 1);
          x = 2 * xl + (par & 1);
          valid = yl < p.hin && xl < p.win;
          const int r0 = sg * 128 + q * 32;  // this warp's first row
          bc1 = par & 1;                      // px
          bc2 = tx * p.bw + r0 % p.bw;        // xl
          bc3 = par >> 1;                     // py
          bc4 = img * p.hin + ty * p.bh + r0 / p.bw;
        }
        row = (static_cast<long long>(img) * p.hout + y) * p.wout + x;
        const long long hw = static_cast<long long>(p.hout) * p.wout;
        const int n_idx = img / p.t, t_idx = img % p.t;
        cstride = hw * p.t;
        nchw0 = static_cast<long long>(n_idx) * p.cout * cstride + t_idx * hw +
                static_cast<long long>(y) * p.wout + x;
      }
      const float rbias = (MODE == 2 && p.bias_per_row && p.bias && valid) ? p.bias[row] : 0.f;
      float rs_m = -INFINITY, rs_s = 0.f;  // softmax statistics of this row (rs_out)

      constexpr int kChunks = BN / C::CH;  // column chunks of the tile
      const int cb = half * (kChunks / kHalves), ce = cb + kChunks / kHalves;
#pragma unroll 1
      for (int c = cb; c < ce; ++c) {
        float v[C::CH];
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
            static_cast<uint32_t>(buf * C::ACC_COLS + sub * BN + c * C::CH);
        if (C::CH == 32)
          tmem_ld_32cols(taddr, v);
        else
          tmem_ld_16cols(taddr, v);
        if (C::CH == 32 && (w.tail || w.head)) {
          // slot layout [sub][chunk][j][128 rows] of float4: a warp's 32
          // lanes touch 32 consecutive float4 per access
          const size_t off = static_cast<size_t>((sub * (BN / 32) + c) * 8) * 128 + q * 32 + lane;
          if (w.tail) {
            float4 *dst = reinterpret_cast<float4 *>(p.sk_part) + blockIdx.x * sk_slot_f4 + off;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              __stcg(dst + j * 128, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
            continue;
          }
          const float4 *src =
              reinterpret_cast<const float4 *>(p.sk_part) + (blockIdx.x + C::NCTA) * sk_slot_f4 + off;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 t = __ldcg(src + j * 128);
            v[4 * j] += t.x;
            v[4 * j + 1] += t.y;
            v[4 * j + 2] += t.z;
            v[4 * j + 3] += t.w;
          }
        }
        const int col0 = n0 + c * C::CH;
        if (col0 >= p.cout) continue;  // warp-uniform
        const int ncols = min(C::CH, p.cout - col0);
        // bias + scale (vector loads when the whole chunk is in range)
        if (!p.bias_per_row && p.bias && ncols == C::CH) {
#pragma unroll
          for (int i = 0; i < C::CH; i += 4) {
            const float4 b4 = __ldg(reinterpret_cast<const float4 *>(p.bias + col0 + i));
            v[i] = fmaf(v[i], p.alpha, b4.x);
            v[i + 1] = fmaf(v[i + 1], p.alpha, b4.y);
            v[i + 2] = fmaf(v[i + 2], p.alpha, b4.z);
            v[i + 3] = fmaf(v[i + 3], p.alpha, b4.w);
          }
        } else {
#pragma unroll
          for (int i = 0; i < C::CH; ++i) {
            float b = rbias;
            if (!p.bias_per_row && p.bias && i < ncols) b = __ldg(p.bias + col0 + i);
            v[i] = fmaf(v[i], p.alpha, b);
          }
        }
        if (MODE == 2 && p.rs_out) {
          // running (max, sum of exp) of v * rs_scale over the valid columns
          float mc = -INFINITY;
#pragma unroll
          for (int i = 0; i < C::CH; ++i)
            if (col0 + i < p.rs_cols) mc = fmaxf(mc, v[i] * p.rs_scale);
          if (mc != -INFINITY) {
            float sc = 0.f;
#pragma unroll
            for (int i = 0; i < C::CH; ++i)
              if (col0 + i < p.rs_cols) sc += __expf(v[i] * p.rs_scale - mc);
            if (mc > rs_m) {
              rs_s = rs_s * __expf(rs_m - mc) + sc;
              rs_m = mc;
            } else {
              rs_s += sc * __expf(mc - rs_m);
            }
          }
        }
        if (C::CH == 32 && p.epi_tma) {
          // Stage the warp's 32 x 32 block in the 128-byte-swizzled layout the
          // TMA store reads (row r, 16-byte chunk j at j ^ (r % 8)); rows and
          // channels outside the tensor are clipped by the store.
          float *sb = stg + sbuf * 1024;
          // The residual block of channels from c0 lands in staging buffer b
          // (its 4 KB box, clipped rows and channels read as zero).
          auto load_res = [&](int b, int c0) {
            uint64_t *bar = &res_bar[ew * 2 + b];
            mbar_arrive_expect_tx(bar, 4096);
            float *dst = stg + b * 1024;
            if (MODE == 2)
              tma_load_2d(dst, &tmR, bar, c0, bc1);
            else if (kConv)
              tma_load_4d(dst, &tmR, bar, c0, bc1, bc2, bc3);
            else
              tma_load_5d(dst, &tmR, bar, c0, bc1, bc2, bc3, bc4);
          };
          if (p.has_res) {
            // With two buffers the next block's residual is requested before
            // this one is processed, so its latency overlaps this block.
            if (lane == 0) {
              if (!(res_pending & (1u << sbuf))) {  // first block of the row range
                bulk_wait_read<0>();
                load_res(sbuf, col0);
              }
              if (C::NSTG == 2 && c + 1 < ce && col0 + C::CH < p.cout) {
                bulk_wait_read<0>();  // the store from the other buffer has read it
                load_res(sbuf ^ 1, col0 + C::CH);
              }
            }
            res_pending |= 1u << sbuf;
            if (C::NSTG == 2 && c + 1 < ce && col0 + C::CH < p.cout)
              res_pending |= 1u << (sbuf ^ 1);
            __syncwarp();
            bool rok = mbar_wait(&res_bar[ew * 2 + sbuf], (res_phase >> sbuf) & 1u, abort,
                                 p.wait_ns);
            rok = __all_sync(0xffffffffu, rok);
            res_phase ^= 1u << sbuf;
            res_pending &= ~(1u << sbuf);
            if (!rok) {
              if (lane == 0) raise_error(p, abort);
              failed = true;
              break;
            }
          } else {
            if (lane == 0) bulk_wait_read<C::NSTG - 1>();  // the store that used sb last is done
            __syncwarp();
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float4 *slot = reinterpret_cast<float4 *>(sb + lane * 32 + ((j ^ (lane & 7)) * 4));
            float4 val = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            if (p.has_res) {
              const float4 rv = *slot;
              val.x += rv.x;
              val.y += rv.y;
              val.z += rv.z;
              val.w += rv.w;
            }
            if (p.round_out) {
              val.x = round_tf32(val.x);
              val.y = round_tf32(val.y);
              val.z = round_tf32(val.z);
              val.w = round_tf32(val.w);
            }
            *slot = val;
            v[4 * j] = val.x;  // keep the stored values for the statistics
            v[4 * j + 1] = val.y;
            v[4 * j + 2] = val.z;
            v[4 * j + 3] = val.w;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (MODE == 2)
              tma_store_2d(&tmO, sb, col0, bc1);
            else if (kConv)
              tma_store_4d(&tmO, sb, col0, bc1, bc2, bc3);
            else
              tma_store_5d(&tmO, sb, col0, bc1, bc2, bc3, bc4);
            bulk_commit();
          }
          if (C::NSTG == 2) sbuf ^= 1;
          if (MODE != 2 && p.stat_part) {
            const int per_img = p.tiles_x * p.tiles_y * (MODE == 1 ? 4 : 1);
            const int img = mt / per_img;
            const long long slot =
                ((static_cast<long long>(img % p.t) * per_img + mt % per_img) * C::ROWS + sg) * 4 +
                q;
            const int gbase = col0 / p.stat_cg;
            float *out = p.stat_part +
                         ((static_cast<long long>(img / p.t) * p.stat_groups + gbase) *
                              p.stat_slots + slot) * 3;
            const long long gs = static_cast<long long>(p.stat_slots) * 3;
            const float nrows = static_cast<float>(__popc(__ballot_sync(0xffffffffu, valid)));
            switch (p.stat_cg) {
              case 1: emit_group_stats<1>(v, valid, nrows, out, gs, lane); break;
              case 2: emit_group_stats<2>(v, valid, nrows, out, gs, lane); break;
              case 4: emit_group_stats<4>(v, valid, nrows, out, gs, lane); break;
              case 8: emit_group_stats<8>(v, valid, nrows, out, gs, lane); break;
              case 16: emit_group_stats<16>(v, valid, nrows, out, gs, lane); break;
              default: emit_group_stats<32>(v, valid, nrows, out, gs, lane); break;
            }
          }
          continue;
        }
        if (!valid) continue;
        if (p.out_nchw) {
          float *o = obase + nchw0 + static_cast<long long>(col0) * cstride;
          const float *r = p.residual ? p.residual + nchw0 + static_cast<long long>(col0) * cstride
                                      : nullptr;
#pragma unroll
          for (int i = 0; i < C::CH; ++i) {
            if (i < ncols) {
              float val = v[i];
              if (r) val += r[i * cstride];
              if (p.round_out) val = round_tf32(val);
              o[i * cstride] = val;
            }
          }
        } else {
          float *o = obase + row * p.ldo + col0;
          const float *r = p.residual ? p.residual + row * p.ldo + col0 : nullptr;
          if (ncols == C::CH) {
#pragma unroll
            for (int i = 0; i < C::CH; i += 4) {
              float4 val = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
              if (r) {
                const float4 rv = *reinterpret_cast<const float4 *>(r + i);
                val.x += rv.x;
                val.y += rv.y;
                val.z += rv.z;
                val.w += rv.w;
              }
              if (p.round_out) {
                val.x = round_tf32(val.x);
                val.y = round_tf32(val.y);
                val.z = round_tf32(val.z);
                val.w = round_tf32(val.w);
              }
              *reinterpret_cast<float4 *>(o + i) = val;
            }
          } else {
#pragma unroll
            for (int i = 0; i < C::CH; ++i) {
              if (i < ncols) {
                float val = v[i];
                if (r) val += r[i];
                if (p.round_out) val = round_tf32(val);
                o[i] = val;
              }
            }
          }
        }
      }
      if (failed) break;
      if (MODE == 2 && p.rs_out && valid)
        p.rs_out[row * p.rs_ld + mn % p.n_tiles] = make_float2(rs_m, rs_s);
      }  // sub-tiles
      if (w.tail && !failed) {  // this warp's raw sums are out: raise its flag
        __threadfence();
        __syncwarp();
        // (The test hook withholds the flag so that the head's bounded wait
        // runs out; nothing else differs.)
        if (lane == 0 && !(p.inject & VAE_INJECT_WITHHOLD_STREAMK_FLAG))
          st_release_gpu(p.sk_flag + blockIdx.x * 4 + q, 1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !failed) {
        if (!PAIR || leader)
          mbar_arrive(&acc_empty[buf]);
        else
          mbar_arrive_cluster(acc_empty_c + buf * 8);
      }
    }
    // Every TMA store of this warp must finish reading shared memory (and
    // land), and a residual load still in flight after an abort must land,
    // before the CTA exits.
    if (lane == 0 && p.epi_tma) bulk_wait_all();
    for (int b = 0; b < 2; ++b)
      if (lane == 0 && (res_pending & (1u << b)))
        mbar_wait_drain(&res_bar[ew * 2 + b], (res_phase >> b) & 1u, p.wait_ns);
  } else if constexpr (SPLIT) {
    // ------------------------------------------------------------ split (SPLIT)
    // Each landed stage, in place: v -> hi = tf32(v), and lo = tf32(v - hi)
    // at the same offset in the lo half. The stage's parts then reach the
    // tensor core through the async proxy.
    const int tt = threadIdx.x - kThreads;  // 0..127
    uint32_t stage = 0, phase = 0;
    bool failed = false;
    auto split = [&](uint8_t *base, uint32_t bytes) {
      float4 *hi = reinterpret_cast<float4 *>(base);
      float4 *lo = reinterpret_cast<float4 *>(base + bytes);
      for (uint32_t i = tt; i < bytes / 16; i += 128) {
        const float4 v = hi[i];
        float4 h, l;
        h.x = round_tf32(v.x);
        h.y = round_tf32(v.y);
        h.z = round_tf32(v.z);
        h.w = round_tf32(v.w);
        l.x = round_tf32(v.x - h.x);
        l.y = round_tf32(v.y - h.y);
        l.z = round_tf32(v.z - h.z);
        l.w = round_tf32(v.w - h.w);
        hi[i] = h;
        lo[i] = l;
      }
    };
    WorkIter<MODE> it(p, wid, wcount);
    Work w;
    while (!failed && it.next(p, w)) {
      for (int ks = w.k0; ks < w.k1; ++ks) {
        bool ok = mbar_wait(&full[stage], phase, abort, p.wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) raise_error(p, abort);
          failed = true;
          break;
        }
        split(sA + stage * C::A_BYTES, C::A_LOAD);
        split(sB + stage * C::B_BYTES, C::B_LOAD);
        fence_proxy_async_smem();
        mbar_arrive(&xfull[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if constexpr (XF == 1) {
    // ------------------------------------------------------------ GroupNorm (XF 1)
    // Each landed halo buffer, in place: v -> silu(v * scale[c] + shift[c])
    // (the same arithmetic as the separate GroupNorm apply), TF32-rounded
    // as an MMA operand; pixels outside the image stay 0 (the conv's zero
    // padding, not silu(shift)). Then the leader's a_full learns that this
    // CTA's buffer is ready. Thread tt touches the 16-byte words tt + 128 j:
    // pixel rows (tt >> 3) + 16 j, always the same 4-channel group (the
    // 128-byte swizzle XORs the word index with the row's low 3 bits, which
    // 16 j leaves alone), so its scale and shift load once per chunk; the
    // words go through in batches of kU for independent loads and math.
    constexpr int kWords = (MS + 2) * 130 * 8;
    constexpr int kU = 5;
    constexpr int kBatches = (kWords + 128 * kU - 1) / (128 * kU);
    const int tt = threadIdx.x - kThreads;  // 0..127
    const int lc = (tt & 7) ^ ((tt >> 3) & 7);
    const uint32_t afull_c = PAIR ? mapa_rank(a_full, 0) : 0u;
    const int yoff = PAIR ? static_cast<int>(rank) * (p.bh >> 1) : 0;
    uint32_t abuf = 0, aphase = 0;
    bool failed = false;
    WorkIter<MODE> it(p, wid, wcount);
    Work w;
    while (!failed && it.next(p, w)) {
      const int mn = w.tile % (p.m_tiles * p.n_tiles);
      const int mt = mn / p.n_tiles;
      const int per_img = p.tiles_x * p.tiles_y;
      const int img = mt / per_img, rem = mt % per_img;
      const int ty = rem / p.tiles_x, tx = rem % p.tiles_x;
      const int y0 = ty * p.bh + yoff - 1, x0 = tx * p.bw - 1;
      const long long ss0 = static_cast<long long>(img / p.t) * p.cin_pad + lc * 4;
      for (int cc = w.k0; cc < w.k1; ++cc) {
        const float4 sa = __ldg(reinterpret_cast<const float4 *>(p.gn_scale + ss0 + cc * 32));
        const float4 sb = __ldg(reinterpret_cast<const float4 *>(p.gn_shift + ss0 + cc * 32));
        bool ok = mbar_wait(&h_full[abuf], aphase, abort, p.wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) raise_error(p, abort);
          failed = true;
          break;
        }
        float4 *buf = reinterpret_cast<float4 *>(sH + abuf * C::HALO_BYTES);
#pragma unroll 1
        for (int bt = 0; bt < kBatches; ++bt) {
          float4 v[kU];
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int i = tt + 128 * (bt * kU + u);
            if (i < kWords) v[u] = buf[i];
          }
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int R = (tt >> 3) + 16 * (bt * kU + u);  // halo pixel
            const int hr = R / 130, hc = R - hr * 130;
            const int y = y0 + hr, x = x0 + hc;
            if (y >= 0 && y < p.hin && x >= 0 && x < p.win) {
              float e[4] = {fmaf(v[u].x, sa.x, sb.x), fmaf(v[u].y, sa.y, sb.y),
                            fmaf(v[u].z, sa.z, sb.z), fmaf(v[u].w, sa.w, sb.w)};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                if (p.gn_silu) e[k] = __fdividef(e[k], 1.0f + __expf(-e[k]));
                e[k] = round_tf32(e[k]);
              }
              v[u] = make_float4(e[0], e[1], e[2], e[3]);
            } else {
              v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int i = tt + 128 * (bt * kU + u);
            if (i < kWords) buf[i] = v[u];
          }
        }
        fence_proxy_async_smem();  // generic writes -> the tensor core's reads
        __syncwarp();
        if (lane == 0) {
          if (!PAIR || leader)
            mbar_arrive(&a_full[abuf]);
          else
            mbar_arrive_cluster(afull_c + abuf * 8);
        }
        if (++abuf == C::HALO_BUFS) {
          abuf = 0;
          aphase ^= 1u;
        }
      }
    }
  } else if constexpr (XF == 2) {
    // ------------------------------------------------------------ softmax (XF 2)
    // Each landed A stage of raw scores, in place: s -> exp(s * scale -
    // m[row]) * inv_l[row] (the row softmax, with the row statistics known),
    // TF32-rounded; keys beyond the valid count read 0. Thread tt touches
    // the 16-byte words tt + 128 j (j < 8): rows (tt >> 3) + 16 j, always
    // the same 4 keys of the stage's 32, so the eight rows' statistics load
    // once per tile.
    const int tt = threadIdx.x - kThreads;  // 0..127
    const int lc = (tt & 7) ^ ((tt >> 3) & 7);
    const uint32_t xfull_c = PAIR ? mapa_rank(xfull, 0) : 0u;
    static_assert(C::A_LOAD / 16 == 8 * 128, "one 128-row stage: eight words per thread");
    uint32_t stage = 0, phase = 0;
    bool failed = false;
    WorkIter<MODE> it(p, wid, wcount);
    Work w;
    while (!failed && it.next(p, w)) {
      const int mn = w.tile % (p.m_tiles * p.n_tiles);
      const int mt = mn / p.n_tiles;
      const int row0 = mt * C::ROWS * kBM + static_cast<int>(rank) * kBM + (tt >> 3);
      float rm[8], ril[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int row = min(row0 + 16 * j, p.M - 1);
        rm[j] = __ldg(p.sm_m + row);
        ril[j] = __ldg(p.sm_inv_l + row);
      }
      for (int ks = w.k0; ks < w.k1; ++ks) {
        bool ok = mbar_wait(&xa_full[stage], phase, abort, p.wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) raise_error(p, abort);
          failed = true;
          break;
        }
        float4 *a = reinterpret_cast<float4 *>(sA + stage * C::A_BYTES);
        const int key = ks * 32 + lc * 4;
        const bool k0 = key < p.sm_cols, k1 = key + 1 < p.sm_cols, k2 = key + 2 < p.sm_cols,
                   k3 = key + 3 < p.sm_cols;
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = a[tt + 128 * j];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[j].x = k0 ? round_tf32(__expf(v[j].x * p.sm_scale - rm[j]) * ril[j]) : 0.f;
          v[j].y = k1 ? round_tf32(__expf(v[j].y * p.sm_scale - rm[j]) * ril[j]) : 0.f;
          v[j].z = k2 ? round_tf32(__expf(v[j].z * p.sm_scale - rm[j]) * ril[j]) : 0.f;
          v[j].w = k3 ? round_tf32(__expf(v[j].w * p.sm_scale - rm[j]) * ril[j]) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) a[tt + 128 * j] = v[j];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (!PAIR || leader)
            mbar_arrive(&xfull[stage]);
          else
            mbar_arrive_cluster(xfull_c + stage * 8);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }

  if constexpr (XF == 3) {
    if (warp >= 6) {
      // ---------------------------------------------------------- GroupNorm ahead (XF 3)
      // Rows in the order the counter hands them out (lowest first, so the
      // first tiles' rows come first): t = tf32(silu(x * scale + shift)),
      // the same arithmetic as the separate GroupNorm apply; then the row's
      // flag. Thread tt keeps channel quad tt % (cin / 4) (128 is a multiple
      // of cin / 4), loading its affine once per row; eight 16-byte loads in
      // flight per thread.
      __shared__ int s_unit;
      constexpr int kU = 8;
      const int tt = threadIdx.x - kThreads;  // 0..127
      const int c4 = p.cin_pad >> 2;
      const int q4 = tt % c4;
      const int units = p.imgs * p.hin;
      const long long row_f4 = static_cast<long long>(p.win) * c4;
      while (true) {
        if (tt == 0) s_unit = *abort ? units : atomicAdd(p.ga_next, 1);
        named_barrier_sync(1, 128);
        const int u = s_unit;
        if (u >= units) break;
        const int sample = (u / p.hin) / p.t;
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p.ga_scale) +
                               static_cast<long long>(sample) * c4 + q4);
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p.ga_shift) +
                               static_cast<long long>(sample) * c4 + q4);
        const float4 *src = reinterpret_cast<const float4 *>(p.ga_x) + u * row_f4;
        float4 *dst = reinterpret_cast<float4 *>(p.ga_t) + u * row_f4;
        for (long long i0 = tt; i0 < row_f4; i0 += 128 * kU) {
          float4 v[kU];
#pragma unroll
          for (int k = 0; k < kU; ++k)
            if (i0 + 128 * k < row_f4) v[k] = __ldg(src + i0 + 128 * k);
#pragma unroll
          for (int k = 0; k < kU; ++k) {
            float e[4] = {fmaf(v[k].x, a.x, b.x), fmaf(v[k].y, a.y, b.y),
                          fmaf(v[k].z, a.z, b.z), fmaf(v[k].w, a.w, b.w)};
#pragma unroll
            for (int j = 0; j < 4; ++j) e[j] = round_tf32(__fdividef(e[j], 1.0f + __expf(-e[j])));
            v[k] = make_float4(e[0], e[1], e[2], e[3]);
          }
#pragma unroll
          for (int k = 0; k < kU; ++k)
            if (i0 + 128 * k < row_f4) dst[i0 + 128 * k] = v[k];
        }
        named_barrier_sync(1, 128);  // every store of the row issued (and s_unit read)
        if (tt == 0) {
          __threadfence();
          st_release_gpu(p.ga_flags + u, p.ga_epoch);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  if constexpr (PAIR) {
    // Neither CTA frees TMEM or leaves while the pair's MMAs, copies or
    // arrivals may still touch it.
    cluster_sync();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
  } else {
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
  }
}

template <int BN, int MODE, int MS, bool PAIR = false, bool SPLIT = false, int XF = 0>
int launch_typed(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ts,
                 const CUtensorMap &to, const CUtensorMap &tr, const KParams &kp,
                 cudaStream_t stream) {
  using C = Cfg<BN, MS, MODE, PAIR, SPLIT, XF>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(igemm_kernel<BN, MODE, MS, PAIR, SPLIT, XF>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(C::SMEM));
  });
  VAE_CUDA_TRY(attr_err);
  // PAIR: one cluster of two CTAs per SM pair, two CTAs per worker.
  const int workers = PAIR ? num_sms() / 2 : num_sms();
  const int grid = std::min(kp.total_tiles, workers) * (PAIR ? 2 : 1);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[1];
  cfg.attrs = attrs;
  cfg.numAttrs = 0;
  if (PAIR) {
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = 2;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
  } else if (kp.sk) {
    // Stream-K CTAs wait on their neighbour's flags: a cooperative launch
    // guarantees that the whole grid is resident.
    attrs[0].id = cudaLaunchAttributeCooperative;
    attrs[0].val.cooperative = 1;
    cfg.numAttrs = 1;
  }
  VAE_CUDA_TRY(
      cudaLaunchKernelEx(&cfg, igemm_kernel<BN, MODE, MS, PAIR, SPLIT, XF>, ta, tb, ts, to, tr, kp));
  VAE_LAUNCH_CHECK();
  count_launches(1);
  return VAE_OK;
}

// Split-TF32 instantiations (igemm_split.cu): MODE 0 (conv), 1 (upsample) or
// 2 (GEMM) at output-channel tile bn.
int launch_split(int mode, int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                 const CUtensorMap &ts, const CUtensorMap &to, const CUtensorMap &tr,
                 const KParams &kp, cudaStream_t s);

// Operand-transform instantiations (igemm_xf.cu): xf 1 (input GroupNorm,
// halo conv), 2 (softmax A, GEMM) or 3 (GroupNorm ahead; mode 3 halo or 4
// channel-major), paired or not where the mode has pairs.
int launch_xf(int xf, int mode, bool pair, const CUtensorMap &ta, const CUtensorMap &tb,
              const CUtensorMap &ts, const CUtensorMap &to, const CUtensorMap &tr,
              const KParams &kp, cudaStream_t s);

}  // namespace igk
}  // namespace vae
