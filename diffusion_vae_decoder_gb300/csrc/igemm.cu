// igemm.cu -- implicit-GEMM convolution and plain GEMM on the tcgen05 tensor
// cores (TF32 operands, FP32 accumulation in TMEM), sm_103a.
//
// The convolution is the decoder's hot path ("VAE decode -> GPU handoff
// (FLUX/LTX render services)", "The CPU VAE code": the late up-block convs at
// full resolution dominate). That page plans an im2col buffer followed by an
// SGEMM ("GPU plan -- im2col + cuBLAS SGEMM", steps 1-2); here the im2col
// matrix is never stored. Output pixels are the GEMM rows, output channels the
// columns, and (tap, input channel) the reduction index. Each reduction step
// is one tap x 32 input channels: a TMA tiled copy of the NHWC activation
// shifted by the tap offset (out-of-range coordinates read as zero, which is
// exactly the zero padding), plus a TMA copy of the packed weights.
//
// CTA layout (192 threads, persistent over output tiles):
//   warp 0     TMA producer (one thread) filling a STAGES-deep smem ring
//   warp 1     TMEM allocator + MMA issuer (one thread)
//   warps 2-5  epilogue: TMEM -> registers, bias / residual / scale, stores
// The accumulator is double-buffered in TMEM so the epilogue of tile i
// overlaps the MMAs of tile i+1.
//
// Operand tiles: 128 rows x 32 f32 (128 bytes per row) with the 128-byte
// swizzle, i.e. the K-major SW128 canonical layout tcgen05 reads directly.
//
// A-operand modes
//   Conv      NHWC input, k x k (x kt causal) taps; the 1x1 resnet shortcut is
//             appended as extra reduction steps over its own input.
//   Upsample  nearest-2x upsample folded into a 3x3 conv (cortiq-engine
//             "Module vae", VaeUpRef). Every output pixel of parity (py, px)
//             sees its 3x3 taps land on only 2 x 2 distinct low-res pixels
//             (tap ky reads low-res row offset floor((py + ky - 1) / 2)), so
//             the layer is four 2x2 convs of the low-res input with summed
//             weights: 4 instead of 9 taps per output pixel. A tile is a
//             block of low-res pixels of one parity; each step is one plain
//             TMA box, and the upsampled tensor is never materialised.
//   Gemm      row-major A [M, K] (token-major activations for attention).
//   Halo      3x3 conv, 256-channel tiles of 128 pixels in one row: per
//             32-channel chunk one 3 x 130-pixel box (the tile's rows with a
//             one-pixel border) is staged once; each tap's A operand is a
//             view starting at row ky * 130 + kx of that swizzled buffer, so
//             the ring stages carry weights only.
//   Channel-major  3x3 conv, 128-channel tiles of 256 pixels: the MMA's M
//             is the 128 output channels (weights as the A operand), N the
//             256 pixels; per 32-channel chunk and kx one band of bh + 2
//             rows serves the three ky taps (views from row ky * bw). The
//             epilogue transposes each 32 x 32 block into pixel-major rows.
//
// Work distribution: whole tiles strided over the persistent CTAs; split-K
// slices when the tiles alone fill few SMs; stream-K ranges (a tile may be
// cut between two neighbouring CTAs, the tail's raw sums handed over through
// a workspace slot and a flag) when whole tiles would leave the last round
// of SMs mostly idle.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "igemm_kernel.cuh"

namespace vae {

using namespace igk;

namespace {

// ---------------------------------------------------------------- host side
int pow2_at_least(int v) {
  int r = 1;
  while (r < v) r <<= 1;
  return r;
}

template <int MODE>
int launch_mode(int bn, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ts,
                const CUtensorMap &to, const CUtensorMap &tr, const KParams &kp,
                cudaStream_t s) {
  switch (bn) {
    case 256: return launch_typed<256, MODE, 1>(ta, tb, ts, to, tr, kp, s);
    case 128:
      return MODE != 2 ? launch_typed<128, MODE, 2>(ta, tb, ts, to, tr, kp, s)
                       : launch_typed<128, MODE, 1>(ta, tb, ts, to, tr, kp, s);
    case 64: return launch_typed<64, MODE, 1>(ta, tb, ts, to, tr, kp, s);
    case 32: return launch_typed<32, MODE, 1>(ta, tb, ts, to, tr, kp, s);
    default: return launch_typed<16, MODE, 1>(ta, tb, ts, to, tr, kp, s);
  }
}

// VAE_CONV=taps turns the buffered-A modes (halo, channel-major) off, leaving
// every conv on per-tap staging (comparisons).
bool buffered_a_enabled() {
  static const bool on = [] {
    const char *e = std::getenv("VAE_CONV");
    return !(e && std::strcmp(e, "taps") == 0);
  }();
  return on;
}

int pick_bn(int cout) {
  if (cout > 128) return 256;
  if (cout > 64) return 128;
  if (cout > 32) return 64;
  if (cout > 16) return 32;
  return 16;
}

// VAE_SPLIT=force forms every product in split-TF32 (tests of that path on
// the single-op entry points).
bool split_forced() {
  static const bool v = [] {
    const char *e = std::getenv("VAE_SPLIT");
    return e && std::strcmp(e, "force") == 0;
  }();
  return v;
}

// VAE_PAIR=off keeps every conv on 1-SM tiles, VAE_PAIR=force pairs every conv
// that can be paired (comparisons and tests); default: by the estimate below.
int pair_setting() {
  static const int v = [] {
    const char *e = std::getenv("VAE_PAIR");
    if (e && std::strcmp(e, "off") == 0) return 0;
    if (e && std::strcmp(e, "force") == 0) return 2;
    return 1;
  }();
  return v;
}

// Output tiles per image of a conv / upsample conv whose tiles hold `rows`
// pixel rows (per output parity tile for the upsample conv).
long long tiles_per_image(const IgemmDesc &d, int rows, int max_bw = 128) {
  const int bw = std::min(max_bw, pow2_at_least(d.win));
  const int bh = rows / bw;
  long long t = static_cast<long long>(ceil_div(d.win, bw)) * ceil_div(d.hin, bh);
  if (d.mode == AMode::Upsample) t *= 4;  // one tile per output parity
  return t;
}

// Whether a launch runs as paired-CTA tiles (Cfg, PAIR): 256-column tiles of
// the pixel-major conv modes and of the GEMM mode, outside the split-K
// regime, when the pairs' 256-row tiles (about 0.8 of a 1-SM tile's time
// each: shared memory stops being the bound) finish sooner than 1-SM
// 128-row tiles, counting the stream-K balance the 1-SM conv path would get.
// (128-channel convs stay on the 1-SM channel-major tiles: paired halo tiles
// of 128 channels, one or two rows per CTA, measured 5-10 % slower on the
// 1024^2 layers.)
bool use_pair(const IgemmDesc &d) {
  const int setting = pair_setting();
  if (setting == 0) return false;
  if (pick_bn(d.cout) != 256) return false;
  const int sms = num_sms();
  if (sms < 2) return false;
  if (setting == 2) return true;
  const long long n_tiles = ceil_div(d.cout, 256);
  const bool gemm = d.mode == AMode::Gemm;
  const long long tiles1 = gemm ? ceil_div(d.M, kBM) * n_tiles
                                : static_cast<long long>(d.imgs) * tiles_per_image(d, kBM) * n_tiles;
  const long long tiles2 = gemm ? ceil_div(d.M, 2 * kBM) * n_tiles
                                : static_cast<long long>(d.imgs) * tiles_per_image(d, 2 * kBM) *
                                      n_tiles;
  if (tiles1 * 5 < static_cast<long long>(sms) * 3) return false;  // split-K regime
  const double r1 = static_cast<double>(tiles1) / sms;
  // stream-K balance (convs only) or whole rounds
  const double est1 = !gemm && r1 / std::ceil(r1) < 0.9 ? r1 : std::ceil(r1);
  const double est2 = 0.8 * std::ceil(static_cast<double>(tiles2) / (sms / 2));
  return est2 <= est1;
}

long long stat_slots_for(const IgemmDesc &d, bool pair, int max_bw) {
  if (!(d.mode == AMode::Conv || d.mode == AMode::Upsample)) return 0;
  const int ms = (pair || pick_bn(d.cout) == 128) ? 2 : 1;
  return static_cast<long long>(d.t > 0 ? d.t : 1) * tiles_per_image(d, ms * kBM, max_bw) * ms * 4;
}

// Channel-major tiles (MODE 4, see igemm_launch) take bands at most 64 pixels
// wide; this is the row width the conv's tiles get when they may run so.
int conv_max_bw(const IgemmDesc &d, bool split) {
  const bool swap_geom = !split && d.mode == AMode::Conv && pick_bn(d.cout) == 128 && d.k == 3 &&
                         d.kt == 1 && !d.out_nchw && buffered_a_enabled();
  return swap_geom ? 64 : 128;
}

}  // namespace

int igemm_col_tile(int cout) { return pick_bn(cout); }

// The operand transforms (input GroupNorm, softmax A) run only with
// VAE_FUSE=on. Measured on GB300 they lose to the separate passes: the
// GroupNorm+SiLU of a halo buffer sits between its copy and the MMAs of a
// two-buffer ring, so the 128^2 x 512-channel conv goes from 0.103 to 0.218
// ms (0.113 ms with the transform's arithmetic removed), while the separate
// apply pass it replaces costs about 0.035 ms; the softmax-normalised P.V
// GEMM takes 1.2 ms even with an empty transform (0.3 ms plain) and the
// statistics epilogue adds about 0.25 ms to the score GEMM, against the
// 0.3 ms row-softmax pass.
bool operand_transforms_enabled() {
  static const bool v = [] {
    const char *e = std::getenv("VAE_FUSE");
    return e && std::strcmp(e, "on") == 0;
  }();
  return v;
}

// The halo-staged path (see igemm_launch), less its no-split-K condition:
// a launch with an input GroupNorm never splits K.
bool halo_candidate(const IgemmDesc &d, bool split) {
  return !split && d.mode == AMode::Conv && d.k == 3 && d.kt == 1 &&
         pow2_at_least(d.win) >= 128 && pick_bn(d.cout) == 256 && !d.sc && d.sc_c == 0 &&
         buffered_a_enabled();
}

bool igemm_input_gn_ok(const IgemmDesc &d) {
  return operand_transforms_enabled() && halo_candidate(d, d.precise || split_forced());
}

// GroupNorm ahead runs only with VAE_GNA=on. Measured on GB300 it loses to
// the separate apply pass (which streams at about 0.9 of HBM bandwidth): in
// the 1024^2 decode the 1024^2 x 128-channel convs go from 0.39-0.45 ms to
// 0.69-0.73 ms (0.79-0.83 ms with sixteen loads in flight per thread), the
// 256^2 x 512-channel ones from 0.30 to 0.39 ms, against 0.05-0.17 ms saved
// per GroupNorm: the four extra warps' row stream competes with the conv's
// own copies and stores, and the first tiles wait for their rows.
bool gn_ahead_enabled() {
  static const bool v = [] {
    const char *e = std::getenv("VAE_GNA");
    return e && std::strcmp(e, "on") == 0;
  }();
  return v;
}

bool igemm_gn_ahead_ok(const IgemmDesc &d) {
  if (!gn_ahead_enabled() || d.precise || split_forced() || d.mode != AMode::Conv || d.k != 3 ||
      d.kt != 1 || d.out_nchw || !buffered_a_enabled())
    return false;
  if (d.a_c <= 0 || d.a_c > 512 || 128 % (d.a_c / 4) != 0 || d.a_c % 32) return false;
  const int bn = pick_bn(d.cout);
  if (bn == 256) return halo_candidate(d, false);
  return bn == 128 && d.win >= 2;
}

bool igemm_softmax_a_ok(const IgemmDesc &d) {
  return operand_transforms_enabled() && d.mode == AMode::Gemm && !d.precise &&
         !split_forced() && pick_bn(d.cout) == 256;
}

// Upper bound over the tile geometries a launch may take (callers size the
// partials buffer with it; the launch reports the stride it used).
long long igemm_stat_slots(const IgemmDesc &d) {
  return std::max({stat_slots_for(d, false, 128), stat_slots_for(d, false, 64),
                   stat_slots_for(d, true, 128)});
}

int igemm_launch(const IgemmDesc &d, cudaStream_t stream) {
  if (!d.a || !d.b || !d.out || d.cout <= 0) return VAE_EINVAL;
  auto misaligned = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) != 0; };
  if (misaligned(d.a) || misaligned(d.b) || (d.sc && misaligned(d.sc)) ||
      (d.bias && misaligned(d.bias)))
    return VAE_EINVAL;

  const int bn = pick_bn(d.cout);
  // Paired-CTA tiles (256 pixel rows across a CTA pair; see Cfg).
  // Split-TF32 products (split_setting: VAE_SPLIT=force makes every launch
  // split, for tests); they run on per-step A and B stages only.
  const bool split = d.precise || split_forced();
  const bool pair = !split && use_pair(d);
  // operand transforms: only on the paths that implement them
  const int xf = d.gn_scale ? 1 : d.sm_m ? 2 : d.ga_x ? 3 : 0;
  if ((d.gn_scale != nullptr) + (d.sm_m != nullptr) + (d.ga_x != nullptr) > 1) return VAE_EINVAL;
  if (xf == 3 && (!igemm_gn_ahead_ok(d) || !d.ga_scale || !d.ga_shift || !d.ga_flags ||
                  !d.ga_next || d.ga_epoch == 0))
    return VAE_EUNSUPPORTED;
  if (xf == 1 && (!igemm_input_gn_ok(d) || !d.gn_shift)) return VAE_EUNSUPPORTED;
  if (xf == 2 && (!igemm_softmax_a_ok(d) || !d.sm_inv_l || d.sm_cols <= 0)) return VAE_EUNSUPPORTED;
  if (d.rs_out && (d.mode != AMode::Gemm || d.rs_ld < ceil_div(d.cout, bn) || d.rs_cols <= 0))
    return VAE_EINVAL;
  KParams kp{};
  kp.err = device_error_word();
  if (!kp.err) return VAE_ECUDA;
  kp.wait_ns = wait_limit_ns();
  kp.inject = injected_faults();
  kp.cout = d.cout;
  kp.out = d.out;
  kp.ldo = d.ldo;
  kp.out_nchw = d.out_nchw;
  kp.bias = d.bias;
  kp.bias_per_row = d.bias_per_row;
  kp.residual = d.residual;
  kp.alpha = d.alpha;
  kp.round_out = d.round_out;
  kp.t = d.t > 0 ? d.t : 1;
  kp.imgs = d.imgs;
  kp.n_tiles = ceil_div(d.cout, bn);
  kp.gn_scale = d.gn_scale;
  kp.gn_shift = d.gn_shift;
  kp.gn_silu = d.gn_silu;
  kp.sm_m = d.sm_m;
  kp.sm_inv_l = d.sm_inv_l;
  kp.sm_scale = d.sm_scale;
  kp.sm_cols = d.sm_cols;
  kp.rs_out = d.rs_out;
  kp.rs_scale = d.rs_scale;
  kp.rs_cols = d.rs_cols;
  kp.rs_ld = d.rs_ld;
  if (xf == 1 && ((reinterpret_cast<uintptr_t>(d.gn_scale) | reinterpret_cast<uintptr_t>(d.gn_shift)) & 15))
    return VAE_EINVAL;
  kp.ga_x = d.ga_x;
  kp.ga_scale = d.ga_scale;
  kp.ga_shift = d.ga_shift;
  kp.ga_t = const_cast<float *>(d.a);
  kp.ga_flags = d.ga_flags;
  kp.ga_next = d.ga_next;
  kp.ga_epoch = d.ga_epoch;
  if (xf == 3 && ((reinterpret_cast<uintptr_t>(d.ga_scale) | reinterpret_cast<uintptr_t>(d.ga_shift) |
                   reinterpret_cast<uintptr_t>(d.ga_x)) & 15))
    return VAE_EINVAL;

  CUtensorMap ta{}, tb{}, ts{};
  int bkdim;
  if (d.mode == AMode::Gemm) {
    if (d.kdim <= 0 || d.kdim % 32 || d.M <= 0 || d.lda % 4) return VAE_EINVAL;
    kp.M = d.M;
    kp.m_tiles = ceil_div(d.M, pair ? 2 * kBM : kBM);  // paired tiles: 256 rows
    kp.taps = 1;
    kp.cin_chunks = d.kdim / 32;
    kp.cin_pad = d.kdim;
    kp.k_stages = kp.cin_chunks;
    const uint64_t dims[2] = {static_cast<uint64_t>(d.kdim), static_cast<uint64_t>(d.M)};
    const uint64_t str[1] = {static_cast<uint64_t>(d.lda) * 4};
    const uint32_t box[2] = {32, static_cast<uint32_t>(kBM)};
    VAE_TRY(encode_tiled(&ta, d.a, 2, dims, str, box));
    bkdim = d.kdim;
  } else {
    if (d.a_c <= 0 || d.a_c % 32 || d.hin <= 0 || d.win <= 0 || d.imgs <= 0) return VAE_EINVAL;
    kp.hin = d.hin;
    kp.win = d.win;
    kp.cin_chunks = d.a_c / 32;
    kp.cin_pad = d.a_c;
    uint32_t box[4];
    if (d.mode == AMode::Conv) {
      if (!(d.k == 1 || d.k == 3) || !(d.kt == 1 || d.kt == 3)) return VAE_EUNSUPPORTED;
      kp.k = d.k;
      kp.kt = d.kt;
      kp.taps = d.k * d.k * d.kt;
      kp.hout = d.hin;
      kp.wout = d.win;
      const int rows = (bn == 128 || pair ? 2 : 1) * kBM;  // M sub-tiles (see Cfg)
      kp.bw = std::min(conv_max_bw(d, split), pow2_at_least(d.win));
      kp.bh = rows / kp.bw;
      kp.tiles_x = ceil_div(d.win, kp.bw);
      kp.tiles_y = ceil_div(d.hin, kp.bh);
      kp.sc_chunks = d.sc ? d.sc_c / 32 : 0;
      if (d.sc && (d.sc_c <= 0 || d.sc_c % 32)) return VAE_EINVAL;
      box[0] = 32;
      box[1] = kp.bw;
      box[2] = pair ? kp.bh / 2 : kp.bh;  // a paired CTA loads its own 128 rows
      box[3] = 1;
    } else {
      // Nearest-2x upsample + 3x3 conv as four parity-specific 2x2 convs of
      // the low-res input (weights packed by pack_upsample_weights): a tile
      // is bw x bh low-res pixels of one output parity.
      kp.taps = 4;
      kp.hout = 2 * d.hin;
      kp.wout = 2 * d.win;
      const int rows = (bn == 128 || pair ? 2 : 1) * kBM;
      kp.bw = std::min(128, pow2_at_least(d.win));
      kp.bh = rows / kp.bw;
      kp.tiles_x = ceil_div(d.win, kp.bw);
      kp.tiles_y = ceil_div(d.hin, kp.bh);
      box[0] = 32;
      box[1] = kp.bw;
      box[2] = pair ? kp.bh / 2 : kp.bh;
      box[3] = 1;
    }
    kp.m_tiles = d.imgs * kp.tiles_x * kp.tiles_y * (d.mode == AMode::Upsample ? 4 : 1);
    kp.k_stages = kp.taps * kp.cin_chunks + kp.sc_chunks;
    const uint64_t dims[4] = {static_cast<uint64_t>(d.a_c), static_cast<uint64_t>(d.win),
                              static_cast<uint64_t>(d.hin), static_cast<uint64_t>(d.imgs)};
    const uint64_t str[3] = {static_cast<uint64_t>(d.a_c) * 4,
                             static_cast<uint64_t>(d.win) * d.a_c * 4,
                             static_cast<uint64_t>(d.hin) * d.win * d.a_c * 4};
    VAE_TRY(encode_tiled(&ta, d.a, 4, dims, str, box));
    if (kp.sc_chunks) {
      const uint64_t sdims[4] = {static_cast<uint64_t>(d.sc_c), static_cast<uint64_t>(kp.wout),
                                 static_cast<uint64_t>(kp.hout), static_cast<uint64_t>(d.imgs)};
      const uint64_t sstr[3] = {static_cast<uint64_t>(d.sc_c) * 4,
                                static_cast<uint64_t>(kp.wout) * d.sc_c * 4,
                                static_cast<uint64_t>(kp.hout) * kp.wout * d.sc_c * 4};
      VAE_TRY(encode_tiled(&ts, d.sc, 4, sdims, sstr, box));
    } else {
      ts = ta;
    }
    bkdim = d.ldb;
  }
  if (d.ldb % 4 || bkdim <= 0) return VAE_EINVAL;
  {
    // Upsample: four parities' weight rows, parity-major
    const uint64_t brows = static_cast<uint64_t>(d.cout) * (d.mode == AMode::Upsample ? 4 : 1);
    const uint64_t dims[2] = {static_cast<uint64_t>(bkdim), brows};
    const uint64_t str[1] = {static_cast<uint64_t>(d.ldb) * 4};
    const uint32_t box[2] = {32, static_cast<uint32_t>(pair ? bn / 2 : bn)};  // paired: a half
    VAE_TRY(encode_tiled(&tb, d.b, 2, dims, str, box));
  }
  const long long total = static_cast<long long>(kp.m_tiles) * kp.n_tiles;
  if (total <= 0 || total > (1ll << 31) - 1) return VAE_EUNSUPPORTED;

  // Split-K when the output tiles fill less than ~60% of the SMs: each split
  // accumulates a slice of the reduction into the caller's split workspace and
  // a fixed-order reduce applies bias, residual and rounding.
  kp.splits = 1;
  kp.ks_per = kp.k_stages;
  kp.split_stride = 0;
  const long long rows_total = d.mode == AMode::Gemm
                                   ? static_cast<long long>(d.M)
                                   : static_cast<long long>(d.imgs) * kp.hout * kp.wout;
  if (!pair && !xf && d.split_ws && d.mode != AMode::Gemm && !d.out_nchw && d.cout % 4 == 0 &&
      d.ldo == d.cout && !d.bias_per_row) {
    const int sms = num_sms();
    if (total * 5 < static_cast<long long>(sms) * 3) {
      long long sp = std::min<long long>(sms / total, kp.k_stages / 8);
      sp = std::min<long long>(sp, 16);
      const long long per = rows_total * d.cout;
      while (sp > 1 && sp * per > static_cast<long long>(d.split_ws_floats)) --sp;
      if (sp > 1) {
        kp.ks_per = ceil_div(kp.k_stages, sp);
        kp.splits = ceil_div(kp.k_stages, kp.ks_per);
        kp.split_stride = per;
      }
    }
  }
  if (total * kp.splits > (1ll << 31) - 1) return VAE_EUNSUPPORTED;
  kp.total_tiles = static_cast<int>(total * kp.splits);
  if (kp.splits > 1) {  // the kernel writes raw partial sums
    kp.out = d.split_ws;
    kp.ldo = d.cout;
    kp.bias = nullptr;
    kp.residual = nullptr;
    kp.round_out = 0;
    kp.alpha = 1.0f;
  }

  // Output (and residual) tensor maps for the staged TMA-store epilogue: one
  // box per epilogue warp = 32 rows x 32 channels.
  CUtensorMap to = tb, tr = tb;
  kp.has_res = kp.residual != nullptr;
  kp.stat_part = nullptr;
  auto al16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  bool epi = kp.splits == 1 && !d.out_nchw && bn >= 32 && !d.bias_per_row && d.ldo % 4 == 0 &&
             al16(d.out) && (!d.residual || al16(d.residual));
  if (d.mode == AMode::Upsample && d.imgs > 1 && d.hin % kp.bh) epi = false;  // rows would wrap
  if (epi) {
    auto encode_out = [&](CUtensorMap *m, const float *base) -> int {
      const uint64_t ld4 = static_cast<uint64_t>(d.ldo) * 4;
      if (d.mode == AMode::Gemm) {
        const uint64_t dims[2] = {static_cast<uint64_t>(d.cout), static_cast<uint64_t>(d.M)};
        const uint64_t str[1] = {ld4};
        const uint32_t box[2] = {32, 32};
        return encode_tiled(m, base, 2, dims, str, box);
      }
      if (d.mode == AMode::Conv) {
        const uint32_t bw = std::min(kp.bw, 32);
        const uint64_t dims[4] = {static_cast<uint64_t>(d.cout), static_cast<uint64_t>(kp.wout),
                                  static_cast<uint64_t>(kp.hout), static_cast<uint64_t>(d.imgs)};
        const uint64_t str[3] = {ld4, ld4 * kp.wout, ld4 * kp.wout * kp.hout};
        const uint32_t box[4] = {32, bw, 32 / bw, 1};
        return encode_tiled(m, base, 4, dims, str, box);
      }
      // Upsample: output [imgs*hin][py][win][px][cout]; a warp's 32 rows of
      // one parity are box (32, 1, min(bw, 32), 1, 32 / min(bw, 32)).
      const uint32_t bw = std::min(kp.bw, 32);
      const uint64_t dims[5] = {static_cast<uint64_t>(d.cout), 2, static_cast<uint64_t>(d.win),
                                2, static_cast<uint64_t>(d.imgs) * d.hin};
      const uint64_t str[4] = {ld4, 2 * ld4, ld4 * kp.wout, 2 * ld4 * kp.wout};
      const uint32_t box[5] = {32, 1, bw, 1, 32 / bw};
      return encode_tiled(m, base, 5, dims, str, box);
    };
    VAE_TRY(encode_out(&to, d.out));
    if (d.residual) VAE_TRY(encode_out(&tr, d.residual));
  }
  kp.epi_tma = epi ? 1 : 0;
  // Fused GroupNorm statistics need the staged epilogue and groups that sit
  // inside one 32-channel chunk; otherwise the caller computes them itself.
  if (d.stat_part) {
    const int cg = d.stat_groups > 0 ? d.cout / d.stat_groups : 0;
    const long long slots =
        stat_slots_for(d, pair, d.mode == AMode::Conv ? conv_max_bw(d, split) : 128);
    if (epi && d.mode != AMode::Gemm && d.cout % 32 == 0 && d.stat_groups > 0 &&
        d.cout % d.stat_groups == 0 && cg >= 1 && cg <= 32 && (cg & (cg - 1)) == 0 &&
        slots > 0 && slots < (1ll << 31)) {
      kp.stat_part = d.stat_part;
      kp.stat_cg = cg;
      kp.stat_groups = d.stat_groups;
      kp.stat_slots = static_cast<int>(slots);
    }
  }
  if (d.stat_ok) *d.stat_ok = kp.stat_part != nullptr;
  if (d.stat_slots) *d.stat_slots = kp.stat_part ? kp.stat_slots : 0;

  // Halo staging for 3x3 single-frame convs with 256-channel tiles spanning
  // 128 pixels of a row: one 3 x 130-pixel box per 32-channel chunk serves
  // all nine taps. Per reduction step shared memory then takes in 37.6 KB
  // instead of 48 KB, while the MMAs read 48 KB from it; with the two near
  // its bandwidth, that is 7-12% per conv on GB300. Measured slower (so left
  // to the per-tap path): 128-channel tiles (two 128-row sub-tiles), and
  // convs with an appended shortcut (with its tiles one or three to an A
  // buffer alike: 0.537 -> 0.607 ms on 512 -> 256 channels at 512^2).
  const bool halo = halo_candidate(d, split) && kp.splits == 1;
  if (xf == 1 && !halo) return VAE_EUNSUPPORTED;  // (not reached: no split-K with xf)
  // Channel-major tiles for 3x3 single-frame convs with 65-128 output
  // channels: the MMA runs M = 128 channels x N = 256 pixels (one wide
  // instruction where the pixel-major tile needs two 128 x 128 ones that both
  // read the weights), and per 32-channel chunk one band of bh + 2 rows per
  // kx serves the three ky taps (bands at most 64 pixels wide: 4 rows + 2
  // halo rows, three of them in flight). Needs the staged epilogue (it
  // transposes).
  const bool swap = !split && !halo && d.mode == AMode::Conv && kp.k == 3 && kp.kt == 1 &&
                    bn == 128 && kp.splits == 1 && epi && kp.bw >= 2 && kp.bw <= 64 &&
                    (kp.bh + 2) * kp.bw * 128 <= 49152 && buffered_a_enabled();
  if (swap) {
    const uint64_t dims[4] = {static_cast<uint64_t>(d.a_c), static_cast<uint64_t>(d.win),
                              static_cast<uint64_t>(d.hin), static_cast<uint64_t>(d.imgs)};
    const uint64_t str[3] = {static_cast<uint64_t>(d.a_c) * 4,
                             static_cast<uint64_t>(d.win) * d.a_c * 4,
                             static_cast<uint64_t>(d.hin) * d.win * d.a_c * 4};
    const uint32_t box[4] = {32, static_cast<uint32_t>(kp.bw), static_cast<uint32_t>(kp.bh + 2),
                             1};
    VAE_TRY(encode_tiled(&ta, d.a, 4, dims, str, box));
  }
  if (xf == 3 && !(halo || swap)) return VAE_EUNSUPPORTED;
  if (halo) {
    const uint64_t dims[4] = {static_cast<uint64_t>(d.a_c), static_cast<uint64_t>(d.win),
                              static_cast<uint64_t>(d.hin), static_cast<uint64_t>(d.imgs)};
    const uint64_t str[3] = {static_cast<uint64_t>(d.a_c) * 4,
                             static_cast<uint64_t>(d.win) * d.a_c * 4,
                             static_cast<uint64_t>(d.hin) * d.win * d.a_c * 4};
    // (paired: each CTA stages its own row with its one-pixel border)
    const uint32_t box[4] = {32, 130, static_cast<uint32_t>((pair ? kp.bh / 2 : kp.bh) + 2), 1};
    VAE_TRY(encode_tiled(&ta, d.a, 4, dims, str, box));
  }

  // Stream-K for convs on 1-SM tiles whose whole tiles would leave the last
  // round of SMs mostly idle (e.g. 256 tiles on 152 SMs: 1.68 rounds run as
  // 2). (On paired tiles -- ranges per pair, each CTA handing its rows to the
  // same-rank CTA of the next pair, a cooperative cluster launch -- it was
  // exact but measured slower: the 128^2 x 512-channel convs 0.100-0.109 ->
  // 0.102-0.119 ms.) Not for
  // the attention GEMMs (measured slower): their n-tiles of one row block
  // share a large A operand through L2 only while they run side by side,
  // which the stream-K ranges undo.
  kp.sk = 0;
  if (!pair && !split && d.mode == AMode::Conv && !swap && kp.splits == 1 && d.split_ws &&
      bn >= 32) {
    const int sms = num_sms();
    const long long tiles = total;
    const int units = halo ? kp.cin_chunks : kp.k_stages;
    const double rounds = static_cast<double>(tiles) / sms;
    const double eff = rounds / std::ceil(rounds);
    const int ms = (!halo && bn == 128) ? 2 : 1;
    // raw partial sums of one CTA's rows of a tile: ms x 128 rows x bn
    const size_t slot = static_cast<size_t>(ms) * bn * kBM;
    const size_t need = static_cast<size_t>(sms) * slot + static_cast<size_t>(sms) * 4;
    // Only long reductions: on short ones the tail/head partials would cost
    // more than the idle round.
    const int steps = halo ? kp.cin_chunks * 9 : kp.k_stages;
    if (tiles >= sms && eff < 0.9 && units >= 4 && steps >= 64 &&
        need <= d.split_ws_floats) {
      kp.sk = 1;
      kp.sk_units = units;
      kp.sk_total = tiles * units;
      kp.sk_part = d.split_ws;
      kp.sk_flag = reinterpret_cast<int *>(d.split_ws + static_cast<size_t>(sms) * slot);
      if (cudaMemsetAsync(kp.sk_flag, 0, static_cast<size_t>(sms) * 4 * sizeof(int), stream) !=
          cudaSuccess)
        return VAE_ECUDA;
    }
  }

  int rc;
  if (split) {
    rc = launch_split(static_cast<int>(d.mode), bn, ta, tb, ts, to, tr, kp, stream);
  } else if (xf) {
    rc = launch_xf(xf, swap ? 4 : halo ? 3 : 2, pair, ta, tb, ts, to, tr, kp, stream);
  } else switch (d.mode) {
    case AMode::Conv:
      if (pair)
        rc = halo ? launch_typed<256, 3, 1, true>(ta, tb, ts, to, tr, kp, stream)
                  : launch_typed<256, 0, 1, true>(ta, tb, ts, to, tr, kp, stream);
      else
        rc = halo   ? launch_typed<256, 3, 1>(ta, tb, ts, to, tr, kp, stream)
             : swap ? launch_typed<128, 4, 2>(ta, tb, ts, to, tr, kp, stream)
                    : launch_mode<0>(bn, ta, tb, ts, to, tr, kp, stream);
      break;
    case AMode::Upsample:
      rc = pair ? launch_typed<256, 1, 1, true>(ta, tb, ts, to, tr, kp, stream)
                : launch_mode<1>(bn, ta, tb, ts, to, tr, kp, stream);
      break;
    default:
      rc = pair ? launch_typed<256, 2, 1, true>(ta, tb, ts, to, tr, kp, stream)
                : launch_mode<2>(bn, ta, tb, ts, to, tr, kp, stream);
      break;
  }
  if (rc != VAE_OK || kp.splits == 1) return rc;
  // Split-K: fixed-order reduce + epilogue (+ GroupNorm partials of the output).
  long long slots = 0;
  VAE_TRY(splitk_reduce(d.split_ws, kp.splits, kp.split_stride, d.imgs / kp.t,
                        rows_total / (d.imgs / kp.t), d.cout, d.bias, d.alpha, d.residual,
                        d.round_out, d.out, d.stat_part, d.stat_groups, &slots, stream));
  if (d.stat_ok) *d.stat_ok = slots > 0;
  if (d.stat_slots) *d.stat_slots = slots;
  return VAE_OK;
}

}  // namespace vae
