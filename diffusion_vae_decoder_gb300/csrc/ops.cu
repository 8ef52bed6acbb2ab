// ops.cu -- the single-op C-ABI entry points: conv2d (with the fused resnet
// skip), upsample+conv, GroupNorm+SiLU, mid-block attention and the 3-D
// causal conv. Each one stages its operands into the NHWC, 32-channel-padded
// layout the tensor-core kernel reads, packs its weights (TF32-rounded) into
// the caller's workspace, and enqueues kernels on the caller's stream.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "common.cuh"
#include "ops.cuh"

namespace vae {

int stage_nhwc(const float *x, int n, int c, long long spatial, int layout, float *staging,
               int cpad, float alpha, float beta, int round, const float **out,
               cudaStream_t s) {
  const bool passthrough =
      layout == VAE_NHWC && c == cpad && alpha == 1.0f && beta == 0.0f && !round;
  if (passthrough) {
    *out = x;
    return VAE_OK;
  }
  if (!staging) return VAE_EINVAL;
  if (spatial > 0x7fffffffll) return VAE_EUNSUPPORTED;
  if (cpad != c)
    VAE_CUDA_TRY(cudaMemsetAsync(staging, 0, static_cast<size_t>(n) * spatial * cpad * 4, s));
  if (layout == VAE_NCHW) {
    VAE_TRY(transpose(x, static_cast<long long>(c) * spatial, static_cast<int>(spatial), staging,
                      spatial * cpad, cpad, n, c, static_cast<int>(spatial), alpha, beta, round,
                      s));
  } else {
    if (alpha != 1.0f || beta != 0.0f || round) return VAE_EINVAL;
    VAE_TRY(pad_rows(x, static_cast<long long>(n) * spatial, c, staging, cpad, s));
  }
  *out = staging;
  return VAE_OK;
}

int unstage_nchw(const float *src_nhwc, int n, int c, long long spatial, float *dst_nchw,
                 cudaStream_t s) {
  if (spatial > 0x7fffffffll) return VAE_EUNSUPPORTED;
  return transpose(src_nhwc, spatial * c, c, dst_nchw, static_cast<long long>(c) * spatial,
                   static_cast<int>(spatial), n, static_cast<int>(spatial), c, 1.0f, 0.0f, 0, s);
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool needs_stage(int layout, int c) { return layout == VAE_NCHW || c % 32 != 0; }

// ---------------------------------------------------------------- conv2d
struct ConvWs {
  float *packed, *bias_sum, *xs, *scs, *split;
  size_t split_floats;
};

// out_scale: output pixels per input pixel (4 for the upsample conv).
// The upsample conv's packed weights (4 parities x 2x2 taps) take the room of
// a 16-tap pack.
constexpr int kUpsamplePackTaps = 16;
ConvWs carve_conv(Carver &cv, int n, int cin, long long spatial, int layout, int cout, int taps,
                  int sc_cin, int out_scale = 1) {
  ConvWs w{};
  const int ldb = packed_ldb(cin, taps, sc_cin);
  w.packed = cv.take<float>(static_cast<size_t>(cout) * ldb);
  w.bias_sum = sc_cin ? cv.take<float>(cout) : nullptr;
  w.xs = needs_stage(layout, cin)
             ? cv.take<float>(static_cast<size_t>(n) * spatial * round_up32(cin))
             : nullptr;
  w.scs = (sc_cin && needs_stage(layout, sc_cin))
              ? cv.take<float>(static_cast<size_t>(n) * spatial * round_up32(sc_cin))
              : nullptr;
  // split-K partials: at most 16 splits of the output
  w.split_floats = std::min<size_t>(kSplitWsFloats,
                            16ull * n * static_cast<size_t>(spatial) * out_scale * cout);
  w.split = cv.take<float>(w.split_floats);
  return w;
}

// ---------------------------------------------------------------- attention
struct AttnWs {
  float *xs, *t, *wqkv, *bqkv, *wo, *qkv, *vt, *s, *o, *y, *rs;
  void *gn;
};

AttnWs carve_attn(Carver &cv, int n, int c, int L, int layout) {
  AttnWs w{};
  const size_t nl = static_cast<size_t>(n) * L;
  const size_t lp = static_cast<size_t>(round_up32(L));
  w.xs = layout == VAE_NCHW ? cv.take<float>(nl * c) : nullptr;
  w.t = cv.take<float>(nl * c);
  w.wqkv = cv.take<float>(3ull * c * c);
  w.bqkv = cv.take<float>(3ull * c);
  w.wo = cv.take<float>(static_cast<size_t>(c) * c);
  w.qkv = cv.take<float>(nl * 3 * c);
  w.vt = cv.take<float>(static_cast<size_t>(c) * lp);
  w.s = cv.take<float>(static_cast<size_t>(L) * lp);
  w.o = cv.take<float>(nl * c);
  w.y = layout == VAE_NCHW ? cv.take<float>(nl * c) : nullptr;
  w.gn = cv.take<char>(groupnorm_ws_bytes(n, c, L, c));  // groups <= c
  w.rs = cv.take<float>(attn_rs_floats(L));
  return w;
}

// ---------------------------------------------------------------- causal stack
struct StackWs {
  float *packed, *xs, *ring[3], *h;
  void *gn;
};

StackWs carve_stack(Carver &cv, int n, int c, long long vox, int layout, int n_layers,
                    int groups) {
  StackWs w{};
  const size_t act = static_cast<size_t>(n) * vox * c;
  w.packed = cv.take<float>(static_cast<size_t>(n_layers) * c * packed_ldb(c, 27, 0));
  w.xs = layout == VAE_NCHW ? cv.take<float>(act) : nullptr;
  for (int i = 0; i < 3; ++i) w.ring[i] = cv.take<float>(act);
  w.h = cv.take<float>(act);
  w.gn = cv.take<char>(groupnorm_ws_bytes(n, c, vox, groups));
  return w;
}

}  // namespace

size_t attn_rs_floats(int L) {
  const size_t tiles = static_cast<size_t>(ceil_div(L, igemm_col_tile(L)));
  return 2 * static_cast<size_t>(L) * tiles + 2 * static_cast<size_t>(L);
}

size_t attn_ws_bytes(int n, int c, int L, int layout) {
  Carver cv(nullptr, 0);
  carve_attn(cv, n, c, L, layout);
  return cv.used;
}

// Which attention path runs. The fused kernel keeps S on chip but TMEM holds
// at most a 256-column slice of O next to S, so a wider head recomputes S once
// per slice (1.5x the FLOPs at c = 512); measured on GB300 at 16384 tokens,
// c = 512, that is 1.71 ms against 1.37 ms for the score-matrix path (GEMM,
// row softmax, GEMM). Default: fused when the head fits one slice.
// VAE_ATTN=flash or VAE_ATTN=unfused forces a path (profiling comparisons).
bool use_fused_attention(int c) {
  static const int mode = [] {
    const char *e = std::getenv("VAE_ATTN");
    if (e && std::strcmp(e, "unfused") == 0) return 1;
    if (e && std::strcmp(e, "flash") == 0) return 2;
    return 0;
  }();
  if (!flash_supported(c) || mode == 1) return false;
  return mode == 2 || c <= 256;
}

// Attention on NHWC data (token-major): x_nhwc [n][L][c] -> y_nhwc (may equal
// x_nhwc). Weights are pre-packed: wqkv [3c][c], bqkv [3c], wo [c][c].
int attention_nhwc(const float *x, int n, int c, int L, int groups, float eps,
                   const float *gn_w, const float *gn_b, const float *wqkv, const float *bqkv,
                   const float *wo, const float *bo, float *y, const AttnScratch &sc,
                   cudaStream_t s, bool exact) {
  const int lp = round_up32(L);
  const int rnd = exact ? 0 : 1;  // MMA operands are stored TF32-rounded unless split
  // t = GroupNorm(x), no SiLU; TF32-rounded because it is an MMA operand.
  VAE_TRY(groupnorm_silu(x, n, c, L, 1, groups, eps, gn_w, gn_b, 0, rnd, sc.t, sc.gn, s));
  // [q | k | v] = t [Wq; Wk; Wv]^T + [bq; bk; bv], one GEMM for all images.
  {
    IgemmDesc d;
    d.mode = AMode::Gemm;
    d.a = sc.t;
    d.lda = c;
    d.M = n * L;
    d.kdim = c;
    d.b = wqkv;
    d.ldb = c;
    d.cout = 3 * c;
    d.out = sc.qkv;
    d.ldo = 3 * c;
    d.bias = bqkv;
    d.round_out = rnd;
    d.precise = exact;
    VAE_TRY(igemm_launch(d, s));
  }
  if (lp != L) VAE_CUDA_TRY(cudaMemsetAsync(sc.vt, 0, static_cast<size_t>(c) * lp * 4, s));
  const bool fused = !exact && use_fused_attention(c);
  const float scale = 1.0f / std::sqrt(static_cast<float>(c));
  for (int b = 0; b < n; ++b) {
    const float *qkv_b = sc.qkv + static_cast<size_t>(b) * L * 3 * c;
    // V^T [c][L] (row stride lp): the K-major B operand of P.V.
    VAE_TRY(transpose(qkv_b + 2 * c, 0, 3 * c, sc.vt, 0, lp, 1, L, c, 1.0f, 0.0f, 0, s));
    if (fused) {  // scores stay on chip
      VAE_TRY(flash_attention(qkv_b, qkv_b + c, 3 * c, sc.vt, lp, L, c, scale,
                              sc.o + static_cast<size_t>(b) * L * c, c, s));
      continue;
    }
    // o = P V with P = softmax(S * scale) row-wise
    IgemmDesc pv;
    pv.mode = AMode::Gemm;
    pv.a = sc.s;
    pv.lda = lp;
    pv.M = L;
    pv.kdim = lp;
    pv.b = sc.vt;
    pv.ldb = lp;
    pv.cout = c;
    pv.out = sc.o + static_cast<size_t>(b) * L * c;
    pv.ldo = c;
    pv.round_out = rnd;
    pv.precise = exact;
    // The softmax folded into the two GEMMs when the P.V kernel normalises
    // its A stages (opt-in, see igemm_softmax_a_ok): the score GEMM's
    // epilogue gathers each row's
    // (max, sum of exponentials) per column tile, a merge turns them into the
    // row's max and 1 / sum, and the P.V kernel reads exp(s * scale - max) /
    // sum from the raw scores.
    const bool fold = igemm_softmax_a_ok(pv);
    const int rs_tiles = ceil_div(L, igemm_col_tile(L));
    float2 *rs = reinterpret_cast<float2 *>(sc.rs);
    float *row_m = sc.rs + 2 * static_cast<size_t>(L) * rs_tiles, *row_il = row_m + L;
    // S = q k^T (scale applied by the softmax).
    {
      IgemmDesc d;
      d.mode = AMode::Gemm;
      d.a = qkv_b;
      d.lda = 3 * c;
      d.M = L;
      d.kdim = c;
      d.b = qkv_b + c;
      d.ldb = 3 * c;
      d.cout = L;
      d.out = sc.s;
      d.ldo = lp;
      d.precise = exact;
      if (fold) {
        d.rs_out = rs;
        d.rs_scale = scale;
        d.rs_cols = L;
        d.rs_ld = rs_tiles;
      }
      VAE_TRY(igemm_launch(d, s));
    }
    if (fold) {
      VAE_TRY(softmax_merge_stats(rs, L, rs_tiles, rs_tiles, row_m, row_il, s));
      pv.sm_m = row_m;
      pv.sm_inv_l = row_il;
      pv.sm_scale = scale;
      pv.sm_cols = L;
    } else {
      VAE_TRY(softmax_rows(sc.s, L, L, lp, scale, s, rnd));
    }
    VAE_TRY(igemm_launch(pv, s));
  }
  // y = x + (o Wo^T + bo)
  IgemmDesc d;
  d.mode = AMode::Gemm;
  d.a = sc.o;
  d.lda = c;
  d.M = n * L;
  d.kdim = c;
  d.b = wo;
  d.ldb = c;
  d.cout = c;
  d.out = y;
  d.ldo = c;
  d.bias = bo;
  d.residual = x;
  d.precise = exact;
  return igemm_launch(d, s);
}

}  // namespace vae

using namespace vae;

extern "C" {

// ------------------------------------------------------------------ conv2d
size_t vae_conv2d_workspace_size(int n, int cin, int h, int w, int layout, int cout, int k,
                                 int sc_cin) {
  if (n <= 0 || cin <= 0 || h <= 0 || w <= 0 || cout <= 0 || k <= 0 || sc_cin < 0) return 0;
  Carver cv(nullptr, 0);
  carve_conv(cv, n, cin, static_cast<long long>(h) * w, layout, cout, k * k, sc_cin);
  return cv.used;
}

namespace {

// The layout of a weight pack made by vae_conv2d_pack / vae_upsample_conv_pack:
// the GEMM-layout weights (rows x ldb floats, TF32-rounded), then the bias
// (cout floats, the shortcut's folded in; zeros without one), each carve
// 256-byte aligned.
struct ConvPack {
  float *w, *bias;
};
ConvPack carve_pack(Carver &cv, size_t rows, int ldb, int cout) {
  ConvPack p{};
  p.w = cv.take<float>(rows * static_cast<size_t>(ldb));
  p.bias = cv.take<float>(static_cast<size_t>(cout));
  return p;
}

int conv_args_ok(const float *x, float *y, int n, int cin, int h, int w, int layout, int cout,
                 int k, const float *residual, const float *sc_x, int sc_cin) {
  if (!x || !y || n <= 0 || cin <= 0 || h <= 0 || w <= 0 || cout <= 0) return VAE_EINVAL;
  if (layout != VAE_NCHW && layout != VAE_NHWC) return VAE_EINVAL;
  if (k != 1 && k != 3) return VAE_EUNSUPPORTED;
  if (sc_x && sc_cin <= 0) return VAE_EINVAL;
  if (cin > 4096 || cout > 4096 || sc_cin > 4096 || h > 65535 || w > 65535)
    return VAE_EUNSUPPORTED;
  if (!aligned16(x) || !aligned16(y) || (residual && !aligned16(residual)) ||
      (sc_x && !aligned16(sc_x)))
    return VAE_EINVAL;
  if (layout == VAE_NHWC && cout % 4) return VAE_EUNSUPPORTED;
  return VAE_OK;
}

// The conv on packed weights (cw: the call's workspace; its packed area is
// not used when the weights come packed).
int conv2d_run(const float *x, int n, int cin, int h, int w, int layout, const float *packed,
               const float *bias, int cout, int k, const float *residual, const float *sc_x,
               int scc, float *y, const ConvWs &cw, cudaStream_t s) {
  const long long spatial = static_cast<long long>(h) * w;
  const float *xa = nullptr, *sca = nullptr;
  VAE_TRY(stage_nhwc(x, n, cin, spatial, layout, cw.xs, round_up32(cin), 1.f, 0.f, 0, &xa, s));
  if (scc)
    VAE_TRY(stage_nhwc(sc_x, n, scc, spatial, layout, cw.scs, round_up32(scc), 1.f, 0.f, 0,
                       &sca, s));
  IgemmDesc d;
  d.mode = AMode::Conv;
  d.a = xa;
  d.imgs = n;
  d.hin = h;
  d.win = w;
  d.a_c = round_up32(cin);
  d.k = k;
  d.sc = sca;
  d.sc_c = scc ? round_up32(scc) : 0;
  d.b = packed;
  d.ldb = packed_ldb(cin, k * k, scc);
  d.cout = cout;
  d.out = y;
  d.ldo = cout;
  d.out_nchw = layout == VAE_NCHW;
  d.bias = bias;
  d.residual = residual;
  d.split_ws = cw.split;
  d.split_ws_floats = cw.split_floats;
  return igemm_launch(d, s);
}

int upsample_run(const float *x, int n, int cin, int h, int w, int layout, const float *packed,
                 const float *bias, int cout, float *y, const ConvWs &cw, cudaStream_t s) {
  const float *xa = nullptr;
  VAE_TRY(stage_nhwc(x, n, cin, static_cast<long long>(h) * w, layout, cw.xs, round_up32(cin),
                     1.f, 0.f, 0, &xa, s));
  IgemmDesc d;
  d.mode = AMode::Upsample;
  d.a = xa;
  d.imgs = n;
  d.hin = h;
  d.win = w;
  d.a_c = round_up32(cin);
  d.b = packed;
  d.ldb = upsample_ldb(cin);
  d.cout = cout;
  d.out = y;
  d.ldo = cout;
  d.out_nchw = layout == VAE_NCHW;
  d.bias = bias;
  d.split_ws = cw.split;
  d.split_ws_floats = cw.split_floats;
  return igemm_launch(d, s);
}

int upsample_args_ok(const float *x, float *y, int n, int cin, int h, int w, int layout,
                     int cout) {
  if (!x || !y || n <= 0 || cin <= 0 || h <= 0 || w <= 0 || cout <= 0) return VAE_EINVAL;
  if (layout != VAE_NCHW && layout != VAE_NHWC) return VAE_EINVAL;
  if (cin > 4096 || cout > 4096 || h > 32767 || w > 32767) return VAE_EUNSUPPORTED;
  if (!aligned16(x) || !aligned16(y)) return VAE_EINVAL;
  if (layout == VAE_NHWC && cout % 4) return VAE_EUNSUPPORTED;
  return VAE_OK;
}

}  // namespace

int vae_conv2d(const float *x, int n, int cin, int h, int w, int layout, const float *weight,
               const float *bias, int cout, int k, const float *residual, const float *sc_x,
               const float *sc_w, const float *sc_b, int sc_cin, float *y, void *ws,
               size_t ws_bytes, vae_stream_t stream) {
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (!weight || !ws) return VAE_EINVAL;
  const bool has_sc = sc_x != nullptr || sc_w != nullptr;
  if (has_sc && (!sc_x || !sc_w || sc_cin <= 0)) return VAE_EINVAL;
  const int scc = has_sc ? sc_cin : 0;
  VAE_TRY(conv_args_ok(x, y, n, cin, h, w, layout, cout, k, residual, sc_x, scc));
  Carver cv(ws, ws_bytes);
  ConvWs cw = carve_conv(cv, n, cin, static_cast<long long>(h) * w, layout, cout, k * k, scc);
  if (!cv.ok()) return VAE_EWORKSPACE;
  VAE_TRY(pack_conv_weights(weight, cout, cin, k * k, sc_w, scc, cw.packed, cout,
                            packed_ldb(cin, k * k, scc), s));
  const float *bsum = bias;
  if (has_sc && (bias || sc_b)) {
    VAE_TRY(add_bias(cw.bias_sum, bias, sc_b, cout, s));
    bsum = cw.bias_sum;
  }
  return conv2d_run(x, n, cin, h, w, layout, cw.packed, bsum, cout, k, residual, sc_x, scc, y, cw,
                    s);
}

size_t vae_conv2d_pack_bytes(int cout, int cin, int k, int sc_cin) {
  if (cout <= 0 || cin <= 0 || (k != 1 && k != 3) || sc_cin < 0) return 0;
  Carver cv(nullptr, 0);
  carve_pack(cv, cout, packed_ldb(cin, k * k, sc_cin), cout);
  return cv.used;
}

int vae_conv2d_pack(const float *weight, const float *bias, int cout, int cin, int k,
                    const float *sc_w, const float *sc_b, int sc_cin, void *packed,
                    size_t packed_bytes, vae_stream_t stream) {
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (!weight || !packed || cout <= 0 || cin <= 0 || sc_cin < 0 || (sc_w && sc_cin <= 0) ||
      (!sc_w && (sc_b || sc_cin)))
    return VAE_EINVAL;
  if (k != 1 && k != 3) return VAE_EUNSUPPORTED;
  if (cin > 4096 || cout > 4096 || sc_cin > 4096) return VAE_EUNSUPPORTED;
  const int ldb = packed_ldb(cin, k * k, sc_cin);
  Carver cv(packed, packed_bytes);
  ConvPack p = carve_pack(cv, cout, ldb, cout);
  if (!cv.ok()) return VAE_EWORKSPACE;
  VAE_TRY(pack_conv_weights(weight, cout, cin, k * k, sc_w, sc_cin, p.w, cout, ldb, s));
  if (bias || sc_b) {
    VAE_TRY(add_bias(p.bias, bias, sc_b, cout, s));
  } else {
    VAE_CUDA_TRY(cudaMemsetAsync(p.bias, 0, static_cast<size_t>(cout) * sizeof(float), s));
  }
  return VAE_OK;
}

int vae_conv2d_packed(const float *x, int n, int cin, int h, int w, int layout,
                      const void *packed, int cout, int k, const float *residual,
                      const float *sc_x, int sc_cin, float *y, void *ws, size_t ws_bytes,
                      vae_stream_t stream) {
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (!packed || !ws || sc_cin < 0 || (sc_cin > 0) != (sc_x != nullptr)) return VAE_EINVAL;
  VAE_TRY(conv_args_ok(x, y, n, cin, h, w, layout, cout, k, residual, sc_x, sc_cin));
  Carver pc(const_cast<void *>(packed), ~size_t(0));
  const ConvPack p = carve_pack(pc, cout, packed_ldb(cin, k * k, sc_cin), cout);
  Carver cv(ws, ws_bytes);
  ConvWs cw = carve_conv(cv, n, cin, static_cast<long long>(h) * w, layout, cout, k * k, sc_cin);
  if (!cv.ok()) return VAE_EWORKSPACE;
  return conv2d_run(x, n, cin, h, w, layout, p.w, p.bias, cout, k, residual, sc_x, sc_cin, y, cw,
                    s);
}

// ------------------------------------------------------------------ upsample + conv
size_t vae_upsample_conv_workspace_size(int n, int cin, int h, int w, int layout, int cout) {
  if (n <= 0 || cin <= 0 || h <= 0 || w <= 0 || cout <= 0) return 0;
  Carver cv(nullptr, 0);
  carve_conv(cv, n, cin, static_cast<long long>(h) * w, layout, cout, kUpsamplePackTaps, 0, 4);
  return cv.used;
}

int vae_upsample_conv(const float *x, int n, int cin, int h, int w, int layout,
                      const float *weight, const float *bias, int cout, float *y, void *ws,
                      size_t ws_bytes, vae_stream_t stream) {
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (!weight || !ws) return VAE_EINVAL;
  VAE_TRY(upsample_args_ok(x, y, n, cin, h, w, layout, cout));
  Carver cv(ws, ws_bytes);
  ConvWs cw = carve_conv(cv, n, cin, static_cast<long long>(h) * w, layout, cout,
                         kUpsamplePackTaps, 0, 4);
  if (!cv.ok()) return VAE_EWORKSPACE;
  VAE_TRY(pack_upsample_weights(weight, cout, cin, cw.packed, s));
  return upsample_run(x, n, cin, h, w, layout, cw.packed, bias, cout, y, cw, s);
}

size_t vae_upsample_conv_pack_bytes(int cout, int cin) {
  if (cout <= 0 || cin <= 0) return 0;
  Carver cv(nullptr, 0);
  carve_pack(cv, 4ull * cout, upsample_ldb(cin), cout);
  return cv.used;
}

int vae_upsample_conv_pack(const float *weight, const float *bias, int cout, int cin,
                           void *packed, size_t packed_bytes, vae_stream_t stream) {
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (!weight || !packed || cout <= 0 || cin <= 0) return VAE_EINVAL;
  if (cin > 4096 || cout > 4096) return VAE_EUNSUPPORTED;
  Carver cv(packed, packed_bytes);
  ConvPack p = carve_pack(cv, 4ull * cout, upsample_ldb(cin), cout);
  if (!cv.ok()) return VAE_EWORKSPACE;
  VAE_TRY(pack_upsample_weights(weight, cout, cin, p.w, s));
  if (bias) {
    VAE_CUDA_TRY(cudaMemcpyAsync(p.bias, bias, static_cast<size_t>(cout) * sizeof(float),
                                 cudaMemcpyDeviceToDevice, s));
  } else {
    VAE_CUDA_TRY(cudaMemsetAsync(p.bias, 0, static_cast<size_t>(cout) * sizeof(float), s));
  }
  return VAE_OK;
}

int vae_upsample_conv_packed(const float *x, int n, int cin, int h, int w, int layout,
                             const void *packed, int cout, float *y, void *ws, size_t ws_bytes,
                             vae_stream_t stream) {
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (!packed || !ws) return VAE_EINVAL;
  VAE_TRY(upsample_args_ok(x, y, n, cin, h, w, layout, cout));
  Carver pc(const_cast<void *>(packed), ~size_t(0));
  const ConvPack p = carve_pack(pc, 4ull * cout, upsample_ldb(cin), cout);
  Carver cv(ws, ws_bytes);
  ConvWs cw = carve_conv(cv, n, cin, static_cast<long long>(h) * w, layout, cout,
                         kUpsamplePackTaps, 0, 4);
  if (!cv.ok()) return VAE_EWORKSPACE;
  return upsample_run(x, n, cin, h, w, layout, p.w, p.bias, cout, y, cw, s);
}

// ------------------------------------------------------------------ GroupNorm + SiLU
size_t vae_groupnorm_silu_workspace_size(int n, int c, long long spatial, int layout,
                                         int groups) {
  (void)layout;
  if (n <= 0 || c <= 0 || spatial <= 0 || groups <= 0) return 0;
  return groupnorm_ws_bytes(n, c, spatial, groups);
}

int vae_groupnorm_silu(const float *x, int n, int c, long long spatial, int layout, int groups,
                       float eps, const float *gamma, const float *beta, int apply_silu,
                       float *y, void *ws, size_t ws_bytes, vae_stream_t stream) {
  if (layout != VAE_NCHW && layout != VAE_NHWC) return VAE_EINVAL;
  if (n <= 0 || c <= 0 || spatial <= 0 || groups <= 0) return VAE_EINVAL;
  if (ws_bytes < groupnorm_ws_bytes(n, c, spatial, groups)) return VAE_EWORKSPACE;
  return groupnorm_silu(x, n, c, spatial, layout == VAE_NHWC, groups, eps, gamma, beta,
                        apply_silu != 0, 0, y, ws, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ mid attention
size_t vae_mid_attn_workspace_size(int n, int c, int h, int w, int layout) {
  if (n <= 0 || c <= 0 || h <= 0 || w <= 0) return 0;
  Carver cv(nullptr, 0);
  const size_t a = attn_ws_bytes(n, c, h * w, layout);
  cv.take<char>(a);
  return cv.used;
}

int vae_mid_attn(const float *x, int n, int c, int h, int w, int layout, int groups, float eps,
                 const float *gn_w, const float *gn_b, const float *wq, const float *bq,
                 const float *wk, const float *bk, const float *wv, const float *bv,
                 const float *wo, const float *bo, float *y, void *ws, size_t ws_bytes,
                 vae_stream_t stream) {
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (!x || !y || !ws || !gn_w || !gn_b || !wq || !bq || !wk || !bk || !wv || !bv || !wo || !bo)
    return VAE_EINVAL;
  if (n <= 0 || c <= 0 || h <= 0 || w <= 0 || groups <= 0) return VAE_EINVAL;
  if (layout != VAE_NCHW && layout != VAE_NHWC) return VAE_EINVAL;
  if (c % 32 || c > 1024 || c % groups) return VAE_EUNSUPPORTED;
  const long long Lll = static_cast<long long>(h) * w;
  if (Lll > 65536) return VAE_EUNSUPPORTED;
  const int L = static_cast<int>(Lll);
  if (!aligned16(x) || !aligned16(y)) return VAE_EINVAL;
  Carver cv(ws, ws_bytes);
  AttnWs aw = carve_attn(cv, n, c, L, layout);
  if (!cv.ok()) return VAE_EWORKSPACE;

  // Pack [Wq; Wk; Wv] and Wo (TF32-rounded, K-major rows) and [bq; bk; bv].
  const size_t cc = static_cast<size_t>(c) * c;
  VAE_TRY(pack_conv_weights(wq, c, c, 1, nullptr, 0, aw.wqkv, c, c, s));
  VAE_TRY(pack_conv_weights(wk, c, c, 1, nullptr, 0, aw.wqkv + cc, c, c, s));
  VAE_TRY(pack_conv_weights(wv, c, c, 1, nullptr, 0, aw.wqkv + 2 * cc, c, c, s));
  VAE_TRY(pack_conv_weights(wo, c, c, 1, nullptr, 0, aw.wo, c, c, s));
  VAE_CUDA_TRY(cudaMemcpyAsync(aw.bqkv, bq, c * 4, cudaMemcpyDeviceToDevice, s));
  VAE_CUDA_TRY(cudaMemcpyAsync(aw.bqkv + c, bk, c * 4, cudaMemcpyDeviceToDevice, s));
  VAE_CUDA_TRY(cudaMemcpyAsync(aw.bqkv + 2 * c, bv, c * 4, cudaMemcpyDeviceToDevice, s));

  const float *xa = x;
  float *ya = y;
  if (layout == VAE_NCHW) {
    VAE_TRY(stage_nhwc(x, n, c, L, layout, aw.xs, c, 1.f, 0.f, 0, &xa, s));
    ya = aw.y;
  }
  AttnScratch sc{aw.t, aw.qkv, aw.vt, aw.s, aw.o, aw.gn, aw.rs};
  VAE_TRY(attention_nhwc(xa, n, c, L, groups, eps, gn_w, gn_b, aw.wqkv, aw.bqkv, aw.wo, bo, ya,
                         sc, s));
  if (layout == VAE_NCHW) VAE_TRY(unstage_nchw(ya, n, c, L, y, s));
  return VAE_OK;
}

// ------------------------------------------------------------------ 3-D causal conv
size_t vae_conv3d_causal_workspace_size(int n, int cin, int t, int h, int w, int layout,
                                        int cout) {
  if (n <= 0 || cin <= 0 || t <= 0 || h <= 0 || w <= 0 || cout <= 0) return 0;
  Carver cv(nullptr, 0);
  carve_conv(cv, n, cin, static_cast<long long>(t) * h * w, layout, cout, 27, 0);
  return cv.used;
}

int vae_conv3d_causal(const float *x, int n, int cin, int t, int h, int w, int layout,
                      const float *weight, const float *bias, int cout, const float *residual,
                      float *y, void *ws, size_t ws_bytes, vae_stream_t stream) {
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (!x || !weight || !y || !ws || n <= 0 || cin <= 0 || t <= 0 || h <= 0 || w <= 0 ||
      cout <= 0)
    return VAE_EINVAL;
  if (layout != VAE_NCHW && layout != VAE_NHWC) return VAE_EINVAL;
  if (cin > 4096 || cout > 4096 || h > 65535 || w > 65535 || static_cast<long long>(n) * t > 65535)
    return VAE_EUNSUPPORTED;
  if (!aligned16(x) || !aligned16(y) || (residual && !aligned16(residual))) return VAE_EINVAL;
  if (layout == VAE_NHWC && cout % 4) return VAE_EUNSUPPORTED;
  const long long spatial = static_cast<long long>(t) * h * w;
  Carver cv(ws, ws_bytes);
  ConvWs cw = carve_conv(cv, n, cin, spatial, layout, cout, 27, 0);
  if (!cv.ok()) return VAE_EWORKSPACE;
  const int ldb = packed_ldb(cin, 27, 0);
  VAE_TRY(pack_conv_weights(weight, cout, cin, 27, nullptr, 0, cw.packed, cout, ldb, s));
  const float *xa = nullptr;
  VAE_TRY(stage_nhwc(x, n, cin, spatial, layout, cw.xs, round_up32(cin), 1.f, 0.f, 0, &xa, s));
  IgemmDesc d;
  d.mode = AMode::Conv;
  d.a = xa;
  d.imgs = n * t;
  d.t = t;
  d.hin = h;
  d.win = w;
  d.a_c = round_up32(cin);
  d.k = 3;
  d.kt = 3;
  d.b = cw.packed;
  d.ldb = ldb;
  d.cout = cout;
  d.out = y;
  d.ldo = cout;
  d.out_nchw = layout == VAE_NCHW;
  d.bias = bias;
  d.residual = residual;
  d.split_ws = cw.split;
  d.split_ws_floats = cw.split_floats;
  return igemm_launch(d, s);
}

// ------------------------------------------------------------------ 3-D causal stack
size_t vae_causal_stack_workspace_size(int n, int c, int t, int h, int w, int layout,
                                       int n_layers) {
  if (n <= 0 || c <= 0 || t <= 0 || h <= 0 || w <= 0 || n_layers <= 0) return 0;
  Carver cv(nullptr, 0);
  carve_stack(cv, n, c, static_cast<long long>(t) * h * w, layout, n_layers, c);
  return cv.used;
}

int vae_causal_stack(const float *x, int n, int c, int t, int h, int w, int layout,
                     int n_layers, const float *const *weight, const float *const *bias,
                     const float *const *gn_w, const float *const *gn_b, int groups, float eps,
                     float *y, void *ws, size_t ws_bytes, vae_stream_t stream) {
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (!x || !y || !ws || !weight || !bias || !gn_w || !gn_b || n <= 0 || c <= 0 || t <= 0 ||
      h <= 0 || w <= 0 || groups <= 0 || n_layers <= 0)
    return VAE_EINVAL;
  if (layout != VAE_NCHW && layout != VAE_NHWC) return VAE_EINVAL;
  if (n_layers > 64 || c % 32 || c % groups || c > 1024 || h > 65535 || w > 65535 ||
      static_cast<long long>(n) * t > 65535)
    return VAE_EUNSUPPORTED;
  for (int i = 0; i < n_layers; ++i)
    if (!weight[i] || !gn_w[i] || !gn_b[i]) return VAE_EINVAL;
  if (!aligned16(x) || !aligned16(y) || x == y) return VAE_EINVAL;
  const long long vox = static_cast<long long>(t) * h * w;
  Carver cv(ws, ws_bytes);
  // groups <= c, so carving with c groups is an upper bound
  StackWs sw = carve_stack(cv, n, c, vox, layout, n_layers, c);
  if (!cv.ok()) return VAE_EWORKSPACE;
  const int ldb = packed_ldb(c, 27, 0);
  for (int i = 0; i < n_layers; ++i)
    VAE_TRY(pack_conv_weights(weight[i], c, c, 27, nullptr, 0,
                              sw.packed + static_cast<size_t>(i) * c * ldb, c, ldb, s));
  const float *u0 = nullptr;
  VAE_TRY(stage_nhwc(x, n, c, vox, layout, sw.xs, c, 1.f, 0.f, 0, &u0, s));
  std::vector<const float *> u(n_layers + 1);
  u[0] = u0;
  for (int i = 1; i <= n_layers; ++i) {
    IgemmDesc d;
    d.mode = AMode::Conv;
    d.a = u[i - 1];
    d.imgs = n * t;
    d.t = t;
    d.hin = h;
    d.win = w;
    d.a_c = c;
    d.k = 3;
    d.kt = 3;
    d.b = sw.packed + static_cast<size_t>(i - 1) * c * ldb;
    d.ldb = ldb;
    d.cout = c;
    d.out = sw.h;
    d.ldo = c;
    d.bias = bias[i - 1];
    VAE_TRY(igemm_launch(d, s));
    // u_i goes to a ring buffer holding neither u_{i-1} nor u_{i-2}; the last
    // layer writes the caller's y directly when y is NDHWC.
    float *dst = nullptr;
    if (i == n_layers && layout == VAE_NHWC) {
      dst = y;
    } else {
      for (float *cand : sw.ring)
        if (cand != u[i - 1] && (i < 2 || cand != u[i - 2])) {
          dst = cand;
          break;
        }
    }
    const float *res = (i % 2 == 0) ? u[i - 2] : nullptr;
    VAE_TRY(groupnorm_silu(sw.h, n, c, vox, 1, groups, eps, gn_w[i - 1], gn_b[i - 1], 1,
                           i < n_layers ? 1 : 0, dst, sw.gn, s, res));
    u[i] = dst;
  }
  if (layout == VAE_NCHW) VAE_TRY(unstage_nchw(u[n_layers], n, c, vox, y, s));
  return VAE_OK;
}

}  // extern "C"
