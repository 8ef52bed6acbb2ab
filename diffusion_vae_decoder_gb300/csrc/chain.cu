// chain.cu -- the whole decoder as one device-resident chain.
//
// cortiq-engine "Module vae": VaeChainArgs lists the decoder in execution
// order (conv_in -> mid_res1 -> mid_attn -> mid_res2 -> ups[..] ->
// norm_out+SiLU -> conv_out) and carries a stable key so a backend uploads
// the weights once; VaeDecoder adds the latent de-normalisation
// z / scaling_factor + shift_factor. "VAE decode -> GPU handoff", step 3:
// activations stay on the device and only the RGB image comes back.
//
// vae_chain_prepare packs every weight once into GEMM layout (TF32-rounded,
// and unrounded as well unless the chain is TF32-only; each resnet's 1x1
// shortcut appended to conv2's reduction with the summed bias) and returns
// the handle that plays the role of that key. A decode whose products are
// split-TF32 (vae_precision) keeps its activations in FP32 instead of storing
// the MMA operands TF32-rounded.
// vae_decode_chain then walks the chain on the caller's stream with no host
// synchronisation, ping-ponging NHWC activations through the workspace:
//   X, Y  the residual stream (a resnet without a shortcut updates it in
//         place: conv2's epilogue adds the skip element by element)
//   T     GroupNorm+SiLU output (TF32-rounded: it is the next conv's operand)
//   H     conv1 output
// plus the latent staging buffer, the GroupNorm partials that conv epilogues
// write with the per-group arrival counters of their finalize (zeroed at the
// start of every decode), the split-K area and the attention scratch.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_set>
#include <vector>

#include "common.cuh"
#include "ops.cuh"

namespace vae {

namespace {

// Registry of live handles: entry points check a handle here instead of
// reading through it, so a destroyed handle is rejected without touching
// freed memory.
std::mutex g_live_mu;
std::unordered_set<const void *> g_live;

bool is_live(const void *h) {
  if (!h) return false;
  std::lock_guard<std::mutex> lk(g_live_mu);
  return g_live.count(h) != 0;
}

// Copies each step's output into the caller's trace buffers (in order).
struct Tracer {
  float *const *bufs = nullptr;
  int n = 0;
  int idx = 0;
  int status = VAE_OK;
  void emit(const void *src, size_t bytes, cudaStream_t s) {
    if (idx < n && bufs[idx] &&
        cudaMemcpyAsync(bufs[idx], src, bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      status = VAE_ECUDA;
    ++idx;
  }
};

struct ConvW {
  float *w = nullptr, *b = nullptr;
  float *w_exact = nullptr;  // the same pack unrounded (split-TF32 products)
  int cin = 0, cout = 0, k = 0, ldb = 0, sc_cin = 0;
  int kt = 1;  // time taps: 3 for the causal 3x3x3 convs of the 3-D decoder
};
struct NormW {
  float *g = nullptr, *b = nullptr;
  int c = 0;
};
struct ResW {
  NormW n1, n2;
  ConvW c1, c2;  // c2 carries the shortcut (sc_cin > 0) when present
};
struct AttnW {
  NormW n;
  float *wqkv = nullptr, *bqkv = nullptr, *wo = nullptr, *bo = nullptr;
  float *wqkv_exact = nullptr, *wo_exact = nullptr;  // unrounded (split-TF32)
  int c = 0;
};
struct UpW {
  std::vector<ResW> res;
  bool has_up = false;
  ConvW up;
};

// Per-step CUDA-event profiler (enabled through vae_chain_profile).
struct Profiler {
  struct Rec {
    vae_prof_record r;
    int ev0, ev1;
    long long launches0;
  };
  bool on = false;
  std::vector<cudaEvent_t> events;
  std::vector<Rec> recs;
  int next = 0;

  int event(cudaStream_t s) {
    if (next == static_cast<int>(events.size())) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return -1;
      events.push_back(e);
    }
    // Inside a stream capture an external record becomes an event-record
    // node of the graph, so every replay re-records it; outside one that
    // flag is refused (and would linger as the thread's last error), so a
    // plain record.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return -1;
    const cudaError_t e = cap == cudaStreamCaptureStatusActive
                              ? cudaEventRecordWithFlags(events[next], s, cudaEventRecordExternal)
                              : cudaEventRecord(events[next], s);
    if (e != cudaSuccess) return -1;
    return next++;
  }
  // Opens a step; returns its record index, or -1 when profiling is off.
  int open(int kind, double flops, double bytes, cudaStream_t s) {
    if (!on) return -1;
    Rec rec{};
    rec.r.kind = kind;
    rec.r.flops = flops;
    rec.r.bytes = bytes;
    rec.launches0 = launch_count();
    rec.ev0 = event(s);
    rec.ev1 = -1;
    recs.push_back(rec);
    return static_cast<int>(recs.size()) - 1;
  }
  void close(int idx, cudaStream_t s) {
    if (idx < 0) return;
    recs[idx].ev1 = event(s);
    recs[idx].r.kernels = static_cast<int>(launch_count() - recs[idx].launches0);
  }
  void reset() {
    recs.clear();
    next = 0;
  }
  ~Profiler() {
    for (cudaEvent_t e : events) cudaEventDestroy(e);
  }
};

struct Chain {
  Profiler prof;
  Tracer *tr = nullptr;  // set for the duration of a traced decode
  // 3-D causal decoder (vae_causal_decoder_prepare): causal 3x3x3 convs, no
  // attention, mid resnets in mid3, nearest-2x spatial upsample materialised
  // before each upsample conv; `frames` is the current decode's frame count
  // (1 for the 2-D decoder).
  bool causal = false;
  std::vector<ResW> mid3;
  int frames = 1;
  int precision = VAE_PRECISION_TF32;
  bool exact = false;  // this decode forms split-TF32 products (set per decode)
  int device = 0;
  int latent_c = 0, groups = 32;
  float eps = 1e-6f, sf = 1.f, sh = 0.f;
  ConvW conv_in, conv_out;
  ResW mid1, mid2;
  AttnW attn;
  std::vector<UpW> ups;
  NormW norm_out;
  float *head_w = nullptr;  // conv_out packed for the fused CUDA-core head (cout <= 4)
  float *head_tc_w = nullptr;  // conv_out packed for the tensor-core head (TF32 decodes)
  std::vector<void *> allocs;
  // GroupNorm ahead (igemm_gn_ahead_ok): the current decode's row flags and
  // per-conv row counters (zeroed at its start), and how many such convs it
  // has launched (conv i uses counter i and flag value i + 1).
  int *ga_flags = nullptr, *ga_next = nullptr;
  int ga_idx = 0;
};
constexpr int kMaxGnAheadConvs = 64;

struct Builder {
  Chain *ch;
  cudaStream_t s;
  std::vector<void *> temps;
  int status = VAE_OK;

  template <class T>
  T *dev(size_t count) {
    void *p = nullptr;
    if (status != VAE_OK) return nullptr;
    if (take_alloc_failure() ||
        cudaMalloc(&p, std::max<size_t>(count, 1) * sizeof(T)) != cudaSuccess) {
      status = VAE_ENOMEM;
      return nullptr;
    }
    ch->allocs.push_back(p);
    return static_cast<T *>(p);
  }
  const float *upload_tmp(const float *src, size_t count) {
    void *p = nullptr;
    if (status != VAE_OK) return nullptr;
    if (!src) {
      status = VAE_EINVAL;
      return nullptr;
    }
    if (take_alloc_failure() || cudaMalloc(&p, count * sizeof(float)) != cudaSuccess) {
      status = VAE_ENOMEM;
      return nullptr;
    }
    temps.push_back(p);
    if (cudaMemcpyAsync(p, src, count * sizeof(float), cudaMemcpyDefault, s) != cudaSuccess)
      status = VAE_ECUDA;
    return static_cast<const float *>(p);
  }
  float *upload(const float *src, size_t count) {
    float *p = dev<float>(count);
    if (status != VAE_OK) return nullptr;
    if (!src) {
      status = VAE_EINVAL;
      return nullptr;
    }
    if (cudaMemcpyAsync(p, src, count * sizeof(float), cudaMemcpyDefault, s) != cudaSuccess)
      status = VAE_ECUDA;
    return p;
  }
  void fail(int st) {
    if (status == VAE_OK) status = st;
  }

  NormW norm(const vae_norm_ref &r, int c) {
    NormW n;
    if (r.c != c || c % ch->groups) fail(VAE_EINVAL);
    n.c = c;
    n.g = upload(r.weight, c);
    n.b = upload(r.bias, c);
    return n;
  }
  // Conv (optionally with the 1x1 shortcut appended to its reduction).
  // kt = 3: a causal 3x3x3 conv, weight [cout][cin][3][3][3].
  ConvW conv(const vae_conv_ref &r, int cin, int cout, const vae_conv_ref *sc = nullptr,
             int kt = 1) {
    ConvW c;
    if (r.cin != cin || r.cout != cout || !(r.k == 1 || r.k == 3)) fail(VAE_EINVAL);
    const bool has_sc = sc && sc->weight;
    if (has_sc && (sc->k != 1 || sc->cout != cout)) fail(VAE_EINVAL);
    if (status != VAE_OK) return c;
    c.cin = cin;
    c.cout = cout;
    c.k = r.k;
    c.kt = kt;
    c.sc_cin = has_sc ? sc->cin : 0;
    const int taps = r.k * r.k * kt;
    c.ldb = packed_ldb(cin, taps, c.sc_cin);
    const float *wt = upload_tmp(r.weight, static_cast<size_t>(cout) * cin * taps);
    const float *wsc = has_sc ? upload_tmp(sc->weight, static_cast<size_t>(cout) * c.sc_cin)
                              : nullptr;
    c.w = dev<float>(static_cast<size_t>(cout) * c.ldb);
    if (ch->precision != VAE_PRECISION_TF32)
      c.w_exact = dev<float>(static_cast<size_t>(cout) * c.ldb);
    if (status != VAE_OK) return c;
    fail(pack_conv_weights(wt, cout, cin, taps, wsc, c.sc_cin, c.w, cout, c.ldb, s));
    if (c.w_exact)
      fail(pack_conv_weights(wt, cout, cin, taps, wsc, c.sc_cin, c.w_exact, cout, c.ldb, s, 0));
    if (has_sc) {
      const float *b1 = r.bias ? upload_tmp(r.bias, cout) : nullptr;
      const float *b2 = sc->bias ? upload_tmp(sc->bias, cout) : nullptr;
      c.b = dev<float>(cout);
      if (status == VAE_OK) fail(add_bias(c.b, b1, b2, cout, s));
    } else if (r.bias) {
      c.b = upload(r.bias, cout);
    }
    return c;
  }
  // Upsample conv: 3x3 weights packed as four parity-specific 2x2 kernels
  // (k = 2 in the returned ConvW: 4 taps per output pixel).
  ConvW upconv(const vae_conv_ref &r, int cin, int cout) {
    ConvW c;
    if (r.cin != cin || r.cout != cout || r.k != 3) fail(VAE_EINVAL);
    if (status != VAE_OK) return c;
    c.cin = cin;
    c.cout = cout;
    c.k = 2;
    c.ldb = upsample_ldb(cin);
    const float *wt = upload_tmp(r.weight, static_cast<size_t>(cout) * cin * 9);
    c.w = dev<float>(4ull * cout * c.ldb);
    if (ch->precision != VAE_PRECISION_TF32) c.w_exact = dev<float>(4ull * cout * c.ldb);
    if (status != VAE_OK) return c;
    fail(pack_upsample_weights(wt, cout, cin, c.w, s));
    if (c.w_exact) fail(pack_upsample_weights(wt, cout, cin, c.w_exact, s, 0));
    if (r.bias) c.b = upload(r.bias, cout);
    return c;
  }
  ResW resnet(const vae_resnet_ref &r, int cin, int cout, int kt = 1) {
    ResW w;
    if ((cin != cout) != (r.shortcut.weight != nullptr)) fail(VAE_EINVAL);
    w.n1 = norm(r.norm1, cin);
    w.c1 = conv(r.conv1, cin, cout, nullptr, kt);
    w.n2 = norm(r.norm2, cout);
    w.c2 = conv(r.conv2, cout, cout, &r.shortcut, kt);
    if (w.c2.sc_cin && w.c2.sc_cin != cin) fail(VAE_EINVAL);
    if (w.c1.k != 3 || w.c2.k != 3) fail(VAE_EINVAL);
    return w;
  }
  AttnW attention(const vae_attn_ref &r, int c) {
    AttnW a;
    a.c = c;
    if (c % 32) fail(VAE_EUNSUPPORTED);
    a.n = norm(r.norm, c);
    const vae_conv_ref *p[3] = {&r.q, &r.k, &r.v};
    const bool exact = ch->precision != VAE_PRECISION_TF32;
    a.wqkv = dev<float>(3ull * c * c);
    if (exact) a.wqkv_exact = dev<float>(3ull * c * c);
    a.bqkv = dev<float>(3ull * c);
    for (int i = 0; i < 3 && status == VAE_OK; ++i) {
      if (p[i]->cin != c || p[i]->cout != c || p[i]->k != 1) fail(VAE_EINVAL);
      const float *wt = upload_tmp(p[i]->weight, static_cast<size_t>(c) * c);
      if (status != VAE_OK) break;
      fail(pack_conv_weights(wt, c, c, 1, nullptr, 0, a.wqkv + static_cast<size_t>(i) * c * c,
                             c, c, s));
      if (exact)
        fail(pack_conv_weights(wt, c, c, 1, nullptr, 0,
                               a.wqkv_exact + static_cast<size_t>(i) * c * c, c, c, s, 0));
      if (!p[i]->bias) fail(VAE_EINVAL);
      if (status == VAE_OK &&
          cudaMemcpyAsync(a.bqkv + i * c, p[i]->bias, c * 4, cudaMemcpyDefault, s) != cudaSuccess)
        fail(VAE_ECUDA);
    }
    if (r.out.cin != c || r.out.cout != c || r.out.k != 1) fail(VAE_EINVAL);
    const float *wo = upload_tmp(r.out.weight, static_cast<size_t>(c) * c);
    a.wo = dev<float>(static_cast<size_t>(c) * c);
    if (exact) a.wo_exact = dev<float>(static_cast<size_t>(c) * c);
    if (status == VAE_OK) fail(pack_conv_weights(wo, c, c, 1, nullptr, 0, a.wo, c, c, s));
    if (status == VAE_OK && exact)
      fail(pack_conv_weights(wo, c, c, 1, nullptr, 0, a.wo_exact, c, c, s, 0));
    a.bo = upload(r.out.bias, c);
    return a;
  }
};

// Sizes of the ping-pong buffers for one decode.
struct Plan {
  size_t max_elems = 0;  // largest activation (n * H * W * C) of the chain
  int max_c = 0;
  int attn_c = 0, attn_l = 0;
  long long max_slots = 0;  // GroupNorm partial slots of the largest producer conv
  long long max_rows = 0;   // n * H of the tallest activation
};

long long stat_slots_of(AMode mode, int hin, int win, int cout) {
  IgemmDesc d;
  d.mode = mode;
  d.hin = hin;
  d.win = win;
  d.cout = cout;
  return igemm_stat_slots(d);
}

Plan make_plan(const Chain &ch, int n, int h, int w) {
  Plan p;
  auto see = [&](long long hh, long long ww, int c) {
    p.max_elems = std::max(p.max_elems, static_cast<size_t>(n * hh * ww * c));
    p.max_rows = std::max(p.max_rows, n * hh);
    p.max_c = std::max(p.max_c, c);
    p.max_slots = std::max(p.max_slots, stat_slots_of(AMode::Conv, static_cast<int>(hh),
                                                      static_cast<int>(ww), c));
  };
  long long hh = h, ww = w;
  see(hh, ww, ch.conv_in.cout);
  p.attn_c = ch.attn.c;
  p.attn_l = static_cast<int>(hh * ww);
  for (const UpW &u : ch.ups) {
    for (const ResW &r : u.res) {
      see(hh, ww, r.c1.cin);
      see(hh, ww, r.c1.cout);
    }
    if (u.has_up) {
      p.max_slots = std::max(p.max_slots, stat_slots_of(AMode::Upsample, static_cast<int>(hh),
                                                        static_cast<int>(ww), u.up.cout));
      hh *= 2;
      ww *= 2;
      see(hh, ww, u.up.cout);
    }
  }
  return p;
}

struct DecodeWs {
  float *lat, *X, *Y, *T, *H;
  float *ss;    // GroupNorm scale / shift for the fused head
  float *part;  // GroupNorm partials written by the producer conv's epilogue
  float *split; // split-K partial sums of the low-resolution convs
  unsigned *gn_cnt;  // per-(sample, group) arrival counters of the GroupNorm finalize
  int *ga_next, *ga_flags;  // GroupNorm-ahead counters and row flags (right after gn_cnt)
  size_t zero_bytes;        // gn_cnt .. ga_flags, zeroed at the start of a decode
  AttnScratch attn;
  void *gn;
};

// Whether `part` currently holds the statistics of the tensor about to be
// normalised, and with how many slots per (sample, group).
struct Stats {
  bool ready = false;
  long long slots = 0;
};

DecodeWs carve_decode(Carver &cv, const Chain &ch, const Plan &p, int n, int h, int w) {
  DecodeWs d{};
  d.lat = cv.take<float>(static_cast<size_t>(n) * h * w * round_up32(ch.latent_c));
  d.X = cv.take<float>(p.max_elems);
  d.Y = cv.take<float>(p.max_elems);
  d.T = cv.take<float>(p.max_elems);
  d.H = cv.take<float>(p.max_elems);
  d.ss = cv.take<float>(2ull * n * std::max(p.max_c, ch.norm_out.c));
  d.split = cv.take<float>(kSplitWsFloats);
  // slots: the largest tile-based count, and at least the 1024 CTAs a split-K
  // reduce may use
  d.part = cv.take<float>(static_cast<size_t>(n) * ch.groups * std::max(1024ll, p.max_slots) * 3);
  d.gn_cnt = cv.take<unsigned>(static_cast<size_t>(n) * ch.groups);
  d.ga_next = cv.take<int>(kMaxGnAheadConvs);
  d.ga_flags = cv.take<int>(static_cast<size_t>(std::max(1ll, p.max_rows)));
  d.zero_bytes = static_cast<size_t>(reinterpret_cast<char *>(d.ga_flags + std::max(1ll, p.max_rows)) -
                                     reinterpret_cast<char *>(d.gn_cnt));
  const size_t nl = static_cast<size_t>(n) * p.attn_l;
  const size_t lp = static_cast<size_t>(round_up32(p.attn_l));
  const int c = p.attn_c;
  d.attn.t = cv.take<float>(nl * c);
  d.attn.qkv = cv.take<float>(nl * 3 * c);
  d.attn.vt = cv.take<float>(static_cast<size_t>(c) * lp);
  d.attn.s = cv.take<float>(static_cast<size_t>(p.attn_l) * lp);
  d.attn.o = cv.take<float>(nl * c);
  d.attn.rs = cv.take<float>(attn_rs_floats(p.attn_l));
  d.gn = cv.take<char>(groupnorm_ws_bytes(n, p.max_c, 1, ch.groups));
  d.attn.gn = d.gn;
  return d;
}

// RAII bracket of one profiled step.
struct Step {
  Profiler &p;
  cudaStream_t s;
  int idx;
  Step(Profiler &prof, int kind, double flops, double bytes, cudaStream_t st)
      : p(prof), s(st), idx(prof.open(kind, flops, bytes, st)) {}
  ~Step() { p.close(idx, s); }
};

// How a conv gets its GroupNorm+SiLU input (run_gn_for): `act` is the
// tensor it reads; with `fold` the kernel applies the affine (scale, shift)
// to its halo itself, with `ahead` it makes `act` from x while it runs.
struct GnIn {
  const float *act = nullptr;
  const float *scale = nullptr, *shift = nullptr, *x = nullptr;
  bool fold = false, ahead = false;
};

double conv_flops(const ConvW &c, long long out_pixels) {
  return 2.0 * out_pixels * c.cout * (static_cast<double>(c.cin) * c.k * c.k + c.sc_cin);
}

int run_conv(Chain &ch, const ConvW &c, const float *in, int n, int h, int w,
             const float *sc_in, const float *residual, float *out, int round_out,
             cudaStream_t s, bool upsample = false, bool nchw_out = false,
             Stats *st = nullptr, float *part = nullptr, int groups = 0,
             float *split = nullptr, const GnIn *gin = nullptr) {
  const long long in_px = static_cast<long long>(n) * ch.frames * h * w;
  const long long out_px = in_px * (upsample ? 4 : 1);
  // algorithmic bytes: the input, the output, a residual and a shortcut
  // input, each moved once
  const double bytes = 4.0 * (static_cast<double>(in_px) * c.cin + out_px * c.cout +
                              (residual ? static_cast<double>(out_px) * c.cout : 0.0) +
                              (c.sc_cin ? static_cast<double>(out_px) * c.sc_cin : 0.0));
  Step step(ch.prof, upsample ? VAE_PROF_UPSAMPLE_CONV : VAE_PROF_CONV3X3,
            conv_flops(c, out_px), bytes, s);
  IgemmDesc d;
  d.mode = upsample ? AMode::Upsample : AMode::Conv;
  d.a = in;
  d.imgs = n * ch.frames;  // one image per frame
  d.t = ch.frames;
  d.kt = c.kt;
  d.hin = h;
  d.win = w;
  d.a_c = round_up32(c.cin);
  d.k = c.k;
  d.sc = c.sc_cin ? sc_in : nullptr;
  d.sc_c = c.sc_cin ? round_up32(c.sc_cin) : 0;
  d.b = ch.exact ? c.w_exact : c.w;
  d.precise = ch.exact ? 1 : 0;
  d.ldb = c.ldb;
  d.cout = c.cout;
  d.out = out;
  d.ldo = c.cout;
  d.out_nchw = nchw_out;
  d.bias = c.b;
  d.residual = residual;
  d.round_out = ch.exact ? 0 : round_out;  // split-TF32 operands stay FP32
  d.split_ws = split;
  d.split_ws_floats = split ? kSplitWsFloats : 0;
  if (gin && gin->fold) {  // the input's GroupNorm+SiLU, applied in the kernel
    d.gn_scale = gin->scale;
    d.gn_shift = gin->shift;
  }
  const bool ahead = gin && gin->ahead;
  if (ahead) {  // `in` made by the launch itself from gin->x
    d.ga_x = gin->x;
    d.ga_scale = gin->scale;
    d.ga_shift = gin->shift;
    d.ga_flags = ch.ga_flags;
    d.ga_next = ch.ga_next + ch.ga_idx;
    d.ga_epoch = ch.ga_idx + 1;
  }
  int fused = 0;
  long long slots = 0;
  if (st) {
    d.stat_part = part;
    d.stat_groups = groups;
    d.stat_ok = &fused;
    d.stat_slots = &slots;
  }
  int rc = igemm_launch(d, s);
  if (ahead && rc == VAE_OK) ++ch.ga_idx;
  if (ahead && rc == VAE_EUNSUPPORTED) {  // another path: the separate apply pass first
    VAE_TRY(groupnorm_apply(gin->x, n, c.cin, in_px / n, gin->scale, gin->shift, 1, 1,
                            const_cast<float *>(in), s));
    d.ga_x = nullptr;
    rc = igemm_launch(d, s);
  }
  if (st) {
    st->ready = rc == VAE_OK && fused && slots > 0;
    st->slots = st->ready ? slots : 0;
  }
  return rc;
}

// One resnet on NHWC data: `in` [n,h,w,cin] -> `out` [n,h,w,cout]; out == in
// is allowed when there is no shortcut.
// GroupNorm+SiLU of `in` into `out` (TF32-rounded: the next conv's operand).
// With statistics fused into the producer conv only the finalize and apply
// passes run (8 bytes per element); otherwise the two-pass kernels (12).
int run_gn(Chain &ch, const NormW &nw, const float *in, int n, long long sp, float *out,
           const DecodeWs &ws, const Stats &stats, cudaStream_t s) {
  Step step(ch.prof, VAE_PROF_GROUPNORM, 0, (stats.ready ? 8.0 : 12.0) * n * sp * nw.c, s);
  if (stats.ready)
    return groupnorm_from_partials(in, n, nw.c, sp, ch.groups, ch.eps, nw.g, nw.b, 1, !ch.exact,
                                   ws.part,
                                   stats.slots, out, ws.gn, s, nullptr, ws.gn_cnt);
  return groupnorm_silu(in, n, nw.c, sp, 1, ch.groups, ch.eps, nw.g, nw.b, 1, !ch.exact, out,
                        ws.gn, s);
}

// Whether conv `c` over w-pixel rows applies its input's GroupNorm+SiLU
// itself (on the halo it stages; opt-in, see igemm_input_gn_ok), so that
// only the normalisation's per-(sample, channel) affine is computed
// beforehand.
bool gn_folds_into(const Chain &ch, const ConvW &c, int w) {
  IgemmDesc d;
  d.mode = AMode::Conv;
  d.k = c.k;
  d.kt = c.kt;
  d.win = w;
  d.cout = c.cout;
  d.sc_c = c.sc_cin;
  d.precise = ch.exact ? 1 : 0;
  return igemm_input_gn_ok(d);
}

// VAE_HEAD=cuda keeps TF32 decodes on the CUDA-core head (comparisons).
bool head_tc_enabled() {
  static const bool v = [] {
    const char *e = std::getenv("VAE_HEAD");
    return !(e && std::strcmp(e, "cuda") == 0);
  }();
  return v;
}

// Whether a decode (exact: with split-TF32 products) runs norm_out + conv_out
// as the fused tensor-core head, or as one of the fused heads at all.
bool uses_tc_head(const Chain &ch, bool exact) {
  return !exact && ch.head_tc_w && head_tc_enabled();
}
bool uses_fused_head(const Chain &ch, bool exact) {
  return uses_tc_head(ch, exact) || ch.head_w != nullptr;
}

// Whether the decode of an [n, *, h, w] latent forms split-TF32 products.
bool decode_exact(const Chain &ch, int n, int h, int w);

// Whether conv `c` (input rows w pixels wide) makes its GroupNorm+SiLU input
// itself while it runs (GroupNorm ahead).
bool gn_ahead_into(const Chain &ch, const ConvW &c, int w) {
  if (!ch.ga_flags || ch.ga_idx >= kMaxGnAheadConvs || ch.exact || ch.frames != 1) return false;
  IgemmDesc d;
  d.mode = AMode::Conv;
  d.k = c.k;
  d.kt = c.kt;
  d.win = w;
  d.cout = c.cout;
  d.sc_c = c.sc_cin;
  d.a_c = round_up32(c.cin);
  return igemm_gn_ahead_ok(d);
}

// The GroupNorm+SiLU of `in` that conv `c` reads: applied here into ws.T, or
// reduced to its per-(sample, channel) affine in ws.ss for the conv to apply
// (fold) or to make ws.T with while it runs (ahead). A trace receives the
// normalised tensor here, or after the conv when the conv makes it.
int run_gn_for(Chain &ch, const NormW &nw, const ConvW &c, const float *in, int n, int w,
               long long sp, const DecodeWs &ws, const Stats &st, GnIn *g, cudaStream_t s) {
  *g = GnIn{};
  g->act = in;
  const size_t bytes = 4ull * n * sp * nw.c;
  const bool fold = gn_folds_into(ch, c, w);
  const bool ahead = !fold && gn_ahead_into(ch, c, w);
  if (!fold && !ahead) {
    VAE_TRY(run_gn(ch, nw, in, n, sp, ws.T, ws, st, s));
    if (ch.tr) ch.tr->emit(ws.T, bytes, s);
    g->act = ws.T;
    return VAE_OK;
  }
  float *sc = ws.ss, *sh = ws.ss + static_cast<size_t>(n) * nw.c;
  {
    // bytes: the statistics pass over the input when they were not fused
    // into its producer, else only the partials
    Step step(ch.prof, VAE_PROF_GN_AFFINE, 0,
              st.ready ? 12.0 * n * ch.groups * st.slots : 4.0 * n * sp * nw.c, s);
    VAE_TRY(groupnorm_scale_shift(in, n, nw.c, sp, ch.groups, ch.eps, nw.g, nw.b,
                                  st.ready ? ws.part : nullptr, st.slots, sc, sh, ws.gn, s,
                                  ws.gn_cnt));
  }
  g->scale = sc;
  g->shift = sh;
  if (ahead) {
    g->ahead = true;
    g->x = in;
    g->act = ws.T;
    return VAE_OK;
  }
  g->fold = true;
  if (ch.tr) {
    VAE_TRY(groupnorm_apply(in, n, nw.c, sp, sc, sh, 1, !ch.exact, ws.T, s));
    ch.tr->emit(ws.T, bytes, s);
  }
  return VAE_OK;
}

// One resnet on NHWC data; `st` holds the statistics of `in` on entry and
// those of `out` on return.
int run_resnet(Chain &ch, const ResW &r, const float *in, float *out, const DecodeWs &ws, int n,
               int h, int w, int round_out, Stats &st, cudaStream_t s) {
  const long long sp = static_cast<long long>(h) * w * ch.frames;  // GroupNorm extent
  const size_t out_bytes = 4ull * n * sp * r.c1.cout;
  const size_t in_bytes = 4ull * n * sp * r.c1.cin;
  GnIn g;
  VAE_TRY(run_gn_for(ch, r.n1, r.c1, in, n, w, sp, ws, st, &g, s));
  VAE_TRY(run_conv(ch, r.c1, g.act, n, h, w, nullptr, nullptr, ws.H, 0, s, false, false, &st,
                   ws.part, ch.groups, ws.split, &g));
  if (ch.tr && g.ahead) ch.tr->emit(g.act, in_bytes, s);
  if (ch.tr) ch.tr->emit(ws.H, out_bytes, s);
  VAE_TRY(run_gn_for(ch, r.n2, r.c2, ws.H, n, w, sp, ws, st, &g, s));
  if (r.c2.sc_cin)
    VAE_TRY(run_conv(ch, r.c2, g.act, n, h, w, in, nullptr, out, round_out, s, false, false,
                     &st, ws.part, ch.groups, ws.split, &g));
  else
    VAE_TRY(run_conv(ch, r.c2, g.act, n, h, w, nullptr, in, out, round_out, s, false, false,
                     &st, ws.part, ch.groups, ws.split, &g));
  if (ch.tr && g.ahead) ch.tr->emit(g.act, out_bytes, s);
  if (ch.tr) ch.tr->emit(out, out_bytes, s);
  return VAE_OK;
}

// The trace points of a decode, in the order decode_impl emits them.
std::vector<vae_trace_point> trace_points(const Chain &ch, int n, int h, int w) {
  std::vector<vae_trace_point> pts;
  auto add = [&](int kind, int c, int hh, int ww, int input, int skip) {
    vae_trace_point p{};
    p.kind = kind;
    p.c = c;
    p.h = hh;
    p.w = ww;
    p.input = input;
    p.skip = skip;
    p.bytes = 4ull * n * hh * ww * c;
    pts.push_back(p);
    return static_cast<int>(pts.size()) - 1;
  };
  auto resnet = [&](const ResW &r, int x, int hh, int ww) {
    const int g1 = add(VAE_TRACE_GROUPNORM, r.c1.cin, hh, ww, x, -1);
    const int c1 = add(VAE_TRACE_CONV, r.c1.cout, hh, ww, g1, -1);
    const int g2 = add(VAE_TRACE_GROUPNORM, r.c1.cout, hh, ww, c1, -1);
    return add(VAE_TRACE_RESNET, r.c1.cout, hh, ww, g2, x);
  };
  int cur = add(VAE_TRACE_LATENT, round_up32(ch.latent_c), h, w, -1, -1);
  cur = add(VAE_TRACE_CONV, ch.conv_in.cout, h, w, cur, -1);
  cur = resnet(ch.mid1, cur, h, w);
  cur = add(VAE_TRACE_ATTENTION, ch.attn.c, h, w, cur, -1);
  cur = resnet(ch.mid2, cur, h, w);
  int hh = h, ww = w;
  for (const UpW &u : ch.ups) {
    for (const ResW &r : u.res) cur = resnet(r, cur, hh, ww);
    if (u.has_up) {
      hh *= 2;
      ww *= 2;
      cur = add(VAE_TRACE_UPSAMPLE, u.up.cout, hh, ww, cur, -1);
    }
  }
  if (!uses_fused_head(ch, decode_exact(ch, n, h, w)))
    cur = add(VAE_TRACE_GROUPNORM, ch.norm_out.c, hh, ww, cur, -1);
  add(VAE_TRACE_RGB, ch.conv_out.cout, hh, ww, cur, -1);
  return pts;
}

}  // namespace

}  // namespace vae

using namespace vae;

extern "C" {

int vae_chain_prepare(const vae_chain_args *a, void **handle, vae_stream_t stream) {
  if (!a || !handle) return VAE_EINVAL;
  *handle = nullptr;
  if (a->latent_channels <= 0 || a->groups <= 0 || a->n_ups < 0 || (a->n_ups && !a->ups) ||
      a->scaling_factor == 0.f)
    return VAE_EINVAL;
  auto s = reinterpret_cast<cudaStream_t>(stream);
  Chain *ch = new Chain();
  cudaGetDevice(&ch->device);
  ch->latent_c = a->latent_channels;
  ch->groups = a->groups;
  ch->eps = a->eps;
  ch->sf = a->scaling_factor;
  ch->sh = a->shift_factor;
  if (a->precision < VAE_PRECISION_AUTO || a->precision > VAE_PRECISION_SPLIT_TF32) {
    delete ch;
    return VAE_EINVAL;
  }
  ch->precision = a->precision;
  Builder b{ch, s};
  const int c0 = a->conv_in.cout;
  ch->conv_in = b.conv(a->conv_in, a->latent_channels, c0);
  if (ch->conv_in.k != 3) b.fail(VAE_EINVAL);
  ch->mid1 = b.resnet(a->mid_res1, c0, c0);
  ch->attn = b.attention(a->mid_attn, c0);
  ch->mid2 = b.resnet(a->mid_res2, c0, c0);
  int c = c0;
  for (int i = 0; i < a->n_ups && b.status == VAE_OK; ++i) {
    const vae_up_ref &u = a->ups[i];
    UpW uw;
    if (u.n_resnets <= 0 || !u.resnets) b.fail(VAE_EINVAL);
    for (int j = 0; j < u.n_resnets && b.status == VAE_OK; ++j) {
      const int cout = u.resnets[j].conv1.cout;
      uw.res.push_back(b.resnet(u.resnets[j], c, cout));
      c = cout;
    }
    uw.has_up = u.upsample_conv.weight != nullptr;
    if (uw.has_up) {
      uw.up = b.upconv(u.upsample_conv, c, u.upsample_conv.cout);
      c = u.upsample_conv.cout;
    }
    ch->ups.push_back(std::move(uw));
  }
  ch->norm_out = b.norm(a->norm_out, c);
  ch->conv_out = b.conv(a->conv_out, c, a->conv_out.cout);
  if (ch->conv_out.k != 3 && b.status == VAE_OK) b.fail(VAE_EINVAL);
  // The fused heads: TF32 decodes run norm_out + conv_out on the tensor cores,
  // split-TF32 ones on the FP32 CUDA cores (cout <= 4); other shapes take the
  // GroupNorm pass and the implicit-GEMM conv.
  const bool cuda_head = head_supported(c, a->conv_out.cout, a->conv_out.k);
  const bool tc_head = a->conv_out.k == 3 && ch->precision != VAE_PRECISION_SPLIT_TF32 &&
                       head_tc_supported(c, a->conv_out.cout);
  if (b.status == VAE_OK && (cuda_head || tc_head)) {
    const float *wt =
        b.upload_tmp(a->conv_out.weight, static_cast<size_t>(a->conv_out.cout) * c * 9);
    if (cuda_head) {
      ch->head_w = b.dev<float>(head_packed_floats(c));
      if (b.status == VAE_OK) b.fail(head_pack_weights(wt, a->conv_out.cout, c, ch->head_w, s));
    }
    if (tc_head) {
      ch->head_tc_w = b.dev<float>(head_tc_packed_floats(c, a->conv_out.cout));
      if (b.status == VAE_OK)
        b.fail(head_tc_pack_weights(wt, a->conv_out.cout, c, ch->head_tc_w, s));
    }
  }
  if (b.status == VAE_OK && cudaStreamSynchronize(s) != cudaSuccess) b.fail(VAE_ECUDA);
  cudaStreamSynchronize(s);
  for (void *p : b.temps) cudaFree(p);
  if (b.status != VAE_OK) {
    for (void *p : ch->allocs) cudaFree(p);
    delete ch;
    return b.status;
  }
  {
    std::lock_guard<std::mutex> lk(g_live_mu);
    g_live.insert(ch);
  }
  *handle = ch;
  return VAE_OK;
}

size_t vae_chain_workspace_size(const void *handle, int n, int h, int w) {
  if (!is_live(handle) || n <= 0 || h <= 0 || w <= 0) return 0;
  const Chain *ch = static_cast<const Chain *>(handle);
  if (ch->causal) return 0;
  const Plan p = make_plan(*ch, n, h, w);
  Carver cv(nullptr, 0);
  carve_decode(cv, *ch, p, n, h, w);
  return cv.used;
}

}  // extern "C"

namespace vae {
namespace {

// Conv work of one decode (GFLOP, 2 per multiply-add at the definition's tap
// count), which the AUTO precision compares with VAE_SPLIT_AUTO_GFLOP.
double decode_conv_gflops(const Chain &ch, int n, int h, int w) {
  auto conv = [&](const ConvW &c, double px) {
    return 2.0 * px * c.cout * (static_cast<double>(c.cin) * (c.k == 2 ? 9 : c.k * c.k) + c.sc_cin);
  };
  double px = static_cast<double>(n) * h * w, f = conv(ch.conv_in, px);
  for (const ResW *r : {&ch.mid1, &ch.mid2}) f += conv(r->c1, px) + conv(r->c2, px);
  for (const UpW &u : ch.ups) {
    for (const ResW &r : u.res) f += conv(r.c1, px) + conv(r.c2, px);
    if (u.has_up) {
      px *= 4;
      f += conv(u.up, px);
    }
  }
  return (f + conv(ch.conv_out, px)) / 1e9;
}

bool decode_exact(const Chain &ch, int n, int h, int w) {
  return ch.precision == VAE_PRECISION_SPLIT_TF32 ||
         (ch.precision == VAE_PRECISION_AUTO &&
          decode_conv_gflops(ch, n, h, w) <= VAE_SPLIT_AUTO_GFLOP);
}

int decode_impl(Chain *ch, const float *z, int n, int h, int w, float *rgb, void *ws,
                size_t ws_bytes, cudaStream_t s) {
  if (ch->causal) return VAE_EINVAL;  // a 3-D causal decoder: vae_decode_causal
  ch->frames = 1;
  if (!z || !rgb || !ws || n <= 0 || h <= 0 || w <= 0) return VAE_EINVAL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != ch->device) return VAE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(z) | reinterpret_cast<uintptr_t>(rgb)) & 15) return VAE_EINVAL;
  const long long L = static_cast<long long>(h) * w;
  if (L > 65536 || static_cast<long long>(n) * L > 0x7fffffffll) return VAE_EUNSUPPORTED;
  const Plan p = make_plan(*ch, n, h, w);
  Carver cv(ws, ws_bytes);
  DecodeWs d = carve_decode(cv, *ch, p, n, h, w);
  if (!cv.ok()) return VAE_EWORKSPACE;
  ch->exact = decode_exact(*ch, n, h, w);

  // The GroupNorm finalize counters start every decode at zero (each
  // finalize leaves them at zero; this also clears what an aborted decode
  // may have left).
  // (with the GroupNorm-ahead counters and row flags right after them)
  if (cudaMemsetAsync(d.gn_cnt, 0, d.zero_bytes, s) != cudaSuccess) return VAE_ECUDA;
  ch->ga_flags = d.ga_flags;
  ch->ga_next = d.ga_next;
  ch->ga_idx = 0;
  // z / scaling_factor + shift_factor, NCHW -> NHWC (channels padded to 32).
  const float *lat = nullptr;
  {
    const int cp = round_up32(ch->latent_c);
    Step st(ch->prof, VAE_PROF_LAYOUT, 0, 4.0 * n * L * (ch->latent_c + cp), s);
    VAE_TRY(stage_nhwc(z, n, ch->latent_c, L, VAE_NCHW, d.lat, cp, 1.0f / ch->sf, ch->sh,
                       !ch->exact, &lat, s));
    if (ch->tr) ch->tr->emit(lat, 4ull * n * L * cp, s);
  }
  float *cur = d.X, *other = d.Y;
  int hh = h, ww = w;
  Stats st;
  VAE_TRY(run_conv(*ch, ch->conv_in, lat, n, hh, ww, nullptr, nullptr, cur, 0, s, false,
                   false, &st, d.part, ch->groups, d.split));
  if (ch->tr) ch->tr->emit(cur, 4ull * n * L * ch->conv_in.cout, s);
  VAE_TRY(run_resnet(*ch, ch->mid1, cur, cur, d, n, hh, ww, 0, st, s));
  {
    const double c = ch->attn.c;
    Step st(ch->prof, VAE_PROF_ATTENTION, n * (4.0 * L * L * c + 8.0 * L * c * c), 0, s);
    const AttnW &a = ch->attn;
    VAE_TRY(attention_nhwc(cur, n, a.c, static_cast<int>(L), ch->groups, ch->eps, a.n.g, a.n.b,
                           ch->exact ? a.wqkv_exact : a.wqkv, a.bqkv,
                           ch->exact ? a.wo_exact : a.wo, a.bo, cur, d.attn, s, ch->exact));
  }
  if (ch->tr) ch->tr->emit(cur, 4ull * n * L * ch->attn.c, s);
  st.ready = false;  // the attention changed `cur`
  VAE_TRY(run_resnet(*ch, ch->mid2, cur, cur, d, n, hh, ww, 0, st, s));
  for (const UpW &u : ch->ups) {
    for (size_t j = 0; j < u.res.size(); ++j) {
      const ResW &r = u.res[j];
      // The block's last resnet output is only read by the upsample conv as
      // an MMA operand, so it is stored TF32-rounded.
      const int round = (u.has_up && j + 1 == u.res.size()) ? 1 : 0;
      float *dst = r.c2.sc_cin ? other : cur;
      VAE_TRY(run_resnet(*ch, r, cur, dst, d, n, hh, ww, round, st, s));
      if (dst != cur) std::swap(cur, other);
    }
    if (u.has_up) {
      // Output rounded: the next resnet may read it through its shortcut MMA.
      VAE_TRY(run_conv(*ch, u.up, cur, n, hh, ww, nullptr, nullptr, other, 1, s, true,
                       false, &st, d.part, ch->groups, d.split));
      std::swap(cur, other);
      hh *= 2;
      ww *= 2;
      if (ch->tr) ch->tr->emit(cur, 4ull * n * hh * ww * u.up.cout, s);
    }
  }
  const long long hw = static_cast<long long>(hh) * ww;
  if (uses_fused_head(*ch, ch->exact)) {
    const int c = ch->norm_out.c, co = ch->conv_out.cout;
    Step step(ch->prof, VAE_PROF_HEAD, 2.0 * 9 * c * co * n * hw, (4.0 * c + 4.0 * co) * n * hw,
              s);
    float *scale = d.ss, *shift = d.ss + static_cast<size_t>(n) * c;
    VAE_TRY(groupnorm_scale_shift(cur, n, c, hw, ch->groups, ch->eps, ch->norm_out.g,
                                  ch->norm_out.b, st.ready ? d.part : nullptr, st.slots, scale,
                                  shift, d.gn, s, d.gn_cnt));
    if (uses_tc_head(*ch, ch->exact))
      VAE_TRY(head_tc_gn_silu_conv(cur, n, hh, ww, c, scale, shift, ch->head_tc_w,
                                   ch->conv_out.b, co, rgb, s));
    else
      VAE_TRY(head_gn_silu_conv(cur, n, hh, ww, c, scale, shift, ch->head_w, ch->conv_out.b,
                                co, rgb, s));
    if (ch->tr) ch->tr->emit(rgb, 4ull * n * hw * co, s);
    return VAE_OK;
  }
  VAE_TRY(run_gn(*ch, ch->norm_out, cur, n, hw, d.T, d, st, s));
  if (ch->tr) ch->tr->emit(d.T, 4ull * n * hw * ch->norm_out.c, s);
  VAE_TRY(run_conv(*ch, ch->conv_out, d.T, n, hh, ww, nullptr, nullptr, rgb, 0, s, false,
                   true));
  if (ch->tr) ch->tr->emit(rgb, 4ull * n * hw * ch->conv_out.cout, s);
  return VAE_OK;
}

// ---------------------------------------------------------------- 3-D causal decoder
// Activations NDHWC: [n * t frames][h][w][c], one image per frame for the
// conv kernel (whose causal taps read frames max(f + kt - 2, 0) of the same
// sample); GroupNorm statistics over (t, h, w) of each sample.
struct CausalPlan {
  size_t max_elems = 0, up_elems = 0;
  int max_c = 0;
  long long max_slots = 0;
};

long long stat_slots_frames(AMode mode, int hin, int win, int cout, int t) {
  IgemmDesc d;
  d.mode = mode;
  d.hin = hin;
  d.win = win;
  d.cout = cout;
  d.t = t;
  return igemm_stat_slots(d);
}

CausalPlan make_causal_plan(const Chain &ch, int n, int t, int h, int w) {
  CausalPlan p;
  auto see = [&](long long hh, long long ww, int c) {
    p.max_elems = std::max(p.max_elems, static_cast<size_t>(static_cast<long long>(n) * t * hh *
                                                            ww * c));
    p.max_c = std::max(p.max_c, c);
    p.max_slots = std::max(p.max_slots, stat_slots_frames(AMode::Conv, static_cast<int>(hh),
                                                          static_cast<int>(ww), c, t));
  };
  long long hh = h, ww = w;
  see(hh, ww, ch.conv_in.cout);
  for (const UpW &u : ch.ups) {
    for (const ResW &r : u.res) {
      see(hh, ww, r.c1.cin);
      see(hh, ww, r.c1.cout);
    }
    if (u.has_up) {
      p.up_elems = std::max(p.up_elems, static_cast<size_t>(static_cast<long long>(n) * t * 4 *
                                                            hh * ww * u.up.cin));
      hh *= 2;
      ww *= 2;
      see(hh, ww, u.up.cout);
    }
  }
  return p;
}

struct CausalWs {
  float *lat, *X, *Y, *T, *H, *U, *part, *split;
  unsigned *gn_cnt;
  void *gn;
};

CausalWs carve_causal(Carver &cv, const Chain &ch, const CausalPlan &p, int n, int t, int h,
                      int w) {
  CausalWs d{};
  d.lat = cv.take<float>(static_cast<size_t>(n) * t * h * w * round_up32(ch.latent_c));
  d.X = cv.take<float>(p.max_elems);
  d.Y = cv.take<float>(p.max_elems);
  d.T = cv.take<float>(p.max_elems);
  d.H = cv.take<float>(p.max_elems);
  d.U = cv.take<float>(std::max<size_t>(p.up_elems, 1));
  d.split = cv.take<float>(kSplitWsFloats);
  d.part = cv.take<float>(static_cast<size_t>(n) * ch.groups * std::max(1024ll, p.max_slots) * 3);
  d.gn_cnt = cv.take<unsigned>(static_cast<size_t>(n) * ch.groups);
  d.gn = cv.take<char>(groupnorm_ws_bytes(n, std::max(p.max_c, ch.norm_out.c), 1, ch.groups));
  return d;
}

int decode_causal_impl(Chain *ch, const float *z, int n, int t, int h, int w, float *out,
                       void *ws, size_t ws_bytes, cudaStream_t s) {
  if (!ch->causal) return VAE_EINVAL;
  if (!z || !out || !ws || n <= 0 || t <= 0 || h <= 0 || w <= 0) return VAE_EINVAL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != ch->device) return VAE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(z) | reinterpret_cast<uintptr_t>(out)) & 15) return VAE_EINVAL;
  if (static_cast<long long>(n) * t > 65535 || h > 65535 || w > 65535) return VAE_EUNSUPPORTED;
  const CausalPlan p = make_causal_plan(*ch, n, t, h, w);
  Carver cv(ws, ws_bytes);
  CausalWs d = carve_causal(cv, *ch, p, n, t, h, w);
  if (!cv.ok()) return VAE_EWORKSPACE;
  ch->frames = t;
  ch->exact = ch->precision == VAE_PRECISION_SPLIT_TF32 ||
              (ch->precision == VAE_PRECISION_AUTO &&
               decode_conv_gflops(*ch, n, h, w) * 3.0 * t <= VAE_SPLIT_AUTO_GFLOP);
  // DecodeWs view of the buffers run_resnet / run_gn use
  DecodeWs dw{};
  dw.X = d.X;
  dw.Y = d.Y;
  dw.T = d.T;
  dw.H = d.H;
  dw.part = d.part;
  dw.split = d.split;
  dw.gn_cnt = d.gn_cnt;
  dw.gn = d.gn;
  if (cudaMemsetAsync(d.gn_cnt, 0, static_cast<size_t>(n) * ch->groups * sizeof(unsigned), s) !=
      cudaSuccess)
    return VAE_ECUDA;
  ch->ga_flags = ch->ga_next = nullptr;  // (its convs have time taps: no GroupNorm ahead)
  ch->ga_idx = 0;
  const long long vox = static_cast<long long>(t) * h * w;
  const float *lat = nullptr;
  {
    const int cp = round_up32(ch->latent_c);
    Step st(ch->prof, VAE_PROF_LAYOUT, 0, 4.0 * n * vox * (ch->latent_c + cp), s);
    VAE_TRY(stage_nhwc(z, n, ch->latent_c, vox, VAE_NCHW, d.lat, cp, 1.0f / ch->sf, ch->sh,
                       !ch->exact, &lat, s));
  }
  float *cur = d.X, *other = d.Y;
  int hh = h, ww = w;
  Stats st;
  VAE_TRY(run_conv(*ch, ch->conv_in, lat, n, hh, ww, nullptr, nullptr, cur, 0, s, false, false,
                   &st, d.part, ch->groups, d.split));
  for (const ResW &r : ch->mid3) VAE_TRY(run_resnet(*ch, r, cur, cur, dw, n, hh, ww, 0, st, s));
  for (const UpW &u : ch->ups) {
    for (size_t j = 0; j < u.res.size(); ++j) {
      const ResW &r = u.res[j];
      const int round = (u.has_up && j + 1 == u.res.size()) ? 1 : 0;
      float *dst = r.c2.sc_cin ? other : cur;
      VAE_TRY(run_resnet(*ch, r, cur, dst, dw, n, hh, ww, round, st, s));
      if (dst != cur) std::swap(cur, other);
    }
    if (u.has_up) {
      // every frame upsampled, then the causal conv at the doubled size
      VAE_TRY(upsample_nearest2x_nhwc(cur, static_cast<long long>(n) * t, hh, ww, u.up.cin, d.U,
                                      s));
      hh *= 2;
      ww *= 2;
      VAE_TRY(run_conv(*ch, u.up, d.U, n, hh, ww, nullptr, nullptr, other, 1, s, false, false,
                       &st, d.part, ch->groups, d.split));
      std::swap(cur, other);
    }
  }
  const long long sp = static_cast<long long>(t) * hh * ww;
  VAE_TRY(run_gn(*ch, ch->norm_out, cur, n, sp, d.T, dw, st, s));
  return run_conv(*ch, ch->conv_out, d.T, n, hh, ww, nullptr, nullptr, out, 0, s, false, true);
}

// ---------------------------------------------------------------- tiled decode
int up_factor(const Chain &ch) {
  int r = 1;
  for (const UpW &u : ch.ups)
    if (u.has_up) r *= 2;
  return r;
}

// Tile schedule and batch of a tiled decode; tile / min_overlap in output
// pixels, multiples of the decoder's latent-to-pixel factor.
int tiled_plan(const Chain &ch, int n, int h, int w, int tile, int min_overlap, int per_batch,
               TileSchedule *ts, int *batch) {
  if (n <= 0 || h <= 0 || w <= 0 || tile <= 0 || min_overlap < 0 || min_overlap >= tile)
    return VAE_EINVAL;
  const int r = up_factor(ch);
  if (tile % r || min_overlap % r) return VAE_EINVAL;
  VAE_TRY(make_tile_schedule(h * r, w * r, r, tile, min_overlap, ts));
  const long long total = static_cast<long long>(n) * ts->ny * ts->nx;
  if (total > 0x7fffffffll) return VAE_EUNSUPPORTED;
  *batch = static_cast<int>(per_batch <= 0 ? total : std::min<long long>(per_batch, total));
  return VAE_OK;
}

struct TiledWs {
  float *lat = nullptr, *tiles = nullptr;
  void *inner = nullptr;
  size_t inner_bytes = 0;
};

TiledWs carve_tiled(Carver &cv, const Chain &ch, int n, const TileSchedule &ts, int batch) {
  TiledWs t;
  t.lat = cv.take<float>(static_cast<size_t>(batch) * ch.latent_c * ts.tzh * ts.tzw);
  t.tiles = cv.take<float>(static_cast<size_t>(n) * ts.ny * ts.nx * ch.conv_out.cout * ts.th *
                           ts.tw);
  const Plan p = make_plan(ch, batch, ts.tzh, ts.tzw);
  Carver inner(nullptr, 0);
  carve_decode(inner, ch, p, batch, ts.tzh, ts.tzw);
  t.inner_bytes = inner.used;
  t.inner = cv.take<char>(t.inner_bytes);
  return t;
}

}  // namespace
}  // namespace vae

extern "C" {

int vae_causal_decoder_prepare(const vae_causal_decoder_args *a, void **handle,
                               vae_stream_t stream) {
  if (!a || !handle) return VAE_EINVAL;
  *handle = nullptr;
  if (a->latent_channels <= 0 || a->groups <= 0 || a->n_ups < 0 || (a->n_ups && !a->ups) ||
      a->n_mid < 0 || (a->n_mid && !a->mid) || a->scaling_factor == 0.f ||
      a->precision < VAE_PRECISION_AUTO || a->precision > VAE_PRECISION_SPLIT_TF32)
    return VAE_EINVAL;
  auto s = reinterpret_cast<cudaStream_t>(stream);
  Chain *ch = new Chain();
  cudaGetDevice(&ch->device);
  ch->causal = true;
  ch->latent_c = a->latent_channels;
  ch->groups = a->groups;
  ch->eps = a->eps;
  ch->sf = a->scaling_factor;
  ch->sh = a->shift_factor;
  ch->precision = a->precision;
  Builder b{ch, s};
  const int c0 = a->conv_in.cout;
  ch->conv_in = b.conv(a->conv_in, a->latent_channels, c0, nullptr, 3);
  if (ch->conv_in.k != 3) b.fail(VAE_EINVAL);
  for (int m = 0; m < a->n_mid && b.status == VAE_OK; ++m)
    ch->mid3.push_back(b.resnet(a->mid[m], c0, c0, 3));
  int c = c0;
  for (int i = 0; i < a->n_ups && b.status == VAE_OK; ++i) {
    const vae_up_ref &u = a->ups[i];
    UpW uw;
    if (u.n_resnets <= 0 || !u.resnets) b.fail(VAE_EINVAL);
    for (int j = 0; j < u.n_resnets && b.status == VAE_OK; ++j) {
      const int cout = u.resnets[j].conv1.cout;
      uw.res.push_back(b.resnet(u.resnets[j], c, cout, 3));
      c = cout;
    }
    uw.has_up = u.upsample_conv.weight != nullptr;
    if (uw.has_up) {
      uw.up = b.conv(u.upsample_conv, c, u.upsample_conv.cout, nullptr, 3);
      if (uw.up.k != 3 || c % 4) b.fail(VAE_EINVAL);
      c = u.upsample_conv.cout;
    }
    ch->ups.push_back(std::move(uw));
  }
  ch->norm_out = b.norm(a->norm_out, c);
  ch->conv_out = b.conv(a->conv_out, c, a->conv_out.cout, nullptr, 3);
  if (ch->conv_out.k != 3 && b.status == VAE_OK) b.fail(VAE_EINVAL);
  if (b.status == VAE_OK && cudaStreamSynchronize(s) != cudaSuccess) b.fail(VAE_ECUDA);
  cudaStreamSynchronize(s);
  for (void *p : b.temps) cudaFree(p);
  if (b.status != VAE_OK) {
    for (void *p : ch->allocs) cudaFree(p);
    delete ch;
    return b.status;
  }
  {
    std::lock_guard<std::mutex> lk(g_live_mu);
    g_live.insert(ch);
  }
  *handle = ch;
  return VAE_OK;
}

size_t vae_causal_decoder_workspace_size(const void *handle, int n, int t, int h, int w) {
  if (!is_live(handle) || n <= 0 || t <= 0 || h <= 0 || w <= 0) return 0;
  const Chain &ch = *static_cast<const Chain *>(handle);
  if (!ch.causal) return 0;
  const CausalPlan p = make_causal_plan(ch, n, t, h, w);
  Carver cv(nullptr, 0);
  carve_causal(cv, ch, p, n, t, h, w);
  return cv.used;
}

int vae_decode_causal(void *handle, const float *z, int n, int t, int h, int w, float *out,
                      void *ws, size_t ws_bytes, vae_stream_t stream) {
  if (!is_live(handle)) return VAE_ENOTPREPARED;
  Chain *ch = static_cast<Chain *>(handle);
  ch->tr = nullptr;
  return decode_causal_impl(ch, z, n, t, h, w, out, ws, ws_bytes,
                            reinterpret_cast<cudaStream_t>(stream));
}

size_t vae_chain_tiled_workspace_size(const void *handle, int n, int h, int w, int tile,
                                      int min_overlap, int tiles_per_batch) {
  if (!is_live(handle)) return 0;
  const Chain &ch = *static_cast<const Chain *>(handle);
  if (ch.causal) return 0;
  TileSchedule ts;
  int batch = 0;
  if (tiled_plan(ch, n, h, w, tile, min_overlap, tiles_per_batch, &ts, &batch) != VAE_OK) return 0;
  Carver cv(nullptr, 0);
  carve_tiled(cv, ch, n, ts, batch);
  return cv.used;
}

int vae_decode_chain_tiled(void *handle, const float *z, int n, int h, int w, int tile,
                           int min_overlap, int tiles_per_batch, float *rgb, void *ws,
                           size_t ws_bytes, vae_stream_t stream) {
  if (!is_live(handle)) return VAE_ENOTPREPARED;
  if (!z || !rgb || !ws) return VAE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(z) | reinterpret_cast<uintptr_t>(rgb)) & 15) return VAE_EINVAL;
  Chain *ch = static_cast<Chain *>(handle);
  if (ch->causal) return VAE_EINVAL;
  auto s = reinterpret_cast<cudaStream_t>(stream);
  TileSchedule ts;
  int batch = 0;
  VAE_TRY(tiled_plan(*ch, n, h, w, tile, min_overlap, tiles_per_batch, &ts, &batch));
  Carver cv(ws, ws_bytes);
  const TiledWs t = carve_tiled(cv, *ch, n, ts, batch);
  if (!cv.ok()) return VAE_EWORKSPACE;
  const int co = ch->conv_out.cout;
  const long long total = static_cast<long long>(n) * ts.ny * ts.nx;
  const size_t tile_floats = static_cast<size_t>(co) * ts.th * ts.tw;
  ch->tr = nullptr;
  for (long long t0 = 0; t0 < total; t0 += batch) {
    const int cnt = static_cast<int>(std::min<long long>(batch, total - t0));
    VAE_TRY(gather_latent_tiles(z, ch->latent_c, h, w, ts, t0, cnt, t.lat, s));
    VAE_TRY(decode_impl(ch, t.lat, cnt, ts.tzh, ts.tzw, t.tiles + t0 * tile_floats, t.inner,
                        t.inner_bytes, s));
  }
  const int r = up_factor(*ch);
  return blend_decoded_tiles(t.tiles, n, co, ts, h * r, w * r, rgb, s);
}

int vae_decode_chain(void *handle, const float *z, int n, int h, int w, float *rgb, void *ws,
                     size_t ws_bytes, vae_stream_t stream) {
  if (!is_live(handle)) return VAE_ENOTPREPARED;
  Chain *ch = static_cast<Chain *>(handle);
  ch->tr = nullptr;
  return decode_impl(ch, z, n, h, w, rgb, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int vae_chain_trace_points(const void *handle, int n, int h, int w, vae_trace_point *out,
                           int capacity, int *count) {
  if (!is_live(handle)) return VAE_ENOTPREPARED;
  if (!count || n <= 0 || h <= 0 || w <= 0 || (capacity > 0 && !out)) return VAE_EINVAL;
  if (static_cast<const Chain *>(handle)->causal) return VAE_EINVAL;
  const std::vector<vae_trace_point> pts =
      trace_points(*static_cast<const Chain *>(handle), n, h, w);
  *count = static_cast<int>(pts.size());
  for (int i = 0; i < capacity && i < *count; ++i) out[i] = pts[i];
  return VAE_OK;
}

int vae_decode_chain_traced(void *handle, const float *z, int n, int h, int w, float *rgb,
                            void *ws, size_t ws_bytes, float *const *trace, int n_trace,
                            vae_stream_t stream) {
  if (!is_live(handle)) return VAE_ENOTPREPARED;
  if (n_trace < 0 || (n_trace > 0 && !trace)) return VAE_EINVAL;
  Chain *ch = static_cast<Chain *>(handle);
  Tracer tr;
  tr.bufs = trace;
  tr.n = n_trace;
  ch->tr = &tr;
  const int rc =
      decode_impl(ch, z, n, h, w, rgb, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
  ch->tr = nullptr;
  return rc != VAE_OK ? rc : tr.status;
}

int vae_chain_profile(void *handle, int enable) {
  if (!is_live(handle)) return VAE_ENOTPREPARED;
  Chain *ch = static_cast<Chain *>(handle);
  ch->prof.on = enable != 0;
  if (ch->prof.on) ch->prof.reset();
  return VAE_OK;
}

int vae_chain_profile_read(void *handle, vae_prof_record *out, int capacity, int *count) {
  if (!is_live(handle)) return VAE_ENOTPREPARED;
  Chain *ch = static_cast<Chain *>(handle);
  if (!count || (capacity > 0 && !out)) return VAE_EINVAL;
  Profiler &p = ch->prof;
  const int n = static_cast<int>(p.recs.size());
  *count = n;
  for (int i = 0; i < n && i < capacity; ++i) {
    Profiler::Rec &r = p.recs[i];
    float ms = 0.f;
    if (r.ev0 < 0 || r.ev1 < 0) return VAE_ECUDA;
    if (cudaEventSynchronize(p.events[r.ev1]) != cudaSuccess) return VAE_ECUDA;
    if (cudaEventElapsedTime(&ms, p.events[r.ev0], p.events[r.ev1]) != cudaSuccess)
      return VAE_ECUDA;
    r.r.ms = ms;
    out[i] = r.r;
  }
  return VAE_OK;
}

int vae_chain_destroy(void *handle) {
  {
    std::lock_guard<std::mutex> lk(g_live_mu);
    if (!handle || g_live.erase(handle) == 0) return VAE_ENOTPREPARED;
  }
  Chain *ch = static_cast<Chain *>(handle);
  for (void *p : ch->allocs) cudaFree(p);
  delete ch;
  return VAE_OK;
}

}  // extern "C"
