// common.cuh -- internal host/device helpers shared by the kernels' launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>

#include "../../include/vae.h"

namespace vae {

// True when e is an error; with VAE_VERBOSE=1 in the environment the error
// and the call site go to stderr.
bool cuda_failed(cudaError_t e, const char *file, int line);
#define VAE_CUDA_TRY(expr)                                         \
  do {                                                             \
    if (::vae::cuda_failed((expr), __FILE__, __LINE__)) return VAE_ECUDA; \
  } while (0)
// After a kernel launch: the launch's own error (configuration, resources).
#define VAE_LAUNCH_CHECK() VAE_CUDA_TRY(cudaGetLastError())

#define VAE_TRY(expr)                                   \
  do {                                                  \
    int s__ = (expr);                                   \
    if (s__ != VAE_OK) return s__;                      \
  } while (0)

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }
inline int round_up32(int c) { return (c + 31) / 32 * 32; }

// Bump allocator over a caller-provided workspace. Every carve is 256-byte
// aligned. With base == nullptr it only measures.
struct Carver {
  char *base;
  size_t cap;
  size_t used = 0;
  Carver(void *b, size_t c) : base(static_cast<char *>(b)), cap(c) {}
  template <class T>
  T *take(size_t count) {
    size_t off = align_up(used, 256);
    used = off + count * sizeof(T);
    return base ? reinterpret_cast<T *>(base + off) : nullptr;
  }
  bool ok() const { return base == nullptr || used <= cap; }
};

// Device error word of the current device (int), via the library's
// __device__ symbol; resolved once per device and context.
int *device_error_word();
// The CUDA context current on this thread (CUcontext), or nullptr.
void *current_context();
// Limit of the kernels' device-side waits (vae_debug_set_wait_limit).
constexpr uint64_t kDefaultWaitNs = 4000000000ull;
uint64_t wait_limit_ns();
// VAE_INJECT_* bits set by vae_debug_inject (0 in normal operation).
int injected_faults();
// True when the allocation about to be made should fail (vae_debug_fail_allocation).
bool take_alloc_failure();
int num_sms();
// Every kernel launch of the library bumps this process-wide counter.
void count_launches(int n);
long long launch_count();

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
// swizzle128 = false: plain row-major boxes in shared memory.
int encode_tiled(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                 const uint64_t *strides_bytes /* rank-1 entries */, const uint32_t *box,
                 bool swizzle128 = true);

// ------------------------------------------------------------------ kernels
// Implicit-GEMM convolution / GEMM on tcgen05 (igemm.cu).
enum class AMode : int { Conv = 0, Upsample = 1, Gemm = 2 };

struct IgemmDesc {
  AMode mode = AMode::Conv;
  // --- A operand (activations, NHWC; channels padded to a multiple of 32)
  const float *a = nullptr;  // Conv/Upsample: [imgs, Hin, Win, a_c]; Gemm: [M, lda]
  int imgs = 1;              // images (n * t for 3-D)
  int t = 1;                 // frames per sample (3-D); imgs = n * t
  int hin = 1, win = 1;      // input spatial dims (Upsample: low-res)
  int a_c = 32;              // channel count of `a` (multiple of 32)
  int lda = 0;               // Gemm: row stride of A in floats
  int M = 0;                 // Gemm: rows
  int k = 3;                 // Conv: spatial kernel (1 or 3)
  int kt = 1;                // Conv: temporal taps (1 or 3, causal)
  // --- 1x1 shortcut operand (Conv only), same spatial dims as the output
  const float *sc = nullptr;
  int sc_c = 0;  // channels of sc (multiple of 32), 0 = none
  // --- B operand: packed weights [rows >= cout][ldb] K-major, TF32-rounded
  const float *b = nullptr;
  int ldb = 0;   // floats per row (the packed K extent)
  int kdim = 0;  // Gemm: K (multiple of 32)
  int cout = 0;  // N extent
  // --- epilogue
  float *out = nullptr;
  int ldo = 0;           // NHWC / Gemm: floats between consecutive rows
  int out_nchw = 0;      // write [n, cout, t, h, w] instead of rows
  const float *bias = nullptr;
  int bias_per_row = 0;  // Gemm: bias indexed by row instead of column
  const float *residual = nullptr;  // same layout / ld as out
  float alpha = 1.0f;
  int round_out = 0;  // store TF32-rounded values (output feeds another MMA)
  // Optional GroupNorm statistics of the stored output (Conv / Upsample
  // modes, NHWC): partials [n][stat_groups][igemm_stat_slots(d)] x (count,
  // mean, M2), consumed by groupnorm_from_partials.
  float *stat_part = nullptr;
  int stat_groups = 0;
  int *stat_ok = nullptr;  // set on the host: 1 if the statistics were requested and fused
  long long *stat_slots = nullptr;  // set on the host: partial slots per (sample, group)
  // Optional split-K workspace (NHWC Conv / Upsample with ldo == cout): used
  // when the output tiles alone would leave most SMs idle.
  float *split_ws = nullptr;
  size_t split_ws_floats = 0;
  // Split-TF32 products (Conv / Upsample / Gemm): A and B are FP32 and every
  // product is formed as a_hi b_hi + a_lo b_hi + a_hi b_lo with each part
  // rounded to TF32 (three MMAs per step, about FP32 accuracy).
  int precise = 0;
  // Optional GroupNorm (+SiLU) of the A operand applied inside the kernel
  // (Conv; only where igemm_input_gn_ok(d)): a -> silu(a * gn_scale[s][c] +
  // gn_shift[s][c]), TF32-rounded, zero padding outside the image, with
  // s = image / t and [s][a_c] arrays. Replaces a separate normalisation pass
  // over the conv's input.
  const float *gn_scale = nullptr, *gn_shift = nullptr;
  int gn_silu = 1;
  // Gemm (only where igemm_softmax_a_ok(d)): A holds raw scores s and the MMA
  // reads the row softmax p = exp(s * sm_scale - sm_m[row]) * sm_inv_l[row],
  // 0 for columns >= sm_cols.
  const float *sm_m = nullptr, *sm_inv_l = nullptr;
  float sm_scale = 1.0f;
  int sm_cols = 0;
  // Gemm: per row and column tile of igemm_col_tile(cout) columns, the
  // softmax statistics of the stored values v (max of v * rs_scale over the
  // columns < rs_cols, and the sum of exp(v * rs_scale - max)), at
  // rs_out[row * rs_ld + column tile]; (-inf, 0) for a tile with no valid
  // column.
  float2 *rs_out = nullptr;
  float rs_scale = 1.0f;
  int rs_cols = 0, rs_ld = 0;
  // GroupNorm ahead (Conv; only where igemm_gn_ahead_ok(d)): `a` is not an
  // input but made by the launch itself, a = tf32(silu(ga_x * ga_scale[s][c]
  // + ga_shift[s][c])) ([s][a_c] arrays, s = image / t), row by row ahead of
  // the tiles that read it. ga_flags: imgs * hin ints, none equal to ga_epoch
  // on entry (a row is made when its flag reads ga_epoch); ga_next: an int
  // that is 0 on entry (the row counter).
  const float *ga_x = nullptr, *ga_scale = nullptr, *ga_shift = nullptr;
  int *ga_flags = nullptr, *ga_next = nullptr;
  int ga_epoch = 0;
};
// Output-channel (column) tile of a launch with `cout` columns.
int igemm_col_tile(int cout);
// Whether igemm_launch applies an input GroupNorm (gn_scale) for this
// descriptor: 3x3 single-frame convs whose 256-channel tiles stage a halo
// of input rows at least 65 pixels wide, without shortcut operand or
// split-TF32 products. Both transforms are opt-in (VAE_FUSE=on; slower than
// the separate passes on GB300) and these return false without it.
bool igemm_input_gn_ok(const IgemmDesc &d);
// Whether igemm_launch takes a softmax-normalised A (sm_m) for this GEMM.
bool igemm_softmax_a_ok(const IgemmDesc &d);
// Whether igemm_launch can make its A operand from ga_x (GroupNorm ahead):
// 3x3 single-frame convs on the halo (256-channel tiles, rows wider than 64,
// no shortcut) or channel-major (65-128 output channels) paths, TF32
// products, a_c in {32, 64, 128, 256, 512}, output NHWC; opt-in (VAE_GNA=on:
// slower than the separate pass on GB300). A launch that ends up on another
// path returns VAE_EUNSUPPORTED before doing anything.
bool igemm_gn_ahead_ok(const IgemmDesc &d);
// Split-K reduce (splitk.cu): out = alpha * sum of the partials + bias
// (+ residual), rounded on request; GroupNorm partials [samples][groups][slots]
// of the result when stat_part is given (*stat_slots receives slots, 0 if none).
int splitk_reduce(const float *part, int splits, long long split_stride, int samples,
                  long long rows_per_sample, int cout, const float *bias, float alpha,
                  const float *residual, int round, float *out, float *stat_part,
                  int stat_groups, long long *stat_slots, cudaStream_t s);
// Split-K workspace that always suffices for one conv (floats).
constexpr size_t kSplitWsFloats = 160ull * 65536;
long long igemm_stat_slots(const IgemmDesc &d);
int igemm_launch(const IgemmDesc &d, cudaStream_t stream);

// Weight packing (layout.cu): w [cout][cin][taps] (+ shortcut [cout][sc_cin])
// -> dst [cout_rows][ldb] with K index tap * cin_pad + c, TF32-rounded, zeros in
// the padding.
// round = 0 keeps the FP32 values (split-TF32 products split them in the kernel).
int pack_conv_weights(const float *w, int cout, int cin, int taps, const float *w_sc,
                      int sc_cin, float *dst, int cout_rows, int ldb, cudaStream_t s,
                      int round = 1);
inline int packed_ldb(int cin, int taps, int sc_cin) {
  return taps * round_up32(cin) + (sc_cin ? round_up32(sc_cin) : 0);
}
// Upsample conv weights as four parity-specific 2x2 kernels (layout.cu):
// w [cout][cin][3][3] -> dst [4 parities][cout][upsample_ldb(cin)], K index
// (a * 2 + b) * cin_pad + c, parity = py * 2 + px.
inline int upsample_ldb(int cin) { return 4 * round_up32(cin); }
int pack_upsample_weights(const float *w, int cout, int cin, float *dst, cudaStream_t s,
                          int round = 1);

// Layout transforms (layout.cu). src [outer][rows][cols] (row stride src_ld)
// -> dst [outer][cols][rows] (row stride dst_ld), dst = src * alpha + beta,
// optionally TF32-rounded. Used for NCHW <-> NHWC and V^T.
int transpose(const float *src, long long src_outer_stride, int src_ld, float *dst,
              long long dst_outer_stride, int dst_ld, int outer, int rows, int cols,
              float alpha, float beta, int round, cudaStream_t s);
// Copy rows of `cols` floats into rows of `dst_cols` (zero padded).
int pad_rows(const float *src, long long rows, int cols, float *dst, int dst_cols,
             cudaStream_t s);
int add_bias(float *dst, const float *a, const float *b, int n, cudaStream_t s);
// Nearest-2x spatial upsample of NHWC images [imgs][h][w][c] (c % 4 == 0).
int upsample_nearest2x_nhwc(const float *src, long long imgs, int h, int w, int c, float *dst,
                            cudaStream_t s);

// GroupNorm (+SiLU) (groupnorm.cu). `x` NHWC [n][spatial][c] or NCHW.
size_t groupnorm_ws_bytes(int n, int c, long long spatial, int groups);
int groupnorm_silu(const float *x, int n, int c, long long spatial, int nhwc, int groups,
                   float eps, const float *gamma, const float *beta, int silu, int round_out,
                   float *y, void *ws, cudaStream_t s, const float *residual = nullptr);

// GroupNorm(+SiLU) of NHWC x whose statistics were produced by the conv
// epilogue (float partials [n][groups][slots][3]); ws: groupnorm_ws_bytes(n,
// c, ., groups) bytes (holds the compacted partials when slots > 64).
// With more than 64 partials per group, `counters` (n * groups unsigned ints,
// zero on entry and again on return) is required: the compaction's last
// block per group finalizes the statistics.
int groupnorm_from_partials(const float *x, int n, int c, long long spatial, int groups,
                            float eps, const float *gamma, const float *beta, int silu,
                            int round_out, const float *part, long long slots, float *y,
                            void *ws, cudaStream_t s, const float *residual = nullptr,
                            unsigned *counters = nullptr);

// Only the per-(sample, channel) affine of GroupNorm: y = x * scale + shift
// (from fused partials when `part` is given, else from a statistics pass over
// NHWC x using ws as groupnorm_ws_bytes describes). `counters` as above: with
// them (and more than 64 partials) the partials are compacted and finalized
// in one launch, using ws for the compacted slots.
int groupnorm_scale_shift(const float *x, int n, int c, long long spatial, int groups, float eps,
                          const float *gamma, const float *beta, const float *part,
                          long long slots, float *scale, float *shift, void *ws, cudaStream_t s,
                          unsigned *counters = nullptr);

// y = act(x * scale[s][c] + shift[s][c]) over NHWC x [n][spatial][c]
// (act = SiLU when silu), TF32-rounded when round_out.
int groupnorm_apply(const float *x, int n, int c, long long spatial, const float *scale,
                    const float *shift, int silu, int round_out, float *y, cudaStream_t s);

// Fused norm_out GroupNorm+SiLU + conv_out (3x3, cout <= 4) on the CUDA cores
// (head.cu): x NHWC [n][h][w][c], y NCHW [n][cout][h][w].
bool head_supported(int cin, int cout, int k);
size_t head_packed_floats(int cin);
int head_pack_weights(const float *w, int cout, int cin, float *dst, cudaStream_t s);
int head_gn_silu_conv(const float *x, int n, int h, int w, int c, const float *scale,
                      const float *shift, const float *wpk, const float *bias, int cout,
                      float *y, cudaStream_t s);
// The same on the tensor cores with TF32 operands (head_tc.cu; cout <= 7 and
// cin * 16 * ceil(9 * cout / 16) * 4 <= 32 KB): weights packed [NT][cin],
// NT = 16 * ceil(9 * cout / 16), row t * cout + o = tap t of output o.
bool head_tc_supported(int cin, int cout);
size_t head_tc_packed_floats(int cin, int cout);
int head_tc_pack_weights(const float *w, int cout, int cin, float *dst, cudaStream_t s);
int head_tc_gn_silu_conv(const float *x, int n, int h, int w, int c, const float *scale,
                         const float *shift, const float *wpk, const float *bias, int cout,
                         float *y, cudaStream_t s);

// Fused attention (flash.cu): O = softmax(Q K^T * scale) V for one head of
// width d; q, k token-major [L][ld]; vt [d][ldv] (zero beyond L); out [L][ldo].
bool flash_supported(int d);
int flash_attention(const float *q, const float *k, int ld, const float *vt, int ldv, int L, int d,
                    float scale, float *out, int ldo, cudaStream_t s);

// Row softmax in place: s[r][:L] <- softmax(scale * s[r][:L]), TF32-rounded
// unless round == 0.
int softmax_rows(float *s, long long rows, int L, int ld, float scale, cudaStream_t st,
                 int round = 1);
// Per-row softmax statistics from the per-column-tile pairs a GEMM epilogue
// wrote (IgemmDesc::rs_out: part[row * ld + tile] = (max, sum of exp(v -
// max))): m[row] = the row max, inv_l[row] = 1 / the row's sum of exp(v - m).
int softmax_merge_stats(const float2 *part, int rows, int tiles, int ld, float *m, float *inv_l,
                        cudaStream_t st);

}  // namespace vae
