/*
 * vae.h -- C ABI of the GB300 (sm_103a) FLUX-class AutoencoderKL latent decoder.
 *
 * The decoder is the one the cortiq-engine 0.7.7 "Module vae" page documents
 * (structs VaeDecoder, VaeChainArgs, VaeConvRef, VaeNormRef, VaeResnetRef,
 * VaeAttnRef, VaeUpRef): latent [B,16,h,w] -> RGB [B,3,8h,8w].
 *
 * Conventions shared by every entry point
 *   - Tensor pointers (x, y, residual, z, rgb, weights of the single-op calls,
 *     ws) are DEVICE pointers owned by the caller, float32, 16-byte aligned.
 *     Weights given to vae_chain_prepare may be host or device pointers.
 *   - layout: VAE_NCHW (NCDHW for the 3-D call) or VAE_NHWC (NDHWC).
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). No entry point allocates device memory (vae_chain_prepare is the
 *     one exception) or synchronises; scratch comes from `ws`, `ws_bytes` long,
 *     whose required size the matching *_workspace_size call returns.
 *   - Return value: VAE_OK (0) or a negative vae_status. On a nonzero status
 *     the contents of the outputs are unspecified. Argument and shape checks
 *     run before any launch. There is no CPU fallback.
 *   - Arithmetic: 3x3 / 1x1 / 3x3x3 convolutions, attention projections and
 *     the attention products run on the tcgen05 tensor cores with TF32
 *     operands and FP32 accumulation; weights are rounded to TF32
 *     (round-to-nearest) when packed; normalisation, softmax and epilogues are
 *     FP32. The chain can instead form every product in split-TF32 (see
 *     vae_precision).
 *   - Outputs may not alias inputs, except y == residual (vae_conv2d,
 *     vae_conv3d_causal) and y == x (vae_groupnorm_silu).
 *   - Device-side waits are bounded: a kernel that gives up records
 *     VAE_EDEVICE_TIMEOUT in a device error word that vae_device_error reads.
 */
#ifndef VAE_GB300_H
#define VAE_GB300_H

#include <stddef.h>

#if defined(__GNUC__)
#define VAE_API __attribute__((visibility("default")))
#else
#define VAE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *vae_stream_t; /* identical to cudaStream_t */

typedef enum {
  VAE_OK = 0,
  VAE_EINVAL = -1,          /* null pointer, non-positive size, bad layout  */
  VAE_EUNSUPPORTED = -2,    /* shape outside what the kernels handle        */
  VAE_EWORKSPACE = -3,      /* ws_bytes below the *_workspace_size value    */
  VAE_ECUDA = -4,           /* a CUDA runtime/driver call or launch failed  */
  VAE_ENOTPREPARED = -5,    /* null or destroyed chain handle               */
  VAE_EDEVICE_TIMEOUT = -6, /* a bounded device-side wait expired           */
  VAE_ENOMEM = -7           /* vae_chain_prepare could not allocate         */
} vae_status;

typedef enum { VAE_NCHW = 0, VAE_NHWC = 1 } vae_layout;

/* ------------------------------------------------------------------------
 * vae_conv2d -- 2-D convolution, stride 1, square kernel k in {1,3}, zero
 * padding k/2 (cortiq-engine "Module vae", structs Conv2d and VaeConvRef):
 *   y[n,o,i,j] = bias[o] + sum_{c,ky,kx} weight[o,c,ky,kx] x[n,c,i+ky-k/2,j+kx-k/2]
 *              (+ residual[n,o,i,j])
 *              (+ sum_c sc_w[o,c] sc_x[n,c,i,j] + sc_b[o])
 * The residual and the 1x1 shortcut form the resnet skip of VaeResnetRef
 * ("x + conv2(...)", "the skip through the 1x1 shortcut"); both are optional
 * (NULL). The shortcut is fused as extra reduction steps into the same
 * accumulator.
 *   x        [n,cin,h,w] (layout)          weight [cout,cin,k,k] row-major
 *   bias     [cout] or NULL                residual [n,cout,h,w] or NULL
 *   sc_x     [n,sc_cin,h,w] or NULL        sc_w [cout,sc_cin], sc_b [cout] or NULL
 *   y        [n,cout,h,w]
 * Limits: cin, sc_cin <= 4096; cout <= 4096; h, w <= 65535.
 */
VAE_API size_t vae_conv2d_workspace_size(int n, int cin, int h, int w, int layout, int cout, int k,
                                 int sc_cin);
VAE_API int vae_conv2d(const float *x, int n, int cin, int h, int w, int layout, const float *weight,
               const float *bias, int cout, int k, const float *residual, const float *sc_x,
               const float *sc_w, const float *sc_b, int sc_cin, float *y, void *ws,
               size_t ws_bytes, vae_stream_t stream);

/* Weights packed once (the GEMM layout vae_conv2d builds on every call), for
 * a conv applied many times:
 *   vae_conv2d_pack_bytes  size of the pack for (cout, cin, k, sc_cin)
 *   vae_conv2d_pack        weight [cout,cin,k,k], bias or NULL, and the 1x1
 *                          shortcut's sc_w [cout,sc_cin] / sc_b or NULL (with
 *                          sc_cin = 0 and NULLs when there is none) into the
 *                          caller's device buffer `packed` (>= the size above,
 *                          256-byte aligned); stream-ordered, no allocation
 *   vae_conv2d_packed      vae_conv2d on such a pack: the same arguments and
 *                          workspace (vae_conv2d_workspace_size), with cin, k,
 *                          cout and sc_cin as given to vae_conv2d_pack (not
 *                          checked against the pack: it holds only numbers);
 *                          sc_x non-NULL exactly when sc_cin > 0.
 * The pack is read-only for vae_conv2d_packed and may serve concurrent calls.
 * Errors: VAE_EINVAL (NULLs, bad sizes, shortcut arguments that disagree),
 * VAE_EUNSUPPORTED (sizes beyond the limits above), VAE_EWORKSPACE
 * (packed_bytes or ws_bytes too small). */
VAE_API size_t vae_conv2d_pack_bytes(int cout, int cin, int k, int sc_cin);
VAE_API int vae_conv2d_pack(const float *weight, const float *bias, int cout, int cin, int k,
                            const float *sc_w, const float *sc_b, int sc_cin, void *packed,
                            size_t packed_bytes, vae_stream_t stream);
VAE_API int vae_conv2d_packed(const float *x, int n, int cin, int h, int w, int layout,
                              const void *packed, int cout, int k, const float *residual,
                              const float *sc_x, int sc_cin, float *y, void *ws, size_t ws_bytes,
                              vae_stream_t stream);

/* ------------------------------------------------------------------------
 * vae_upsample_conv -- nearest-2x upsample followed by a 3x3 stride-1 pad-1
 * convolution (cortiq-engine "Module vae", struct VaeUpRef):
 *   u[n,c,i,j] = x[n,c,i/2,j/2];  y = conv3x3(u) + bias
 * The upsampled tensor is never stored: per output parity (py, px) the 3x3
 * taps land on 2x2 distinct low-resolution pixels, so the weights are summed
 * (then rounded to TF32) into four 2x2 kernels applied to x directly; the
 * result equals the definition up to where the rounding happens.
 *   x [n,cin,h,w]; weight [cout,cin,3,3]; bias [cout] or NULL; y [n,cout,2h,2w]
 */
VAE_API size_t vae_upsample_conv_workspace_size(int n, int cin, int h, int w, int layout, int cout);
VAE_API int vae_upsample_conv(const float *x, int n, int cin, int h, int w, int layout,
                      const float *weight, const float *bias, int cout, float *y, void *ws,
                      size_t ws_bytes, vae_stream_t stream);
/* The same with the weights packed once (as for vae_conv2d_pack): the pack
 * holds the four parity kernels and the bias; vae_upsample_conv_packed takes
 * vae_upsample_conv's arguments and workspace with the pack in place of
 * weight and bias. Errors as for vae_conv2d_pack / vae_conv2d_packed. */
VAE_API size_t vae_upsample_conv_pack_bytes(int cout, int cin);
VAE_API int vae_upsample_conv_pack(const float *weight, const float *bias, int cout, int cin,
                                   void *packed, size_t packed_bytes, vae_stream_t stream);
VAE_API int vae_upsample_conv_packed(const float *x, int n, int cin, int h, int w, int layout,
                                     const void *packed, int cout, float *y, void *ws,
                                     size_t ws_bytes, vae_stream_t stream);

/* ------------------------------------------------------------------------
 * vae_groupnorm_silu -- GroupNorm (cortiq-engine "Module vae", structs
 * GroupNorm and VaeNormRef; statistics as vae3d.rs GroupNorm::apply computes
 * them): per (sample, group) over the group's c/groups channels and all
 * `spatial` positions (H*W, or T*H*W for 5-D data),
 *   mean, var = biased variance,  y = (x-mean)/sqrt(var+eps)*gamma[c] + beta[c]
 * then, if apply_silu != 0, y = y / (1 + exp(-y)) (vae3d.rs fn silu).
 *   x, y [n,c,spatial] (layout; y == x allowed); gamma, beta [c]
 * Limits: c % groups == 0, c % 4 == 0, c <= 1024.
 */
VAE_API size_t vae_groupnorm_silu_workspace_size(int n, int c, long long spatial, int layout,
                                         int groups);
VAE_API int vae_groupnorm_silu(const float *x, int n, int c, long long spatial, int layout, int groups,
                       float eps, const float *gamma, const float *beta, int apply_silu,
                       float *y, void *ws, size_t ws_bytes, vae_stream_t stream);

/* vae_groupnorm_silu_noalloc -- the same GroupNorm(+SiLU) for callers that
 * must not allocate device memory, not even a workspace: e.g. a plug-in inside
 * a host application that owns the whole device-memory budget and forbids
 * libraries to allocate, or a latency-critical loop that cannot take the cost
 * (and possible implicit device synchronisation) of cudaMalloc. The pages
 * have no counterpart; this is a deployment convenience.
 * Arguments and results are those of vae_groupnorm_silu without ws/ws_bytes.
 * Its statistics scratch is one fixed 4 MiB array compiled into the library
 * (held in the global memory of every GPU that loads the library until the
 * process exits): enough for up to 10 samples at 32 groups; larger requests
 * return VAE_EUNSUPPORTED before anything is launched. The first call on a
 * device looks up the array's device address for that device, and so does
 * the first call after the device's context was replaced (cudaDeviceReset
 * moves the array); make that first call before any stream capture. All
 * calls share the array, so calls
 * that overlap on the GPU (e.g. on two streams at once) race; calls on one
 * stream are ordered and safe. No part of the array needs clearing between
 * calls. Allocates nothing. */
VAE_API int vae_groupnorm_silu_noalloc(const float *x, int n, int c, long long spatial, int layout,
                                       int groups, float eps, const float *gamma,
                                       const float *beta, int apply_silu, float *y,
                                       vae_stream_t stream);

/* ------------------------------------------------------------------------
 * vae_mid_attn -- mid-block single-head spatial attention (cortiq-engine
 * "Module vae", struct VaeAttnRef): t = GroupNorm(x); tokens p = i*w + j;
 * q,k,v = t W^T + b with W [c,c] row-major (out x in);
 * o = softmax(q k^T / sqrt(c)) v (row softmax with max subtraction, vae3d.rs
 * fn softmax_inplace); y = x + (o wo^T + bo).
 *   x, y [n,c,h,w] (layout); gn_w, gn_b [c]; wq..wo [c,c]; bq..bo [c]
 * Limits: c % 32 == 0, c <= 1024, h*w <= 65536.
 */
VAE_API size_t vae_mid_attn_workspace_size(int n, int c, int h, int w, int layout);
VAE_API int vae_mid_attn(const float *x, int n, int c, int h, int w, int layout, int groups, float eps,
                 const float *gn_w, const float *gn_b, const float *wq, const float *bq,
                 const float *wk, const float *bk, const float *wv, const float *bv,
                 const float *wo, const float *bo, float *y, void *ws, size_t ws_bytes,
                 vae_stream_t stream);

/* ------------------------------------------------------------------------
 * vae_conv3d_causal -- 3-D convolution with causal time padding ("VAE decode
 * -> GPU handoff (FLUX/LTX render services)", sections "The CPU VAE code"
 * and "GPU plan" step 1): kernel 3x3x3, stride 1, spatial zero padding 1,
 * time padded by prepending two copies of the first frame:
 *   y[n,o,t,i,j] = bias[o] + sum w[o,c,kt,ky,kx] x[n,c,max(t+kt-2,0),i+ky-1,j+kx-1]
 *                  (+ residual[n,o,t,i,j])
 *   x [n,cin,t,h,w] (NCDHW or NDHWC); weight [cout,cin,3,3,3]; y [n,cout,t,h,w]
 */
VAE_API size_t vae_conv3d_causal_workspace_size(int n, int cin, int t, int h, int w, int layout,
                                        int cout);
VAE_API int vae_conv3d_causal(const float *x, int n, int cin, int t, int h, int w, int layout,
                      const float *weight, const float *bias, int cout, const float *residual,
                      float *y, void *ws, size_t ws_bytes, vae_stream_t stream);

/* ------------------------------------------------------------------------
 * vae_causal_stack -- the LTX-style 3-D causal conv slice ("VAE decode -> GPU
 * handoff (FLUX/LTX render services)", "The CPU VAE code": a 3-D causal conv
 * stack with causal padding on the time axis): for i = 1..n_layers
 *   u_i = silu(GroupNorm_i(conv3d_causal_i(u_{i-1})))   (+ u_{i-2} when i is even)
 * with u_0 = x and y = u_{n_layers}; "residual every 2 convs" is read as adding
 * the input of each pair of layers to the pair's output.
 *   x, y [n,c,t,h,w] (NCDHW or NDHWC; y must not alias x)
 *   weight, bias, gn_w, gn_b: HOST arrays of n_layers DEVICE pointers to
 *   [c,c,3,3,3], [c], [c], [c]
 * Limits: c % 32 == 0, c % groups == 0, c <= 1024, 1 <= n_layers <= 64.
 */
VAE_API size_t vae_causal_stack_workspace_size(int n, int c, int t, int h, int w, int layout,
                                               int n_layers);
VAE_API int vae_causal_stack(const float *x, int n, int c, int t, int h, int w, int layout,
                             int n_layers, const float *const *weight, const float *const *bias,
                             const float *const *gn_w, const float *const *gn_b, int groups,
                             float eps, float *y, void *ws, size_t ws_bytes, vae_stream_t stream);

/* ------------------------------------------------------------------------
 * The whole decoder (cortiq-engine "Module vae", structs VaeChainArgs and
 * VaeDecoder), in execution order: z/scaling_factor + shift_factor ->
 * conv_in -> mid_res1 -> mid_attn -> mid_res2 -> ups[0..n_ups) ->
 * GroupNorm+SiLU (norm_out) -> conv_out. Activations stay in device memory
 * (NHWC inside the chain); only the RGB output is written to `rgb`.
 * A conv_ref with weight == NULL is absent (shortcut, upsample conv).
 * Attention projections are conv_refs with k = 1, cin = cout = c.
 */
typedef struct {
  const float *weight; /* [cout, cin, k, k] row-major */
  const float *bias;   /* [cout] */
  int cout, cin, k;
} vae_conv_ref;

typedef struct {
  const float *weight; /* gamma [c] */
  const float *bias;   /* beta [c] */
  int c;
} vae_norm_ref;

typedef struct {
  vae_norm_ref norm1;
  vae_conv_ref conv1;
  vae_norm_ref norm2;
  vae_conv_ref conv2;
  vae_conv_ref shortcut; /* 1x1, weight NULL when cin == cout */
} vae_resnet_ref;

typedef struct {
  vae_norm_ref norm;
  vae_conv_ref q, k, v, out;
} vae_attn_ref;

typedef struct {
  int n_resnets;
  const vae_resnet_ref *resnets;
  vae_conv_ref upsample_conv; /* weight NULL: no upsample */
} vae_up_ref;

/* Arithmetic of the chain's tensor-core products.
 *   TF32        TF32 operands (rounded to nearest), FP32 accumulation.
 *   SPLIT_TF32  every operand split into two TF32 parts, hi + lo, and each
 *               product formed as hi*hi + lo*hi + hi*lo (three MMAs), FP32
 *               accumulation: about FP32 accuracy at three times the MMA work.
 *   AUTO        SPLIT_TF32 for a decode whose conv work is at most
 *               VAE_SPLIT_AUTO_GFLOP (small, low-channel decoders, where the
 *               extra products cost next to nothing), TF32 otherwise. */
typedef enum {
  VAE_PRECISION_AUTO = 0,
  VAE_PRECISION_TF32 = 1,
  VAE_PRECISION_SPLIT_TF32 = 2
} vae_precision;
#define VAE_SPLIT_AUTO_GFLOP 20.0

typedef struct {
  int latent_channels;
  float scaling_factor, shift_factor;
  int groups;
  float eps;
  vae_conv_ref conv_in;
  vae_resnet_ref mid_res1;
  vae_attn_ref mid_attn;
  vae_resnet_ref mid_res2;
  int n_ups;
  const vae_up_ref *ups;
  vae_norm_ref norm_out;
  vae_conv_ref conv_out;
  int precision; /* vae_precision */
} vae_chain_args;

/* Packs every weight once (TF32-rounded, GEMM layout) into device memory owned
 * by the returned handle, which the key-cached weight set of VaeChainArgs
 * corresponds to. Allocates; enqueues copies on `stream` and synchronises it. */
VAE_API int vae_chain_prepare(const vae_chain_args *args, void **handle, vae_stream_t stream);
/* Workspace for one vae_decode_chain call on a [n,latent_channels,h,w] latent;
 * 0 for a null handle. */
VAE_API size_t vae_chain_workspace_size(const void *handle, int n, int h, int w);
/*   z   [n,latent_channels,h,w] NCHW (not yet de-normalised)
 *   rgb [n,3,8h,8w] NCHW (raw decoder output, not clamped)
 * The workspace needs no initialisation (the decode clears the counters and
 * flags it relies on) and holds one decode's intermediate state, so decodes
 * that may overlap on the GPU need workspaces of their own. Every reduction
 * has a fixed order: the same inputs give the same bits. */
VAE_API int vae_decode_chain(void *handle, const float *z, int n, int h, int w, float *rgb, void *ws,
                     size_t ws_bytes, vae_stream_t stream);
/* ------------------------------------------------------------------------
 * Tiled decode, for outputs the whole-image decode cannot hold (its
 * activations and attention grow with the image; a latent above 65536
 * tokens is refused by vae_decode_chain). The tile schedule and the
 * cross-fade follow cortiq-engine 0.8.78's vae3d.rs (fn split_tiles,
 * fn blend, fn crop, VideoVae::decode_clip), written there for another
 * decoder:
 *   - along each axis of the output plane (8h x 8w pixels), the fewest
 *     tiles of `tile` pixels whose overlaps are at least `min_overlap`,
 *     the slack added to the overlaps one latent cell (8 pixels) at a time,
 *     round robin; a single tile when the axis fits in one;
 *   - every tile's latent crop is decoded on its own (GroupNorm statistics
 *     and attention see only that tile, so the output differs from the
 *     whole-image decode unless one tile covers the image);
 *   - in raster order, a tile's first overlap rows are cross-faded with the
 *     last rows of the tile above as that tile was decoded (weights
 *     1 - k/e and k/e at row k of the e-row overlap), then its first
 *     overlap columns likewise with the tile to its left; a tile keeps its
 *     last overlap rows / columns only if it is the last of its column /
 *     row (the next tile's cross-fade replaces them).
 * tile, min_overlap: output pixels, multiples of the latent-to-pixel factor
 * (8), min_overlap < tile; at most 128 tiles per axis. tiles_per_batch: how
 * many tiles one pass of the chain decodes (0 = all), which bounds the
 * workspace. z, rgb as vae_decode_chain. */
VAE_API size_t vae_chain_tiled_workspace_size(const void *handle, int n, int h, int w, int tile,
                                              int min_overlap, int tiles_per_batch);
VAE_API int vae_decode_chain_tiled(void *handle, const float *z, int n, int h, int w, int tile,
                                   int min_overlap, int tiles_per_batch, float *rgb, void *ws,
                                   size_t ws_bytes, vae_stream_t stream);

/* Frees the handle's device memory. Handles are tracked in a registry of live
 * handles: every entry point given a destroyed (or never prepared) handle
 * returns VAE_ENOTPREPARED without touching it. */
VAE_API int vae_chain_destroy(void *handle);

/* ------------------------------------------------------------------------
 * Layer trace of one decode, for per-layer parity checks: the same decode as
 * vae_decode_chain (identical kernels and arithmetic) that also copies each
 * step's output tensor, right after the step, into caller buffers. The
 * points follow the chain's execution order ("Module vae", VaeChainArgs):
 *   LATENT     de-normalised latent, NHWC with channels padded to 32
 *   CONV       3x3 conv output: conv_in, a resnet's conv1
 *   GROUPNORM  GroupNorm+SiLU output: a resnet's norm1 / norm2, and norm_out
 *              when conv_out does not take the fused head
 *   RESNET     resnet output: conv2 + bias + skip (identity or 1x1 shortcut)
 *   ATTENTION  mid attention block output: x + out-projection
 *   UPSAMPLE   nearest-2x upsample + conv output
 *   RGB        decoder output, NCHW: conv_out of the GroupNorm point before
 *              it, or norm_out + SiLU + conv_out (fused head) of the point
 *              before it when that point is not a GROUPNORM
 * Activations are NHWC [n][h][w][c] float32, stored as the next step reads
 * them (operands of a tensor-core product are TF32-rounded values). */
typedef enum {
  VAE_TRACE_LATENT = 0,
  VAE_TRACE_CONV = 1,
  VAE_TRACE_GROUPNORM = 2,
  VAE_TRACE_RESNET = 3,
  VAE_TRACE_ATTENTION = 4,
  VAE_TRACE_UPSAMPLE = 5,
  VAE_TRACE_RGB = 6
} vae_trace_kind;

typedef struct {
  int kind;     /* vae_trace_kind */
  int c, h, w;  /* tensor channels and spatial size (per image) */
  int input;    /* index of the point holding this step's input (-1: none) */
  int skip;     /* RESNET: index of the point holding the resnet's input */
  size_t bytes; /* n * h * w * c * 4 */
} vae_trace_point;

/* Describes the trace points of a decode of a [n,latent_channels,h,w]
 * latent: copies min(capacity, total) of them to `out`, *count = total. */
VAE_API int vae_chain_trace_points(const void *handle, int n, int h, int w, vae_trace_point *out,
                                   int capacity, int *count);
/* vae_decode_chain plus the trace: trace[i] (device, bytes of point i) or
 * NULL to skip point i; n_trace may be smaller than the point count. */
VAE_API int vae_decode_chain_traced(void *handle, const float *z, int n, int h, int w,
                                    float *rgb, void *ws, size_t ws_bytes, float *const *trace,
                                    int n_trace, vae_stream_t stream);

/* ------------------------------------------------------------------------
 * 3-D causal decoder: an LTX-style video decoder ("VAE decode -> GPU handoff
 * (FLUX/LTX render services)", "The CPU VAE code": LtxVaeDecoder::decode, a
 * 3-D causal conv over time x H x W with causal padding on the time axis)
 * as a structural decoder, since the pages give no LTX architecture
 * constants: the 2-D decoder's order (VaeChainArgs) with every 3x3 conv a
 * causal 3x3x3 conv (vae_conv3d_causal's definition: two copies of the
 * first frame in front, zero spatial padding) and GroupNorm over (t, h, w):
 *   z / scaling_factor + shift_factor -> conv_in -> mid resnets (no
 *   attention) -> ups[i]: resnets, then (if upsample_conv.weight) nearest-2x
 *   upsample of every frame and upsample_conv -> GroupNorm+SiLU -> conv_out.
 * Frames stay frames (no temporal upsampling).
 *   conv refs with k = 3: weight [cout][cin][3][3][3]; shortcuts k = 1:
 *   [cout][cin] (1x1x1); norms as for the chain.
 *   z   [n, latent_channels, t, h, w] NCDHW; out [n, conv_out.cout, t, f*h,
 *   f*w] NCDHW, f = 2^(upsampling up-blocks).
 * The handle is freed with vae_chain_destroy; the 2-D entry points refuse it
 * (VAE_EINVAL), as vae_decode_causal refuses a 2-D chain. */
typedef struct {
  int latent_channels;
  float scaling_factor, shift_factor;
  int groups;
  float eps;
  vae_conv_ref conv_in;
  int n_mid;
  const vae_resnet_ref *mid;
  int n_ups;
  const vae_up_ref *ups;
  vae_norm_ref norm_out;
  vae_conv_ref conv_out;
  int precision; /* vae_precision; AUTO compares the decode's conv work */
} vae_causal_decoder_args;

VAE_API int vae_causal_decoder_prepare(const vae_causal_decoder_args *args, void **handle,
                                       vae_stream_t stream);
VAE_API size_t vae_causal_decoder_workspace_size(const void *handle, int n, int t, int h, int w);
VAE_API int vae_decode_causal(void *handle, const float *z, int n, int t, int h, int w,
                              float *out, void *ws, size_t ws_bytes, vae_stream_t stream);

/* ------------------------------------------------------------------------
 * Step profiler of the chain: when enabled, vae_decode_chain brackets every
 * step (one conv, one GroupNorm+SiLU, the attention block, the latent
 * staging) with CUDA events on the caller's stream and stores the step's
 * algorithmic work. Enabling clears earlier records; records accumulate over
 * decode calls until read. Inside a stream capture the events become
 * event-record nodes of the graph: every replay re-records them, and a read
 * after replays returns the last replay's times. */
typedef enum {
  VAE_PROF_CONV3X3 = 0,        /* 3x3 conv (flops: 2*cin*cout*9 per output pixel, + shortcut;
                                  bytes: input, output, residual and shortcut input once)     */
  VAE_PROF_UPSAMPLE_CONV = 1,  /* nearest-2x upsample + 3x3 conv (flops executed: 2*cin*cout*4
                                  per output pixel, four parity 2x2 kernels; bytes: low-res
                                  input and output once)                                      */
  VAE_PROF_GROUPNORM = 2,      /* GroupNorm(+SiLU) (bytes: 8 per element, read + write, when
                                  the producing conv supplied the statistics; 12 otherwise)    */
  VAE_PROF_ATTENTION = 3,      /* mid attention block (flops: 4*L*L*c + 8*L*c*c per image)   */
  VAE_PROF_LAYOUT = 4,         /* latent de-normalisation / layout staging (bytes)           */
  VAE_PROF_HEAD = 5,           /* norm_out GroupNorm+SiLU fused into conv_out (tensor cores in
                                  TF32 decodes, FP32 CUDA cores in split-TF32 ones): flops
                                  2*9*cin*cout, bytes 4*cin + 4*cout per output pixel */
  VAE_PROF_GN_AFFINE = 6       /* a GroupNorm reduced to its per-channel affine, applied by the
                                  conv that reads it (bytes: the statistics read: 12 per
                                  partial, or 4 per element without fused partials)          */
} vae_prof_kind;

typedef struct {
  int kind;     /* vae_prof_kind */
  int kernels;  /* kernel launches inside the step */
  double flops; /* algorithmic floating-point operations of the step */
  double bytes; /* algorithmic HBM bytes of the step (memory-bound kinds) */
  double ms;    /* device time between the step's two events */
} vae_prof_record;

VAE_API int vae_chain_profile(void *handle, int enable);
/* Synchronises the recorded events; copies min(capacity, recorded) records. */
VAE_API int vae_chain_profile_read(void *handle, vae_prof_record *out, int capacity, int *count);

/* ------------------------------------------------------------------------
 * Diagnostics. */
/* Kernels this library has launched in this process (monotonic counter). */
VAE_API long long vae_kernel_launch_count(void);
VAE_API const char *vae_status_string(int status);
/* Synchronises `stream`, then reads and clears the device error word of the
 * current device; *code receives 0 or the VAE_E* status a kernel recorded. */
VAE_API int vae_device_error(vae_stream_t stream, int *code);
/* Number of SMs the kernels size their persistent grids for (current device). */
VAE_API int vae_num_sms(void);
/* Measures this GPU's tcgen05 kind::tf32 tensor-pipe rate, the denominator of
 * the convolution's roofline fraction: one CTA per SM issues iters x 4
 * MMAs of M = 128, N = 256, K = 8 on operands resident in shared memory
 * (no global-memory traffic), accumulating in TMEM. *flops receives the
 * floating-point operations executed, *ms their device time (CUDA events on
 * `stream`, synchronised before returning). */
VAE_API int vae_measure_tf32_mma(int iters, double *flops, float *ms, vae_stream_t stream);

/* ------------------------------------------------------------------------
 * Test hooks for the failure paths; none of them faults, traps or hangs a
 * GPU. Process-wide settings, read when a kernel is launched.
 *
 * vae_debug_set_wait_limit: every device-side wait of the implicit-GEMM conv
 * gives up after `ns` nanoseconds (0 restores the default, 4 s) and records
 * VAE_EDEVICE_TIMEOUT, drains its own copies and MMAs, frees its TMEM and
 * returns.
 * vae_debug_inject: VAE_INJECT_WITHHOLD_STREAMK_FLAG makes the conv's
 * stream-K CTAs skip the flag that hands a tile's tail over to the CTA that
 * finishes it, so that CTA's bounded wait runs out (0 clears).
 * vae_debug_fail_allocation: the nth device allocation vae_chain_prepare
 * makes from now on (1 = the next) fails as if the device were out of
 * memory: prepare frees what it allocated and returns VAE_ENOMEM (0 clears). */
typedef enum { VAE_INJECT_WITHHOLD_STREAMK_FLAG = 1 } vae_inject_bits;
VAE_API int vae_debug_set_wait_limit(unsigned long long ns);
VAE_API int vae_debug_inject(int bits);
VAE_API int vae_debug_fail_allocation(int nth);

#ifdef __cplusplus
}
#endif
#endif /* VAE_GB300_H */
