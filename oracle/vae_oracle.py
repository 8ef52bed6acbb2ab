"""Plain float64 CPU oracle of the FLUX-class VAE decoder (test infrastructure).

Sources (cited by page title and section):
  [vae]   cortiq-engine 0.7.7, "Module vae" (docs.rs): structs Conv2d, GroupNorm,
          VaeConvRef, VaeNormRef, VaeResnetRef, VaeAttnRef, VaeUpRef,
          VaeChainArgs, VaeDecoder.
  [vae3d] cortiq-engine 0.8.78, source of vae3d.rs: fn silu, fn softmax_inplace,
          struct GroupNorm (apply).
  [hand]  "VAE decode -> GPU handoff (FLUX/LTX render services)": sections
          "The CPU VAE code" and "GPU plan -- im2col + cuBLAS SGEMM".
  [tile]  cortiq-engine 0.8.78, source of vae3d.rs: fn split_tiles, fn crop,
          fn blend and VideoVae::decode_clip (the spatial tile schedule and
          the cross-fade of neighbouring tiles, written there for another
          decoder and applied here to this one).

Layout: NCHW (NCTHW for the 3-D case), as the pages' decoders store tensors.
Every input is widened to float64 first; every step is float64. Where a page
is silent the reading taken is stated on the function.

Parity status: every function here is pinned by tests in
tests/test_oracle_pins.py (brute force on tiny inputs, closed forms,
invariants, library special cases). The composition ``decode`` is pinned by an
independent restatement through torch.nn.functional float64 ops and by
structural invariants; its agreement with a trained diffusers decode is
"parity unpinned" (no trained weights exist here).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "denormalize", "conv2d", "group_norm", "silu", "group_norm_silu",
    "upsample_nearest2x", "upsample_conv", "resnet", "softmax_rows",
    "mid_attention", "up_block", "decode", "conv3d_causal", "causal_stack",
    "conv2d_at", "upsample_conv_at", "mid_attention_at",
    "split_tiles", "blend_tiles", "tiled_decode",
    "upsample_nearest2x_spatial", "resnet3d", "causal_decode",
]


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def denormalize(z, scaling_factor, shift_factor):
    """[vae] VaeDecoder: the diffusers latent de-normalisation
    z / scaling_factor + shift_factor, elementwise."""
    return _f64(z) / scaling_factor + shift_factor


def conv2d(x, weight, bias=None):
    """[vae] Conv2d / VaeConvRef: stride 1, square kernel k, symmetric zero
    padding k // 2, weight [oc, ic, k, k].

    y[n,o,i,j] = b[o] + sum_{c,ky,kx} w[o,c,ky,kx] * x[n,c,i+ky-p,j+kx-p],
    x taken as 0 outside the image. Reading (pages silent on kernel flip):
    cross-correlation, the diffusers/PyTorch convention, which is also how the
    im2col in vae3d.rs EncConv::apply indexes (oy + ky - pad, no flip).

    The sum over (c, ky, kx) is written as one matrix product per tap over the
    zero-padded input: tap (ky, kx) contributes w[:, :, ky, kx] @ x_shifted.
    """
    x = _f64(x)
    w = _f64(weight)
    n, cin, h, wd = x.shape
    cout, cin_w, k, k2 = w.shape
    assert cin == cin_w and k == k2
    p = k // 2
    xp = np.zeros((n, cin, h + 2 * p, wd + 2 * p))
    xp[:, :, p:p + h, p:p + wd] = x
    y = np.zeros((n, cout, h, wd))
    for b in range(n):
        for ky in range(k):
            for kx in range(k):
                shifted = xp[b, :, ky:ky + h, kx:kx + wd].reshape(cin, h * wd)
                y[b] += (w[:, :, ky, kx] @ shifted).reshape(cout, h, wd)
    if bias is not None:
        y += _f64(bias)[None, :, None, None]
    return y


def conv2d_at(x, weight, bias, pixels, upsample=False):
    """The conv2d definition evaluated at chosen output pixels only (for
    outputs too large to compute whole): ``pixels`` is an int array [S, 3] of
    (image, row, col); returns [S, cout].

    y[o] = b[o] + sum_{c,ky,kx} w[o,c,ky,kx] * u[c, i+ky-p, j+kx-p], zero
    outside the image, where u is x itself, or with ``upsample`` the
    nearest-2x upsample of x ([vae] VaeUpRef: u[c,i,j] = x[c,i//2,j//2] on the
    doubled grid). ``x`` is NCHW (any array that supports numpy indexing,
    e.g. a transposed view); only the gathered taps are widened to float64."""
    w = _f64(weight)
    cout, cin, k, _ = w.shape
    p = k // 2
    pix = np.asarray(pixels, dtype=np.int64)
    b_idx, i_idx, j_idx = pix[:, 0], pix[:, 1], pix[:, 2]
    h, wd = x.shape[2], x.shape[3]
    if upsample:
        h, wd = 2 * h, 2 * wd
    y = np.zeros((len(pix), cout))
    for ky in range(k):
        for kx in range(k):
            r = i_idx + ky - p
            c = j_idx + kx - p
            inside = (r >= 0) & (r < h) & (c >= 0) & (c < wd)
            rs, cs = np.where(inside, r, 0), np.where(inside, c, 0)
            if upsample:
                rs, cs = rs // 2, cs // 2
            taps = _f64(x[b_idx, :, rs, cs]) * inside[:, None]  # [S, cin]
            y += taps @ w[:, :, ky, kx].T
    if bias is not None:
        y += _f64(bias)[None, :]
    return y


def upsample_conv_at(x, weight, bias, pixels):
    """upsample_conv at chosen output pixels of the doubled grid ([S, cout])."""
    return conv2d_at(x, weight, bias, pixels, upsample=True)


def group_norm(x, gamma, beta, groups=32, eps=1e-6):
    """[vae] GroupNorm / VaeNormRef (eps 1e-6, affine); statistics as in
    [vae3d] struct GroupNorm::apply: per (sample, group) over the group's
    channels and every spatial (and temporal) position, mean, then the biased
    variance sum((x - mean)^2) / count, both in float64;
    y = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c]."""
    x = _f64(x)
    n, c = x.shape[:2]
    assert c % groups == 0
    cg = c // groups
    y = np.empty_like(x)
    for b in range(n):
        for g in range(groups):
            seg = x[b, g * cg:(g + 1) * cg]
            mean = seg.sum() / seg.size
            var = ((seg - mean) ** 2).sum() / seg.size
            y[b, g * cg:(g + 1) * cg] = (seg - mean) / np.sqrt(var + eps)
    shape = (1, c) + (1,) * (x.ndim - 2)
    return y * _f64(gamma).reshape(shape) + _f64(beta).reshape(shape)


def silu(x):
    """[vae3d] fn silu: v / (1 + exp(-v))."""
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


def group_norm_silu(x, gamma, beta, groups=32, eps=1e-6):
    return silu(group_norm(x, gamma, beta, groups, eps))


def upsample_nearest2x(x):
    """[vae] VaeUpRef: nearest-2x upsample, u[n,c,i,j] = x[n,c,i//2,j//2]."""
    x = _f64(x)
    h, w = x.shape[2], x.shape[3]
    rows = np.arange(2 * h) // 2
    cols = np.arange(2 * w) // 2
    return x[:, :, rows][:, :, :, cols]


def upsample_conv(x, weight, bias):
    """[vae] VaeUpRef: nearest-2x upsample followed by the upsample conv."""
    return conv2d(upsample_nearest2x(x), weight, bias)


def resnet(x, p, groups=32, eps=1e-6):
    """[vae] VaeResnetRef: x + conv2(silu(norm2(conv1(silu(norm1(x)))))), the
    skip going through the 1x1 shortcut when in/out channels differ.

    ``p`` holds norm1/conv1/norm2/conv2 (and conv_shortcut) as
    (weight, bias) pairs. Reading (page silent): the shortcut is a 1x1 conv
    with bias (a VaeConvRef carries a bias), and there is no output scale."""
    h = conv2d(group_norm_silu(x, *p["norm1"], groups, eps), *p["conv1"])
    h = conv2d(group_norm_silu(h, *p["norm2"], groups, eps), *p["conv2"])
    skip = conv2d(x, *p["conv_shortcut"]) if "conv_shortcut" in p else _f64(x)
    return skip + h


def softmax_rows(s):
    """[vae3d] fn softmax_inplace: subtract the row maximum, exponentiate,
    divide by the row sum."""
    s = _f64(s)
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def mid_attention(x, p, groups=32, eps=1e-6):
    """[vae] VaeAttnRef: GroupNorm, then token-major q/k/v Linear [c, c]
    (row-major out x in) + bias, softmax(q k^T / sqrt(c)) v, out Linear + bias,
    residual add onto the block input. Token index = i * W + j (row-major
    spatial order); c = channel count."""
    x = _f64(x)
    n, c, h, w = x.shape
    t = group_norm(x, *p["group_norm"], groups, eps)
    y = np.empty_like(x)
    for b in range(n):
        tok = t[b].reshape(c, h * w).T  # [HW, c]
        q = tok @ _f64(p["to_q"][0]).T + _f64(p["to_q"][1])
        k = tok @ _f64(p["to_k"][0]).T + _f64(p["to_k"][1])
        v = tok @ _f64(p["to_v"][0]).T + _f64(p["to_v"][1])
        a = softmax_rows(q @ k.T / np.sqrt(c)) @ v
        o = a @ _f64(p["to_out"][0]).T + _f64(p["to_out"][1])
        y[b] = x[b] + o.T.reshape(c, h, w)
    return y


def mid_attention_at(x, p, tokens, groups=32, eps=1e-6):
    """mid_attention evaluated for chosen query tokens only: the GroupNorm,
    k and v of every token, q and the softmax rows of the chosen tokens.
    ``tokens`` index i * W + j; returns [n, c, len(tokens)] (block output
    x + out-projection at those tokens)."""
    x = _f64(x)
    n, c, h, w = x.shape
    tokens = np.asarray(tokens, dtype=np.int64)
    t = group_norm(x, *p["group_norm"], groups, eps)
    y = np.empty((n, c, len(tokens)))
    for b in range(n):
        tok = t[b].reshape(c, h * w).T  # [HW, c]
        q = tok[tokens] @ _f64(p["to_q"][0]).T + _f64(p["to_q"][1])
        k = tok @ _f64(p["to_k"][0]).T + _f64(p["to_k"][1])
        v = tok @ _f64(p["to_v"][0]).T + _f64(p["to_v"][1])
        a = softmax_rows(q @ k.T / np.sqrt(c)) @ v
        o = a @ _f64(p["to_out"][0]).T + _f64(p["to_out"][1])
        y[b] = x[b].reshape(c, h * w)[:, tokens] + o.T
    return y


def _pairs(weights, prefix, names):
    out = {}
    for nm in names:
        key = f"{prefix}.{nm}.weight"
        if key in weights:
            out[nm] = (weights[key], weights[f"{prefix}.{nm}.bias"])
    return out


_RES = ("norm1", "conv1", "norm2", "conv2", "conv_shortcut")
_ATT = ("group_norm", "to_q", "to_k", "to_v", "to_out")


def up_block(x, weights, i, n_resnets, groups=32, eps=1e-6):
    """[vae] VaeUpRef: the block's resnets in order, then (if present) the
    nearest-2x upsample followed by the upsample conv."""
    for j in range(n_resnets):
        x = resnet(x, _pairs(weights, f"up_blocks.{i}.resnets.{j}", _RES), groups, eps)
    key = f"up_blocks.{i}.upsamplers.0.conv"
    if key + ".weight" in weights:
        x = upsample_conv(x, weights[key + ".weight"], weights[key + ".bias"])
    return x


def decode(z, weights, scaling_factor, shift_factor, n_up_blocks, n_resnets=3,
           groups=32, eps=1e-6, trace=None):
    """[vae] VaeDecoder / VaeChainArgs execution order: de-normalise, conv_in,
    mid resnet, mid attention, mid resnet, up blocks, GroupNorm + SiLU,
    conv_out. Returns the raw conv_out output (reading: the pages state no
    clamp or output range).

    ``trace``, when a list, receives (layer name, output) after each layer."""
    def rec(name, v):
        if trace is not None:
            trace.append((name, v))
        return v

    x = rec("denorm", denormalize(z, scaling_factor, shift_factor))
    x = rec("conv_in", conv2d(x, weights["conv_in.weight"], weights["conv_in.bias"]))
    x = rec("mid.res0", resnet(x, _pairs(weights, "mid.resnets.0", _RES), groups, eps))
    x = rec("mid.attn", mid_attention(x, _pairs(weights, "mid.attentions.0", _ATT), groups, eps))
    x = rec("mid.res1", resnet(x, _pairs(weights, "mid.resnets.1", _RES), groups, eps))
    for i in range(n_up_blocks):
        x = rec(f"up{i}", up_block(x, weights, i, n_resnets, groups, eps))
    x = rec("norm_out", group_norm_silu(x, weights["conv_norm_out.weight"],
                                        weights["conv_norm_out.bias"], groups, eps))
    return rec("conv_out", conv2d(x, weights["conv_out.weight"], weights["conv_out.bias"]))


def conv3d_causal(x, weight, bias=None):
    """[hand] "The CPU VAE code" (LTX: 3-D causal conv, causal padding on the
    time axis) and "GPU plan" step 1 (the 3-D im2col rows are
    out_t*out_h*out_w pixels by Cin*kt*kh*kw taps, with causal time padding).

    y[n,o,t,i,j] = b[o] + sum_{c,kt,ky,kx} w[o,c,kt,ky,kx] *
                   x[n, c, max(t + kt - (KT-1), 0), i + ky - 1, j + kx - 1]
    with zero spatial padding. Reading: the causal time padding prepends KT-1
    copies of the first frame (replicate padding), so frame indices below 0
    read frame 0."""
    x = _f64(x)
    w = _f64(weight)
    n, cin, t, h, wd = x.shape
    cout, _, kt_n, k, _ = w.shape
    p = k // 2
    xp = np.zeros((n, cin, t, h + 2 * p, wd + 2 * p))
    xp[:, :, :, p:p + h, p:p + wd] = x
    y = np.zeros((n, cout, t, h, wd))
    for b in range(n):
        for tt in range(t):
            for kt in range(kt_n):
                src = max(tt + kt - (kt_n - 1), 0)
                for ky in range(k):
                    for kx in range(k):
                        sh = xp[b, :, src, ky:ky + h, kx:kx + wd].reshape(cin, h * wd)
                        y[b, :, tt] += (w[:, :, kt, ky, kx] @ sh).reshape(cout, h, wd)
    if bias is not None:
        y += _f64(bias)[None, :, None, None, None]
    return y


def causal_stack(x, layers, groups=32, eps=1e-6):
    """The LTX-style 3-D causal conv slice: u_i = silu(gn_i(conv_i(u_{i-1})))
    for each layer. Reading of "residual every 2 convs": after every second
    layer the input of that pair is added (u_2 += u_0, u_4 += u_2, ...)."""
    u = [_f64(x)]
    for i, L in enumerate(layers, start=1):
        v = group_norm_silu(conv3d_causal(u[-1], L["weight"], L["bias"]),
                            L["gn_weight"], L["gn_bias"], groups, eps)
        if i % 2 == 0:
            v = v + u[i - 2]
        u.append(v)
    return u[-1]


def split_tiles(length, ratio, tile=256, min_overlap=64):
    """[tile] fn split_tiles: (starts, lens, overlaps) of one axis in pixels.
    At or under one tile: a single tile of the whole length. Otherwise the
    fewest tiles of exactly ``tile`` pixels whose overlaps, all at least
    ``min_overlap``, cover the length; the slack is then added to the
    overlaps ``ratio`` pixels at a time, round robin from the first, so that
    every tile start stays on the latent grid."""
    if tile >= length:
        return [0], [length], []
    n = -(-length // tile)
    while tile * n < min_overlap * (n - 1) + length:
        n += 1
    overlaps = [min_overlap] * (n - 1)
    slack = tile * n - sum(overlaps) - length
    for i in range(slack // ratio):
        overlaps[i % (n - 1)] += ratio
    starts = [0]
    for i in range(n - 1):
        starts.append(starts[i] + tile - overlaps[i])
    return starts, [tile] * n, overlaps


def blend_tiles(tiles, height, width, ys, yo, xs, xo):
    """[tile] VideoVae::decode_clip's assembly of decoded tiles
    ``tiles[i][j]`` ([c, th, tw] each) into a [c, height, width] image, in
    raster order. Tile (i, j): its first yo[i-1] rows are cross-faded with the
    last yo[i-1] rows of the tile above as that tile was decoded (before its
    own blending), weights 1 - k/e and k/e at row k (fn blend, dim 2); then
    its first xo[j-1] columns likewise with the last xo[j-1] columns of the
    tile to its left as decoded (dim 3); then its last yo[i] rows and xo[j]
    columns are dropped
    (fn crop) unless it is the last of its row / column, and what is left is
    written at the running output position."""
    c = tiles[0][0].shape[0]
    out = np.zeros((c, height, width))
    oy = 0
    for i in range(len(ys)):
        ox = 0
        th = tw = 0
        for j in range(len(xs)):
            raw = _f64(tiles[i][j])
            th, tw = raw.shape[1], raw.shape[2]
            t = raw.copy()
            if i > 0:
                above = _f64(tiles[i - 1][j])
                e = min(yo[i - 1], above.shape[1], th)
                for k in range(e):
                    wb = k / e
                    t[:, k, :] = above[:, above.shape[1] - e + k, :] * (1 - wb) + t[:, k, :] * wb
            if j > 0:
                left = _f64(tiles[i][j - 1])
                e = min(xo[j - 1], left.shape[2], tw)
                for k in range(e):
                    wb = k / e
                    t[:, :, k] = left[:, :, left.shape[2] - e + k] * (1 - wb) + t[:, :, k] * wb
            if i + 1 < len(ys):
                t = t[:, :th - yo[i], :]
            if j + 1 < len(xs):
                t = t[:, :, :tw - xo[j]]
            out[:, oy:oy + t.shape[1], ox:ox + t.shape[2]] = t
            ox += t.shape[2]
            th = t.shape[1]
        oy += th
    return out


def tiled_decode(z, weights, scaling_factor, shift_factor, n_up_blocks, tile=256,
                 min_overlap=64, n_resnets=3, groups=32, eps=1e-6):
    """[tile] decode_clip applied to this decoder: split the output plane
    with split_tiles along each axis (ratio = the decoder's 2^upsamples
    latent-to-pixel factor), decode each tile's latent crop on its own with
    ``decode``, and assemble them with blend_tiles. Each tile sees only its
    own latents (GroupNorm statistics and attention included), so the
    result differs from the whole-image decode except when one tile covers
    the image."""
    z = _f64(z)
    n, _, zh, zw = z.shape
    up = [f"up_blocks.{i}.upsamplers.0.conv.weight" in weights for i in range(n_up_blocks)]
    r = 2 ** sum(up)
    height, width = zh * r, zw * r
    ys, yl, yo = split_tiles(height, r, tile, min_overlap)
    xs, xl, xo = split_tiles(width, r, tile, min_overlap)
    outs = []
    for b in range(n):
        tiles = [[decode(z[b:b + 1, :, ys[i] // r:(ys[i] + yl[i]) // r,
                           xs[j] // r:(xs[j] + xl[j]) // r],
                         weights, scaling_factor, shift_factor, n_up_blocks, n_resnets,
                         groups, eps)[0]
                  for j in range(len(xs))] for i in range(len(ys))]
        outs.append(blend_tiles(tiles, height, width, ys, yo, xs, xo))
    return np.stack(outs)


def upsample_nearest2x_spatial(x):
    """Nearest-2x upsample of every frame of a [n, c, t, h, w] video
    ([vae] VaeUpRef's upsample, per frame; time is kept)."""
    x = _f64(x)
    h, w = x.shape[3], x.shape[4]
    rows = np.arange(2 * h) // 2
    cols = np.arange(2 * w) // 2
    return x[:, :, :, rows][:, :, :, :, cols]


def resnet3d(x, p, groups=32, eps=1e-6):
    """resnet with every 3x3 conv a causal 3x3x3 conv (conv3d_causal) and
    GroupNorm over (t, h, w); the 1x1 shortcut acts on every frame."""
    x = _f64(x)
    h = conv3d_causal(group_norm_silu(x, *p["norm1"], groups, eps), *p["conv1"])
    h = conv3d_causal(group_norm_silu(h, *p["norm2"], groups, eps), *p["conv2"])
    if "conv_shortcut" in p:
        w, b = p["conv_shortcut"]
        w = _f64(w).reshape(w.shape[0], -1)
        skip = np.einsum("oc,ncthw->nothw", w, x) + _f64(b)[None, :, None, None, None]
    else:
        skip = x
    return skip + h


def causal_decode(z, weights, scaling_factor, shift_factor, n_up_blocks, n_mid=2,
                  n_resnets=2, groups=32, eps=1e-6):
    """[hand] "The CPU VAE code" (LtxVaeDecoder::decode: a 3-D causal decode,
    causal padding on the time axis) as a structural decoder: the pages give
    no LTX architecture constants, so the structure is the 2-D decoder's
    ([vae] VaeChainArgs order) with every conv a causal 3x3x3 conv and
    GroupNorm over (t, h, w): de-normalise, conv_in, the mid resnets (no
    attention), up blocks of resnets each followed (but the last) by a
    per-frame nearest-2x spatial upsample and a causal conv, GroupNorm+SiLU,
    conv_out. z [n, c, t, h, w] -> [n, 3, t, 8h, 8w] for three upsamples;
    frames stay frames (no temporal upsampling is read into the pages)."""
    x = denormalize(z, scaling_factor, shift_factor)
    x = conv3d_causal(x, weights["conv_in.weight"], weights["conv_in.bias"])
    for m in range(n_mid):
        x = resnet3d(x, _pairs(weights, f"mid.resnets.{m}", _RES), groups, eps)
    for i in range(n_up_blocks):
        for j in range(n_resnets):
            x = resnet3d(x, _pairs(weights, f"up_blocks.{i}.resnets.{j}", _RES), groups, eps)
        key = f"up_blocks.{i}.upsamplers.0.conv"
        if key + ".weight" in weights:
            x = conv3d_causal(upsample_nearest2x_spatial(x), weights[key + ".weight"],
                              weights[key + ".bias"])
    x = group_norm_silu(x, weights["conv_norm_out.weight"], weights["conv_norm_out.bias"],
                        groups, eps)
    return conv3d_causal(x, weights["conv_out.weight"], weights["conv_out.bias"])
