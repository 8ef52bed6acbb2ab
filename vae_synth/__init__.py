"""Seeded synthetic inputs for the FLUX-class AutoencoderKL latent decoder.

This module draws random numbers and fixes tensor shapes and names; it holds
none of the decoder's arithmetic. Both the CPU oracle (through the tests and the
bench) and the CUDA path receive the arrays made here, so the two sides always
see identical inputs.

Shapes follow the decoder the cortiq-engine ``vae`` module documents
(structs ``VaeDecoder``, ``VaeChainArgs``, ``VaeResnetRef``, ``VaeAttnRef``,
``VaeUpRef``): latent ``[B,16,h,w]`` -> RGB ``[B,3,8h,8w]``; conv_in; a mid block
of resnet / single-head attention / resnet; up blocks over
``reversed(block_out_channels)`` with three resnets each (1x1 shortcut when the
channel count changes) and a nearest-2x upsample + 3x3 conv on all but the last;
GroupNorm(32)+SiLU; conv_out to 3 channels.

Init recipe (variances, not standard deviations): conv / linear weights
``N(0, 1/(Cin*k*k))``, biases ``N(0, 0.01)``, GroupNorm gamma ``1 + N(0, 0.1)``,
beta ``N(0, 0.1)``, latents ``N(0, 1)``. Every tensor is drawn in float64 from
``numpy.random.default_rng`` and cast to float32, one tensor after the other in
chain execution order.
"""
from __future__ import annotations

import numpy as np

LATENT_CHANNELS = 16
SCALING_FACTOR = 0.3611
SHIFT_FACTOR = 0.1159
GN_GROUPS = 32
GN_EPS = 1e-6
RESNETS_PER_UP_BLOCK = 3

# Named decoder architectures: block_out_channels as a diffusers config lists them.
ARCHS = {
    "tiny": (32, 64, 128, 128),
    "flux": (128, 256, 512, 512),
}

# Workloads (name -> description). Seeds are 1000 + index.
WORKLOADS = {
    "tiny_decoder": dict(index=0, arch="tiny", latent=(1, 16, 8, 8)),
    "op_sweep": dict(index=1, convs=((128, 512), (256, 256), (512, 128), (512, 64))),
    "decoder_256": dict(index=2, arch="flux", latent=(1, 16, 32, 32)),
    "decoder_1024": dict(index=3, arch="flux", latent=(1, 16, 128, 128)),
    "decoder_512_b4": dict(index=3, arch="flux", latent=(4, 16, 64, 64)),
    "causal3d_stack": dict(index=4, shape=(1, 128, 17, 128, 128), n_convs=5),
}


def seed_of(workload: str) -> int:
    return 1000 + WORKLOADS[workload]["index"]


class _Drawer:
    """One float64 normal stream; each draw is cast to float32."""

    def __init__(self, seed):
        self.rng = np.random.default_rng(seed)

    def normal(self, shape, var, mean=0.0):
        v = self.rng.standard_normal(size=shape) * np.sqrt(var) + mean
        return v.astype(np.float32)


def _conv(d, out, name, cout, cin, k):
    out[name + ".weight"] = d.normal((cout, cin, k, k), 1.0 / (cin * k * k))
    out[name + ".bias"] = d.normal((cout,), 0.01)


def _norm(d, out, name, c):
    out[name + ".weight"] = d.normal((c,), 0.1, mean=1.0)
    out[name + ".bias"] = d.normal((c,), 0.1)


def _linear(d, out, name, c):
    out[name + ".weight"] = d.normal((c, c), 1.0 / c)
    out[name + ".bias"] = d.normal((c,), 0.01)


def _resnet(d, out, name, cin, cout):
    _norm(d, out, name + ".norm1", cin)
    _conv(d, out, name + ".conv1", cout, cin, 3)
    _norm(d, out, name + ".norm2", cout)
    _conv(d, out, name + ".conv2", cout, cout, 3)
    if cin != cout:
        _conv(d, out, name + ".conv_shortcut", cout, cin, 1)


def decoder_layout(arch: str):
    """Up-block plan: list of (cin_of_first_resnet, cout, has_upsample)."""
    rev = list(reversed(ARCHS[arch]))
    plan, prev = [], rev[0]
    for i, c in enumerate(rev):
        plan.append((prev, c, i < len(rev) - 1))
        prev = c
    return rev, plan


def make_decoder_weights(arch: str, seed: int) -> dict:
    """All decoder tensors, float32, keyed by diffusers-style names."""
    d = _Drawer([seed, 0])
    rev, plan = decoder_layout(arch)
    c0 = rev[0]
    w: dict = {}
    _conv(d, w, "conv_in", c0, LATENT_CHANNELS, 3)
    _resnet(d, w, "mid.resnets.0", c0, c0)
    _norm(d, w, "mid.attentions.0.group_norm", c0)
    for p in ("to_q", "to_k", "to_v", "to_out"):
        _linear(d, w, "mid.attentions.0." + p, c0)
    _resnet(d, w, "mid.resnets.1", c0, c0)
    for i, (cin, cout, up) in enumerate(plan):
        for j in range(RESNETS_PER_UP_BLOCK):
            _resnet(d, w, f"up_blocks.{i}.resnets.{j}", cin if j == 0 else cout, cout)
        if up:
            _conv(d, w, f"up_blocks.{i}.upsamplers.0.conv", cout, cout, 3)
    _norm(d, w, "conv_norm_out", rev[-1])
    _conv(d, w, "conv_out", 3, rev[-1], 3)
    return w


# 3-D causal decoders (LTX-style structure, random init): block_out_channels
# as for the 2-D decoder; latent channels; resnets in the mid block.
CAUSAL_ARCHS = {
    "causal_tiny": dict(channels=(32, 32, 64, 64), latent_channels=16, mid_resnets=2),
    "causal_small": dict(channels=(64, 128, 256, 256), latent_channels=16, mid_resnets=2),
}


def _conv3(d, out, name, cout, cin):
    out[name + ".weight"] = d.normal((cout, cin, 3, 3, 3), 1.0 / (cin * 27))
    out[name + ".bias"] = d.normal((cout,), 0.01)


def _resnet3(d, out, name, cin, cout):
    _norm(d, out, name + ".norm1", cin)
    _conv3(d, out, name + ".conv1", cout, cin)
    _norm(d, out, name + ".norm2", cout)
    _conv3(d, out, name + ".conv2", cout, cout)
    if cin != cout:
        _conv(d, out, name + ".conv_shortcut", cout, cin, 1)


def causal_decoder_layout(arch: str):
    """(reversed channels, up-block plan [(cin, cout, has_upsample)], latent
    channels, mid resnets) of a 3-D causal decoder architecture."""
    a = CAUSAL_ARCHS[arch]
    rev = list(reversed(a["channels"]))
    plan, prev = [], rev[0]
    for i, c in enumerate(rev):
        plan.append((prev, c, i < len(rev) - 1))
        prev = c
    return rev, plan, a["latent_channels"], a["mid_resnets"]


def make_causal_decoder_weights(arch: str, seed: int, resnets_per_block: int = 2) -> dict:
    """All tensors of a 3-D causal decoder (3x3x3 convs [cout, cin, 3, 3, 3],
    1x1x1 shortcuts stored [cout, cin, 1, 1]), float32, diffusers-style names,
    drawn in execution order with the 2-D decoder's init recipe (conv weights
    N(0, 1/(Cin*27)))."""
    d = _Drawer([seed, 8])
    rev, plan, lc, n_mid = causal_decoder_layout(arch)
    c0 = rev[0]
    w: dict = {}
    _conv3(d, w, "conv_in", c0, lc)
    for m in range(n_mid):
        _resnet3(d, w, f"mid.resnets.{m}", c0, c0)
    for i, (cin, cout, up) in enumerate(plan):
        for j in range(resnets_per_block):
            _resnet3(d, w, f"up_blocks.{i}.resnets.{j}", cin if j == 0 else cout, cout)
        if up:
            _conv3(d, w, f"up_blocks.{i}.upsamplers.0.conv", cout, cout)
    _norm(d, w, "conv_norm_out", rev[-1])
    _conv3(d, w, "conv_out", 3, rev[-1])
    return w


def make_latent(shape, seed: int) -> np.ndarray:
    return _Drawer([seed, 1]).normal(shape, 1.0)


def make_normal(shape, seed: int, var: float = 1.0, stream: int = 2) -> np.ndarray:
    return _Drawer([seed, stream]).normal(shape, var)


def make_conv_params(cout, cin, k, seed, stream=3):
    d = _Drawer([seed, stream])
    w = {}
    _conv(d, w, "c", cout, cin, k)
    return w["c.weight"], w["c.bias"]


def make_norm_params(c, seed, stream=4):
    d = _Drawer([seed, stream])
    w = {}
    _norm(d, w, "n", c)
    return w["n.weight"], w["n.bias"]


def make_attn_params(c, seed, stream=5):
    d = _Drawer([seed, stream])
    w = {}
    _norm(d, w, "group_norm", c)
    for p in ("to_q", "to_k", "to_v", "to_out"):
        _linear(d, w, p, c)
    return w


def make_causal_stack(shape, n_convs, seed):
    """Input and params for the 3-D causal conv stack (3x3x3 kernels)."""
    n, c, t, h, w_ = shape
    d = _Drawer([seed, 6])
    x = d.normal(shape, 1.0)
    layers = []
    for _ in range(n_convs):
        wt = d.normal((c, c, 3, 3, 3), 1.0 / (c * 27))
        b = d.normal((c,), 0.01)
        g = d.normal((c,), 0.1, mean=1.0)
        be = d.normal((c,), 0.1)
        layers.append(dict(weight=wt, bias=b, gn_weight=g, gn_bias=be))
    return x, layers


def integer_tensor(shape, seed, lo=-4, hi=4, stream=7):
    """Small integers stored as float32: products and sums of these are exact in
    TF32 x TF32 -> FP32 arithmetic, so index/gather errors show as exact mismatches."""
    rng = np.random.default_rng([seed, stream])
    return rng.integers(lo, hi + 1, size=shape).astype(np.float32)
