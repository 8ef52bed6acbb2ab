"""Pins for the CPU oracle: each function is checked against something other
than itself -- hand-worked values, brute force on tiny inputs, closed forms,
invariants, and library routines in float64 where the operation reduces to one.
No GPU is used."""
import itertools
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
import vae_synth as S

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ conv2d

def _conv_brute(x, w, b):
    """Pure-Python loops straight from the definition (tiny inputs only)."""
    n, cin, h, wd = x.shape
    cout, _, k, _ = w.shape
    p = k // 2
    y = np.zeros((n, cout, h, wd))
    for bb, o, i, j in itertools.product(range(n), range(cout), range(h), range(wd)):
        acc = 0.0 if b is None else float(b[o])
        for c, ky, kx in itertools.product(range(cin), range(k), range(k)):
            ii, jj = i + ky - p, j + kx - p
            if 0 <= ii < h and 0 <= jj < wd:
                acc += float(w[o, c, ky, kx]) * float(x[bb, c, ii, jj])
        y[bb, o, i, j] = acc
    return y


def test_conv_hand_golden(golden_dir):
    g = _load(golden_dir, "conv3x3_hand.json")
    x = np.array(g["x"], dtype=np.float64)[None, None]
    for case in g["cases"]:
        w = np.array(case["kernel"], dtype=np.float64)[None, None]
        y = O.conv2d(x, w, np.array([case["bias"]]))
        np.testing.assert_array_equal(y[0, 0], np.array(case["y"], dtype=np.float64))


@pytest.mark.parametrize("k", [1, 3])
@pytest.mark.parametrize("shape", [(1, 2, 3, 4), (2, 3, 5, 2), (1, 1, 1, 1)])
def test_conv_brute_force(k, shape):
    r = _rng(11)
    x = r.standard_normal(shape)
    w = r.standard_normal((3, shape[1], k, k))
    b = r.standard_normal(3)
    np.testing.assert_allclose(O.conv2d(x, w, b), _conv_brute(x, w, b), rtol=0, atol=1e-12)


def test_conv_1x1_identity_reproduces_input():
    x = _rng(1).standard_normal((2, 5, 4, 3))
    w = np.eye(5)[:, :, None, None]
    np.testing.assert_array_equal(O.conv2d(x, w), x)


def test_conv_3x3_centre_identity_reproduces_input():
    x = _rng(2).standard_normal((1, 4, 5, 6))
    w = np.zeros((4, 4, 3, 3))
    for c in range(4):
        w[c, c, 1, 1] = 1.0
    np.testing.assert_array_equal(O.conv2d(x, w), x)


def test_conv_linear():
    r = _rng(3)
    x1, x2 = r.standard_normal((2, 1, 3, 6, 5))
    w = r.standard_normal((4, 3, 3, 3))
    a, b = 0.7, -1.9
    np.testing.assert_allclose(O.conv2d(a * x1 + b * x2, w),
                               a * O.conv2d(x1, w) + b * O.conv2d(x2, w), atol=1e-12)


@pytest.mark.parametrize("i0,j0", [(2, 3), (0, 0), (4, 5), (0, 5)])
def test_conv_impulse_response(i0, j0):
    """A unit impulse at (i0,j0) lands w[o,c,ky,kx] at (i0-ky+1, j0-kx+1);
    taps that would fall outside the image are dropped (zero padding)."""
    h, w_ = 5, 6
    x = np.zeros((1, 2, h, w_))
    x[0, 1, i0, j0] = 1.0
    w = _rng(4).standard_normal((3, 2, 3, 3))
    y = O.conv2d(x, w)
    expect = np.zeros((1, 3, h, w_))
    for ky, kx in itertools.product(range(3), range(3)):
        i, j = i0 - ky + 1, j0 - kx + 1
        if 0 <= i < h and 0 <= j < w_:
            expect[0, :, i, j] = w[:, 1, ky, kx]
    np.testing.assert_array_equal(y, expect)


@pytest.mark.parametrize("k", [1, 3])
def test_conv_vs_torch_float64(k):
    r = _rng(5)
    x = r.standard_normal((2, 7, 9, 11))
    w = r.standard_normal((5, 7, k, k))
    b = r.standard_normal(5)
    ref = F.conv2d(_t(x), _t(w), _t(b), padding=k // 2).numpy()
    np.testing.assert_allclose(O.conv2d(x, w, b), ref, atol=1e-11)


# ------------------------------------------------------------------ GroupNorm

def test_groupnorm_hand_golden(golden_dir):
    g = _load(golden_dir, "groupnorm_hand.json")
    y = O.group_norm(np.array(g["x"]), np.array(g["gamma"]), np.array(g["beta"]),
                     groups=g["groups"], eps=g["eps"])
    np.testing.assert_allclose(y, np.array(g["y"]), rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("shape,groups", [((2, 64, 5, 3), 32), ((1, 32, 4, 4), 32),
                                          ((1, 64, 2, 3, 3), 32), ((1, 6, 3, 3), 3)])
def test_groupnorm_moments_before_affine(shape, groups):
    """With gamma=1, beta=0 every (sample, group) has mean 0 and variance
    var/(var+eps) exactly (biased variance)."""
    r = _rng(6)
    x = 3.0 + 2.5 * r.standard_normal(shape)
    c = shape[1]
    eps = 1e-6
    y = O.group_norm(x, np.ones(c), np.zeros(c), groups, eps)
    cg = c // groups
    for b in range(shape[0]):
        for gi in range(groups):
            seg_x = x[b, gi * cg:(gi + 1) * cg]
            seg_y = y[b, gi * cg:(gi + 1) * cg]
            v = seg_x.var()
            assert abs(seg_y.mean()) < 1e-12
            assert abs(seg_y.var() - v / (v + eps)) < 1e-12


def test_groupnorm_constant_group_gives_beta():
    x = np.full((1, 4, 3, 3), 7.25)
    gamma = np.array([2.0, 3.0, 4.0, 5.0])
    beta = np.array([0.1, -0.2, 0.3, -0.4])
    y = O.group_norm(x, gamma, beta, groups=2)
    np.testing.assert_array_equal(y, np.broadcast_to(beta[None, :, None, None], x.shape))


@pytest.mark.parametrize("shape", [(2, 64, 6, 5), (1, 128, 3, 2, 4)])
def test_groupnorm_vs_torch_float64(shape):
    r = _rng(7)
    x = r.standard_normal(shape) + 0.5
    c = shape[1]
    gamma, beta = r.standard_normal(c), r.standard_normal(c)
    ref = F.group_norm(_t(x), 32, _t(gamma), _t(beta), eps=1e-6).numpy()
    np.testing.assert_allclose(O.group_norm(x, gamma, beta, 32, 1e-6), ref, atol=1e-12)


# ------------------------------------------------------------------ SiLU

def test_silu_closed_forms():
    x = np.linspace(-30, 30, 1001)
    s = O.silu(x)
    # silu(x) - silu(-x) = x * (sigma(x) + sigma(-x)) = x
    np.testing.assert_allclose(s - O.silu(-x), x, atol=1e-12)
    assert O.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(O.silu(np.array([np.log(3.0)])), [np.log(3.0) * 0.75], rtol=1e-15)
    np.testing.assert_allclose(s, F.silu(_t(x)).numpy(), atol=1e-14)


# ------------------------------------------------------------------ softmax / attention

def test_softmax_hand_golden(golden_dir):
    g = _load(golden_dir, "softmax_hand.json")
    np.testing.assert_allclose(O.softmax_rows(np.array(g["s"])), np.array(g["p"]), rtol=1e-15)


def test_softmax_rows_sum_to_one_and_shift_invariant():
    s = _rng(8).standard_normal((7, 33)) * 20
    p = O.softmax_rows(s)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    np.testing.assert_allclose(O.softmax_rows(s + 123.0), p, atol=1e-14)
    np.testing.assert_allclose(p, torch.softmax(_t(s), dim=-1).numpy(), atol=1e-15)


def _attn_params(c, seed):
    w = S.make_attn_params(c, seed)
    return {k: (w[k + ".weight"], w[k + ".bias"]) for k in
            ("group_norm", "to_q", "to_k", "to_v", "to_out")}


def _attn_torch(x, p, groups=32):
    """Independent restatement with torch float64 library routines."""
    xt = _t(x)
    n, c, h, w = xt.shape
    t = F.group_norm(xt, groups, _t(p["group_norm"][0]), _t(p["group_norm"][1]), eps=1e-6)
    tok = t.reshape(n, c, h * w).transpose(1, 2)
    q = F.linear(tok, _t(p["to_q"][0]), _t(p["to_q"][1]))
    k = F.linear(tok, _t(p["to_k"][0]), _t(p["to_k"][1]))
    v = F.linear(tok, _t(p["to_v"][0]), _t(p["to_v"][1]))
    a = F.scaled_dot_product_attention(q[:, None], k[:, None], v[:, None])[:, 0]
    o = F.linear(a, _t(p["to_out"][0]), _t(p["to_out"][1]))
    return (xt + o.transpose(1, 2).reshape(n, c, h, w)).numpy()


def test_attention_hand_golden(golden_dir):
    """Two tokens, two channels, worked by hand (the fixture states the
    steps): pins GroupNorm before the projections, the out x in orientation of
    every Linear, the biases, the 1/sqrt(c) scale and the residual add."""
    g = _load(golden_dir, "attention_hand.json")
    a = {k: np.array(v, dtype=np.float64) for k, v in g.items() if k not in ("source",)}
    p = {"group_norm": (a["gamma"], a["beta"]), "to_q": (a["wq"], a["bq"]),
         "to_k": (a["wk"], a["bk"]), "to_v": (a["wv"], a["bv"]), "to_out": (a["wo"], a["bo"])}
    y = O.mid_attention(a["x"], p, groups=int(g["groups"]), eps=float(g["eps"]))
    np.testing.assert_allclose(y, a["y"], rtol=0, atol=1e-13)


@pytest.mark.parametrize("shape", [(1, 64, 4, 5), (2, 32, 3, 3)])
def test_attention_vs_torch_sdpa(shape):
    x = _rng(9).standard_normal(shape)
    p = _attn_params(shape[1], 9)
    np.testing.assert_allclose(O.mid_attention(x, p), _attn_torch(x, p), atol=1e-11)


def test_attention_single_token_ignores_q_and_k():
    """One token: the softmax row is [1], so q and k weights cannot matter."""
    x = _rng(10).standard_normal((1, 64, 1, 1))
    p = _attn_params(64, 10)
    p2 = dict(p)
    r = _rng(99)
    p2["to_q"] = (r.standard_normal((64, 64)), r.standard_normal(64))
    p2["to_k"] = (r.standard_normal((64, 64)), r.standard_normal(64))
    np.testing.assert_allclose(O.mid_attention(x, p), O.mid_attention(x, p2), atol=1e-12)


def test_attention_identical_keys_average_values():
    """Equal keys for every token (zero k weight): uniform attention, so the
    block adds (mean of v) @ Wo^T + bo to every token."""
    c = 32
    x = _rng(12).standard_normal((1, c, 3, 4))
    p = _attn_params(c, 12)
    p["to_k"] = (np.zeros((c, c)), p["to_k"][1])
    y = O.mid_attention(x, p)
    t = O.group_norm(x, *p["group_norm"], 32, 1e-6)[0].reshape(c, -1).T
    v = t @ p["to_v"][0].astype(np.float64).T + p["to_v"][1]
    o = v.mean(axis=0) @ p["to_out"][0].astype(np.float64).T + p["to_out"][1]
    np.testing.assert_allclose(y[0] - x[0], np.broadcast_to(o[:, None, None], x[0].shape), atol=1e-12)


def test_attention_permutation_equivariant():
    """GroupNorm and softmax attention commute with a spatial permutation."""
    x = _rng(13).standard_normal((1, 32, 4, 6))
    p = _attn_params(32, 13)
    perm = _rng(14).permutation(24)
    xp = x.reshape(1, 32, 24)[:, :, perm].reshape(1, 32, 4, 6)
    y = O.mid_attention(x, p).reshape(1, 32, 24)[:, :, perm].reshape(1, 32, 4, 6)
    np.testing.assert_allclose(O.mid_attention(xp, p), y, atol=1e-12)


# ------------------------------------------------------------------ upsample

def test_upsample_hand_golden(golden_dir):
    g = _load(golden_dir, "upsample_hand.json")
    y = O.upsample_nearest2x(np.array(g["x"], dtype=np.float64)[None, None])
    np.testing.assert_array_equal(y[0, 0], np.array(g["y"], dtype=np.float64))


def test_upsample_replicates_2x2_blocks_and_matches_torch():
    x = _rng(15).standard_normal((2, 3, 5, 7))
    u = O.upsample_nearest2x(x)
    assert u.shape == (2, 3, 10, 14)
    for dy, dx in itertools.product(range(2), range(2)):
        np.testing.assert_array_equal(u[:, :, dy::2, dx::2], x)
    np.testing.assert_array_equal(u, F.interpolate(_t(x), scale_factor=2, mode="nearest").numpy())


def test_upsample_conv_vs_torch():
    r = _rng(16)
    x = r.standard_normal((1, 4, 5, 6))
    w, b = r.standard_normal((3, 4, 3, 3)), r.standard_normal(3)
    ref = F.conv2d(F.interpolate(_t(x), scale_factor=2, mode="nearest"), _t(w), _t(b), padding=1)
    np.testing.assert_allclose(O.upsample_conv(x, w, b), ref.numpy(), atol=1e-11)


# ------------------------------------------------------------------ 3-D causal conv

def test_causal3d_hand_golden(golden_dir):
    g = _load(golden_dir, "causal3d_hand.json")
    x = np.array(g["x_frames"])[None, None, :, None, None]
    w = np.zeros((1, 1, 3, 3, 3))
    w[0, 0, :, 1, 1] = g["kt_weights"]
    y = O.conv3d_causal(x, w)
    np.testing.assert_array_equal(y[0, 0, :, 0, 0], np.array(g["y_frames"]))


def _causal_torch(x, w, b):
    """Replicate-pad the first frame KT-1 times, zero-pad space, F.conv3d."""
    xt = _t(x)
    kt = w.shape[2]
    front = xt[:, :, :1].expand(-1, -1, kt - 1, -1, -1)
    xp = torch.cat([front, xt], dim=2)
    return F.conv3d(xp, _t(w), _t(b), padding=(0, 1, 1)).numpy()


def test_causal3d_vs_torch_conv3d():
    r = _rng(17)
    x = r.standard_normal((1, 3, 5, 4, 6))
    w, b = r.standard_normal((2, 3, 3, 3, 3)), r.standard_normal(2)
    np.testing.assert_allclose(O.conv3d_causal(x, w, b), _causal_torch(x, w, b), atol=1e-11)


def test_causal3d_single_frame_is_2d_conv_with_summed_time_taps():
    r = _rng(18)
    x = r.standard_normal((1, 3, 1, 5, 4))
    w, b = r.standard_normal((2, 3, 3, 3, 3)), r.standard_normal(2)
    y = O.conv3d_causal(x, w, b)[:, :, 0]
    y2 = O.conv2d(x[:, :, 0], w.sum(axis=2), b)
    np.testing.assert_allclose(y, y2, atol=1e-12)


def test_causal3d_is_causal():
    r = _rng(19)
    x = r.standard_normal((1, 2, 6, 3, 3))
    w = r.standard_normal((2, 2, 3, 3, 3))
    y = O.conv3d_causal(x, w)
    x2 = x.copy()
    x2[:, :, 4] += 5.0
    y2 = O.conv3d_causal(x2, w)
    np.testing.assert_array_equal(y[:, :, :4], y2[:, :, :4])
    assert np.abs(y[:, :, 4:] - y2[:, :, 4:]).max() > 1e-3


def test_causal_stack_vs_torch_restatement():
    x, layers = S.make_causal_stack((1, 32, 4, 5, 6), 5, seed=20)
    u = [_t(x)]
    for i, L in enumerate(layers, start=1):
        v = F.silu(F.group_norm(_t(_causal_torch(u[-1].numpy(), L["weight"], L["bias"])), 32,
                                _t(L["gn_weight"]), _t(L["gn_bias"]), eps=1e-6))
        if i % 2 == 0:
            v = v + u[i - 2]
        u.append(v)
    np.testing.assert_allclose(O.causal_stack(x, layers), u[-1].numpy(), atol=1e-10)


# ------------------------------------------------------------------ resnet / chain

def _res_params(cin, cout, seed):
    w = {}
    d = S._Drawer([seed, 50])
    S._resnet(d, w, "r", cin, cout)
    return {k[2:].rsplit(".", 1)[0]: (w[k], w[k[:-6] + "bias"]) for k in w if k.endswith("weight")}


def test_resnet_zero_branch_is_skip():
    x = _rng(21).standard_normal((1, 64, 4, 4))
    p = _res_params(64, 64, 21)
    p["conv2"] = (np.zeros_like(p["conv2"][0]), np.zeros_like(p["conv2"][1]))
    np.testing.assert_array_equal(O.resnet(x, p), x)
    p = _res_params(64, 32, 22)
    p["conv2"] = (np.zeros_like(p["conv2"][0]), np.zeros_like(p["conv2"][1]))
    np.testing.assert_allclose(O.resnet(x, p), O.conv2d(x, *p["conv_shortcut"]), atol=0)


def _decode_torch(z, w, sf, sh, n_up):
    """The decoder restated with torch.nn.functional float64 calls."""
    T = lambda k: _t(w[k])  # noqa: E731

    def gns(x, pre, silu=True):
        y = F.group_norm(x, 32, T(pre + ".weight"), T(pre + ".bias"), eps=1e-6)
        return F.silu(y) if silu else y

    def conv(x, pre):
        wt = T(pre + ".weight")
        return F.conv2d(x, wt, T(pre + ".bias"), padding=wt.shape[-1] // 2)

    def res(x, pre):
        h = conv(gns(x, pre + ".norm1"), pre + ".conv1")
        h = conv(gns(h, pre + ".norm2"), pre + ".conv2")
        s = conv(x, pre + ".conv_shortcut") if pre + ".conv_shortcut.weight" in w else x
        return s + h

    def attn(x, pre):
        n, c, hh, ww = x.shape
        t = gns(x, pre + ".group_norm", silu=False).reshape(n, c, -1).transpose(1, 2)
        q, k, v = (F.linear(t, T(f"{pre}.{nm}.weight"), T(f"{pre}.{nm}.bias"))
                   for nm in ("to_q", "to_k", "to_v"))
        a = F.scaled_dot_product_attention(q[:, None], k[:, None], v[:, None])[:, 0]
        o = F.linear(a, T(pre + ".to_out.weight"), T(pre + ".to_out.bias"))
        return x + o.transpose(1, 2).reshape(n, c, hh, ww)

    x = _t(z) / sf + sh
    x = conv(x, "conv_in")
    x = res(x, "mid.resnets.0")
    x = attn(x, "mid.attentions.0")
    x = res(x, "mid.resnets.1")
    for i in range(n_up):
        for j in range(3):
            x = res(x, f"up_blocks.{i}.resnets.{j}")
        if f"up_blocks.{i}.upsamplers.0.conv.weight" in w:
            x = conv(F.interpolate(x, scale_factor=2, mode="nearest"), f"up_blocks.{i}.upsamplers.0.conv")
    x = gns(x, "conv_norm_out")
    return conv(x, "conv_out").numpy()


def test_denormalize_closed_forms():
    """z / scaling_factor + shift_factor, elementwise: z = s maps to 1 + t,
    z = 0 to t, and z = -t*s to 0 (it undoes the encoder-side (x - t) * s); a
    swapped order (z + t) / s or a product z * s + t fails every case."""
    s, t = 0.3611, 0.1159
    z = np.array([[[[s, 0.0], [-t * s, 2.0 * s]]]])
    want = np.array([[[[1.0 + t, t], [0.0, 2.0 + t]]]])
    np.testing.assert_allclose(O.denormalize(z, s, t), want, rtol=0, atol=1e-15)
    x = _rng(21).standard_normal((2, 16, 3, 5))
    np.testing.assert_allclose(O.denormalize((x - t) * s, s, t), x, rtol=0, atol=1e-14)


def test_tiny_decoder_vs_torch_restatement():
    w = S.make_decoder_weights("tiny", seed=1000)
    z = S.make_latent((1, 16, 4, 4), seed=1000)
    trace = []
    y = O.decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4, trace=trace)
    assert y.shape == (1, 3, 32, 32)
    assert [t[0] for t in trace] == ["denorm", "conv_in", "mid.res0", "mid.attn", "mid.res1",
                                     "up0", "up1", "up2", "up3", "norm_out", "conv_out"]
    ref = _decode_torch(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    np.testing.assert_allclose(y, ref, atol=1e-9, rtol=1e-9)


def test_decoder_weight_plan_shapes():
    """Structural pins of the up-block plan for the FLUX-class channel list."""
    w = S.make_decoder_weights("tiny", seed=0)
    assert w["conv_in.weight"].shape == (128, 16, 3, 3)
    assert w["up_blocks.2.resnets.0.conv_shortcut.weight"].shape == (64, 128, 1, 1)
    assert w["up_blocks.3.resnets.0.conv_shortcut.weight"].shape == (32, 64, 1, 1)
    assert "up_blocks.3.upsamplers.0.conv.weight" not in w
    assert "up_blocks.0.resnets.0.conv_shortcut.weight" not in w
    assert w["conv_out.weight"].shape == (3, 32, 3, 3)
    rev, plan = S.decoder_layout("flux")
    assert rev == [512, 512, 256, 128]
    assert plan == [(512, 512, True), (512, 512, True), (512, 256, True), (256, 128, False)]


# ------------------------------------------------------------------ sampled outputs
# The full-size parity tests evaluate the definitions at sampled outputs only;
# these pins hold the sampled forms to library routines and brute force.

@pytest.mark.parametrize("k", [1, 3])
def test_conv2d_at_every_pixel_matches_torch_and_brute_force(k):
    r = _rng(40 + k)
    x = r.standard_normal((2, 3, 5, 7))
    w, b = r.standard_normal((4, 3, k, k)), r.standard_normal(4)
    pix = np.array(list(itertools.product(range(2), range(5), range(7))))
    got = O.conv2d_at(x, w, b, pix)
    ref = F.conv2d(_t(x), _t(w), _t(b), padding=k // 2).numpy()
    np.testing.assert_allclose(got, ref[pix[:, 0], :, pix[:, 1], pix[:, 2]], atol=1e-12)
    brute = _conv_brute(x, w, b)
    np.testing.assert_allclose(got, brute[pix[:, 0], :, pix[:, 1], pix[:, 2]], atol=1e-12)


def test_conv2d_at_reads_a_channels_last_view():
    """The tests hand it NHWC activations as an NCHW view (no copy)."""
    r = _rng(44)
    x = r.standard_normal((1, 6, 4, 8)).astype(np.float32)
    w, b = r.standard_normal((5, 6, 3, 3)), r.standard_normal(5)
    nhwc = np.ascontiguousarray(np.moveaxis(x, 1, -1))
    pix = np.array([[0, 0, 0], [0, 3, 7], [0, 1, 4], [0, 2, 0]])
    np.testing.assert_array_equal(O.conv2d_at(np.moveaxis(nhwc, -1, 1), w, b, pix),
                                  O.conv2d_at(x, w, b, pix))


def test_upsample_conv_at_matches_torch():
    r = _rng(45)
    x = r.standard_normal((2, 4, 3, 5))
    w, b = r.standard_normal((3, 4, 3, 3)), r.standard_normal(3)
    ref = F.conv2d(F.interpolate(_t(x), scale_factor=2, mode="nearest"), _t(w), _t(b),
                   padding=1).numpy()
    pix = np.array(list(itertools.product(range(2), range(6), range(10))))
    np.testing.assert_allclose(O.upsample_conv_at(x, w, b, pix),
                               ref[pix[:, 0], :, pix[:, 1], pix[:, 2]], atol=1e-11)


def test_mid_attention_at_matches_torch_sdpa():
    x = _rng(46).standard_normal((2, 64, 4, 5))
    p = _attn_params(64, 46)
    tokens = np.array([0, 7, 19, 3])
    ref = _attn_torch(x, p).reshape(2, 64, 20)[:, :, tokens]
    np.testing.assert_allclose(O.mid_attention_at(x, p, tokens), ref, atol=1e-11)


# ------------------------------------------------------------------ tiled decode

def test_split_tiles_matches_the_page_values(golden_dir):
    g = _load(golden_dir, "tile_schedule.json")
    for case in g["cases"]:
        s, ln, o = O.split_tiles(case["length"], case["ratio"], g["tile"], g["min_overlap"])
        assert (s, ln, o) == (case["starts"], case["lens"], case["overlaps"]), case


@pytest.mark.parametrize("length,ratio,tile,ov", [(1024, 8, 256, 64), (800, 8, 256, 64),
                                                  (1000, 8, 512, 64), (264, 8, 256, 64),
                                                  (4096, 8, 512, 128)])
def test_split_tiles_cover_the_axis_on_the_latent_grid(length, ratio, tile, ov):
    s, ln, o = O.split_tiles(length, ratio, tile, ov)
    assert s[0] == 0 and s[-1] + ln[-1] == length and all(x == tile for x in ln)
    assert all(x >= ov for x in o) and all(x % ratio == 0 for x in s)
    assert all(s[i + 1] == s[i] + tile - o[i] for i in range(len(o)))


def _crops(img, ys, yl, xs, xl):
    return [[img[:, ys[i]:ys[i] + yl[i], xs[j]:xs[j] + xl[j]] for j in range(len(xs))]
            for i in range(len(ys))]


def test_blend_of_consistent_crops_rebuilds_the_image():
    """Tiles cut from one image agree on their overlaps, so every cross-fade
    returns the shared value: any offset, crop or placement mistake shows."""
    img = _rng(50).standard_normal((3, 800, 1000))
    ys, yl, yo = O.split_tiles(800, 8, 256, 64)
    xs, xl, xo = O.split_tiles(1000, 8, 256, 64)
    out = O.blend_tiles(_crops(img, ys, yl, xs, xl), 800, 1000, ys, yo, xs, xo)
    np.testing.assert_allclose(out, img, atol=1e-12)


def test_blend_cross_fades_linearly_from_the_earlier_tile():
    """Two tiles side by side, constant a and b: across the overlap of e
    columns the result runs a*(1 - k/e) + b*k/e, the earlier tile fading
    out; outside it each tile's own value."""
    xs, xl, xo = O.split_tiles(288, 16, 256, 64)  # two tiles, overlap 224
    a = np.full((1, 4, 256), 2.0)
    b = np.full((1, 4, 256), -3.0)
    out = O.blend_tiles([[a, b]], 4, 288, [0], [], xs, xo)
    e = xo[0]
    k = np.arange(e)
    np.testing.assert_allclose(out[0, :, xs[1]:xs[1] + e], np.broadcast_to(
        2.0 * (1 - k / e) + -3.0 * (k / e), (4, e)), atol=1e-14)
    assert (out[0, :, :xs[1]] == 2.0).all() and (out[0, :, xs[1] + e:] == -3.0).all()


def test_tiled_decode_with_one_tile_is_the_decode():
    w = S.make_decoder_weights("tiny", 3)
    z = S.make_latent((1, 16, 6, 7), 3)
    ref = O.decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    got = O.tiled_decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4, tile=64, min_overlap=16)
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------------ 3-D causal decoder

def _causal_conv_torch(x, w, b):
    """torch restatement: replicate frame 0 twice in front, zero-pad space,
    F.conv3d (cross-correlation)."""
    xp = torch.cat([x[:, :, :1], x[:, :, :1], x], dim=2)
    xp = F.pad(xp, (1, 1, 1, 1, 0, 0))
    return F.conv3d(xp, _t(w), _t(b))


def _causal_decode_torch(z, wts, n_up=4, n_mid=2, n_res=2):
    def gs(x, pre):
        return F.silu(F.group_norm(x, 32, _t(wts[pre + ".weight"]), _t(wts[pre + ".bias"]),
                                   eps=1e-6))

    def res(x, pre):
        h = _causal_conv_torch(gs(x, pre + ".norm1"), wts[pre + ".conv1.weight"],
                               wts[pre + ".conv1.bias"])
        h = _causal_conv_torch(gs(h, pre + ".norm2"), wts[pre + ".conv2.weight"],
                               wts[pre + ".conv2.bias"])
        if pre + ".conv_shortcut.weight" in wts:
            sw = _t(wts[pre + ".conv_shortcut.weight"])[:, :, :, :, None]
            x = F.conv3d(x, sw, _t(wts[pre + ".conv_shortcut.bias"]))
        return x + h

    x = _t(z) / S.SCALING_FACTOR + S.SHIFT_FACTOR
    x = _causal_conv_torch(x, wts["conv_in.weight"], wts["conv_in.bias"])
    for m in range(n_mid):
        x = res(x, f"mid.resnets.{m}")
    for i in range(n_up):
        for j in range(n_res):
            x = res(x, f"up_blocks.{i}.resnets.{j}")
        k = f"up_blocks.{i}.upsamplers.0.conv"
        if k + ".weight" in wts:
            x = F.interpolate(x, scale_factor=(1, 2, 2), mode="nearest")
            x = _causal_conv_torch(x, wts[k + ".weight"], wts[k + ".bias"])
    x = gs(x, "conv_norm_out")
    return _causal_conv_torch(x, wts["conv_out.weight"], wts["conv_out.bias"]).numpy()


def test_causal_decoder_vs_torch_restatement():
    w = S.make_causal_decoder_weights("causal_tiny", 11)
    z = S.make_latent((2, 16, 3, 3, 4), 11)
    got = O.causal_decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    assert got.shape == (2, 3, 3, 24, 32)
    np.testing.assert_allclose(got, _causal_decode_torch(z, w), atol=1e-10)


def test_causal_decoder_single_frame_is_the_2d_decoder_with_summed_time_taps():
    """With one frame every causal conv reads frame 0 through all three time
    taps, so the decoder is the 2-D decoder (no attention) whose 3x3 kernels
    are the 3x3x3 kernels summed over time: composed here from the pinned
    2-D oracle functions."""
    w = S.make_causal_decoder_weights("causal_tiny", 12)
    z = S.make_latent((1, 16, 1, 4, 3), 12)
    got = O.causal_decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)

    def w2(name):
        return np.asarray(w[name + ".weight"], np.float64).sum(axis=2), w[name + ".bias"]

    def res2(x, pre):
        p = {"norm1": (w[pre + ".norm1.weight"], w[pre + ".norm1.bias"]),
             "norm2": (w[pre + ".norm2.weight"], w[pre + ".norm2.bias"]),
             "conv1": w2(pre + ".conv1"), "conv2": w2(pre + ".conv2")}
        if pre + ".conv_shortcut.weight" in w:
            p["conv_shortcut"] = (w[pre + ".conv_shortcut.weight"], w[pre + ".conv_shortcut.bias"])
        return O.resnet(x, p)

    x = O.conv2d(O.denormalize(z[:, :, 0], S.SCALING_FACTOR, S.SHIFT_FACTOR), *w2("conv_in"))
    for m in range(2):
        x = res2(x, f"mid.resnets.{m}")
    for i in range(4):
        for j in range(2):
            x = res2(x, f"up_blocks.{i}.resnets.{j}")
        if f"up_blocks.{i}.upsamplers.0.conv.weight" in w:
            x = O.upsample_conv(x, *w2(f"up_blocks.{i}.upsamplers.0.conv"))
    x = O.group_norm_silu(x, w["conv_norm_out.weight"], w["conv_norm_out.bias"])
    ref = O.conv2d(x, *w2("conv_out"))
    np.testing.assert_allclose(got[:, :, 0], ref, atol=1e-10)
