"""Per-layer parity inside the decoder chain: every step of a decode, traced
out of the chain through vae_decode_chain_traced, against the float64 oracle
fed the GPU's own input for that step (cortiq-engine "Module vae",
VaeChainArgs execution order; VaeResnetRef, VaeAttnRef, VaeUpRef).

Each traced tensor is compared with relative L2 <= 1e-3 and cosine >= 0.99999
(the per-layer bar), and so is the residual branch of every resnet (the
output minus its skip term). At the full 1024^2 size the oracle evaluates
sampled outputs: the conv-type layers at sampled pixels (all corners and
edges plus seeded random pixels, every output channel), GroupNorm on whole
sampled groups, the 16384-token attention at sampled query tokens; smaller
decodes compare every element. The 1024^2 decode covers the layers that
exist only inside the chain: GroupNorm from conv-epilogue partials, the
stream-K convs of the 128^2 layers and the c = 512 attention."""
import numpy as np
import pytest

import oracle as O
import vae_synth as S
from tests._parity import COS_MIN, REL_L2_MAX, RGB_MAXABS, metrics

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SAMPLE_PIXELS = 1536  # per conv-type layer at full size
SAMPLE_TOKENS = 96    # attention query tokens at full size
SAMPLE_GROUPS = 3     # GroupNorm groups checked whole


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_vae_decoder_gb300 as pkg
    pkg.load_library()
    yield
    assert pkg.vae_device_error() == 0


def expected_steps(weights, n_up=4, n_res=3):
    """(kind, weight prefix) of every trace point, in the chain's order."""
    steps = [("latent", None), ("conv", "conv_in")]

    def resnet(pre):
        steps.extend([("groupnorm", pre + ".norm1"), ("conv", pre + ".conv1"),
                      ("groupnorm", pre + ".norm2"), ("resnet", pre)])

    resnet("mid.resnets.0")
    steps.append(("attention", "mid.attentions.0"))
    resnet("mid.resnets.1")
    for i in range(n_up):
        for j in range(n_res):
            resnet(f"up_blocks.{i}.resnets.{j}")
        if f"up_blocks.{i}.upsamplers.0.conv.weight" in weights:
            steps.append(("upsample", f"up_blocks.{i}.upsamplers.0.conv"))
    steps.append(("rgb", "conv_out"))
    return steps


def _pixels(n, h, w, count, seed):
    """Every pixel when there are few; else corners, edge midpoints and the
    four image borders' samples, plus seeded random pixels."""
    if n * h * w <= count:
        return np.array([(b, i, j) for b in range(n) for i in range(h) for j in range(w)])
    r = np.random.default_rng(seed)
    fixed = []
    for b in range(n):
        for i in (0, 1, h // 2, h - 2, h - 1):
            for j in (0, 1, w // 2, w - 2, w - 1):
                fixed.append((b, i, j))
    k = count - len(fixed)
    rnd = np.stack([r.integers(0, n, k), r.integers(0, h, k), r.integers(0, w, k)], axis=1)
    return np.concatenate([np.array(fixed), rnd])


def _nchw(t_nhwc):
    """Host NHWC activation seen as NCHW (a view, no copy)."""
    return np.moveaxis(t_nhwc, -1, 1)


def _check(got, ref, what, results):
    m = metrics(got, ref)
    results.append((what, m))
    print(f"{what:60s} rel_l2 {m['rel_l2']:.2e} cos {m['cos']:.8f} max {m['max_abs']:.2e}")
    assert np.isfinite(got).all(), what
    assert m["cos"] >= COS_MIN and m["rel_l2"] <= REL_L2_MAX, (what, m)
    return m


def _trace_decode(workload_latent, seed, arch="flux"):
    import diffusion_vae_decoder_gb300 as pkg
    w = S.make_decoder_weights(arch, seed)
    z = S.make_latent(workload_latent, seed)
    chain = pkg.VaeChain(w, n_up_blocks=4)
    n, _, h, ww = workload_latent
    pts = chain.trace_points(n, h, ww)
    bufs = [torch.empty(p["bytes"] // 4, dtype=torch.float32, device="cuda") for p in pts]
    rgb = chain.decode_traced(torch.from_numpy(z).cuda(), bufs)
    torch.cuda.synchronize()
    assert pkg.vae_device_error() == 0
    chain.close()
    return w, z, pts, bufs, rgb


def run_layer_parity(latent, seed, arch="flux"):
    w, z, pts, bufs, rgb = _trace_decode(latent, seed, arch)
    steps = expected_steps(w)
    assert [p["kind"] for p in pts] == [k for k, _ in steps]
    n = latent[0]
    host = {}

    def get(i):  # host copy of trace point i ([n, h, w, c]; RGB [n, c, h, w])
        if i not in host:
            if len(host) > 3:
                host.pop(next(iter(host)))
            p = pts[i]
            shape = (n, p["c"], p["h"], p["w"]) if p["kind"] == "rgb" else \
                (n, p["h"], p["w"], p["c"])
            host[i] = bufs[i].cpu().numpy().reshape(shape)
        return host[i]

    results = []
    for i, ((kind, pre), p) in enumerate(zip(steps, pts)):
        what = f"{i:3d} {kind} {pre or ''} [{p['c']}x{p['h']}x{p['w']}]"
        seed_i = 1000 + i
        if kind == "latent":
            got = get(i)
            ref = O.denormalize(z, S.SCALING_FACTOR, S.SHIFT_FACTOR)
            _check(_nchw(got)[:, :16], ref, what, results)
            assert (got[..., 16:] == 0).all(), what  # channel padding stays zero
            continue
        if kind in ("conv", "upsample"):
            x = _nchw(get(p["input"]))[:, :w[pre + ".weight"].shape[1]]  # drop channel padding
            pix = _pixels(n, p["h"], p["w"], SAMPLE_PIXELS, seed_i)
            fn = O.upsample_conv_at if kind == "upsample" else O.conv2d_at
            ref = fn(x, w[pre + ".weight"], w[pre + ".bias"], pix)
            got = get(i)[pix[:, 0], pix[:, 1], pix[:, 2]]
            _check(got, ref, what, results)
            continue
        if kind == "groupnorm":
            x = get(p["input"])
            c = p["c"]
            cg = c // 32
            gsel = sorted({0, 31, int(np.random.default_rng(seed_i).integers(1, 31))})
            gsel = gsel[:SAMPLE_GROUPS]
            ch = np.concatenate([np.arange(g * cg, (g + 1) * cg) for g in gsel])
            xs = np.ascontiguousarray(_nchw(x[..., ch]))
            ref = O.group_norm_silu(xs, w[pre + ".weight"][ch], w[pre + ".bias"][ch],
                                    len(gsel), 1e-6)
            got = _nchw(get(i)[..., ch])
            _check(got, ref, what, results)
            continue
        if kind == "resnet":
            t = _nchw(get(p["input"]))
            xin = _nchw(get(p["skip"]))
            pix = _pixels(n, p["h"], p["w"], SAMPLE_PIXELS, seed_i)
            branch = O.conv2d_at(t, w[pre + ".conv2.weight"], w[pre + ".conv2.bias"], pix)
            if pre + ".conv_shortcut.weight" in w:
                skip = O.conv2d_at(xin, w[pre + ".conv_shortcut.weight"],
                                   w[pre + ".conv_shortcut.bias"], pix)
            else:
                skip = xin[pix[:, 0], :, pix[:, 1], pix[:, 2]].astype(np.float64)
            got = get(i)[pix[:, 0], pix[:, 1], pix[:, 2]].astype(np.float64)
            _check(got, branch + skip, what, results)
            # The branch alone, where the output is stored unrounded: an
            # up-block's last resnet feeds the upsample conv's MMA and is
            # stored TF32-rounded, a rounding of the whole output (skip
            # included) that is not the branch's arithmetic.
            rounded = i + 1 < len(steps) and steps[i + 1][0] == "upsample"
            if pre + ".conv_shortcut.weight" not in w and not rounded:
                _check(got - skip, branch, what + " branch", results)
            continue
        if kind == "attention":
            x = np.ascontiguousarray(_nchw(get(p["input"])), dtype=np.float64)
            L = p["h"] * p["w"]
            r = np.random.default_rng(seed_i)
            tokens = np.arange(L) if L <= SAMPLE_TOKENS else np.unique(np.concatenate(
                [[0, L - 1], r.integers(0, L, SAMPLE_TOKENS)]))
            pa = {k: (w[f"{pre}.{k}.weight"], w[f"{pre}.{k}.bias"]) for k in
                  ("group_norm", "to_q", "to_k", "to_v", "to_out")}
            ref = O.mid_attention_at(x, pa, tokens)  # [n, c, S]
            got = get(i).reshape(n, L, p["c"])[:, tokens].transpose(0, 2, 1)
            xt = x.reshape(n, p["c"], L)[:, :, tokens]
            _check(got, ref, what, results)
            _check(got - xt, ref - xt, what + " branch", results)
            continue
        if kind == "rgb":
            src = get(p["input"])
            pix = _pixels(n, p["h"], p["w"], 4 * SAMPLE_PIXELS, seed_i)
            if pts[p["input"]]["kind"] == "groupnorm":
                act = _nchw(src)
            else:  # fused head: norm_out GroupNorm + SiLU of the whole input, then conv_out
                act = O.group_norm_silu(_nchw(src), w["conv_norm_out.weight"],
                                        w["conv_norm_out.bias"], 32, 1e-6)
            ref = O.conv2d_at(act, w["conv_out.weight"], w["conv_out.bias"], pix)
            got = get(i)[pix[:, 0], :, pix[:, 1], pix[:, 2]]
            m = _check(got, ref, what, results)
            assert m["max_abs"] <= RGB_MAXABS, (what, m)
            # the traced RGB is the decode's output
            assert torch.equal(bufs[i].view_as(rgb), rgb)
            continue
        raise AssertionError(kind)
    return results


def test_layer_parity_tiny_decoder():
    run_layer_parity((1, 16, 8, 8), S.seed_of("tiny_decoder"), arch="tiny")


def test_layer_parity_decoder_256():
    run_layer_parity((1, 16, 32, 32), S.seed_of("decoder_256"))


def test_layer_parity_decoder_1024():
    """Full size: the 16384-token c = 512 attention, GroupNorms finalised from
    conv-epilogue partials, the stream-K convs of the 128^2 layers."""
    run_layer_parity((1, 16, 128, 128), S.seed_of("decoder_1024"))
