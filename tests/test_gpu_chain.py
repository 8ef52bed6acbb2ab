"""GPU parity of the whole decoder chain (vae_decode_chain) against the
float64 CPU oracle, on the seeded synthetic latents and random-init weights
of the decoder workloads: RGB cosine >= 0.99999 and max |err| <= 5e-3."""
import numpy as np
import pytest

import oracle as O
import vae_synth as S
from tests._parity import COS_MIN, REL_L2_MAX, RGB_MAXABS, SENTINEL, assert_all_written, metrics

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_vae_decoder_gb300 as pkg
    pkg.load_library()
    yield
    assert pkg.vae_device_error() == 0


def _decode(arch, latent_shape, seed, n_up=4, precision=None):
    import diffusion_vae_decoder_gb300 as pkg
    w = S.make_decoder_weights(arch, seed)
    z = S.make_latent(latent_shape, seed)
    kw = {} if precision is None else {"precision": precision}
    chain = pkg.VaeChain(w, n_up_blocks=n_up, **kw)
    n, _, h, ww = latent_shape
    out = torch.full((n, 3, 8 * h, 8 * ww), SENTINEL, dtype=torch.float32, device="cuda")
    chain.decode(torch.from_numpy(z).cuda(), out=out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    chain.close()
    return w, z, got


def _check(got, ref, what, rel_l2=True):
    """The RGB bar (cosine, max |err|), and relative L2 <= 1e-3 end to end
    too unless rel_l2 is False."""
    assert_all_written(got, what)
    m = metrics(got, ref)
    print(what, m)
    assert m["cos"] >= COS_MIN and m["max_abs"] <= RGB_MAXABS, (what, m)
    assert not rel_l2 or m["rel_l2"] <= REL_L2_MAX, (what, m)
    return m


def test_tiny_decoder_parity():
    """The configured tiny decoder. Its whole decode is about 2.4 GFLOP of
    convs, so the default precision forms every tensor-core product in
    split-TF32; the bar is met with a wide margin (at least 20 %)."""
    seed = S.seed_of("tiny_decoder")
    w, z, got = _decode("tiny", (1, 16, 8, 8), seed)
    ref = O.decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    m = _check(got, ref, "tiny [1,16,8,8]")
    assert m["max_abs"] <= 0.8 * RGB_MAXABS, m


def test_tiny_decoder_tf32_products():
    """The same decode with plain TF32 products (VAE_PRECISION_TF32): inside
    the RGB bar, with end-to-end relative L2 near 1.1e-3 (TF32 rounding of
    both operands of every product accumulates over the 30 layers; the
    per-layer bar is met layer by layer)."""
    import diffusion_vae_decoder_gb300 as pkg
    seed = S.seed_of("tiny_decoder")
    w, z, got = _decode("tiny", (1, 16, 8, 8), seed, precision=pkg.PRECISION_TF32)
    ref = O.decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    _check(got, ref, "tiny [1,16,8,8], TF32", rel_l2=False)


def test_tiny_decoder_batch_and_ragged_latent():
    """Batch of 2 on a latent whose sides are not powers of two."""
    seed = 77
    w, z, got = _decode("tiny", (2, 16, 5, 7), seed)
    ref = O.decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    m = _check(got, ref, "tiny [2,16,5,7]")
    assert m["max_abs"] <= 0.8 * RGB_MAXABS, m
    for b in range(2):  # every image of the batch decodes like it would alone
        mb = metrics(got[b], ref[b])
        assert mb["cos"] >= COS_MIN, (b, mb)


def test_decoder_256_split_tf32_products():
    """The 256^2 decoder with every product in split-TF32
    (VAE_PRECISION_SPLIT_TF32): close to FP32 accuracy, far inside the bar."""
    import diffusion_vae_decoder_gb300 as pkg
    seed = S.seed_of("decoder_256")
    w, z, got = _decode("flux", (1, 16, 32, 32), seed, precision=pkg.PRECISION_SPLIT_TF32)
    ref = O.decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    m = _check(got, ref, "flux [1,16,32,32], split-TF32")
    assert m["rel_l2"] <= 5e-5 and m["max_abs"] <= 5e-4, m


@pytest.mark.parametrize("cout", [1, 2, 4, 5])
def test_tiny_decoder_other_output_widths(cout):
    """conv_out widths other than RGB: the fused norm_out + conv_out head has
    one kernel instantiation per width up to 4; wider outputs take the
    implicit-GEMM conv after a separate GroupNorm+SiLU."""
    import diffusion_vae_decoder_gb300 as pkg
    seed = S.seed_of("tiny_decoder")
    w = dict(S.make_decoder_weights("tiny", seed))
    cin = w["conv_out.weight"].shape[1]
    w["conv_out.weight"], w["conv_out.bias"] = S.make_conv_params(cout, cin, 3, seed + 7)
    z = S.make_latent((1, 16, 8, 8), seed)
    chain = pkg.VaeChain(w, n_up_blocks=4)
    out = torch.full((1, cout, 64, 64), SENTINEL, dtype=torch.float32, device="cuda")
    chain.decode(torch.from_numpy(z).cuda(), out=out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    chain.close()
    ref = O.decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    _check(got, ref, f"tiny, {cout} output channels")


def test_decoder_256_parity():
    seed = S.seed_of("decoder_256")
    w, z, got = _decode("flux", (1, 16, 32, 32), seed)
    ref = O.decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    _check(got, ref, "flux [1,16,32,32] -> 256^2")


def test_chain_rejects_small_workspace():
    import diffusion_vae_decoder_gb300 as pkg
    w = S.make_decoder_weights("tiny", 5)
    chain = pkg.VaeChain(w, n_up_blocks=4)
    z = torch.zeros((1, 16, 8, 8), device="cuda")
    need = chain.workspace_size(1, 8, 8)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.VaeError) as e:
        chain.decode(z, ws=ws)
    assert e.value.status == -3
    chain.close()


@pytest.mark.parametrize("workload", ["decoder_256", "decoder_1024"])
def test_decode_is_bitwise_repeatable_on_a_dirty_workspace(workload):
    """Every reduction of the decode has a fixed order (split-K slices,
    stream-K hand-offs between neighbouring CTAs, GroupNorm partial merges
    whichever block of a group finishes last), and no step depends on what
    the workspace held before: decodes on a workspace filled with 0xFF bytes,
    eager or replayed from a CUDA graph, give the same bits every time. The
    1024^2 decode covers the stream-K layers, the 256^2 one split-K."""
    import diffusion_vae_decoder_gb300 as pkg
    spec = S.WORKLOADS[workload]
    seed = S.seed_of(workload)
    n, _, h, w = spec["latent"]
    chain = pkg.VaeChain(S.make_decoder_weights("flux", seed), n_up_blocks=4)
    z = torch.from_numpy(S.make_latent(spec["latent"], seed)).cuda()
    ws = torch.full((chain.workspace_size(n, h, w),), 255, dtype=torch.uint8, device="cuda")

    def fresh():
        return torch.full((n, 3, 8 * h, 8 * w), SENTINEL, dtype=torch.float32, device="cuda")

    outs = []
    for _ in range(2):
        outs.append(chain.decode(z, out=fresh(), ws=ws))
    g_out = fresh()
    graph = chain.capture_graph(z, g_out, ws)
    ws.fill_(255)
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        outs.append(g_out.clone())
    assert pkg.vae_device_error() == 0
    got = [o.cpu().numpy() for o in outs]
    chain.close()
    assert_all_written(got[0], workload)
    assert np.isfinite(got[0]).all()
    for i, g in enumerate(got[1:], 1):
        np.testing.assert_array_equal(g, got[0], err_msg=f"{workload}: decode {i} differs")
