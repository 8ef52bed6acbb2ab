"""The 3-D causal decoder (vae_causal_decoder_prepare / vae_decode_causal):
an LTX-style structural video decoder ("VAE decode -> GPU handoff", "The
CPU VAE code": LtxVaeDecoder::decode, 3-D causal convs with causal time
padding) with random-init weights, against the float64 oracle's
causal_decode; the decoder's RGB bar (cosine >= 0.99999, max |err| <=
5e-3), on every frame."""
import ctypes

import numpy as np
import pytest

import oracle as O
import vae_synth as S
from tests._parity import COS_MIN, RGB_MAXABS, SENTINEL, assert_all_written, metrics

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_vae_decoder_gb300 as p
    p.load_library()
    yield p
    assert p.vae_device_error() == 0


def _run(pkg, arch, latent, seed, **kw):
    w = S.make_causal_decoder_weights(arch, seed)
    z = S.make_latent(latent, seed)
    dec = pkg.VaeCausalDecoder(w, n_up_blocks=4, **kw)
    n, _, t, h, ww = latent
    f = dec.up_factor
    out = torch.full((n, 3, t, f * h, f * ww), SENTINEL, device="cuda")
    dec.decode(torch.from_numpy(z).cuda(), out=out)
    torch.cuda.synchronize()
    dec.close()
    got = out.cpu().numpy()
    ref = O.causal_decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    assert_all_written(got, arch)
    return got, ref


def _bar(got, ref, what):
    m = metrics(got, ref)
    print(what, m)
    assert m["cos"] >= COS_MIN and m["max_abs"] <= RGB_MAXABS, (what, m)
    for f in range(got.shape[2]):
        mf = metrics(got[:, :, f], ref[:, :, f])
        assert mf["cos"] >= COS_MIN, (what, f, mf)


def test_causal_tiny_batch_ragged(pkg):
    got, ref = _run(pkg, "causal_tiny", (2, 16, 3, 5, 7), 91)
    _bar(got, ref, "causal tiny [2,16,3,5,7]")


def test_causal_tiny_tf32_products(pkg):
    got, ref = _run(pkg, "causal_tiny", (1, 16, 4, 6, 6), 92, precision=pkg.PRECISION_TF32)
    _bar(got, ref, "causal tiny TF32 [1,16,4,6,6]")


def test_causal_small_decoder(pkg):
    """Channels 256/256/128/64, latent [1,16,5,16,16] -> 5 frames of 128^2:
    TF32 products, paired and 1-SM conv tiles, GroupNorm from conv partials
    over (t, h, w)."""
    got, ref = _run(pkg, "causal_small", (1, 16, 5, 16, 16), 93)
    _bar(got, ref, "causal small [1,16,5,16,16]")


def test_handles_of_the_other_kind_are_refused(pkg):
    lib = pkg.load_library()
    chain = pkg.VaeChain(S.make_decoder_weights("tiny", 5), n_up_blocks=4)
    dec = pkg.VaeCausalDecoder(S.make_causal_decoder_weights("causal_tiny", 5), n_up_blocks=4)
    z = torch.zeros((1, 16, 1, 8, 8), device="cuda")
    out = torch.empty((1, 3, 1, 64, 64), device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert lib.vae_decode_causal(chain.handle, p(z), 1, 1, 8, 8, p(out), p(ws), ws.numel(),
                                 None) == -1
    assert lib.vae_decode_chain(dec.handle, p(z), 1, 8, 8, p(out), p(ws), ws.numel(), None) == -1
    assert lib.vae_chain_workspace_size(dec.handle, 1, 8, 8) == 0
    assert lib.vae_causal_decoder_workspace_size(chain.handle, 1, 1, 8, 8) == 0
    chain.close()
    dec.close()
