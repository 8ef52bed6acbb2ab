"""Failure paths on the GPU, exercised without a fault, a trap or a hang
(bounded device waits with an error word; "VAE decode -> GPU handoff", section
"Correctness gate": a status comes back instead of a silent fallback):

  * a bounded device-side wait that runs out: the conv's stream-K hand-off
    flag is withheld through a test hook and the wait limit shortened to
    2 ms; the kernel records VAE_EDEVICE_TIMEOUT, drains its copies and MMAs,
    frees TMEM and returns, and the same process then runs the conv again
    with full parity;
  * vae_chain_prepare failing to allocate: VAE_ENOMEM, nothing leaked;
  * a destroyed chain handle: VAE_ENOTPREPARED from every entry point."""
import numpy as np
import pytest

import oracle as O
import vae_synth as S
from tests._parity import assert_layer_parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_vae_decoder_gb300 as p
    p.load_library()
    yield p
    p.vae_debug_inject(0)
    p.vae_debug_set_wait_limit(0)
    p.vae_debug_fail_allocation(0)
    assert p.vae_device_error() == 0


def _conv_case():
    """256 -> 64 channels at 192 x 128, NHWC: 192 one-SM output tiles of 64
    channels (1.26 rounds of the SMs) and 72 reduction steps each, which the
    conv runs with stream-K ranges (a tile cut between two CTAs)."""
    x = S.make_normal((1, 192, 128, 256), 61)
    w, b = S.make_conv_params(64, 256, 3, 62)
    return x, w, b


def test_expired_device_wait_reports_timeout_and_recovers(pkg):
    x, w, b = _conv_case()
    xd, wd, bd = (torch.from_numpy(a).cuda() for a in (x, w, b))
    y = torch.empty((1, 192, 128, 64), device="cuda")
    assert pkg.vae_device_error() == 0
    pkg.vae_debug_set_wait_limit(2_000_000)  # 2 ms
    pkg.vae_debug_inject(pkg.INJECT_WITHHOLD_STREAMK_FLAG)
    try:
        pkg.vae_conv2d(xd, wd, bd, layout=pkg.VAE_NHWC, out=y)
        torch.cuda.synchronize()
    finally:
        pkg.vae_debug_inject(0)
        pkg.vae_debug_set_wait_limit(0)
    assert pkg.vae_device_error() == -6  # VAE_EDEVICE_TIMEOUT, read and cleared
    # the context is intact: the same conv runs again, exactly as it should
    y.fill_(-12345.0)
    pkg.vae_conv2d(xd, wd, bd, layout=pkg.VAE_NHWC, out=y)
    torch.cuda.synchronize()
    assert pkg.vae_device_error() == 0
    got = np.moveaxis(y.cpu().numpy(), -1, 1)
    r = np.random.default_rng(3)
    pix = np.array([[0, i, j] for i in (0, 1, 95, 191) for j in (0, 5, 64, 127)] +
                   [[0, int(i), int(j)] for i, j in
                    zip(r.integers(0, 192, 400), r.integers(0, 128, 400))])
    ref = O.conv2d_at(np.moveaxis(x, -1, 1), w, b, pix)
    assert_layer_parity(got[0][:, pix[:, 1], pix[:, 2]].T, ref, "conv after a timeout")


def test_prepare_allocation_failure_returns_enomem_and_frees(pkg):
    w = S.make_decoder_weights("tiny", 5)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for nth in (1, 7, 40):
        pkg.vae_debug_fail_allocation(nth)
        with pytest.raises(pkg.VaeError) as e:
            pkg.VaeChain(w, n_up_blocks=4)
        assert e.value.status == -7
    pkg.vae_debug_fail_allocation(0)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0 - (8 << 20)  # nothing left allocated
    chain = pkg.VaeChain(w, n_up_blocks=4)  # and the next prepare works
    out = chain.decode(torch.zeros((1, 16, 8, 8), device="cuda"))
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    chain.close()


def test_destroyed_handle_is_rejected(pkg):
    import ctypes
    lib = pkg.load_library()
    chain = pkg.VaeChain(S.make_decoder_weights("tiny", 6), n_up_blocks=4)
    h = chain.handle
    z = torch.zeros((1, 16, 8, 8), device="cuda")
    rgb = torch.empty((1, 3, 64, 64), device="cuda")
    ws = torch.empty(chain.workspace_size(1, 8, 8), dtype=torch.uint8, device="cuda")
    chain.close()
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert lib.vae_decode_chain(h, p(z), 1, 8, 8, p(rgb), p(ws), ws.numel(), None) == -5
    assert lib.vae_chain_workspace_size(h, 1, 8, 8) == 0
    assert lib.vae_chain_destroy(h) == -5
    cnt = ctypes.c_int(0)
    assert lib.vae_chain_trace_points(h, 1, 8, 8, None, 0, ctypes.byref(cnt)) == -5
    assert pkg.vae_device_error() == 0
