"""The allocation-free GroupNorm(+SiLU) entry point, for callers that must not
allocate device memory (for example a plug-in whose host application owns the
whole device-memory budget): its statistics scratch is a fixed array inside
the library instead of a caller workspace.

Checked through the C ABI against the workspace entry point,
vae_groupnorm_silu, with the tolerance the GroupNorm parity tests use, on two
calls in a row with different shapes and layouts (the shared scratch keeps
the previous call's contents), against the float64 oracle's GroupNorm(+SiLU)
on both, plus the size limit. This file is collected last on purpose so
that a run stopping at the first failure has run every other test before
it."""
import ctypes

import numpy as np
import pytest

import oracle as O
import vae_synth as S
from tests._parity import metrics

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_vae_decoder_gb300 as pkg
    return pkg.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _both(lib, x, g, b, layout, silu):
    n = x.shape[0]
    c = x.shape[1] if layout == 0 else x.shape[-1]
    spatial = x.numel() // (n * c)
    ref = torch.empty_like(x)
    ws_bytes = lib.vae_groupnorm_silu_workspace_size(n, c, spatial, layout, 32)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    assert lib.vae_groupnorm_silu(_p(x), n, c, spatial, layout, 32, 1e-6, _p(g), _p(b), silu,
                                  _p(ref), _p(ws), ws_bytes, _stream()) == 0
    got = torch.full_like(x, -12345.0)
    assert lib.vae_groupnorm_silu_noalloc(_p(x), n, c, spatial, layout, 32, 1e-6, _p(g), _p(b),
                                          silu, _p(got), _stream()) == 0
    torch.cuda.synchronize()
    return got.cpu().numpy(), ref.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_twice(lib):
    cases = [((2, 128, 24, 40), 0, 1, 41), ((1, 20, 36, 512), 1, 0, 42)]
    for shape, layout, silu, seed in cases:
        c = shape[1] if layout == 0 else shape[-1]
        x = torch.from_numpy(S.make_normal(shape, seed) * 2.0 + 0.5).cuda()
        g, b = (torch.from_numpy(a).cuda() for a in S.make_norm_params(c, seed))
        got, ref = _both(lib, x, g, b, layout, silu)
        assert not (got == -12345.0).any()
        m = metrics(got, ref)
        assert m["rel_l2"] < 2e-6 and m["max_abs"] < 2e-5, (shape, m)
        # and against the oracle itself (NCHW view of the input)
        xh = x.cpu().numpy()
        xn = xh if layout == 0 else np.moveaxis(xh, -1, 1)
        gh, bh = g.cpu().numpy(), b.cpu().numpy()
        want = O.group_norm_silu(xn, gh, bh, 32, 1e-6) if silu else \
            O.group_norm(xn, gh, bh, 32, 1e-6)
        if layout == 1:
            want = np.moveaxis(want, 1, -1)
        mo = metrics(got, want)
        assert mo["rel_l2"] < 2e-6 and mo["cos"] >= 0.99999, (shape, mo)


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    x = torch.zeros((11, 64, 4, 4), device="cuda")
    g = torch.ones(64, device="cuda")
    b = torch.zeros(64, device="cuda")
    y = torch.empty_like(x)
    # 11 samples x 32 groups needs more than the fixed 4 MiB of scratch
    assert lib.vae_groupnorm_silu_noalloc(_p(x), 11, 64, 16, 0, 32, 1e-6, _p(g), _p(b), 1,
                                          _p(y), _stream()) == -2
    assert lib.vae_groupnorm_silu_noalloc(_p(x), 10, 64, 16, 0, 32, 1e-6, _p(g), _p(b), 1,
                                          _p(y), _stream()) == 0
    torch.cuda.synchronize()
    import diffusion_vae_decoder_gb300 as pkg
    assert pkg.vae_device_error() == 0
