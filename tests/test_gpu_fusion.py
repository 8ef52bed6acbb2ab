"""GroupNorm and softmax work moved into the tensor-core kernels
(cortiq-engine "Module vae": VaeResnetRef GroupNorm -> SiLU -> conv;
VaeAttnRef softmax(q k^T / sqrt(c)) v), against the float64 oracle:

* the resnets' GroupNorm+SiLU made by extra warps of the conv that reads
  it, row by row ahead of its tiles (GroupNorm ahead: opt-in, VAE_GNA=on,
  measured slower than the separate pass on GB300; run in a child process);
* opt-in (VAE_FUSE=on: measured slower than the separate passes on GB300,
  run in a child process): the resnets' GroupNorm+SiLU applied by the 3x3
  conv that reads it, on the halo rows it stages, where the conv runs
  256-channel halo tiles; and the c = 512 attention's row softmax folded into
  its two GEMMs (row statistics from the score GEMM's epilogue, normalisation
  of the P.V kernel's A stages).

Each child runs this module, the 256^2 decoder parity and its layer-by-layer
trace (the settings are read once per process)."""
import os
import subprocess
import sys

import pytest

import oracle as O
import vae_synth as S
from tests._parity import COS_MIN, REL_L2_MAX, RGB_MAXABS, SENTINEL, assert_all_written, metrics

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_vae_decoder_gb300 as p
    p.load_library()
    yield p
    assert p.vae_device_error() == 0


def _fuse_on():
    return os.environ.get("VAE_FUSE", "") == "on"


def test_ragged_batch_decode(pkg):
    """Two images of a 12 x 20 latent: the 256-channel level is 48 x 80, so
    its halo tiles (128 pixels wide) hold 48 columns outside the image, where
    the transform must keep the conv's zero padding; the per-sample affine
    differs between the two images. The GroupNorm steps that fold into their
    conv move only the statistics' partials."""
    seed = 91
    w = S.make_decoder_weights("flux", seed)
    z = S.make_latent((2, 16, 12, 20), seed)
    chain = pkg.VaeChain(w, n_up_blocks=4)
    out = torch.full((2, 3, 96, 160), SENTINEL, device="cuda")
    chain.profile(True)
    chain.decode(torch.from_numpy(z).cuda(), out=out)
    torch.cuda.synchronize()
    steps = chain.profile_read()
    chain.close()
    got = out.cpu().numpy()
    ref = O.decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    assert_all_written(got, "ragged batch")
    m = metrics(got, ref)
    print(m)
    # the RGB bar (TF32 products: about 1e-3 relative L2 accumulates over
    # the 30 layers end to end; the per-layer bar is checked layer by layer
    # in test_ragged_batch_layers)
    assert m["cos"] >= COS_MIN and m["max_abs"] <= RGB_MAXABS, m
    for b in range(2):
        assert metrics(got[b], ref[b])["cos"] >= COS_MIN, b
    # GroupNorm steps reduced to the per-channel affine, their apply running
    # inside the conv. At 48 x 80 (256-channel halo convs) the five ahead of
    # a conv without a shortcut operand (the 512 -> 256 resnet's norm1, both
    # norms of the other two resnets; its norm2 feeds a conv with a 1x1
    # shortcut); at 96 x 160 all six (channel-major convs) with GroupNorm
    # ahead (VAE_FUSE=on's halo transform covers only the 48 x 80 ones).
    affine = [s for s in steps if s["kind"] == "groupnorm_affine"]
    gna_on = os.environ.get("VAE_GNA") == "on"
    expect = 11 if gna_on else (5 if _fuse_on() else 0)
    assert len(affine) == expect, [s for s in steps if s["kind"].startswith("groupnorm")]


def test_ragged_batch_layers(pkg):
    """The same decode traced layer by layer: every GroupNorm, folded conv,
    resnet and upsample against the oracle fed the GPU's own input for that
    layer (relative L2 <= 1e-3, cosine >= 0.99999)."""
    from tests.test_gpu_layers import run_layer_parity
    run_layer_parity((2, 16, 12, 20), 91)


def test_attention_softmax_folded_on_ragged_keys(pkg):
    """c = 512 attention over 20 x 26 = 520 tokens: three 256-key column
    tiles of statistics, the last with 8 valid keys, and a P.V reduction
    padded to 544 keys."""
    x = S.make_normal((1, 512, 20, 26), 92)
    wt = S.make_attn_params(512, 93)
    p = {k: (wt[k + ".weight"], wt[k + ".bias"]) for k in
         ("group_norm", "to_q", "to_k", "to_v", "to_out")}
    pd = {k: (torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()) for k, (a, b) in p.items()}
    got = pkg.vae_mid_attn(torch.from_numpy(x).cuda(), pd).cpu().numpy()
    ref = O.mid_attention(x, p)
    for a, b, what in ((got, ref, "attn"), (got - x, ref - x, "attn branch")):
        m = metrics(a, b)
        print(what, m)
        assert m["cos"] >= COS_MIN and m["rel_l2"] <= REL_L2_MAX, (what, m)


def test_groupnorm_ahead_on():
    """The same checks, the decoder_256 parity and its layer trace with the
    GroupNorm made ahead of the conv's tiles (VAE_GNA=on)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if os.environ.get("VAE_GNA") == "on" or _fuse_on():
        pytest.skip("already a child")
    env = dict(os.environ, VAE_GNA="on")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                        "tests/test_gpu_fusion.py", "tests/test_gpu_chain.py::test_decoder_256_parity",
                        "tests/test_gpu_layers.py::test_layer_parity_decoder_256"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


def test_operand_transforms_on():
    """The same checks, the decoder_256 parity and the layer-by-layer trace of
    the 256^2 decode with VAE_FUSE=on."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if _fuse_on() or os.environ.get("VAE_GNA") == "on":
        pytest.skip("already a child")
    env = dict(os.environ, VAE_FUSE="on")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                        "tests/test_gpu_fusion.py", "tests/test_gpu_chain.py::test_decoder_256_parity",
                        "tests/test_gpu_layers.py::test_layer_parity_decoder_256"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
