"""The decoder's last two steps, norm_out GroupNorm+SiLU and conv_out
(cortiq-engine "Module vae", VaeDecoder), on the tensor-core head that TF32
decodes use: the traced RGB against the float64 oracle fed the GPU's own
input of the head, every pixel, for conv_out widths 1-7, batches and image
sides that leave a ragged last column strip (strips of equal width, at most
126 output columns per CTA) and ragged row segments. Per-layer bar: relative L2 <= 1e-3, cosine >= 0.99999,
and the RGB max |err| bar."""
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


def _head_parity(latent, cout, seed):
    """Decode with TF32 products (tensor-core head) and compare the head's
    output with the oracle's norm_out + conv_out of the traced head input."""
    import diffusion_vae_decoder_gb300 as pkg
    w = dict(S.make_decoder_weights("tiny", seed))
    cin = w["conv_out.weight"].shape[1]
    w["conv_out.weight"], w["conv_out.bias"] = S.make_conv_params(cout, cin, 3, seed + 7)
    z = S.make_latent(latent, seed)
    chain = pkg.VaeChain(w, n_up_blocks=4, precision=pkg.PRECISION_TF32)
    n, _, h, ww = latent
    pts = chain.trace_points(n, h, ww)
    assert pts[-1]["kind"] == "rgb"
    # the fused head: its trace input is the un-normalised last activation
    src_pt = pts[pts[-1]["input"]]
    assert src_pt["kind"] != "groupnorm"
    bufs = [torch.full((p["bytes"] // 4,), SENTINEL, dtype=torch.float32, device="cuda")
            for p in pts]
    rgb = chain.decode_traced(torch.from_numpy(z).cuda(), bufs)
    torch.cuda.synchronize()
    assert pkg.vae_device_error() == 0
    chain.close()
    H, W = src_pt["h"], src_pt["w"]
    src = bufs[pts[-1]["input"]].cpu().numpy().reshape(n, H, W, src_pt["c"])
    act = O.group_norm_silu(np.moveaxis(src, -1, 1), w["conv_norm_out.weight"],
                            w["conv_norm_out.bias"], 32, 1e-6)
    pix = np.array([(b, i, j) for b in range(n) for i in range(H) for j in range(W)])
    ref = O.conv2d_at(act, w["conv_out.weight"], w["conv_out.bias"], pix)
    got_all = rgb.cpu().numpy()
    assert got_all.shape == (n, cout, H, W)
    assert_all_written(got_all, f"head cout={cout}")
    got = got_all[pix[:, 0], :, pix[:, 1], pix[:, 2]]
    m = metrics(got, ref)
    print(f"head {latent} cout={cout}: {m}")
    assert m["cos"] >= COS_MIN and m["rel_l2"] <= REL_L2_MAX, m
    assert m["max_abs"] <= RGB_MAXABS, m
    return m


@pytest.mark.parametrize("cout", [1, 2, 3, 4, 5, 7])
def test_tensor_core_head_widths(cout):
    """Every conv_out width the tensor-core head takes (N = 16, 32, 48, 64
    columns of tap projections), batch 2, a 40 x 280 output: three column
    strips of 94 columns, the last 92 wide."""
    _head_parity((2, 16, 5, 35), cout, 300 + cout)


def test_tensor_core_head_ragged_rows():
    """A 320 x 168 output: three rows per CTA, the last segment two rows."""
    _head_parity((1, 16, 40, 21), 3, 311)


def test_tensor_core_head_matches_cuda_core_head():
    """The tensor-core head and the FP32 CUDA-core head (VAE_HEAD=cuda, in a
    child process) decode the same latent to RGB within the RGB bar of each
    other."""
    import os
    import subprocess
    import sys
    import tempfile
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import sys, numpy as np, torch\n"
        f"sys.path.insert(0, {root!r})\n"
        "import vae_synth as S, diffusion_vae_decoder_gb300 as pkg\n"
        "w = S.make_decoder_weights('tiny', 321)\n"
        "z = torch.from_numpy(S.make_latent((1, 16, 12, 20), 321)).cuda()\n"
        "c = pkg.VaeChain(w, n_up_blocks=4, precision=pkg.PRECISION_TF32)\n"
        "out = c.decode(z); torch.cuda.synchronize()\n"
        "assert pkg.vae_device_error() == 0\n"
        "np.save(sys.argv[1], out.cpu().numpy())\n")
    outs = []
    with tempfile.TemporaryDirectory() as tmp:
        for env_head in (None, "cuda"):
            env = dict(os.environ)
            env.pop("VAE_HEAD", None)
            if env_head:
                env["VAE_HEAD"] = env_head
            path = os.path.join(tmp, f"head_{env_head or 'tc'}.npy")
            subprocess.run([sys.executable, "-c", code, path], env=env, check=True, timeout=600)
            outs.append(np.load(path))
    m = metrics(outs[0], outs[1].astype(np.float64))
    print("tensor-core head vs CUDA-core head", m)
    assert m["cos"] >= COS_MIN and m["max_abs"] <= RGB_MAXABS, m
    assert not np.array_equal(outs[0], outs[1])  # two different kernels ran
