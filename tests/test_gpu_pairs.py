"""Paired-CTA conv tiles (tcgen05.mma.cta_group::2: a 256-pixel-row x
256-channel tile on two SMs, each staging its own rows and half of the
weights; "VAE decode -> GPU handoff", "GPU plan" step 2, the GEMM this
replaces).

The default picks paired tiles by an estimate of which finishes first, so
the small exact-integer shapes of test_gpu_ops.py run on 1-SM tiles and the
full-size parity tests on paired ones. Here the exact-integer and attention
tests are run again with VAE_PAIR=force (every 256-column conv, upsample
conv and attention GEMM paired, ragged GEMM rows included:
per-tap staging with the appended 1x1 shortcut and the in-place residual,
halo staging, the upsample parities, ragged rows where one CTA of a pair
holds only rows outside the image), and the full-size sweep again with
VAE_PAIR=off (1-SM tiles where the default pairs them). Child processes:
the setting is read once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child_pytest(setting, args):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, VAE_PAIR=setting)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        "-m", "gpu", *args], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


def test_exact_integer_convs_on_forced_pairs():
    _child_pytest("force", ["tests/test_gpu_ops.py", "-k",
                            "exact_integer or shortcut_and_residual or causal_float or "
                            "mid_attn_parity or growing_scores"])


def test_full_size_sweep_on_single_sm_tiles():
    _child_pytest("off", ["tests/test_gpu_configs.py", "tests/test_gpu_ops.py", "-k",
                          "sweep or stream_k"])
