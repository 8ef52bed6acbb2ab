"""Split-TF32 products on the single-op entry points: the exact-integer tests
of test_gpu_ops.py (conv with per-tap staging, appended 1x1 shortcut and
in-place residual, upsample parities, causal 3-D conv, ragged tiles, both
layouts) and the floating-point conv / attention parity tests run again with
VAE_SPLIT=force, so every implicit-GEMM launch (conv, upsample conv, the
attention GEMMs) forms a_hi b_hi + a_lo b_hi + a_hi b_lo on its FP32
operands. Integer operands split into hi = v, lo = 0, so the exact tests must
still match bit for bit. Child process: the setting is read once per
process. (The chain's split-TF32 decodes are covered by test_gpu_chain.py and
the per-layer test of the tiny decoder.)"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_single_ops_on_forced_split_products():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, VAE_SPLIT="force")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m",
                        "gpu", "tests/test_gpu_ops.py", "-k",
                        "exact_integer or shortcut_and_residual or float_parity or "
                        "mid_attn_parity"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
