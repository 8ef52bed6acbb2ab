"""Parity metrics shared by the GPU tests (the tolerances are the ones the
decoder's acceptance bar states: cosine >= 0.99999, per-layer relative L2
<= 1e-3, max |err| <= 5e-3 on RGB outputs)."""
import numpy as np

COS_MIN = 0.99999
REL_L2_MAX = 1e-3
RGB_MAXABS = 5e-3
SENTINEL = -12345.0


def metrics(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    diff = got - ref
    nr = np.sqrt((ref * ref).sum())
    ng = np.sqrt((got * got).sum())
    cos = float((got * ref).sum() / (nr * ng)) if nr > 0 and ng > 0 else float(nr == ng)
    rel = float(np.sqrt((diff * diff).sum()) / nr) if nr > 0 else float(np.abs(diff).max())
    return dict(cos=cos, rel_l2=rel, max_abs=float(np.abs(diff).max()),
                rel_rms=rel, pct_gt_1_255=float((np.abs(diff) > 1 / 255).mean() * 100))


def assert_layer_parity(got, ref, what=""):
    m = metrics(got, ref)
    assert np.isfinite(np.asarray(got)).all(), f"{what}: non-finite output"
    assert m["cos"] >= COS_MIN and m["rel_l2"] <= REL_L2_MAX, f"{what}: {m}"
    return m


def assert_all_written(arr, what=""):
    a = np.asarray(arr)
    n = int((a == SENTINEL).sum())
    assert n == 0, f"{what}: {n} of {a.size} output elements never written"
