"""Host-side model of the SiLU the CUDA kernels apply before TF32 operands
(csrc/silu.cuh): u / (1 + e^-u) with e^-u from the exp2 unit, u clamped at
-80, the reciprocal by two Newton steps from an integer-subtraction seed, and
round-to-nearest-TF32 (ties away from zero) on the bit pattern. Emulated in
float32 with numpy (exp2 correctly rounded here; the device's exp2 is within
a few ulps), it must stay within the TF32 half-ulp (2^-11, relative) of the
float64 SiLU (plus the Newton steps' 7e-6), stay finite everywhere, and
round exactly like the TF32 definition on the values it produces."""
import numpy as np

F32 = np.float32
SEED = 0x7EF30000  # the seed constant in csrc/silu.cuh


def _bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def _from_bits(b):
    return np.asarray(b, dtype=np.uint32).view(np.float32)


def tf32_rna(y):
    """Round float32 to 10 explicit mantissa bits, ties away from zero."""
    return _from_bits((_bits(y).astype(np.uint64) + 0x1000 & 0xFFFFE000).astype(np.uint32))


def silu_model(u):
    u = np.asarray(u, dtype=np.float32)
    c = np.maximum(u, F32(-80))
    t = (c * F32(-1.4426950408889634)).astype(np.float32)
    e = np.exp2(t.astype(np.float64)).astype(np.float32)
    nd = (e * F32(-1) + F32(-1)).astype(np.float32)            # -(1 + e)
    r = _from_bits(((0xFEF30000 - _bits(nd).astype(np.int64)) & 0xFFFFFFFF).astype(np.uint32))
    for _ in range(2):
        q = (nd * r + F32(1)).astype(np.float32)
        r = (r * q + r).astype(np.float32)
    return tf32_rna((u * r).astype(np.float32))


def test_seed_identity():
    """0xfef30000 - bits(-d) equals 0x7ef30000 - bits(d) for d >= 1, and the
    seed is within 5.1 % of 1/d over a binade."""
    d = np.linspace(1, 2, 100001, endpoint=False).astype(np.float32)
    a = (0xFEF30000 - _bits(-d).astype(np.int64)) & 0xFFFFFFFF
    b = (SEED - _bits(d).astype(np.int64)) & 0xFFFFFFFF
    assert (a == b).all()
    r0 = _from_bits(b.astype(np.uint32)).astype(np.float64)
    assert np.abs(r0 * d - 1).max() <= 0.0508


def test_silu_within_tf32_half_ulp():
    u = np.concatenate([np.linspace(-100, 40, 400001), np.geomspace(1e-30, 1e4, 2001),
                        -np.geomspace(1e-30, 1e4, 2001)]).astype(np.float32)
    got = silu_model(u).astype(np.float64)
    ud = u.astype(np.float64)
    with np.errstate(over="ignore"):
        ref = ud / (1 + np.exp(-ud))
    assert np.isfinite(got).all()
    big = np.abs(ref) > 1e-30
    rel = np.abs(got[big] - ref[big]) / np.abs(ref[big])
    # the TF32 half-ulp of the rounded value plus the Newton reciprocal's
    # 7e-6 (a value that lands next to a rounding boundary can go either way)
    assert rel.max() <= 2.0 ** -11 * (1 + 1e-5) + 1e-5, rel.max()
    # below the clamp SiLU is 0 to far below float resolution
    tail = ud < -80
    assert (np.abs(got[tail]) < 1e-30).all()


def test_tf32_rounding_definition():
    """The bit-pattern rounding is round-to-nearest on 11 significant bits,
    ties away from zero, for finite float32 values."""
    rng = np.random.default_rng(5)
    y = rng.standard_normal(200000).astype(np.float32) * F32(3.7)
    got = tf32_rna(y).astype(np.float64)
    m, ex = np.frexp(y.astype(np.float64))          # y = m * 2^ex, 0.5 <= |m| < 1
    q = np.sign(m) * np.floor(np.abs(m) * 2048 + 0.5) / 2048
    want = np.ldexp(q, ex)
    assert np.array_equal(got, want)
    ties = _from_bits((_bits(np.float32([1.5, -1.5])) & 0xFFFFE000) | 0x1000)
    assert np.array_equal(np.abs(tf32_rna(ties)), np.abs(_from_bits(
        (_bits(ties) & 0xFFFFE000) + 0x2000)))
