"""The identity the tensor-core head is built on (csrc/head_tc.cu): a 3x3
stride-1 pad-1 conv of C channels to CO outputs equals, per input row, one
matrix product Y = A W (A: pixels x C, W: C x 9*CO, column t*CO + o = tap t
of output o) followed by adding three rows' projections shifted by the tap
offsets, zero outside the image -- checked in float64 against the oracle's
conv2d (cortiq-engine "Module vae": conv_out, 3x3, padding 1), including the
per-pixel split of the epilogue (kx = 0 / 1 / 2 partial sums taken from the
left neighbour, the pixel itself and the right neighbour)."""
import numpy as np

import oracle as O


def _head_by_projections(a, w, b):
    """a [C][H][W], w [CO][C][3][3], b [CO] -> [CO][H][W] via tap projections."""
    C, H, W = a.shape
    CO = w.shape[0]
    wt = np.zeros((C, 9 * CO))
    for o in range(CO):
        for ky in range(3):
            for kx in range(3):
                wt[:, (ky * 3 + kx) * CO + o] = w[o, :, ky, kx]
    # one GEMM per input row (pixels x C) @ (C x 9*CO), rows -1 and H are zero
    Y = np.zeros((H + 2, W + 2, 9 * CO))  # padded: row r + 1, column x + 1
    for r in range(H):
        Y[r + 1, 1:W + 1] = a[:, r, :].T @ wt
    out = np.zeros((CO, H, W))
    for r in range(H):
        # z[kx][x][o]: sum over ky of rows r-1, r, r+1 at the pixel itself
        z = np.zeros((3, W + 2, CO))
        for ky in range(3):
            for kx in range(3):
                z[kx] += Y[r + ky, :, (ky * 3 + kx) * CO:(ky * 3 + kx + 1) * CO]
        # output pixel x takes kx = 0 from x - 1, kx = 1 from x, kx = 2 from x + 1
        for x in range(W):
            out[:, r, x] = b + z[0, x] + z[1, x + 1] + z[2, x + 2]
    return out


def test_tap_projection_identity():
    rng = np.random.default_rng(11)
    for C, H, W, CO in [(32, 7, 13, 3), (64, 5, 9, 1), (32, 4, 6, 7)]:
        a = rng.standard_normal((C, H, W))
        w = rng.standard_normal((CO, C, 3, 3))
        b = rng.standard_normal(CO)
        got = _head_by_projections(a, w, b)
        want = O.conv2d(a[None], w, b)[0]
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_identity_fails_on_a_flipped_kernel():
    """The check is sharp: the same decomposition with the kernel flipped (a
    plausible indexing mistake) does not match."""
    rng = np.random.default_rng(12)
    a = rng.standard_normal((32, 6, 8))
    w = rng.standard_normal((3, 32, 3, 3))
    b = np.zeros(3)
    got = _head_by_projections(a, w[:, :, ::-1, ::-1].copy(), b)
    want = O.conv2d(a[None], w, b)[0]
    assert np.abs(got - want).max() > 1e-3
