"""Pins for the oracle's FP64 GEMMs (no GPU).

FProp Y = X W^T, DGrad dX = dY W, WGrad dW = dY^T X (Jet-RL papercache
summary, section 2.2).  Pinned by: an exact rational sum over K = 256 of
dequantized E4M3 products (Python fractions), a scaled-identity weight that
reduces FProp to dequantization, the transpose identities that tie the three
GEMMs to one another, sampled-vs-full agreement, and a non-square,
non-symmetric case against numpy's matmul.
"""
from fractions import Fraction

import numpy as np

import oracle
import synth


def _deq_row_pair(N, D, C, seed):
    x = synth.activation(N, C, seed=seed, stream="x")
    w = synth.weight(D, C, seed=seed, stream="w")
    qx, sx = oracle.quant_rowgroups(x)
    qw, sw, _, _ = oracle.quant_blocks(w)
    return oracle.dequant_rowgroups(qx, sx), oracle.dequant_blocks(qw, sw), (qx, sx, qw, sw)


def test_fprop_exact_rational_k256():
    N, D, C = 3, 5 * 0 + 128, 256
    X, W, (qx, sx, qw, sw) = _deq_row_pair(N, D, C, 0)
    y, bound = oracle.fprop(X, W)
    vals = oracle.e4m3_decode(np.arange(256))
    for n in range(N):
        for d in (0, 17, 127):
            exact = Fraction(0)
            for c in range(C):
                a = Fraction(float(vals[qx[n, c]])) * Fraction(float(sx[c // 128, n]))
                b = Fraction(float(vals[qw[d, c]])) * Fraction(float(sw[d // 128, c // 128]))
                exact += a * b
            assert abs(Fraction(y[n, d]) - exact) <= Fraction(2) ** -45 * Fraction(bound[n, d])
            assert bound[n, d] >= abs(y[n, d])


def test_fprop_with_scaled_identity_weight_is_dequantization():
    N, C = 4, 256
    x = synth.activation(N, C, seed=1, stream="x")
    eye = np.eye(C, dtype=np.float32) * np.float32(448.0 * 2.0 ** -3)
    qw, sw, _, _ = oracle.quant_blocks(synth.bf16_bits(eye))
    assert np.all(sw[np.eye(2, dtype=bool)] == 2.0 ** -3) and np.all(sw[~np.eye(2, dtype=bool)] == 0)
    qx, sx = oracle.quant_rowgroups(x)
    X = oracle.dequant_rowgroups(qx, sx)
    y, _ = oracle.fprop(X, oracle.dequant_blocks(qw, sw))
    assert np.array_equal(y, X * 56.0)


def test_transpose_identities_tie_the_three_gemms():
    rng = np.random.default_rng(0)
    N, D, C = 7, 5, 3
    X = rng.standard_normal((N, C))
    W = rng.standard_normal((D, C))
    dY = rng.standard_normal((N, D))
    # DGrad(dY, W) == FProp(dY, W^T): the same terms in the same order
    a, _ = oracle.dgrad(dY, W)
    b, _ = oracle.fprop(dY, np.ascontiguousarray(W.T))
    assert np.array_equal(a, b)
    # WGrad(dY, X) == FProp(dY^T, X^T)
    a, _ = oracle.wgrad(dY, X)
    b, _ = oracle.fprop(np.ascontiguousarray(dY.T), np.ascontiguousarray(X.T))
    assert np.array_equal(a, b)
    # and each equals the textbook product on non-square, non-symmetric operands
    assert np.allclose(oracle.fprop(X, W)[0], X @ W.T, rtol=1e-13, atol=1e-13)
    assert np.allclose(oracle.dgrad(dY, W)[0], dY @ W, rtol=1e-13, atol=1e-13)
    assert np.allclose(oracle.wgrad(dY, X)[0], dY.T @ X, rtol=1e-13, atol=1e-13)


def test_hand_computed_two_by_two():
    X = np.array([[1.0, 2.0], [3.0, -4.0]])
    W = np.array([[0.5, 0.25], [-1.0, 8.0]])
    dY = np.array([[2.0, -1.0], [0.0, 3.0]])
    assert np.array_equal(oracle.fprop(X, W)[0], [[1.0, 15.0], [0.5, -35.0]])
    assert np.array_equal(oracle.fprop(X, W)[1], [[1.0, 17.0], [2.5, 35.0]])
    assert np.array_equal(oracle.dgrad(dY, W)[0], [[2.0, -7.5], [-3.0, 24.0]])
    assert np.array_equal(oracle.wgrad(dY, X)[0], [[2.0, 4.0], [8.0, -14.0]])


def test_sampled_outputs_equal_full():
    X, W, _ = _deq_row_pair(9, 256, 384, 2)
    full, fb = oracle.fprop(X, W)
    at = np.array([[0, 0], [8, 255], [3, 100], [5, 7]])
    y, b = oracle.fprop(X, W, at=at)
    assert np.array_equal(y, full[at[:, 0], at[:, 1]]) and np.array_equal(b, fb[at[:, 0], at[:, 1]])
    dY = oracle.dequant_rowgroups(*oracle.quant_rowgroups(synth.gradient(9, 256, seed=2)))
    full, _ = oracle.dgrad(dY, W)
    y, _ = oracle.dgrad(dY, W, at=at[:, ::-1] * 0 + at)  # (n, c) pairs
    assert np.array_equal(y, full[at[:, 0], at[:, 1]])
    full, _ = oracle.wgrad(dY, X)
    at2 = np.array([[0, 0], [255, 383], [17, 5]])
    y, _ = oracle.wgrad(dY, X, at=at2)
    assert np.array_equal(y, full[at2[:, 0], at2[:, 1]])
