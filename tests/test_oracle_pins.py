"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code (CPU only).

Sources: Tuteja et al., "Theoretical and Empirical Analysis of Sparse
Convolution" (Sec. 3 Eq.(1)-(3), Sec. 4 Eq.(4)-(8), Table 1); Escoin, arXiv
1802.10280 ("Sparse convolution": lowering O = W * I with W of M x CRS and I of
CRS x EF; CSR; Algorithms 1 and 2).
"""
import itertools
import os

import numpy as np
import pytest

import oracle
import workloads
from sparse_weight_direct_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers written in the tests, independently of oracle/spconv_oracle.c
# --------------------------------------------------------------------------

def im2col_bruteforce(x, R, S, stride, pad):
    """Escoin's lowering: gather the input of one image into I (CRS x EF) by
    explicit zero-padded copies (duplicating inputs, as the page describes)."""
    C, H, W = x.shape
    Hp, Wp = H + 2 * pad, W + 2 * pad
    xp = np.zeros((C, Hp, Wp))
    xp[:, pad:pad + H, pad:pad + W] = x
    E = (Hp - R) // stride + 1
    F = (Wp - S) // stride + 1
    I = np.zeros((C * R * S, E * F))
    for c in range(C):
        for r in range(R):
            for s in range(S):
                row = (c * R + r) * S + s
                for e in range(E):
                    for f in range(F):
                        I[row, e * F + f] = xp[c, e * stride + r, f * stride + s]
    return I, E, F


def int_tensor(rng, shape, lo, hi):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64)


def dense_from_csr(rowptr, colidx, value, M, C, R, S):
    return oracle.csr_to_dense(rowptr, colidx, value, M, C, R, S)


# --------------------------------------------------------------------------
# Eq.(2): output extent
# --------------------------------------------------------------------------

def test_output_extent_closed_form():
    # Worked values: 3x3/s1/p1 keeps the size; 11x11/s4/p0 on 227 gives 55;
    # 5x5/s1/p2 on 27 keeps 27; kernel larger than the padded input gives 0.
    assert oracle.out_dim(16, 3, 1, 1) == 16
    assert oracle.out_dim(14, 3, 1, 1) == 14
    assert oracle.out_dim(56, 3, 1, 1) == 56
    assert oracle.out_dim(28, 3, 1, 1) == 28
    assert oracle.out_dim(227, 11, 4, 0) == 55
    assert oracle.out_dim(27, 5, 1, 2) == 27
    assert oracle.out_dim(2, 5, 1, 1) == 0
    assert oracle.out_dim(7, 3, 2, 0) == 3
    assert oracle.out_dim(8, 3, 2, 0) == 3
    assert oracle.out_dim(9, 3, 2, 0) == 4
    for layer in workloads.LAYERS.values():
        assert oracle.out_dim(layer.H, layer.R, layer.stride, layer.pad) == layer.E
        # the page's garbled print reads ceil((H + 2P - K + 1) / s); for
        # integers it equals the floor form
        num = layer.H + 2 * layer.pad - layer.R + 1
        assert -(-num // layer.stride) == layer.E


# --------------------------------------------------------------------------
# Lowering identity O = W (M x CRS) . I (CRS x EF), exact on integers
# --------------------------------------------------------------------------

CASES = [(R, S, st, p) for R, S in [(1, 1), (2, 2), (3, 3), (5, 5), (3, 2), (1, 3)]
         for st in (1, 2, 4) for p in (0, 1, 2)]


@pytest.mark.parametrize("R,S,stride,pad", CASES)
def test_lowering_identity(R, S, stride, pad):
    rng = np.random.default_rng(R * 1000 + S * 100 + stride * 10 + pad)
    N, C, M = 2, 3, 4
    H, W = 7, 6  # non-square so a transposed index shows
    if H + 2 * pad < R or W + 2 * pad < S:
        pytest.skip("kernel larger than padded input")
    x = int_tensor(rng, (N, C, H, W), 0, 7)
    w = int_tensor(rng, (M, C, R, S), -3, 3)
    y, _ = oracle.dense7(x, w, stride, pad)
    Wmat = w.reshape(M, C * R * S)
    for n in range(N):
        I, E, F = im2col_bruteforce(x[n], R, S, stride, pad)
        O = Wmat @ I
        assert y.shape[2:] == (E, F)
        np.testing.assert_array_equal(y[n].reshape(M, E * F), O)


# --------------------------------------------------------------------------
# Special case reducing to a library routine: torch CPU conv2d in float64
# --------------------------------------------------------------------------

@pytest.mark.parametrize("R,S,stride,pad", [(3, 3, 1, 1), (5, 5, 1, 2), (3, 3, 2, 0),
                                            (11, 11, 4, 0), (1, 1, 1, 0), (3, 5, 2, 1)])
def test_dense7_matches_torch_conv2d(R, S, stride, pad):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    H = W = 23 if R < 11 else 31
    x = rng.standard_normal((2, 3, H, W))
    w = rng.standard_normal((5, 3, R, S))
    y, _ = oracle.dense7(x, w, stride, pad)
    ref = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(w),
                                     stride=stride, padding=pad).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_tiny_layer_matches_torch_conv2d():
    torch = pytest.importorskip("torch")
    L = workloads.LAYERS["tiny"]
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L)
    w = dense_from_csr(rowptr, colidx, value, L.M, L.C, L.R, L.S)
    y, _ = oracle.dense7(x, w, L.stride, L.pad)
    ref = torch.nn.functional.conv2d(torch.from_numpy(x.astype(np.float64)),
                                     torch.from_numpy(w), stride=L.stride,
                                     padding=L.pad).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)
    yc, _ = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
    np.testing.assert_allclose(yc, ref, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------
# Sparse == dense (Eq.(3) is Eq.(1) restricted to nonzeros)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("density", [1.0, 0.5, 0.1, 0.02, 0.0])
@pytest.mark.parametrize("R,stride,pad", [(3, 1, 1), (5, 1, 2), (3, 2, 0), (11, 4, 0)])
def test_csr_equals_dense_integer(density, R, stride, pad):
    rng = np.random.default_rng(int(density * 100) + R)
    N, C, M = 2, 4, 6
    H = W = 13 if R < 11 else 27
    rowptr, colidx, value = workloads.random_csr(M, C * R * R, density, rng, integer=True)
    x = workloads.random_input((N, C, H, W), rng, integer=True)
    w = dense_from_csr(rowptr, colidx, value, M, C, R, R)
    yd, ad = oracle.dense7(x, w, stride, pad)
    yc, ac = oracle.csr(x, rowptr, colidx, value, M, R, R, stride, pad, threads=3)
    np.testing.assert_array_equal(yc, yd)
    np.testing.assert_array_equal(ac, ad)
    if density == 0.0:
        assert not yc.any()


def test_csr_equals_dense_float_all_configs_small():
    rng = np.random.default_rng(11)
    for density in (1.0, 0.3, 0.1):
        rowptr, colidx, value = workloads.random_csr(8, 5 * 9, density, rng)
        x = workloads.random_input((1, 5, 9, 10), rng)
        w = dense_from_csr(rowptr, colidx, value, 8, 5, 3, 3)
        yd, ad = oracle.dense7(x, w, 1, 1)
        yc, ac = oracle.csr(x, rowptr, colidx, value, 8, 3, 3, 1, 1)
        assert np.all(np.abs(yc - yd) <= 1e-12 * ad + 1e-300)
        np.testing.assert_allclose(ac, ad, rtol=1e-12)


def test_csr_points_match_full():
    L = workloads.LAYERS["tiny"]
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L)
    y, a = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad)
    rng = np.random.default_rng(3)
    idx = rng.integers(0, y.size, size=500)
    yp, ap = oracle.csr_points(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad, idx)
    np.testing.assert_array_equal(yp, y.reshape(-1)[idx])
    np.testing.assert_array_equal(ap, a.reshape(-1)[idx])


# --------------------------------------------------------------------------
# Linearity in the weights and in the input (exact on integers)
# --------------------------------------------------------------------------

def test_linearity():
    rng = np.random.default_rng(5)
    N, C, M, H, W, R = 2, 3, 4, 9, 8, 3
    x1 = int_tensor(rng, (N, C, H, W), 0, 7)
    x2 = int_tensor(rng, (N, C, H, W), 0, 7)
    w1 = int_tensor(rng, (M, C, R, R), -3, 3)
    w2 = int_tensor(rng, (M, C, R, R), -3, 3)
    a, b = 3.0, -2.0
    f = lambda x, w: oracle.dense7(x, w, 1, 1)[0]
    np.testing.assert_array_equal(f(x1, a * w1 + b * w2), a * f(x1, w1) + b * f(x1, w2))
    np.testing.assert_array_equal(f(a * x1 + b * x2, w1), a * f(x1, w1) + b * f(x2, w1))


# --------------------------------------------------------------------------
# Identity / shifted-delta filters (orientation and padding pins)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("K", [1, 3, 5])
def test_identity_delta_passes_input_through(K):
    rng = np.random.default_rng(K)
    C = 4
    x = workloads.random_input((2, C, 11, 9), rng)
    w = np.zeros((C, C, K, K))
    for c in range(C):
        w[c, c, K // 2, K // 2] = 1.0
    y, _ = oracle.dense7(x, w, 1, (K - 1) // 2)
    np.testing.assert_array_equal(y, x.astype(np.float64))
    # same through the CSR walker
    flat = w.reshape(C, -1)
    rowptr = np.concatenate([[0], np.cumsum((flat != 0).sum(1))]).astype(np.int32)
    colidx = np.nonzero(flat)[1].astype(np.int32)
    value = flat[flat != 0].astype(np.float32)
    yc, _ = oracle.csr(x, rowptr, colidx, value, C, K, K, 1, (K - 1) // 2)
    np.testing.assert_array_equal(yc, x.astype(np.float64))


# Hand-computed outputs of a 3x3 input X = [[1,2,3],[4,5,6],[7,8,9]] under
# single-nonzero 3x3 filters (weight 1 at kernel row r, column s), pad 1,
# stride 1.  Eq.(1) reads X[h + r - P, w + s - P] (cross-correlation, no
# flip), so tap (0,0) shifts the image down-right and tap (2,2) up-left.
X33 = np.array([[1, 2, 3], [4, 5, 6], [7, 8, 9]], dtype=np.float64)
HAND = {
    (0, 0): [[0, 0, 0], [0, 1, 2], [0, 4, 5]],
    (0, 1): [[0, 0, 0], [1, 2, 3], [4, 5, 6]],
    (0, 2): [[0, 0, 0], [2, 3, 0], [5, 6, 0]],
    (1, 0): [[0, 1, 2], [0, 4, 5], [0, 7, 8]],
    (1, 1): [[1, 2, 3], [4, 5, 6], [7, 8, 9]],
    (1, 2): [[2, 3, 0], [5, 6, 0], [8, 9, 0]],
    (2, 0): [[0, 4, 5], [0, 7, 8], [0, 0, 0]],
    (2, 1): [[4, 5, 6], [7, 8, 9], [0, 0, 0]],
    (2, 2): [[5, 6, 0], [8, 9, 0], [0, 0, 0]],
}


@pytest.mark.parametrize("tap", sorted(HAND))
def test_single_nonzero_enumeration_pad1(tap):
    r, s = tap
    x = X33.reshape(1, 1, 3, 3)
    w = np.zeros((1, 1, 3, 3))
    w[0, 0, r, s] = 1.0
    y, a = oracle.dense7(x, w, 1, 1)
    np.testing.assert_array_equal(y[0, 0], np.array(HAND[tap], dtype=np.float64))
    np.testing.assert_array_equal(a, y)  # nonnegative terms: |sum| == sum of |.|
    rowptr = np.array([0, 1], dtype=np.int32)
    colidx = np.array([r * 3 + s], dtype=np.int32)
    yc, _ = oracle.csr(x, rowptr, colidx, np.array([1.0], np.float32), 1, 3, 3, 1, 1)
    np.testing.assert_array_equal(yc[0, 0], np.array(HAND[tap], dtype=np.float64))


def test_single_nonzero_enumeration_pad0():
    # Without padding the 3x3 filter fits once: the output is X[r, s].
    x = X33.reshape(1, 1, 3, 3)
    for r, s in itertools.product(range(3), range(3)):
        w = np.zeros((1, 1, 3, 3))
        w[0, 0, r, s] = -2.0
        y, a = oracle.dense7(x, w, 1, 0)
        assert y.shape == (1, 1, 1, 1)
        assert y[0, 0, 0, 0] == -2.0 * X33[r, s]
        assert a[0, 0, 0, 0] == 2.0 * X33[r, s]


def test_channel_index_convention():
    # colidx = (c*R + r)*S + s: a single nonzero in column 1*9 + 0*3 + 2 = 11
    # reads channel 1 at tap (0, 2).
    x = np.stack([X33, 10 * X33]).reshape(1, 2, 3, 3)
    rowptr = np.array([0, 1], dtype=np.int32)
    colidx = np.array([11], dtype=np.int32)
    y, _ = oracle.csr(x, rowptr, colidx, np.array([1.0], np.float32), 1, 3, 3, 1, 1)
    np.testing.assert_array_equal(y[0, 0], 10 * np.array(HAND[(0, 2)], dtype=np.float64))


# --------------------------------------------------------------------------
# abs_sum properties
# --------------------------------------------------------------------------

def test_abs_sum_properties():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, 3, 8, 7))
    w = rng.standard_normal((4, 3, 3, 3))
    y, a = oracle.dense7(x, w, 1, 1)
    assert np.all(a >= np.abs(y) - 1e-12)
    ya, _ = oracle.dense7(np.abs(x), np.abs(w), 1, 1)
    np.testing.assert_allclose(a, ya, rtol=1e-13)


def test_oracle_rejects_bad_csr():
    x = np.ones((1, 1, 3, 3))
    with pytest.raises(ValueError):
        oracle.csr(x, np.array([0, 1], np.int32), np.array([9], np.int32),
                   np.array([1.0], np.float32), 1, 3, 3, 1, 1)
    with pytest.raises(ValueError):
        oracle.csr(x, np.array([1, 1], np.int32), np.array([0], np.int32),
                   np.array([1.0], np.float32), 1, 3, 3, 1, 1)


def test_oracle_threads_agree():
    L = workloads.LAYERS["tiny"]
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L)
    y1, a1, t1 = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad,
                            threads=1, return_threads=True)
    y4, a4, t4 = oracle.csr(x, rowptr, colidx, value, L.M, L.R, L.S, L.stride, L.pad,
                            threads=4, return_threads=True)
    assert t1 == 1 and t4 == 4
    np.testing.assert_array_equal(y1, y4)
    np.testing.assert_array_equal(a1, a4)


# --------------------------------------------------------------------------
# Accounting: Table 1 and the ridge points, from the printed values
# --------------------------------------------------------------------------

def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_table1_arithmetic_intensity():
    rows = _read_golden("table1_arithmetic_intensity.txt")
    n = 0
    for key, printed in rows:
        if key == "dense":
            ai = roofline.ai_dense(32, 256, 256, 32, 64, 3)
            assert abs(ai - float(printed)) < 0.5
            assert abs(ai - 95.99) < 0.01
            continue
        ai = roofline.ai_sparse(32, 256, 256, 32, 64, 3, float(key))
        # every printed cell is within 0.06 of Eq.(7)/(8); one (0.94 -> 5.76
        # printed as 5.7) is truncated rather than rounded
        assert abs(ai - float(printed)) <= 0.06 + 1e-9, (key, ai, printed)
        n += 1
    assert n == 9


def test_table1_rejects_two_byte_activations():
    # With the text's P = 2 the table would double: the pin is sensitive to it.
    ai = roofline.ai_sparse(32, 256, 256, 32, 64, 3, 0.90, P=2, P_entry=4)
    assert ai > 15


def test_ridge_points():
    for _dev, tf, gbs, printed in _read_golden("ridge_points.txt"):
        r = roofline.ridge(float(tf) * 1e12, float(gbs) * 1e9)
        assert abs(r - float(printed)) < 0.01, (_dev, r, printed)


# --------------------------------------------------------------------------
# Generators (seeded, reproducible, documented distributions)
# --------------------------------------------------------------------------

def test_generators_reproducible_and_valid():
    for name in ("tiny", "tiny_int", "resnet3x3", "sweep90", "alex11x11"):
        L = workloads.LAYERS[name]
        a = workloads.make_weights(L)
        b = workloads.make_weights(L)
        for u, v in zip(a, b):
            np.testing.assert_array_equal(u, v)
        rowptr, colidx, value = a
        assert rowptr[0] == 0 and np.all(np.diff(rowptr) >= 0)
        assert rowptr[-1] == colidx.size == value.size
        assert colidx.min() >= 0 and colidx.max() < L.CRS
        for m in range(L.M):
            seg = colidx[rowptr[m]:rowptr[m + 1]]
            assert np.all(np.diff(seg) > 0)
        dens = colidx.size / (L.M * L.CRS)
        assert abs(dens - L.density) < 0.15 * L.density + 0.01
        if L.integer:
            assert set(np.unique(value)) <= {-3, -2, -1, 1, 2, 3}
            x = workloads.make_input(L)
            assert x.min() >= 0 and x.max() <= 7 and np.all(x == np.round(x))


def test_lognormal_rows_are_skewed():
    L = workloads.LAYERS["sweep90"]
    rowptr, _, _ = workloads.make_weights(L)
    counts = np.diff(rowptr)
    assert abs(counts.mean() / L.CRS - L.density) < 0.01 * L.density + 1e-3
    assert counts.max() > 3 * counts.mean()
    assert counts.min() < 0.5 * counts.mean()
