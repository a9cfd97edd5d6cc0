"""Pins for the CPU oracle: each check rests on something other than the oracle.

Pages (by title): P47 = "Kimi-K2.6__l2_p47" (conv3d + Mish + Tanh),
P8 = "Kimi-K2.6__l2_p8" (conv3d + /2 + maxpool + mean + bias + channel sum),
P86 = "Kimi-K2.6__l1_p86" (depthwise-separable conv2d).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.optimize
import scipy.signal

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


@pytest.fixture(scope="module")
def facts():
    with open(GOLDEN) as f:
        return json.load(f)


def rel_err(a, b):
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b) / (1e-300 + np.maximum(1.0, np.abs(b))))) if a.size else 0.0


# ------------------------------------------------------------------ printed facts
def test_printed_dims_and_counts(facts):
    for e in facts["conv3d_out_dims"]:
        assert list(oracle.conv3d_out_dims(*e["in"])) == e["out"], e["cite"]
    for e in facts["conv3d_out_count"]:
        N, Cin, D, H, W = e["shape"]
        assert N * e["cout"] * math.prod(oracle.conv3d_out_dims(D, H, W)) == e["count"], e["cite"]
    for e in facts["conv3d_macs"]:
        N, Cin, D, H, W = e["shape"]
        assert oracle.conv3d_macs(N, Cin, D, H, W, e["cout"]) == e["macs"], e["cite"]
    for e in facts["pooled_dims"]:
        p = oracle.pooled_dims(*e["conv_out"], pool=e["pool"])
        assert list(p) == e["pooled"] and math.prod(p) == e["cells"], e["cite"]
    for e in facts["dwsep_counts"]:
        N, C, H, W = e["shape"]
        assert N * H * W == e["pixels"]
        assert oracle.dwsep_macs(N, C, H, W, e["cout"]) == e["pixels"] * e["macs_per_pixel"], e["cite"]


def test_oracle_output_shape_follows_dims():
    x = np.zeros((1, 2, 5, 6, 7), np.float32)
    w = np.zeros((3, 2, 3, 3, 3), np.float32)
    assert oracle.conv3d(x, w).shape == (1, 3, 3, 4, 5)


# ------------------------------------------------------------------ conv3d
def im2col_conv3d(x, w, b):
    """Brute force: explicit [M x K] patch matrix times W^T, float64 (numpy matmul)."""
    x = x.astype(np.float64); w = w.astype(np.float64)
    N, Cin, D, H, W = x.shape
    Cout = w.shape[0]
    OD, OH, OW = D - 2, H - 2, W - 2
    cols = np.empty((N, OD, OH, OW, Cin, 3, 3, 3))
    for kd in range(3):
        for kh in range(3):
            for kw in range(3):
                patch = x[:, :, kd:kd + OD, kh:kh + OH, kw:kw + OW]  # N,C,OD,OH,OW
                cols[..., kd, kh, kw] = np.moveaxis(patch, 1, -1)
    A = cols.reshape(N * OD * OH * OW, Cin * 27)
    Y = A @ w.reshape(Cout, Cin * 27).T
    if b is not None:
        Y = Y + b.astype(np.float64)[None, :]
    return np.moveaxis(Y.reshape(N, OD, OH, OW, Cout), -1, 1)


def test_conv3d_tiny_workload_vs_im2col():
    wl = si.tiny_conv3d()
    t = wl.generate_all()
    y = oracle.conv3d(t["x"], t["w"], t["b"])
    assert y.shape == (2, 8, 6, 6, 6)
    assert rel_err(y, im2col_conv3d(t["x"], t["w"], t["b"])) < 1e-12


@pytest.mark.parametrize("shape", [(1, 1, 3, 3, 3, 1), (2, 3, 5, 4, 7, 2), (1, 5, 4, 9, 3, 3),
                                   (2, 2, 6, 5, 5, 4)])
def test_conv3d_odd_shapes_vs_im2col(shape):
    N, Cin, D, H, W, Cout = shape
    rng = np.random.default_rng(sum(shape))
    x = rng.standard_normal((N, Cin, D, H, W)).astype(np.float32)
    w = rng.uniform(-1, 1, (Cout, Cin, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-1, 1, Cout).astype(np.float32)
    assert rel_err(oracle.conv3d(x, w, b), im2col_conv3d(x, w, b)) < 1e-12
    assert rel_err(oracle.conv3d(x, w, None), im2col_conv3d(x, w, None)) < 1e-12


def test_conv3d_vs_scipy_correlate():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((2, 3, 6, 7, 8)).astype(np.float32)
    w = rng.uniform(-1, 1, (4, 3, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-1, 1, 4).astype(np.float32)
    ref = np.zeros((2, 4, 4, 5, 6))
    for n in range(2):
        for k in range(4):
            ref[n, k] = b[k]
            for c in range(3):
                ref[n, k] += scipy.signal.correlate(x[n, c].astype(np.float64),
                                                    w[k, c].astype(np.float64),
                                                    mode="valid", method="direct")
    assert rel_err(oracle.conv3d(x, w, b), ref) < 1e-12


def test_conv3d_single_tap_pins_orientation():
    # One nonzero tap at (kd, kh, kw) = (0, 1, 2) reads x[od, oh+1, ow+2]: no flip, no transpose.
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, 1, 5, 6, 7)).astype(np.float32)
    w = np.zeros((1, 1, 3, 3, 3), np.float32)
    w[0, 0, 0, 1, 2] = 1.0
    y = oracle.conv3d(x, w)
    assert np.array_equal(y[0, 0], x[0, 0, 0:3, 1:5, 2:7].astype(np.float64))


def test_conv3d_delta_kernel_is_centre_crop():
    rng = np.random.default_rng(4)
    C = 3
    x = rng.standard_normal((2, C, 5, 6, 7)).astype(np.float32)
    w = np.zeros((C, C, 3, 3, 3), np.float32)
    for k in range(C):
        w[k, k, 1, 1, 1] = 1.0
    assert np.array_equal(oracle.conv3d(x, w), x[:, :, 1:-1, 1:-1, 1:-1].astype(np.float64))


def test_conv3d_constant_input():
    rng = np.random.default_rng(5)
    x = np.ones((1, 4, 5, 5, 5), np.float32)
    w = rng.uniform(-1, 1, (3, 4, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-1, 1, 3).astype(np.float32)
    y = oracle.conv3d(x, w, b)
    expect = w.astype(np.float64).reshape(3, -1).sum(1) + b
    assert rel_err(y, np.broadcast_to(expect[None, :, None, None, None], y.shape)) < 1e-13


def test_conv3d_linearity_exact_on_integers():
    # Small integers keep every float64 sum exact, so linearity must hold bit for bit.
    rng = np.random.default_rng(6)
    x1 = rng.integers(-4, 5, (1, 3, 5, 6, 5)).astype(np.float32)
    x2 = rng.integers(-4, 5, (1, 3, 5, 6, 5)).astype(np.float32)
    w1 = rng.integers(-3, 4, (2, 3, 3, 3, 3)).astype(np.float32)
    w2 = rng.integers(-3, 4, (2, 3, 3, 3, 3)).astype(np.float32)
    assert np.array_equal(oracle.conv3d(x1 + x2, w1), oracle.conv3d(x1, w1) + oracle.conv3d(x2, w1))
    assert np.array_equal(oracle.conv3d(x1, w1 + w2), oracle.conv3d(x1, w1) + oracle.conv3d(x1, w2))
    assert np.array_equal(oracle.conv3d(3 * x1, w1), 3 * oracle.conv3d(x1, w1))


def test_conv3d_translation_equivariance():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((1, 2, 7, 8, 9)).astype(np.float32)
    w = rng.uniform(-1, 1, (2, 2, 3, 3, 3)).astype(np.float32)
    y = oracle.conv3d(x, w)
    ys = oracle.conv3d(x[:, :, 1:, 2:, 3:], w)
    assert np.array_equal(ys, y[:, :, 1:, 2:, 3:])


def test_conv3d_at_matches_full():
    wl = si.tiny_conv3d()
    t = wl.generate_all()
    y = oracle.conv3d(t["x"], t["w"], t["b"])
    rng = np.random.default_rng(9)
    idx = np.stack([rng.integers(0, s, 50) for s in y.shape], 1)
    assert np.array_equal(oracle.conv3d_at(t["x"], t["w"], t["b"], idx), y[tuple(idx.T)])


# ------------------------------------------------------------------ padded conv3d
# [P47] the padding discussion: input coordinate od + kd - padding, zero outside the
# tensor, output size D + 2*padding - 2.
@pytest.mark.parametrize("shape,pad", [((1, 2, 3, 4, 5, 3), 1), ((2, 3, 4, 3, 6, 2), 1),
                                       ((1, 2, 3, 3, 3, 2), 2), ((1, 1, 1, 1, 1, 1), 1),
                                       ((2, 2, 5, 4, 3, 2), 0)])
def test_conv3d_pad_vs_numpy_pad_and_im2col(shape, pad):
    N, Cin, D, H, W, Cout = shape
    rng = np.random.default_rng(100 + sum(shape) + pad)
    x = rng.standard_normal((N, Cin, D, H, W)).astype(np.float32)
    w = rng.uniform(-1, 1, (Cout, Cin, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-1, 1, Cout).astype(np.float32)
    xp = np.pad(x, ((0, 0), (0, 0), (pad, pad), (pad, pad), (pad, pad)))
    y = oracle.conv3d_pad(x, w, b, pad)
    assert y.shape == (N, Cout, D + 2 * pad - 2, H + 2 * pad - 2, W + 2 * pad - 2)
    assert rel_err(y, im2col_conv3d(xp, w, b)) < 1e-12


def test_conv3d_pad_vs_scipy_same():
    rng = np.random.default_rng(101)
    x = rng.standard_normal((1, 2, 5, 6, 4)).astype(np.float32)
    w = rng.uniform(-1, 1, (3, 2, 3, 3, 3)).astype(np.float32)
    ref = np.zeros((1, 3, 5, 6, 4))
    for k in range(3):
        for c in range(2):
            ref[0, k] += scipy.signal.correlate(x[0, c].astype(np.float64), w[k, c].astype(np.float64),
                                                mode="same", method="direct")
    assert rel_err(oracle.conv3d_pad(x, w, None, 1), ref) < 1e-12


def test_conv3d_pad_delta_kernel_is_identity():
    rng = np.random.default_rng(102)
    C = 3
    x = rng.standard_normal((2, C, 4, 5, 6)).astype(np.float32)
    w = np.zeros((C, C, 3, 3, 3), np.float32)
    for k in range(C):
        w[k, k, 1, 1, 1] = 1.0
    assert np.array_equal(oracle.conv3d_pad(x, w, None, 1), x.astype(np.float64))


def test_conv3d_pad_constant_input_corner_and_interior():
    rng = np.random.default_rng(103)
    x = np.ones((1, 2, 5, 5, 5), np.float32)
    w = rng.uniform(-1, 1, (3, 2, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-1, 1, 3).astype(np.float32)
    y = oracle.conv3d_pad(x, w, b, 1)
    w64 = w.astype(np.float64)
    # Corner (0,0,0): only taps with kd, kh, kw >= 1 land inside.
    corner = b + w64[:, :, 1:, 1:, 1:].reshape(3, -1).sum(1)
    # Interior: every tap lands inside.
    interior = b + w64.reshape(3, -1).sum(1)
    assert rel_err(y[0, :, 0, 0, 0], corner) < 1e-13
    assert rel_err(y[0, :, 2, 2, 2], interior) < 1e-13


def test_conv3d_pad_zero_equals_valid_and_at_matches_full():
    rng = np.random.default_rng(104)
    x = rng.standard_normal((1, 2, 5, 6, 7)).astype(np.float32)
    w = rng.uniform(-1, 1, (2, 2, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-1, 1, 2).astype(np.float32)
    assert np.array_equal(oracle.conv3d_pad(x, w, b, 0), oracle.conv3d(x, w, b))
    y = oracle.conv3d_pad(x, w, b, 1)
    idx = np.stack([rng.integers(0, s, 40) for s in y.shape], 1)
    assert np.array_equal(oracle.conv3d_pad_at(x, w, b, 1, idx), y[tuple(idx.T)])


# ------------------------------------------------------------------ strided conv3d
# [P47] the stride and padding discussion: input window of output d_out starts at
# d_out*stride - padding; OD = (D + 2*padding - KD)/stride + 1.
def strided_im2col(xp, w, b, S):
    """Brute force on an already padded input: strided [M x K] patches times W^T (float64)."""
    xp = xp.astype(np.float64); w = w.astype(np.float64)
    N, Cin, D, H, W = xp.shape
    Cout = w.shape[0]
    OD, OH, OW = (D - 3) // S + 1, (H - 3) // S + 1, (W - 3) // S + 1
    cols = np.empty((N, OD, OH, OW, Cin, 3, 3, 3))
    for kd in range(3):
        for kh in range(3):
            for kw in range(3):
                patch = xp[:, :, kd:kd + S * (OD - 1) + 1:S, kh:kh + S * (OH - 1) + 1:S,
                           kw:kw + S * (OW - 1) + 1:S]
                cols[..., kd, kh, kw] = np.moveaxis(patch, 1, -1)
    Y = cols.reshape(N * OD * OH * OW, Cin * 27) @ w.reshape(Cout, Cin * 27).T
    if b is not None:
        Y = Y + b.astype(np.float64)[None, :]
    return np.moveaxis(Y.reshape(N, OD, OH, OW, Cout), -1, 1)


@pytest.mark.parametrize("shape,pad,stride", [((1, 2, 5, 6, 7, 3), 0, 2), ((2, 3, 6, 5, 8, 2), 1, 2),
                                              ((1, 2, 4, 4, 4, 2), 2, 2), ((1, 1, 3, 3, 3, 1), 0, 2),
                                              ((1, 2, 7, 9, 6, 2), 1, 3), ((1, 2, 4, 5, 6, 2), 1, 1)])
def test_conv3d_ex_vs_numpy_pad_and_strided_im2col(shape, pad, stride):
    N, Cin, D, H, W, Cout = shape
    rng = np.random.default_rng(200 + sum(shape) + 7 * pad + stride)
    x = rng.standard_normal((N, Cin, D, H, W)).astype(np.float32)
    w = rng.uniform(-1, 1, (Cout, Cin, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-1, 1, Cout).astype(np.float32)
    xp = np.pad(x, ((0, 0), (0, 0), (pad, pad), (pad, pad), (pad, pad)))
    y = oracle.conv3d_ex(x, w, b, pad, stride)
    assert y.shape[2:] == tuple((s + 2 * pad - 3) // stride + 1 for s in (D, H, W))
    assert rel_err(y, strided_im2col(xp, w, b, stride)) < 1e-12


def test_conv3d_ex_vs_scipy_valid_subsampled():
    rng = np.random.default_rng(201)
    x = rng.standard_normal((1, 2, 7, 8, 9)).astype(np.float32)
    w = rng.uniform(-1, 1, (2, 2, 3, 3, 3)).astype(np.float32)
    xp = np.pad(x, ((0, 0), (0, 0), (1, 1), (1, 1), (1, 1))).astype(np.float64)
    ref = np.zeros((1, 2) + tuple((s + 2 - 3) // 2 + 1 for s in (7, 8, 9)))
    for k in range(2):
        full = sum(scipy.signal.correlate(xp[0, c], w[k, c].astype(np.float64), mode="valid", method="direct")
                   for c in range(2))
        ref[0, k] = full[::2, ::2, ::2]
    assert rel_err(oracle.conv3d_ex(x, w, None, 1, 2), ref) < 1e-12


def test_conv3d_ex_centre_delta_subsamples():
    rng = np.random.default_rng(202)
    C = 2
    x = rng.standard_normal((1, C, 7, 6, 5)).astype(np.float32)
    w = np.zeros((C, C, 3, 3, 3), np.float32)
    for k in range(C):
        w[k, k, 1, 1, 1] = 1.0
    # pad 1, stride 2: output (od, oh, ow) reads x[2od, 2oh, 2ow]
    assert np.array_equal(oracle.conv3d_ex(x, w, None, 1, 2), x[:, :, ::2, ::2, ::2].astype(np.float64))


def test_conv3d_ex_stride1_is_padded_and_at_matches_full():
    rng = np.random.default_rng(203)
    x = rng.standard_normal((1, 2, 5, 6, 7)).astype(np.float32)
    w = rng.uniform(-1, 1, (2, 2, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-1, 1, 2).astype(np.float32)
    assert np.array_equal(oracle.conv3d_ex(x, w, b, 1, 1), oracle.conv3d_pad(x, w, b, 1))
    y = oracle.conv3d_ex(x, w, b, 1, 2)
    idx = np.stack([rng.integers(0, s, 30) for s in y.shape], 1)
    assert np.array_equal(oracle.conv3d_ex_at(x, w, b, 1, 2, idx), y[tuple(idx.T)])


# ------------------------------------------------------------------ tanh(mish)
def test_tanh_mish_zero():
    assert oracle.tanh_mish_scalar(0.0) == 0.0


def test_tanh_mish_identity_form_high_precision():
    # With n = e^y: tanh(log(1 + n)) = ((1+n)^2 - 1) / ((1+n)^2 + 1) = n(n+2) / (n(n+2) + 2),
    # an algebraic identity, evaluated here at 50 digits.
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    ys = np.concatenate([np.linspace(-30, 30, 1201), [-1e-8, 1e-8, 0.5, -0.5, 19.99, 20.01]])
    got = oracle.tanh_mish(ys)
    for y, g in zip(ys, got):
        n = mp.e ** mp.mpf(float(y))
        t = n * (n + 2)
        ref = mp.tanh(mp.mpf(float(y)) * t / (t + 2))
        assert abs(g - float(ref)) <= 4e-16 * max(1.0, abs(float(ref))) + 1e-300, y


def test_tanh_mish_asymptotes():
    for y in [20.0, 25.0, 50.0, 200.0, 800.0, 1e5]:
        assert abs(oracle.tanh_mish_scalar(y) - math.tanh(y)) < 1e-15
    for y in [-40.0, -100.0, -1000.0]:
        v = oracle.tanh_mish_scalar(y)
        assert -1e-15 < v <= 0.0


def test_tanh_mish_minimum_matches_mish_minimum():
    # Mish has its global minimum of about -0.30884 near y = -1.1924 (Misra, 2019);
    # tanh is increasing, so tanh(mish) has its minimum at the same point.
    res = scipy.optimize.minimize_scalar(oracle.tanh_mish_scalar, bounds=(-3, 0), method="bounded",
                                         options={"xatol": 1e-10})
    # Both textbook figures are quoted to about five digits.
    assert abs(res.x - (-1.1924)) < 1e-3
    assert abs(math.atanh(res.fun) - (-0.30884)) < 1e-5


# ------------------------------------------------------------------ pool-reduce
def enumerate_pool_reduce(y, divisor, pool, bias2):
    """Brute force by visiting every element once and keeping a running max per window."""
    N, C, OD, OH, OW = y.shape
    PD, PH, PW = OD // pool, OH // pool, OW // pool
    out = []
    for n in range(N):
        total = 0.0
        for c in range(C):
            best = {}
            for d in range(PD * pool):
                for h in range(PH * pool):
                    for w in range(PW * pool):
                        key = (d // pool, h // pool, w // pool)
                        v = y[n, c, d, h, w] / divisor
                        if key not in best or v > best[key]:
                            best[key] = v
            cells = PD * PH * PW
            total += math.fsum(best.values()) / cells + float(bias2[c])
        out.append(total)
    return np.array(out)


@pytest.mark.parametrize("dims", [(4, 6, 6), (5, 7, 6), (3, 4, 9), (2, 2, 2)])
def test_pool_reduce_vs_enumeration(dims):
    rng = np.random.default_rng(sum(dims))
    y = rng.standard_normal((2, 3) + dims)
    bias2 = rng.standard_normal(3).astype(np.float32)
    for div in (2.0, 3.0, -1.0):
        got = oracle.pool_reduce(y, div, 2, bias2)
        assert rel_err(got, enumerate_pool_reduce(y, div, 2, bias2)) < 1e-12


def test_pool_reduce_identity_form():
    # out[n] = S[n] / (divisor * cells) + sum_c bias2[c], S = sum over channels and cells
    # of the window max of the undivided conv output (valid for divisor > 0).
    rng = np.random.default_rng(11)
    y = rng.standard_normal((3, 4, 6, 8, 10))
    bias2 = rng.standard_normal(4).astype(np.float32)
    blocks = y.reshape(3, 4, 3, 2, 4, 2, 5, 2).max(axis=(3, 5, 7))
    S = blocks.reshape(3, -1).sum(1)
    expect = S / (2.0 * 3 * 4 * 5) + bias2.astype(np.float64).sum()
    assert rel_err(oracle.pool_reduce(y, 2.0, 2, bias2), expect) < 1e-12


def test_pool_reduce_constant_and_floor_mode():
    bias2 = np.array([0.5, -1.25, 2.0], np.float32)
    y = np.full((1, 3, 5, 7, 9), 3.0)
    assert oracle.pool_reduce(y, 2.0, 2, bias2)[0] == pytest.approx(3 * 1.5 + 1.25, abs=1e-14)
    # Floor mode: the last plane, row and column (odd sizes) belong to no window.
    y[:, :, 4, :, :] = 1e6
    y[:, :, :, 6, :] = 1e6
    y[:, :, :, :, 8] = 1e6
    assert oracle.pool_reduce(y, 2.0, 2, bias2)[0] == pytest.approx(3 * 1.5 + 1.25, abs=1e-14)


def test_pool_reduce_planted_maxima():
    # Each 2x2x2 window holds zeros except one planted value at a varying corner.
    rng = np.random.default_rng(12)
    y = np.zeros((1, 2, 4, 4, 6))
    planted = rng.uniform(1, 2, (2, 2, 2, 3))
    for c in range(2):
        for i in range(2):
            for j in range(2):
                for l in range(3):
                    a, b_, e = (i + c) % 2, (j + l) % 2, (l + i) % 2
                    y[0, c, 2 * i + a, 2 * j + b_, 2 * l + e] = planted[c, i, j, l]
    bias2 = np.zeros(2, np.float32)
    expect = sum(planted[c].sum() / 2.0 / 12 for c in range(2))
    assert oracle.pool_reduce(y, 2.0, 2, bias2)[0] == pytest.approx(expect, rel=1e-14)


def test_conv3d_pool_reduce_zero_weights_closed_form():
    wl = si.conv3d_workload("t", 2, 3, 6, 8, 8, 4, seed=21, epilogue="pool_reduce", bias2=True)
    t = wl.generate_all()
    w0 = np.zeros_like(t["w"])
    got = oracle.conv3d_pool_reduce(t["x"], w0, t["b"], 2.0, 2, t["bias2"])
    expect = t["b"].astype(np.float64).sum() / 2.0 + t["bias2"].astype(np.float64).sum()
    assert np.allclose(got, expect, rtol=0, atol=1e-13)


# ------------------------------------------------------------------ depthwise-separable
def scipy_dwsep(x, w_dw, w_pw, b):
    N, C, H, W = x.shape
    dw = np.empty((N, C, H, W))
    for n in range(N):
        for c in range(C):
            dw[n, c] = scipy.signal.correlate2d(x[n, c].astype(np.float64),
                                                w_dw[c, 0].astype(np.float64),
                                                mode="same", boundary="fill", fillvalue=0.0)
    out = np.einsum("oc,nchw->nohw", w_pw[:, :, 0, 0].astype(np.float64), dw)
    if b is not None:
        out += b.astype(np.float64)[None, :, None, None]
    return out


@pytest.mark.parametrize("shape", [(1, 3, 5, 7, 4), (2, 4, 8, 6, 5), (1, 1, 1, 1, 1), (1, 2, 2, 9, 3)])
def test_dwsep_vs_scipy(shape):
    N, C, H, W, Cout = shape
    rng = np.random.default_rng(sum(shape))
    x = rng.standard_normal((N, C, H, W)).astype(np.float32)
    w_dw = rng.uniform(-1, 1, (C, 1, 3, 3)).astype(np.float32)
    w_pw = rng.uniform(-1, 1, (Cout, C, 1, 1)).astype(np.float32)
    b = rng.uniform(-1, 1, Cout).astype(np.float32)
    for bb in (None, b):
        ref = scipy_dwsep(x, w_dw, w_pw, bb)
        assert rel_err(oracle.dwsep(x, w_dw, w_pw, bb), ref) < 1e-12
        assert rel_err(oracle.dwsep_single_sum(x, w_dw, w_pw, bb), ref) < 1e-12


def test_dwsep_two_stage_equals_single_sum():
    wl = si.dwsep_workload("t", 2, 6, 9, 11, 5, seed=31, with_bias=True)
    t = wl.generate_all()
    a = oracle.dwsep(t["x"], t["w_dw"], t["w_pw"], t["b"])
    s = oracle.dwsep_single_sum(t["x"], t["w_dw"], t["w_pw"], t["b"])
    assert rel_err(a, s) < 1e-13


def test_dwsep_special_cases():
    rng = np.random.default_rng(32)
    x = rng.standard_normal((1, 4, 6, 7)).astype(np.float32)
    w_pw = rng.uniform(-1, 1, (3, 4, 1, 1)).astype(np.float32)
    # Centre-delta depthwise: the result is the pointwise GEMM of x.
    w_dw = np.zeros((4, 1, 3, 3), np.float32); w_dw[:, 0, 1, 1] = 1.0
    ref = np.einsum("oc,nchw->nohw", w_pw[:, :, 0, 0].astype(np.float64), x.astype(np.float64))
    assert rel_err(oracle.dwsep(x, w_dw, w_pw), ref) < 1e-14
    # Identity pointwise: the result is the depthwise conv alone; a one-tap kernel at
    # (kh, kw) = (0, 2) reads x[h-1, w+1] with zeros outside (padding 1, no flip).
    eye = np.eye(4, dtype=np.float32).reshape(4, 4, 1, 1)
    w_dw = np.zeros((4, 1, 3, 3), np.float32); w_dw[:, 0, 0, 2] = 1.0
    shifted = np.zeros_like(x, dtype=np.float64)
    shifted[:, :, 1:, :-1] = x[:, :, :-1, 1:]
    assert np.array_equal(oracle.dwsep(x, w_dw, eye), shifted)
    # The bias adds b[o] to every output of channel o.
    b = rng.uniform(-1, 1, 3).astype(np.float32)
    w_dw = rng.uniform(-1, 1, (4, 1, 3, 3)).astype(np.float32)
    d = oracle.dwsep(x, w_dw, w_pw, b) - oracle.dwsep(x, w_dw, w_pw, None)
    assert np.allclose(d, b.astype(np.float64)[None, :, None, None], atol=1e-14, rtol=0)


def test_dwsep_at_matches_full():
    wl = si.dwsep_workload("t", 2, 5, 8, 9, 6, seed=33)
    t = wl.generate_all()
    full = oracle.dwsep(t["x"], t["w_dw"], t["w_pw"])
    rng = np.random.default_rng(34)
    idx = np.stack([rng.integers(0, s, 60) for s in full.shape], 1)
    got = oracle.dwsep_at(t["x"], t["w_dw"], t["w_pw"], None, idx)
    assert rel_err(got, full[tuple(idx.T)]) < 1e-14


# ------------------------------------------------------------------ dwsep, K x K
# [P86] the discussion of kernel sizes other than 3 (templated on K, dispatched for 1,
# 3, 5, 7); reading: stride 1, dilation 1, padding (K-1)/2.
@pytest.mark.parametrize("K", [1, 3, 5, 7])
def test_dwsep_k_vs_scipy_same_and_einsum(K):
    rng = np.random.default_rng(300 + K)
    N, C, H, W, Cout = 2, 3, 9, 8, 4
    x = rng.standard_normal((N, C, H, W)).astype(np.float32)
    w_dw = rng.uniform(-1, 1, (C, 1, K, K)).astype(np.float32)
    w_pw = rng.uniform(-1, 1, (Cout, C, 1, 1)).astype(np.float32)
    b = rng.uniform(-1, 1, Cout).astype(np.float32)
    dw = np.zeros((N, C, H, W))
    for n in range(N):
        for c in range(C):
            dw[n, c] = scipy.signal.correlate2d(x[n, c].astype(np.float64), w_dw[c, 0].astype(np.float64),
                                                mode="same", boundary="fill")
    ref = np.einsum("oc,nchw->nohw", w_pw[:, :, 0, 0].astype(np.float64), dw) + b[None, :, None, None]
    got = oracle.dwsep_k(x, w_dw, w_pw, b)
    assert rel_err(got, ref) < 1e-12
    idx = np.stack([rng.integers(0, s, 40) for s in got.shape], 1)
    assert rel_err(oracle.dwsep_k_at(x, w_dw, w_pw, b, idx), got[tuple(idx.T)]) < 1e-12


def test_dwsep_k3_equals_dwsep_and_centre_delta():
    rng = np.random.default_rng(310)
    x = rng.standard_normal((1, 3, 7, 6)).astype(np.float32)
    w3 = rng.uniform(-1, 1, (3, 1, 3, 3)).astype(np.float32)
    w_pw = rng.uniform(-1, 1, (2, 3, 1, 1)).astype(np.float32)
    assert np.array_equal(oracle.dwsep_k(x, w3, w_pw), oracle.dwsep(x, w3, w_pw))
    w5 = np.zeros((3, 1, 5, 5), np.float32)
    w5[:, 0, 2, 2] = 1.0        # centre tap: the depthwise stage is the identity
    ref = np.einsum("oc,nchw->nohw", w_pw[:, :, 0, 0].astype(np.float64), x.astype(np.float64))
    assert rel_err(oracle.dwsep_k(x, w5, w_pw), ref) < 1e-14

