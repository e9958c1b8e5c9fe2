"""Pins for the convolution oracle against what the definition fixes.

Expected values come from elsewhere than the oracle's formula: seven nested
loops over exact rationals (``fractions.Fraction``) on tiny inputs, closed
forms (a delta filter copies or shifts the input, a 1 x 1 stride-1
convolution is a plain matrix product of the pinned GEMM oracle, a box filter
on a constant image counts the taps inside the image), and the per-point
evaluator against the full one. The last test plants mistakes in copies of
the oracle and checks that a pin catches each.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import conv_oracle as co
from half_precision_dense_gb300 import inputs


def rand16(shape, dtype, seed, tid):
    n = int(np.prod(shape))
    t = inputs.generate((1, n), dtype, seed, tid)
    return inputs.bits(t).reshape(shape)


def ones16(shape, dtype):
    one = inputs.bits(torch.ones(1, 1, dtype=inputs.TORCH_DTYPES[dtype]))[0, 0]
    return np.full(shape, one, dtype=np.uint16)


def brute(x, w, dtype, stride, pad):
    """y as exact rationals from the definition, seven nested loops."""
    N, H, W, C = x.shape
    R, S, _, K = w.shape
    P, Q = co.out_size(H, W, R, S, stride, pad)
    xv = oracle.decode(x, dtype)
    wv = oracle.decode(w, dtype)
    y = {}
    for n in range(N):
        for p in range(P):
            for q in range(Q):
                for k in range(K):
                    acc = Fraction(0)
                    for r in range(R):
                        for s in range(S):
                            h, ww = p * stride - pad + r, q * stride - pad + s
                            if 0 <= h < H and 0 <= ww < W:
                                for c in range(C):
                                    acc += Fraction(float(xv[n, h, ww, c])) * Fraction(float(wv[r, s, c, k]))
                    y[(n, p, q, k)] = acc
    return y, (N, P, Q, K)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [
    # (N, H, W, C, R, S, K, stride, pad)
    (1, 4, 4, 2, 3, 3, 2, 1, 1),
    (2, 5, 3, 3, 2, 2, 1, 2, 0),
    (1, 6, 5, 1, 3, 1, 3, 1, 2),
    (1, 7, 7, 2, 5, 3, 2, 3, 1),
])
def test_brute_force_exact_rationals(dtype, shape):
    N, H, W, C, R, S, K, stride, pad = shape
    x = rand16((N, H, W, C), dtype, 1, 0)
    w = rand16((R, S, C, K), dtype, 1, 1)
    y, yshape = brute(x, w, dtype, stride, pad)
    got = co.conv_f64(x, w, dtype, stride, pad)
    assert got.shape == yshape
    for idx, v in y.items():
        assert Fraction(float(got[idx])) == v or abs(Fraction(float(got[idx])) - v) <= abs(v) * Fraction(1, 2 ** 50), idx


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_delta_filter_copies_and_shifts(dtype):
    x = rand16((2, 6, 5, 4), dtype, 2, 0)
    # w[r0, s0, c, c] = 1: output = input at offset (r0 - pad, s0 - pad)
    w = np.zeros((3, 3, 4, 4), dtype=np.uint16)
    one = ones16((1,), dtype)[0]
    for c in range(4):
        w[1, 1, c, c] = one
    y = co.conv(x, w, dtype, stride=1, pad=1)
    assert np.array_equal(y, x)
    w2 = np.zeros((3, 3, 4, 4), dtype=np.uint16)
    for c in range(4):
        w2[0, 2, c, c] = one
    y2 = co.conv_f64(x, w2, dtype, stride=1, pad=1)      # y[p, q] = x[p - 1, q + 1]
    xv = oracle.decode(x, dtype)
    assert np.array_equal(y2[:, 1:, :-1], xv[:, :-1, 1:])
    assert np.all(y2[:, 0] == 0) and np.all(y2[:, :, -1] == 0)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_pointwise_conv_is_the_gemm(dtype):
    x = rand16((2, 5, 7, 16), dtype, 3, 0)
    w = rand16((1, 1, 16, 12), dtype, 3, 1)
    y = co.conv(x, w, dtype)
    g = oracle.gemm(x.reshape(-1, 16), w.reshape(16, 12), dtype)
    assert np.array_equal(y.reshape(-1, 12), g)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_box_filter_counts_taps_inside_the_image(dtype):
    # all-ones image and 3 x 3 all-ones filter, pad 1: every output is the
    # number of taps that land inside (9 inside, 6 on edges, 4 at corners) x C
    C = 3
    x = ones16((1, 5, 6, C), dtype)
    w = ones16((3, 3, C, 1), dtype)
    y = co.conv_f64(x, w, dtype, stride=1, pad=1)[0, :, :, 0]
    rows = np.array([2, 3, 3, 3, 2])
    cols = np.array([2, 3, 3, 3, 3, 2])
    assert np.array_equal(y, C * np.outer(rows, cols))


def test_point_evaluator_agrees():
    dtype = "bf16"
    x = rand16((2, 9, 8, 5), dtype, 4, 0)
    w = rand16((3, 2, 5, 6), dtype, 4, 1)
    full = co.conv_f64(x, w, dtype, 2, 1)
    pts = [(0, 0, 0), (1, 4, 3), (0, 2, 1), (1, 0, 4)]
    got = co.conv_at(x, w, dtype, 2, 1, pts)
    for i, (n, p, q) in enumerate(pts):
        assert np.allclose(got[i], full[n, p, q], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Planted mistakes: each broken copy must fail at least one pin above.

def _flipped(x, w, dtype, stride=1, pad=0):          # convolution instead of correlation
    return co.conv_f64(x, w[::-1, ::-1].copy(), dtype, stride, pad)


def _pad_one_side(x, w, dtype, stride=1, pad=0):    # padding only at the start
    y = co.conv_f64(np.pad(x, ((0, 0), (pad, 0), (pad, 0), (0, 0))), w, dtype, stride, 0)
    return y


def _swapped_rs(x, w, dtype, stride=1, pad=0):
    return co.conv_f64(x, np.ascontiguousarray(np.swapaxes(w, 0, 1)).reshape(w.shape), dtype, stride, pad)


def _stride_ignored(x, w, dtype, stride=1, pad=0):
    return co.conv_f64(x, w, dtype, 1, pad)


BROKEN = {"flipped_kernel": _flipped, "pad_one_side": _pad_one_side, "swapped_r_s": _swapped_rs,
          "stride_ignored": _stride_ignored}


def _pins_pass(conv_f64):
    try:
        for shape in [(1, 4, 4, 2, 3, 3, 2, 1, 1), (2, 5, 3, 3, 2, 2, 1, 2, 0), (1, 7, 7, 2, 5, 3, 2, 3, 1)]:
            N, H, W, C, R, S, K, stride, pad = shape
            x = rand16((N, H, W, C), "bf16", 1, 0)
            w = rand16((R, S, C, K), "bf16", 1, 1)
            y, yshape = brute(x, w, "bf16", stride, pad)
            got = conv_f64(x, w, "bf16", stride, pad)
            if got.shape != yshape:
                return False
            for idx, v in y.items():
                if abs(Fraction(float(got[idx])) - v) > abs(v) * Fraction(1, 2 ** 50):
                    return False
    except Exception:
        return False
    return True


def test_pins_pass_for_the_oracle():
    assert _pins_pass(co.conv_f64)


@pytest.mark.parametrize("broken", sorted(BROKEN))
def test_pins_catch_planted_mistakes(broken):
    assert not _pins_pass(BROKEN[broken])
