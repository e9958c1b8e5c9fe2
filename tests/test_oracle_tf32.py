"""Pins for the TF32 oracle against what the definition and plain mathematics fix.

Expected values come from elsewhere than the oracle's own formulas: operands
built from integer (significand, exponent) pairs with Python integers, exact
rational sums (``fractions.Fraction``) rounded to fp32 by searching float32
neighbours, closed forms (identity, all-ones, small integers), and the
transpose symmetry. The last test plants mistakes in copies of the oracle and
checks that a pin catches each.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import tf32_oracle as tf


def make_fp32(sig24: np.ndarray, exp: np.ndarray, neg: np.ndarray) -> np.ndarray:
    """fp32 values (-1)^neg * sig24 * 2^exp for 24-bit integer significands
    (2^23 <= sig24 < 2^24), built with exact integer scaling."""
    out = np.empty(sig24.shape, dtype=np.float32)
    for idx in np.ndindex(sig24.shape):
        v = math.ldexp(int(sig24[idx]), int(exp[idx]))
        out[idx] = -v if neg[idx] else v
    return out


def expected_trunc(sig24, exp, neg):
    """The tf32 value: the significand's low 13 bits dropped (integers only)."""
    return make_fp32((sig24 >> 13) << 13, exp, neg)


def random_operands(shape, rng, emin=-30, emax=-20):
    sig = rng.integers(1 << 23, 1 << 24, size=shape, dtype=np.int64)
    exp = rng.integers(emin, emax, size=shape)
    neg = rng.integers(0, 2, size=shape).astype(bool)
    return sig, exp, neg


def nearest_fp32(s: Fraction) -> np.float32:
    """Round an exact rational to the nearest fp32 (ties to an even significand)
    by comparing it with float32 neighbours exactly."""
    if s == 0:
        return np.float32(0.0)
    guess = np.float32(float(s))
    cands = {guess, np.nextafter(guess, np.float32(np.inf)), np.nextafter(guess, np.float32(-np.inf))}
    best = None
    for c in cands:
        d = abs(Fraction(float(c)) - s)
        key = (d, int(np.array(c, dtype=np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return np.float32(best[1])


# ---------------------------------------------------------------------------
def test_trunc_matches_integer_construction():
    rng = np.random.default_rng(1)
    sig, exp, neg = random_operands((4000,), rng, -140, 100)
    x = make_fp32(sig, exp, neg)
    want = expected_trunc(sig, exp, neg)
    assert np.array_equal(tf.trunc_tf32(x).view(np.uint32), want.view(np.uint32))


def test_trunc_low_bits_are_dropped_not_rounded():
    one_plus = np.float32(1 + 2.0 ** -11 + 2.0 ** -12)   # rounds up to 1 + 2^-10 at 10 bits
    keep = np.float32(1 + 2.0 ** -10)
    got = tf.trunc_tf32(np.array([one_plus, keep, -one_plus], dtype=np.float32))
    assert got.tolist() == [1.0, float(keep), -1.0]
    C = tf.gemm(np.array([[one_plus]], dtype=np.float32), np.array([[np.float32(3.0)]], dtype=np.float32))
    assert C[0, 0] == np.float32(3.0)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 4), (3, 2, 7), (5, 4, 3), (4, 6, 9)])
def test_brute_force_exact_rationals(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    sa, ea, na = random_operands((M, K), rng)
    sb, eb, nb = random_operands((K, N), rng)
    A = make_fp32(sa, ea, na)
    B = make_fp32(sb, eb, nb)
    At = expected_trunc(sa, ea, na)
    Bt = expected_trunc(sb, eb, nb)
    got = tf.gemm(A, B)
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(float(At[i, k])) * Fraction(float(Bt[k, j])) for k in range(K))
            assert got[i, j] == nearest_fp32(s), (i, j)


def test_identity_and_orientation():
    rng = np.random.default_rng(3)
    B = rng.standard_normal((6, 5)).astype(np.float32)
    assert np.array_equal(tf.gemm(np.eye(6, dtype=np.float32), B), tf.trunc_tf32(B))
    A = rng.standard_normal((4, 6)).astype(np.float32)
    assert np.array_equal(tf.gemm(A, np.eye(6, dtype=np.float32)), tf.trunc_tf32(A))
    # a unit row picks a row of B, a unit column a column of A
    e = np.zeros((1, 6), dtype=np.float32)
    e[0, 2] = 1
    assert np.array_equal(tf.gemm(e, B)[0], tf.trunc_tf32(B)[2])


def test_all_ones_and_small_integers():
    K = 3000
    C = tf.gemm(np.ones((3, K), np.float32), np.ones((K, 2), np.float32))
    assert np.all(C == K)
    rng = np.random.default_rng(4)
    Ai = rng.integers(-7, 8, size=(9, 50))
    Bi = rng.integers(-7, 8, size=(50, 11))
    assert np.array_equal(tf.gemm(Ai.astype(np.float32), Bi.astype(np.float32)), (Ai @ Bi).astype(np.float32))


def test_transpose_symmetry():
    rng = np.random.default_rng(5)
    A = rng.standard_normal((7, 13)).astype(np.float32)
    B = rng.standard_normal((13, 5)).astype(np.float32)
    assert np.array_equal(tf.gemm(B.T.copy(), A.T.copy()), tf.gemm(A, B).T)


def test_degenerate_shapes():
    assert tf.gemm(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32)).tolist() == [[0.0] * 4] * 3
    assert tf.gemm(np.zeros((0, 5), np.float32), np.zeros((5, 2), np.float32)).shape == (0, 2)


def test_tolerance_covers_a_sequential_fp32_sum():
    # an fp32 left-to-right accumulation of the exact products stays inside
    # the bound, and the bound is not vacuous (far below |C|)
    rng = np.random.default_rng(6)
    M, N, K = 16, 16, 2048
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    At = tf.trunc_tf32(A)
    Bt = tf.trunc_tf32(B)
    acc = np.zeros((M, N), np.float32)
    for k in range(K):
        acc = (acc + np.outer(At[:, k], Bt[k, :]).astype(np.float32)).astype(np.float32)
    ref = tf.gemm(A, B)
    S = tf.abs_gemm(A, B)
    tol = tf.tolerance(S, ref, K)
    assert np.all(np.abs(acc.astype(np.float64) - ref) <= tol)
    assert np.median(tol / np.maximum(np.abs(ref), 1e-30)) < 0.05


# ---------------------------------------------------------------------------
# Planted mistakes: each broken copy must fail at least one pin above.

def _round_tf32(x):
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bits = (bits + (1 << 12)) & ~np.uint64((1 << 13) - 1)
    return bits.astype(np.uint32).view(np.float32)


BROKEN = {
    "rounds_instead_of_truncating": lambda A, B: (_round_tf32(A).astype(np.float64) @
                                                  _round_tf32(B).astype(np.float64)).astype(np.float32),
    "no_truncation": lambda A, B: (A.astype(np.float64) @ B.astype(np.float64)).astype(np.float32),
    # B read column-major (element (k, j) taken from offset j*K + k)
    "transposed_b": lambda A, B: (tf.trunc_tf32(A).astype(np.float64) @
                                  tf.trunc_tf32(np.ascontiguousarray(B.T).reshape(B.shape)).astype(np.float64)
                                  ).astype(np.float32),
    "drops_last_k": lambda A, B: (tf.trunc_tf32(A[:, :-1]).astype(np.float64) @
                                  tf.trunc_tf32(B[:-1]).astype(np.float64)).astype(np.float32),
}


def _pins_pass(gemm):
    rng = np.random.default_rng(7)
    try:
        # truncation pin
        one_plus = np.float32(1 + 2.0 ** -11 + 2.0 ** -12)
        if gemm(np.array([[one_plus]], np.float32), np.array([[np.float32(3.0)]], np.float32))[0, 0] != 3.0:
            return False
        # brute-force pin
        sa, ea, na = random_operands((3, 4), rng)
        sb, eb, nb = random_operands((4, 3), rng)
        A, B = make_fp32(sa, ea, na), make_fp32(sb, eb, nb)
        At, Bt = expected_trunc(sa, ea, na), expected_trunc(sb, eb, nb)
        got = gemm(A, B)
        for i in range(3):
            for j in range(3):
                s = sum(Fraction(float(At[i, k])) * Fraction(float(Bt[k, j])) for k in range(4))
                if got[i, j] != nearest_fp32(s):
                    return False
        # all-ones pin
        if not np.all(gemm(np.ones((2, 300), np.float32), np.ones((300, 2), np.float32)) == 300):
            return False
    except Exception:
        return False
    return True


def test_pins_pass_for_the_oracle():
    assert _pins_pass(tf.gemm)


@pytest.mark.parametrize("broken", sorted(BROKEN))
def test_pins_catch_planted_mistakes(broken):
    assert not _pins_pass(BROKEN[broken])
