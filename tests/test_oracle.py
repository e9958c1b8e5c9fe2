"""Pins for the CPU oracle against what the pages and plain mathematics fix.

None of these re-types the oracle's formulas. Each pin takes its expected value
from somewhere else: exact rational arithmetic (``fractions.Fraction``), an
independent library conversion (numpy's binary16, PyTorch's bfloat16), integer
matrix products, closed forms (identity, all-ones), a symmetry of the product
(transpose), or numbers printed on the pages (``tests/golden``). The last
section plants mistakes in copies of the oracle and checks that the pins catch
each one.
"""

import bisect
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from half_precision_dense_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DTYPES = ["f16", "bf16"]


# ---------------------------------------------------------------------------
# Independent references: library decodes of every 16-bit pattern.

def lib_decode_all(dtype):
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    if dtype == "f16":
        return allbits, allbits.view(np.float16).astype(np.float64)
    t = torch.from_numpy(allbits.view(np.int16).copy()).view(torch.bfloat16)
    return allbits, t.to(torch.float64).numpy()


_TABLES = {}


def rational_table(dtype):
    """Sorted non-negative finite values (as Fractions) with their bit patterns."""
    if dtype not in _TABLES:
        b, v = lib_decode_all(dtype)
        keep = np.isfinite(v) & ~np.signbit(v)
        pairs = sorted((Fraction(float(x)), int(bb)) for x, bb in zip(v[keep], b[keep]))
        vals = [p[0] for p in pairs]
        pats = [p[1] for p in pairs]
        _TABLES[dtype] = (vals, pats)
    return _TABLES[dtype]


def rne_by_search(s: Fraction, dtype):
    """Round an exact rational to the nearest representable value (ties to even
    pattern), by searching the library's own table of values."""
    vals, pats = rational_table(dtype)
    sign = 0x8000 if s < 0 else 0
    a = -s if s < 0 else s
    top = vals[-1]
    half_gap_top = (vals[-1] - vals[-2]) / 2
    if a >= top + half_gap_top:
        inf = 0x7C00 if dtype == "f16" else 0x7F80
        return inf | sign
    i = bisect.bisect_left(vals, a)
    if i < len(vals) and vals[i] == a:
        return pats[i] | sign
    lo, hi = vals[i - 1], vals[i]
    dl, dh = a - lo, hi - a
    if dl < dh:
        pick = pats[i - 1]
    elif dh < dl:
        pick = pats[i]
    else:
        pick = pats[i - 1] if pats[i - 1] % 2 == 0 else pats[i]
    return pick | sign


def lib_values(bits16, dtype):
    b, v = lib_decode_all(dtype)
    return v[bits16.astype(np.int64)]


def random_operands(rng, M, N, K, dtype, scale=1.0):
    A = torch.from_numpy((rng.uniform(-1, 1, (M, K)) * scale).astype(np.float32))
    B = torch.from_numpy((rng.uniform(-1, 1, (K, N)) * scale).astype(np.float32))
    t = inputs.TORCH_DTYPES[dtype]
    return inputs.bits(A.to(t)), inputs.bits(B.to(t))


# ---------------------------------------------------------------------------
# Pins, written as functions of the oracle so the mutation tests can reuse them.

def pin_brute_force(gemm, dtype, seed=0, trials=40):
    """Every output equals the exact rational sum rounded once, on tiny shapes."""
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        M, N, K = (int(v) for v in rng.integers(1, 8, size=3))
        A, B = random_operands(rng, M, N, K, dtype, scale=float(rng.choice([1.0, 8.0, 1e-3])))
        av = lib_values(A, dtype)
        bv = lib_values(B, dtype)
        got = gemm(A, B, dtype)
        for i in range(M):
            for j in range(N):
                s = sum((Fraction(float(av[i, k])) * Fraction(float(bv[k, j])) for k in range(K)),
                        Fraction(0))
                want = rne_by_search(s, dtype)
                if int(got[i, j]) != want:
                    return False
    return True


def pin_identity(gemm, dtype):
    """I.B = B and A.I = A for square identity operands."""
    rng = np.random.default_rng(1)
    for M, N in [(5, 7), (16, 3), (33, 65)]:
        A, B = random_operands(rng, M, N, M, dtype)             # A: M x M, B: M x N
        eye = inputs.bits(torch.eye(M, dtype=inputs.TORCH_DTYPES[dtype]))
        if not np.array_equal(gemm(eye, B, dtype), B):
            return False
        if not np.array_equal(gemm(A, eye, dtype), A):
            return False
    return True


def pin_right_identity(gemm, dtype):
    rng = np.random.default_rng(2)
    M, K = 9, 12
    A, _ = random_operands(rng, M, 1, K, dtype)
    eye = inputs.bits(torch.eye(K, dtype=inputs.TORCH_DTYPES[dtype]))
    return np.array_equal(gemm(A, eye, dtype), A)                 # A . I = A


def pin_all_ones(gemm, dtype):
    """C = K for all-ones operands; exact while K is representable (2^(p+1))."""
    one = 0x3C00 if dtype == "f16" else 0x3F80
    limit = 2048 if dtype == "f16" else 256
    for K in [1, 2, 3, 64, 255, limit]:
        A = np.full((3, K), one, dtype=np.uint16)
        B = np.full((K, 4), one, dtype=np.uint16)
        c = lib_values(gemm(A, B, dtype), dtype)
        if not np.all(c == K):
            return False
    return True


def pin_small_integers(gemm, dtype):
    """Small-integer operands: products and sums are exact; compare with an
    integer matrix product."""
    rng = np.random.default_rng(3)
    t = inputs.TORCH_DTYPES[dtype]
    for M, N, K in [(7, 9, 11), (32, 17, 20), (64, 64, 28)]:
        Ai = rng.integers(-3, 4, (M, K))
        Bi = rng.integers(-3, 4, (K, N))
        A = inputs.bits(torch.from_numpy(Ai.astype(np.float32)).to(t))
        B = inputs.bits(torch.from_numpy(Bi.astype(np.float32)).to(t))
        want = Ai @ Bi                       # |C| <= 9K <= 252: exact in bf16 and f16
        got = lib_values(gemm(A, B, dtype), dtype)
        if not np.array_equal(got, want.astype(np.float64)):
            return False
    return True


def pin_transpose(gemm, dtype):
    """(A.B)^T = B^T.A^T, bit for bit."""
    rng = np.random.default_rng(4)
    for M, N, K in [(13, 29, 31), (64, 48, 80)]:
        A, B = random_operands(rng, M, N, K, dtype)
        c1 = gemm(A, B, dtype)
        c2 = gemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T), dtype)
        if not np.array_equal(c1.T, c2):
            return False
    return True


def pin_rectangular_orientation(gemm, dtype):
    """Row i of A and column j of B meet in C[i][j] (no operand transposed):
    A = e_r (a unit row) picks row r of B; B = e_c picks column c of A."""
    rng = np.random.default_rng(5)
    M, N, K = 6, 10, 8
    A, B = random_operands(rng, M, N, K, dtype)
    one = 0x3C00 if dtype == "f16" else 0x3F80
    for r in [0, 3, K - 1]:
        e = np.zeros((1, K), dtype=np.uint16)
        e[0, r] = one
        if not np.array_equal(gemm(e, B, dtype)[0], B[r]):
            return False
    for c in [0, 5, K - 1]:
        e = np.zeros((K, 1), dtype=np.uint16)
        e[c, 0] = one
        if not np.array_equal(gemm(A, e, dtype)[:, 0], A[:, c]):
            return False
    return True


PINS = [pin_brute_force, pin_identity, pin_right_identity, pin_all_ones,
        pin_small_integers, pin_transpose, pin_rectangular_orientation]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pins(pin, dtype):
    assert pin(oracle.gemm, dtype)


# ---------------------------------------------------------------------------
# The 16-bit codecs against independent library conversions.

@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_exhaustive(dtype):
    b, want = lib_decode_all(dtype)
    got = oracle.decode(b, dtype)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(want[~np.isnan(want)]))


def test_round_f16_matches_numpy_binary16():
    rng = np.random.default_rng(10)
    mags = np.exp2(rng.uniform(-30, 18, 400000))
    x = mags * rng.choice([-1.0, 1.0], mags.size)
    # exact ties and near-ties around every binade
    b, v = lib_decode_all("f16")
    fin = v[np.isfinite(v)]
    fin = np.unique(fin)
    mids = (fin[:-1] + fin[1:]) / 2
    x = np.concatenate([x, fin, mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf),
                        [0.0, -0.0, np.inf, -np.inf, 65504.0, 65519.99, 65520.0, 1e10,
                         2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -26]])
    got = oracle.round_rne(x, "f16")
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_round_bf16_matches_torch_from_fp32():
    rng = np.random.default_rng(11)
    raw = rng.integers(0, 1 << 32, 1 << 20, dtype=np.uint64).astype(np.uint32)
    f32 = raw.view(np.float32)
    f32 = f32[np.isfinite(f32)]
    edge = np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 3.4e38, 1e-45, 1e-40,
                     1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 - 2.0 ** -24], dtype=np.float32)
    f32 = np.concatenate([f32, edge])
    want = inputs.bits(torch.from_numpy(f32.copy()).to(torch.bfloat16))
    got = oracle.round_rne(f32.astype(np.float64), "bf16")
    assert np.array_equal(got, want)


def test_round_specials():
    # ties to even: 1 + 2^-11 lies halfway between 1 and 1 + 2^-10 in f16
    assert oracle.round_rne(np.array([1 + 2.0 ** -11]), "f16")[0] == 0x3C00
    assert oracle.round_rne(np.array([1 + 3 * 2.0 ** -11]), "f16")[0] == 0x3C02
    # the largest finite values and the overflow thresholds
    assert oracle.round_rne(np.array([65504.0]), "f16")[0] == 0x7BFF
    assert oracle.round_rne(np.array([65520.0]), "f16")[0] == 0x7C00
    bf_max = (2 - 2.0 ** -7) * 2.0 ** 127
    assert oracle.round_rne(np.array([bf_max]), "bf16")[0] == 0x7F7F
    assert oracle.round_rne(np.array([(2 - 2.0 ** -8) * 2.0 ** 127]), "bf16")[0] == 0x7F80
    # gradual underflow
    assert oracle.round_rne(np.array([2.0 ** -24]), "f16")[0] == 0x0001
    assert oracle.round_rne(np.array([2.0 ** -25]), "f16")[0] == 0x0000
    assert oracle.round_rne(np.array([-(2.0 ** -133)]), "bf16")[0] == 0x8001
    # NaN stays NaN
    assert np.isnan(oracle.decode(oracle.round_rne(np.array([np.nan]), "bf16"), "bf16")[0])


def test_degenerate_shapes():
    A = np.zeros((3, 0), dtype=np.uint16)
    B = np.zeros((0, 5), dtype=np.uint16)
    assert np.array_equal(oracle.gemm(A, B, "bf16"), np.zeros((3, 5), dtype=np.uint16))
    assert oracle.gemm(np.zeros((0, 4), np.uint16), np.zeros((4, 2), np.uint16), "f16").shape == (0, 2)
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((2, 3), np.uint16), np.zeros((4, 2), np.uint16), "f16")


def test_rows_and_cols_agree_with_full():
    rng = np.random.default_rng(6)
    A, B = random_operands(rng, 40, 50, 60, "bf16")
    full = oracle.gemm(A, B, "bf16")
    rows = [0, 7, 39]
    cols = [1, 2, 49]
    assert np.array_equal(oracle.gemm_rows(A, B, "bf16", rows)[0], full[rows])
    assert np.array_equal(oracle.gemm_cols(A, B, "bf16", cols)[0], full[:, cols])


# ---------------------------------------------------------------------------
# Numbers printed on the pages.

def _golden_rows(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_page_benchmark_table_reproduces_flop_convention():
    rows = _golden_rows("hgemm_4096_benchmark.txt")
    flop = oracle.flops(4096, 4096, 4096)
    t_torch = float(rows[0][1])
    for name, ms, speedup, tflops in rows:
        t = float(ms)
        assert round(flop / (t * 1e-3) / 1e12, 2) == float(tflops), name
        if speedup != "-":
            assert round(t_torch / t, 2) == float(speedup), name


def test_page_flop_count_example():
    (M, N, K, gflop, peak, ms), = _golden_rows("flop_count_example.txt")
    f = oracle.flops(int(M), int(N), int(K))
    assert round(f / 1e9, 1) == float(gflop)
    assert round(f / (float(peak) * 1e12) * 1e3, 1) == float(ms)


# ---------------------------------------------------------------------------
# Planted mistakes: each broken copy of the oracle must fail at least one pin.

def _broken_transposed_b(A, B, dtype):
    B = np.asarray(B)
    Bt = np.ascontiguousarray(B.T) if B.shape[0] == B.shape[1] else B[::-1]
    return oracle.round_rne(oracle.decode(A, dtype) @ oracle.decode(Bt, dtype), dtype)


def _broken_dropped_term(A, B, dtype):
    A = np.asarray(A)
    B = np.asarray(B)
    if A.shape[1] <= 1:
        return oracle.gemm(A, B, dtype)
    return oracle.gemm(A[:, :-1], B[:-1, :], dtype)


def _broken_truncating_round(A, B, dtype):
    c = oracle.gemm_f64(A, B, dtype)
    f = oracle.FORMATS[dtype]
    with np.errstate(divide="ignore"):
        e = np.maximum(np.floor(np.log2(np.abs(np.where(c == 0, 1, c)))), f.emin)
    q = np.exp2(e - f.p)
    return oracle.round_rne(np.trunc(c / q) * q, dtype)


def _broken_sign(A, B, dtype):
    c = oracle.gemm_f64(A, B, dtype)
    return oracle.round_rne(np.abs(c), dtype)


def _broken_round_half_up(A, B, dtype):
    c = oracle.gemm_f64(A, B, dtype)
    f = oracle.FORMATS[dtype]
    with np.errstate(divide="ignore"):
        e = np.maximum(np.floor(np.log2(np.abs(np.where(c == 0, 1, c)))), f.emin)
    q = np.exp2(e - f.p)
    return oracle.round_rne(np.sign(c) * np.floor(np.abs(c) / q + 0.5) * q, dtype)


@pytest.mark.parametrize("broken", [_broken_transposed_b, _broken_dropped_term,
                                    _broken_truncating_round, _broken_sign,
                                    _broken_round_half_up], ids=lambda f: f.__name__)
def test_pins_catch_planted_mistakes(broken):
    caught = []
    for dtype in DTYPES:
        for pin in PINS:
            try:
                ok = pin(broken, dtype)
            except Exception:
                ok = False
            caught.append(not ok)
    assert any(caught), f"{broken.__name__} passed every pin"


def test_brute_force_table_is_consistent():
    # the search-based rounding agrees with the library on exact float inputs
    for dtype in DTYPES:
        b, v = lib_decode_all(dtype)
        for x in [1.0, 0.5, 3.0, 1e-3, 100.5]:
            r = rne_by_search(Fraction(x), dtype)
            assert r == int(oracle.round_rne(np.array([x]), dtype)[0])
        assert math.isinf(float(lib_values(np.array([rne_by_search(Fraction(10 ** 40), dtype)],
                                                    dtype=np.uint16), dtype)[0]))
