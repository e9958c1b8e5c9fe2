"""Pins for the FP8 oracle against what the definitions and plain mathematics fix.

Expected values come from elsewhere than the oracle's formulas: PyTorch's own
float8 types decode every bit pattern (an independent library), exact rational
sums (``fractions.Fraction``) rounded to bf16 by searching PyTorch's bf16
values, closed forms (all-ones, powers-of-two scales) and the transpose
symmetry. The last test plants mistakes in copies of the oracle and checks
that a pin catches each.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp8_oracle as f8

TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
FMTS = sorted(TORCH_FP8)


def lib_decode(fmt):
    pats = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return pats.view(TORCH_FP8[fmt]).to(torch.float64).numpy()


def random_fp8(shape, fmt, rng, lo=-4.0, hi=4.0):
    """Finite fp8 patterns: uniform values quantised by PyTorch, as uint8."""
    x = torch.from_numpy(rng.uniform(lo, hi, size=shape).astype(np.float32))
    return x.to(TORCH_FP8[fmt]).view(torch.uint8).numpy()


def nearest_bf16(s: Fraction) -> int:
    """bf16 pattern nearest to an exact rational (ties to an even pattern), by
    comparing it with PyTorch bf16 neighbours exactly."""
    if s == 0:
        return 0
    g = torch.tensor(float(s), dtype=torch.float64).to(torch.bfloat16)
    bits = int(g.view(torch.int16).item()) & 0xFFFF
    cands = {bits, (bits + 1) & 0xFFFF, (bits - 1) & 0xFFFF}
    best = None
    for c in cands:
        v = torch.tensor([c], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).to(torch.float64).item()
        if not np.isfinite(v):
            continue
        key = (abs(Fraction(v) - s), c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", FMTS)
def test_decode_exhaustive_against_torch(fmt):
    got = f8.decode(np.arange(256, dtype=np.uint8), fmt)
    want = lib_decode(fmt)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_format_landmarks():
    # E4M3: largest finite 448, no infinity (0x7F is NaN); E5M2: 0x7C is +inf
    assert f8.decode(np.array([0x7E], np.uint8), "e4m3")[0] == 448.0
    assert np.isnan(f8.decode(np.array([0x7F], np.uint8), "e4m3")[0])
    assert f8.decode(np.array([0x7C], np.uint8), "e5m2")[0] == np.inf
    assert f8.decode(np.array([0x7B], np.uint8), "e5m2")[0] == 57344.0
    # smallest subnormals
    assert f8.decode(np.array([0x01], np.uint8), "e4m3")[0] == 2.0 ** -9
    assert f8.decode(np.array([0x01], np.uint8), "e5m2")[0] == 2.0 ** -16


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 5), (4, 2, 9), (3, 3, 16)])
def test_brute_force_exact_rationals(fmt, M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A = random_fp8((M, K), fmt, rng)
    B = random_fp8((K, N), fmt, rng)
    sa = rng.uniform(0.1, 3, M).astype(np.float32)
    sb = rng.uniform(0.1, 3, N).astype(np.float32)
    dA, dB = lib_decode(fmt)[A], lib_decode(fmt)[B]
    got = f8.gemm(A, B, fmt, sa, sb)
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(float(dA[i, k])) * Fraction(float(dB[k, j])) for k in range(K))
            s *= Fraction(float(sa[i])) * Fraction(float(sb[j]))
            assert int(got[i, j]) == nearest_bf16(s), (i, j)


@pytest.mark.parametrize("fmt", FMTS)
def test_all_ones_and_power_of_two_scales(fmt):
    one = {"e4m3": 0x38, "e5m2": 0x3C}[fmt]
    K = 200
    A = np.full((3, K), one, np.uint8)
    B = np.full((K, 4), one, np.uint8)
    c = f8.gemm_f64(A, B, fmt)
    assert np.all(c == K)
    sa = np.array([1, 2, 0.25], np.float32)
    sb = np.array([1, 4, 0.5, 8], np.float32)
    assert np.array_equal(f8.gemm_f64(A, B, fmt, sa, sb), K * np.outer(sa, sb).astype(np.float64))


@pytest.mark.parametrize("fmt", FMTS)
def test_transpose_symmetry(fmt):
    rng = np.random.default_rng(3)
    A = random_fp8((5, 11), fmt, rng)
    B = random_fp8((11, 7), fmt, rng)
    sa = rng.uniform(0.5, 2, 5).astype(np.float32)
    sb = rng.uniform(0.5, 2, 7).astype(np.float32)
    assert np.array_equal(f8.gemm(B.T.copy(), A.T.copy(), fmt, sb, sa), f8.gemm(A, B, fmt, sa, sb).T)


def test_tolerance_covers_an_fp32_accumulation():
    rng = np.random.default_rng(4)
    fmt = "e4m3"
    M, N, K = 8, 8, 1024
    A = random_fp8((M, K), fmt, rng)
    B = random_fp8((K, N), fmt, rng)
    sa = rng.uniform(0.01, 0.1, M).astype(np.float32)
    sb = rng.uniform(0.01, 0.1, N).astype(np.float32)
    dA = lib_decode(fmt)[A].astype(np.float32)
    dB = lib_decode(fmt)[B].astype(np.float32)
    acc = np.zeros((M, N), np.float32)
    for k in range(K):
        acc = (acc + np.outer(dA[:, k], dB[k]).astype(np.float32)).astype(np.float32)
    v = (acc * (sa[:, None] * sb[None, :]).astype(np.float32)).astype(np.float32)
    gpu_like = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    c64 = f8.gemm_f64(A, B, fmt, sa, sb)
    ref = torch.from_numpy(f8.gemm(A, B, fmt, sa, sb).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    tol = f8.tolerance(f8.abs_gemm(A, B, fmt, sa, sb), c64, K)
    assert np.all(np.abs(gpu_like - ref) <= tol)


# ---------------------------------------------------------------------------
# Planted mistakes: each broken copy must fail at least one pin above.

def _bad_decode_bias(b, fmt):
    v = f8.decode(b, fmt)
    return v * 0.5 if fmt == "e4m3" else v


def _bad_decode_e4m3_inf(b, fmt):
    v = f8.decode(b, fmt)
    if fmt == "e4m3":
        x = np.asarray(b).astype(np.int64)
        v = np.where((x & 0x7F) == 0x78, np.where(x & 0x80, -np.inf, np.inf), v)
    return v


def _make(decode=None, swap_scales=False, drop_b_scale=False):
    dec = decode or f8.decode

    def gemm(A, B, fmt, a_scale=None, b_scale=None):
        M, N = A.shape[0], B.shape[1]
        sa = np.ones(M) if a_scale is None else np.asarray(a_scale, np.float64)
        sb = np.ones(N) if b_scale is None else np.asarray(b_scale, np.float64)
        c = dec(A, fmt) @ dec(B, fmt)
        if swap_scales and M == N:
            c = c * sa[None, :] * sb[:, None]
        elif swap_scales:
            c = c * sa.mean() * sb.mean()
        else:
            c = c * sa[:, None] * (1.0 if drop_b_scale else sb[None, :])
        return f8.round_rne(c, "bf16")
    return gemm


BROKEN = {
    "e4m3_bias_8": _make(decode=_bad_decode_bias),
    "e4m3_with_infinity": _make(decode=_bad_decode_e4m3_inf),
    "scales_swapped": _make(swap_scales=True),
    "b_scale_dropped": _make(drop_b_scale=True),
}


def _bf16_value(bits) -> float:
    return torch.tensor([int(bits)], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).item()


def _pins_pass(gemm):
    try:
        for fmt in FMTS:
            # decode pin through a 1 x 1 product with unit scales
            pats = np.arange(256, dtype=np.uint8)
            want = lib_decode(fmt)
            one = np.array([[{"e4m3": 0x38, "e5m2": 0x3C}[fmt]]], np.uint8)
            for p in pats:
                if np.isnan(want[p]):
                    continue
                got = gemm(np.array([[p]], np.uint8), one, fmt)[0, 0]
                # compare values (a zero's sign is not part of the pin)
                if _bf16_value(got) != _bf16_value(f8.round_rne(np.array([want[p]]), "bf16")[0]):
                    return False
            # brute force with scales
            rng = np.random.default_rng(11)
            A = random_fp8((3, 4), fmt, rng)
            B = random_fp8((4, 2), fmt, rng)
            sa = rng.uniform(0.1, 3, 3).astype(np.float32)
            sb = rng.uniform(0.1, 3, 2).astype(np.float32)
            got = gemm(A, B, fmt, sa, sb)
            dA, dB = lib_decode(fmt)[A], lib_decode(fmt)[B]
            for i in range(3):
                for j in range(2):
                    s = sum(Fraction(float(dA[i, k])) * Fraction(float(dB[k, j])) for k in range(4))
                    s *= Fraction(float(sa[i])) * Fraction(float(sb[j]))
                    if int(got[i, j]) != nearest_bf16(s):
                        return False
    except Exception:
        return False
    return True


def test_pins_pass_for_the_oracle():
    assert _pins_pass(f8.gemm)


@pytest.mark.parametrize("broken", sorted(BROKEN))
def test_pins_catch_planted_mistakes(broken):
    assert not _pins_pass(BROKEN[broken])
