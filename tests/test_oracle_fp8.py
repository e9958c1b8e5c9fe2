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


# ---------------------------------------------------------------------------
# Block-scaled variant: one fp32 factor per bs x bs sub-block of A and of B.

def _block_scales(rows, cols, bs, rng, pow2=False):
    shape = f8.scale_grid(rows, cols, bs)
    if pow2:
        return np.ldexp(1.0, rng.integers(-3, 4, size=shape)).astype(np.float32)
    return rng.uniform(0.05, 4.0, size=shape).astype(np.float32)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("bs,M,N,K", [(32, 33, 35, 70), (32, 5, 64, 96), (64, 65, 66, 130), (64, 3, 2, 64)])
def test_blockscaled_brute_force_exact_rationals(fmt, bs, M, N, K):
    # every element as an exact rational sum over k of value(A[i,k]) value(B[k,j]),
    # each value decoded by PyTorch and scaled by its own sub-block's factor
    # (index arithmetic written here per element), rounded to bf16 by search
    rng = np.random.default_rng(bs + M + N + K)
    A = random_fp8((M, K), fmt, rng)
    B = random_fp8((K, N), fmt, rng)
    sa = _block_scales(M, K, bs, rng)
    sb = _block_scales(K, N, bs, rng)
    dA, dB = lib_decode(fmt)[A], lib_decode(fmt)[B]
    fa = [[Fraction(float(dA[i, k])) * Fraction(float(sa[i // bs, k // bs])) for k in range(K)] for i in range(M)]
    fb = [[Fraction(float(dB[k, j])) * Fraction(float(sb[k // bs, j // bs])) for j in range(N)] for k in range(K)]
    got = f8.gemm_blockscaled(A, B, fmt, sa, sb, bs)
    for i in range(M):
        for j in range(N):
            s = sum(fa[i][k] * fb[k][j] for k in range(K))
            assert int(got[i, j]) == nearest_bf16(s), (i, j)


@pytest.mark.parametrize("bs", [32, 64])
def test_blockscaled_constant_along_k_is_the_per_channel_product(bs):
    # scales that do not vary along K factor out of the sum: the result is the
    # (separately pinned) per-channel product with row factor a[i // bs] and
    # column factor b[j // bs]; power-of-two factors keep both exact in fp64
    rng = np.random.default_rng(bs)
    M, N, K = 150, 140, 3 * bs + 5
    A = random_fp8((M, K), "e4m3", rng)
    B = random_fp8((K, N), "e4m3", rng)
    ra = np.ldexp(1.0, rng.integers(-4, 5, size=-(-M // bs))).astype(np.float32)
    cb = np.ldexp(1.0, rng.integers(-4, 5, size=-(-N // bs))).astype(np.float32)
    sa = np.repeat(ra[:, None], -(-K // bs), axis=1)
    sb = np.repeat(cb[None, :], -(-K // bs), axis=0)
    want = f8.gemm(A, B, "e4m3", ra[np.arange(M) // bs], cb[np.arange(N) // bs])
    assert np.array_equal(f8.gemm_blockscaled(A, B, "e4m3", sa, sb, bs), want)
    # all ones: exactly the unscaled product
    ones_a = np.ones(f8.scale_grid(M, K, bs), np.float32)
    ones_b = np.ones(f8.scale_grid(K, N, bs), np.float32)
    assert np.array_equal(f8.gemm_blockscaled(A, B, "e4m3", ones_a, ones_b, bs), f8.gemm(A, B, "e4m3"))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("bs", [32, 64])
def test_blockscaled_is_the_sum_of_scaled_k_slices(fmt, bs):
    # C = sum over K blocks kb of (a_scale[:, kb] (x) b_scale[kb, :]) * the
    # unscaled product of the kb-th K slice (the per-channel oracle with unit
    # scales); power-of-two scales keep every step exact in fp64
    rng = np.random.default_rng(7 * bs)
    M, N, K = 2 * bs + 3, bs + 9, 4 * bs - 7
    A = random_fp8((M, K), fmt, rng)
    B = random_fp8((K, N), fmt, rng)
    sa = _block_scales(M, K, bs, rng, pow2=True)
    sb = _block_scales(K, N, bs, rng, pow2=True)
    rows = np.arange(M) // bs
    cols = np.arange(N) // bs
    want = np.zeros((M, N))
    for kb in range(-(-K // bs)):
        k0, k1 = kb * bs, min(K, (kb + 1) * bs)
        part = f8.gemm_f64(A[:, k0:k1], B[k0:k1, :], fmt)
        want += part * np.outer(sa[rows, kb].astype(np.float64), sb[kb, cols].astype(np.float64))
    assert np.array_equal(f8.gemm_blockscaled_f64(A, B, fmt, sa, sb, bs), want)


@pytest.mark.parametrize("bs", [32, 64])
def test_blockscaled_transpose_symmetry(bs):
    # (A B)^T = B^T A^T: the transposed operands carry transposed scale grids
    rng = np.random.default_rng(11 + bs)
    M, N, K = 70, 45, 100
    A = random_fp8((M, K), "e5m2", rng)
    B = random_fp8((K, N), "e5m2", rng)
    sa = _block_scales(M, K, bs, rng)
    sb = _block_scales(K, N, bs, rng)
    got = f8.gemm_blockscaled(B.T.copy(), A.T.copy(), "e5m2", sb.T.copy(), sa.T.copy(), bs)
    assert np.array_equal(got, f8.gemm_blockscaled(A, B, "e5m2", sa, sb, bs).T)


def test_blockscaled_rejects_wrong_scale_grids():
    A = np.zeros((40, 70), np.uint8)
    B = np.zeros((70, 33), np.uint8)
    with pytest.raises(ValueError):
        f8.gemm_blockscaled(A, B, "e4m3", np.ones((2, 2), np.float32), np.ones((3, 2), np.float32), 32)
    with pytest.raises(ValueError):
        f8.gemm_blockscaled(A, B, "e4m3", np.ones((2, 3), np.float32), np.ones((3, 2), np.float32), 16)
    assert f8.gemm_blockscaled(A, B, "e4m3", np.ones((2, 3), np.float32),
                               np.ones((3, 2), np.float32), 32).shape == (40, 33)


def test_blockscaled_tolerance_covers_a_blockwise_fp32_accumulation():
    # a GPU-like evaluation: each K block's products summed in fp32, its factor
    # a_scale * b_scale formed in fp32 and added into an fp32 accumulator by a
    # fused multiply-add, then one rounding to bf16
    rng = np.random.default_rng(5)
    fmt, bs = "e4m3", 32
    M, N, K = 8, 8, 512
    A = random_fp8((M, K), fmt, rng)
    B = random_fp8((K, N), fmt, rng)
    sa = _block_scales(M, K, bs, rng)
    sb = _block_scales(K, N, bs, rng)
    dA = lib_decode(fmt)[A].astype(np.float32)
    dB = lib_decode(fmt)[B].astype(np.float32)
    acc = np.zeros((M, N), np.float32)
    for kb in range(K // bs):
        part = np.zeros((M, N), np.float32)
        for k in range(kb * bs, (kb + 1) * bs):
            part = (part + np.outer(dA[:, k], dB[k]).astype(np.float32)).astype(np.float32)
        s = (sa[np.arange(M) // bs, kb][:, None] * sb[kb, np.arange(N) // bs][None, :]).astype(np.float32)
        acc = (acc.astype(np.float64) + s.astype(np.float64) * part.astype(np.float64)).astype(np.float32)
    gpu_like = torch.from_numpy(acc).to(torch.bfloat16).to(torch.float64).numpy()
    c64 = f8.gemm_blockscaled_f64(A, B, fmt, sa, sb, bs)
    ref = torch.from_numpy(f8.gemm_blockscaled(A, B, fmt, sa, sb, bs).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()
    tol = f8.tolerance_blockscaled(f8.abs_gemm_blockscaled(A, B, fmt, sa, sb, bs), c64, K, bs)
    assert np.all(np.abs(gpu_like - ref) <= tol)


# Planted mistakes in the block-scaled oracle: each broken copy must fail a pin.

def _make_bs(a_index=None, b_index=None, k_once=False, block_override=None):
    def gemm(A, B, fmt, sa, sb, bs):
        eff = block_override or bs
        M, K = A.shape
        N = B.shape[1]
        sa = np.asarray(sa, np.float64)
        sb = np.asarray(sb, np.float64)
        i = np.arange(M)
        k = np.arange(K)
        j = np.arange(N)
        ia, ka = (a_index or (lambda i, k, b: (i // b, k // b)))(i[:, None], k[None, :], eff)
        kb_, jb = (b_index or (lambda k, j, b: (k // b, j // b)))(k[:, None], j[None, :], eff)
        if k_once:
            ka = np.zeros_like(ka)
            kb_ = np.zeros_like(kb_)
        ia = np.clip(ia, 0, sa.shape[0] - 1)
        ka = np.clip(ka, 0, sa.shape[1] - 1)
        kb_ = np.clip(kb_, 0, sb.shape[0] - 1)
        jb = np.clip(jb, 0, sb.shape[1] - 1)
        a = f8.decode(A, fmt) * sa[ia, ka]
        b = f8.decode(B, fmt) * sb[kb_, jb]
        return f8.round_rne(a @ b, "bf16")
    return gemm


BROKEN_BS = {
    # A's factor looked up with the block indices swapped
    "a_index_swapped": _make_bs(a_index=lambda i, k, b: (k // b, i // b)),
    # B's factor taken by (column block, K block)
    "b_index_swapped": _make_bs(b_index=lambda k, j, b: (j // b, k // b)),
    # the first K block's factors used for the whole sum (per channel)
    "k_block_ignored": _make_bs(k_once=True),
    # the other block size of the page
    "wrong_block_size": _make_bs(block_override=16),
    # the factor of the block one row further down
    "row_block_off_by_one": _make_bs(a_index=lambda i, k, b: ((i + 1) // b, k // b)),
}


def _bs_pins_pass(gemm):
    try:
        for fmt in FMTS:
            for bs, (M, N, K) in ((32, (35, 34, 70)), (64, (66, 67, 130))):
                rng = np.random.default_rng(bs + K)
                A = random_fp8((M, K), fmt, rng)
                B = random_fp8((K, N), fmt, rng)
                sa = _block_scales(M, K, bs, rng)
                sb = _block_scales(K, N, bs, rng)
                dA, dB = lib_decode(fmt)[A], lib_decode(fmt)[B]
                got = gemm(A, B, fmt, sa, sb, bs)
                for (i, j) in ((0, 0), (M - 1, N - 1), (bs, bs - 1), (bs - 1, bs), (M // 2, N // 3)):
                    s = sum(Fraction(float(dA[i, k])) * Fraction(float(sa[i // bs, k // bs])) *
                            Fraction(float(dB[k, j])) * Fraction(float(sb[k // bs, j // bs])) for k in range(K))
                    if int(got[i, j]) != nearest_bf16(s):
                        return False
    except Exception:
        return False
    return True


def test_blockscaled_pins_pass_for_the_oracle():
    assert _bs_pins_pass(f8.gemm_blockscaled)


@pytest.mark.parametrize("broken", sorted(BROKEN_BS))
def test_blockscaled_pins_catch_planted_mistakes(broken):
    assert not _bs_pins_pass(BROKEN_BS[broken])
