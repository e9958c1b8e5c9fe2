"""GPU parity of the block-scaled FP8 GEMM (hgemm_fp8_blockscaled) against the
CPU oracle (oracle.fp8_oracle.gemm_blockscaled): one fp32 factor per 32 x 32 or
64 x 64 sub-block of A and of B, bf16 C.

Inputs are the seeded generators' fp8 patterns (uniform over [-8, 8) rounded to
the format) and factors uniform in [0.5, 2); the bound per element is the
oracle's tolerance_blockscaled, and the relative Frobenius error must stay
under 5e-3 (bf16). Small-integer operands with power-of-two factors are exact
in every step, so there the GPU must match the oracle bit for bit."""

import numpy as np
import pytest
import torch

from half_precision_dense_gb300 import binding as hg
from half_precision_dense_gb300 import inputs
from oracle import fp8_oracle as f8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from half_precision_dense_gb300 import build as hbuild
    hbuild.build()
    hg.load_library()


def operands(M, N, K, fmt, bs, seed):
    A = inputs.generate_fp8((M, K), fmt, seed, 0, 8.0)
    B = inputs.generate_fp8((K, N), fmt, seed, 1, 8.0)
    ga, gb = f8.scale_grid(M, K, bs), f8.scale_grid(K, N, bs)
    sa = inputs.generate_scales(ga[0] * ga[1], seed, 2).reshape(ga)
    sb = inputs.generate_scales(gb[0] * gb[1], seed, 3).reshape(gb)
    return A, B, sa, sb


def run_gpu(A, B, sa, sb, fmt, bs, config=None, C_init=None):
    M, K = A.shape
    N = B.shape[1]
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dsa = torch.from_numpy(np.ascontiguousarray(sa)).cuda()
    dsb = torch.from_numpy(np.ascontiguousarray(sb)).cuda()
    C = torch.full((M, N), -7.0 if C_init is None else C_init, dtype=torch.bfloat16, device="cuda")
    hg.hgemm_fp8_blockscaled(dA, dB, C, dsa, dsb, M, N, K, bs, fmt, config)
    torch.cuda.synchronize()
    st, info = hg.get_device_status(0, reset=True)
    assert st == 0, (st, hex(info))
    return C.cpu()


def check(A, B, sa, sb, fmt, bs, config=None):
    K = A.shape[1]
    C = run_gpu(A, B, sa, sb, fmt, bs, config)
    got = C.to(torch.float64).numpy()
    c64 = f8.gemm_blockscaled_f64(A, B, fmt, sa, sb, bs)
    ref = torch.from_numpy(f8.gemm_blockscaled(A, B, fmt, sa, sb, bs).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()
    tol = f8.tolerance_blockscaled(f8.abs_gemm_blockscaled(A, B, fmt, sa, sb, bs), c64, K, bs)
    err = np.abs(got - ref)
    bad = int((err > tol).sum())
    assert bad == 0, f"{bad} elements over the bound; worst {np.max(err - tol):.3g}"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= 5e-3, rel


SHAPES = [
    (300, 520, 700),     # ragged in M, N and K; several tiles
    (128, 384, 1024),    # one tile row (single CTAs)
    (257, 129, 96),      # a tile row of one row, K shorter than a stage
    (1000, 1000, 2000),  # many tiles per CTA
]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_matches_oracle(fmt, bs, shape):
    M, N, K = shape
    A, B, sa, sb = operands(M, N, K, fmt, bs, 40 + bs)
    check(A, B, sa, sb, fmt, bs)


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("bs", [32, 64])
def test_tile_kinds(cta_group, bs):
    A, B, sa, sb = operands(520, 700, 1100, "e4m3", bs, 50)
    check(A, B, sa, sb, "e4m3", bs, hg.Config(cta_group=cta_group))


@pytest.mark.parametrize("M,N,K", [(200, 1000, 520), (130, 520, 1001), (200, 777, 333)])
def test_unaligned_pitches(M, N, K):
    # K or N not a multiple of 16 bytes: A or B goes through the 16-byte-pitch
    # copy; N = 777 also leaves C's rows unaligned (element stores)
    A, B, sa, sb = operands(M, N, K, "e4m3", 64, 51)
    check(A, B, sa, sb, "e4m3", 64)


def test_persistent_loop_with_few_clusters():
    # many tiles per CTA: the TMEM partial ring and the register accumulators
    # carry over from tile to tile
    A, B, sa, sb = operands(1024, 1024, 512, "e4m3", 32, 52)
    check(A, B, sa, sb, "e4m3", 32, hg.Config(cta_group=2, max_clusters=3))
    check(A, B, sa, sb, "e4m3", 32, hg.Config(cta_group=1, max_clusters=5, group_m=3))


@pytest.mark.parametrize("bs", [32, 64])
def test_small_integers_are_exact(bs):
    # operands in {-1, 0, 1}, factors 1 or 2, K = 64: every partial sum, factor
    # and accumulation is exact in fp32 and |C| <= 256 is exact in bf16
    rng = np.random.default_rng(bs)
    M, N, K = 384, 256, 64
    one, neg = 0x38, 0xB8   # E4M3 +1 and -1
    A = rng.choice(np.array([0, one, neg], np.uint8), size=(M, K))
    B = rng.choice(np.array([0, one, neg], np.uint8), size=(K, N))
    sa = rng.choice(np.array([1.0, 2.0], np.float32), size=f8.scale_grid(M, K, bs))
    sb = rng.choice(np.array([1.0, 2.0], np.float32), size=f8.scale_grid(K, N, bs))
    C = run_gpu(A, B, sa, sb, "e4m3", bs)
    want = f8.gemm_blockscaled(A, B, "e4m3", sa, sb, bs)
    assert np.array_equal(C.view(torch.int16).numpy().view(np.uint16), want)


def test_a_scale_block_reaches_only_its_block():
    # one factor of A changed: only that sub-block's rows (all columns) move,
    # and by exactly the change of that block's share of the sum
    M, N, K, bs = 256, 256, 256, 64
    A, B, sa, sb = operands(M, N, K, "e4m3", bs, 53)
    sa = np.ones_like(sa)
    sb = np.ones_like(sb)
    base = run_gpu(A, B, sa, sb, "e4m3", bs).to(torch.float64).numpy()
    sa2 = sa.copy()
    sa2[1, 2] = 0.0
    moved = run_gpu(A, B, sa2, sb, "e4m3", bs).to(torch.float64).numpy()
    rows = np.zeros(M, bool)
    rows[64:128] = True
    assert np.array_equal(base[~rows], moved[~rows])
    want = f8.gemm_blockscaled(A, B, "e4m3", sa2, sb, bs)
    got = torch.from_numpy(moved).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    c64 = f8.gemm_blockscaled_f64(A, B, "e4m3", sa2, sb, bs)
    tol = f8.tolerance_blockscaled(f8.abs_gemm_blockscaled(A, B, "e4m3", sa2, sb, bs), c64, K, bs)
    wv = torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.all(np.abs(moved - wv) <= tol)
    assert got.shape == (M, N)


def test_degenerate_shapes():
    # K = 0: the empty sum; M = 0 or N = 0: nothing is written
    C = run_gpu(np.zeros((40, 0), np.uint8), np.zeros((0, 50), np.uint8), np.zeros((2, 0), np.float32),
                np.zeros((0, 2), np.float32), "e4m3", 32, C_init=5.0)
    assert torch.all(C == 0)
    for (M, N) in ((0, 50), (40, 0)):
        A = np.zeros((M, 64), np.uint8)
        B = np.zeros((64, N), np.uint8)
        hg.hgemm_fp8_blockscaled(torch.from_numpy(A).cuda() if M else None,
                                 torch.from_numpy(B).cuda() if N else None,
                                 torch.empty((max(M, 1), max(N, 1)), dtype=torch.bfloat16, device="cuda"),
                                 None, None, M, N, 64, 32, "e4m3")
    # K shorter than one scale block
    A, B, sa, sb = operands(130, 140, 5, "e5m2", 32, 54)
    check(A, B, sa, sb, "e5m2", 32)


def test_rejects_bad_arguments():
    A = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    s = torch.ones((2, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(hg.HgemmError):
        hg.hgemm_fp8_blockscaled(A, A, C, s, s, 64, 64, 64, 16, "e4m3")      # block 16
    with pytest.raises(hg.HgemmError):
        hg.hgemm_fp8_blockscaled(A, A, C, None, s, 64, 64, 64, 32, "e4m3")   # no a_scale
    with pytest.raises(hg.HgemmError):
        hg.hgemm_fp8_blockscaled(A, A, C, s, s, 64, 64, 64, 32, "bf16")      # not fp8
    with pytest.raises(hg.HgemmError):
        hg.hgemm_fp8_blockscaled(A, A, C, s, s, 64, 64, 64, 32, "e4m3", hg.Config(block_n=256))


@pytest.mark.parametrize("bs", [32, 64])
def test_full_size_4096(bs):
    # the bench workload's shape and launch (4096^3 E4M3), every element
    # against the oracle
    M = N = K = 4096
    A = inputs.generate_fp8((M, K), "e4m3", 1, 0, 8.0)
    B = inputs.generate_fp8((K, N), "e4m3", 1, 1, 8.0)
    ga, gb = f8.scale_grid(M, K, bs), f8.scale_grid(K, N, bs)
    sa = inputs.generate_scales(ga[0] * ga[1], 1, 2).reshape(ga)
    sb = inputs.generate_scales(gb[0] * gb[1], 1, 3).reshape(gb)
    check(A, B, sa, sb, "e4m3", bs)
