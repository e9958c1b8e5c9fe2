"""GPU parity of the FP8 variant (E4M3 / E5M2 operands, per-channel fp32
scales, bf16 C) against the FP8 oracle on the same seeded inputs: bit-exact
where every product, sum and scale product is exact, elsewhere within the
bound of an fp32 accumulation followed by the scale products and one bf16
rounding (``oracle.fp8_oracle.tolerance``). Shapes span several tiles and
ragged tails, every tile configuration, the persistent loop, unaligned
pitches, every store mode, stream-K, null scales, K = 0 and the 4096^3 shape
(sampled)."""

import numpy as np
import pytest
import torch

from half_precision_dense_gb300 import binding as hg
from half_precision_dense_gb300 import inputs
from oracle import fp8_oracle as f8

pytestmark = pytest.mark.gpu

CONFIGS = [
    hg.Config(cta_group=1, block_n=64),
    hg.Config(cta_group=1, block_n=128),
    hg.Config(cta_group=1, block_n=256),
    hg.Config(cta_group=2, block_n=128),
    hg.Config(cta_group=2, block_n=224),
    hg.Config(cta_group=2, block_n=256),
]
CFG_IDS = ["cg1_n64", "cg1_n128", "cg1_n256", "cg2_n128", "cg2_n224", "cg2_n256"]
FMTS = ["e4m3", "e5m2"]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from half_precision_dense_gb300 import build as hbuild
    hbuild.build()
    hg.load_library()
    hg.get_device_status(0, reset=True)
    yield
    st, info = hg.get_device_status(0)
    assert st == 0, f"a kernel reported status {st} (info {info:#x})"


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def run_gpu(A, B, fmt, sa=None, sb=None, config=None, guard=64):
    M, K = A.shape
    N = B.shape[1]
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dsa = torch.from_numpy(sa).cuda() if sa is not None else None
    dsb = torch.from_numpy(sb).cuda() if sb is not None else None
    buf = torch.full((2 * guard + M * N,), -7.0, dtype=torch.bfloat16, device="cuda")
    C = buf[guard:guard + M * N]
    hg.hgemm_fp8(dA, dB, C, dsa, dsb, M, N, K, fmt, config)
    torch.cuda.synchronize()
    if guard:
        canary = torch.full((guard,), -7.0, dtype=torch.bfloat16, device="cuda")
        assert torch.equal(buf[:guard], canary) and torch.equal(buf[guard + M * N:], canary), \
            "write outside C"
    return C.view(M, N).cpu().view(torch.int16).numpy().view(np.uint16)


def assert_close(got_bits, A, B, fmt, sa=None, sb=None):
    K = A.shape[1]
    c64 = f8.gemm_f64(A, B, fmt, sa, sb)
    ref = bf16_values(f8.gemm(A, B, fmt, sa, sb))
    got = bf16_values(got_bits)
    tol = f8.tolerance(f8.abs_gemm(A, B, fmt, sa, sb), c64, K)
    err = np.abs(got - ref)
    bad = np.argwhere(~(err <= tol))
    assert len(bad) == 0, (f"{len(bad)} elements out of bound; first {bad[:4].tolist()}: "
                           f"got {got[tuple(bad[0])]} want {ref[tuple(bad[0])]} tol {tol[tuple(bad[0])]}")
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert fro <= 5e-3, fro


def operands(M, N, K, fmt, seed, scales=True):
    A = inputs.generate_fp8((M, K), fmt, seed, 0)
    B = inputs.generate_fp8((K, N), fmt, seed, 1)
    if not scales:
        return A, B, None, None
    return A, B, inputs.generate_scales(M, seed, 2), inputs.generate_scales(N, seed, 3)


def check(M, N, K, fmt, seed, config=None, scales=True):
    A, B, sa, sb = operands(M, N, K, fmt, seed, scales)
    assert_close(run_gpu(A, B, fmt, sa, sb, config), A, B, fmt, sa, sb)


def int_fp8(shape, fmt, rng):
    v = rng.integers(-3, 4, shape).astype(np.float32)
    return torch.from_numpy(v).to(getattr(torch, inputs.FP8_TORCH[fmt])).view(torch.uint8).numpy()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_small_integers_and_power_of_two_scales_bit_exact(cfg, fmt):
    rng = np.random.default_rng(1)
    M, N, K = 300, 520, 24
    A = int_fp8((M, K), fmt, rng)
    B = int_fp8((K, N), fmt, rng)
    sa = (2.0 ** rng.integers(-2, 3, M)).astype(np.float32)
    sb = (2.0 ** rng.integers(-2, 3, N)).astype(np.float32)
    got = run_gpu(A, B, fmt, sa, sb, cfg)
    exact = f8.gemm_f64(A, B, fmt, sa, sb)      # |C| <= 9 * 24 * 16: every value exact in bf16
    assert np.array_equal(bf16_values(got), exact)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("shape", [(256, 256, 256), (1000, 520, 336), (129, 72, 48), (640, 768, 1024)])
def test_random_shapes(cfg, fmt, shape):
    check(*shape, fmt, 2, cfg)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_persistent_loop(cfg):
    check(1024, 1280, 384, "e4m3", 3, hg.Config(cfg.cta_group, cfg.block_n, 0, 2))


@pytest.mark.parametrize("block_n", [224, 256])
@pytest.mark.parametrize("store_mode", [1, 2, 3, 4, 5])
def test_store_modes(store_mode, block_n):
    # 224: the last 32-column chunk of every tile goes through each store path
    check(700, 1024, 512, "e4m3", 4, hg.Config(cta_group=2, block_n=block_n, store_mode=store_mode))


@pytest.mark.parametrize("epi", [8, 16])
@pytest.mark.parametrize("tile", [(1, 256), (2, 224), (2, 256)], ids=["cg1_n256", "cg2_n224", "cg2_n256"])
@pytest.mark.parametrize("fmt", FMTS)
def test_epilogue_warps(tile, epi, fmt):
    # the wide tiles with 8 epilogue warps on 64-column chunks and 16 on
    # 32-column chunks (the planner's default for them), ragged M and N, the
    # persistent loop
    check(1000, 520, 336, fmt, 10, hg.Config(cta_group=tile[0], block_n=tile[1], max_clusters=3, epi_warps=epi))


@pytest.mark.parametrize("block_n", [224, 256])
@pytest.mark.parametrize("mode,clusters", [(2, 3), (3, 5), (4, 7)])
def test_stream_k(mode, clusters, block_n):
    check(1024, 1280, 1408, "e5m2", 5,
          hg.Config(cta_group=2, block_n=block_n, max_clusters=clusters, stream_k=mode))


@pytest.mark.parametrize("shape", [(333, 517, 259), (256, 250, 130), (100, 3, 7)])
def test_unaligned_pitches(shape):
    # K not a multiple of 16 bytes (A repacked), N not a multiple of 8 (C with
    # plain stores)
    check(*shape, "e4m3", 6)


def test_null_scales_and_k_zero():
    check(512, 1024, 2048, "e4m3", 7, scales=False)
    got = run_gpu(np.zeros((64, 0), np.uint8), np.zeros((0, 96), np.uint8), "e4m3")
    assert np.array_equal(bf16_values(got), np.zeros((64, 96)))


@pytest.mark.parametrize("fmt", FMTS)
def test_workload_4096_sampled(fmt):
    M = N = K = 4096
    A, B, sa, sb = operands(M, N, K, fmt, 1)
    got = run_gpu(A, B, fmt, sa, sb, guard=0)
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([rng.integers(0, M, 24), [0, 127, 128, 255, 256, M - 1]]))
    cols = np.unique(np.concatenate([rng.integers(0, N, 24), [0, 127, 128, 255, 256, N - 1]]))
    assert_close(got[rows], A[rows], B, fmt, sa[rows], sb)
    assert_close(got[:, cols], A, B[:, cols], fmt, sa, sb[cols])
