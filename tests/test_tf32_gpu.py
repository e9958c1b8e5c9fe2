"""GPU parity of the TF32 variant (dtype HGEMM_TF32: fp32 A, B, C) against the
TF32 oracle on the same seeded inputs: bit-exact where every product and sum
is exact, elsewhere within the per-element bound of an fp32 accumulation
(``oracle.tf32_oracle.tolerance``). Shapes span several tiles and ragged
tails, every tf32 tile configuration, the persistent loop, unaligned
pitches, every store mode, stream-K, the degenerate shapes and the 4096^3
workload (sampled)."""

import numpy as np
import pytest
import torch

from half_precision_dense_gb300 import binding as hg
from half_precision_dense_gb300 import inputs
from oracle import tf32_oracle as tf

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


def operands(M, N, K, seed, dist="uniform", sigma=1.0):
    return (inputs.generate((M, K), "f32", seed, 0, dist, sigma).numpy(),
            inputs.generate((K, N), "f32", seed, 1, dist, sigma).numpy())


def run_gpu(A, B, config=None, guard=64):
    M, K = A.shape
    N = B.shape[1]
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    buf = torch.full((2 * guard + M * N,), -7.0, dtype=torch.float32, device="cuda")
    C = buf[guard:guard + M * N]
    hg.hgemm_ex(dA, dB, C, M, N, K, "tf32", config)
    torch.cuda.synchronize()
    if guard:
        canary = torch.full((guard,), -7.0, dtype=torch.float32, device="cuda")
        assert torch.equal(buf[:guard], canary) and torch.equal(buf[guard + M * N:], canary), \
            "write outside C"
    return C.view(M, N).cpu().numpy()


def assert_close(got, A, B):
    ref = tf.gemm(A, B)
    tol = tf.tolerance(tf.abs_gemm(A, B), ref, A.shape[1])
    err = np.abs(got.astype(np.float64) - ref)
    bad = np.argwhere(~(err <= tol))
    assert len(bad) == 0, (f"{len(bad)} elements out of bound; first {bad[:4].tolist()}, "
                           f"got {got[tuple(bad[0])]} want {ref[tuple(bad[0])]} tol {tol[tuple(bad[0])]}")
    fro = np.linalg.norm(got.astype(np.float64) - ref) / max(np.linalg.norm(ref), 1e-300)
    assert fro <= 1e-5, fro


def check(M, N, K, seed, config=None, dist="uniform"):
    A, B = operands(M, N, K, seed, dist)
    assert_close(run_gpu(A, B, config), A, B)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_small_integers_bit_exact(cfg):
    rng = np.random.default_rng(1)
    M, N, K = 300, 520, 330
    Ai = rng.integers(-3, 4, (M, K))
    Bi = rng.integers(-3, 4, (K, N))
    got = run_gpu(Ai.astype(np.float32), Bi.astype(np.float32), cfg)
    assert np.array_equal(got, (Ai @ Bi).astype(np.float32))


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_low_fraction_bits_are_ignored(cfg):
    # every A element is 1 + 2^-11 + 2^-12: its tf32 part is 1.0 (the dropped
    # bits would round it up to 1 + 2^-10); B is the identity, so C = tf32(A)
    M, K = 256, 256
    A = np.full((M, K), np.float32(1 + 2.0 ** -11 + 2.0 ** -12), dtype=np.float32)
    B = np.eye(K, dtype=np.float32)
    got = run_gpu(A, B, cfg)
    assert np.array_equal(got, np.ones((M, K), np.float32))
    assert np.array_equal(got, tf.gemm(A, B))


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("shape", [(256, 256, 256), (1000, 520, 330), (129, 65, 31), (640, 768, 1024)])
def test_random_shapes(cfg, shape):
    check(*shape, 2, cfg)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_persistent_loop(cfg):
    c = hg.Config(cfg.cta_group, cfg.block_n, 0, 2)
    check(1024, 1280, 320, 3, c)


@pytest.mark.parametrize("block_n", [224, 256])
@pytest.mark.parametrize("store_mode", [1, 2, 3, 4])
def test_store_modes(store_mode, block_n):
    # 224: every tile's last chunk is one 32-column half, in each store path
    check(700, 1024, 256, 4, hg.Config(cta_group=2, block_n=block_n, store_mode=store_mode))


@pytest.mark.parametrize("block_n", [224, 256])
@pytest.mark.parametrize("mode,clusters", [(2, 3), (3, 5), (4, 7)])
def test_stream_k(mode, clusters, block_n):
    check(1024, 1280, 704, 5,
          hg.Config(cta_group=2, block_n=block_n, max_clusters=clusters, stream_k=mode))


@pytest.mark.parametrize("shape", [(333, 517, 259), (256, 250, 130), (100, 3, 7)])
def test_unaligned_pitches(shape):
    # K or N not a multiple of 4 floats: the operand is repacked, C written
    # with plain stores
    check(*shape, 6)


def test_planner_and_k_zero():
    check(512, 1024, 2048, 7)
    A = np.zeros((64, 0), np.float32)
    B = np.zeros((0, 96), np.float32)
    got = run_gpu(np.ones((64, 1), np.float32)[:, :0].copy(), B)
    assert np.array_equal(got, np.zeros((64, 96), np.float32))
    del A


def test_host_entry_and_matmul_wrapper():
    M, N, K = 300, 400, 500
    A, B = operands(M, N, K, 8)
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
    dA = torch.empty_like(hA, device="cuda")
    dB = torch.empty_like(hB, device="cuda")
    dC = torch.empty_like(hC, device="cuda")
    hg.hgemm_host(hA, hB, hC, M, N, K, "tf32", dA, dB, dC)
    assert_close(hC.numpy(), A, B)
    out = hg.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    assert out.dtype == torch.float32
    assert_close(out.cpu().numpy(), A, B)


def test_workload_4096_sampled():
    # the 4096^3 shape at full size: every element of sampled rows and columns
    M = N = K = 4096
    A, B = operands(M, N, K, 1)
    got = run_gpu(A, B, guard=0)
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([rng.integers(0, M, 24), [0, 127, 128, 255, 256, M - 1]]))
    cols = np.unique(np.concatenate([rng.integers(0, N, 24), [0, 127, 128, 255, 256, N - 1]]))
    assert_close(got[rows], A[rows], B)
    assert_close(got[:, cols], A, B[:, cols])
