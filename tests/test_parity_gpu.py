"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, elementwise, within the stated tolerance; bit-exact where
every product and sum is exact. Shapes span several tiles and ragged tails,
every kernel configuration, the persistent loop (few CTAs, many tiles each),
unaligned pitches, the degenerate shapes, and every workload at full size
(sampled rows and columns where the full oracle would be too slow)."""

import numpy as np
import pytest
import torch

import oracle
from half_precision_dense_gb300 import binding as hg
from half_precision_dense_gb300 import inputs
from tests._check import compare

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


def run_gpu(A, B, dtype, config=None, guard=0):
    """C through the C ABI; with guard > 0 the output sits between canary bands."""
    M, K = A.shape
    N = B.shape[1]
    dA = A.cuda()
    dB = B.cuda()
    t = inputs.TORCH_DTYPES[dtype]
    buf = torch.full((2 * guard + M * N,), -7.0, dtype=t, device="cuda")
    C = buf[guard:guard + M * N]
    hg.hgemm_ex(dA, dB, C, M, N, K, dtype, config)
    torch.cuda.synchronize()
    if guard:
        canary = torch.full((guard,), -7.0, dtype=t, device="cuda")
        assert torch.equal(buf[:guard], canary) and torch.equal(buf[guard + M * N:], canary), \
            "write outside C"
    return inputs.bits(C.view(M, N).cpu())


def check_full(A, B, dtype, config=None, guard=64):
    a, b = inputs.bits(A), inputs.bits(B)
    got = run_gpu(A, B, dtype, config, guard)
    ref64 = oracle.gemm_f64(a, b, dtype)
    ref = oracle.round_rne(ref64, dtype)
    r = compare(got, ref, ref64, dtype, A.shape[1])
    assert r["ok"], r
    return got, ref


def operands(M, N, K, dtype, seed, dist="uniform", sigma=1.0):
    return (inputs.generate((M, K), dtype, seed, 0, dist, sigma),
            inputs.generate((K, N), dtype, seed, 1, dist, sigma))


def int_operands(M, N, K, dtype, seed):
    rng = np.random.default_rng(seed)
    t = inputs.TORCH_DTYPES[dtype]
    Ai = rng.integers(-3, 4, (M, K)).astype(np.float32)
    Bi = rng.integers(-3, 4, (K, N)).astype(np.float32)
    return torch.from_numpy(Ai).to(t), torch.from_numpy(Bi).to(t)


# ------------------------------------------------------------ exact cases

@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_small_integers_bit_exact(cfg, dtype):
    # |C| <= 9 * 28 = 252: exact in fp32 accumulation and in both output types
    A, B = int_operands(300, 520, 28, dtype, 11)
    got = run_gpu(A, B, dtype, cfg, guard=64)
    assert np.array_equal(got, oracle.gemm(inputs.bits(A), inputs.bits(B), dtype))


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
def test_identity_and_unit_vectors(cfg):
    dtype = "bf16"
    _, B = operands(384, 320, 384, dtype, 21)
    eye = torch.eye(384, dtype=torch.bfloat16)
    got = run_gpu(eye, B, dtype, cfg)
    assert np.array_equal(got, inputs.bits(B))          # I . B = B exactly
    A, _ = operands(200, 1, 192, dtype, 22)
    eyeK = torch.eye(192, dtype=torch.bfloat16)
    got = run_gpu(A, eyeK, dtype, cfg)
    assert np.array_equal(got, inputs.bits(A))          # A . I = A exactly


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_all_ones_gives_k(dtype):
    K = 256 if dtype == "bf16" else 2048
    t = inputs.TORCH_DTYPES[dtype]
    A = torch.ones((256, K), dtype=t)
    B = torch.ones((K, 384), dtype=t)
    got = run_gpu(A, B, dtype)
    assert np.all(got == inputs.bits(torch.tensor([float(K)], dtype=t))[0])


def test_transpose_identity():
    A, B = operands(320, 448, 512, "bf16", 23)
    c1 = run_gpu(A, B, "bf16")
    c2 = run_gpu(B.t().contiguous(), A.t().contiguous(), "bf16")
    r = compare(c2, np.ascontiguousarray(c1.T), oracle.gemm_f64(inputs.bits(A), inputs.bits(B), "bf16").T,
                "bf16", 512)
    assert r["ok"], r


# ----------------------------------------------------- random shapes, tails

SHAPES = [(256, 256, 256), (128, 64, 64), (1, 1, 1), (7, 9, 11), (129, 65, 63), (255, 257, 130),
          (300, 520, 1000), (511, 383, 129), (640, 768, 576), (1000, 1000, 72)]


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_random_shapes(cfg, shape):
    M, N, K = shape
    A, B = operands(M, N, K, "bf16", 5)
    check_full(A, B, "bf16", cfg)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("max_clusters", [1, 3])
def test_persistent_loop_many_tiles_per_cta(cfg, max_clusters):
    # few CTAs walk many tiles: ring phases and both accumulators wrap many times
    c = hg.Config(cfg.cta_group, cfg.block_n, 0, max_clusters, 0, 0, cfg.multicast)
    A, B = operands(1024, 1280, 320, "f16", 6)
    check_full(A, B, "f16", c)


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("mode,clusters", [(2, 3), (3, 3), (3, 7), (4, 7)])
def test_stream_k(cfg, mode, clusters):
    # a few clusters share the leftover tiles plus a wave (mode 2), every tile
    # (mode 3) or the leftover tiles alone (mode 4) in equal ranges of K
    # blocks; owners add their partners' partial sums
    c = hg.Config(cfg.cta_group, cfg.block_n, 0, clusters, 0, mode, cfg.multicast)
    A, B = operands(1024, 1280, 704, "bf16", 14)
    check_full(A, B, "bf16", c)


@pytest.mark.parametrize("shape", [(512, 1024, 8192), (300, 700, 130), (128, 2048, 4096), (256, 512, 64),
                                   (128, 1000, 3000)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_planner_choices(shape, dtype):
    # whatever the planner picks (whole tiles; the narrowest single-CTA tiles
    # for one tile row on a long K loop)
    M, N, K = shape
    A, B = operands(M, N, K, dtype, 15)
    check_full(A, B, dtype)


SPLITS = [(2, 128), (4, 128), (2, 256), (4, 256), (8, 256)]


@pytest.mark.parametrize("split,bn", SPLITS, ids=[f"s{s}_n{b}" for s, b in SPLITS])
@pytest.mark.parametrize("shape", [(128, 3072, 4096), (77, 1000, 2056), (1, 520, 4096), (200, 1536, 1000),
                                   (129, 65, 63), (256, 1536, 2048)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_split_k(split, bn, shape, dtype):
    # the K loop of each tile split over a cluster, the partial sums reduced
    # through distributed shared memory: ragged M, N and K, a K shorter than
    # the split (CTAs with no K block add zeros), several tile rows. At most
    # 12 tiles under an 8-way split: 15 clusters of 8 fit on a 152-SM GB300.
    M, N, K = shape
    cfg = hg.Config(block_n=bn, split_k=split)
    p = hg.plan(M, N, K, dtype, cfg)
    assert p["split_k"] == split and p["grid_ctas"] == p["num_tiles"] * split
    A, B = operands(M, N, K, dtype, 18)
    check_full(A, B, dtype, cfg)


@pytest.mark.parametrize("store_mode", [1, 2, 3, 4])
def test_split_k_store_modes_and_repeat(store_mode):
    # every store mode (the reduction writes C itself: 8-byte vectors, plain
    # stores for mode 2), and the same bits on a second call
    cfg = hg.Config(block_n=256, split_k=4, store_mode=store_mode)
    A, B = operands(128, 2056, 3000, "bf16", 19)
    got, _ = check_full(A, B, "bf16", cfg)
    again, _ = check_full(A, B, "bf16", cfg)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("shape", [(128, 4864, 8192), (100, 4736, 8200)])
def test_split_k_planner_fallback(shape):
    # the planner's split of 4 on 37-38 tiles: fewer clusters of 4 are
    # resident than tiles, so the launch takes a split of 2 (or whole tiles),
    # and the plan for the current device reports the split it keeps
    M, N, K = shape
    p152 = hg.plan(M, N, K, "bf16", sm_count=152)
    assert p152["split_k"] == 4 and p152["num_tiles"] * 4 <= 152 and p152["num_tiles"] > 32
    p = hg.plan(M, N, K, "bf16")
    assert p["split_k"] in (1, 2) and p["num_tiles"] == p152["num_tiles"]
    A, B = operands(M, N, K, "bf16", 21)
    check_full(A, B, "bf16")


def test_split_k_unaligned_c():
    # N = 1001: C rows are not 16-byte multiples, element stores only
    A, B = operands(100, 1001, 2048, "f16", 20)
    check_full(A, B, "f16", hg.Config(block_n=128, split_k=4))


def test_stream_k_repeated_calls_reuse_workspace():
    # the pool hands the same workspace back; fresh launch epochs keep stale
    # partial-sum marks from being taken for new ones
    A, B = operands(512, 1024, 2048, "f16", 16)
    cfg = hg.Config(stream_k=3)
    assert hg.plan(512, 1024, 2048, "f16", cfg)["sk_tiles"] > 0
    a, b = inputs.bits(A), inputs.bits(B)
    ref64 = oracle.gemm_f64(a, b, "f16")
    ref = oracle.round_rne(ref64, "f16")
    dA, dB = A.cuda(), B.cuda()
    for i in range(4):
        C = torch.empty((512, 1024), dtype=torch.float16, device="cuda")
        hg.hgemm_ex(dA, dB, C, 512, 1024, 2048, "f16", cfg)
        torch.cuda.synchronize()
        r = compare(inputs.bits(C.cpu()), ref, ref64, "f16", 2048)
        assert r["ok"], (i, r)


@pytest.mark.parametrize("group_m", [1, 2, 5, 64])
def test_raster_groups(group_m):
    A, B = operands(1536, 1024, 256, "bf16", 7)
    check_full(A, B, "bf16", hg.Config(cta_group=2, block_n=128, group_m=group_m))


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("store_mode", [2, 3, 4, 5])
def test_store_modes_match(cfg, store_mode):
    # plain 2-byte stores, direct 16-byte vector stores, smem-staged
    # coalesced stores and realigned staged stores (on an aligned C), ragged
    # M and N
    c = hg.Config(cfg.cta_group, cfg.block_n, 0, 0, store_mode, 0, cfg.multicast)
    A, B = operands(700, 520, 300, "bf16", 8)
    check_full(A, B, "bf16", c)


EPI16 = [(1, 256), (2, 224), (2, 256)]
EPI16_IDS = ["cg1_n256", "cg2_n224", "cg2_n256"]


@pytest.mark.parametrize("tile", EPI16, ids=EPI16_IDS)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("store_mode", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("shape", [(700, 520, 64), (1000, 1800, 300), (4096, 4096, 64)])
def test_sixteen_epilogue_warps(tile, dtype, store_mode, shape):
    # 16 epilogue warps on 32-column chunks of 224- and 256-wide tiles, every
    # store mode, ragged M and N, short and longer K loops, and the
    # persistent loop (a cap on the clusters: several tiles per CTA, both
    # accumulator buffers)
    M, N, K = shape
    A, B = operands(M, N, K, dtype, 60)
    for mc in ((0, 3) if M * N < 4_000_000 else (0,)):
        check_full(A, B, dtype, hg.Config(cta_group=tile[0], block_n=tile[1], max_clusters=mc,
                                          store_mode=store_mode, epi_warps=16))


@pytest.mark.parametrize("tile", EPI16, ids=EPI16_IDS)
@pytest.mark.parametrize("store_mode", [1, 2, 3, 4, 5])
def test_eight_epilogue_warps_on_wide_tiles(tile, store_mode):
    # the 8-warp epilogue (64-column chunks) that the planner no longer takes
    # for these tiles, forced: every store mode, ragged M and N, the
    # persistent loop
    A, B = operands(700, 520, 300, "bf16", 63)
    check_full(A, B, "bf16", hg.Config(cta_group=tile[0], block_n=tile[1], max_clusters=2, store_mode=store_mode,
                                       epi_warps=8))


@pytest.mark.parametrize("tile", EPI16, ids=EPI16_IDS)
@pytest.mark.parametrize("N", [4095, 777])
def test_sixteen_epilogue_warps_unaligned_c(tile, N):
    # a C pitch that is not a multiple of 16 bytes: realigned stores (5)
    A, B = operands(300, N, 128, "bf16", 61)
    check_full(A, B, "bf16", hg.Config(cta_group=tile[0], block_n=tile[1], epi_warps=16))


def test_sixteen_epilogue_warps_bit_exact_and_planner_default():
    # small integers: every product and sum is exact, so 16 and 8 warps,
    # and the planner's own choice, agree bit for bit with the oracle
    M, N, K = 1536, 2304, 192
    A, B = int_operands(M, N, K, "bf16", 62)
    assert hg.plan(M, N, K, "bf16")["epi_warps"] == 16
    outs = [check_full(A, B, "bf16", cfg)[0] for cfg in
            (None, hg.Config(cta_group=1, block_n=256, epi_warps=8),
             hg.Config(cta_group=1, block_n=256, epi_warps=16, max_clusters=5))]
    ref = oracle.round_rne(oracle.gemm_f64(inputs.bits(A), inputs.bits(B), "bf16"), "bf16")
    for o in outs:
        assert np.array_equal(o, ref)


@pytest.mark.parametrize("store_mode", [1, 3, 4])
def test_store_modes_with_stream_k(store_mode):
    c = hg.Config(2, 224, 0, 3, store_mode, 3)
    A, B = operands(1024, 1344, 512, "f16", 17)
    check_full(A, B, "f16", c)


@pytest.mark.parametrize("shape", [(300, 517, 264), (129, 4095, 257), (64, 100, 1001), (33, 7, 5)])
def test_unaligned_pitches(shape):
    # N or K not a multiple of 8: repacked operand and/or plain stores of C
    M, N, K = shape
    A, B = operands(M, N, K, "bf16", 9)
    check_full(A, B, "bf16")


@pytest.mark.parametrize("cfg", CONFIGS, ids=CFG_IDS)
@pytest.mark.parametrize("store_mode", [2, 5])
@pytest.mark.parametrize("N", [4095, 1001, 777, 130])
def test_unaligned_c_store_modes(cfg, store_mode, N):
    # row pitches of N 16-bit elements that are not multiples of 8: every row
    # starts at a different offset inside a 16-byte segment; the realigned
    # stores (5) must touch exactly the columns of C, as the element stores (2)
    # do (the canary bands around C stay intact), on ragged M and N
    M, K = 300, 200
    A, B = operands(M, N, K, "bf16", 36)
    check_full(A, B, "bf16", hg.Config(cfg.cta_group, cfg.block_n, 0, 0, store_mode, 0, 0))


def test_unaligned_c_offset_base_and_split_k():
    # a C base 2 bytes past a 16-byte boundary with an aligned pitch (every
    # row misaligned the same way), through the planner's realigned stores,
    # and the K split's own stores on the same C
    M, N, K = 200, 264, 1536
    A, B = operands(M, N, K, "f16", 37)
    a, b = inputs.bits(A), inputs.bits(B)
    ref64 = oracle.gemm_f64(a, b, "f16")
    for cfg in (None, hg.Config(block_n=128, split_k=2)):
        dC = torch.zeros(M * N + 9, dtype=torch.float16, device="cuda")
        C = dC[1:1 + M * N]
        hg.hgemm_ex(A.cuda(), B.cuda(), C, M, N, K, "f16", cfg)
        torch.cuda.synchronize()
        assert dC[0].item() == 0 and torch.count_nonzero(dC[1 + M * N:]).item() == 0
        got = inputs.bits(C.view(M, N).cpu())
        r = compare(got, oracle.round_rne(ref64, "f16"), ref64, "f16", K)
        assert r["ok"], r


def test_unaligned_base_pointers():
    M, N, K = 200, 264, 136
    A, B = operands(M, N, K, "f16", 10)
    dA = torch.empty(M * K + 1, dtype=torch.float16, device="cuda")[1:]
    dB = torch.empty(K * N + 3, dtype=torch.float16, device="cuda")[3:]
    dC = torch.zeros(M * N + 5, dtype=torch.float16, device="cuda")[5:]
    dA.copy_(A.reshape(-1))
    dB.copy_(B.reshape(-1))
    hg.hgemm(dA, dB, dC, M, N, K, "f16")
    torch.cuda.synchronize()
    got = inputs.bits(dC.view(M, N).cpu())
    a, b = inputs.bits(A), inputs.bits(B)
    ref64 = oracle.gemm_f64(a, b, "f16")
    r = compare(got, oracle.round_rne(ref64, "f16"), ref64, "f16", K)
    assert r["ok"], r


def test_k_zero_writes_zeros_and_empty_is_noop():
    C = torch.full((37, 41), 3.0, dtype=torch.bfloat16, device="cuda")
    a = torch.empty((37, 0), dtype=torch.bfloat16, device="cuda")
    b = torch.empty((0, 41), dtype=torch.bfloat16, device="cuda")
    hg.hgemm(a, b, C, 37, 41, 0, "bf16")
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0
    D = torch.full((4, 4), 3.0, dtype=torch.bfloat16, device="cuda")
    hg.hgemm(None, None, D, 0, 4, 4, "bf16")
    torch.cuda.synchronize()
    assert torch.all(D == 3.0)


def test_overlap_rejected_on_device():
    X = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(hg.HgemmError):
        hg.hgemm(X[:1024], X[1024:2048], X[512:1536], 32, 32, 32, "bf16")


def test_host_entry_point():
    M, N, K = 512, 384, 256
    A, B = operands(M, N, K, "bf16", 12)
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    dA = torch.empty_like(A, device="cuda")
    dB = torch.empty_like(B, device="cuda")
    dC = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    hg.hgemm_host(hA, hB, hC, M, N, K, "bf16", dA, dB, dC, torch.cuda.current_stream())
    a, b = inputs.bits(A), inputs.bits(B)
    ref64 = oracle.gemm_f64(a, b, "bf16")
    r = compare(inputs.bits(hC), oracle.round_rne(ref64, "bf16"), ref64, "bf16", K)
    assert r["ok"], r


@pytest.mark.parametrize("M", [4100, 1100])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_host_entry_point_in_bands(dtype, M):
    # M = 4100: four row bands (three of 1280 rows and one of 260); M = 1100:
    # three (512, 512 and 76). Each band is copied in, multiplied and copied
    # out on the internal streams; work already on the caller's stream (a
    # long fill of dC) runs first
    N, K = 384, 256
    A, B = operands(M, N, K, dtype, 17)
    hA, hB = A.pin_memory(), B.pin_memory()
    t = torch.bfloat16 if dtype == "bf16" else torch.float16
    hC = torch.empty((M, N), dtype=t).pin_memory()
    dA = torch.empty_like(A, device="cuda")
    dB = torch.empty_like(B, device="cuda")
    dC = torch.empty((M, N), dtype=t, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(2_000_000)
        dC.fill_(7)
        hg.hgemm_host(hA, hB, hC, M, N, K, dtype, dA, dB, dC, s)
    a, b = inputs.bits(A), inputs.bits(B)
    ref64 = oracle.gemm_f64(a, b, dtype)
    r = compare(inputs.bits(hC), oracle.round_rne(ref64, dtype), ref64, dtype, K)
    assert r["ok"], r
    # K = 0: every band writes zeros
    hg.hgemm_host(hA, hB, hC, M, N, 0, dtype, dA, dB, dC)
    assert bool((hC == 0).all())


def test_matmul_wrapper_and_stream():
    A, B = operands(256, 192, 320, "f16", 13)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = hg.matmul(A.cuda(), B.cuda())
    s.synchronize()
    a, b = inputs.bits(A), inputs.bits(B)
    ref64 = oracle.gemm_f64(a, b, "f16")
    r = compare(inputs.bits(C.cpu()), oracle.round_rne(ref64, "f16"), ref64, "f16", 320)
    assert r["ok"], r


# --------------------------------------------------------- the workloads

FULL = ["square256_bf16", "square4096_f16", "square4096_bf16", "skinny_bf16", "tails_bf16",
        "shortk_bf16"]
SAMPLED = ["square8192_bf16", "mlp_up_bf16", "mlp_down_bf16"]


@pytest.mark.parametrize("name", FULL)
def test_workload_full_oracle(name):
    A, B, (M, N, K, dtype) = inputs.workload_operands(name)
    check_full(A, B, dtype, guard=256)


def sample_indices(n, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 127, 128, 255, 256, n - 1]
    return np.unique(np.concatenate([rng.integers(0, n, 32), [i for i in fixed if i < n]]))


@pytest.mark.parametrize("name", SAMPLED)
def test_workload_sampled_rows_and_cols(name):
    A, B, (M, N, K, dtype) = inputs.workload_operands(name)
    got = run_gpu(A, B, dtype, guard=256)
    a, b = inputs.bits(A), inputs.bits(B)
    rows = sample_indices(M, 1)
    cols = sample_indices(N, 2)
    ref_r, ref64_r = oracle.gemm_rows(a, b, dtype, rows)
    r = compare(got[rows], ref_r, ref64_r, dtype, K)
    assert r["ok"], ("rows", r)
    ref_c, ref64_c = oracle.gemm_cols(a, b, dtype, cols)
    r = compare(got[:, cols], ref_c, ref64_c, dtype, K)
    assert r["ok"], ("cols", r)
    # a property at any size: every element is finite
    v = torch.from_numpy(got.view(np.int16).copy()).view(inputs.TORCH_DTYPES[dtype]).double()
    assert torch.isfinite(v).all()
