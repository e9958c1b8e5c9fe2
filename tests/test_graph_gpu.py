"""CUDA-graph capture: each entry point recorded into a graph and replayed
gives the same bits as the eager call (same plan, same accumulation order),
replay after replay, with the operands changed between replays (the graph
holds pointers, not values). The cases cover the launches a graph must carry
besides the GEMM kernel: the stream-K phase (its partial-sum marks are
cleared by the captured call), the pool's workspace allocation, the
16-byte-pitch repack and the explicit im2col matrix. The no-alloc entry
point captures with its fixed array."""

import pytest
import torch

from half_precision_dense_gb300 import binding as hg

pytestmark = pytest.mark.gpu

REPLAYS = 4


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from half_precision_dense_gb300 import build as hbuild
    hbuild.build()
    hg.load_library()
    hg.get_device_status(0, reset=True)
    yield
    hg.conv2d_set_mode(0)
    st, info = hg.get_device_status(0)
    assert st == 0, f"a kernel reported status {st} (info {info:#x})"


def check_graph(call, operands, out, refresh):
    """Capture call(stream), then replay it REPLAYS times; before each replay
    refresh() gives the operands new values, and the replayed output must
    equal an eager call's output bit for bit."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)                                  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    torch.cuda.synchronize()
    for i in range(REPLAYS):
        if i:
            refresh()
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        got = out.clone()
        call(torch.cuda.current_stream())        # eager, same operands
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.uint8), out.view(torch.uint8)), f"replay {i} differs from the eager call"
        assert bool(got.ne(0).any()), "the replay wrote nothing"
    del g


def rnd(shape, dtype, scale=1.0):
    return (torch.randn(*shape, device="cuda") * scale).to(dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(1024, 1536, 2048), (128, 4096, 8192), (4096, 4096, 1024)])
def test_gemm(dtype, M, N, K):
    t = torch.bfloat16 if dtype == "bf16" else torch.float16
    A, B = rnd((M, K), t), rnd((K, N), t)
    C = torch.empty(M, N, device="cuda", dtype=t)
    check_graph(lambda s: hg.hgemm(A, B, C, M, N, K, dtype, s), (A, B), C,
                lambda: (A.copy_(rnd((M, K), t)), B.copy_(rnd((K, N), t))))


SK_CONFIGS = {"leftover_plus_wave": hg.Config(stream_k=2), "all_tiles": hg.Config(stream_k=3),
              "leftover_only": hg.Config(stream_k=4)}


@pytest.mark.parametrize("mode", sorted(SK_CONFIGS))
def test_gemm_stream_k(mode):
    # stream-K forced: partial sums and their marks go through the pool
    # workspace inside the graph, and the marks are cleared by the captured call
    M, N, K = 1024, 1536, 2048
    cfg = SK_CONFIGS[mode]
    assert hg.plan(M, N, K, "bf16", cfg)["sk_tiles"] > 0
    A, B = rnd((M, K), torch.bfloat16), rnd((K, N), torch.bfloat16)
    C = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    check_graph(lambda s: hg.hgemm_ex(A, B, C, M, N, K, "bf16", cfg, s), (A, B), C,
                lambda: (A.copy_(rnd((M, K), torch.bfloat16)), B.copy_(rnd((K, N), torch.bfloat16))))


@pytest.mark.parametrize("split,bn", [(4, 256), (2, 128)])
def test_gemm_split_k(split, bn):
    # the in-cluster K split: its barriers are initialised by each launch
    M, N, K = 128, 2048, 4096
    cfg = hg.Config(block_n=bn, split_k=split)
    A, B = rnd((M, K), torch.bfloat16), rnd((K, N), torch.bfloat16)
    C = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    check_graph(lambda s: hg.hgemm_ex(A, B, C, M, N, K, "bf16", cfg, s), (A, B), C,
                lambda: (A.copy_(rnd((M, K), torch.bfloat16)), B.copy_(rnd((K, N), torch.bfloat16))))


def test_gemm_unaligned_repack():
    # K = 1001: rows of A are not 16-byte multiples, so A is repacked in the
    # pool workspace inside the graph
    M, N, K = 700, 520, 1001
    A, B = rnd((M, K), torch.bfloat16), rnd((K, N), torch.bfloat16)
    C = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    assert hg.plan(M, N, K, "bf16")["workspace_bytes"] > 0
    check_graph(lambda s: hg.hgemm(A, B, C, M, N, K, "bf16", s), (A, B), C,
                lambda: A.copy_(rnd((M, K), torch.bfloat16)))


@pytest.mark.parametrize("M,N,K,sk", [(128, 4096, 8192, 3), (128, 4096, 8192, 0), (2048, 2048, 2048, 0)])
def test_noalloc(M, N, K, sk):
    # sk 3: every tile's K blocks shared; partial sums and marks in the fixed array
    cfg = hg.Config(stream_k=sk) if sk else None
    if sk:
        assert hg.plan(M, N, K, "bf16", cfg)["sk_tiles"] > 0
    A, B = rnd((M, K), torch.bfloat16), rnd((K, N), torch.bfloat16)
    C = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    check_graph(lambda s: hg.hgemm_noalloc(A, B, C, M, N, K, "bf16", s, config=cfg), (A, B), C,
                lambda: B.copy_(rnd((K, N), torch.bfloat16)))


def test_tf32():
    M, N, K = 512, 768, 4096
    A, B = rnd((M, K), torch.float32), rnd((K, N), torch.float32)
    C = torch.empty(M, N, device="cuda", dtype=torch.float32)
    check_graph(lambda s: hg.hgemm(A, B, C, M, N, K, "tf32", s), (A, B), C,
                lambda: A.copy_(rnd((M, K), torch.float32)))


def test_fp8():
    M, N, K = 1024, 1024, 4096
    A = rnd((M, K), torch.float8_e4m3fn, 2.0).view(torch.uint8)
    B = rnd((K, N), torch.float8_e4m3fn, 2.0).view(torch.uint8)
    sa = torch.rand(M, device="cuda") + 0.5
    sb = torch.rand(N, device="cuda") + 0.5
    C = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    check_graph(lambda s: hg.hgemm_fp8(A, B, C, sa, sb, M, N, K, "e4m3", stream=s), (A, B), C,
                lambda: (B.copy_(rnd((K, N), torch.float8_e4m3fn, 2.0).view(torch.uint8)),
                         sb.copy_(torch.rand(N, device="cuda") + 0.5)))


@pytest.mark.parametrize("mode", [0, 1])
def test_conv(mode):
    # mode 0: implicit GEMM (TMA im2col); mode 1: explicit im2col matrix in the pool
    Nb, H, W, Cc, K, R, S, stride, pad = 4, 14, 14, 128, 192, 3, 3, 1, 1
    hg.conv2d_set_mode(mode)
    try:
        x, w = rnd((Nb, H, W, Cc), torch.bfloat16), rnd((R, S, Cc, K), torch.bfloat16)
        y = torch.empty(Nb, H, W, K, device="cuda", dtype=torch.bfloat16)
        check_graph(lambda s: hg.hgemm_conv2d(x, w, y, Nb, H, W, Cc, K, R, S, stride, pad, "bf16", s), (x, w), y,
                    lambda: x.copy_(rnd((Nb, H, W, Cc), torch.bfloat16)))
    finally:
        hg.conv2d_set_mode(0)
