"""hgemm_noalloc: the entry point for callers that cannot allocate device
memory (graph captures that forbid allocation, pipelines that reserve all
memory up front, hosts whose memory belongs to another runtime's pool).

It must give the same results as hgemm on shapes that need the repack
workspace, call after call (the library's fixed scratch array is shared and
keeps the previous call's contents), and refuse shapes whose workspace would
not fit. This file is collected last so that a first-failure run has already
run every other test; it also passes on its own in a fresh process."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from half_precision_dense_gb300 import binding as hg
from half_precision_dense_gb300 import inputs
from tests._check import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from half_precision_dense_gb300 import build as hbuild
    hbuild.build()
    return hg.load_library()


def _call(lib, fn, A, B, C, M, N, K, dtype):
    code = hg.HGEMM_BF16 if dtype == "bf16" else hg.HGEMM_F16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = fn(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
            ctypes.c_void_p(C.data_ptr()), M, N, K, code, stream)
    return st


# Each shape needs the workspace: N (and for the second, K) not a multiple of 8.
CALLS = [((300, 517, 264), "bf16", 31), ((129, 4095, 257), "f16", 32), ((1000, 4095, 4104), "bf16", 33)]


def test_noalloc_matches_hgemm_on_consecutive_calls(lib):
    assert lib.hgemm_noalloc_scratch_bytes() == 64 << 20
    for (M, N, K), dtype, seed in CALLS:
        A = inputs.generate((M, K), dtype, seed, 0)
        B = inputs.generate((K, N), dtype, seed, 1)
        dA, dB = A.cuda(), B.cuda()
        t = inputs.TORCH_DTYPES[dtype]
        C_ref = torch.full((M, N), -3.0, dtype=t, device="cuda")
        C_new = torch.full((M, N), -5.0, dtype=t, device="cuda")
        assert _call(lib, lib.hgemm, dA, dB, C_ref, M, N, K, dtype) == 0
        assert _call(lib, lib.hgemm_noalloc, dA, dB, C_new, M, N, K, dtype) == 0
        torch.cuda.synchronize()
        got_ref = inputs.bits(C_ref.cpu())
        got_new = inputs.bits(C_new.cpu())
        # against the existing entry point, with the parity tolerance
        ref64 = oracle.gemm_f64(inputs.bits(A), inputs.bits(B), dtype)
        r = compare(got_new, got_ref, ref64, dtype, K)
        assert r["ok"], r
        # and both against the oracle
        want = oracle.round_rne(ref64, dtype)
        assert compare(got_new, want, ref64, dtype, K)["ok"]
        assert compare(got_ref, want, ref64, dtype, K)["ok"]
    st, info = hg.get_device_status(0)
    assert st == 0, (st, info)


def test_noalloc_rejects_workspace_beyond_its_scratch(lib):
    # B of 8200 x 4097 needs 8200 * 4160 * 2 bytes (> 64 MiB) once copied into
    # 128-byte rows
    M, N, K = 1, 4097, 8200
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    C = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    st = _call(lib, lib.hgemm_noalloc, A, B, C, M, N, K, "bf16")
    assert st == 1
    assert b"scratch" in lib.hgemm_last_error()
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)  # nothing was enqueued


def test_noalloc_reads_a_in_place_when_its_optional_copy_does_not_fit(lib):
    # A's 8208-byte rows (an odd multiple of 16 bytes) on 224-wide pair tiles:
    # hgemm copies A into 128-byte rows for speed. 8192 x 4160 x 2 bytes do not
    # fit the fixed scratch, so the no-alloc call reads A in place instead of
    # refusing the shape (the copy is not needed for correctness)
    M, N, K = 8192, 4096, 4104
    cfg = hg.Config(cta_group=2, block_n=224)
    assert hg.plan(M, N, K, "bf16", cfg)["repack_a"] == 1
    A = inputs.generate((M, K), "bf16", 38, 0)
    B = inputs.generate((K, N), "bf16", 38, 1)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    hg.hgemm_noalloc(A.cuda(), B.cuda(), C, M, N, K, "bf16", config=cfg)
    torch.cuda.synchronize()
    got = inputs.bits(C.cpu())
    rows = np.unique(np.concatenate([np.random.default_rng(5).integers(0, M, 24), [0, 255, 256, M - 1]]))
    ref, ref64 = oracle.gemm_rows(inputs.bits(A), inputs.bits(B), "bf16", rows)
    r = compare(got[rows], ref, ref64, "bf16", K)
    assert r["ok"], r
    st, info = hg.get_device_status(0)
    assert st == 0, (st, info)


@pytest.mark.parametrize("mode", [2, 3, 4])
def test_noalloc_aligned_shape_with_stream_k(lib, mode):
    # aligned operands; the only workspace is the stream-K partial sums (a
    # stream-K schedule asked for through hgemm_noalloc_ex)
    M, N, K = 128, 2048, 4096
    cfg = hg.Config(stream_k=mode)
    assert hg.plan(M, N, K, "bf16", cfg)["sk_tiles"] > 0
    A = inputs.generate((M, K), "bf16", 34, 0)
    B = inputs.generate((K, N), "bf16", 34, 1)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    hg.hgemm_noalloc(A.cuda(), B.cuda(), C, M, N, K, "bf16", config=cfg)
    torch.cuda.synchronize()
    a, b = inputs.bits(A), inputs.bits(B)
    ref64 = oracle.gemm_f64(a, b, "bf16")
    r = compare(inputs.bits(C.cpu()), oracle.round_rne(ref64, "bf16"), ref64, "bf16", K)
    assert r["ok"], r


@pytest.mark.parametrize("dtype", ["tf32", "e4m3"])
def test_other_dtypes_in_scratch(lib, dtype):
    # B is read in place unless its row pitch is not a multiple of 16 bytes
    # (N = 770 floats, 776 bytes): then it is repacked, here into the fixed
    # scratch array
    import numpy as np
    M, N, K = 512, (770 if dtype == "tf32" else 776), 1024
    assert hg.plan(M, N, K, dtype)["repack_b"] == 1
    if dtype == "tf32":
        A = torch.randn(M, K, device="cuda")
        B = torch.randn(K, N, device="cuda")
        C0 = torch.empty(M, N, device="cuda")
        C1 = torch.empty(M, N, device="cuda")
    else:
        A = (torch.rand(M, K, device="cuda") * 8 - 4).to(torch.float8_e4m3fn)
        B = (torch.rand(K, N, device="cuda") * 8 - 4).to(torch.float8_e4m3fn)
        C0 = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        C1 = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    hg.hgemm(A, B, C0, M, N, K, dtype)
    hg.hgemm_noalloc(A, B, C1, M, N, K, dtype)
    torch.cuda.synchronize()
    assert torch.equal(C0, C1)


# Driver node types (CUgraphNodeType) that allocate or free memory.
_CU_GRAPH_NODE_TYPE_MEM_ALLOC = 10
_CU_GRAPH_NODE_TYPE_MEM_FREE = 11


def _capture_node_types(fn, stream):
    """Record `fn()` (which enqueues on `stream`) by stream capture through the
    driver API and return the type of every node of the captured graph."""
    cu = ctypes.CDLL("libcuda.so.1")
    s = ctypes.c_void_p(stream.cuda_stream)
    assert cu.cuStreamBeginCapture_v2(s, 1) == 0          # CU_STREAM_CAPTURE_MODE_THREAD_LOCAL
    try:
        fn()
    finally:
        graph = ctypes.c_void_p()
        rc = cu.cuStreamEndCapture(s, ctypes.byref(graph))
    assert rc == 0
    try:
        n = ctypes.c_size_t(0)
        assert cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) == 0
        nodes = (ctypes.c_void_p * max(1, n.value))()
        assert cu.cuGraphGetNodes(graph, nodes, ctypes.byref(n)) == 0
        types = []
        for i in range(n.value):
            t = ctypes.c_int(-1)
            assert cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
            types.append(t.value)
        return types
    finally:
        cu.cuGraphDestroy(graph)


def test_noalloc_capture_has_no_allocation_node(lib):
    # K = 1001: A's rows are not 16-byte multiples, so the call repacks A into
    # its workspace; captured, hgemm_noalloc must take that workspace from the
    # fixed array (no allocation or free node), while hgemm draws it from its
    # pool (an allocation node).
    M, N, K = 300, 512, 1001
    A = inputs.generate((M, K), "bf16", 35, 0).cuda()
    B = inputs.generate((K, N), "bf16", 35, 1).cuda()
    assert hg.plan(M, N, K, "bf16")["repack_a"] == 1
    C_eager = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C_cap = torch.full((M, N), 9.0, dtype=torch.bfloat16, device="cuda")
    # the first call on the device looks up the array's address: before any capture
    assert _call(lib, lib.hgemm_noalloc, A, B, C_eager, M, N, K, "bf16") == 0
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        types = _capture_node_types(lambda: _call(lib, lib.hgemm_noalloc, A, B, C_cap, M, N, K, "bf16"), s)
    assert types, "nothing was captured"
    assert _CU_GRAPH_NODE_TYPE_MEM_ALLOC not in types and _CU_GRAPH_NODE_TYPE_MEM_FREE not in types, types
    # the pool-backed entry point, captured the same way, does allocate
    with torch.cuda.stream(s):
        types_pool = _capture_node_types(lambda: _call(lib, lib.hgemm, A, B, C_cap, M, N, K, "bf16"), s)
    assert _CU_GRAPH_NODE_TYPE_MEM_ALLOC in types_pool, types_pool
    torch.cuda.synchronize()
    assert torch.all(C_cap == 9.0)   # a captured call only records work
