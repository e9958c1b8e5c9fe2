"""Failure detection on the GPU without a fault: a bounded wait that runs out
reports HGEMM_ERR_TIMEOUT through the device status word, the kernel returns,
and the context stays usable for the next GEMM."""

import pytest
import torch

import oracle
from half_precision_dense_gb300 import binding as hg
from half_precision_dense_gb300 import inputs
from tests._check import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from half_precision_dense_gb300 import build as hbuild
    hbuild.build()
    hg.load_library()
    hg.get_device_status(0, reset=True)
    yield
    hg.test_inject(0)
    hg.set_timeout_ns(2_000_000_000)
    hg.get_device_status(0, reset=True)


def test_k_split_wait_that_runs_out_reports_timeout_and_context_survives():
    # the K split's reduction: rank 0 of every cluster withholds its "ring
    # free" arrival; the peers' bounded waits run out, every CTA returns
    M, N, K = 128, 2048, 8192
    cfg = hg.Config(block_n=128, split_k=4)
    A = inputs.generate((M, K), "bf16", 41, 0).cuda()
    B = inputs.generate((K, N), "bf16", 41, 1).cuda()
    assert hg.plan(M, N, K, "bf16", cfg)["split_k"] == 4
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    hg.set_timeout_ns(50_000_000)  # 50 ms
    hg.test_inject(2)
    hg.hgemm_ex(A, B, C, M, N, K, "bf16", cfg)
    torch.cuda.synchronize()  # the kernel returned on its own
    st, info = hg.get_device_status(0, reset=True)
    assert st == 5, (st, hex(info))
    role, which = info >> 24, (info >> 16) & 0xFF
    assert role == 3 and which in (96, 97, 98), hex(info)  # the epilogue, in the reduction's waits
    # the context is intact: the next GEMM is correct and reports nothing
    hg.test_inject(0)
    hg.set_timeout_ns(2_000_000_000)
    hg.hgemm_ex(A, B, C, M, N, K, "bf16", cfg)
    torch.cuda.synchronize()
    a, b = inputs.bits(A.cpu()), inputs.bits(B.cpu())
    ref64 = oracle.gemm_f64(a, b, "bf16")
    r = compare(inputs.bits(C.cpu()), oracle.round_rne(ref64, "bf16"), ref64, "bf16", K)
    assert r["ok"], r
    assert hg.get_device_status(0)[0] == 0


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    M, N, K = 512, 1024, 2048  # stream-K over every tile: owners wait for partners' marks
    cfg = hg.Config(stream_k=3)
    A = inputs.generate((M, K), "bf16", 40, 0).cuda()
    B = inputs.generate((K, N), "bf16", 40, 1).cuda()
    assert hg.plan(M, N, K, "bf16", cfg)["sk_tiles"] > 0
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    hg.set_timeout_ns(50_000_000)  # 50 ms
    hg.test_inject(1)
    hg.hgemm_ex(A, B, C, M, N, K, "bf16", cfg)
    torch.cuda.synchronize()  # the kernel returned on its own
    st, info = hg.get_device_status(0, reset=True)
    assert st == 5, (st, hex(info))
    role, which = info >> 24, (info >> 16) & 0xFF
    assert role == 3 and which >= 64, hex(info)  # the epilogue, waiting for a partial-sum mark
    # the context is intact: the next GEMM is correct and reports nothing
    hg.test_inject(0)
    hg.set_timeout_ns(2_000_000_000)
    hg.hgemm_ex(A, B, C, M, N, K, "bf16", cfg)
    torch.cuda.synchronize()
    a, b = inputs.bits(A.cpu()), inputs.bits(B.cpu())
    ref64 = oracle.gemm_f64(a, b, "bf16")
    r = compare(inputs.bits(C.cpu()), oracle.round_rne(ref64, "bf16"), ref64, "bf16", K)
    assert r["ok"], r
    assert hg.get_device_status(0)[0] == 0
