"""GPU parity of the im2col convolution (hgemm_conv2d) against the
convolution oracle (the definition, not im2col) on seeded inputs: every
output within the GEMM's tolerance, bit-exact on small integers. Shapes cover
1x1 / 3x3 / 5x5 / 7x1 filters, strides 1-3, zero and non-zero padding,
channel counts that are and are not multiples of 8 (vector and element im2col
copies), ragged output tiles, and a ResNet-style layer sampled at full size."""

import numpy as np
import pytest
import torch

from half_precision_dense_gb300 import binding as hg
from half_precision_dense_gb300 import inputs
from oracle import conv_oracle as co
from tests._check import compare

pytestmark = pytest.mark.gpu


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


def tensors(N, H, W, C, R, S, K, dtype, seed):
    x = inputs.generate((1, N * H * W * C), dtype, seed, 0).view(N, H, W, C)
    w = inputs.generate((1, R * S * C * K), dtype, seed, 1).view(R, S, C, K)
    return x, w


def run_gpu(x, w, stride, pad):
    return hg.conv2d_nhwc(x.cuda(), w.cuda(), stride, pad).cpu()


CASES = [
    # (N, H, W, C, R, S, K, stride, pad); C a multiple of 64 takes the
    # implicit GEMM (TMA im2col), other C the explicit im2col matrix
    (2, 9, 11, 64, 3, 3, 24, 1, 1),
    (2, 13, 10, 128, 5, 5, 40, 2, 2),
    (1, 20, 20, 64, 7, 1, 8, 3, 3),
    (3, 8, 8, 192, 3, 3, 264, 2, 1),
    (1, 15, 17, 64, 2, 4, 72, 1, 0),
    (2, 9, 11, 16, 3, 3, 24, 1, 1),
    (1, 14, 14, 64, 1, 1, 96, 1, 0),
    (2, 13, 10, 8, 5, 5, 40, 2, 2),
    (1, 17, 9, 3, 3, 3, 16, 1, 0),      # C = 3: element-wise im2col copies, R*S*C = 27
    (1, 20, 20, 12, 7, 1, 8, 3, 3),
    (3, 8, 8, 32, 3, 3, 264, 2, 1),     # ragged output tile in N (K = 264)
    (2, 7, 9, 40, 1, 1, 48, 1, 0),      # pointwise: straight to the GEMM
    (2, 7, 9, 40, 1, 1, 48, 2, 0),      # strided pointwise: im2col
    (1, 6, 6, 12, 1, 1, 20, 1, 0),      # pointwise with C * 2 bytes not a 16-byte pitch
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", CASES)
def test_conv_matches_definition(case, dtype):
    N, H, W, C, R, S, K, stride, pad = case
    x, w = tensors(N, H, W, C, R, S, K, dtype, 2)
    got = inputs.bits(run_gpu(x, w, stride, pad).reshape(-1, K))
    xb, wb = inputs.bits(x.reshape(1, -1)).reshape(x.shape), inputs.bits(w.reshape(1, -1)).reshape(w.shape)
    ref64 = co.conv_f64(xb, wb, dtype, stride, pad).reshape(-1, K)
    ref = co.conv(xb, wb, dtype, stride, pad).reshape(-1, K)
    r = compare(got, ref, ref64, dtype, R * S * C)
    assert r["ok"], r


@pytest.mark.parametrize("mode", [0, 1])
def test_implicit_and_explicit_paths_agree(mode):
    # the same C % 64 == 0 shapes through either path
    hg.conv2d_set_mode(mode)
    try:
        for case in [(2, 9, 11, 64, 3, 3, 24, 1, 1), (3, 8, 8, 192, 3, 3, 264, 2, 1)]:
            test_conv_matches_definition(case, "bf16")
    finally:
        hg.conv2d_set_mode(0)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_small_integers_bit_exact(dtype):
    rng = np.random.default_rng(3)
    N, H, W, C, R, S, K = 2, 10, 7, 5, 3, 3, 20
    t = inputs.TORCH_DTYPES[dtype]
    x = torch.from_numpy(rng.integers(-2, 3, (N, H, W, C)).astype(np.float32)).to(t)
    w = torch.from_numpy(rng.integers(-2, 3, (R, S, C, K)).astype(np.float32)).to(t)
    got = run_gpu(x, w, 1, 1)
    xb, wb = inputs.bits(x.reshape(1, -1)).reshape(x.shape), inputs.bits(w.reshape(1, -1)).reshape(w.shape)
    assert np.array_equal(inputs.bits(got.reshape(1, -1)).reshape(got.shape), co.conv(xb, wb, dtype, 1, 1))


@pytest.mark.parametrize("shape", [(2, 9, 9, 16, 3, 3, 32, 1, 1),     # explicit im2col (C = 16)
                                   (2, 9, 9, 64, 3, 3, 32, 1, 1),     # implicit GEMM (C % 32 == 0)
                                   (1, 11, 8, 32, 5, 3, 24, 2, 2)])
def test_tf32_conv(shape):
    from oracle import tf32_oracle as tf
    N, H, W, C, R, S, K, stride, pad = shape
    x = inputs.generate((1, N * H * W * C), "f32", 4, 0).view(N, H, W, C)
    w = inputs.generate((1, R * S * C * K), "f32", 4, 1).view(R, S, C, K)
    got = run_gpu(x, w, stride, pad).numpy().reshape(-1, K)
    # the definition on tf32-truncated operands: im2col on the CPU is only a
    # gather here; products and sums are the TF32 oracle's
    xp = np.pad(x.numpy(), ((0, 0), (pad, pad), (pad, pad), (0, 0)))
    P, Q = co.out_size(H, W, R, S, stride, pad)
    cols = np.stack([xp[:, r:r + stride * (P - 1) + 1:stride, s:s + stride * (Q - 1) + 1:stride, :]
                     for r in range(R) for s in range(S)], axis=3)
    A = np.ascontiguousarray(cols.reshape(N * P * Q, R * S * C))
    Bm = np.ascontiguousarray(w.numpy().reshape(R * S * C, K))
    ref = tf.gemm(A, Bm)
    tol = tf.tolerance(tf.abs_gemm(A, Bm), ref, R * S * C)
    assert np.all(np.abs(got.astype(np.float64) - ref) <= tol)


def test_resnet_layer_sampled():
    # 32 x 28 x 28 x 256 input, 3 x 3 x 256 x 512 filters, stride 1, pad 1:
    # sampled output pixels, every channel, against the definition
    N, H, W, C, R, S, K = 32, 28, 28, 256, 3, 3, 512
    dtype = "bf16"
    x, w = tensors(N, H, W, C, R, S, K, dtype, 5)
    got = run_gpu(x, w, 1, 1)
    xb, wb = inputs.bits(x.reshape(1, -1)).reshape(x.shape), inputs.bits(w.reshape(1, -1)).reshape(w.shape)
    rng = np.random.default_rng(6)
    pts = [(0, 0, 0), (31, 27, 27), (5, 0, 13), (7, 27, 0)] + \
          [tuple(int(v) for v in (rng.integers(0, N), rng.integers(0, 28), rng.integers(0, 28))) for _ in range(28)]
    ref64 = co.conv_at(xb, wb, dtype, 1, 1, pts)
    from oracle import round_rne
    ref = round_rne(ref64, dtype)
    gb = inputs.bits(got.reshape(1, -1)).reshape(got.shape)
    g = np.stack([gb[n, p, q] for (n, p, q) in pts])
    r = compare(g, ref, ref64, dtype, R * S * C)
    assert r["ok"], r


def test_degenerate_and_invalid():
    x = torch.zeros(1, 2, 2, 4, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(3, 3, 4, 8, dtype=torch.bfloat16, device="cuda")
    y = hg.conv2d_nhwc(x, w, 1, 0)          # the filter does not fit: no output pixels
    assert y.numel() == 0
    with pytest.raises(hg.HgemmError):
        hg.hgemm_conv2d(x, w, x, 1, 2, 2, 4, 8, 3, 3, 0, 0, "bf16")   # stride 0
