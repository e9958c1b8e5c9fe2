"""CPU oracle for the FP8 GEMM variants: per-channel scales, and one scale
per square sub-block.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import or call this
module: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs
use it. It shares no code with the CUDA library.

What is computed, and where it is defined
-----------------------------------------
* "深度学习加速核心：GEMM优化从分块到TensorCore的实战解析", section 4.3: FP8
  comes in two variants, E4M3 (more precision, for weights and activations)
  and E5M2 (more range); FP8 values need scale factors because eight bits
  cover a narrow range. Section 2.3: FP8 quantisation goes with per-layer or
  per-channel ("逐层或逐通道") scale factors, and accumulation stays in a wider
  format.
* "[CUDA 优化实战] hgemm - 超越 cuBLAS", section 1: C = A.B with row-major
  A (M x K), B (K x N), C (M x N), fp32 accumulation, C rounded to nearest
  even in a half-precision type.

Readings (the pages leave these open):
* The formats are the OCP 8-bit floats: E4M3 = 1 sign, 4 exponent (bias 7),
  3 fraction bits, no infinities, S.1111.111 is NaN (largest finite 448);
  E5M2 = 1 sign, 5 exponent (bias 15), 2 fraction bits, IEEE infinities and
  NaNs. A and B share one format.
* Scales are per channel: one fp32 factor per row of A (``a_scale[i]``) and
  one per column of B (``b_scale[j]``). Both are constant along K, so they
  factor out of the sum. The section 4.3 sub-block scales (32 x 32 or
  64 x 64 blocks, varying along K) are the block-scaled variant below.
* C is bfloat16 (the series' output type), rounded once to nearest even.

The oracle is the definition in fp64 (each fp8 x fp8 product is exact):

    C64[i][j] = a_scale[i] * b_scale[j] * sum_k A[i][k] * B[k][j]
    C[i][j]   = RNE_bf16(C64[i][j])

The bf16 rounding is the half-precision oracle's own ``round_rne``.

Block-scaled variant ("深度学习加速核心：GEMM优化从分块到TensorCore的实战解析",
section 4.3: FP8 data is usually scaled block-wise, one factor per 32 x 32
or 64 x 64 sub-block, mapping its values into the format's range; section
5.2, the third mishap: a 16-bit sub-block scale overflowed to infinity, and
32-bit scales fixed it). Readings:
* The value of A's element (i, k) is decode(A[i][k]) * a_scale[i // bs][k // bs]
  and that of B's element (k, j) is decode(B[k][j]) * b_scale[k // bs][j // bs]:
  a_scale is ceil(M / bs) x ceil(K / bs), b_scale ceil(K / bs) x ceil(N / bs),
  both row-major fp32; bs is 32 or 64 (the two sizes the page names). The
  last block of a dimension that is not a multiple of bs is partial.
* The product is that of the dequantised matrices, C rounded once to bf16.
  The oracle is that definition written out in fp64 (dequantise, then the
  plain product; the 28-bit dequantised values are exact in fp64):

    C64 = (decode(A) * a_scale[i // bs][k // bs]) @ (decode(B) * b_scale[k // bs][j // bs])
    C   = RNE_bf16(C64)
"""

from __future__ import annotations

import numpy as np

from .hgemm_oracle import round_rne

__all__ = ["FORMATS", "decode", "gemm_f64", "gemm", "abs_gemm", "tolerance", "SCALE_BLOCKS",
           "scale_grid", "dequantise_a", "dequantise_b", "gemm_blockscaled_f64", "gemm_blockscaled",
           "abs_gemm_blockscaled", "tolerance_blockscaled"]

# name -> (exponent bits, fraction bits, bias, has_infinity)
FORMATS = {"e4m3": (4, 3, 7, False), "e5m2": (5, 2, 15, True)}


def decode(b: np.ndarray, fmt: str) -> np.ndarray:
    """Values (fp64) of 8-bit patterns ``b`` (uint8) in ``fmt``.

    normal:    (-1)^s * (2^f + m) * 2^(e - bias - f)
    subnormal: (-1)^s * m * 2^(1 - bias - f)          (exponent field 0)
    E5M2 exponent all ones: +-inf (m = 0) or NaN; E4M3: only S.1111.111 is NaN.
    """
    if fmt not in FORMATS:
        raise ValueError(f"fmt must be one of {sorted(FORMATS)}")
    eb, fb, bias, has_inf = FORMATS[fmt]
    x = np.asarray(b).astype(np.int64)
    s = (x >> 7) & 1
    e = (x >> fb) & ((1 << eb) - 1)
    m = x & ((1 << fb) - 1)
    sub = e == 0
    sig = np.where(sub, m, m + (1 << fb)).astype(np.float64)
    ex = np.where(sub, 1 - bias - fb, e - bias - fb)
    mag = np.ldexp(sig, ex)
    e_max = (1 << eb) - 1
    if has_inf:
        special = e == e_max
        mag = np.where(special, np.where(m == 0, np.inf, np.nan), mag)
    else:
        mag = np.where((e == e_max) & (m == (1 << fb) - 1), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def _check(A, B, a_scale, b_scale):
    A = np.asarray(A)
    B = np.asarray(B)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shapes {A.shape} and {B.shape} do not chain (M x K) . (K x N)")
    if A.dtype != np.uint8 or B.dtype != np.uint8:
        raise TypeError("operands are uint8 bit patterns")
    M, N = A.shape[0], B.shape[1]
    sa = np.ones(M) if a_scale is None else np.asarray(a_scale, dtype=np.float32).astype(np.float64)
    sb = np.ones(N) if b_scale is None else np.asarray(b_scale, dtype=np.float32).astype(np.float64)
    if sa.shape != (M,) or sb.shape != (N,):
        raise ValueError("a_scale has one entry per row of A, b_scale one per column of B")
    return A, B, sa, sb


def gemm_f64(A, B, fmt: str, a_scale=None, b_scale=None) -> np.ndarray:
    """a_scale[i] * b_scale[j] * sum_k A[i,k] * B[k,j] in fp64 (M x N)."""
    A, B, sa, sb = _check(A, B, a_scale, b_scale)
    if A.shape[1] == 0:
        return np.zeros((A.shape[0], B.shape[1]), dtype=np.float64)
    return (decode(A, fmt) @ decode(B, fmt)) * sa[:, None] * sb[None, :]


def gemm(A, B, fmt: str, a_scale=None, b_scale=None) -> np.ndarray:
    """The oracle's C as bfloat16 bit patterns (uint16)."""
    return round_rne(gemm_f64(A, B, fmt, a_scale, b_scale), "bf16")


def abs_gemm(A, B, fmt: str, a_scale=None, b_scale=None) -> np.ndarray:
    """|a_scale[i] * b_scale[j]| * sum_k |A[i,k]| |B[k,j]| (fp64)."""
    A, B, sa, sb = _check(A, B, a_scale, b_scale)
    if A.shape[1] == 0:
        return np.zeros((A.shape[0], B.shape[1]), dtype=np.float64)
    return (np.abs(decode(A, fmt)) @ np.abs(decode(B, fmt))) * np.abs(sa)[:, None] * np.abs(sb)[None, :]


def tolerance(S: np.ndarray, C64: np.ndarray, K: int) -> np.ndarray:
    """Per-element bound on |C_gpu - C_oracle| (both as values): the GPU sums
    K exact products in fp32 in its own order ((K - 1) additions, relative
    error <= 2^-23 each), multiplies by the two scales in fp32 (two more
    roundings) and rounds once to bf16; the oracle rounds the exact value once.
    The two may then differ by the fp32 error bound, (K + 1) 2^-23 S, plus one
    bf16 ulp of |C64| (the two bf16 roundings can fall on either side of a
    rounding boundary)."""
    u = 2.0 ** -23
    ref = np.abs(np.asarray(C64, dtype=np.float64))
    e = np.frexp(np.where(ref > 0, ref, 1.0))[1] - 1
    ulp_bf16 = np.ldexp(1.0, np.maximum(e, -126) - 7)
    return (K + 1) * u * S + ulp_bf16


# ---------------------------------------------------------------------------
# Block-scaled variant: one fp32 factor per bs x bs sub-block of A and of B.

SCALE_BLOCKS = (32, 64)


def scale_grid(rows: int, cols: int, block: int) -> tuple:
    """Shape of the scale array of a rows x cols operand: one factor per
    block x block sub-block, the last block of each dimension partial."""
    return (-(-rows // block), -(-cols // block))


def _check_blocks(A, B, a_scale, b_scale, block):
    A = np.asarray(A)
    B = np.asarray(B)
    if block not in SCALE_BLOCKS:
        raise ValueError(f"block must be one of {SCALE_BLOCKS}")
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shapes {A.shape} and {B.shape} do not chain (M x K) . (K x N)")
    if A.dtype != np.uint8 or B.dtype != np.uint8:
        raise TypeError("operands are uint8 bit patterns")
    M, K = A.shape
    N = B.shape[1]
    sa = np.asarray(a_scale, dtype=np.float32).astype(np.float64)
    sb = np.asarray(b_scale, dtype=np.float32).astype(np.float64)
    if sa.shape != scale_grid(M, K, block) or sb.shape != scale_grid(K, N, block):
        raise ValueError(f"a_scale must be {scale_grid(M, K, block)} and b_scale {scale_grid(K, N, block)}")
    return A, B, sa, sb


def dequantise_a(A, fmt: str, a_scale, block: int) -> np.ndarray:
    """Values of A (M x K, fp64): decode(A[i][k]) * a_scale[i // block][k // block]."""
    A = np.asarray(A)
    sa = np.asarray(a_scale, dtype=np.float32).astype(np.float64)
    i = np.arange(A.shape[0]) // block
    k = np.arange(A.shape[1]) // block
    return decode(A, fmt) * sa[i[:, None], k[None, :]]


def dequantise_b(B, fmt: str, b_scale, block: int) -> np.ndarray:
    """Values of B (K x N, fp64): decode(B[k][j]) * b_scale[k // block][j // block]."""
    B = np.asarray(B)
    sb = np.asarray(b_scale, dtype=np.float32).astype(np.float64)
    k = np.arange(B.shape[0]) // block
    j = np.arange(B.shape[1]) // block
    return decode(B, fmt) * sb[k[:, None], j[None, :]]


def gemm_blockscaled_f64(A, B, fmt: str, a_scale, b_scale, block: int) -> np.ndarray:
    """The product of the dequantised operands, in fp64 (M x N)."""
    A, B, sa, sb = _check_blocks(A, B, a_scale, b_scale, block)
    if A.shape[1] == 0:
        return np.zeros((A.shape[0], B.shape[1]), dtype=np.float64)
    return dequantise_a(A, fmt, sa, block) @ dequantise_b(B, fmt, sb, block)


def gemm_blockscaled(A, B, fmt: str, a_scale, b_scale, block: int) -> np.ndarray:
    """The oracle's block-scaled C as bfloat16 bit patterns (uint16)."""
    return round_rne(gemm_blockscaled_f64(A, B, fmt, a_scale, b_scale, block), "bf16")


def abs_gemm_blockscaled(A, B, fmt: str, a_scale, b_scale, block: int) -> np.ndarray:
    """sum_k |A64[i][k]| |B64[k][j]| of the dequantised operands (fp64)."""
    A, B, sa, sb = _check_blocks(A, B, a_scale, b_scale, block)
    if A.shape[1] == 0:
        return np.zeros((A.shape[0], B.shape[1]), dtype=np.float64)
    return np.abs(dequantise_a(A, fmt, sa, block)) @ np.abs(dequantise_b(B, fmt, sb, block))


def tolerance_blockscaled(S: np.ndarray, C64: np.ndarray, K: int, block: int) -> np.ndarray:
    """Per-element bound on |C_gpu - C_oracle| (both as values) for a GPU that
    sums each K block's exact fp8 products in fp32 (in any order: fewer than K
    additions in all, relative error <= 2^-23 each), forms each block's factor
    a_scale * b_scale in fp32 and adds factor * partial into an fp32
    accumulator (one rounding per block, ceil(K / block) blocks), then rounds
    once to bf16: (K + ceil(K / block) + 2) 2^-23 S, with S the sum of
    |A64| |B64|, plus one bf16 ulp of |C64| for the two roundings to bf16."""
    u = 2.0 ** -23
    nkb = -(-int(K) // int(block))
    ref = np.abs(np.asarray(C64, dtype=np.float64))
    e = np.frexp(np.where(ref > 0, ref, 1.0))[1] - 1
    ulp_bf16 = np.ldexp(1.0, np.maximum(e, -126) - 7)
    return (K + nkb + 2) * u * S + ulp_bf16
