"""CPU oracle for the TF32 GEMM variant C = A.B (fp32 in, fp32 out).

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import or call this
module: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs
use it. It shares no code with the CUDA library.

What is computed, and where it is defined
-----------------------------------------
* "[CUDA 优化实战] hgemm - 超越 cuBLAS", section 1: the series' previous kernel
  used the ``m16n8k8`` tensor-core shape with A and B of type tf32 (the
  half-precision kernel "changes the a/b type from tf32 to f16/bf16"); the
  cp.async / smem pipeline is the same. The product is the same C = A.B with
  row-major A (M x K), B (K x N) and C (M x N), accumulated in fp32.
* "CUDA GEMM 优化实践笔记", second-level tiling section: C = A x B, 2MNK flops.

Readings (the pages name the format, not its arithmetic):
* TF32 keeps the sign, the 8 exponent bits and the top 10 of the 23 fraction
  bits of an fp32 value: a tf32 operand is the fp32 value with its low 13
  fraction bits cleared (truncation toward zero; the tensor core reads fp32
  words and ignores those bits).
* Products of two tf32 values (at most 11 x 11 significant bits) are exact in
  fp32; they are accumulated in fp32 and C is that fp32 accumulator, with no
  further rounding to a narrower type.

So the oracle is the plain definition on the truncated operands, in fp64:

    A32[i][k] = trunc_tf32(A[i][k]),  B32[k][j] = trunc_tf32(B[k][j])
    C64[i][j] = sum_k A32[i][k] * B32[k][j]       (exact products, fp64 sum)
    C[i][j]   = RNE_fp32(C64[i][j])

The fp32 rounding of the fp64 sum is numpy's float64 -> float32 conversion
(round to nearest, ties to even; a library routine used as one step). The GPU
sums in fp32 in an order of its own, so parity is a tolerance derived from
fp32 accumulation (see ``tolerance``).
"""

from __future__ import annotations

import numpy as np

__all__ = ["trunc_tf32", "gemm_f64", "gemm", "abs_gemm", "tolerance"]

_LOW13 = np.uint32((1 << 13) - 1)


def trunc_tf32(x: np.ndarray) -> np.ndarray:
    """fp32 values with the low 13 fraction bits cleared (fp32 result).

    Infinities and zeros are unchanged; a NaN whose payload sits only in the
    cleared bits would become infinity, which the GEMM inputs never contain.
    """
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (bits & ~_LOW13).view(np.float32)


def _check(A: np.ndarray, B: np.ndarray):
    A = np.asarray(A)
    B = np.asarray(B)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shapes {A.shape} and {B.shape} do not chain (M x K) . (K x N)")
    if A.dtype != np.float32 or B.dtype != np.float32:
        raise TypeError("operands are fp32 arrays")
    return A, B


def gemm_f64(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """sum_k trunc(A[i,k]) * trunc(B[k,j]) in fp64 (M x N)."""
    A, B = _check(A, B)
    if A.shape[1] == 0:
        return np.zeros((A.shape[0], B.shape[1]), dtype=np.float64)
    return trunc_tf32(A).astype(np.float64) @ trunc_tf32(B).astype(np.float64)


def gemm(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """The oracle's C (fp32): the fp64 sum rounded once to fp32."""
    return gemm_f64(A, B).astype(np.float32)


def abs_gemm(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """sum_k |trunc(A[i,k])| * |trunc(B[k,j])| (fp64): the scale of each sum."""
    A, B = _check(A, B)
    if A.shape[1] == 0:
        return np.zeros((A.shape[0], B.shape[1]), dtype=np.float64)
    return np.abs(trunc_tf32(A).astype(np.float64)) @ np.abs(trunc_tf32(B).astype(np.float64))


def tolerance(S: np.ndarray, C_ref: np.ndarray, K: int) -> np.ndarray:
    """Per-element bound on |C_gpu - C_ref| for an fp32 accumulation of K
    exact products whose absolute values sum to S.

    Any order of K - 1 fp32 additions, each rounding (or truncating) with
    relative error at most u = 2^-23, stays within (K - 1) u S of the exact
    sum (the standard recursive-summation bound, first order); the reference
    itself is rounded once (half an fp32 ulp), and 2 ulp of |C_ref| more cover
    the GPU's own final rounding.
    """
    u = 2.0 ** -23
    ref = np.abs(np.asarray(C_ref, dtype=np.float64))
    ulp = np.ldexp(1.0, np.maximum(np.frexp(np.where(ref > 0, ref, 1.0))[1] - 1, -126) - 23)
    return max(K - 1, 0) * u * S + 2.0 * ulp
