"""CPU oracle for the dense half-precision GEMM C = A.B.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import or call this
module: only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it. It shares no code with the
CUDA library (no kernels, headers, tables or helpers); the only module both
sides read is the seeded input generator.

What is computed, and where it is defined
-----------------------------------------
* "[CUDA 优化实战] hgemm - 超越 cuBLAS", section 1 (hgemm_naive): A is M x K and
  B is K x N, both row-major ("A/B 都行优先"; element (r, c) of A at
  ``a[r*k + c]``, of B at ``b[r*n + c]``), fp16 or bf16 entries, products
  accumulated in fp32 by ``mma.sync ... .f32.bf16.bf16.f32`` /
  ``.f32.f16.f16.f32``, and the result written to C (``c[r*n + c]``) through
  ``__float22half2_rn`` / ``__float22bfloat162_rn``, i.e. rounded to nearest,
  ties to even, in the input dtype.
* "CUDA GEMM 优化实践笔记", second-level tiling section: C = A x B with
  A in R^{M x K}, B in R^{K x N}, C in R^{M x N}; each C_ij needs row i of A and
  column j of B; 2MNK floating-point operations in total.

The method is exact up to the order of its fp32 additions, so the oracle is
the plain definition written out in higher precision:

    C64[i][j] = sum_k  A[i][k] * B[k][j]          (fp64)
    C[i][j]   = RNE_dtype(C64[i][j])               (one rounding)

Each product of two fp16/bf16 values is exact in fp64 (at most 2 x 11
significant bits), so the only fp64 error is in the sum, about 2**-53 relative
per addition, far below either output format's resolution. The sum itself is
taken by numpy's fp64 matrix product (a library primitive serving as one
step); decoding the 16-bit operands and the final rounding are written out
here from the IEEE 754 binary16 / bfloat16 definitions, bit by bit, and do not
use any library conversion.

Readings where the pages are silent (the full list is in the design notes):
* Out-of-range tile elements contribute zero ("CUDA GEMM 优化实践笔记", the
  register-tiled kernel's bounds-checked loads fill 0.0f), so a GEMM of any
  M, N, K is the plain sum above; K = 0 gives C = 0; M = 0 or N = 0 is empty.
* Overflow rounds to +-inf, gradual underflow is kept, NaN is the canonical
  quiet NaN.
"""

from __future__ import annotations

import numpy as np

__all__ = ["FORMATS", "decode", "round_rne", "gemm_f64", "gemm", "gemm_rows",
           "gemm_cols", "flops"]


class _Fmt:
    def __init__(self, name, ebits, p, bias):
        self.name = name
        self.ebits = ebits          # exponent field width
        self.p = p                  # stored mantissa bits (precision p + 1)
        self.bias = bias
        self.emin = 1 - bias        # smallest normal exponent
        self.emax = bias            # largest finite exponent
        self.exp_all_ones = (1 << ebits) - 1
        self.sign_shift = ebits + p
        self.qnan = (self.exp_all_ones << p) | (1 << (p - 1))
        self.inf = self.exp_all_ones << p


# IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits.
# bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits (the top half of binary32).
FORMATS = {"f16": _Fmt("f16", 5, 10, 15), "bf16": _Fmt("bf16", 8, 7, 127)}


def _fmt(dtype: str) -> _Fmt:
    try:
        return FORMATS[dtype]
    except KeyError:
        raise ValueError(f"dtype must be one of {sorted(FORMATS)}") from None


def decode(b: np.ndarray, dtype: str) -> np.ndarray:
    """Values (fp64) of 16-bit patterns ``b`` (uint16) in format ``dtype``.

    normal:    (-1)^s * (2^p + m) * 2^(e - bias - p)
    subnormal: (-1)^s * m * 2^(emin - p)         (exponent field 0)
    e all ones: +-inf (m = 0) or NaN.
    """
    f = _fmt(dtype)
    x = np.asarray(b).astype(np.int64)
    s = (x >> f.sign_shift) & 1
    e = (x >> f.p) & f.exp_all_ones
    m = x & ((1 << f.p) - 1)
    sub = e == 0
    special = e == f.exp_all_ones
    sig = np.where(sub, m, m + (1 << f.p)).astype(np.float64)
    ex = np.where(sub, f.emin - f.p, e - f.bias - f.p)
    ex = np.where(special, 0, ex)
    mag = np.ldexp(sig, ex)
    mag = np.where(special, np.where(m == 0, np.inf, np.nan), mag)
    return np.where(s == 1, -mag, mag)


def round_rne(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 values ``x`` once, to nearest with ties to even, into ``dtype``.

    For |x| with exponent e = floor(log2|x|), clamped below at emin, the
    representable neighbours are multiples of q = 2^(e - p). |x| / q is exact
    (a power-of-two scaling), is rounded to the nearest integer n with ties to
    even, and n * q is the result. n = 2^(p+1) carries into the next binade;
    a result above the largest finite binade is infinity.
    """
    f = _fmt(dtype)
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    inf = np.isinf(a)
    zero = a == 0
    ok = ~(nan | inf | zero)
    a1 = np.where(ok, a, 1.0)
    _, E = np.frexp(a1)                      # a1 = frac * 2^E, frac in [0.5, 1)
    e = np.maximum(E - 1, f.emin)
    n = np.rint(np.ldexp(a1, -(e - f.p)))    # numpy rint: half to even
    carry = n >= float(1 << (f.p + 1))
    e = np.where(carry, e + 1, e)
    n = np.where(carry, n * 0.5, n).astype(np.int64)
    sub = n < (1 << f.p)                     # only when e == emin
    exp_field = np.where(sub, 0, e + f.bias)
    mant = np.where(sub, n, n - (1 << f.p))
    out = (exp_field << f.p) | mant
    out = np.where(e > f.emax, f.inf, out)
    out = np.where(zero, 0, out)
    out = np.where(inf, f.inf, out)
    out = np.where(neg, out | (1 << f.sign_shift), out)
    out = np.where(nan, f.qnan, out)
    return out.astype(np.uint16)


def _check_operands(A: np.ndarray, B: np.ndarray):
    A = np.asarray(A)
    B = np.asarray(B)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shapes {A.shape} and {B.shape} do not chain (M x K) . (K x N)")
    if A.dtype != np.uint16 or B.dtype != np.uint16:
        raise TypeError("operands are uint16 bit patterns")
    return A, B


def gemm_f64(A: np.ndarray, B: np.ndarray, dtype: str) -> np.ndarray:
    """The unrounded product sum_k A[i,k] * B[k,j] in fp64 (M x N)."""
    A, B = _check_operands(A, B)
    M, K = A.shape
    N = B.shape[1]
    if K == 0:
        return np.zeros((M, N), dtype=np.float64)
    return decode(A, dtype) @ decode(B, dtype)


def gemm(A: np.ndarray, B: np.ndarray, dtype: str) -> np.ndarray:
    """C = RNE_dtype(A . B) as uint16 bit patterns (M x N)."""
    return round_rne(gemm_f64(A, B, dtype), dtype)


def gemm_rows(A: np.ndarray, B: np.ndarray, dtype: str, rows) -> tuple[np.ndarray, np.ndarray]:
    """Rows ``rows`` of C, every column: (bits, fp64) each len(rows) x N."""
    A, B = _check_operands(A, B)
    rows = np.asarray(rows, dtype=np.int64)
    c64 = gemm_f64(A[rows, :], B, dtype)
    return round_rne(c64, dtype), c64


def gemm_cols(A: np.ndarray, B: np.ndarray, dtype: str, cols) -> tuple[np.ndarray, np.ndarray]:
    """Columns ``cols`` of C, every row: (bits, fp64) each M x len(cols)."""
    A, B = _check_operands(A, B)
    cols = np.asarray(cols, dtype=np.int64)
    c64 = gemm_f64(A, B[:, cols], dtype)
    return round_rne(c64, dtype), c64


def flops(M: int, N: int, K: int) -> int:
    """2MNK: one multiply and one add per (i, j, k) ("CUDA GEMM 优化实践笔记",
    second-level tiling section; "深度学习加速核心：GEMM优化从分块到TensorCore的实战解析",
    section 1.2's 4096^3 x 2 example)."""
    return 2 * int(M) * int(N) * int(K)
