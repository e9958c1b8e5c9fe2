"""CPU oracle for 2-D convolution, the workload the im2col path turns into a GEMM.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import or call this
module: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs
use it. It shares no code with the CUDA library, and it does not use im2col:
it is the convolution's own definition.

What is computed, and where it is defined
-----------------------------------------
* "深度学习加速核心：GEMM优化从分块到TensorCore的实战解析", section 1.1: a
  convolution slides the kernel over the input and takes a pointwise
  multiply-and-sum at every position; im2col rearranges the input feature map
  by the kernel's receptive fields into one large matrix, which turns the
  convolution into a single GEMM (at the cost of that matrix's memory).

Readings (the page gives no layout, stride or padding):
* Layouts are channels-last: input x is N x H x W x C, filters w are
  R x S x C x K (so that w, read as an (R*S*C) x K row-major matrix, is the
  GEMM's B), output y is N x P x Q x K (the GEMM's C, (N*P*Q) x K row-major).
* "Pointwise multiply-and-sum of a sliding window" is cross-correlation (no
  kernel flip), with a stride and symmetric zero padding:
      P = (H + 2 pad - R) / stride + 1,  Q = (W + 2 pad - S) / stride + 1,
      y[n,p,q,k] = sum_{r,s,c} x[n, p*stride - pad + r, q*stride - pad + s, c] * w[r,s,c,k]
  with x taken as 0 outside the image.
* Element types and rounding are the GEMM's: fp16/bf16 inputs, an exact
  (fp64) sum, one round-to-nearest-even into the input type.

The oracle sums over (r, s) explicitly; for each filter tap the sum over c
is one fp64 matrix product (a library step) of the shifted input window with
that tap's C x K filter slice.
"""

from __future__ import annotations

import numpy as np

from .hgemm_oracle import decode, round_rne

__all__ = ["out_size", "conv_f64", "conv", "conv_at"]


def out_size(H: int, W: int, R: int, S: int, stride: int, pad: int):
    P = (H + 2 * pad - R) // stride + 1
    Q = (W + 2 * pad - S) // stride + 1
    return P, Q


def _check(x, w, stride, pad):
    x = np.asarray(x)
    w = np.asarray(w)
    if x.ndim != 4 or w.ndim != 4 or x.shape[3] != w.shape[2]:
        raise ValueError(f"x {x.shape} (N,H,W,C) and w {w.shape} (R,S,C,K) do not match")
    if stride < 1 or pad < 0:
        raise ValueError("stride >= 1 and pad >= 0")
    return x, w


def conv_f64(x, w, dtype: str, stride: int = 1, pad: int = 0) -> np.ndarray:
    """The exact convolution (fp64, N x P x Q x K) of 16-bit patterns x, w."""
    x, w = _check(x, w, stride, pad)
    N, H, W, C = x.shape
    R, S, _, K = w.shape
    P, Q = out_size(H, W, R, S, stride, pad)
    xv = np.zeros((N, H + 2 * pad, W + 2 * pad, C), dtype=np.float64)
    xv[:, pad:pad + H, pad:pad + W, :] = decode(x, dtype)
    wv = decode(w, dtype)
    y = np.zeros((N, max(P, 0), max(Q, 0), K), dtype=np.float64)
    if P <= 0 or Q <= 0:
        return y
    for r in range(R):
        for s in range(S):
            win = xv[:, r:r + stride * (P - 1) + 1:stride, s:s + stride * (Q - 1) + 1:stride, :]
            y += win @ wv[r, s]
    return y


def conv(x, w, dtype: str, stride: int = 1, pad: int = 0) -> np.ndarray:
    """The oracle's output as 16-bit patterns (N x P x Q x K)."""
    return round_rne(conv_f64(x, w, dtype, stride, pad), dtype)


def conv_at(x, w, dtype: str, stride: int, pad: int, points) -> np.ndarray:
    """Exact outputs (fp64, one row of K per point) at output pixels
    ``points`` = [(n, p, q), ...], summed tap by tap from the definition."""
    x, w = _check(x, w, stride, pad)
    N, H, W, C = x.shape
    R, S, _, K = w.shape
    wv = decode(w, dtype)
    out = np.zeros((len(points), K), dtype=np.float64)
    for i, (n, p, q) in enumerate(points):
        for r in range(R):
            h = p * stride - pad + r
            if h < 0 or h >= H:
                continue
            for s in range(S):
                ww = q * stride - pad + s
                if ww < 0 or ww >= W:
                    continue
                out[i] += decode(x[n, h, ww], dtype) @ wv[r, s]
    return out
