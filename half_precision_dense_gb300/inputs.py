"""Seeded synthetic inputs for the dense half-precision GEMM.

This module is shared by the CPU oracle's tests and by the GPU tests and the
benchmark, so that both sides read exactly the same operand bits. It holds no
part of the GEMM's arithmetic: it only draws numbers and narrows them to the
operand dtype.

Generator: a counter-based SplitMix64 stream (Steele, Lea & Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014). Element ``e`` of
tensor ``t`` (A = 0, B = 1) under seed ``s`` is the ``e``-th output of the
stream whose state starts at ``key = s * 2**40 + t * 2**36``:

    z = key + (e + 1) * 0x9E3779B97F4A7C15            (mod 2**64)
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9          (mod 2**64)
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB          (mod 2**64)
    out = z ^ (z >> 31)

Distributions (the recipes the workloads name):

* ``uniform``: entries in [-1, 1). The top 24 bits ``k`` of ``out`` give
  ``k / 2**23 - 1``, which fp32 holds exactly, so the only rounding is the
  single round-to-nearest-even step from fp32 to the operand dtype (values
  just below 1 may round to exactly 1.0; that is accepted).
* ``normal``: N(0, sigma**2) by the Box-Muller transform on consecutive pairs
  of outputs (elements 2j and 2j+1 share a pair), computed in fp64, scaled by
  sigma, narrowed to fp32 and then to the operand dtype.

The narrowing to fp16/bf16 uses PyTorch's conversion (round to nearest even).
"""

from __future__ import annotations

import numpy as np
import torch

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)

TORCH_DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}

# Elements generated per chunk: bounds the temporaries to a few hundred MB.
_CHUNK = 1 << 24


def splitmix64(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the stream for (seed, tensor_id), as uint64."""
    if not (0 <= seed < (1 << 24) and 0 <= tensor_id < 16):
        raise ValueError("seed must be in [0, 2**24) and tensor_id in [0, 16)")
    if start < 0 or count < 0 or start + count > (1 << 36):
        raise ValueError("element index out of the stream's range")
    key = np.uint64((seed << 40) | (tensor_id << 36))
    with np.errstate(over="ignore"):
        e = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = key + e * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
        z = z ^ (z >> np.uint64(31))
    return z


def _uniform_f32(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    k = (splitmix64(seed, tensor_id, start, count) >> np.uint64(40)).astype(np.int64)
    return ((k - (1 << 23)).astype(np.float32)) * np.float32(2.0 ** -23)


def _normal_f32(seed: int, tensor_id: int, start: int, count: int, sigma: float) -> np.ndarray:
    # Box-Muller needs whole pairs: widen to even boundaries, then trim.
    lo = start - (start & 1)
    hi = start + count + ((start + count) & 1)
    x = splitmix64(seed, tensor_id, lo, hi - lo)
    x1 = x[0::2]
    x2 = x[1::2]
    u1 = ((x1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (x2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)  # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * np.pi * u2
    out = np.empty(hi - lo, dtype=np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    out = out[start - lo:start - lo + count] * sigma
    return out.astype(np.float32)


def generate(shape, dtype: str, seed: int, tensor_id: int, dist: str = "uniform",
             sigma: float = 1.0) -> torch.Tensor:
    """A contiguous CPU tensor of ``shape`` in ``dtype`` ("bf16", "f16" or "f32";
    the uniform draw k / 2^23 - 1 is exact in f32).

    Elements are numbered in row-major order; element ``e`` is the ``e``-th
    stream output, so a sub-block of a large matrix can be regenerated alone.
    """
    if dtype not in TORCH_DTYPES:
        raise ValueError(f"dtype must be one of {sorted(TORCH_DTYPES)}")
    rows, cols = int(shape[0]), int(shape[1])
    n = rows * cols
    out = torch.empty(n, dtype=TORCH_DTYPES[dtype])
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        if dist == "uniform":
            f = _uniform_f32(seed, tensor_id, s, c)
        elif dist == "normal":
            f = _normal_f32(seed, tensor_id, s, c, sigma)
        else:
            raise ValueError("dist must be 'uniform' or 'normal'")
        out[s:s + c] = torch.from_numpy(f).to(TORCH_DTYPES[dtype])
    return out.view(rows, cols)


def bits(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a CPU fp16/bf16 tensor, as a uint16 numpy array."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray, dtype: str) -> torch.Tensor:
    """A CPU tensor of ``dtype`` holding the uint16 bit patterns ``b``."""
    arr = np.ascontiguousarray(b, dtype=np.uint16)
    return torch.from_numpy(arr.view(np.int16).copy()).view(TORCH_DTYPES[dtype])


# The workloads: (name, M, N, K, dtype, dist, sigma, seed).
WORKLOADS = {
    "square256_bf16": (256, 256, 256, "bf16", "uniform", 1.0, 0),
    "square4096_f16": (4096, 4096, 4096, "f16", "uniform", 1.0, 1),
    "square4096_bf16": (4096, 4096, 4096, "bf16", "uniform", 1.0, 1),
    "square8192_bf16": (8192, 8192, 8192, "bf16", "normal", 1.0, 2),
    "mlp_up_bf16": (16384, 14336, 4096, "bf16", "normal", 0.02, 3),
    "mlp_down_bf16": (16384, 4096, 14336, "bf16", "normal", 0.02, 3),
    "skinny_bf16": (128, 8192, 8192, "bf16", "uniform", 1.0, 4),
    "tails_bf16": (1000, 4095, 4104, "bf16", "uniform", 1.0, 4),
    "shortk_bf16": (4096, 4096, 64, "bf16", "uniform", 1.0, 4),
}


def workload_operands(name: str):
    """(A, B, meta) CPU tensors for a named workload; meta = (M, N, K, dtype)."""
    M, N, K, dtype, dist, sigma, seed = WORKLOADS[name]
    A = generate((M, K), dtype, seed, 0, dist, sigma)
    B = generate((K, N), dtype, seed, 1, dist, sigma)
    return A, B, (M, N, K, dtype)


FP8_TORCH = {"e4m3": "float8_e4m3fn", "e5m2": "float8_e5m2"}


def generate_fp8(shape, fmt: str, seed: int, tensor_id: int, spread: float = 8.0):
    """8-bit patterns (uint8 numpy array) of ``shape``: the uniform stream
    scaled to [-spread, spread) and rounded to the fp8 format by PyTorch."""
    rows, cols = int(shape[0]), int(shape[1])
    f = _uniform_f32(seed, tensor_id, 0, rows * cols) * np.float32(spread)
    t = torch.from_numpy(f).to(getattr(torch, FP8_TORCH[fmt]))
    return t.view(torch.uint8).numpy().reshape(rows, cols)


def generate_scales(n: int, seed: int, tensor_id: int, lo: float = 0.5, hi: float = 2.0) -> np.ndarray:
    """``n`` fp32 factors uniform in [lo, hi) from the stream."""
    u = (_uniform_f32(seed, tensor_id, 0, n) + np.float32(1.0)) * np.float32(0.5)   # [0, 1)
    return (np.float32(lo) + u * np.float32(hi - lo)).astype(np.float32)
