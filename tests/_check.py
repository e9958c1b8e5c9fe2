"""Parity tolerance for GPU results against the oracle.

For each checked element (the bound of the hot path's stated tolerance):

    |C_gpu - C_ref| <= 2 * ulp_dtype(|C_ref64|) + 1e-4 * sqrt(K)

where C_ref is the oracle's rounded result, C_ref64 its unrounded fp64 sum, and
ulp_dtype(x) = 2^(max(floor(log2 x), emin) - p) with (p, emin) = (10, -14) for
fp16 and (7, -126) for bf16. In aggregate, over the checked elements,

    ||C_gpu - C_ref||_F / ||C_ref||_F <= 1e-3 (fp16), 5e-3 (bf16).

The GPU values are decoded with PyTorch's own conversion, independently of the
oracle's decoder.
"""

from __future__ import annotations

import numpy as np
import torch

FRO_BOUND = {"f16": 1e-3, "bf16": 5e-3}
_P_EMIN = {"f16": (10, -14), "bf16": (7, -126)}


def values(bits16: np.ndarray, dtype: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits16).view(np.int16).copy())
    t = t.view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.to(torch.float64).numpy()


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    p, emin = _P_EMIN[dtype]
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, emin), emin)
    return np.exp2(e - p)


def compare(got_bits: np.ndarray, ref_bits: np.ndarray, ref64: np.ndarray, dtype: str, K: int) -> dict:
    got = values(got_bits, dtype)
    ref = values(ref_bits, dtype)
    err = np.abs(got - ref)
    bound = 2.0 * ulp(ref64, dtype) + 1e-4 * np.sqrt(max(K, 0))
    bad = ~(err <= bound)  # NaN counts as bad
    denom = np.sqrt(np.sum(ref * ref))
    rel = float(np.sqrt(np.sum((got - ref) ** 2)) / denom) if denom > 0 else float(np.sqrt(np.sum(got * got)))
    return {
        "n": int(got.size),
        "n_bad": int(bad.sum()),
        "max_err": float(np.nanmax(err)) if err.size else 0.0,
        "max_err_over_bound": float(np.nanmax(err / bound)) if err.size else 0.0,
        "rel_fro": rel,
        "rel_fro_bound": FRO_BOUND[dtype],
        "first_bad": tuple(int(v) for v in np.argwhere(bad)[0]) if bad.any() else None,
        "ok": bool((not bad.any()) and rel <= FRO_BOUND[dtype]),
    }
