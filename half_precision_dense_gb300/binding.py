"""ctypes binding to ``libhgemm.so`` (the C ABI in ``include/hgemm.h``).

Argument marshalling only: every step of the GEMM runs in the library's CUDA
kernels. The binding loads the library on first use and raises
:class:`HgemmError` if it is missing; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

from . import build as _build

_lib = None
_lock = threading.Lock()

HGEMM_F16 = 0
HGEMM_BF16 = 1
HGEMM_TF32 = 2
HGEMM_E4M3 = 3
HGEMM_E5M2 = 4
STATUS_NAMES = {0: "HGEMM_OK", 1: "HGEMM_ERR_INVALID_ARG", 2: "HGEMM_ERR_UNSUPPORTED_DEVICE",
                3: "HGEMM_ERR_CUDA", 4: "HGEMM_ERR_ALLOC", 5: "HGEMM_ERR_TIMEOUT"}


class HgemmError(RuntimeError):
    def __init__(self, status: int, detail: str = ""):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{name}{': ' + detail if detail else ''}")


class _Config(ctypes.Structure):
    _fields_ = [("cta_group", ctypes.c_int32), ("block_n", ctypes.c_int32),
                ("group_m", ctypes.c_int32), ("max_clusters", ctypes.c_int32),
                ("store_mode", ctypes.c_int32), ("stream_k", ctypes.c_int32),
                ("multicast", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("epi_warps", ctypes.c_int32)]


class _Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "cta_group", "block_m", "block_n", "block_k", "stages", "group_m", "tiles_m", "tiles_n",
        "num_tiles", "grid_ctas", "smem_bytes", "tmem_cols", "repack_a", "repack_b", "store_mode",
        "dp_tiles", "sk_tiles", "sk_blocks", "sk_extra", "num_kb", "multicast", "split_k")] + \
        [("workspace_bytes", ctypes.c_int64), ("epi_warps", ctypes.c_int32)]


@dataclass
class Config:
    """Optional launch configuration; 0 = let the planner choose."""
    cta_group: int = 0
    block_n: int = 0
    group_m: int = 0
    max_clusters: int = 0
    store_mode: int = 0
    stream_k: int = 0
    multicast: int = 0
    split_k: int = 0
    epi_warps: int = 0

    def _c(self) -> _Config:
        return _Config(self.cta_group, self.block_n, self.group_m, self.max_clusters, self.store_mode,
                       self.stream_k, self.multicast, self.split_k, self.epi_warps)


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load the library (once). Raises HgemmError if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise HgemmError(3, f"CUDA library not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        lib.hgemm.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int, vp]
        lib.hgemm.restype = ctypes.c_int
        lib.hgemm_ex.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int, ctypes.POINTER(_Config), vp]
        lib.hgemm_ex.restype = ctypes.c_int
        lib.hgemm_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int, vp]
        lib.hgemm_noalloc.restype = ctypes.c_int
        lib.hgemm_noalloc_ex.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int, ctypes.POINTER(_Config), vp]
        lib.hgemm_noalloc_ex.restype = ctypes.c_int
        lib.hgemm_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_int, vp]
        lib.hgemm_fp8.restype = ctypes.c_int
        lib.hgemm_fp8_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_int,
                                     ctypes.POINTER(_Config), vp]
        lib.hgemm_fp8_ex.restype = ctypes.c_int
        lib.hgemm_fp8_blockscaled.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, ctypes.c_int, vp]
        lib.hgemm_fp8_blockscaled.restype = ctypes.c_int
        lib.hgemm_fp8_blockscaled_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, ctypes.c_int,
                                                 ctypes.POINTER(_Config), vp]
        lib.hgemm_fp8_blockscaled_ex.restype = ctypes.c_int
        lib.hgemm_conv2d.argtypes = [vp, vp, vp] + [i32] * 9 + [ctypes.c_int, vp]
        lib.hgemm_conv2d.restype = ctypes.c_int
        lib.hgemm_conv2d_set_mode.argtypes = [ctypes.c_int32]
        lib.hgemm_conv2d_set_mode.restype = None
        lib.hgemm_noalloc_scratch_bytes.argtypes = []
        lib.hgemm_noalloc_scratch_bytes.restype = ctypes.c_uint64
        lib.hgemm_host.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.c_int, vp, vp, vp, vp]
        lib.hgemm_host.restype = ctypes.c_int
        lib.hgemm_plan.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.POINTER(_Config), i32,
                                   ctypes.POINTER(_Plan)]
        lib.hgemm_plan.restype = ctypes.c_int
        lib.hgemm_work_unit.argtypes = [ctypes.POINTER(_Plan), i32, i32] + [ctypes.POINTER(i32)] * 4
        lib.hgemm_work_unit.restype = i32
        lib.hgemm_tile_coord.argtypes = [i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.hgemm_tile_coord.restype = None
        lib.hgemm_split_share.argtypes = [i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.hgemm_split_share.restype = None
        lib.hgemm_get_device_status.argtypes = [i32, i32, ctypes.POINTER(ctypes.c_uint32)]
        lib.hgemm_get_device_status.restype = ctypes.c_int
        lib.hgemm_set_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.hgemm_set_timeout_ns.restype = None
        lib.hgemm_test_inject.argtypes = [ctypes.c_int32]
        lib.hgemm_test_inject.restype = None
        lib.hgemm_status_string.argtypes = [ctypes.c_int]
        lib.hgemm_status_string.restype = ctypes.c_char_p
        lib.hgemm_last_error.argtypes = []
        lib.hgemm_last_error.restype = ctypes.c_char_p
        lib.hgemm_version.argtypes = []
        lib.hgemm_version.restype = ctypes.c_int32
        _lib = lib
        return lib


def _dtype_code(dtype) -> int:
    if dtype in (HGEMM_F16, HGEMM_BF16, HGEMM_TF32, HGEMM_E4M3, HGEMM_E5M2):
        return int(dtype)
    name = str(dtype)
    if name in ("bf16", "bfloat16", "torch.bfloat16"):
        return HGEMM_BF16
    if name in ("f16", "fp16", "float16", "half", "torch.float16"):
        return HGEMM_F16
    if name in ("tf32", "f32", "fp32", "float32", "torch.float32"):
        return HGEMM_TF32
    if name in ("e4m3", "fp8_e4m3", "torch.float8_e4m3fn"):
        return HGEMM_E4M3
    if name in ("e5m2", "fp8_e5m2", "torch.float8_e5m2"):
        return HGEMM_E5M2
    raise ValueError(f"unsupported dtype {dtype!r}")


def _ptr(x) -> int | None:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s) -> int | None:
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def _check(status: int):
    if status != 0:
        lib = load_library()
        raise HgemmError(status, lib.hgemm_last_error().decode())


def hgemm(A, B, C, M: int, N: int, K: int, dtype, stream=None) -> None:
    """C = A.B (device pointers or CUDA tensors), enqueued on ``stream``."""
    lib = load_library()
    _check(lib.hgemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, _dtype_code(dtype), _stream(stream)))


def hgemm_noalloc(A, B, C, M: int, N: int, K: int, dtype, stream=None, config: Config | None = None) -> None:
    """hgemm for callers that cannot allocate: any workspace comes from the
    library's fixed scratch array (see include/hgemm.h); `config` as for hgemm_ex."""
    lib = load_library()
    if config is None:
        _check(lib.hgemm_noalloc(_ptr(A), _ptr(B), _ptr(C), M, N, K, _dtype_code(dtype), _stream(stream)))
    else:
        _check(lib.hgemm_noalloc_ex(_ptr(A), _ptr(B), _ptr(C), M, N, K, _dtype_code(dtype),
                                    ctypes.byref(config._c()), _stream(stream)))


def hgemm_ex(A, B, C, M: int, N: int, K: int, dtype, config: Config | None = None,
             stream=None) -> None:
    lib = load_library()
    cfg = ctypes.byref(config._c()) if config is not None else None
    _check(lib.hgemm_ex(_ptr(A), _ptr(B), _ptr(C), M, N, K, _dtype_code(dtype), cfg, _stream(stream)))


def hgemm_fp8(A, B, C, a_scale, b_scale, M: int, N: int, K: int, dtype, config: Config | None = None,
              stream=None) -> None:
    """C (bf16) = a_scale[i] * b_scale[j] * sum_k A[i,k] B[k,j] for 8-bit E4M3 / E5M2
    operands (device pointers or CUDA tensors; scales fp32 arrays or None)."""
    lib = load_library()
    code = _dtype_code(dtype)
    if config is None:
        _check(lib.hgemm_fp8(_ptr(A), _ptr(B), _ptr(C), _ptr(a_scale), _ptr(b_scale), M, N, K, code,
                             _stream(stream)))
    else:
        _check(lib.hgemm_fp8_ex(_ptr(A), _ptr(B), _ptr(C), _ptr(a_scale), _ptr(b_scale), M, N, K, code,
                                ctypes.byref(config._c()), _stream(stream)))


def hgemm_fp8_blockscaled(A, B, C, a_scale, b_scale, M: int, N: int, K: int, block: int, dtype,
                          config: Config | None = None, stream=None) -> None:
    """C (bf16) = the product of A and B dequantised with one fp32 factor per
    block x block sub-block (block 32 or 64): a_scale is ceil(M/block) x
    ceil(K/block), b_scale ceil(K/block) x ceil(N/block), both row-major fp32
    device arrays (see include/hgemm.h)."""
    lib = load_library()
    code = _dtype_code(dtype)
    if config is None:
        _check(lib.hgemm_fp8_blockscaled(_ptr(A), _ptr(B), _ptr(C), _ptr(a_scale), _ptr(b_scale), M, N, K,
                                         int(block), code, _stream(stream)))
    else:
        _check(lib.hgemm_fp8_blockscaled_ex(_ptr(A), _ptr(B), _ptr(C), _ptr(a_scale), _ptr(b_scale), M, N, K,
                                            int(block), code, ctypes.byref(config._c()), _stream(stream)))


def hgemm_conv2d(x, w, y, N: int, H: int, W: int, C: int, K: int, R: int, S: int, stride: int, pad: int,
                 dtype, stream=None) -> None:
    """y (N x P x Q x K) = conv2d(x (N x H x W x C), w (R x S x C x K)) through im2col
    and the GEMM (device pointers or CUDA tensors; see include/hgemm.h)."""
    lib = load_library()
    _check(lib.hgemm_conv2d(_ptr(x), _ptr(w), _ptr(y), N, H, W, C, K, R, S, stride, pad, _dtype_code(dtype),
                            _stream(stream)))


def conv2d_set_mode(mode: int) -> None:
    """0: implicit GEMM where the shape allows (default); 1: always explicit im2col."""
    load_library().hgemm_conv2d_set_mode(mode)


def conv2d_nhwc(x, w, stride: int = 1, pad: int = 0, stream=None):
    """Channels-last convolution of CUDA tensors x (N, H, W, C) and w (R, S, C, K)
    of dtype float16, bfloat16 or float32 (multiplied as tf32); returns y (N, P, Q, K)."""
    import torch

    if x.dim() != 4 or w.dim() != 4 or x.shape[3] != w.shape[2]:
        raise ValueError(f"x {tuple(x.shape)} (N,H,W,C) and w {tuple(w.shape)} (R,S,C,K) do not match")
    if x.dtype != w.dtype or not (x.is_cuda and w.is_cuda and x.is_contiguous() and w.is_contiguous()):
        raise ValueError("x and w must be contiguous CUDA tensors of one dtype")
    N, H, W, C = x.shape
    R, S, _, K = w.shape
    P = (H + 2 * pad - R) // stride + 1
    Q = (W + 2 * pad - S) // stride + 1
    y = torch.empty((N, max(P, 0), max(Q, 0), K), dtype=x.dtype, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    hgemm_conv2d(x, w, y, N, H, W, C, K, R, S, stride, pad, str(x.dtype), stream)
    return y


def hgemm_host(hA, hB, hC, M: int, N: int, K: int, dtype, dA, dB, dC, stream=None) -> None:
    """Host operands in, host result out, through caller-owned device buffers;
    returns after the stream has been synchronised."""
    lib = load_library()
    _check(lib.hgemm_host(_ptr(hA), _ptr(hB), _ptr(hC), M, N, K, _dtype_code(dtype), _ptr(dA),
                          _ptr(dB), _ptr(dC), _stream(stream)))


def plan(M: int, N: int, K: int, dtype="bf16", config: Config | None = None, sm_count: int = 0) -> dict:
    lib = load_library()
    out = _Plan()
    cfg = ctypes.byref(config._c()) if config is not None else None
    _check(lib.hgemm_plan(M, N, K, _dtype_code(dtype), cfg, sm_count, ctypes.byref(out)))
    return {name: getattr(out, name) for name, _ in _Plan._fields_}


def work_units(plan_dict: dict, cluster: int) -> list[tuple[int, int, int, int]]:
    """The (tile, kb0, kb1, kind) units of one cluster under a plan from plan()."""
    lib = load_library()
    pl = _Plan(**{k: v for k, v in plan_dict.items() if k in dict(_Plan._fields_)})
    out = []
    vals = [ctypes.c_int32() for _ in range(4)]
    i = 0
    while lib.hgemm_work_unit(ctypes.byref(pl), cluster, i, *[ctypes.byref(v) for v in vals]):
        out.append(tuple(v.value for v in vals))
        i += 1
    return out


def split_share(kb0: int, kb1: int, rank: int, parts: int) -> tuple[int, int]:
    """K blocks [lo, hi) of [kb0, kb1) for rank `rank` of a K-split cluster of `parts`."""
    lib = load_library()
    a, b = ctypes.c_int32(-1), ctypes.c_int32(-1)
    lib.hgemm_split_share(kb0, kb1, rank, parts, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def tile_coord(t: int, tiles_m: int, tiles_n: int, group_m: int) -> tuple[int, int]:
    lib = load_library()
    a, b = ctypes.c_int32(), ctypes.c_int32()
    lib.hgemm_tile_coord(t, tiles_m, tiles_n, group_m, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def get_device_status(device: int = 0, reset: bool = False) -> tuple[int, int]:
    """(status, info) of the device status word; status 0 = no kernel timed out."""
    lib = load_library()
    info = ctypes.c_uint32()
    st = lib.hgemm_get_device_status(device, 1 if reset else 0, ctypes.byref(info))
    if st == 3:
        _check(st)
    return st, info.value


def set_timeout_ns(ns: int) -> None:
    load_library().hgemm_set_timeout_ns(int(ns))


def test_inject(kind: int) -> None:
    """Test hook of the failure path (see include/hgemm.h); 0 turns it off."""
    load_library().hgemm_test_inject(int(kind))


def status_string(s: int) -> str:
    return load_library().hgemm_status_string(int(s)).decode()


def version() -> int:
    return load_library().hgemm_version()


def matmul(a, b, out=None, config: Config | None = None, stream=None):
    """C = a @ b for 2-D contiguous CUDA tensors of dtype float16, bfloat16 or
    float32 (float32 operands are multiplied as tf32: see include/hgemm.h)."""
    import torch

    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shapes {tuple(a.shape)} and {tuple(b.shape)} do not chain")
    if a.dtype != b.dtype or a.dtype not in (torch.float16, torch.bfloat16, torch.float32):
        raise ValueError("a and b must share dtype float16, bfloat16 or float32")
    if not (a.is_cuda and b.is_cuda and a.is_contiguous() and b.is_contiguous()):
        raise ValueError("a and b must be contiguous CUDA tensors")
    M, K = a.shape
    N = b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=a.dtype, device=a.device)
    elif out.shape != (M, N) or out.dtype != a.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous (M, N) tensor of the operands' dtype")
    if stream is None:
        stream = torch.cuda.current_stream(a.device)
    hgemm_ex(a, b, out, M, N, K, str(a.dtype), config, stream)
    return out
