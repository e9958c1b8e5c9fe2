"""GB300-native dense half-precision GEMM: C = A.B with fp16/bf16 inputs,
fp32 accumulation in tensor memory, and C rounded to the input dtype.

The compute path is a C-ABI shared library (``libhgemm.so``, declared in
``include/hgemm.h``) whose kernels are hand-written CUDA for sm_103a. The
Python binding in :mod:`half_precision_dense_gb300.binding` only marshals
arguments to it. Importing this package loads nothing; the binding loads the
library on first use and raises if it is missing.
"""

__version__ = "0.2.0"

_BINDING_NAMES = {
    "hgemm", "hgemm_ex", "hgemm_fp8", "hgemm_conv2d", "conv2d_nhwc", "hgemm_noalloc", "hgemm_host", "matmul", "status_string", "version",
    "get_device_status", "plan", "tile_coord", "HgemmError", "Config", "load_library",
    "set_timeout_ns",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
