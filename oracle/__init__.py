"""CPU oracles for the dense GEMM (test infrastructure only): the fp16/bf16
product (``hgemm_oracle``, re-exported here), the TF32 variant
(``oracle.tf32_oracle``) and the FP8 variant with per-channel scales
(``oracle.fp8_oracle``), and 2-D convolution from its definition
(``oracle.conv_oracle``).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package. The product path never does.
"""

from .hgemm_oracle import (FORMATS, decode, flops, gemm, gemm_cols, gemm_f64,  # noqa: F401
                           gemm_rows, round_rne)
