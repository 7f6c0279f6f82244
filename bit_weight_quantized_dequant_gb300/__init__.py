"""Python binding of liblq: fused low-bit dequantize-and-multiply on GB300.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of ``liblq.so``; there is no CPU or PyTorch fallback, and importing the
compute functions without the compiled library raises.

Weight formats (see ``include/lq.h``):
  * 2-bit Lloyd-Max codes, group 32, binary16 scale/offset, binary16 anchor columns
    (otf-llm 4.0.1 README, sections 2-4);
  * NF4, block 64, fp32 absmax (AirQuant README, NF4 block-wise).
"""
from __future__ import annotations

from ._lq import (  # noqa: F401
    LQ_OK, LQ_ERR_INVALID_ARG, LQ_ERR_UNSUPPORTED, LQ_ERR_ALIGNMENT, LQ_ERR_WORKSPACE, LQ_ERR_CUDA,
    LQ_ERR_TIMEOUT, LQ_ERR_RANGE, FMT_2BIT, FMT_NF4, FMT_INT4, FMT_NF4_DQ, F32, F16, BF16, LQError, QuantWeights, Handle, load_library,
    library_path, exported_symbols, EXPORTED, LayerStream, pack_layer,
)
from .build import build  # noqa: F401
