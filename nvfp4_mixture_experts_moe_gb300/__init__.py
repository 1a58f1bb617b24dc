"""Fused NVFP4 Mixture-of-Experts layer for one GB300 GPU (sm_103a).

The compute lives in the CUDA library ``_lib/libmoe_nvfp4.so`` (C ABI in
``include/moe_nvfp4.h``); ``binding`` marshals torch tensors into its calls
and ``layer`` keeps one layer's prepared weights resident on the device.
"""
from . import binding  # noqa: F401
from .binding import MoeError, MOE_W4A16, MOE_W4A4, MOE_MXFP4  # noqa: F401
from .layer import Nvfp4MoeLayer, quantize_bf16, quantize_mx  # noqa: F401
