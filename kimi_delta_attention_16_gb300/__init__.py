"""Kimi Delta Attention (KDA) layer for one GB300 (sm_103a).

The compute lives in libkda.so (hand-written CUDA, C ABI in include/kda.h);
this package holds its PyTorch binding, its build script and the seeded
synthetic-input generators.
"""
from .api import (KDAError, kda_backward, kda_backward_workspace_size, kda_decode_step, kda_gemm,
                  kda_layer, kda_prefill, kda_prefill_noalloc, kda_prefill_plan, kda_prefill_workspace_size,
                  kda_short_conv)

__all__ = ["KDAError", "kda_short_conv", "kda_prefill", "kda_prefill_workspace_size",
           "kda_prefill_plan", "kda_prefill_noalloc", "kda_decode_step", "kda_gemm", "kda_backward", "kda_layer",
           "kda_backward_workspace_size"]
