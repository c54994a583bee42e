"""Exact softmax attention for large head dims (D = 64..1024, tuned for 320..1024) on GB300 (sm_103a).

Forward (O and fp32 LSE) and backward (dQ, dK, dV) with bottom-right causal
masking, GQA/MQA head broadcast and packed varlen batches, computed by
hand-written tcgen05/TMA kernels behind the C ABI of ``include/ffpa.h``.
"""
from .api import (attention, bwd, bwd_workspace_bytes, decode_fwd, decode_supported, fp8_quantize, fwd, fwd_fp8,
                  get_status, varlen_attention, varlen_bwd, varlen_fwd, varlen_fwd_fp8)

__all__ = ["attention", "varlen_attention", "fwd", "bwd", "bwd_workspace_bytes", "varlen_fwd", "varlen_bwd",
           "decode_fwd", "decode_supported", "fwd_fp8", "varlen_fwd_fp8", "fp8_quantize", "get_status"]
