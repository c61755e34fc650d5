"""FlashAttention for one GB300 (sm_103a): Python binding of libfa_b200.

The compute path is the C-ABI library ``libfa_b200.so`` (hand-written CUDA for
sm_103a): forward (dense, grouped-query, split-KV, varlen, paged K/V, strided)
and backward.  This package only marshals arguments; it loads the library
lazily on the first call and raises if it is missing.
"""
from .binding import (FA_DTYPE, FA_LAYOUT, FA_STATUS, FaError, attention, attention_backward,
                      fa_bwd, fa_fwd, fa_fwd_gqa, fa_last_device_error, fa_status_string,
                      flash_attention, load)

__all__ = ["FA_DTYPE", "FA_LAYOUT", "FA_STATUS", "FaError", "attention", "attention_backward",
           "fa_bwd", "fa_fwd", "fa_fwd_gqa", "fa_last_device_error", "fa_status_string",
           "flash_attention", "load"]
