"""libflashattn for GB300 (sm_103a): exact scaled-dot-product attention, forward and backward.

The compute lives in ``libflashattn.so`` (CUDA, built from ``csrc/`` by ``build.py``); this
package is its ctypes binding plus seeded input generators for tests and benchmarks.
"""
from .flashattn import (FA_OK, FlashAttnError, attention_backward, attention_forward, fa_bwd,
                        fa_bwd_fp32, fa_bwd_workspace_bytes, fa_fwd, fa_fwd_fp32,
                        fa_get_device_status, fa_status_string)

__all__ = ["FA_OK", "FlashAttnError", "attention_backward", "attention_forward", "fa_bwd",
           "fa_bwd_fp32", "fa_bwd_workspace_bytes", "fa_fwd", "fa_fwd_fp32",
           "fa_get_device_status", "fa_status_string"]
