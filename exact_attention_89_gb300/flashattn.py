"""ctypes binding of libflashattn with the C ABI's names (argument marshalling only).

Every computation runs in the CUDA library; this module only turns torch tensors into device
pointers and sizes, picks the current CUDA stream and raises on a non-OK status.  There is no
fallback: if ``libflashattn.so`` is missing or the GPU is not sm_103, calls fail loudly.

Low-level functions (same names and argument order as ``include/flashattn.h``):
    fa_fwd, fa_bwd, fa_bwd_workspace_bytes, fa_fwd_fp32, fa_bwd_fp32,
    fa_get_device_status, fa_status_string, fa_bwd_noalloc, fa_fwd_split, fa_merge,
    fa_fwd_masked, fa_bwd_masked, fa_fwd_dropout, fa_bwd_dropout, fa_dropout_mask,
    fa_fwd_kvouter, fa_fwd_kvouter_workspace_bytes, fa_fwd_fp32_tc, fa_fwd_fp32_tc_workspace_bytes,
    fa_bwd_fp32_tc, fa_bwd_fp32_tc_workspace_bytes, fa_bwd_deterministic,
    fa_bwd_deterministic_workspace_bytes
Convenience wrappers that allocate outputs with torch:
    attention_forward, attention_backward (deterministic=True: fa_bwd_deterministic),
    attention_forward_split
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libflashattn.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_WORKSPACE = 4
FA_ERR_CUDA = 5
FA_ERR_DEVICE_TIMEOUT = 6
FA_ERR_DEVICE_BOUNDS = 7

# Every symbol include/flashattn.h declares.
EXPORTED = ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_fwd_fp32", "fa_bwd_fp32",
            "fa_get_device_status", "fa_status_string", "fa_bwd_noalloc", "fa_fwd_split",
            "fa_merge", "fa_fwd_masked", "fa_bwd_masked", "fa_fwd_dropout", "fa_bwd_dropout",
            "fa_dropout_mask", "fa_fwd_kvouter", "fa_fwd_kvouter_workspace_bytes",
            "fa_fwd_fp32_tc", "fa_fwd_fp32_tc_workspace_bytes", "fa_bwd_fp32_tc",
            "fa_bwd_fp32_tc_workspace_bytes", "fa_bwd_deterministic",
            "fa_bwd_deterministic_workspace_bytes")

# Side of the square tiles of a block mask (FA_MASK_BLOCK).
MASK_BLOCK = 128

# Largest number of key ranges fa_fwd_split / fa_merge accept (FA_MAX_SPLITS).
MAX_SPLITS = 256

# Size of the fixed device scratch fa_bwd_noalloc uses (FA_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024

_lock = threading.Lock()
_lib = None


class FlashAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__("%s failed: %s" % (where, fa_status_string(status)))


def lib() -> ctypes.CDLL:
    """The loaded library with argument types set (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libflashattn.so not found at %s; build it with "
                                   "exact_attention_89_gb300.build.build()" % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            dims = [i, i, i, i, i, i, f]
            L.fa_fwd.argtypes = [vp] * 5 + dims + [vp]
            L.fa_fwd.restype = i
            L.fa_bwd.argtypes = [vp] * 9 + dims + [vp, sz, vp]
            L.fa_bwd.restype = i
            L.fa_fwd_fp32.argtypes = [vp] * 5 + dims + [vp]
            L.fa_fwd_fp32.restype = i
            L.fa_bwd_fp32.argtypes = [vp] * 9 + dims + [vp, sz, vp]
            L.fa_bwd_fp32.restype = i
            L.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
            L.fa_bwd_workspace_bytes.restype = sz
            L.fa_get_device_status.argtypes = [vp]
            L.fa_get_device_status.restype = i
            L.fa_status_string.argtypes = [i]
            L.fa_status_string.restype = ctypes.c_char_p
            L.fa_bwd_noalloc.argtypes = [vp] * 9 + dims + [vp]
            L.fa_bwd_noalloc.restype = i
            L.fa_bwd_deterministic.argtypes = [vp] * 9 + dims + [vp, sz, vp]
            L.fa_bwd_deterministic.restype = i
            L.fa_bwd_deterministic_workspace_bytes.argtypes = [i, i, i, i]
            L.fa_bwd_deterministic_workspace_bytes.restype = sz
            L.fa_fwd_split.argtypes = [vp] * 5 + dims + [i, vp]
            L.fa_fwd_split.restype = i
            L.fa_merge.argtypes = [vp, vp, i, ctypes.c_longlong, i, vp, i, vp, vp]
            L.fa_merge.restype = i
            L.fa_fwd_masked.argtypes = [vp] * 5 + dims + [vp, vp, vp, i, vp]
            L.fa_fwd_masked.restype = i
            L.fa_bwd_masked.argtypes = [vp] * 9 + dims + [vp, vp, vp, i, vp, sz, vp]
            L.fa_bwd_masked.restype = i
            u64, u32 = ctypes.c_ulonglong, ctypes.c_uint
            L.fa_fwd_dropout.argtypes = [vp] * 5 + dims + [f, u64, u32, vp]
            L.fa_fwd_dropout.restype = i
            L.fa_bwd_dropout.argtypes = [vp] * 9 + dims + [f, u64, u32, vp, sz, vp]
            L.fa_bwd_dropout.restype = i
            L.fa_dropout_mask.argtypes = [i, i, f, u64, u32, vp, vp]
            L.fa_dropout_mask.restype = i
            L.fa_fwd_kvouter.argtypes = [vp] * 5 + dims + [vp, sz, vp]
            L.fa_fwd_kvouter.restype = i
            L.fa_fwd_kvouter_workspace_bytes.argtypes = [i, i, i, i]
            L.fa_fwd_kvouter_workspace_bytes.restype = sz
            L.fa_fwd_fp32_tc.argtypes = [vp] * 5 + dims + [vp, sz, vp]
            L.fa_fwd_fp32_tc.restype = i
            L.fa_fwd_fp32_tc_workspace_bytes.argtypes = [i, i, i, i, i]
            L.fa_fwd_fp32_tc_workspace_bytes.restype = sz
            L.fa_bwd_fp32_tc.argtypes = [vp] * 9 + dims + [vp, sz, vp]
            L.fa_bwd_fp32_tc.restype = i
            L.fa_bwd_fp32_tc_workspace_bytes.argtypes = [i, i, i, i, i]
            L.fa_bwd_fp32_tc_workspace_bytes.restype = sz
            _lib = L
    return _lib


def fa_status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _dims(Q, K):
    B, Hq, N, d = Q.shape
    return B, Hq, K.shape[1], N, d


def _check(status: int, where: str, check: bool):
    if check and status != FA_OK:
        raise FlashAttnError(status, where)
    return status


def fa_fwd(Q, K, V, O, LSE, causal: bool, scale: float, stream=None, check: bool = True) -> int:
    """O, LSE <- attention(Q, K, V); bf16 [B,H,N,d] tensors, LSE fp32 [B,Hq,N]."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    st = lib().fa_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, Hq, Hkv, N, d,
                      int(bool(causal)), float(scale), _stream(stream))
    return _check(st, "fa_fwd", check)


def fa_bwd_workspace_bytes(B: int, Hq: int, N: int, d: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, Hq, N, d))


def fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, causal: bool, scale: float, workspace,
           stream=None, check: bool = True) -> int:
    """dQ, dK, dV <- gradients of attention; workspace is a byte tensor on the device."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().fa_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                      _ptr(dK), _ptr(dV), B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                      _ptr(workspace), wbytes, _stream(stream))
    return _check(st, "fa_bwd", check)


def fa_bwd_deterministic_workspace_bytes(B: int, Hq: int, N: int, d: int) -> int:
    return int(lib().fa_bwd_deterministic_workspace_bytes(B, Hq, N, d))


def fa_bwd_deterministic(Q, K, V, O, dO, LSE, dQ, dK, dV, causal: bool, scale: float, workspace,
                         stream=None, check: bool = True) -> int:
    """fa_bwd with the dQ reductions in a fixed order (bitwise reproducible dQ); the workspace
    holds fa_bwd_deterministic_workspace_bytes bytes."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().fa_bwd_deterministic(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE),
                                    _ptr(dQ), _ptr(dK), _ptr(dV), B, Hq, Hkv, N, d,
                                    int(bool(causal)), float(scale), _ptr(workspace), wbytes,
                                    _stream(stream))
    return _check(st, "fa_bwd_deterministic", check)


def fa_bwd_noalloc(Q, K, V, O, dO, LSE, dQ, dK, dV, causal: bool, scale: float, stream=None,
                   check: bool = True) -> int:
    """fa_bwd for callers that cannot allocate: the scratch is the library's own fixed array of
    NOALLOC_SCRATCH_BYTES per device, shared by every call (calls must not overlap on the GPU)."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    st = lib().fa_bwd_noalloc(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                              _ptr(dK), _ptr(dV), B, Hq, Hkv, N, d, int(bool(causal)),
                              float(scale), _stream(stream))
    return _check(st, "fa_bwd_noalloc", check)


def fa_fwd_split(Q, K, V, O_parts, LSE_parts, causal: bool, scale: float, num_splits: int,
                 stream=None, check: bool = True) -> int:
    """Partial results of num_splits key ranges: O_parts fp32 [S,B,Hq,N,d], LSE_parts fp32
    [S,B,Hq,N] (-inf where a row has no key in the range)."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    st = lib().fa_fwd_split(_ptr(Q), _ptr(K), _ptr(V), _ptr(O_parts), _ptr(LSE_parts), B, Hq,
                            Hkv, N, d, int(bool(causal)), float(scale), int(num_splits),
                            _stream(stream))
    return _check(st, "fa_fwd_split", check)


def fa_merge(O_parts, LSE_parts, O, LSE, stream=None, check: bool = True) -> int:
    """O, LSE <- merge of the parts along dim 0; O bf16 or fp32 by its dtype."""
    S = O_parts.shape[0]
    d = O_parts.shape[-1]
    rows = LSE_parts.numel() // S if S > 0 else 0
    st = lib().fa_merge(_ptr(O_parts), _ptr(LSE_parts), int(S), int(rows), int(d), _ptr(O),
                        int(O.dtype == torch.bfloat16), _ptr(LSE), _stream(stream))
    return _check(st, "fa_merge", check)


def _mask_ptrs(q_len, k_len, block_mask):
    mh = 0 if block_mask is None else int(block_mask.shape[0])
    return _ptr(q_len), _ptr(k_len), _ptr(block_mask), mh


def fa_fwd_masked(Q, K, V, O, LSE, causal: bool, scale: float, q_len=None, k_len=None,
                  block_mask=None, stream=None, check: bool = True) -> int:
    """fa_fwd under a general mask: q_len / k_len int32 [B] and block_mask uint8
    [mask_heads, nb, nb] device tensors (or None)."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    st = lib().fa_fwd_masked(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, Hq, Hkv, N, d,
                             int(bool(causal)), float(scale),
                             *_mask_ptrs(q_len, k_len, block_mask), _stream(stream))
    return _check(st, "fa_fwd_masked", check)


def fa_bwd_masked(Q, K, V, O, dO, LSE, dQ, dK, dV, causal: bool, scale: float, workspace,
                  q_len=None, k_len=None, block_mask=None, stream=None, check: bool = True) -> int:
    """fa_bwd under the general mask fa_fwd_masked used."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().fa_bwd_masked(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                             _ptr(dK), _ptr(dV), B, Hq, Hkv, N, d, int(bool(causal)),
                             float(scale), *_mask_ptrs(q_len, k_len, block_mask),
                             _ptr(workspace), wbytes, _stream(stream))
    return _check(st, "fa_bwd_masked", check)


def fa_fwd_dropout(Q, K, V, O, LSE, causal: bool, scale: float, p_drop: float, seed: int,
                   offset: int = 0, stream=None, check: bool = True) -> int:
    """fa_fwd with dropout on P (keep decisions from Philox4x32-10 at (seed, offset))."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    st = lib().fa_fwd_dropout(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, Hq, Hkv, N, d,
                              int(bool(causal)), float(scale), float(p_drop), int(seed),
                              int(offset), _stream(stream))
    return _check(st, "fa_fwd_dropout", check)


def fa_bwd_dropout(Q, K, V, O, dO, LSE, dQ, dK, dV, causal: bool, scale: float, p_drop: float,
                   seed: int, offset: int, workspace, stream=None, check: bool = True) -> int:
    """Backward of fa_fwd_dropout with the same (p_drop, seed, offset)."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().fa_bwd_dropout(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                              _ptr(dK), _ptr(dV), B, Hq, Hkv, N, d, int(bool(causal)),
                              float(scale), float(p_drop), int(seed), int(offset),
                              _ptr(workspace), wbytes, _stream(stream))
    return _check(st, "fa_bwd_dropout", check)


def fa_dropout_mask(Z, p_drop: float, seed: int, offset: int = 0, stream=None,
                    check: bool = True) -> int:
    """Z: uint8 device tensor [BH, N, N] <- the keep decisions (1 = keep)."""
    BH, N = Z.shape[0], Z.shape[-1]
    st = lib().fa_dropout_mask(int(BH), int(N), float(p_drop), int(seed), int(offset), _ptr(Z),
                               _stream(stream))
    return _check(st, "fa_dropout_mask", check)


def fa_fwd_kvouter_workspace_bytes(B: int, Hq: int, N: int, d: int) -> int:
    return int(lib().fa_fwd_kvouter_workspace_bytes(B, Hq, N, d))


def fa_fwd_kvouter(Q, K, V, O, LSE, causal: bool, scale: float, workspace, stream=None,
                   check: bool = True) -> int:
    """The forward in the key/value-outer loop order (same O and LSE as fa_fwd)."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().fa_fwd_kvouter(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, Hq, Hkv, N, d,
                              int(bool(causal)), float(scale), _ptr(workspace), wbytes,
                              _stream(stream))
    return _check(st, "fa_fwd_kvouter", check)


def fa_fwd_fp32_tc_workspace_bytes(B: int, Hq: int, Hkv: int, N: int, d: int) -> int:
    return int(lib().fa_fwd_fp32_tc_workspace_bytes(B, Hq, Hkv, N, d))


def fa_fwd_fp32_tc(Q, K, V, O, LSE, causal: bool, scale: float, workspace, stream=None,
                   check: bool = True) -> int:
    """fp32 forward on the tensor cores (three TF32 products per product); fp32 tensors."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().fa_fwd_fp32_tc(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, Hq, Hkv, N, d,
                              int(bool(causal)), float(scale), _ptr(workspace), wbytes,
                              _stream(stream))
    return _check(st, "fa_fwd_fp32_tc", check)


def fa_bwd_fp32_tc_workspace_bytes(B: int, Hq: int, Hkv: int, N: int, d: int) -> int:
    return int(lib().fa_bwd_fp32_tc_workspace_bytes(B, Hq, Hkv, N, d))


def fa_bwd_fp32_tc(Q, K, V, O, dO, LSE, dQ, dK, dV, causal: bool, scale: float, workspace,
                   stream=None, check: bool = True) -> int:
    """fp32 backward on the tensor cores (three TF32 products per product); fp32 tensors."""
    B, Hq, Hkv, N, d = _dims(Q, K)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().fa_bwd_fp32_tc(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                              _ptr(dK), _ptr(dV), B, Hq, Hkv, N, d, int(bool(causal)),
                              float(scale), _ptr(workspace), wbytes, _stream(stream))
    return _check(st, "fa_bwd_fp32_tc", check)


def fa_fwd_fp32(Q, K, V, O, LSE, causal: bool, scale: float, stream=None, check: bool = True):
    B, Hq, Hkv, N, d = _dims(Q, K)
    st = lib().fa_fwd_fp32(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, Hq, Hkv, N, d,
                           int(bool(causal)), float(scale), _stream(stream))
    return _check(st, "fa_fwd_fp32", check)


def fa_bwd_fp32(Q, K, V, O, dO, LSE, dQ, dK, dV, causal: bool, scale: float, workspace,
                stream=None, check: bool = True):
    B, Hq, Hkv, N, d = _dims(Q, K)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().fa_bwd_fp32(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                           _ptr(dK), _ptr(dV), B, Hq, Hkv, N, d, int(bool(causal)),
                           float(scale), _ptr(workspace), wbytes, _stream(stream))
    return _check(st, "fa_bwd_fp32", check)


def fa_get_device_status(stream=None) -> int:
    return int(lib().fa_get_device_status(_stream(stream)))


# ----------------------------------------------------------------------------- convenience
def attention_forward(Q, K, V, causal: bool, scale: float | None = None, stream=None):
    """Allocates O and LSE and runs the forward (bf16 or fp32 by Q's dtype)."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    B, Hq, N, d = Q.shape
    O = torch.empty_like(Q)
    LSE = torch.empty((B, Hq, N), dtype=torch.float32, device=Q.device)
    f = fa_fwd_fp32 if Q.dtype == torch.float32 else fa_fwd
    f(Q, K, V, O, LSE, causal, scale, stream)
    return O, LSE


def attention_forward_split(Q, K, V, causal: bool, scale: float | None = None,
                            num_splits: int = 2, stream=None, return_parts: bool = False):
    """bf16 forward as fa_fwd_split over num_splits key ranges followed by fa_merge; returns O
    (bf16) and LSE, plus the partials when return_parts is set."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    B, Hq, N, d = Q.shape
    O_parts = torch.empty((num_splits, B, Hq, N, d), dtype=torch.float32, device=Q.device)
    LSE_parts = torch.empty((num_splits, B, Hq, N), dtype=torch.float32, device=Q.device)
    fa_fwd_split(Q, K, V, O_parts, LSE_parts, causal, scale, num_splits, stream)
    O = torch.empty_like(Q)
    LSE = torch.empty((B, Hq, N), dtype=torch.float32, device=Q.device)
    fa_merge(O_parts, LSE_parts, O, LSE, stream)
    if return_parts:
        return O, LSE, O_parts, LSE_parts
    return O, LSE


def attention_forward_masked(Q, K, V, causal: bool, scale: float | None = None, q_len=None,
                             k_len=None, block_mask=None, stream=None):
    """Allocates O and LSE and runs fa_fwd_masked."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    B, Hq, N, d = Q.shape
    O = torch.empty_like(Q)
    LSE = torch.empty((B, Hq, N), dtype=torch.float32, device=Q.device)
    fa_fwd_masked(Q, K, V, O, LSE, causal, scale, q_len, k_len, block_mask, stream)
    return O, LSE


def attention_backward_masked(Q, K, V, O, dO, LSE, causal: bool, scale: float | None = None,
                              q_len=None, k_len=None, block_mask=None, workspace=None,
                              stream=None):
    """Allocates dQ, dK, dV (and the workspace unless given) and runs fa_bwd_masked."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    B, Hq, N, d = Q.shape
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_bytes(B, Hq, N, d), dtype=torch.uint8,
                                device=Q.device)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    fa_bwd_masked(Q, K, V, O, dO, LSE, dQ, dK, dV, causal, scale, workspace, q_len, k_len,
                  block_mask, stream)
    return dQ, dK, dV


def attention_forward_dropout(Q, K, V, causal: bool, scale: float | None, p_drop: float,
                              seed: int, offset: int = 0, stream=None):
    """Allocates O and LSE and runs fa_fwd_dropout."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    B, Hq, N, d = Q.shape
    O = torch.empty_like(Q)
    LSE = torch.empty((B, Hq, N), dtype=torch.float32, device=Q.device)
    fa_fwd_dropout(Q, K, V, O, LSE, causal, scale, p_drop, seed, offset, stream)
    return O, LSE


def attention_backward_dropout(Q, K, V, O, dO, LSE, causal: bool, scale: float | None,
                               p_drop: float, seed: int, offset: int = 0, workspace=None,
                               stream=None):
    """Allocates dQ, dK, dV (and the workspace unless given) and runs fa_bwd_dropout."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    B, Hq, N, d = Q.shape
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_bytes(B, Hq, N, d), dtype=torch.uint8,
                                device=Q.device)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    fa_bwd_dropout(Q, K, V, O, dO, LSE, dQ, dK, dV, causal, scale, p_drop, seed, offset,
                   workspace, stream)
    return dQ, dK, dV


def attention_forward_kvouter(Q, K, V, causal: bool, scale: float | None = None,
                              workspace=None, stream=None):
    """Allocates O, LSE (and the workspace unless given) and runs fa_fwd_kvouter."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    B, Hq, N, d = Q.shape
    if workspace is None:
        workspace = torch.empty(fa_fwd_kvouter_workspace_bytes(B, Hq, N, d), dtype=torch.uint8,
                                device=Q.device)
    O = torch.empty_like(Q)
    LSE = torch.empty((B, Hq, N), dtype=torch.float32, device=Q.device)
    fa_fwd_kvouter(Q, K, V, O, LSE, causal, scale, workspace, stream)
    return O, LSE


def attention_forward_fp32_tc(Q, K, V, causal: bool, scale: float | None = None,
                              workspace=None, stream=None):
    """Allocates O, LSE (and the workspace unless given) and runs fa_fwd_fp32_tc."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    B, Hq, N, d = Q.shape
    if workspace is None:
        workspace = torch.empty(fa_fwd_fp32_tc_workspace_bytes(B, Hq, K.shape[1], N, d),
                                dtype=torch.uint8, device=Q.device)
    O = torch.empty_like(Q)
    LSE = torch.empty((B, Hq, N), dtype=torch.float32, device=Q.device)
    fa_fwd_fp32_tc(Q, K, V, O, LSE, causal, scale, workspace, stream)
    return O, LSE


def attention_backward_fp32_tc(Q, K, V, O, dO, LSE, causal: bool, scale: float | None = None,
                               workspace=None, stream=None):
    """Allocates dQ, dK, dV (and the workspace unless given) and runs fa_bwd_fp32_tc."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    B, Hq, N, d = Q.shape
    if workspace is None:
        workspace = torch.empty(fa_bwd_fp32_tc_workspace_bytes(B, Hq, K.shape[1], N, d),
                                dtype=torch.uint8, device=Q.device)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    fa_bwd_fp32_tc(Q, K, V, O, dO, LSE, dQ, dK, dV, causal, scale, workspace, stream)
    return dQ, dK, dV


def attention_backward(Q, K, V, O, dO, LSE, causal: bool, scale: float | None = None,
                       workspace=None, stream=None, deterministic: bool = False):
    """Allocates dQ, dK, dV (and the workspace unless given) and runs the backward
    (deterministic: the bf16 backward with the dQ reductions in a fixed order)."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    B, Hq, N, d = Q.shape
    if deterministic and Q.dtype == torch.float32:
        raise ValueError("the deterministic backward is the bf16 one; the fp32 backward "
                         "(fa_bwd_fp32) is reproducible as it is")
    if workspace is None:
        size = (fa_bwd_deterministic_workspace_bytes if deterministic else
                fa_bwd_workspace_bytes)(B, Hq, N, d)
        workspace = torch.empty(size, dtype=torch.uint8, device=Q.device)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    f = (fa_bwd_fp32 if Q.dtype == torch.float32 else
         fa_bwd_deterministic if deterministic else fa_bwd)
    f(Q, K, V, O, dO, LSE, dQ, dK, dV, causal, scale, workspace, stream)
    return dQ, dK, dV
