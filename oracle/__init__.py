"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The CUDA library never calls it and shares no code with it; the two meet
only through the seeded input generators, which hold none of the method's arithmetic.

The arithmetic lives in ``attention_oracle.c`` (plain C, fp64, OpenMP over independent rows or
key columns).  This module compiles it with gcc on first use (or through ``build()``) and wraps
it with ctypes over numpy float64 arrays laid out [B, H, N, d].

What the oracle computes (see the C file for the page citations):
  P = softmax(scale * Q K^T, masked pairs weight 0), O = P V, LSE = m + ln l (natural log),
  dS = P * (dO V^T - D), D = rowsum(dO * O), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO,
  with dK, dV summed over the query heads of a KV group (query head hq reads KV head hq // G).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)
_L = ctypes.POINTER(ctypes.c_int64)
_U8 = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile attention_oracle.c into liboracle.so next to it (gcc -O2 -fopenmp). Returns path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            common = [ctypes.c_int] * 6 + [ctypes.c_double]
            lib.oracle_attention_forward.argtypes = common + [_D, _D, _D, ctypes.c_int, _I, _D, _D, _D]
            lib.oracle_attention_backward.argtypes = common + [_D, _D, _D, _D, ctypes.c_int, _I, _D, _D, _D]
            lib.oracle_forward_rows.argtypes = common + [_D, _D, _D, ctypes.c_int, _L, _D, _D]
            lib.oracle_backward_dq_rows.argtypes = common + [_D, _D, _D, _D, ctypes.c_int, _L, _D]
            lib.oracle_backward_dkv_cols.argtypes = common + [_D, _D, _D, _D, ctypes.c_int, _L, _D, _D]
            lib.oracle_attention_forward_keys.argtypes = common + [_D, _D, _D, ctypes.c_int, ctypes.c_int,
                                                                   ctypes.c_int, _I, _D, _D]
            lib.oracle_merge_partials.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, _D, _D, _D, _D]
            masked = [ctypes.c_int] * 6 + [_I, _I, _U8, ctypes.c_int, ctypes.c_int, ctypes.c_double]
            lib.oracle_attention_forward_masked.argtypes = masked + [_D, _D, _D, ctypes.c_int, _I, _D, _D]
            lib.oracle_attention_backward_masked.argtypes = masked + [_D, _D, _D, _D, ctypes.c_int, _I,
                                                                      _D, _D, _D]
            lib.oracle_forward_rows_masked.argtypes = masked + [_D, _D, _D, ctypes.c_int, _L, _D, _D]
            lib.oracle_backward_dq_rows_masked.argtypes = masked + [_D, _D, _D, _D, ctypes.c_int, _L, _D]
            lib.oracle_backward_dkv_cols_masked.argtypes = masked + [_D, _D, _D, _D, ctypes.c_int, _L,
                                                                     _D, _D]
            u32, u64, dbl = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double
            _U32P = ctypes.POINTER(ctypes.c_uint32)
            lib.oracle_philox4x32_10.argtypes = [_U32P, _U32P, _U32P]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_dropout_threshold.argtypes = [dbl]
            lib.oracle_dropout_threshold.restype = u32
            lib.oracle_dropout_mask.argtypes = [ctypes.c_int, ctypes.c_int, u64, u32, dbl, _U8]
            drop = [ctypes.c_int] * 6 + [dbl, dbl, u64, u32]
            lib.oracle_attention_forward_dropout.argtypes = drop + [_D, _D, _D, _D, _D]
            lib.oracle_attention_backward_dropout.argtypes = drop + [_D, _D, _D, _D, _D, _D, _D]
            for name in ("oracle_dropout_mask", "oracle_attention_forward_dropout",
                         "oracle_attention_backward_dropout"):
                getattr(lib, name).restype = ctypes.c_int
            for name in ("oracle_attention_forward", "oracle_attention_backward",
                         "oracle_forward_rows", "oracle_backward_dq_rows",
                         "oracle_backward_dkv_cols", "oracle_num_threads",
                         "oracle_attention_forward_keys", "oracle_merge_partials",
                         "oracle_attention_forward_masked", "oracle_attention_backward_masked",
                         "oracle_forward_rows_masked", "oracle_backward_dq_rows_masked",
                         "oracle_backward_dkv_cols_masked"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS or all cores)."""
    return int(_load().oracle_num_threads())


def _f64(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def _ptr(a: np.ndarray, typ=_D):
    return a.ctypes.data_as(typ)


def _shape(Q, K):
    B, Hq, N, d = Q.shape
    Bk, Hkv, Nk, dk = K.shape
    if (Bk, Nk, dk) != (B, N, d) or Hq % Hkv:
        raise ValueError("shape mismatch: Q %s K %s" % (Q.shape, K.shape))
    return B, Hq, Hkv, N, d


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("%s failed (code %d)" % (what, rc))


def forward(Q, K, V, causal: bool, scale: float, heads=None, want_P: bool = False):
    """Full forward for the listed heads (b*Hq + hq; default all).

    Returns (O [nh, N, d], LSE [nh, N]) and P [nh, N, N] if want_P; with heads=None the outputs
    are reshaped to [B, Hq, N, d] / [B, Hq, N] (/ [B, Hq, N, N]).
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, Hq, Hkv, N, d = _shape(Q, K)
    full = heads is None
    hs = np.arange(B * Hq, dtype=np.int32) if full else np.asarray(heads, dtype=np.int32)
    hs = np.ascontiguousarray(hs)
    nh = len(hs)
    O = np.zeros((nh, N, d))
    L = np.zeros((nh, N))
    P = np.zeros((nh, N, N)) if want_P else None
    rc = _load().oracle_attention_forward(B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                                          _ptr(Q), _ptr(K), _ptr(V), nh, _ptr(hs, _I),
                                          _ptr(O), _ptr(L), _ptr(P) if want_P else None)
    _check(rc, "oracle_attention_forward")
    if full:
        O, L = O.reshape(B, Hq, N, d), L.reshape(B, Hq, N)
        if want_P:
            P = P.reshape(B, Hq, N, N)
    return (O, L, P) if want_P else (O, L)


def backward(Q, K, V, dO, causal: bool, scale: float, groups=None):
    """Full backward for the listed KV groups (b*Hkv + hk; default all).

    Returns (dQ [ng, G, N, d], dK [ng, N, d], dV [ng, N, d]); with groups=None reshaped to
    [B, Hq, N, d] and [B, Hkv, N, d].
    """
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, Hq, Hkv, N, d = _shape(Q, K)
    G = Hq // Hkv
    full = groups is None
    gs = np.arange(B * Hkv, dtype=np.int32) if full else np.asarray(groups, dtype=np.int32)
    gs = np.ascontiguousarray(gs)
    ng = len(gs)
    dQ = np.zeros((ng, G, N, d))
    dK = np.zeros((ng, N, d))
    dV = np.zeros((ng, N, d))
    rc = _load().oracle_attention_backward(B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                                           _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), ng, _ptr(gs, _I),
                                           _ptr(dQ), _ptr(dK), _ptr(dV))
    _check(rc, "oracle_attention_backward")
    if full:
        return dQ.reshape(B, Hq, N, d), dK.reshape(B, Hkv, N, d), dV.reshape(B, Hkv, N, d)
    return dQ, dK, dV


def forward_rows(Q, K, V, causal: bool, scale: float, rows):
    """Sampled rows (flat index (b*Hq + hq)*N + i) -> (O_rows [n, d], LSE_rows [n])."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, Hq, Hkv, N, d = _shape(Q, K)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    O = np.zeros((len(rows), d))
    L = np.zeros(len(rows))
    rc = _load().oracle_forward_rows(B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                                     _ptr(Q), _ptr(K), _ptr(V), len(rows), _ptr(rows, _L),
                                     _ptr(O), _ptr(L))
    _check(rc, "oracle_forward_rows")
    return O, L


def backward_dq_rows(Q, K, V, dO, causal: bool, scale: float, rows):
    """Sampled dQ rows (flat index (b*Hq + hq)*N + i) -> [n, d]."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, Hq, Hkv, N, d = _shape(Q, K)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dQ = np.zeros((len(rows), d))
    rc = _load().oracle_backward_dq_rows(B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                                         _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), len(rows),
                                         _ptr(rows, _L), _ptr(dQ))
    _check(rc, "oracle_backward_dq_rows")
    return dQ


def backward_dkv_cols(Q, K, V, dO, causal: bool, scale: float, cols):
    """Sampled dK/dV rows (flat index (b*Hkv + hk)*N + j) -> (dK [n, d], dV [n, d])."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, Hq, Hkv, N, d = _shape(Q, K)
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    dK = np.zeros((len(cols), d))
    dV = np.zeros((len(cols), d))
    rc = _load().oracle_backward_dkv_cols(B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                                          _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), len(cols),
                                          _ptr(cols, _L), _ptr(dK), _ptr(dV))
    _check(rc, "oracle_backward_dkv_cols")
    return dK, dV


def forward_keys(Q, K, V, causal: bool, scale: float, key_begin: int, key_end: int):
    """Partial forward over the keys key_begin <= j < key_end (and the causal mask): returns
    (O [B, Hq, N, d], LSE [B, Hq, N]); rows with no allowed key get O = 0, LSE = -inf."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, Hq, Hkv, N, d = _shape(Q, K)
    hs = np.ascontiguousarray(np.arange(B * Hq, dtype=np.int32))
    O = np.zeros((B * Hq, N, d))
    L = np.zeros((B * Hq, N))
    rc = _load().oracle_attention_forward_keys(B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                                               _ptr(Q), _ptr(K), _ptr(V), int(key_begin),
                                               int(key_end), len(hs), _ptr(hs, _I), _ptr(O),
                                               _ptr(L))
    _check(rc, "oracle_attention_forward_keys")
    return O.reshape(B, Hq, N, d), L.reshape(B, Hq, N)


def merge_partials(O_parts, LSE_parts):
    """Merge of S partial results over disjoint key sets: O_parts [S, ..., d], LSE_parts [S, ...]
    -> (O [..., d], LSE [...])."""
    O_parts, LSE_parts = _f64(O_parts), _f64(LSE_parts)
    S = O_parts.shape[0]
    d = O_parts.shape[-1]
    rows = int(np.prod(LSE_parts.shape[1:]))
    O = np.zeros(LSE_parts.shape[1:] + (d,))
    L = np.zeros(LSE_parts.shape[1:])
    rc = _load().oracle_merge_partials(S, rows, d, _ptr(O_parts), _ptr(LSE_parts), _ptr(O), _ptr(L))
    _check(rc, "oracle_merge_partials")
    return O, L


# ----------------------------------------------------------------------------- general masks
class Mask:
    """A general mask (see attention_oracle.c): per-batch valid query / key lengths q_len, k_len
    ([B] ints, None = all N) and a 0/1 block mask [mask_heads, nb, nb] over block x block tiles
    (None = all tiles), on top of the causal rule."""

    def __init__(self, q_len=None, k_len=None, block_mask=None, block: int = 128):
        self.q_len = None if q_len is None else np.ascontiguousarray(np.asarray(q_len, np.int32))
        self.k_len = None if k_len is None else np.ascontiguousarray(np.asarray(k_len, np.int32))
        self.block_mask = (None if block_mask is None
                           else np.ascontiguousarray(np.asarray(block_mask, np.uint8)))
        self.block = int(block)

    def args(self, causal):
        """ctypes arguments (causal, q_len, k_len, block_mask, mask_heads, block)."""
        bm = self.block_mask
        return (int(bool(causal)),
                None if self.q_len is None else _ptr(self.q_len, _I),
                None if self.k_len is None else _ptr(self.k_len, _I),
                None if bm is None else _ptr(bm, _U8),
                0 if bm is None else int(bm.shape[0]), self.block)


def forward_masked(Q, K, V, causal: bool, scale: float, mask: Mask, heads=None):
    """forward() under a general mask: (O [B, Hq, N, d], LSE [B, Hq, N]) for all heads, or
    ([nh, N, d], [nh, N]) for the listed heads."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, Hq, Hkv, N, d = _shape(Q, K)
    full = heads is None
    hs = np.ascontiguousarray(np.arange(B * Hq, dtype=np.int32) if full
                              else np.asarray(heads, dtype=np.int32))
    O = np.zeros((len(hs), N, d))
    L = np.zeros((len(hs), N))
    rc = _load().oracle_attention_forward_masked(B, Hq, Hkv, N, d, *mask.args(causal), float(scale),
                                                 _ptr(Q), _ptr(K), _ptr(V), len(hs), _ptr(hs, _I),
                                                 _ptr(O), _ptr(L))
    _check(rc, "oracle_attention_forward_masked")
    if full:
        return O.reshape(B, Hq, N, d), L.reshape(B, Hq, N)
    return O, L


def backward_masked(Q, K, V, dO, causal: bool, scale: float, mask: Mask, groups=None):
    """backward() under a general mask (same return shapes as backward())."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, Hq, Hkv, N, d = _shape(Q, K)
    G = Hq // Hkv
    full = groups is None
    gs = np.ascontiguousarray(np.arange(B * Hkv, dtype=np.int32) if full
                              else np.asarray(groups, dtype=np.int32))
    ng = len(gs)
    dQ = np.zeros((ng, G, N, d))
    dK = np.zeros((ng, N, d))
    dV = np.zeros((ng, N, d))
    rc = _load().oracle_attention_backward_masked(B, Hq, Hkv, N, d, *mask.args(causal),
                                                  float(scale), _ptr(Q), _ptr(K), _ptr(V),
                                                  _ptr(dO), ng, _ptr(gs, _I), _ptr(dQ), _ptr(dK),
                                                  _ptr(dV))
    _check(rc, "oracle_attention_backward_masked")
    if full:
        return dQ.reshape(B, Hq, N, d), dK.reshape(B, Hkv, N, d), dV.reshape(B, Hkv, N, d)
    return dQ, dK, dV


def forward_rows_masked(Q, K, V, causal: bool, scale: float, mask: Mask, rows):
    """forward_rows() under a general mask."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, Hq, Hkv, N, d = _shape(Q, K)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    O = np.zeros((len(rows), d))
    L = np.zeros(len(rows))
    rc = _load().oracle_forward_rows_masked(B, Hq, Hkv, N, d, *mask.args(causal), float(scale),
                                            _ptr(Q), _ptr(K), _ptr(V), len(rows), _ptr(rows, _L),
                                            _ptr(O), _ptr(L))
    _check(rc, "oracle_forward_rows_masked")
    return O, L


def backward_dq_rows_masked(Q, K, V, dO, causal: bool, scale: float, mask: Mask, rows):
    """backward_dq_rows() under a general mask."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, Hq, Hkv, N, d = _shape(Q, K)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dQ = np.zeros((len(rows), d))
    rc = _load().oracle_backward_dq_rows_masked(B, Hq, Hkv, N, d, *mask.args(causal),
                                                float(scale), _ptr(Q), _ptr(K), _ptr(V),
                                                _ptr(dO), len(rows), _ptr(rows, _L), _ptr(dQ))
    _check(rc, "oracle_backward_dq_rows_masked")
    return dQ


def backward_dkv_cols_masked(Q, K, V, dO, causal: bool, scale: float, mask: Mask, cols):
    """backward_dkv_cols() under a general mask."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, Hq, Hkv, N, d = _shape(Q, K)
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    dK = np.zeros((len(cols), d))
    dV = np.zeros((len(cols), d))
    rc = _load().oracle_backward_dkv_cols_masked(B, Hq, Hkv, N, d, *mask.args(causal),
                                                 float(scale), _ptr(Q), _ptr(K), _ptr(V),
                                                 _ptr(dO), len(cols), _ptr(cols, _L), _ptr(dK),
                                                 _ptr(dV))
    _check(rc, "oracle_backward_dkv_cols_masked")
    return dK, dV


# ----------------------------------------------------------------------------- dropout
def philox4x32_10(counter, key):
    """Philox4x32-10 (Salmon et al., SC'11) of a 4-word counter and 2-word key -> 4 words."""
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in counter])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    out = (ctypes.c_uint32 * 4)()
    _load().oracle_philox4x32_10(c, k, out)
    return tuple(int(x) for x in out)


def dropout_threshold(p: float) -> int:
    """floor((1 - p) 2^32): a key is kept when its Philox word is below this."""
    return int(_load().oracle_dropout_threshold(float(p)))


def dropout_mask(BH: int, N: int, seed: int, offset: int, p: float):
    """Keep decisions Z [BH, N, N] uint8 of every (b*Hq + hq, query, key)."""
    Z = np.zeros((BH, N, N), dtype=np.uint8)
    rc = _load().oracle_dropout_mask(BH, N, int(seed), int(offset), float(p), _ptr(Z, _U8))
    _check(rc, "oracle_dropout_mask")
    return Z


def forward_dropout(Q, K, V, causal: bool, scale: float, p: float, seed: int, offset: int):
    """Forward with dropout: (O [B, Hq, N, d], LSE [B, Hq, N])."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, Hq, Hkv, N, d = _shape(Q, K)
    O = np.zeros((B, Hq, N, d))
    L = np.zeros((B, Hq, N))
    rc = _load().oracle_attention_forward_dropout(B, Hq, Hkv, N, d, int(bool(causal)),
                                                  float(scale), float(p), int(seed), int(offset),
                                                  _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(L))
    _check(rc, "oracle_attention_forward_dropout")
    return O, L


def backward_dropout(Q, K, V, dO, causal: bool, scale: float, p: float, seed: int, offset: int):
    """Backward with dropout: (dQ [B, Hq, N, d], dK, dV [B, Hkv, N, d])."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, Hq, Hkv, N, d = _shape(Q, K)
    dQ = np.zeros((B, Hq, N, d))
    dK = np.zeros((B, Hkv, N, d))
    dV = np.zeros((B, Hkv, N, d))
    rc = _load().oracle_attention_backward_dropout(B, Hq, Hkv, N, d, int(bool(causal)),
                                                   float(scale), float(p), int(seed), int(offset),
                                                   _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ),
                                                   _ptr(dK), _ptr(dV))
    _check(rc, "oracle_attention_backward_dropout")
    return dQ, dK, dV
