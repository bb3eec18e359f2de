"""The debug bounds-check build (FA_DEBUG_BOUNDS), the stand-in for a memory checker.

Built with FA_DEBUG_BOUNDS, the bf16 forward and backward kernels check the index of each of
their computed plain global accesses (O and LSE rows written by the forward; LSE and D rows read
and dQ accumulator rows reduced by the backward) against the extent of its buffer; an index out
of range is recorded as FA_ERR_DEVICE_BOUNDS in the status word and the access is skipped,
nothing traps.  The first test runs that build on small ragged shapes (tile tails, odd numbers
of key blocks, GQA, both head dims): no check may fire and the results must match the oracle.
The second builds it with FA_DEBUG_BOUNDS_SHRINK=1, which makes every checked extent one row
shorter, so the last row's accesses are reported and skipped (no access leaves its buffer):
the status must read FA_ERR_DEVICE_BOUNDS, once, for the forward and for the backward."""
import ctypes

import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import make_inputs
from helpers import (BF16_GRAD_REL_FRO, BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, f64, max_abs,
                     rel_fro)

pytestmark = pytest.mark.gpu


def _load(path):
    L = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.fa_fwd.argtypes = [vp] * 5 + [i] * 6 + [f, vp]
    L.fa_fwd.restype = i
    L.fa_bwd.argtypes = [vp] * 9 + [i] * 6 + [f, vp, ctypes.c_size_t, vp]
    L.fa_bwd.restype = i
    L.fa_get_device_status.argtypes = [vp]
    L.fa_get_device_status.restype = i
    return L


def _build(tmp_path_factory, flags, name):
    from exact_attention_89_gb300 import build
    return _load(build.build(extra_flags=flags, out_dir=str(tmp_path_factory.mktemp(name))))


@pytest.fixture(scope="module")
def checked(flash, tmp_path_factory):
    return _build(tmp_path_factory, ["-DFA_DEBUG_BOUNDS"], "bounds")


@pytest.fixture(scope="module")
def shrunk(flash, tmp_path_factory):
    return _build(tmp_path_factory, ["-DFA_DEBUG_BOUNDS", "-DFA_DEBUG_BOUNDS_SHRINK=1"], "shrunk")


def _run(L, flash, Q, K, V, dO, causal, scale, O=None, LSE=None):
    """fa_fwd (unless O / LSE are given) then fa_bwd of library L; returns tensors and statuses."""
    dev = helpers.DEVICE
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    st_f = flash.FA_OK
    if O is None:
        O = torch.empty_like(q)
        LSE = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
        assert L.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), LSE.data_ptr(),
                        B, Hq, Hkv, N, d, int(causal), scale, stream) == flash.FA_OK
        st_f = L.fa_get_device_status(stream)
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = flash.fa_bwd_workspace_bytes(B, Hq, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    assert L.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), do.data_ptr(),
                    LSE.data_ptr(), dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), B, Hq, Hkv, N, d,
                    int(causal), scale, ws.data_ptr(), nbytes, stream) == flash.FA_OK
    st_b = L.fa_get_device_status(stream)
    return O, LSE, (dQ, dK, dV), st_f, st_b


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [(1, 2, 1, 17, 128, True), (2, 4, 2, 300, 128, False),
                                                 (1, 8, 2, 513, 128, True), (2, 2, 2, 129, 64, True),
                                                 (1, 4, 1, 1000, 64, False)])
def test_checked_build_reports_nothing_on_ragged_shapes(flash, oracle_mod, checked,
                                                        B, Hq, Hkv, N, d, causal):
    Q, K, V, dO = make_inputs(B, Hq, Hkv, N, d, seed=500 + N + d)
    scale = 1.0 / np.sqrt(d)
    O, LSE, grads, st_f, st_b = _run(checked, flash, Q, K, V, dO, causal, scale)
    assert (st_f, st_b) == (flash.FA_OK, flash.FA_OK)
    Oo, Lo = oracle_mod.forward(f64(Q), f64(K), f64(V), causal, scale)
    assert max_abs(O.cpu(), Oo) <= BF16_O_MAX_ABS and max_abs(LSE.cpu(), Lo) <= BF16_LSE_MAX_ABS
    ref = oracle_mod.backward(f64(Q), f64(K), f64(V), f64(dO), causal, scale)
    errs = [rel_fro(g.cpu(), r) for g, r in zip(grads, ref)]
    assert all(e <= BF16_GRAD_REL_FRO for e in errs), errs


@pytest.mark.parametrize("d", [128, 64])
def test_shrunk_extents_are_reported_not_faulted(flash, shrunk, d):
    Q, K, V, dO = make_inputs(1, 4, 2, 300, d, seed=600 + d)
    scale = 1.0 / np.sqrt(d)
    stream = torch.cuda.current_stream().cuda_stream
    _, _, _, st_f, st_b = _run(shrunk, flash, Q, K, V, dO, True, scale)
    assert st_f == flash.FA_ERR_DEVICE_BOUNDS          # the forward's last O / LSE row
    assert st_b == flash.FA_ERR_DEVICE_BOUNDS          # the backward's last LSE / D / dQ row
    assert shrunk.fa_get_device_status(stream) == flash.FA_OK   # read and cleared
    # the regular library is unaffected
    dev = helpers.DEVICE
    O, LSE = flash.attention_forward(Q.to(dev), K.to(dev), V.to(dev), True, scale)
    torch.cuda.synchronize()
    assert flash.fa_get_device_status() == flash.FA_OK
