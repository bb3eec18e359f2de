"""Failure detection without a GPU fault: a bounded wait that runs out.

Every mbarrier wait in the library gives up after a time limit, records FA_ERR_DEVICE_TIMEOUT in
the device status word, lets the CTA unwind (copies in flight drained, TMEM freed) and returns;
nothing traps.  These tests build the library with FA_FAULT_INJECT and a 0.2 s wait limit:
CTA 0 of the forward never delivers its first K block, so its MMA warp waits on a barrier that
nothing completes; CTA 0 of the backward stops delivering Q / dO tiles after the first fill of its
ring, so its S^T / dP^T issuer waits in vain while the other roles (second MMA issuer, gradient
and dQ-drain warps) must unwind around it; in the deterministic backward the other CTAs of its
head then wait for dQ turns that CTA 0 never passes, and those waits run out as well.  Each test runs the faulty build, reads the status,
and then checks that the same process and context still compute a correct result with the
regular library."""
import ctypes

import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import make_inputs
from helpers import BF16_GRAD_REL_FRO, BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, f64, max_abs, rel_fro

pytestmark = pytest.mark.gpu


def _load(path):
    L = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.fa_fwd.argtypes = [vp] * 5 + [i] * 6 + [f, vp]
    L.fa_fwd.restype = i
    L.fa_bwd.argtypes = [vp] * 9 + [i] * 6 + [f, vp, ctypes.c_size_t, vp]
    L.fa_bwd.restype = i
    L.fa_bwd_deterministic.argtypes = [vp] * 9 + [i] * 6 + [f, vp, ctypes.c_size_t, vp]
    L.fa_bwd_deterministic.restype = i
    L.fa_get_device_status.argtypes = [vp]
    L.fa_get_device_status.restype = i
    return L


@pytest.fixture(scope="module")
def faulty(flash, tmp_path_factory):
    """The library built with the injected stalls and a 0.2 s wait limit."""
    from exact_attention_89_gb300 import build
    path = build.build(extra_flags=["-DFA_FAULT_INJECT", "-DFA_WAIT_NS=200000000ull"],
                       out_dir=str(tmp_path_factory.mktemp("faulty")))
    return _load(path)


def test_bounded_wait_times_out_and_context_survives(flash, oracle_mod, faulty):
    dev = helpers.DEVICE
    B, Hq, Hkv, N, d = 1, 2, 1, 700, 128
    scale = 1.0 / np.sqrt(d)
    Q, K, V, _ = make_inputs(B, Hq, Hkv, N, d, seed=77, with_dO=False)
    q, k, v = (t.to(dev) for t in (Q, K, V))
    O = torch.empty_like(q)
    LSE = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = faulty.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), LSE.data_ptr(),
                       B, Hq, Hkv, N, d, 1, scale, stream)
    assert st == flash.FA_OK                      # the launch itself is fine
    assert faulty.fa_get_device_status(stream) == flash.FA_ERR_DEVICE_TIMEOUT
    assert faulty.fa_get_device_status(stream) == flash.FA_OK   # read-and-clear
    # the context is still usable: the regular library computes the right answer
    O2, LSE2 = flash.attention_forward(q, k, v, True, scale)
    torch.cuda.synchronize()
    assert flash.fa_get_device_status() == flash.FA_OK
    Oo, Lo = oracle_mod.forward(f64(Q), f64(K), f64(V), True, scale)
    assert max_abs(O2.cpu(), Oo) <= BF16_O_MAX_ABS
    assert max_abs(LSE2.cpu(), Lo) <= BF16_LSE_MAX_ABS


def test_backward_bounded_wait_times_out_and_context_survives(flash, oracle_mod, faulty):
    dev = helpers.DEVICE
    B, Hq, Hkv, N, d = 1, 4, 2, 700, 128
    scale = 1.0 / np.sqrt(d)
    Q, K, V, dO = make_inputs(B, Hq, Hkv, N, d, seed=78)
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    O, LSE = flash.attention_forward(q, k, v, True, scale)    # regular library
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = flash.fa_bwd_workspace_bytes(B, Hq, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = faulty.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), do.data_ptr(),
                       LSE.data_ptr(), dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(),
                       B, Hq, Hkv, N, d, 1, scale, ws.data_ptr(), nbytes, stream)
    assert st == flash.FA_OK                      # the launch itself is fine
    assert faulty.fa_get_device_status(stream) == flash.FA_ERR_DEVICE_TIMEOUT
    assert faulty.fa_get_device_status(stream) == flash.FA_OK   # read-and-clear
    # the context is still usable: the regular library's backward gives the right gradients
    got = flash.attention_backward(q, k, v, O, do, LSE, True, scale)
    torch.cuda.synchronize()
    assert flash.fa_get_device_status() == flash.FA_OK
    ref = oracle_mod.backward(f64(Q), f64(K), f64(V), f64(dO), True, scale)
    errs = [rel_fro(g.cpu(), r) for g, r in zip(got, ref)]
    assert all(e <= BF16_GRAD_REL_FRO for e in errs), errs


def test_deterministic_backward_turn_waits_time_out_and_context_survives(flash, oracle_mod,
                                                                         faulty):
    """CTA 0 of the deterministic backward is the first key block in the reduction order (the
    last block of head 0); without causal masking it has more steps than the ring holds, so the
    injected stall leaves its later dQ turns unpassed and the next key block's turn wait runs
    out (and ends the others')."""
    dev = helpers.DEVICE
    B, Hq, Hkv, N, d = 1, 4, 2, 700, 128
    scale = 1.0 / np.sqrt(d)
    Q, K, V, dO = make_inputs(B, Hq, Hkv, N, d, seed=79)
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    O, LSE = flash.attention_forward(q, k, v, False, scale)    # regular library
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = flash.fa_bwd_deterministic_workspace_bytes(B, Hq, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = faulty.fa_bwd_deterministic(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(),
                                     do.data_ptr(), LSE.data_ptr(), dQ.data_ptr(), dK.data_ptr(),
                                     dV.data_ptr(), B, Hq, Hkv, N, d, 0, scale, ws.data_ptr(),
                                     nbytes, stream)
    assert st == flash.FA_OK                      # the launch itself is fine
    assert faulty.fa_get_device_status(stream) == flash.FA_ERR_DEVICE_TIMEOUT
    assert faulty.fa_get_device_status(stream) == flash.FA_OK   # read-and-clear
    # the same workspace (counters left mid-way, abort word set) serves the regular library:
    # each call clears both before its main kernel
    got = flash.attention_backward(q, k, v, O, do, LSE, False, scale, workspace=ws,
                                   deterministic=True)
    torch.cuda.synchronize()
    assert flash.fa_get_device_status() == flash.FA_OK
    ref = oracle_mod.backward(f64(Q), f64(K), f64(V), f64(dO), False, scale)
    errs = [rel_fro(g.cpu(), r) for g, r in zip(got, ref)]
    assert all(e <= BF16_GRAD_REL_FRO for e in errs), errs
