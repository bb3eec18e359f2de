"""Failure detection without a GPU fault: a bounded wait that runs out.

Every mbarrier wait in the library gives up after a time limit, records FA_ERR_DEVICE_TIMEOUT in
the device status word, lets the CTA unwind (copies in flight drained, TMEM freed) and returns;
nothing traps.  This test builds the library with FA_FAULT_INJECT (CTA 0 of the forward never
delivers its first K block, so its MMA warp waits on a barrier that nothing completes) and a
0.2 s wait limit, runs it, reads the status, and then checks that the same process and context
still compute a correct result with the regular library."""
import ctypes

import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import make_inputs
from helpers import BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, f64, max_abs

pytestmark = pytest.mark.gpu


def _load(path):
    L = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.fa_fwd.argtypes = [vp] * 5 + [i] * 6 + [f, vp]
    L.fa_fwd.restype = i
    L.fa_get_device_status.argtypes = [vp]
    L.fa_get_device_status.restype = i
    return L


def test_bounded_wait_times_out_and_context_survives(flash, oracle_mod, tmp_path):
    from exact_attention_89_gb300 import build
    path = build.build(extra_flags=["-DFA_FAULT_INJECT", "-DFA_WAIT_NS=200000000ull"],
                       out_dir=str(tmp_path))
    faulty = _load(path)
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
