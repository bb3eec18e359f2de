"""The forward in the key/value-outer loop order (fa_fwd_kvouter) against the fp64 oracle, within
the bf16 forward tolerances (O max abs <= 1e-2, mean abs <= 1e-3, LSE max abs <= 1e-3): small
shapes and the full-size workload over every element."""
import numpy as np
import pytest

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import (BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, BF16_O_MEAN_ABS, ErrorTally, f64, max_abs,
                     mean_abs)

pytestmark = pytest.mark.gpu


def gpu_kvouter(flash, Q, K, V, causal, scale):
    dev = helpers.DEVICE
    O, LSE = flash.attention_forward_kvouter(*(t.to(dev) for t in (Q, K, V)), causal, scale)
    assert flash.fa_get_device_status() == flash.FA_OK
    return O.cpu(), LSE.cpu()


def assert_close(O, LSE, Oo, Lo, what=""):
    e = (max_abs(O, Oo), mean_abs(O, Oo), max_abs(LSE, Lo))
    assert e[0] <= BF16_O_MAX_ABS and e[1] <= BF16_O_MEAN_ABS and e[2] <= BF16_LSE_MAX_ABS, (what, e)


@pytest.mark.parametrize("B,Hq,Hkv,N,causal", [(1, 1, 1, 1, True), (1, 2, 1, 17, False),
                                               (2, 2, 2, 129, True), (1, 4, 2, 300, False),
                                               (1, 2, 2, 513, True), (2, 2, 1, 1000, True),
                                               (1, 2, 2, 777, False)])
def test_kvouter_small_shapes(flash, oracle_mod, B, Hq, Hkv, N, causal):
    Q, K, V, _ = make_inputs(B, Hq, Hkv, N, 128, seed=700 + N, with_dO=False)
    scale = 1.0 / np.sqrt(128)
    O, LSE = gpu_kvouter(flash, Q, K, V, causal, scale)
    Oo, Lo = oracle_mod.forward(f64(Q), f64(K), f64(V), causal, scale)
    assert_close(O, LSE, Oo, Lo)


def test_kvouter_full_size_workload(flash, oracle_mod):
    """The benchmark's causal B2 H32 N4096 workload: every element against the oracle (a few
    heads per oracle call)."""
    w = WORKLOADS["kvouter_n4096"]
    Q, K, V, _ = workload_inputs(w)
    O, LSE = gpu_kvouter(flash, Q, K, V, w.causal, w.scale)
    q64, k64, v64 = f64(Q), f64(K), f64(V)
    O2, L2 = O.reshape(w.B * w.Hq, w.N, w.d), LSE.reshape(w.B * w.Hq, w.N)
    to, tl = ErrorTally(), ErrorTally()
    for h0 in range(0, w.B * w.Hq, 8):
        heads = list(range(h0, min(h0 + 8, w.B * w.Hq)))
        Oo, Lo = oracle_mod.forward(q64, k64, v64, w.causal, w.scale, heads=heads)
        to.add(O2[heads], Oo, label="heads %d.." % h0)
        tl.add(L2[heads], Lo)
    print("[parity] kvouter_n4096 forward, every element: O max abs %.3e mean abs %.3e, LSE max "
          "abs %.3e; worst O element %s" % (to.max_abs, to.mean_abs, tl.max_abs, to.worst))
    assert (to.max_abs <= BF16_O_MAX_ABS and to.mean_abs <= BF16_O_MEAN_ABS
            and tl.max_abs <= BF16_LSE_MAX_ABS), (to.max_abs, to.mean_abs, tl.max_abs)
