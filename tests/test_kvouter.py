"""The forward in the key/value-outer loop order (fa_fwd_kvouter) against the fp64 oracle: the
same O and LSE as the query-outer forward, within the bf16 forward tolerances (O max abs <= 1e-2,
mean abs <= 1e-3, LSE max abs <= 1e-3)."""
import numpy as np
import pytest

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import (BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, BF16_O_MEAN_ABS, f64, max_abs, mean_abs,
                     sample_rows)

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
    w = WORKLOADS["kvouter_n4096"]
    Q, K, V, _ = workload_inputs(w)
    O, LSE = gpu_kvouter(flash, Q, K, V, w.causal, w.scale)
    rows = sample_rows(w.B, w.Hq, w.N, 96, seed=w.seed)
    Oo, Lo = oracle_mod.forward_rows(f64(Q), f64(K), f64(V), w.causal, w.scale, rows)
    assert_close(O.reshape(-1, w.d)[rows], LSE.reshape(-1)[rows], Oo, Lo)
    dev = helpers.DEVICE
    O1, L1 = flash.attention_forward(*(t.to(dev) for t in (Q, K, V)), w.causal, w.scale)
    assert max_abs(O, O1.cpu()) <= BF16_O_MAX_ABS and max_abs(LSE, L1.cpu()) <= BF16_LSE_MAX_ABS
