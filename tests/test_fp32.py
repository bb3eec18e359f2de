"""fp32 SIMT path (fa_fwd_fp32 / fa_bwd_fp32) against the fp64 oracle, element by element.
Tolerance: max abs error <= 1e-5 on O, LSE, dQ, dK, dV."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import FP32_MAX_ABS, f64, max_abs

pytestmark = pytest.mark.gpu


def run_fp32(flash, Q, K, V, dO, causal, scale):
    dev = helpers.DEVICE
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    O, LSE = flash.attention_forward(q, k, v, causal, scale)
    dQ, dK, dV = flash.attention_backward(q, k, v, O, do, LSE, causal, scale)
    torch.cuda.synchronize()
    assert flash.fa_get_device_status() == flash.FA_OK
    return [t.cpu() for t in (O, LSE, dQ, dK, dV)]


def check_all(flash, oracle_mod, Q, K, V, dO, causal, scale, tol=FP32_MAX_ABS):
    O, LSE, dQ, dK, dV = run_fp32(flash, Q, K, V, dO, causal, scale)
    qa, ka, va, doa = (f64(t) for t in (Q, K, V, dO))
    Oo, Lo = oracle_mod.forward(qa, ka, va, causal, scale)
    dQo, dKo, dVo = oracle_mod.backward(qa, ka, va, doa, causal, scale)
    errs = {"O": max_abs(O, Oo), "LSE": max_abs(LSE, Lo), "dQ": max_abs(dQ, dQo),
            "dK": max_abs(dK, dKo), "dV": max_abs(dV, dVo)}
    assert all(e <= tol for e in errs.values()), errs
    return errs


def test_tiny_fp32_workload(flash, oracle_mod):
    """B1 H1 N256 d64 non-causal fp32, seed 0: every element within 1e-5 of the oracle."""
    w = WORKLOADS["tiny_fp32"]
    Q, K, V, dO = workload_inputs(w)
    check_all(flash, oracle_mod, Q, K, V, dO, w.causal, w.scale)


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [
    (1, 1, 1, 1, 64, False), (1, 1, 1, 1, 64, True), (2, 2, 1, 17, 8, True),
    (1, 4, 2, 129, 128, True), (1, 3, 3, 200, 33, False), (2, 4, 1, 64, 100, True)])
def test_fp32_edge_shapes(flash, oracle_mod, B, Hq, Hkv, N, d, causal):
    Q, K, V, dO = make_inputs(B, Hq, Hkv, N, d, seed=11 + N + d, dtype=torch.float32)
    check_all(flash, oracle_mod, Q, K, V, dO, causal, 1.0 / np.sqrt(d))
