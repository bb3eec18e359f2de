"""fp32 forward on the tensor cores (fa_fwd_fp32_tc, three TF32 products per product) against the
fp64 oracle with the fp32 tolerance (max abs <= 1e-5 on O and LSE)."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import FP32_MAX_ABS, f64, max_abs, sample_rows

pytestmark = pytest.mark.gpu


def gpu_tc(flash, Q, K, V, causal, scale):
    dev = helpers.DEVICE
    O, LSE = flash.attention_forward_fp32_tc(*(t.to(dev) for t in (Q, K, V)), causal, scale)
    assert flash.fa_get_device_status() == flash.FA_OK
    return O.cpu(), LSE.cpu()


def test_tiny_fp32_workload(flash, oracle_mod):
    w = WORKLOADS["tiny_fp32"]
    Q, K, V, _ = workload_inputs(w)
    O, LSE = gpu_tc(flash, Q, K, V, w.causal, w.scale)
    Oo, Lo = oracle_mod.forward(f64(Q), f64(K), f64(V), w.causal, w.scale)
    assert max_abs(O, Oo) <= FP32_MAX_ABS and max_abs(LSE, Lo) <= FP32_MAX_ABS


@pytest.mark.parametrize("B,Hq,Hkv,N,causal", [(1, 1, 1, 1, True), (1, 2, 1, 17, False),
                                               (2, 2, 2, 100, True), (1, 4, 2, 129, False),
                                               (1, 2, 2, 300, True), (2, 2, 1, 1000, False),
                                               (1, 1, 1, 513, True)])
def test_small_shapes(flash, oracle_mod, B, Hq, Hkv, N, causal):
    Q, K, V, _ = make_inputs(B, Hq, Hkv, N, 64, seed=800 + N, dtype=torch.float32, with_dO=False)
    O, LSE = gpu_tc(flash, Q, K, V, causal, 0.125)
    Oo, Lo = oracle_mod.forward(f64(Q), f64(K), f64(V), causal, 0.125)
    assert max_abs(O, Oo) <= FP32_MAX_ABS and max_abs(LSE, Lo) <= FP32_MAX_ABS


def test_peaked_scores(flash, oracle_mod):
    """Q x 4: scores spread over ~60, one key dominates many rows.  Each TF32 part keeps 11
    significant bits, so a product of three parts errs by up to about 2^-20 of sum_k |q_k k_k|
    (per score, after the scale); a score error ds moves a softmax weight by a factor e^ds and
    O by at most 2 ds max|v|.  The bound below is that, with the fp32 tolerance as a floor."""
    Q, K, V, _ = make_inputs(1, 2, 2, 700, 64, seed=9, dtype=torch.float32, q_mult=4.0,
                             with_dO=False)
    O, LSE = gpu_tc(flash, Q, K, V, True, 0.125)
    Oo, Lo = oracle_mod.forward(f64(Q), f64(K), f64(V), True, 0.125)
    q, k, v = f64(Q), f64(K), f64(V)
    ds = 2.0 ** -20 * 0.125 * np.max(np.abs(q) @ np.abs(k).transpose(0, 1, 3, 2))
    tol_o = max(FP32_MAX_ABS, 2 * ds * np.abs(v).max())
    tol_l = max(FP32_MAX_ABS, ds)
    assert max_abs(O, Oo) <= tol_o and max_abs(LSE, Lo) <= tol_l, (max_abs(O, Oo), tol_o)


def test_fp32tc_full_size_workload(flash, oracle_mod):
    w = WORKLOADS["fp32tc_n4096"]
    Q, K, V, _ = workload_inputs(w)
    O, LSE = gpu_tc(flash, Q, K, V, w.causal, w.scale)
    rows = sample_rows(w.B, w.Hq, w.N, 96, seed=w.seed)
    Oo, Lo = oracle_mod.forward_rows(f64(Q), f64(K), f64(V), w.causal, w.scale, rows)
    assert max_abs(O.reshape(-1, w.d)[rows], Oo) <= FP32_MAX_ABS
    assert max_abs(LSE.reshape(-1)[rows], Lo) <= FP32_MAX_ABS
