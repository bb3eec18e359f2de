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


# ---------------------------------------------------------------------------- backward
def gpu_tc_bwd(flash, Q, K, V, dO, causal, scale):
    """fa_fwd_fp32_tc then fa_bwd_fp32_tc on the device; returns dQ, dK, dV on the host."""
    dev = helpers.DEVICE
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    O, LSE = flash.attention_forward_fp32_tc(q, k, v, causal, scale)
    dQ, dK, dV = flash.attention_backward_fp32_tc(q, k, v, O, do, LSE, causal, scale)
    assert flash.fa_get_device_status() == flash.FA_OK
    return dQ.cpu(), dK.cpu(), dV.cpu()


def grad_tol(ref) -> float:
    """fp32 tolerance for a gradient, relative to its largest element.  A product of three TF32
    parts errs by about 2^-21 of the sum of |terms|, and a gradient element sums up to N such
    terms (dV_k = sum_q P_qk dO_q), so its error scales with the gradient's magnitude rather
    than staying under an absolute 1e-5 once |dV| reaches 10 or more; 1e-5 of max|ref| still
    fails by ~50x a path that used one TF32 product (relative error 2^-11)."""
    return FP32_MAX_ABS * max(1.0, float(np.abs(np.asarray(ref)).max()))


def check_bwd(flash, oracle_mod, Q, K, V, dO, causal, scale, relative=True):
    dQ, dK, dV = gpu_tc_bwd(flash, Q, K, V, dO, causal, scale)
    dQo, dKo, dVo = oracle_mod.backward(f64(Q), f64(K), f64(V), f64(dO), causal, scale)
    errs = {n: (max_abs(a, r), grad_tol(r) if relative else FP32_MAX_ABS)
            for n, a, r in (("dQ", dQ, dQo), ("dK", dK, dKo), ("dV", dV, dVo))}
    assert all(e <= t for e, t in errs.values()), errs


def test_bwd_tiny_fp32_workload(flash, oracle_mod):
    """B1 H1 N256 d64 non-causal: every gradient element within 1e-5 of the fp64 oracle."""
    w = WORKLOADS["tiny_fp32"]
    Q, K, V, dO = workload_inputs(w)
    check_bwd(flash, oracle_mod, Q, K, V, dO, w.causal, w.scale, relative=False)


@pytest.mark.parametrize("B,Hq,Hkv,N,causal", [(1, 1, 1, 1, True), (1, 2, 1, 17, False),
                                               (2, 2, 2, 100, True), (1, 4, 2, 129, False),
                                               (1, 2, 2, 300, True), (2, 2, 1, 1000, False),
                                               (1, 4, 1, 513, True), (1, 1, 1, 160, True)])
def test_bwd_small_shapes(flash, oracle_mod, B, Hq, Hkv, N, causal):
    """Ragged N (one row, a partial 32-row block, partial 128-row tiles), GQA groups of 1-4."""
    Q, K, V, dO = make_inputs(B, Hq, Hkv, N, 64, seed=900 + N, dtype=torch.float32)
    check_bwd(flash, oracle_mod, Q, K, V, dO, causal, 0.125)


def test_bwd_matches_simt_path(flash):
    """The tensor-core and CUDA-core fp32 backward passes agree to the fp32 tolerance (relative
    to each gradient's largest element, as against the oracle)."""
    dev = helpers.DEVICE
    Q, K, V, dO = (t.to(dev) for t in make_inputs(2, 4, 2, 700, 64, seed=31, dtype=torch.float32))
    O, LSE = flash.attention_forward(Q, K, V, True, 0.125)
    tc = flash.attention_backward_fp32_tc(Q, K, V, O, dO, LSE, True, 0.125)
    simt = flash.attention_backward(Q, K, V, O, dO, LSE, True, 0.125)
    assert flash.fa_get_device_status() == flash.FA_OK
    for a, b in zip(tc, simt):
        assert max_abs(a.cpu(), b.cpu()) <= grad_tol(b.cpu())


def test_bwd_fp32tc_full_size_workload(flash, oracle_mod):
    """B2 H16 N4096 d64 causal: sampled dQ rows and dK / dV rows against the oracle."""
    w = WORKLOADS["fp32tc_n4096"]
    Q, K, V, dO = workload_inputs(w)
    dQ, dK, dV = gpu_tc_bwd(flash, Q, K, V, dO, w.causal, w.scale)
    q, k, v, do = f64(Q), f64(K), f64(V), f64(dO)
    rows = sample_rows(w.B, w.Hq, w.N, 64, seed=w.seed)
    dQo = oracle_mod.backward_dq_rows(q, k, v, do, w.causal, w.scale, rows)
    assert max_abs(dQ.reshape(-1, w.d)[rows], dQo) <= grad_tol(dQo)
    cols = sample_rows(w.B, w.Hkv, w.N, 64, seed=w.seed + 1)
    dKo, dVo = oracle_mod.backward_dkv_cols(q, k, v, do, w.causal, w.scale, cols)
    assert max_abs(dK.reshape(-1, w.d)[cols], dKo) <= grad_tol(dKo)
    assert max_abs(dV.reshape(-1, w.d)[cols], dVo) <= grad_tol(dVo)
