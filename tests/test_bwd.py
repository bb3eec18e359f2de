"""bf16 backward on tcgen05 (fa_bwd) against the fp64 oracle on the same seeded inputs.

Tolerance: relative Frobenius error <= 2e-2 for each of dQ, dK, dV.  The GPU backward consumes
the GPU forward's O and LSE (as a user would); the oracle recomputes everything in fp64 from the
same bf16 inputs.  Full-size workloads are checked on one whole (batch, KV-group) slice (N <= 8192)
and on sampled dQ rows and dK/dV rows computed by the oracle one by one."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import BF16_GRAD_REL_FRO, f64, group_slice, rel_fro, sample_rows

pytestmark = pytest.mark.gpu


def gpu_fwd_bwd(flash, Q, K, V, dO, causal, scale):
    dev = helpers.DEVICE
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    O, LSE = flash.attention_forward(q, k, v, causal, scale)
    dQ, dK, dV = flash.attention_backward(q, k, v, O, do, LSE, causal, scale)
    assert flash.fa_get_device_status() == flash.FA_OK
    return dQ.cpu(), dK.cpu(), dV.cpu()


def assert_grads_close(got, ref, what=""):
    errs = [rel_fro(g, r) for g, r in zip(got, ref)]
    assert all(e <= BF16_GRAD_REL_FRO for e in errs), (what, errs)
    return errs


SMALL = [
    # B, Hq, Hkv, N, causal
    (1, 1, 1, 1, False), (1, 1, 1, 1, True), (1, 2, 1, 17, True), (2, 2, 2, 127, False),
    (1, 4, 2, 128, True), (1, 2, 2, 129, False), (2, 4, 1, 200, True), (1, 2, 1, 256, True),
    (1, 2, 2, 300, False), (1, 8, 2, 513, True), (2, 2, 1, 1000, False),
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B,Hq,Hkv,N,causal", SMALL)
def test_backward_small_shapes(flash, oracle_mod, B, Hq, Hkv, N, causal, d):
    Q, K, V, dO = make_inputs(B, Hq, Hkv, N, d, seed=200 + N + d)
    scale = 1.0 / np.sqrt(d)
    got = gpu_fwd_bwd(flash, Q, K, V, dO, causal, scale)
    ref = oracle_mod.backward(f64(Q), f64(K), f64(V), f64(dO), causal, scale)
    assert_grads_close(got, ref)


def test_backward_invariants_on_gpu(flash):
    """sum_j dK_j = 0 (rows of dS sum to 0) and sum_j dV_j = sum over the group of sum_i dO_i,
    checked on the GPU result alone (these hold at any size)."""
    Q, K, V, dO = make_inputs(1, 4, 2, 700, 128, seed=9)
    dQ, dK, dV = gpu_fwd_bwd(flash, Q, K, V, dO, True, 1 / np.sqrt(128))
    sdv = dV.double().sum(2)
    ref = dO.double().reshape(1, 2, 2, 700, 128).sum((2, 3))
    assert rel_fro(sdv, ref) <= BF16_GRAD_REL_FRO
    assert float(dK.double().sum(2).abs().max()) <= 0.05 * float(dK.double().abs().sum(2).max())


@pytest.mark.parametrize("name", ["causal_n4096", "gqa_n8192", "long_n32768",
                                  "causal_d64_n4096"])
def test_backward_full_size_workloads(flash, oracle_mod, name):
    w = WORKLOADS[name]
    Q, K, V, dO = workload_inputs(w)
    dQ, dK, dV = gpu_fwd_bwd(flash, Q, K, V, dO, w.causal, w.scale)
    G = w.Hq // w.Hkv
    b, hk = 0, w.Hkv - 1
    q, k, v, do = (f64(t) for t in group_slice(Q, K, V, dO, b, hk))
    if w.N <= 8192:
        ref = oracle_mod.backward(q, k, v, do, w.causal, w.scale)
        got = (dQ[b:b + 1, hk * G:(hk + 1) * G].reshape(ref[0].shape),
               dK[b:b + 1, hk:hk + 1].reshape(ref[1].shape),
               dV[b:b + 1, hk:hk + 1].reshape(ref[2].shape))
        assert_grads_close(got, ref, name + " group")
    # sampled rows of the same group (sub-problem indices) and across all heads for dQ
    rows = sample_rows(1, G, w.N, 48, seed=w.seed)
    dq_ref = oracle_mod.backward_dq_rows(q, k, v, do, w.causal, w.scale, rows)
    dq_got = dQ[b:b + 1, hk * G:(hk + 1) * G].reshape(-1, w.d)[rows]
    cols = sample_rows(1, 1, w.N, 48, seed=w.seed + 1)
    dk_ref, dv_ref = oracle_mod.backward_dkv_cols(q, k, v, do, w.causal, w.scale, cols)
    dk_got = dK[b:b + 1, hk:hk + 1].reshape(-1, w.d)[cols]
    dv_got = dV[b:b + 1, hk:hk + 1].reshape(-1, w.d)[cols]
    assert_grads_close((dq_got, dk_got, dv_got), (dq_ref, dk_ref, dv_ref), name + " rows")
