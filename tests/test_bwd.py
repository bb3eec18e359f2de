"""bf16 backward on tcgen05 (fa_bwd) against the fp64 oracle on the same seeded inputs.

Tolerance: relative Frobenius error <= 2e-2 for each of dQ, dK, dV.  The GPU backward consumes
the GPU forward's O and LSE (as a user would); the oracle recomputes everything in fp64 from the
same bf16 inputs.  Full-size workloads up to N = 8192 are checked over every element; the
N = 32768 workload over every dQ, dK and dV element of four whole KV groups drawn by seed plus
dQ rows sampled over all heads."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import (BF16_GRAD_REL_FRO, ErrorTally, chosen_groups, f64, group_slice, rel_fro,
                     sample_rows)

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


# Workloads whose every element the oracle checks (a few KV groups per oracle call), and the
# one too long for that: its check covers whole KV groups drawn by seed.
EVERY_ELEMENT = ["causal_n4096", "gqa_n8192", "causal_d64_n4096"]
WHOLE_GROUPS = {"long_n32768": 4}


@pytest.mark.parametrize("name", EVERY_ELEMENT)
def test_backward_full_size_every_element(flash, oracle_mod, name):
    """Full-size workloads in the launch configuration the benchmark times: every element of dQ,
    dK and dV against the oracle, which runs a few KV groups at a time."""
    w = WORKLOADS[name]
    Q, K, V, dO = workload_inputs(w)
    dQ, dK, dV = gpu_fwd_bwd(flash, Q, K, V, dO, w.causal, w.scale)
    G = w.Hq // w.Hkv
    q64, k64, v64, do64 = f64(Q), f64(K), f64(V), f64(dO)
    dQg = dQ.reshape(w.B * w.Hkv, G, w.N, w.d)
    dKg, dVg = dK.reshape(w.B * w.Hkv, w.N, w.d), dV.reshape(w.B * w.Hkv, w.N, w.d)
    tq, tk, tv = ErrorTally(), ErrorTally(), ErrorTally()
    step = max(1, 8 // G)
    for g0 in range(0, w.B * w.Hkv, step):
        groups = list(range(g0, min(g0 + step, w.B * w.Hkv)))
        rq, rk, rv = oracle_mod.backward(q64, k64, v64, do64, w.causal, w.scale, groups=groups)
        tq.add(dQg[groups], rq)
        tk.add(dKg[groups], rk)
        tv.add(dVg[groups], rv)
    errs = (tq.rel_fro, tk.rel_fro, tv.rel_fro)
    print("[parity] %s backward, every element: rel fro dQ %.3e dK %.3e dV %.3e" % ((name,) + errs))
    assert tq.count == w.B * w.Hq * w.N * w.d and tk.count == w.B * w.Hkv * w.N * w.d
    assert all(e <= BF16_GRAD_REL_FRO for e in errs), (name, errs)


@pytest.mark.parametrize("name", sorted(WHOLE_GROUPS))
def test_backward_full_size_whole_groups(flash, oracle_mod, name):
    """The longest workload: every dQ row and every dK / dV row of KV groups drawn by seed
    (exact for those heads: groups are independent), plus dQ rows sampled over all heads."""
    w = WORKLOADS[name]
    Q, K, V, dO = workload_inputs(w)
    dQ, dK, dV = gpu_fwd_bwd(flash, Q, K, V, dO, w.causal, w.scale)
    G = w.Hq // w.Hkv
    tq, tk, tv = ErrorTally(), ErrorTally(), ErrorTally()
    groups = chosen_groups(w.B * w.Hkv, WHOLE_GROUPS[name], w.seed)
    for bk in groups:
        b, hk = divmod(bk, w.Hkv)
        q, k, v, do = (f64(t) for t in group_slice(Q, K, V, dO, b, hk))
        # the full backward of the group's sub-problem (it holds one N x N matrix, 8.6 GB here)
        rq, rk, rv = oracle_mod.backward(q, k, v, do, w.causal, w.scale)
        tq.add(dQ[b, hk * G:(hk + 1) * G], rq[0])
        tk.add(dK[b, hk], rk[0, 0])
        tv.add(dV[b, hk], rv[0, 0])
    errs = (tq.rel_fro, tk.rel_fro, tv.rel_fro)
    rows = sample_rows(w.B, w.Hq, w.N, 48, seed=w.seed)
    dq_rows = oracle_mod.backward_dq_rows(f64(Q), f64(K), f64(V), f64(dO), w.causal, w.scale, rows)
    err_rows = rel_fro(dQ.reshape(-1, w.d)[rows], dq_rows)
    print("[parity] %s backward, groups %s: rel fro dQ %.3e dK %.3e dV %.3e; %d sampled dQ rows "
          "%.3e" % ((name, groups) + errs + (len(rows), err_rows)))
    assert all(e <= BF16_GRAD_REL_FRO for e in errs + (err_rows,)), (name, errs, err_rows)
