"""bf16 forward on tcgen05 (fa_fwd) against the fp64 oracle on the same seeded inputs.

Tolerances: O max abs <= 1e-2 and mean abs <= 1e-3; LSE max abs <= 1e-3.
Small shapes are compared over every element; the full-size workloads are compared over whole
(batch, KV-group) slices or sampled rows that the oracle computes one by one."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import (BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, BF16_O_MEAN_ABS, f64, group_slice,
                     max_abs, mean_abs, sample_rows)

pytestmark = pytest.mark.gpu


def gpu_forward(flash, Q, K, V, causal, scale):
    dev = helpers.DEVICE
    q, k, v = (t.to(dev) for t in (Q, K, V))
    O, LSE = flash.attention_forward(q, k, v, causal, scale)
    assert flash.fa_get_device_status() == flash.FA_OK
    return O.cpu(), LSE.cpu()


def assert_fwd_close(O, LSE, Oo, Lo, what=""):
    e = (max_abs(O, Oo), mean_abs(O, Oo), max_abs(LSE, Lo))
    assert e[0] <= BF16_O_MAX_ABS and e[1] <= BF16_O_MEAN_ABS and e[2] <= BF16_LSE_MAX_ABS, (what, e)
    return e


SMALL = [
    # B, Hq, Hkv, N, d, causal
    (1, 1, 1, 1, 128, False), (1, 1, 1, 1, 64, True),
    (1, 2, 1, 17, 128, True), (2, 2, 2, 127, 64, False),
    (1, 4, 2, 128, 128, True), (1, 2, 2, 129, 128, False),
    (2, 4, 1, 200, 64, True), (1, 2, 1, 256, 128, True),
    (1, 2, 2, 300, 128, False), (1, 8, 2, 513, 128, True),
    (1, 4, 4, 640, 64, True), (2, 2, 1, 1000, 128, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", SMALL)
def test_forward_small_shapes(flash, oracle_mod, B, Hq, Hkv, N, d, causal):
    Q, K, V, _ = make_inputs(B, Hq, Hkv, N, d, seed=100 + N + d, with_dO=False)
    scale = 1.0 / np.sqrt(d)
    O, LSE = gpu_forward(flash, Q, K, V, causal, scale)
    Oo, Lo = oracle_mod.forward(f64(Q), f64(K), f64(V), causal, scale)
    assert_fwd_close(O, LSE, Oo, Lo)


def test_forward_single_key_returns_v0(flash):
    """N = 1: the only weight is 1, so O equals V exactly and LSE equals the scaled score."""
    Q, K, V, _ = make_inputs(2, 4, 2, 1, 128, seed=5, with_dO=False)
    O, LSE = gpu_forward(flash, Q, K, V, True, 0.125)
    assert torch.equal(O, V.repeat_interleave(2, dim=1))
    s = 0.125 * (Q.float() * K.float().repeat_interleave(2, dim=1)).sum(-1)
    assert torch.allclose(LSE, s, atol=1e-5, rtol=0)


def test_forward_equal_scores_give_mean(flash):
    """Q = 0: every allowed key gets the same weight; causal row i is the mean of V[:i+1]."""
    _, K, V, _ = make_inputs(1, 2, 2, 300, 128, seed=6, with_dO=False)
    Q = torch.zeros(1, 2, 300, 128, dtype=torch.bfloat16)
    O, LSE = gpu_forward(flash, Q, K, V, True, 0.1)
    ref = V.double().cumsum(2) / torch.arange(1, 301, dtype=torch.float64).view(1, 1, -1, 1)
    assert max_abs(O, ref) <= BF16_O_MAX_ABS
    assert max_abs(LSE, torch.log(torch.arange(1, 301, dtype=torch.float64))) <= BF16_LSE_MAX_ABS


def test_forward_fwd_d64_workload(flash, oracle_mod):
    """B4 H16 N1024 d64 non-causal, seed 1: every element against the oracle."""
    w = WORKLOADS["fwd_d64"]
    Q, K, V, _ = workload_inputs(w)
    O, LSE = gpu_forward(flash, Q, K, V, w.causal, w.scale)
    Oo, Lo = oracle_mod.forward(f64(Q), f64(K), f64(V), w.causal, w.scale)
    assert_fwd_close(O, LSE, Oo, Lo, w.name)


@pytest.mark.parametrize("name", ["causal_n4096", "gqa_n8192", "long_n32768",
                                  "causal_d64_n4096"])
def test_forward_full_size_workloads(flash, oracle_mod, name):
    """Full-size causal workloads in the launch configuration the benchmark times: one whole
    (batch, KV-group) slice (N <= 8192) plus rows sampled over all heads."""
    w = WORKLOADS[name]
    Q, K, V, _ = workload_inputs(w)
    O, LSE = gpu_forward(flash, Q, K, V, w.causal, w.scale)
    if w.N <= 8192:
        b, hk = w.B - 1, w.Hkv - 1
        q, k, v, _ = group_slice(Q, K, V, None, b, hk)
        Oo, Lo = oracle_mod.forward(f64(q), f64(k), f64(v), w.causal, w.scale)
        G = w.Hq // w.Hkv
        assert_fwd_close(O[b:b + 1, hk * G:(hk + 1) * G], LSE[b:b + 1, hk * G:(hk + 1) * G],
                         Oo, Lo, name + " group")
    rows = sample_rows(w.B, w.Hq, w.N, 96, seed=w.seed)
    Or, Lr = oracle_mod.forward_rows(f64(Q), f64(K), f64(V), w.causal, w.scale, rows)
    assert_fwd_close(O.reshape(-1, w.d)[rows], LSE.reshape(-1)[rows], Or, Lr, name + " rows")
