"""bf16 forward on tcgen05 (fa_fwd) against the fp64 oracle on the same seeded inputs.

Tolerances: O max abs <= 1e-2 and mean abs <= 1e-3; LSE max abs <= 1e-3.
Small shapes and every full-size workload are compared over every element.  On the N = 32768
workload (queries scaled by 4, so rows put nearly all their weight on a few keys and |O| reaches
4 and more) a few elements cannot be within 1e-2 of the exact value in the arithmetic the method
prescribes (P rounded to bf16, a bf16 output: half a bf16 ulp alone is 0.0156 for |O| >= 4);
there each element is held to the worst case of that arithmetic instead (helpers.
bf16_forward_allowed), and the test prints how many elements exceed 1e-2."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import (BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, BF16_O_MEAN_ABS, ErrorTally,
                     bf16_forward_allowed, f64, group_slice, max_abs, mean_abs)

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


# Workloads whose every element the oracle checks (a few heads per oracle call), and the one
# too long for that: its whole-group check covers KV groups drawn by seed.
EVERY_ELEMENT = ["causal_n4096", "gqa_n8192", "causal_d64_n4096"]
WHOLE_GROUPS = ["long_n32768"]


@pytest.mark.parametrize("name", EVERY_ELEMENT)
def test_forward_full_size_every_element(flash, oracle_mod, name):
    """Full-size causal workloads in the launch configuration the benchmark times, compared with
    the oracle over every element of O and LSE (the oracle runs a few heads at a time)."""
    w = WORKLOADS[name]
    Q, K, V, _ = workload_inputs(w)
    O, LSE = gpu_forward(flash, Q, K, V, w.causal, w.scale)
    q64, k64, v64 = f64(Q), f64(K), f64(V)
    O2, L2 = O.reshape(w.B * w.Hq, w.N, w.d), LSE.reshape(w.B * w.Hq, w.N)
    to, tl = ErrorTally(), ErrorTally()
    step = 8
    for h0 in range(0, w.B * w.Hq, step):
        heads = list(range(h0, min(h0 + step, w.B * w.Hq)))
        Oo, Lo = oracle_mod.forward(q64, k64, v64, w.causal, w.scale, heads=heads)
        to.add(O2[heads], Oo, label="heads %d.." % h0)
        tl.add(L2[heads], Lo, label="heads %d.." % h0)
    print("[parity] %s forward, every element: O max abs %.3e mean abs %.3e, LSE max abs %.3e; "
          "worst O element %s" % (name, to.max_abs, to.mean_abs, tl.max_abs, to.worst))
    assert to.count == w.B * w.Hq * w.N * w.d
    assert (to.max_abs <= BF16_O_MAX_ABS and to.mean_abs <= BF16_O_MEAN_ABS
            and tl.max_abs <= BF16_LSE_MAX_ABS), (name, to.max_abs, to.mean_abs, tl.max_abs)


@pytest.mark.parametrize("name", WHOLE_GROUPS)
def test_forward_full_size_whole_groups(flash, oracle_mod, name):
    """The longest workload, every element, one KV group per oracle call (the oracle computes it
    row by row).  Each element within 1e-2, or within the worst case of the prescribed bf16
    arithmetic where that is larger (the oracle's attention applied to |V| gives the weighted
    |V| the bound needs)."""
    w = WORKLOADS[name]
    Q, K, V, _ = workload_inputs(w)
    O, LSE = gpu_forward(flash, Q, K, V, w.causal, w.scale)
    G = w.Hq // w.Hkv
    to, tl = ErrorTally(), ErrorTally()
    over, beyond, worst_ratio = 0, 0, 0.0
    for bk in range(w.B * w.Hkv):
        b, hk = divmod(bk, w.Hkv)
        q, k, v, _ = group_slice(Q, K, V, None, b, hk)
        rows = np.arange(G * w.N, dtype=np.int64)
        q64, k64, v64 = f64(q), f64(k), f64(v)
        Oo, Lo = oracle_mod.forward_rows(q64, k64, v64, w.causal, w.scale, rows)
        Oa, _ = oracle_mod.forward_rows(q64, k64, np.abs(v64), w.causal, w.scale, rows)
        got = O[b, hk * G:(hk + 1) * G].reshape(-1, w.d)
        err = np.abs(f64(got) - Oo)
        allowed = bf16_forward_allowed(Oo, Oa)
        over += int((err > BF16_O_MAX_ABS).sum())
        beyond += int((err > allowed).sum())
        worst_ratio = max(worst_ratio, float((err / allowed).max()))
        to.add(got, Oo, label="group %d" % bk)
        tl.add(LSE[b, hk * G:(hk + 1) * G].reshape(-1), Lo, label="group %d" % bk)
    print("[parity] %s forward, every element of all %d KV groups: O max abs %.3e mean abs %.3e, "
          "LSE max abs %.3e; worst O element %s; %d elements above %.0e, %d above the bound of "
          "the prescribed arithmetic (largest error / bound %.3f)"
          % (name, w.B * w.Hkv, to.max_abs, to.mean_abs, tl.max_abs, to.worst, over,
             BF16_O_MAX_ABS, beyond, worst_ratio))
    assert beyond == 0, (name, beyond, worst_ratio)
    # The bound is a worst case, loose where it applies; as a guard against a regression hiding
    # under it, elements above 1e-2 must stay rare (a kernel-faithful model of the current
    # arithmetic puts 13 to 15 of the 537 M elements there).
    assert over <= 1e-6 * O.numel(), (name, over)
    assert to.mean_abs <= BF16_O_MEAN_ABS and tl.max_abs <= BF16_LSE_MAX_ABS, (
        name, to.mean_abs, tl.max_abs)
