"""Dropout on P (fa_fwd_dropout / fa_bwd_dropout / fa_dropout_mask) against the fp64 oracle.

The keep decisions are integer work: fa_dropout_mask must equal oracle.dropout_mask bit for bit.
Outputs: LSE max abs <= 1e-3, O mean abs <= 1e-3, gradients relative Frobenius error <= 2e-2
(the bf16 tolerances), and O elementwise |O - O_ref| <= 1e-2 + 2^-8 |O_ref|: the scale
1 / (1 - p) lets kept outputs exceed 4 in magnitude, where rounding O to bf16 alone (half an
ulp, 2^-9 |O| relative, 0.0156 at |O| = 8) exceeds a flat 1e-2; 2^-8 |O_ref| covers that
rounding with a factor of 2 to spare."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import (BF16_GRAD_REL_FRO, BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, BF16_O_MEAN_ABS, f64,
                     max_abs, rel_fro)


def assert_dropout_fwd_close(O, LSE, Oo, Lo):
    err = np.abs(f64(O) - Oo)
    worst = float(np.max(err - 2.0 ** -8 * np.abs(Oo)))
    e = (worst, float(err.mean()), max_abs(LSE, Lo))
    assert e[0] <= BF16_O_MAX_ABS and e[1] <= BF16_O_MEAN_ABS and e[2] <= BF16_LSE_MAX_ABS, e

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("BH,N,p,seed,offset", [(3, 300, 0.1, 1, 0), (2, 129, 0.5, 2 ** 40 + 7, 9),
                                                (1, 1, 0.3, 5, 1), (4, 64, 0.9, 123456789, 77)])
def test_mask_equals_the_oracle_bit_for_bit(flash, oracle_mod, BH, N, p, seed, offset):
    Z = torch.empty(BH, N, N, dtype=torch.uint8, device=helpers.DEVICE)
    flash.fa_dropout_mask(Z, p, seed, offset)
    assert flash.fa_get_device_status() == flash.FA_OK
    assert np.array_equal(Z.cpu().numpy(), oracle_mod.dropout_mask(BH, N, seed, offset, p))


def gpu_drop(flash, Q, K, V, dO, causal, scale, p, seed, offset):
    dev = helpers.DEVICE
    q, k, v = (t.to(dev) for t in (Q, K, V))
    O, LSE = flash.attention_forward_dropout(q, k, v, causal, scale, p, seed, offset)
    grads = None
    if dO is not None:
        grads = flash.attention_backward_dropout(q, k, v, O, dO.to(dev), LSE, causal, scale, p,
                                                 seed, offset)
        grads = tuple(g.cpu() for g in grads)
    assert flash.fa_get_device_status() == flash.FA_OK
    return O.cpu(), LSE.cpu(), grads


CASES = [
    # B, Hq, Hkv, N, d, causal, p
    (1, 1, 1, 17, 128, False, 0.5), (1, 2, 1, 300, 128, True, 0.1), (2, 2, 2, 257, 64, False, 0.2),
    (1, 4, 2, 513, 128, True, 0.3), (2, 2, 1, 1000, 128, False, 0.05), (1, 2, 2, 640, 64, True, 0.5),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,p", CASES)
def test_dropout_forward_and_backward_small_shapes(flash, oracle_mod, B, Hq, Hkv, N, d, causal, p):
    Q, K, V, dO = make_inputs(B, Hq, Hkv, N, d, seed=600 + N + d)
    scale, seed, offset = 1.0 / np.sqrt(d), 1000 + N, 3
    O, LSE, (dQ, dK, dV) = gpu_drop(flash, Q, K, V, dO, causal, scale, p, seed, offset)
    Oo, Lo = oracle_mod.forward_dropout(f64(Q), f64(K), f64(V), causal, scale, p, seed, offset)
    assert_dropout_fwd_close(O, LSE, Oo, Lo)
    ref = oracle_mod.backward_dropout(f64(Q), f64(K), f64(V), f64(dO), causal, scale, p, seed, offset)
    errs = [rel_fro(g, r) for g, r in zip((dQ, dK, dV), ref)]
    assert all(x <= BF16_GRAD_REL_FRO for x in errs), errs


def test_zero_probability_is_the_plain_path(flash):
    Q, K, V, dO = make_inputs(1, 2, 2, 333, 128, seed=41)
    dev = helpers.DEVICE
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    O1, L1 = flash.attention_forward(q, k, v, True, 0.1)
    O2, L2 = flash.attention_forward_dropout(q, k, v, True, 0.1, 0.0, 5)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    g1 = flash.attention_backward(q, k, v, O1, do, L1, True, 0.1)
    g2 = flash.attention_backward_dropout(q, k, v, O1, do, L1, True, 0.1, 0.0, 5)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])


def test_offset_and_seed_draw_fresh_masks(flash):
    Q, K, V, _ = make_inputs(1, 1, 1, 256, 128, seed=42, with_dO=False)
    outs = [gpu_drop(flash, Q, K, V, None, False, 0.1, 0.5, s, o)[0] for s, o in ((1, 0), (1, 1), (2, 0), (1, 0))]
    assert not torch.equal(outs[0], outs[1]) and not torch.equal(outs[0], outs[2])
    assert torch.equal(outs[0], outs[3])


def test_dropout_full_size_workload_first_group(flash, oracle_mod):
    """dropout_n4096 (B2 H32 N4096 causal, p = 0.1): the whole first (batch, head) slice, whose
    global head index 0 the oracle reproduces on the slice, forward and backward."""
    w = WORKLOADS["dropout_n4096"]
    Q, K, V, dO = workload_inputs(w)
    O, LSE, (dQ, dK, dV) = gpu_drop(flash, Q, K, V, dO, w.causal, w.scale, w.dropout, w.seed, 0)
    sl = (slice(0, 1), slice(0, 1))
    q, k, v, do = (f64(t[sl]) for t in (Q, K, V, dO))
    Oo, Lo = oracle_mod.forward_dropout(q, k, v, w.causal, w.scale, w.dropout, w.seed, 0)
    assert_dropout_fwd_close(O[sl], LSE[sl], Oo, Lo)
    ref = oracle_mod.backward_dropout(q, k, v, do, w.causal, w.scale, w.dropout, w.seed, 0)
    errs = [rel_fro(g[sl], r) for g, r in zip((dQ, dK, dV), ref)]
    assert all(x <= BF16_GRAD_REL_FRO for x in errs), errs
