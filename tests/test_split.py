"""Split-KV forward (fa_fwd_split) and the merge of partial results (fa_merge) against the fp64
oracle on the same seeded inputs.

The partial of range s is checked against the oracle's forward restricted to that range's keys
(oracle.forward_keys): the rows with no allowed key must carry LSE = -inf exactly, the others
meet the bf16 forward tolerances (O max abs <= 1e-2, LSE max abs <= 1e-3).  Split + merge is
checked against the one-pass oracle forward with the same tolerances (plus O mean abs <= 1e-3),
and the merge alone against oracle.merge_partials in fp32 (max abs <= 1e-5)."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import (BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, BF16_O_MEAN_ABS, FP32_MAX_ABS, f64,
                     max_abs, mean_abs, sample_rows)

pytestmark = pytest.mark.gpu

BN = 128     # keys per block: the unit the ranges are cut in


def key_ranges(N, S):
    """[begin, end) of each range: ceil(nb / S) blocks of 128 keys each, the last ones empty."""
    nb = -(-N // BN)
    c = -(-nb // S)
    return [(min(N, s * c * BN), min(N, (s + 1) * c * BN)) for s in range(S)]


def gpu_split(flash, Q, K, V, causal, scale, S):
    dev = helpers.DEVICE
    q, k, v = (t.to(dev) for t in (Q, K, V))
    O, LSE, Op, Lp = flash.attention_forward_split(q, k, v, causal, scale, num_splits=S,
                                                   return_parts=True)
    assert flash.fa_get_device_status() == flash.FA_OK
    return O.cpu(), LSE.cpu(), Op.cpu(), Lp.cpu()


def assert_parts_match(oracle_mod, Q, K, V, causal, scale, S, Op, Lp):
    for s, (k0, k1) in enumerate(key_ranges(Q.shape[2], S)):
        Oo, Lo = oracle_mod.forward_keys(f64(Q), f64(K), f64(V), causal, scale, k0, k1)
        got_l = f64(Lp[s])
        empty = np.isneginf(Lo)
        assert np.array_equal(np.isneginf(got_l), empty), ("-inf pattern", s)
        full = ~empty
        if full.any():
            assert np.max(np.abs(got_l[full] - Lo[full])) <= BF16_LSE_MAX_ABS, s
            assert np.max(np.abs(f64(Op[s])[full] - Oo[full])) <= BF16_O_MAX_ABS, s


CASES = [
    # B, Hq, Hkv, N, d, causal, S
    (1, 1, 1, 1, 128, True, 1), (1, 1, 1, 1, 128, False, 3),
    (1, 2, 1, 300, 128, True, 2), (1, 2, 1, 300, 64, False, 3),
    (2, 4, 2, 513, 128, True, 4), (1, 2, 2, 1000, 128, False, 5),
    (1, 4, 1, 640, 64, True, 8), (1, 2, 1, 1024, 128, True, 3),
    (1, 2, 2, 200, 128, True, 7),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,S", CASES)
def test_split_parts_and_merge_small_shapes(flash, oracle_mod, B, Hq, Hkv, N, d, causal, S):
    Q, K, V, _ = make_inputs(B, Hq, Hkv, N, d, seed=300 + N + d + S, with_dO=False)
    scale = 1.0 / np.sqrt(d)
    O, LSE, Op, Lp = gpu_split(flash, Q, K, V, causal, scale, S)
    assert_parts_match(oracle_mod, Q, K, V, causal, scale, S, Op, Lp)
    Oo, Lo = oracle_mod.forward(f64(Q), f64(K), f64(V), causal, scale)
    e = (max_abs(O, Oo), mean_abs(O, Oo), max_abs(LSE, Lo))
    assert e[0] <= BF16_O_MAX_ABS and e[1] <= BF16_O_MEAN_ABS and e[2] <= BF16_LSE_MAX_ABS, e


def test_one_range_reproduces_the_one_pass_forward_exactly(flash):
    """With a single range the partial is the whole result and the merge multiplies by
    e^0 = 1, so split + merge gives fa_fwd's O and LSE bit for bit."""
    Q, K, V, _ = make_inputs(1, 4, 2, 777, 128, seed=31, with_dO=False)
    dev = helpers.DEVICE
    q, k, v = (t.to(dev) for t in (Q, K, V))
    O1, L1 = flash.attention_forward(q, k, v, True, 0.09)
    O2, L2, _, Lp = flash.attention_forward_split(q, k, v, True, 0.09, num_splits=1,
                                                  return_parts=True)
    assert flash.fa_get_device_status() == flash.FA_OK
    assert torch.equal(O1, O2) and torch.equal(L1, L2) and torch.equal(Lp[0], L1)


def random_parts(S, rows, d, seed):
    g = torch.Generator().manual_seed(seed)
    O = torch.randn(S, rows, d, generator=g)
    L = torch.rand(S, rows, generator=g) * 10 - 5
    drop = torch.rand(S, rows, generator=g) < 0.3
    L[drop] = -float("inf")
    L[:, 0] = -float("inf")                 # a row with no key in any part
    L[:, 1] = -float("inf")
    L[S // 2, 1] = 2.5                      # a row with exactly one non-empty part
    return O, L


@pytest.mark.parametrize("S,rows,d", [(1, 5, 128), (2, 300, 128), (5, 1000, 64), (8, 77, 4),
                                      (33, 64, 256), (3, 129, 1024)])
def test_merge_against_oracle(flash, oracle_mod, S, rows, d):
    Op, Lp = random_parts(S, rows, d, seed=S * 1000 + d)
    Oo, Lo = oracle_mod.merge_partials(f64(Op), f64(Lp))
    dev = helpers.DEVICE
    op, lp = Op.to(dev), Lp.to(dev)
    O = torch.empty(rows, d, dtype=torch.float32, device=dev)
    L = torch.empty(rows, dtype=torch.float32, device=dev)
    flash.fa_merge(op, lp, O, L)
    Ob = torch.empty(rows, d, dtype=torch.bfloat16, device=dev)
    Lb = torch.empty(rows, dtype=torch.float32, device=dev)
    flash.fa_merge(op, lp, Ob, Lb)
    assert flash.fa_get_device_status() == flash.FA_OK
    O, L, Ob, Lb = O.cpu(), L.cpu(), Ob.cpu(), Lb.cpu()
    assert np.array_equal(np.isneginf(f64(L)), np.isneginf(Lo))
    fin = ~np.isneginf(Lo)
    assert np.max(np.abs(f64(L)[fin] - Lo[fin])) <= FP32_MAX_ABS
    assert np.all(f64(O)[~fin] == 0.0)
    assert max_abs(O, Oo) <= FP32_MAX_ABS
    # bf16 output: the fp32 result rounded once (half an ulp, 2^-9 relative, plus fp32 slack)
    assert np.all(np.abs(f64(Ob) - Oo) <= 2.0 ** -8 * np.abs(Oo) + FP32_MAX_ABS)
    assert torch.equal(Lb, L)


def test_split_full_size_workload(flash, oracle_mod):
    """One head, N = 32768, causal, four key ranges: sampled rows against the oracle, and the
    split result against the one-pass forward on the GPU (both within the bf16 tolerances)."""
    w = WORKLOADS["splitkv_n32768"]
    Q, K, V, _ = workload_inputs(w)
    O, LSE, _, Lp = gpu_split(flash, Q, K, V, w.causal, w.scale, w.num_splits)
    rows = sample_rows(w.B, w.Hq, w.N, 64, seed=w.seed)
    Oo, Lo = oracle_mod.forward_rows(f64(Q), f64(K), f64(V), w.causal, w.scale, rows)
    got_o = O.reshape(-1, w.d)[rows]
    got_l = LSE.reshape(-1)[rows]
    assert max_abs(got_o, Oo) <= BF16_O_MAX_ABS and max_abs(got_l, Lo) <= BF16_LSE_MAX_ABS
    # rows of range 0 only see keys of range 0 under the causal mask
    c = key_ranges(w.N, w.num_splits)[0][1]
    assert torch.all(torch.isneginf(Lp[1:, :, :, :c]))
    dev = helpers.DEVICE
    O1, L1 = flash.attention_forward(*(t.to(dev) for t in (Q, K, V)), w.causal, w.scale)
    assert max_abs(O, O1.cpu()) <= BF16_O_MAX_ABS and max_abs(LSE, L1.cpu()) <= BF16_LSE_MAX_ABS
