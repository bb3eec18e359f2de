"""The deterministic backward (fa_bwd_deterministic): gradients within the bf16 backward
tolerance of the fp64 oracle, the same as fa_bwd's up to the order of the fp32 dQ sums, and dQ,
dK, dV bitwise equal from call to call (with other work and a scrambled workspace in between)."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import BF16_GRAD_REL_FRO, chosen_groups, f64, group_slice, rel_fro

pytestmark = pytest.mark.gpu

# fa_bwd and fa_bwd_deterministic run the same products; only the order of the fp32 additions
# into the dQ accumulator differs, so their results agree to about one bf16 rounding of dQ.
SAME_KERNELS_REL_FRO = 1e-3


def det_backward(flash, q, k, v, O, do, LSE, causal, scale, workspace=None):
    out = flash.attention_backward(q, k, v, O, do, LSE, causal, scale, workspace=workspace,
                                   deterministic=True)
    assert flash.fa_get_device_status() == flash.FA_OK
    return out


def on_device(*ts):
    return tuple(t.to(helpers.DEVICE) for t in ts)


SMALL = [
    # B, Hq, Hkv, N, causal
    (1, 1, 1, 1, True), (1, 2, 1, 17, False), (2, 2, 2, 127, True), (1, 4, 2, 129, False),
    (2, 4, 1, 200, True), (1, 2, 2, 300, False), (1, 8, 2, 513, True), (2, 2, 1, 1000, False),
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B,Hq,Hkv,N,causal", SMALL)
def test_deterministic_small_shapes(flash, oracle_mod, B, Hq, Hkv, N, causal, d):
    Q, K, V, dO = make_inputs(B, Hq, Hkv, N, d, seed=900 + N + d)
    scale = 1.0 / np.sqrt(d)
    q, k, v, do = on_device(Q, K, V, dO)
    O, LSE = flash.attention_forward(q, k, v, causal, scale)
    got = det_backward(flash, q, k, v, O, do, LSE, causal, scale)
    ref = oracle_mod.backward(f64(Q), f64(K), f64(V), f64(dO), causal, scale)
    errs = [rel_fro(g.cpu(), r) for g, r in zip(got, ref)]
    assert all(e <= BF16_GRAD_REL_FRO for e in errs), errs
    plain = flash.attention_backward(q, k, v, O, do, LSE, causal, scale)
    diffs = [rel_fro(g.cpu(), p.cpu()) for g, p in zip(got, plain)]
    assert all(e <= SAME_KERNELS_REL_FRO for e in diffs), diffs
    # dK and dV involve no cross-CTA sum: the two entry points give the same bits
    assert torch.equal(got[1], plain[1]) and torch.equal(got[2], plain[2])


def test_deterministic_workspace_size(flash):
    for B, Hq, N, d in [(1, 1, 1, 64), (2, 32, 4096, 128), (1, 16, 32768, 128), (3, 5, 1000, 64)]:
        base = flash.fa_bwd_workspace_bytes(B, Hq, N, d)
        assert flash.fa_bwd_deterministic_workspace_bytes(B, Hq, N, d) == \
            base + B * Hq * ((N + 63) // 64) * 16 + 16
    # one byte short is refused before any launch
    Q, K, V, dO = make_inputs(1, 2, 1, 300, 128, seed=3)
    q, k, v, do = on_device(Q, K, V, dO)
    O, LSE = flash.attention_forward(q, k, v, True, 0.1)
    ws = torch.empty(flash.fa_bwd_deterministic_workspace_bytes(1, 2, 300, 128) - 16,
                     dtype=torch.uint8, device=helpers.DEVICE)
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = flash.fa_bwd_deterministic(q, k, v, O, do, LSE, dQ, dK, dV, True, 0.1, ws, check=False)
    assert st == flash.FA_ERR_WORKSPACE


# The benchmark's workload, the grouped-query one and head dim 64, in the launch configuration
# the benchmark times.
REPRO = ["causal_n4096", "gqa_n8192", "causal_d64_n4096"]


@pytest.mark.parametrize("name", REPRO)
def test_deterministic_full_size_bitwise_repeat(flash, oracle_mod, name):
    """Three calls on the full-size workload give the same bits; between them fa_bwd runs on the
    same buffers and the workspace is overwritten with noise.  The result matches fa_bwd to the
    rounding of the fp32 sums and the oracle on every element of one whole KV group."""
    w = WORKLOADS[name]
    Q, K, V, dO = workload_inputs(w)
    q, k, v, do = on_device(Q, K, V, dO)
    O, LSE = flash.attention_forward(q, k, v, w.causal, w.scale)
    ws = torch.empty(flash.fa_bwd_deterministic_workspace_bytes(w.B, w.Hq, w.N, w.d),
                     dtype=torch.uint8, device=helpers.DEVICE)
    runs = []
    for r in range(3):
        runs.append([t.clone() for t in det_backward(flash, q, k, v, O, do, LSE, w.causal,
                                                     w.scale, workspace=ws)])
        plain = flash.attention_backward(q, k, v, O, do, LSE, w.causal, w.scale)
        ws.random_(0, 256)
    for r in (1, 2):
        for name_t, a, b in zip(("dQ", "dK", "dV"), runs[0], runs[r]):
            assert torch.equal(a, b), (name_t, r, int((a != b).sum()))
    diffs = [rel_fro(g.cpu(), p.cpu()) for g, p in zip(runs[0], plain)]
    assert all(e <= SAME_KERNELS_REL_FRO for e in diffs), diffs
    ndiff = int((runs[0][0] != plain[0]).sum())
    print("[determinism] %s: 3 calls bitwise equal; dQ elements differing from fa_bwd: %d of %d"
          % (name, ndiff, runs[0][0].numel()))
    # one whole KV group against the oracle
    G = w.Hq // w.Hkv
    (gi,) = chosen_groups(w.B * w.Hkv, 1, seed=31)
    b, hk = divmod(gi, w.Hkv)
    Qs, Ks, Vs, dOs = group_slice(Q, K, V, dO, b, hk)
    ref = oracle_mod.backward(f64(Qs), f64(Ks), f64(Vs), f64(dOs), w.causal, w.scale)
    dQ, dK, dV = (t.cpu() for t in runs[0])
    got = (dQ[b, hk * G:(hk + 1) * G][None], dK[b, hk][None, None], dV[b, hk][None, None])
    errs = [rel_fro(g, r) for g, r in zip(got, ref)]
    assert all(e <= BF16_GRAD_REL_FRO for e in errs), errs
