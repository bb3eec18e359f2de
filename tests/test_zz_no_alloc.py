"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (a plugin handed only its input and output buffers by a framework that owns all
allocations, or a runtime that forbids allocating once it is serving) cannot pass fa_bwd a
workspace.  fa_bwd_noalloc runs the same backward with the library's fixed scratch array.

These tests check its results against the fp64 oracle (backward tolerance) and against fa_bwd
on the same inputs (a much tighter bound: the same kernels run, only the scratch differs), on two
calls in a row with a call on other, larger inputs in between, so that anything the array kept
from an earlier call (D, the fp32 dQ accumulator) would show.  They also check that sizes whose
scratch would not fit are rejected.  This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import make_inputs
from helpers import BF16_GRAD_REL_FRO, f64, rel_fro

# fa_bwd_noalloc against fa_bwd on the same inputs: only the order of the fp32 dQ reductions
# differs between the two runs.
SAME_KERNELS_REL_FRO = 1e-3


def test_noalloc_rejects_sizes_beyond_the_scratch(built_lib):
    """Too large for the fixed scratch: FA_ERR_WORKSPACE, returned before any CUDA call."""
    L = built_lib.lib()
    A = 0x10000
    B, Hq, N, d = 2, 32, 4096, 128     # needs about 135 MB of scratch
    assert built_lib.fa_bwd_workspace_bytes(B, Hq, N, d) > built_lib.NOALLOC_SCRATCH_BYTES
    st = L.fa_bwd_noalloc(*([A] * 9), B, Hq, Hq, N, d, 1, 0.088, None)
    assert st == built_lib.FA_ERR_WORKSPACE


def _noalloc(flash, q, k, v, O, do, LSE, causal, scale):
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flash.fa_bwd_noalloc(q, k, v, O, do, LSE, dQ, dK, dV, causal, scale)
    torch.cuda.synchronize()
    assert flash.fa_get_device_status() == flash.FA_OK
    return dQ, dK, dV


@pytest.mark.gpu
@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [(1, 4, 2, 1000, 128, True),
                                                 (1, 8, 8, 4096, 128, True),
                                                 (2, 2, 1, 777, 128, False),
                                                 (1, 4, 2, 1000, 64, True),
                                                 (2, 4, 4, 1500, 64, False)])
def test_noalloc_matches_oracle_and_fa_bwd_twice(flash, oracle_mod, B, Hq, Hkv, N, d, causal):
    scale = 1.0 / np.sqrt(d)
    assert flash.fa_bwd_workspace_bytes(B, Hq, N, d) <= flash.NOALLOC_SCRATCH_BYTES
    dev = helpers.DEVICE
    Q, K, V, dO = make_inputs(B, Hq, Hkv, N, d, seed=900 + N + d)
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    O, LSE = flash.attention_forward(q, k, v, causal, scale)
    ref_gpu = [t.cpu() for t in flash.attention_backward(q, k, v, O, do, LSE, causal, scale)]
    ref = oracle_mod.backward(f64(Q), f64(K), f64(V), f64(dO), causal, scale)
    # Other inputs for the call between the two checked ones: a different seed and more rows
    # (8 heads of 8192), so its D and dQ accumulator cover every byte of scratch ours use.
    Np = 8192
    assert 8 * Np >= B * Hq * N
    assert flash.fa_bwd_workspace_bytes(1, 8, Np, d) <= flash.NOALLOC_SCRATCH_BYTES
    P = make_inputs(1, 8, 2, Np, d, seed=31 + d)
    p = [t.to(dev) for t in P]
    Op, Lp = flash.attention_forward(p[0], p[1], p[2], True, scale)
    for call in range(2):
        if call == 1:
            _noalloc(flash, p[0], p[1], p[2], Op, p[3], Lp, True, scale)
        got = [t.cpu() for t in _noalloc(flash, q, k, v, O, do, LSE, causal, scale)]
        errs_oracle = [rel_fro(g, r) for g, r in zip(got, ref)]
        errs_gpu = [rel_fro(g, r) for g, r in zip(got, ref_gpu)]
        assert all(e <= BF16_GRAD_REL_FRO for e in errs_oracle), (call, errs_oracle)
        assert all(e <= SAME_KERNELS_REL_FRO for e in errs_gpu), (call, errs_gpu)
