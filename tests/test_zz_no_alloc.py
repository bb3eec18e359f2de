"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (a plugin handed only its input and output buffers by a framework that owns all
allocations, or a runtime that forbids allocating once it is serving) cannot pass fa_bwd a
workspace.  fa_bwd_noalloc runs the same backward with the library's fixed scratch array.
These tests check that its results match fa_bwd's within the backward tolerance on two calls in
a row (the second call reuses the array left over from the first), and that it rejects sizes
whose scratch would not fit.  This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import make_inputs
from helpers import BF16_GRAD_REL_FRO, rel_fro


def test_noalloc_rejects_sizes_beyond_the_scratch(built_lib):
    """Too large for the fixed scratch: FA_ERR_WORKSPACE, returned before any CUDA call."""
    L = built_lib.lib()
    A = 0x10000
    B, Hq, N, d = 2, 32, 4096, 128     # needs about 135 MB of scratch
    assert built_lib.fa_bwd_workspace_bytes(B, Hq, N, d) > built_lib.NOALLOC_SCRATCH_BYTES
    st = L.fa_bwd_noalloc(*([A] * 9), B, Hq, Hq, N, d, 1, 0.088, None)
    assert st == built_lib.FA_ERR_WORKSPACE


@pytest.mark.gpu
@pytest.mark.parametrize("B,Hq,Hkv,N,causal", [(1, 4, 2, 1000, True), (1, 8, 8, 4096, True),
                                               (2, 2, 1, 777, False)])
def test_noalloc_matches_fa_bwd_twice(flash, B, Hq, Hkv, N, causal):
    d = 128
    scale = 1.0 / np.sqrt(d)
    assert flash.fa_bwd_workspace_bytes(B, Hq, N, d) <= flash.NOALLOC_SCRATCH_BYTES
    dev = helpers.DEVICE
    q, k, v, do = (t.to(dev) for t in make_inputs(B, Hq, Hkv, N, d, seed=900 + N))
    O, LSE = flash.attention_forward(q, k, v, causal, scale)
    ref = flash.attention_backward(q, k, v, O, do, LSE, causal, scale)
    for call in range(2):
        dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        flash.fa_bwd_noalloc(q, k, v, O, do, LSE, dQ, dK, dV, causal, scale)
        torch.cuda.synchronize()
        assert flash.fa_get_device_status() == flash.FA_OK
        errs = [rel_fro(g.cpu(), r.cpu()) for g, r in zip((dQ, dK, dV), ref)]
        assert all(e <= BF16_GRAD_REL_FRO for e in errs), (call, errs)
