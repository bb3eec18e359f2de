"""The entry points inside a CUDA graph: one forward + backward step captured once and replayed on
new inputs written into the captured buffers gives the same bits as the same calls made eagerly
(the deterministic backward, so dQ is comparable bit for bit too), and within the bf16
tolerances of the fp64 oracle.  After their first call on a device the compute entry points
allocate nothing and never synchronise, which is what capture needs."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import make_inputs
from helpers import BF16_GRAD_REL_FRO, BF16_O_MAX_ABS, f64, max_abs, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [(2, 4, 2, 1000, 128, True),
                                                 (1, 4, 1, 777, 64, False)])
def test_step_replays_in_a_cuda_graph(flash, oracle_mod, B, Hq, Hkv, N, d, causal):
    dev = helpers.DEVICE
    scale = 1.0 / np.sqrt(d)
    first = make_inputs(B, Hq, Hkv, N, d, seed=40 + d)
    second = make_inputs(B, Hq, Hkv, N, d, seed=41 + d)
    q, k, v, do = (t.to(dev) for t in first)
    O = torch.empty_like(q)
    LSE = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(flash.fa_bwd_deterministic_workspace_bytes(B, Hq, N, d), dtype=torch.uint8,
                     device=dev)

    def step():
        flash.fa_fwd(q, k, v, O, LSE, causal, scale)
        flash.fa_bwd_deterministic(q, k, v, O, do, LSE, dQ, dK, dV, causal, scale, ws)

    step()                                          # first calls outside the capture
    torch.cuda.synchronize()
    eager_first = [t.clone() for t in (O, LSE, dQ, dK, dV)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    # replay on the first inputs, then on the second ones copied into the captured buffers
    g.replay()
    torch.cuda.synchronize()
    assert flash.fa_get_device_status() == flash.FA_OK
    for a, b in zip((O, LSE, dQ, dK, dV), eager_first):
        assert torch.equal(a, b)
    for dst, src in zip((q, k, v, do), second):
        dst.copy_(src.to(dev))
    g.replay()
    torch.cuda.synchronize()
    assert flash.fa_get_device_status() == flash.FA_OK
    replayed = [t.clone() for t in (O, LSE, dQ, dK, dV)]
    step()                                          # the same calls, eagerly, on the same data
    torch.cuda.synchronize()
    for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), replayed, (O, LSE, dQ, dK, dV)):
        assert torch.equal(a, b), name
    Q2, K2, V2, dO2 = second
    Oo, _ = oracle_mod.forward(f64(Q2), f64(K2), f64(V2), causal, scale)
    assert max_abs(replayed[0].cpu(), Oo) <= BF16_O_MAX_ABS
    ref = oracle_mod.backward(f64(Q2), f64(K2), f64(V2), f64(dO2), causal, scale)
    errs = [rel_fro(g_.cpu(), r) for g_, r in zip(replayed[2:], ref)]
    assert all(e <= BF16_GRAD_REL_FRO for e in errs), errs
