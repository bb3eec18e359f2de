"""Forward under a general mask (fa_fwd_masked) against the fp64 oracle (oracle.forward_masked)
on the same seeded inputs and masks.

Rows with no allowed key (padding rows, or rows whose tiles are all masked) must carry O = 0
and LSE = -inf exactly; every other row meets the bf16 forward tolerances (O max abs <= 1e-2,
mean abs <= 1e-3, LSE max abs <= 1e-3)."""
import numpy as np
import pytest
import torch

import helpers
from exact_attention_89_gb300.inputs import WORKLOADS, make_inputs, workload_inputs, workload_mask
from helpers import BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, BF16_O_MEAN_ABS, f64, max_abs, mean_abs

pytestmark = pytest.mark.gpu

BLK = 128


def dev_or_none(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(helpers.DEVICE)


def gpu_masked(flash, Q, K, V, causal, scale, q_len, k_len, bm):
    dev = helpers.DEVICE
    q, k, v = (t.to(dev) for t in (Q, K, V))
    O, LSE = flash.attention_forward_masked(q, k, v, causal, scale, dev_or_none(q_len),
                                            dev_or_none(k_len), dev_or_none(bm))
    assert flash.fa_get_device_status() == flash.FA_OK
    return O.cpu(), LSE.cpu()


def assert_masked_close(O, LSE, Oo, Lo, what=""):
    L, Lo = f64(LSE), np.asarray(Lo)
    dead = np.isneginf(Lo)
    assert np.array_equal(np.isneginf(L), dead), (what, "-inf pattern")
    Og = f64(O)
    assert np.all(Og[dead] == 0.0), what
    live = ~dead
    if live.any():
        e = (np.abs(Og[live] - Oo[live]).max(), np.abs(Og[live] - Oo[live]).mean(),
             np.abs(L[live] - Lo[live]).max())
        assert e[0] <= BF16_O_MAX_ABS and e[1] <= BF16_O_MEAN_ABS and e[2] <= BF16_LSE_MAX_ABS, (what, e)


def random_block_mask(heads, N, density, seed, diag=True):
    nb = -(-N // BLK)
    rng = np.random.default_rng(seed)
    bm = (rng.random((heads, nb, nb)) < density).astype(np.uint8)
    if diag:
        bm[:, np.arange(nb), np.arange(nb)] = 1
    return bm


CASES = [
    # B, Hq, Hkv, N, d, causal, lens, mask (density, heads: 1 | "Hq" | "BHq"), diag
    (2, 2, 1, 300, 128, True, [300, 130], None, True),
    (3, 2, 2, 257, 64, False, [1, 200, 257], None, True),
    (2, 4, 2, 513, 128, False, None, (0.5, 1), True),
    (1, 4, 4, 640, 128, True, None, (0.4, "Hq"), True),
    (2, 2, 1, 700, 64, True, [700, 333], (0.5, "BHq"), True),
    (1, 2, 2, 1000, 128, False, [999, 1000], (0.3, 1), False),     # rows with no tile at all
    (1, 2, 1, 384, 128, True, [0, 0], None, True),                 # empty sequences (B = 1: [0])
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,lens,mspec,diag", CASES)
def test_masked_forward_small_shapes(flash, oracle_mod, B, Hq, Hkv, N, d, causal, lens, mspec,
                                     diag):
    lens = None if lens is None else np.asarray(lens[:B], np.int32)
    Q, K, V, _ = make_inputs(B, Hq, Hkv, N, d, seed=400 + N + d, with_dO=False)
    bm = None
    if mspec is not None:
        dens, heads = mspec
        nh = {1: 1, "Hq": Hq, "BHq": B * Hq}[heads]
        bm = random_block_mask(nh, N, dens, seed=N, diag=diag)
    scale = 1.0 / np.sqrt(d)
    O, LSE = gpu_masked(flash, Q, K, V, causal, scale, lens, lens, bm)
    m = oracle_mod.Mask(q_len=lens, k_len=lens, block_mask=bm, block=BLK)
    Oo, Lo = oracle_mod.forward_masked(f64(Q), f64(K), f64(V), causal, scale, m)
    assert_masked_close(O, LSE, Oo, Lo)


def test_separate_query_and_key_lengths(flash, oracle_mod):
    Q, K, V, _ = make_inputs(2, 2, 2, 400, 128, seed=77, with_dO=False)
    ql, kl = np.array([400, 250], np.int32), np.array([130, 400], np.int32)
    for causal in (False, True):
        O, LSE = gpu_masked(flash, Q, K, V, causal, 0.09, ql, kl, None)
        Oo, Lo = oracle_mod.forward_masked(f64(Q), f64(K), f64(V), causal, 0.09,
                                           oracle_mod.Mask(q_len=ql, k_len=kl, block=BLK))
        assert_masked_close(O, LSE, Oo, Lo, causal)


def test_all_ones_mask_reproduces_the_unmasked_forward_exactly(flash):
    """Full lengths and an all-ones tile mask select every block in the same order, so the
    masked kernel's arithmetic is the unmasked one's, bit for bit."""
    Q, K, V, _ = make_inputs(2, 4, 2, 777, 128, seed=8, with_dO=False)
    dev = helpers.DEVICE
    q, k, v = (t.to(dev) for t in (Q, K, V))
    bm = torch.ones(1, 7, 7, dtype=torch.uint8, device=dev)
    lens = torch.full((2,), 777, dtype=torch.int32, device=dev)
    for causal in (False, True):
        O1, L1 = flash.attention_forward(q, k, v, causal, 0.1)
        O2, L2 = flash.attention_forward_masked(q, k, v, causal, 0.1, lens, lens, bm)
        assert flash.fa_get_device_status() == flash.FA_OK
        assert torch.equal(O1, O2) and torch.equal(L1, L2)


def test_padding_rows_ignore_their_contents(flash):
    """Changing the padding positions of Q (finite values) changes nothing in the output."""
    Q, K, V, _ = make_inputs(2, 2, 2, 300, 128, seed=12, with_dO=False)
    lens = np.array([300, 170], np.int32)
    O1, L1 = gpu_masked(flash, Q, K, V, True, 0.1, lens, lens, None)
    Q2, K2, V2 = Q.clone(), K.clone(), V.clone()
    Q2[1, :, 170:] = 3.0
    K2[1, :, 170:] = -2.0
    V2[1, :, 170:] = 5.0
    O2, L2 = gpu_masked(flash, Q2, K2, V2, True, 0.1, lens, lens, None)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


@pytest.mark.parametrize("name", ["varlen_n8192", "local_n16384"])
def test_masked_forward_full_size_workloads(flash, oracle_mod, name):
    w = WORKLOADS[name]
    Q, K, V, _ = workload_inputs(w)
    ql, kl, bm = workload_mask(w)
    O, LSE = gpu_masked(flash, Q, K, V, w.causal, w.scale, ql, kl, bm)
    m = oracle_mod.Mask(q_len=ql, k_len=kl, block_mask=bm, block=BLK)
    rng = np.random.default_rng(w.seed)
    rows = np.unique(np.concatenate([
        rng.integers(0, w.B * w.Hq * w.N, size=96),
        [(b * w.Hq) * w.N + i for b in range(w.B) for i in (0, 127, 128, w.N - 1)]]))
    Oo, Lo = oracle_mod.forward_rows_masked(f64(Q), f64(K), f64(V), w.causal, w.scale, m, rows)
    assert_masked_close(O.reshape(-1, w.d)[rows], LSE.reshape(-1)[rows], Oo, Lo, name)


# ----------------------------------------------------------------------------- backward
from helpers import BF16_GRAD_REL_FRO, rel_fro, sample_rows  # noqa: E402


def gpu_masked_fwd_bwd(flash, Q, K, V, dO, causal, scale, q_len, k_len, bm):
    dev = helpers.DEVICE
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    ql, kl, m = dev_or_none(q_len), dev_or_none(k_len), dev_or_none(bm)
    O, LSE = flash.attention_forward_masked(q, k, v, causal, scale, ql, kl, m)
    grads = flash.attention_backward_masked(q, k, v, O, do, LSE, causal, scale, ql, kl, m)
    assert flash.fa_get_device_status() == flash.FA_OK
    return tuple(g.cpu() for g in grads)


def assert_masked_grads_close(got, ref, what="", dead_rows=None, dead_keys=None):
    """Relative Frobenius error per gradient; rows with no allowed key (dead_rows, [B, Hq, N])
    must have dQ exactly 0 and padding keys (dead_keys, [B, Hkv, N]) dK = dV = 0 exactly."""
    errs = [rel_fro(g, r) for g, r in zip(got, ref)]
    assert all(e <= BF16_GRAD_REL_FRO for e in errs), (what, errs)
    if dead_rows is not None:
        assert np.all(f64(got[0])[dead_rows] == 0.0), what
    if dead_keys is not None:
        assert np.all(f64(got[1])[dead_keys] == 0.0) and np.all(f64(got[2])[dead_keys] == 0.0), what


def padding_keys(B, Hkv, N, k_len):
    if k_len is None:
        return None
    return np.broadcast_to(np.arange(N)[None, None, :] >= np.asarray(k_len)[:, None, None],
                           (B, Hkv, N))


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,lens,mspec,diag", CASES)
def test_masked_backward_small_shapes(flash, oracle_mod, B, Hq, Hkv, N, d, causal, lens, mspec,
                                      diag):
    lens = None if lens is None else np.asarray(lens[:B], np.int32)
    Q, K, V, dO = make_inputs(B, Hq, Hkv, N, d, seed=500 + N + d)
    bm = None
    if mspec is not None:
        dens, heads = mspec
        nh = {1: 1, "Hq": Hq, "BHq": B * Hq}[heads]
        bm = random_block_mask(nh, N, dens, seed=N + 1, diag=diag)
    scale = 1.0 / np.sqrt(d)
    got = gpu_masked_fwd_bwd(flash, Q, K, V, dO, causal, scale, lens, lens, bm)
    m = oracle_mod.Mask(q_len=lens, k_len=lens, block_mask=bm, block=BLK)
    ref = oracle_mod.backward_masked(f64(Q), f64(K), f64(V), f64(dO), causal, scale, m)
    _, Lo = oracle_mod.forward_masked(f64(Q), f64(K), f64(V), causal, scale, m)
    assert_masked_grads_close(got, ref, dead_rows=np.isneginf(Lo),
                              dead_keys=padding_keys(B, Hkv, N, lens))


def test_masked_backward_separate_lengths(flash, oracle_mod):
    Q, K, V, dO = make_inputs(2, 4, 2, 400, 128, seed=78)
    ql, kl = np.array([400, 250], np.int32), np.array([130, 400], np.int32)
    for causal in (False, True):
        got = gpu_masked_fwd_bwd(flash, Q, K, V, dO, causal, 0.09, ql, kl, None)
        m = oracle_mod.Mask(q_len=ql, k_len=kl, block=BLK)
        ref = oracle_mod.backward_masked(f64(Q), f64(K), f64(V), f64(dO), causal, 0.09, m)
        _, Lo = oracle_mod.forward_masked(f64(Q), f64(K), f64(V), causal, 0.09, m)
        assert_masked_grads_close(got, ref, causal, dead_rows=np.isneginf(Lo),
                                  dead_keys=padding_keys(2, 2, 400, kl))


def test_all_ones_mask_reproduces_the_unmasked_backward(flash):
    """Same steps in the same order: dK and dV bit for bit; dQ (fp32 atomics in any order)
    to fp32 rounding."""
    Q, K, V, dO = make_inputs(2, 4, 2, 777, 128, seed=9)
    dev = helpers.DEVICE
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    bm = torch.ones(1, 7, 7, dtype=torch.uint8, device=dev)
    lens = torch.full((2,), 777, dtype=torch.int32, device=dev)
    for causal in (False, True):
        O, L = flash.attention_forward(q, k, v, causal, 0.1)
        a = flash.attention_backward(q, k, v, O, do, L, causal, 0.1)
        b = flash.attention_backward_masked(q, k, v, O, do, L, causal, 0.1, lens, lens, bm)
        assert flash.fa_get_device_status() == flash.FA_OK
        assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
        assert rel_fro(b[0].cpu(), a[0].cpu()) <= 1e-2


@pytest.mark.parametrize("name", ["varlen_n8192", "local_n16384"])
def test_masked_backward_full_size_workloads(flash, oracle_mod, name):
    w = WORKLOADS[name]
    Q, K, V, dO = workload_inputs(w)
    ql, kl, bm = workload_mask(w)
    dQ, dK, dV = gpu_masked_fwd_bwd(flash, Q, K, V, dO, w.causal, w.scale, ql, kl, bm)
    m = oracle_mod.Mask(q_len=ql, k_len=kl, block_mask=bm, block=BLK)
    # the last batch entry: a shorter sequence for varlen
    b = w.B - 1
    sl = slice(b, b + 1)
    q, k, v, do = (f64(t[sl]) for t in (Q, K, V, dO))
    mb = oracle_mod.Mask(q_len=None if ql is None else ql[sl], k_len=None if kl is None else kl[sl],
                         block_mask=bm, block=BLK)
    rows = sample_rows(1, w.Hq, w.N, 40, seed=w.seed)
    dq_ref = oracle_mod.backward_dq_rows_masked(q, k, v, do, w.causal, w.scale, mb, rows)
    cols = sample_rows(1, w.Hkv, w.N, 40, seed=w.seed + 1)[:48]
    dk_ref, dv_ref = oracle_mod.backward_dkv_cols_masked(q, k, v, do, w.causal, w.scale, mb, cols)
    got = (dQ[sl].reshape(-1, w.d)[rows], dK[sl].reshape(-1, w.d)[cols],
           dV[sl].reshape(-1, w.d)[cols])
    assert_masked_grads_close(got, (dq_ref, dk_ref, dv_ref), name)
    del m
