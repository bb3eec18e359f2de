"""Pins of the oracle's general masks (per-batch valid lengths and 0/1 block masks) against
identities and library routines, on the CPU:

  * padding is truncation: with q_len = k_len = L the first L rows (and keys) of a padded batch
    are exactly the unmasked oracle on the first L positions, every other row has O = 0,
    LSE = -inf and passes no gradient;
  * a block-diagonal block mask is independent attention inside each diagonal tile;
  * arbitrary masks (every row keeping at least one key) equal torch's fp64
    scaled_dot_product_attention with the same boolean mask, and its autograd gradients;
  * a per-head mask agrees with running each head under its own shared mask.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import Mask

F = torch.nn.functional


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def qkv(B, Hq, Hkv, N, d, seed):
    return (rnd((B, Hq, N, d), seed), rnd((B, Hkv, N, d), seed + 1), rnd((B, Hkv, N, d), seed + 2),
            rnd((B, Hq, N, d), seed + 3))


def dense_mask(B, Hq, N, causal, q_len=None, k_len=None, bm=None, block=128):
    """[B, Hq, N, N] boolean allowed-mask, built with numpy broadcasting (not the oracle's loop)."""
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    m = np.ones((B, Hq, N, N), dtype=bool)
    if causal:
        m &= (j <= i)[None, None]
    if q_len is not None:
        m &= (i[None, None] < np.asarray(q_len)[:, None, None, None])
    if k_len is not None:
        m &= (j[None, None] < np.asarray(k_len)[:, None, None, None])
    if bm is not None:
        full = np.kron(np.asarray(bm, bool), np.ones((block, block), bool))[..., :N, :N]
        if full.shape[0] == 1:
            full = np.broadcast_to(full[None], (B, Hq, N, N))
        elif full.shape[0] == Hq and full.shape[0] != B * Hq:
            full = np.broadcast_to(full[None], (B, Hq, N, N))
        else:
            full = full.reshape(B, Hq, N, N)
        m &= full
    return m


def torch_reference(Q, K, V, dO, allowed, scale):
    """fp64 torch SDPA with a boolean mask (rows must keep a key) and its autograd gradients."""
    G = Q.shape[1] // K.shape[1]
    q = torch.tensor(Q, requires_grad=True)
    k = torch.tensor(K, requires_grad=True)
    v = torch.tensor(V, requires_grad=True)
    kk, vv = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    am = torch.tensor(allowed)
    o = F.scaled_dot_product_attention(q, kk, vv, attn_mask=am, scale=scale)
    s = (q @ kk.transpose(-1, -2)) * scale
    lse = torch.logsumexp(s.masked_fill(~am, -float("inf")), dim=-1)
    o.backward(torch.tensor(dO))
    return (o.detach().numpy(), lse.detach().numpy(), q.grad.numpy(), k.grad.numpy(),
            v.grad.numpy())


@pytest.mark.parametrize("causal", [False, True])
def test_padding_is_truncation(causal):
    B, Hq, Hkv, N, d = 3, 4, 2, 70, 8
    Q, K, V, dO = qkv(B, Hq, Hkv, N, d, seed=11)
    L = [70, 33, 1]
    m = Mask(q_len=L, k_len=L, block=16)
    O, LSE = oracle.forward_masked(Q, K, V, causal, 0.4, m)
    dQ, dK, dV = oracle.backward_masked(Q, K, V, dO, causal, 0.4, m)
    for b, n in enumerate(L):
        sl = (slice(b, b + 1), slice(None), slice(0, n))
        Ot, Lt = oracle.forward(Q[sl], K[sl], V[sl], causal, 0.4)
        gq, gk, gv = oracle.backward(Q[sl], K[sl], V[sl], dO[sl], causal, 0.4)
        assert np.abs(O[sl] - Ot).max() < 1e-13 and np.abs(LSE[b, :, :n] - Lt[0]).max() < 1e-13
        assert np.abs(dQ[sl] - gq).max() < 1e-12
        assert np.abs(dK[sl] - gk).max() < 1e-12 and np.abs(dV[sl] - gv).max() < 1e-12
        assert np.all(O[b, :, n:] == 0) and np.all(np.isneginf(LSE[b, :, n:]))
        assert np.all(dQ[b, :, n:] == 0) and np.all(dK[b, :, n:] == 0) and np.all(dV[b, :, n:] == 0)


def test_lengths_clamp_to_the_sequence():
    Q, K, V, _ = qkv(2, 2, 2, 40, 8, seed=3)
    O1, L1 = oracle.forward_masked(Q, K, V, True, 0.3, Mask(q_len=[99, -4], k_len=[40, 7]))
    O2, L2 = oracle.forward_masked(Q, K, V, True, 0.3, Mask(q_len=[40, 0], k_len=[40, 7]))
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    assert np.all(np.isneginf(L1[1]))


def test_block_diagonal_mask_is_attention_inside_each_tile():
    B, H, N, d, blk = 1, 2, 50, 8, 16
    Q, K, V, dO = qkv(B, H, H, N, d, seed=5)
    nb = -(-N // blk)
    m = Mask(block_mask=np.eye(nb, dtype=np.uint8)[None], block=blk)
    O, LSE = oracle.forward_masked(Q, K, V, False, 0.5, m)
    dQ, dK, dV = oracle.backward_masked(Q, K, V, dO, False, 0.5, m)
    for c in range(nb):
        sl = (slice(None), slice(None), slice(c * blk, min(N, (c + 1) * blk)))
        Ot, Lt = oracle.forward(Q[sl], K[sl], V[sl], False, 0.5)
        gq, gk, gv = oracle.backward(Q[sl], K[sl], V[sl], dO[sl], False, 0.5)
        assert np.abs(O[sl] - Ot).max() < 1e-13 and np.abs(LSE[sl[:3]] - Lt).max() < 1e-13
        assert max(np.abs(dQ[sl] - gq).max(), np.abs(dK[sl] - gk).max(),
                   np.abs(dV[sl] - gv).max()) < 1e-12


@pytest.mark.parametrize("causal,heads_mode", [(False, "shared"), (True, "per_head"),
                                               (False, "per_batch_head"), (True, "shared")])
def test_masks_match_torch_sdpa(causal, heads_mode):
    B, Hq, Hkv, N, d, blk = 2, 4, 2, 45, 8, 8
    Q, K, V, dO = qkv(B, Hq, Hkv, N, d, seed=21)
    nb = -(-N // blk)
    rng = np.random.default_rng(7)
    mh = {"shared": 1, "per_head": Hq, "per_batch_head": B * Hq}[heads_mode]
    bm = (rng.random((mh, nb, nb)) < 0.5).astype(np.uint8)
    bm[:, np.arange(nb), np.arange(nb)] = 1          # every row keeps its diagonal tile
    q_len, k_len = [45, 45], [45, 30]                 # keys past 30 of batch 1 are padding
    if causal:
        k_len = [45, 45]                             # (a causal row keeps key 0 .. i)
    m = Mask(q_len=q_len, k_len=k_len, block_mask=bm, block=blk)
    allowed = dense_mask(B, Hq, N, causal, q_len, k_len, bm, blk)
    keep = allowed.any(-1)
    assert keep.all()
    O, LSE = oracle.forward_masked(Q, K, V, causal, 0.35, m)
    dQ, dK, dV = oracle.backward_masked(Q, K, V, dO, causal, 0.35, m)
    Ot, Lt, gq, gk, gv = torch_reference(Q, K, V, dO, allowed, 0.35)
    assert np.abs(O - Ot).max() < 1e-12 and np.abs(LSE - Lt).max() < 1e-12
    assert max(np.abs(dQ - gq).max(), np.abs(dK - gk).max(), np.abs(dV - gv).max()) < 1e-11


def test_per_head_mask_equals_each_head_alone():
    B, Hq, N, d, blk = 2, 3, 40, 8, 8
    Q, K, V, _ = qkv(B, Hq, Hq, N, d, seed=9)
    nb = -(-N // blk)
    rng = np.random.default_rng(1)
    bm = (rng.random((B * Hq, nb, nb)) < 0.6).astype(np.uint8)
    O, LSE = oracle.forward_masked(Q, K, V, True, 0.3, Mask(block_mask=bm, block=blk))
    for b in range(B):
        for h in range(Hq):
            sl = (slice(b, b + 1), slice(h, h + 1))
            Oh, Lh = oracle.forward_masked(Q[sl], K[sl], V[sl], True, 0.3,
                                           Mask(block_mask=bm[b * Hq + h][None], block=blk))
            assert np.array_equal(O[sl], Oh) and np.array_equal(LSE[sl], Lh)


def test_fully_masked_rows_get_zero_and_minus_infinity():
    Q, K, V, dO = qkv(1, 1, 1, 32, 8, seed=4)
    bm = np.array([[[1, 0], [0, 0]]], np.uint8)       # rows 16..31 keep no tile
    m = Mask(block_mask=bm, block=16)
    O, LSE = oracle.forward_masked(Q, K, V, False, 0.5, m)
    dQ, dK, dV = oracle.backward_masked(Q, K, V, dO, False, 0.5, m)
    assert np.all(O[0, 0, 16:] == 0) and np.all(np.isneginf(LSE[0, 0, 16:]))
    assert np.all(dQ[0, 0, 16:] == 0) and np.all(dK[0, 0, 16:] == 0) and np.all(dV[0, 0, 16:] == 0)
    assert np.all(np.isfinite(LSE[0, 0, :16]))


def test_sampled_rows_and_columns_match_the_full_masked_oracle():
    B, Hq, Hkv, N, d, blk = 2, 4, 2, 60, 8, 16
    Q, K, V, dO = qkv(B, Hq, Hkv, N, d, seed=31)
    nb = -(-N // blk)
    bm = (np.random.default_rng(2).random((Hq, nb, nb)) < 0.7).astype(np.uint8)
    m = Mask(q_len=[60, 41], k_len=[55, 41], block_mask=bm, block=blk)
    O, LSE = oracle.forward_masked(Q, K, V, True, 0.3, m)
    dQ, dK, dV = oracle.backward_masked(Q, K, V, dO, True, 0.3, m)
    rows = np.arange(0, B * Hq * N, 7)
    Or, Lr = oracle.forward_rows_masked(Q, K, V, True, 0.3, m, rows)
    assert np.abs(Or - O.reshape(-1, d)[rows]).max() < 1e-13
    assert np.array_equal(np.isneginf(Lr), np.isneginf(LSE.reshape(-1)[rows]))
    fin = ~np.isneginf(Lr)
    assert np.abs(Lr[fin] - LSE.reshape(-1)[rows][fin]).max() < 1e-13
    assert np.abs(oracle.backward_dq_rows_masked(Q, K, V, dO, True, 0.3, m, rows)
                  - dQ.reshape(-1, d)[rows]).max() < 1e-12
    cols = np.arange(0, B * Hkv * N, 5)
    gk, gv = oracle.backward_dkv_cols_masked(Q, K, V, dO, True, 0.3, m, cols)
    assert np.abs(gk - dK.reshape(-1, d)[cols]).max() < 1e-12
    assert np.abs(gv - dV.reshape(-1, d)[cols]).max() < 1e-12


def test_invalid_mask_descriptions_are_rejected():
    Q, K, V, _ = qkv(2, 4, 4, 20, 4, seed=1)
    with pytest.raises(RuntimeError):
        oracle.forward_masked(Q, K, V, False, 0.5, Mask(block_mask=np.ones((3, 2, 2)), block=16))
    with pytest.raises(RuntimeError):
        oracle.forward_masked(Q, K, V, False, 0.5, Mask(block_mask=np.ones((1, 2, 2)), block=0))
