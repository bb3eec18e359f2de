"""Pins for the fp64 oracle, checked against what the pages and the mathematics fix (CPU only).

Each test names the fact it pins.  None of them retypes the oracle's own formula: they use the
pages' worked example, closed forms, invariants, an independent blocked recurrence written from
the pages' update equations, brute-force finite differences and torch fp64 autograd of the naive
definition.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def rand(*shape):
    return RNG.standard_normal(shape)


# --------------------------------------------------------------------------- worked example
def _worked():
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        return json.load(f)


def test_worked_example_output_and_lse(oracle_mod):
    """FlashAttention note (paweldubiel.com), worked example: scores [0,0,ln3,ln3], values
    [0,0,1,1] give 6/8 = 0.75.  Scores are realised with d = 1, q = 1, k_j = s_j, scale = 1."""
    g = _worked()
    s = np.array(g["scores"])
    v = np.array(g["values"])
    N = len(s)
    Q = np.ones((1, 1, N, 1))            # every query row is the same query
    K = s.reshape(1, 1, N, 1)
    V = v.reshape(1, 1, N, 1)
    O, L = oracle_mod.forward(Q, K, V, causal=False, scale=1.0)
    assert np.allclose(O[0, 0, :, 0], g["expected_output"], rtol=0, atol=1e-15)
    assert not np.isclose(O[0, 0, 0, 0], g["naive_block_mean_wrong"])
    assert np.allclose(L[0, 0], math.log(8.0), rtol=0, atol=1e-15)


def test_worked_example_block_means_are_wrong(oracle_mod):
    """Same example: the per-block results are 0 and 1 and their plain mean 0.5 is wrong; the
    oracle restricted to each block reproduces the page's block results."""
    g = _worked()
    s = np.array(g["scores"])
    v = np.array(g["values"])
    res = []
    for blk in (slice(0, 2), slice(2, 4)):
        n = 2
        O, _ = oracle_mod.forward(np.ones((1, 1, n, 1)), s[blk].reshape(1, 1, n, 1),
                                  v[blk].reshape(1, 1, n, 1), causal=False, scale=1.0)
        res.append(O[0, 0, 0, 0])
    assert np.allclose(res, g["block_results"], atol=1e-15)
    assert np.isclose(np.mean(res), g["naive_block_mean_wrong"])


# --------------------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_P_sum_to_one_and_mask_is_zero(oracle_mod, causal):
    """Softmax definition: each row of P sums to 1; masked pairs carry weight exactly 0."""
    Q, K, V = rand(1, 2, 37, 8), rand(1, 2, 37, 8), rand(1, 2, 37, 8)
    _, _, P = oracle_mod.forward(Q, K, V, causal, 0.3, want_P=True)
    assert np.allclose(P.sum(-1), 1.0, rtol=0, atol=1e-14)
    assert (P >= 0).all()
    if causal:
        iu = np.triu_indices(37, k=1)
        assert (P[:, :, iu[0], iu[1]] == 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_give_mean_of_allowed_values(oracle_mod, causal):
    """Q = 0 makes every score 0: O_i is the mean of the allowed v_j, LSE_i = ln(#allowed)."""
    N, d = 29, 5
    Q = np.zeros((2, 3, N, d))
    K, V = rand(2, 3, N, d), rand(2, 3, N, d)
    O, L = oracle_mod.forward(Q, K, V, causal, 0.7)
    for i in range(N):
        n = i + 1 if causal else N
        assert np.allclose(O[:, :, i], V[:, :, :n].mean(axis=2), atol=1e-14)
        assert np.allclose(L[:, :, i], math.log(n), atol=1e-14)


def test_causal_row_zero_returns_v0(oracle_mod):
    """Causal row 0 sees only key 0: O_0 = v_0 exactly and LSE_0 = s_00."""
    Q, K, V = rand(2, 2, 17, 6), rand(2, 2, 17, 6), rand(2, 2, 17, 6)
    O, L = oracle_mod.forward(Q, K, V, True, 0.5)
    assert np.array_equal(O[:, :, 0], V[:, :, 0])
    assert np.allclose(L[:, :, 0], 0.5 * (Q[:, :, 0] * K[:, :, 0]).sum(-1), atol=1e-15)


def test_lse_matches_library_logsumexp(oracle_mod):
    """LSE_i is scipy's logsumexp of the (unmasked) scaled scores, computed here with numpy."""
    from scipy.special import logsumexp
    Q, K, V = rand(1, 1, 40, 7), rand(1, 1, 40, 7), rand(1, 1, 40, 7)
    _, L = oracle_mod.forward(Q, K, V, False, 0.9)
    S = 0.9 * Q[0, 0] @ K[0, 0].T
    assert np.allclose(L[0, 0], logsumexp(S, axis=1), atol=1e-13)


def test_shift_invariance(oracle_mod):
    """Adding the same vector u to every key adds scale*q_i.u to every score of row i: P and O
    are unchanged and LSE_i moves by exactly that amount (the reason the max shift is exact)."""
    Q, K, V = rand(1, 2, 23, 4), rand(1, 2, 23, 4), rand(1, 2, 23, 4)
    u = rand(4)
    for causal in (False, True):
        O1, L1 = oracle_mod.forward(Q, K, V, causal, 0.8)
        O2, L2 = oracle_mod.forward(Q, K + u, V, causal, 0.8)
        assert np.allclose(O1, O2, atol=1e-13)
        assert np.allclose(L2 - L1, 0.8 * Q @ u, atol=1e-12)


def test_large_scores_do_not_overflow(oracle_mod):
    """Scores around 1e3 (exp would overflow without the max shift) still give finite P."""
    Q = rand(1, 1, 16, 4) * 30
    K = rand(1, 1, 16, 4) * 30
    V = rand(1, 1, 16, 4)
    O, L = oracle_mod.forward(Q, K, V, False, 1.0)
    assert np.isfinite(O).all() and np.isfinite(L).all()
    # the largest score dominates: O_i ~ v_argmax within exp(-gap)
    S = Q[0, 0] @ K[0, 0].T
    arg = S.argmax(1)
    gap = np.sort(S, 1)[:, -1] - np.sort(S, 1)[:, -2]
    ok = gap > 50
    assert np.allclose(O[0, 0][ok], V[0, 0][arg[ok]], atol=1e-12)


# --------------------------------------------------------------------------- blocked recurrence
def _blocked_fa1(s, v, bounds):
    """Reading-note (paper.adslab.icu) Methods: per block j, rescale the running sum
    l <- e^{m-m'} l + e^{m~-m'} l~ and the normalised output
    O <- diag(l')^-1 (diag(l) e^{m-m'} O + e^{m~-m'} P~ V_j), with m~, l~, P~ the block's own
    max, sum and unnormalised exp."""
    m, l, o = -np.inf, 0.0, np.zeros(v.shape[1])
    for a, b in bounds:
        sb = s[a:b]
        mt = sb.max()
        pt = np.exp(sb - mt)
        lt = pt.sum()
        mn = max(m, mt)
        ln = math.exp(m - mn) * l + math.exp(mt - mn) * lt
        o = (l * math.exp(m - mn) * o + math.exp(mt - mn) * (pt @ v[a:b])) / ln
        m, l = mn, ln
    return o, m + math.log(l)


def _blocked_deferred(s, v, bounds):
    """FlashAttention note (paweldubiel.com): keep m, l = sum e^{s-m} and u = sum e^{s-m} v;
    when a block raises the max to m', scale l and u by e^{m-m'} first; the result is u / l."""
    m, l, u = -np.inf, 0.0, np.zeros(v.shape[1])
    for a, b in bounds:
        mn = max(m, s[a:b].max())
        alpha = math.exp(m - mn)
        p = np.exp(s[a:b] - mn)
        l = alpha * l + p.sum()
        u = alpha * u + p @ v[a:b]
        m = mn
    return u / l, m + math.log(l)


def _random_bounds(n, rng):
    cuts = sorted(set(rng.integers(1, n, size=rng.integers(0, n)).tolist())) if n > 1 else []
    edges = [0] + cuts + [n]
    return list(zip(edges[:-1], edges[1:]))


def test_worked_example_through_both_recurrences():
    g = _worked()
    s = np.array(g["scores"])
    v = np.array(g["values"]).reshape(-1, 1)
    for f in (_blocked_fa1, _blocked_deferred):
        o, lse = f(s, v, [(0, 2), (2, 4)])
        assert abs(o[0] - 0.75) < 1e-15 and abs(lse - math.log(8)) < 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_blocked_online_softmax_equals_one_shot(oracle_mod, causal):
    """Any partition of the keys into blocks (sizes 1..N, including one key per block, the
    per-token recurrence of the mzeromiko blog) merged with the rescale gives the oracle's
    one-shot result to rounding."""
    rng = np.random.default_rng(7)
    N, d, scale = 48, 6, 0.6
    Q, K, V = rand(1, 1, N, d) * 2, rand(1, 1, N, d) * 2, rand(1, 1, N, d)
    O, L = oracle_mod.forward(Q, K, V, causal, scale)
    for i in range(N):
        n = i + 1 if causal else N
        s = scale * K[0, 0, :n] @ Q[0, 0, i]
        for bounds in (_random_bounds(n, rng), [(j, j + 1) for j in range(n)], [(0, n)]):
            for f in (_blocked_fa1, _blocked_deferred):
                o, lse = f(s, V[0, 0, :n], bounds)
                assert np.allclose(o, O[0, 0, i], atol=1e-13)
                assert abs(lse - L[0, 0, i]) < 1e-13


# --------------------------------------------------------------------------- GQA
def test_gqa_equals_repeated_heads(oracle_mod):
    """Query head hq reads KV head hq // G: the grouped result equals the result with each KV
    head repeated G times, and grouped dK/dV are the sums over the group."""
    B, Hq, Hkv, N, d = 2, 6, 2, 19, 4
    G = Hq // Hkv
    Q, K, V, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    Kr, Vr = np.repeat(K, G, axis=1), np.repeat(V, G, axis=1)
    for causal in (False, True):
        O1, L1 = oracle_mod.forward(Q, K, V, causal, 0.4)
        O2, L2 = oracle_mod.forward(Q, Kr, Vr, causal, 0.4)
        assert np.allclose(O1, O2, atol=1e-14) and np.allclose(L1, L2, atol=1e-14)
        dQ1, dK1, dV1 = oracle_mod.backward(Q, K, V, dO, causal, 0.4)
        dQ2, dK2, dV2 = oracle_mod.backward(Q, Kr, Vr, dO, causal, 0.4)
        assert np.allclose(dQ1, dQ2, atol=1e-13)
        assert np.allclose(dK1, dK2.reshape(B, Hkv, G, N, d).sum(2), atol=1e-13)
        assert np.allclose(dV1, dV2.reshape(B, Hkv, G, N, d).sum(2), atol=1e-13)


# --------------------------------------------------------------------------- backward
def _loss(oracle_mod, Q, K, V, dO, causal, scale):
    O, _ = oracle_mod.forward(Q, K, V, causal, scale)
    return float((O * dO).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("G", [1, 2])
def test_backward_central_finite_differences(oracle_mod, causal, G):
    """dQ, dK, dV equal central differences of L = sum(dO * O) (brute force, tiny sizes)."""
    B, Hkv, N, d, scale = 1, 2, 9, 5, 0.45
    Hq = Hkv * G
    Q, K, V, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    dQ, dK, dV = oracle_mod.backward(Q, K, V, dO, causal, scale)
    h = 1e-5
    for X, grad in ((Q, dQ), (K, dK), (V, dV)):
        num = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = X[idx]
            X[idx] = old + h
            lp = _loss(oracle_mod, Q, K, V, dO, causal, scale)
            X[idx] = old - h
            lm = _loss(oracle_mod, Q, K, V, dO, causal, scale)
            X[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(num - grad) / np.linalg.norm(grad)
        assert err < 1e-6, err


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(oracle_mod, causal):
    """Independent routine: torch fp64 autograd of naive softmax(scale QK^T + mask) V."""
    B, Hq, Hkv, N, d, scale = 2, 4, 2, 33, 8, 0.35
    G = Hq // Hkv
    Q, K, V, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (Q, K, V))
    s = scale * tq @ tk.repeat_interleave(G, 1).transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, -1) @ tv.repeat_interleave(G, 1)
    o.backward(torch.tensor(dO))
    O, L = oracle_mod.forward(Q, K, V, causal, scale)
    assert np.allclose(O, o.detach().numpy(), atol=1e-13)
    assert np.allclose(L, torch.logsumexp(s, -1).detach().numpy(), atol=1e-13)
    dQ, dK, dV = oracle_mod.backward(Q, K, V, dO, causal, scale)
    assert np.allclose(dQ, tq.grad.numpy(), atol=1e-12)
    assert np.allclose(dK, tk.grad.numpy(), atol=1e-12)
    assert np.allclose(dV, tv.grad.numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(oracle_mod, causal):
    """Rows of dS sum to 0, so sum_j dK_j = 0; sum_j dV_j = sum over the group of sum_i dO_i."""
    B, Hq, Hkv, N, d = 1, 4, 2, 31, 6
    Q, K, V, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    _, dK, dV = oracle_mod.backward(Q, K, V, dO, causal, 0.5)
    assert np.allclose(dK.sum(2), 0.0, atol=1e-12)
    assert np.allclose(dV.sum(2), dO.reshape(B, Hkv, 2, N, d).sum((2, 3)), atol=1e-12)


# --------------------------------------------------------------------------- sampled forms
@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_and_columns_match_full(oracle_mod, causal):
    """The row / column-sampled functions used at full sizes agree with the full functions."""
    B, Hq, Hkv, N, d, scale = 2, 4, 2, 27, 5, 0.55
    Q, K, V, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    O, L = oracle_mod.forward(Q, K, V, causal, scale)
    dQ, dK, dV = oracle_mod.backward(Q, K, V, dO, causal, scale)
    rows = np.array([0, 5, N - 1, N + 3, 3 * N + 26, B * Hq * N - 1])
    Or, Lr = oracle_mod.forward_rows(Q, K, V, causal, scale, rows)
    assert np.allclose(Or, O.reshape(-1, d)[rows], atol=1e-14)
    assert np.allclose(Lr, L.reshape(-1)[rows], atol=1e-14)
    dqr = oracle_mod.backward_dq_rows(Q, K, V, dO, causal, scale, rows)
    assert np.allclose(dqr, dQ.reshape(-1, d)[rows], atol=1e-13)
    cols = np.array([0, 7, N - 1, N, 2 * N + 4, B * Hkv * N - 1])
    dkc, dvc = oracle_mod.backward_dkv_cols(Q, K, V, dO, causal, scale, cols)
    assert np.allclose(dkc, dK.reshape(-1, d)[cols], atol=1e-13)
    assert np.allclose(dvc, dV.reshape(-1, d)[cols], atol=1e-13)


def test_subset_of_heads_and_groups(oracle_mod):
    """Head / group selection returns exactly the corresponding slices of the full result."""
    B, Hq, Hkv, N, d = 2, 4, 2, 13, 3
    Q, K, V, dO = rand(B, Hq, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, Hq, N, d)
    O, L = oracle_mod.forward(Q, K, V, True, 0.5)
    Os, Ls = oracle_mod.forward(Q, K, V, True, 0.5, heads=[5, 2])
    assert np.array_equal(Os, O.reshape(-1, N, d)[[5, 2]])
    assert np.array_equal(Ls, L.reshape(-1, N)[[5, 2]])
    dQ, dK, dV = oracle_mod.backward(Q, K, V, dO, True, 0.5)
    gq, gk, gv = oracle_mod.backward(Q, K, V, dO, True, 0.5, groups=[3])
    assert np.allclose(gq, dQ.reshape(B * Hkv, 2, N, d)[[3]], atol=0)
    assert np.allclose(gk, dK.reshape(-1, N, d)[[3]], atol=0)
    assert np.allclose(gv, dV.reshape(-1, N, d)[[3]], atol=0)


def test_invalid_arguments_raise(oracle_mod):
    Q = rand(1, 3, 4, 2)
    K = rand(1, 2, 4, 2)
    with pytest.raises(ValueError):
        oracle_mod.forward(Q, K, K, False, 1.0)
    with pytest.raises(RuntimeError):
        oracle_mod.forward(rand(1, 2, 4, 2), K, K, False, 1.0, heads=[7])


# --------------------------------------------------------------------------- split-KV merge
def test_worked_example_merged_from_its_two_blocks(oracle_mod):
    """FlashAttention note (paweldubiel.com) worked example: the two blocks' own results (0 and 1,
    with LSE ln 2 and ln 6) merged by the rescale recurrence give 0.75 and LSE ln 8, not the
    block mean 0.5."""
    g = _worked()
    O_parts = np.array(g["block_results"]).reshape(2, 1, 1)
    LSE_parts = np.array([math.log(2.0), math.log(6.0)]).reshape(2, 1)
    O, L = oracle_mod.merge_partials(O_parts, LSE_parts)
    assert abs(O[0, 0] - g["expected_output"]) < 1e-15
    assert abs(L[0] - math.log(8.0)) < 1e-15


def test_key_range_partials_merge_to_one_shot(oracle_mod):
    """Any partition of the keys into ranges: each range's partial (O, LSE) from the ranged
    forward, merged, equals the one-shot forward; empty ranges (LSE = -inf) change nothing."""
    rng = np.random.default_rng(3)
    B, Hq, Hkv, N, d, scale = 1, 4, 2, 45, 6, 0.4
    Q, K, V = rand(B, Hq, N, d) * 2, rand(B, Hkv, N, d), rand(B, Hkv, N, d)
    for causal in (False, True):
        O1, L1 = oracle_mod.forward(Q, K, V, causal, scale)
        for bounds in (_random_bounds(N, rng), [(0, N)], [(0, 1), (1, 44), (44, 45)]):
            parts = [oracle_mod.forward_keys(Q, K, V, causal, scale, a, b) for a, b in bounds]
            O, L = oracle_mod.merge_partials(np.stack([p[0] for p in parts]),
                                             np.stack([p[1] for p in parts]))
            assert np.allclose(O, O1, atol=1e-13) and np.allclose(L, L1, atol=1e-13)
        # causal rows before a range's first key see nothing from it
        O0, L0 = oracle_mod.forward_keys(Q, K, V, True, scale, 20, 30)
        assert np.isneginf(L0[:, :, :20]).all() and (O0[:, :, :20] == 0).all()


def test_merge_with_a_single_part_is_identity(oracle_mod):
    O_parts, L_parts = rand(1, 5, 3), rand(1, 5)
    O, L = oracle_mod.merge_partials(O_parts, L_parts)
    assert np.allclose(O, O_parts[0], atol=1e-15) and np.allclose(L, L_parts[0], atol=1e-15)
