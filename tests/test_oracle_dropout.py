"""Pins of the oracle's dropout (Philox4x32-10 keep decisions, inverted dropout on P), on the CPU:

  * Philox4x32-10 reproduces the published known-answer vectors (tests/golden);
  * the keep threshold is floor((1 - p) 2^32), and the kept fraction is 1 - p within binomial
    error over a large mask;
  * the forward equals (P (.) Z / (1 - p)) V with P the undropped probabilities and the same
    keep decisions, and its LSE is the undropped one;
  * the backward equals torch's fp64 autograd of that expression and central finite
    differences of L = sum(dO (.) O);
  * averaged over many seeds the dropped output approaches the undropped one.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_philox_known_answer_vectors():
    kat = json.load(open(os.path.join(HERE, "golden", "philox4x32_10_kat.json")))
    for v in kat["vectors"]:
        got = oracle.philox4x32_10([int(x, 16) for x in v["counter"]], [int(x, 16) for x in v["key"]])
        assert ["%08x" % g for g in got] == v["out"]


def test_threshold():
    assert oracle.dropout_threshold(0.25) == 3 * 2 ** 30
    assert oracle.dropout_threshold(0.5) == 2 ** 31
    assert oracle.dropout_threshold(1e-12) == 2 ** 32 - 1
    assert oracle.dropout_threshold(0.0) == 0 and oracle.dropout_threshold(1.0) == 0


def test_mask_layout_and_kept_fraction():
    BH, N, seed, off, p = 3, 64, 0x1234_5678_9ABC_DEF0, 7, 0.3
    Z = oracle.dropout_mask(BH, N, seed, off, p)
    t = oracle.dropout_threshold(p)
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for bh, i, j in [(0, 0, 0), (2, 63, 63), (1, 5, 17), (0, 40, 3)]:
        words = oracle.philox4x32_10((j // 4, i, bh, off), key)
        assert Z[bh, i, j] == (words[j % 4] < t)
    n = Z.size
    frac = Z.mean()
    assert abs(frac - (1 - p)) < 5 * np.sqrt(p * (1 - p) / n)
    assert not np.array_equal(Z, oracle.dropout_mask(BH, N, seed, off + 1, p))
    assert not np.array_equal(Z, oracle.dropout_mask(BH, N, seed + 1, off, p))


@pytest.mark.parametrize("causal", [False, True])
def test_forward_is_dropped_probabilities_times_v(causal):
    B, Hq, Hkv, N, d, p = 2, 4, 2, 40, 8, 0.2
    Q, K, V = rnd((B, Hq, N, d), 1), rnd((B, Hkv, N, d), 2), rnd((B, Hkv, N, d), 3)
    O, L = oracle.forward_dropout(Q, K, V, causal, 0.4, p, seed=99, offset=3)
    O0, L0, P = oracle.forward(Q, K, V, causal, 0.4, want_P=True)
    Z = oracle.dropout_mask(B * Hq, N, 99, 3, p).reshape(B, Hq, N, N)
    Vr = np.repeat(V, Hq // Hkv, axis=1)
    ref = np.matmul(P * Z / (1 - p), Vr)
    assert np.abs(O - ref).max() < 1e-13
    assert np.array_equal(L, L0)


def torch_dropout_reference(Q, K, V, dO, causal, scale, Z, p):
    G = Q.shape[1] // K.shape[1]
    q = torch.tensor(Q, requires_grad=True)
    k = torch.tensor(K, requires_grad=True)
    v = torch.tensor(V, requires_grad=True)
    s = (q @ k.repeat_interleave(G, 1).transpose(-1, -2)) * scale
    if causal:
        N = Q.shape[2]
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -float("inf"))
    P = torch.softmax(s, dim=-1)
    o = (P * torch.tensor(Z, dtype=torch.float64) / (1 - p)) @ v.repeat_interleave(G, 1)
    o.backward(torch.tensor(dO))
    return o.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(causal):
    B, Hq, Hkv, N, d, p = 2, 4, 2, 33, 8, 0.35
    Q, K, V, dO = (rnd((B, Hq, N, d), 4), rnd((B, Hkv, N, d), 5), rnd((B, Hkv, N, d), 6),
                   rnd((B, Hq, N, d), 7))
    Z = oracle.dropout_mask(B * Hq, N, 5, 11, p).reshape(B, Hq, N, N)
    dQ, dK, dV = oracle.backward_dropout(Q, K, V, dO, causal, 0.3, p, 5, 11)
    O, tq, tk, tv = torch_dropout_reference(Q, K, V, dO, causal, 0.3, Z, p)
    assert max(np.abs(dQ - tq).max(), np.abs(dK - tk).max(), np.abs(dV - tv).max()) < 1e-11
    O2, _ = oracle.forward_dropout(Q, K, V, causal, 0.3, p, 5, 11)
    assert np.abs(O2 - O).max() < 1e-12


def test_backward_matches_finite_differences():
    B, Hq, Hkv, N, d, p, h = 1, 2, 1, 9, 4, 0.4, 1e-6
    Q, K, V, dO = (rnd((B, Hq, N, d), 8), rnd((B, Hkv, N, d), 9), rnd((B, Hkv, N, d), 10),
                   rnd((B, Hq, N, d), 11))
    dQ, dK, dV = oracle.backward_dropout(Q, K, V, dO, True, 0.5, p, 77, 0)

    def loss(q, k, v):
        return float(np.sum(dO * oracle.forward_dropout(q, k, v, True, 0.5, p, 77, 0)[0]))
    for name, X, G in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args = {"Q": (Xp, K, V), "K": (Q, Xp, V), "V": (Q, K, Xp)}[name]
            argm = {"Q": (Xm, K, V), "K": (Q, Xm, V), "V": (Q, K, Xm)}[name]
            fd[idx] = (loss(*args) - loss(*argm)) / (2 * h)
        assert np.linalg.norm(fd - G) <= 1e-6 * np.linalg.norm(G), name


def test_dropout_is_unbiased_over_seeds():
    Q, K, V = rnd((1, 1, 8, 4), 12), rnd((1, 1, 8, 4), 13), rnd((1, 1, 8, 4), 14)
    O0, _ = oracle.forward(Q, K, V, False, 0.5)
    acc = np.zeros_like(O0)
    n = 2000
    for s in range(n):
        acc += oracle.forward_dropout(Q, K, V, False, 0.5, 0.5, seed=s, offset=0)[0]
    # each output is a mean of n independent draws with |P V| <= max |V|: well inside 6 sigma
    assert np.abs(acc / n - O0).max() < 6 * np.abs(V).max() / np.sqrt(n)


def test_invalid_probability_is_rejected():
    Q = rnd((1, 1, 4, 4), 1)
    for p in (0.0, 1.0, -0.1):
        with pytest.raises(RuntimeError):
            oracle.forward_dropout(Q, Q, Q, False, 0.5, p, 1, 0)
