"""Shared helpers for the parity tests: moving tensors to the oracle, slicing independent
(batch, KV-group) sub-problems, and the error measures the tolerances are stated in."""
import numpy as np
import torch

# Device the parity tests run the CUDA path on.
DEVICE = torch.device("cuda:0")


def _np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, np.float64)


def f64(t):
    """Exact fp64 copy of a (bf16 / fp32) tensor as a numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()


def group_slice(Q, K, V, dO, b, hk):
    """The sub-problem of batch b and KV head hk: its G query heads and its one KV head.
    Attention of different (batch, KV head) pairs is independent, so the oracle on the slice
    gives exactly the slice of the full result."""
    G = Q.shape[1] // K.shape[1]
    sl = slice(hk * G, (hk + 1) * G)
    out = [Q[b:b + 1, sl], K[b:b + 1, hk:hk + 1], V[b:b + 1, hk:hk + 1]]
    out.append(dO[b:b + 1, sl] if dO is not None else None)
    return out


def max_abs(a, b):
    return float(np.max(np.abs(_np(a) - _np(b))))


def mean_abs(a, b):
    return float(np.mean(np.abs(_np(a) - _np(b))))


def rel_fro(a, ref):
    """||a - ref||_F / ||ref||_F, with the denominator floored at 1e-3 RMS: where the exact
    gradient is identically zero (one key per query: its weight is exactly 1, so dS = 0) a
    relative error is undefined and the rounding noise is measured against that floor."""
    a = _np(a)
    ref = _np(ref)
    floor = 1e-3 * np.sqrt(ref.size)
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), floor))


# Tolerances of the method's evaluation plan.
FP32_MAX_ABS = 1e-5
BF16_O_MAX_ABS = 1e-2
BF16_O_MEAN_ABS = 1e-3
BF16_LSE_MAX_ABS = 1e-3
BF16_GRAD_REL_FRO = 2e-2

# bf16 unit roundoff (8-bit significand, round to nearest even): |bf16(x) - x| <= 2^-8 |x|.
BF16_U = 2.0 ** -8


def bf16_forward_allowed(o_ref, oabs_ref):
    """Per-element bound on |O - O_ref| for the bf16 forward: BF16_O_MAX_ABS, or where larger the
    worst case of the arithmetic the method prescribes, whatever the kernel.  P is rounded to bf16
    (each weight within u of itself) before P V, while the normaliser sums the unrounded weights,
    so before the output rounding O is within E = u (sum_j P_j |V_j| + |O_ref|); the bf16 output
    then adds at most u |O_ref + E|.  o_ref is the exact O, oabs_ref the same attention applied to
    |V| (sum_j P_j |V_j|).  Where |O_ref| >= 4 half a bf16 ulp alone (0.0156) exceeds 1e-2, so the
    stated bound cannot hold for every bf16 output there."""
    o_ref = np.abs(_np(o_ref))
    e = BF16_U * (_np(oabs_ref) + o_ref)
    return np.maximum(BF16_O_MAX_ABS, e + BF16_U * (o_ref + e))


def sample_rows(B, H, N, n, seed):
    """Flat row indices (b*H + h)*N + i: first / last rows of every tile edge plus random ones."""
    rng = np.random.default_rng(seed)
    edges = [0, 1, 63, 64, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = []
    for bh in rng.choice(B * H, size=min(B * H, 4), replace=False):
        for i in edges:
            if 0 <= i < N:
                rows.append(int(bh) * N + i)
    rows += rng.integers(0, B * H * N, size=n).tolist()
    return np.unique(np.asarray(rows, dtype=np.int64))


def chosen_groups(n_groups, k, seed):
    """k distinct (batch * KV head) group indices out of n_groups, drawn with a seeded generator
    (for workloads whose every group is too slow for the oracle)."""
    rng = np.random.default_rng(seed)
    return sorted(int(g) for g in rng.choice(n_groups, size=min(k, n_groups), replace=False))


class ErrorTally:
    """Running max / mean absolute error and relative Frobenius error over chunks of a tensor,
    so a full-size comparison can run the oracle a few heads at a time."""

    def __init__(self):
        self.max_abs = 0.0
        self.worst = None          # (chunk label, index in the chunk, got, ref) of the max error
        self.abs_sum = 0.0
        self.count = 0
        self.diff_sq = 0.0
        self.ref_sq = 0.0

    def add(self, got, ref, label=None):
        g, r = _np(got), _np(ref)
        diff = g - r
        if diff.size:
            k = int(np.argmax(np.abs(diff)))
            if abs(diff.flat[k]) > self.max_abs:
                self.max_abs = float(abs(diff.flat[k]))
                self.worst = (label, np.unravel_index(k, diff.shape), float(g.flat[k]), float(r.flat[k]))
        self.abs_sum += float(np.sum(np.abs(diff)))
        self.count += diff.size
        self.diff_sq += float(np.sum(diff * diff))
        self.ref_sq += float(np.sum(r * r))

    @property
    def mean_abs(self):
        return self.abs_sum / max(self.count, 1)

    @property
    def rel_fro(self):
        floor = 1e-3 * np.sqrt(max(self.count, 1))
        return float(np.sqrt(self.diff_sq) / max(np.sqrt(self.ref_sq), floor))
