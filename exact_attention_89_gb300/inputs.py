"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers and names workload shapes; it holds none of the attention
arithmetic.  Every tensor is drawn on the CPU with a seeded ``torch.Generator`` in the fixed
order Q, K, V, dO, as iid N(0, 1) fp32, optionally multiplied (the long-sequence stress case
multiplies Q by 4 to widen the score range), then cast to the working dtype with round-to-
nearest-even.  The same host tensors feed both the CUDA path and the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    seed: int
    dtype: torch.dtype
    backward: bool
    q_mult: float = 1.0
    num_splits: int = 1          # key ranges of the split-KV forward (1: the one-pass forward)
    mask: str = ""               # general-mask recipe (see workload_mask), "" for none
    dropout: float = 0.0         # dropout probability on P (keep decisions seeded by `seed`)
    kv_outer: bool = False       # forward in the key/value-outer loop order (IO ablation)
    tensor_fp32: bool = False    # fp32 forward on the tensor cores (three TF32 products)

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    def flops_fwd(self) -> float:
        """4 B Hq N^2 d, halved for causal (the formula, not N(N+1)/2)."""
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        """2.5x the forward count (five contractions instead of two)."""
        return 2.5 * self.flops_fwd()


# The five workloads of the method's evaluation plan, then workloads for the split-KV forward, the
# general masks and dropout.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 1, 1, 256, 64, False, 0, torch.float32, True),
    "fwd_d64": Workload("fwd_d64", 4, 16, 16, 1024, 64, False, 1, torch.bfloat16, False),
    "causal_n4096": Workload("causal_n4096", 2, 32, 32, 4096, 128, True, 2, torch.bfloat16, True),
    "gqa_n8192": Workload("gqa_n8192", 1, 32, 8, 8192, 128, True, 3, torch.bfloat16, True),
    "long_n32768": Workload("long_n32768", 1, 16, 16, 32768, 128, True, 4, torch.bfloat16, True,
                            q_mult=4.0),
    # One head over a long causal sequence: its 128 (256-query) items fill fewer SMs than a
    # GB300 has, the case the split-KV forward (num_splits key ranges + merge) is for.
    "splitkv_n32768": Workload("splitkv_n32768", 1, 1, 1, 32768, 128, True, 5, torch.bfloat16,
                               False, num_splits=4),
    # Padded batch of variable-length sequences (general mask: valid lengths).
    "varlen_n8192": Workload("varlen_n8192", 8, 16, 16, 8192, 128, True, 6, torch.bfloat16, True,
                             mask="varlen"),
    # Block-sparse causal pattern (general mask: tile mask): a local window plus a first tile.
    "local_n16384": Workload("local_n16384", 1, 16, 16, 16384, 128, True, 7, torch.bfloat16, True,
                             mask="local_sink"),
    # The bench workload's shape at head dim 64.
    "causal_d64_n4096": Workload("causal_d64_n4096", 2, 32, 32, 4096, 64, True, 10, torch.bfloat16,
                                 True),
    # The bench workload's shape with dropout p = 0.1 on P.
    "dropout_n4096": Workload("dropout_n4096", 2, 32, 32, 4096, 128, True, 8, torch.bfloat16, True,
                              dropout=0.1),
    # The bench workload's shape, forward only, in the key/value-outer loop order.
    "kvouter_n4096": Workload("kvouter_n4096", 2, 32, 32, 4096, 128, True, 2, torch.bfloat16, False,
                              kv_outer=True),
    # fp32 at the tiny_fp32 head dim, at a size worth timing, forward and backward on the tensor
    # cores.
    "fp32tc_n4096": Workload("fp32tc_n4096", 2, 16, 16, 4096, 64, True, 9, torch.float32, True,
                             tensor_fp32=True),
}

MASK_BLOCK = 128        # side of the tiles a block mask covers
LOCAL_WINDOW_TILES = 8  # local_sink: tiles of keys before (and including) the query's own tile


def workload_mask(w: Workload):
    """(q_len, k_len, block_mask) numpy arrays (int32 [B], int32 [B], uint8 [heads, nb, nb]) of a
    workload's mask recipe, each None when absent.

    varlen: q_len = k_len, the first sequence full length N, the others uniform in [N/8, N]
    (seeded).  local_sink: one mask for every head; query tile a sees key tiles
    a-7 .. a and tile 0."""
    import numpy as np
    if not w.mask:
        return None, None, None
    if w.mask == "varlen":
        rng = np.random.default_rng(w.seed)
        lens = rng.integers(w.N // 8, w.N + 1, size=w.B).astype(np.int32)
        lens[0] = w.N
        return lens, lens.copy(), None
    if w.mask == "local_sink":
        nb = -(-w.N // MASK_BLOCK)
        a = np.arange(nb)[:, None]
        c = np.arange(nb)[None, :]
        bm = ((c <= a) & (c > a - LOCAL_WINDOW_TILES)) | (c == 0)
        return None, None, bm.astype(np.uint8)[None]
    raise ValueError("unknown mask recipe " + w.mask)


def make_inputs(B: int, Hq: int, Hkv: int, N: int, d: int, seed: int,
                dtype: torch.dtype = torch.bfloat16, q_mult: float = 1.0,
                with_dO: bool = True):
    """Q [B,Hq,N,d], K, V [B,Hkv,N,d], dO [B,Hq,N,d] (or None) on the CPU, drawn in that order."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float32)
    if q_mult != 1.0:
        q = q * q_mult
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float32)
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float32)
    do = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float32) if with_dO else None
    out = [t.to(dtype).contiguous() for t in (q, k, v)]
    out.append(do.to(dtype).contiguous() if do is not None else None)
    return tuple(out)


def workload_inputs(w: Workload, seed_offset: int = 0):
    """Inputs for a named workload (seed_offset gives independent replicas per rank)."""
    return make_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed + seed_offset, w.dtype, w.q_mult,
                       with_dO=w.backward)
