"""Benchmark: exact attention forward + backward, bf16 d=128 causal, on GB300.

One step = one pass of the whole path over one batch: fa_fwd (O, LSE) then fa_bwd (dQ, dK, dV)
on the causal B2 H32 N4096 d128 workload (seed 2).  Inputs (Q, K, V, dO, O: 5 x 67 MB) are
larger than the 129 MB L2, so no flush is needed between steps.

Printed JSON line (rank 0):
  value     attention TFLOP/s of fwd+bwd, whole job (all ranks), device-timed with CUDA events,
            inputs resident in HBM; FLOPs = 4 B Hq N^2 d (x2.5 for the backward, /2 for causal).
  e2e       the same metric through the public API with pinned host buffers: every step copies
            Q, K, V, dO host->device and O, LSE, dQ, dK, dV device->host inside the timed region;
            the copies of neighbouring steps overlap the compute (copy streams, two buffer sets).
  roofline  the dominant launch sequence (fa_bwd) against the measured dense bf16 peak.
  cpu_baseline  the fp64 oracle on a bounded sample (whole heads) of the same workload.
--impl reference times the oracle itself (the reference arm) on the same metric.
Multi-GPU (torchrun): every rank runs its own replica (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "causal_n4096"
# The other full-size causal d = 128 workloads, timed the same way in the same run (extra keys).
OTHER_WORKLOADS = ("gqa_n8192", "long_n32768")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300's nominal dense bf16 tensor rate (datasheet), reported beside the measured peak.
NOMINAL_BF16_TFLOPS = 2250.0
# ex2.approx results per clock per SM (MUFU), measured with a single-SM probe on this GPU; the
# forward and backward each evaluate one exponential per allowed (query, key) pair.
MUFU_EX2_PER_CLK_PER_SM = 32.0

# DRAM traffic per launch of the reported kernel from one ncu capture, keyed by
# "<kernel file>:<sha256 prefix of that file and the device headers it includes>:<workload>";
# a key that no longer matches the sources (the kernel changed since the capture) reports null.
NCU_TRAFFIC = {
    # fa_bwd, three kernels per launch (bwd_preprocess + bwd_main + bwd_dq_convert, read + write):
    # causal_n4096 0.206 + 0.644 + 0.160 GB; causal_d64_n4096 0.073 + 0.291 + 0.070 GB;
    # gqa_n8192 0.207 + 0.880 + 0.161 GB; long_n32768 0.476 + 1.344 + 0.355 GB
    "fa_bwd_sm103a.cu:bda22c19073291fe:causal_n4096": 1.010e9,
    "fa_bwd_sm103a.cu:bda22c19073291fe:causal_d64_n4096": 0.433e9,
    "fa_bwd_sm103a.cu:bda22c19073291fe:gqa_n8192": 1.247e9,
    "fa_bwd_sm103a.cu:bda22c19073291fe:long_n32768": 2.174e9,
    # fa_bwd_masked, three kernels: local_n16384 0.206 + 0.630 + 0.160 GB; varlen_n8192
    # 1.014 + 1.900 + 0.766 GB
    "fa_bwd_sm103a.cu:bda22c19073291fe:local_n16384": 0.997e9,
    "fa_bwd_sm103a.cu:bda22c19073291fe:varlen_n8192": 3.680e9,
    # fa_bwd_dropout, three kernels: 0.206 + 0.640 + 0.161 GB
    "fa_bwd_sm103a.cu:bda22c19073291fe:dropout_n4096": 1.007e9,
    # split forward on splitkv_n32768: 25.4 MB read + 0.3 MB write (partials stay in L2)
    "fa_fwd_sm103a.cu:4cb1c4303c86d174:splitkv_n32768": 2.57e7,
    # forward at head dim 64 on fwd_d64: 25.2 MB read (Q, K, V), O written back from L2 later
    "fa_fwd_sm103a.cu:4cb1c4303c86d174:fwd_d64": 2.52e7,
    # key/value-outer forward: 2.374 GB read + 1.765 GB write
    "fa_fwd_kvouter_sm103a.cu:8eb13f6609ed98d2:kvouter_n4096": 4.139e9,
    # fp32 tensor-core backward: split rows 0.343 GB, split transposes 0.239 GB, dq pass
    # 0.328 GB, dkv pass 0.404 GB
    "fa_bwd_tf32x3_sm103a.cu:560f2a16a488a0a8:fp32tc_n4096": 1.314e9,
}


def split_key_ranges(N: int, S: int):
    """[begin, end) keys of each range of the split-KV forward (ceil(nb/S) 128-key blocks)."""
    nb = -(-N // 128)
    c = -(-nb // S)
    return [(min(N, s * c * 128), min(N, (s + 1) * c * 128)) for s in range(S)]


def allowed_pairs(w, q_len, k_len, block_mask, B=None, heads=None) -> float:
    """Number of (query, key) pairs a general mask allows, summed over batches and query heads:
    the work a masked pass does (4 d FLOPs per pair forward).  B / heads restrict the count to
    the first B batch entries and `heads` query heads (a sampled slice)."""
    import numpy as np
    B = w.B if B is None else B
    Hq = w.Hq if heads is None else heads
    N, blk = w.N, 128
    i = np.arange(N)
    total = 0.0
    for b in range(B):
        lq = N if q_len is None else int(min(max(q_len[b], 0), N))
        lk = N if k_len is None else int(min(max(k_len[b], 0), N))
        hi = np.minimum(i + 1 if w.causal else np.full(N, N), lk)[:lq]   # keys j < hi per row
        if block_mask is None:
            total += Hq * float(np.maximum(hi, 0).sum())
            continue
        nb = block_mask.shape[-1]
        c0 = np.arange(nb) * blk                                           # tile starts
        per_tile = np.clip(hi[:, None] - c0[None, :], 0, blk)              # [lq, nb]
        for h in range(Hq):
            mh = block_mask.shape[0]
            m = block_mask[0 if mh == 1 else (b * w.Hq + h if mh == w.B * w.Hq else h)]
            rows_tiles = m[i[:lq] // blk]                                  # [lq, nb]
            total += float((per_tile * rows_tiles).sum())
    return total


def _code_only(src: str) -> str:
    """C++ source without comments, blank lines and trailing blanks: an edit of a comment leaves
    the kernel, and so its key, unchanged."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_sources_hash(kernel_file: str) -> str:
    """Key prefix for NCU_TRAFFIC: the code of the kernel's source file and of the device headers
    it uses (comments excluded)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_89_gb300", "csrc")
    with open(os.path.join(csrc, kernel_file)) as f:
        own = re.findall(r'^#include "(\w+\.cuh)"', f.read(), re.M)
    extra = [fn for fn in own if fn not in ("fa_ptx.cuh", "fa_philox.cuh")]
    for fn in [kernel_file, "fa_ptx.cuh", "fa_philox.cuh"] + extra:
        with open(os.path.join(csrc, fn)) as f:
            h.update(fn.encode() + _code_only(f.read()).encode())
    return "%s:%s" % (kernel_file, h.hexdigest()[:16])


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples (every 200 ms) of SM clock and throttle reasons during a region."""
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        rows = [[c.strip() for c in ln.split(",")] for ln in self.lines if ln]
        buses = sorted({r[1].lower() for r in rows if len(r) > 1})
        if self.bus_id:
            mine = [r for r in rows if len(r) >= 10 and self.bus_id[-12:] in r[1].lower()]
        else:
            mine = []
        if not mine and len(buses) == 1:
            mine = [r for r in rows if len(r) >= 10]
        if not mine:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "gpu not matched"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in mine if num(r[2]) is not None]
        mx = [num(r[3]) for r in mine if num(r[3]) is not None]
        under = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in mine for n, v in zip(names, r[6:10]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(under) if under else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(mine)}


def cpu_info() -> dict:
    """Host CPU model, logical cores and OMP_NUM_THREADS, for the oracle's timings."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith(("model name", "cpu part")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"cpu_model": model, "machine": platform.machine(), "logical_cores": os.cpu_count(),
            "omp_num_threads": os.environ.get("OMP_NUM_THREADS")}


def ex2_ceiling(exps: float, flops: float, ms: float, sm_mhz, num_sms: int) -> dict:
    """The MUFU exponential ceiling of a pass: its exponentials at MUFU_EX2_PER_CLK_PER_SM on
    every SM at the sampled SM clock, as a time floor and as the TFLOP/s that floor allows."""
    mhz = float(sm_mhz) if sm_mhz else 2070.0
    rate = MUFU_EX2_PER_CLK_PER_SM * num_sms * mhz * 1e6
    floor_ms = exps / rate * 1e3
    return {"exps_per_launch": exps, "rate_per_clk_per_sm": MUFU_EX2_PER_CLK_PER_SM,
            "sm_mhz": mhz, "sms": num_sms, "time_floor_ms": floor_ms,
            "ceiling_tflops": flops / (floor_ms * 1e-3) / 1e12,
            "share_of_launch": floor_ms / ms if ms else None}


def time_plain_workload(name: str, steps: int, warmup: int, dev, peak: float) -> dict:
    """fa_fwd then fa_bwd on one of the plain causal workloads, CUDA events around every pass of
    `steps` timed steps after `warmup` untimed ones (the same timing as the main line)."""
    import torch

    from exact_attention_89_gb300 import flashattn as fa
    from exact_attention_89_gb300.inputs import WORKLOADS, workload_inputs
    w = WORKLOADS[name]
    Qh, Kh, Vh, dOh = workload_inputs(w)
    q, k, v, do = (t.to(dev) for t in (Qh, Kh, Vh, dOh))
    O, LSE = torch.empty_like(q), torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsp = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.Hq, w.N, w.d), dtype=torch.uint8,
                      device=dev)
    stream = torch.cuda.current_stream()

    def fwd():
        fa.fa_fwd(q, k, v, O, LSE, w.causal, w.scale)

    def bwd():
        fa.fa_bwd(q, k, v, O, do, LSE, dQ, dK, dV, w.causal, w.scale, wsp)

    for _ in range(max(3, warmup)):
        fwd()
        bwd()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e0, e1, e2 in ev:
        e0.record(stream)
        fwd()
        e1.record(stream)
        bwd()
        e2.record(stream)
    torch.cuda.synchronize()
    st = fa.fa_get_device_status()
    if st != fa.FA_OK:
        raise RuntimeError("device status after %s: %s" % (name, fa.fa_status_string(st)))
    fwd_ms = sum(a.elapsed_time(b) for a, b, _ in ev) / steps
    bwd_ms = sum(b.elapsed_time(c) for _, b, c in ev) / steps
    ff, fb = w.flops_fwd(), w.flops_bwd()
    fwd_t = ff / (fwd_ms * 1e-3) / 1e12
    tot_t = (ff + fb) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12
    return {"config": {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
                       "causal": w.causal, "seed": w.seed, "q_mult": w.q_mult},
            "steps": steps, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "fwd_tflops": fwd_t, "bwd_tflops": fb / (bwd_ms * 1e-3) / 1e12,
            "fwd_bwd_tflops": tot_t,
            "fwd_frac_of_peak": fwd_t / peak, "fwd_bwd_frac_of_peak": tot_t / peak,
            "fwd_frac_of_nominal_peak": fwd_t / NOMINAL_BF16_TFLOPS,
            "fwd_bwd_frac_of_nominal_peak": tot_t / NOMINAL_BF16_TFLOPS}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_seed_offset(rank: int) -> int:
    """Each rank runs its own replica of the workload on inputs seeded seed + rank."""
    return rank


def max_over_ranks(ms: float, ws: int, device) -> float:
    """The slowest rank's time (ms); the process group's MAX reduction when ws > 1."""
    if ws == 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(ws: int, flops_per_step: float, steps: int, max_ms: float) -> float:
    """Weak scaling: every rank processes one full step per step, so the job does ws x the FLOPs."""
    return ws * flops_per_step * steps / (max_ms * 1e-3) / 1e12


def cpu_oracle_rows_sample(w, budget_s: float, inputs=None):
    """Forward-only workloads: times the fp64 oracle on batches of random query rows (each row
    costs its own keys; random rows average to the formula's FLOPs per row)."""
    import numpy as np
    import torch

    import oracle
    from exact_attention_89_gb300.inputs import workload_inputs
    Q, K, V, _ = inputs if inputs is not None else workload_inputs(w)
    q, k, v = (t.to(torch.float64).numpy() for t in (Q, K, V))
    rng = np.random.default_rng(w.seed)
    total_rows = w.B * w.Hq * w.N
    rows_done, t_total = 0, 0.0
    while t_total < budget_s or rows_done == 0:
        rows = rng.integers(0, total_rows, size=64)
        t0 = time.perf_counter()
        oracle.forward_rows(q, k, v, w.causal, w.scale, rows)
        t_total += time.perf_counter() - t0
        rows_done += len(rows)
    per_row = w.flops_fwd() / total_rows
    return {"value": per_row * rows_done / t_total / 1e12, "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d random query rows of %s (B%d Hq%d Hkv%d N%d d%d causal), fp64 forward, "
                      "%.1f s" % (rows_done, w.name, w.B, w.Hq, w.Hkv, w.N, w.d, t_total),
            "seconds": t_total, "rows": rows_done}


def cpu_oracle_masked_sample(w, budget_s: float, inputs=None):
    """Masked workloads: times the fp64 oracle's masked forward + backward on whole KV groups
    (batch entry b, KV head hk), counting the pairs the mask allows in each group."""
    import torch

    import oracle
    from exact_attention_89_gb300.inputs import workload_inputs, workload_mask
    Q, K, V, dO = inputs if inputs is not None else workload_inputs(w)
    ql, kl, bm = workload_mask(w)
    G = w.Hq // w.Hkv
    done, pairs, t_total = 0, 0.0, 0.0
    while t_total < budget_s or done == 0:
        b, hk = divmod(done % (w.B * w.Hkv), w.Hkv)
        sl = slice(hk * G, (hk + 1) * G)
        q = Q[b:b + 1, sl].to(torch.float64).numpy()
        k = K[b:b + 1, hk:hk + 1].to(torch.float64).numpy()
        v = V[b:b + 1, hk:hk + 1].to(torch.float64).numpy()
        do = dO[b:b + 1, sl].to(torch.float64).numpy()
        qb = None if ql is None else ql[b:b + 1]
        kb = None if kl is None else kl[b:b + 1]
        mb = bm if bm is None or bm.shape[0] == 1 else bm[b * w.Hq + hk * G:b * w.Hq + (hk + 1) * G]
        m = oracle.Mask(q_len=qb, k_len=kb, block_mask=mb, block=128)
        t0 = time.perf_counter()
        oracle.forward_masked(q, k, v, w.causal, w.scale, m)
        oracle.backward_masked(q, k, v, do, w.causal, w.scale, m)
        t_total += time.perf_counter() - t0
        from types import SimpleNamespace
        sub = SimpleNamespace(B=1, Hq=G, N=w.N, causal=w.causal)
        pairs += allowed_pairs(sub, qb, kb, mb, B=1, heads=G)
        done += 1
    flops = 4.0 * w.d * pairs * 3.5
    return {"value": flops / t_total / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "%d whole KV group(s) of %s (B%d Hq%d Hkv%d N%d d%d, mask %s), fp64 masked "
                      "forward+backward, %.1f s" % (done, w.name, w.B, w.Hq, w.Hkv, w.N, w.d,
                                                    w.mask, t_total),
            "seconds": t_total}


def cpu_oracle_dropout_sample(w, budget_s: float, inputs=None):
    """Dropout workloads: times the fp64 oracle's dropout forward + backward on the first
    (batch, query head) slice, whose global head index the oracle reproduces on the slice."""
    import torch

    import oracle
    from exact_attention_89_gb300.inputs import workload_inputs
    Q, K, V, dO = inputs if inputs is not None else workload_inputs(w)
    sl = (slice(0, 1), slice(0, 1))
    q, k, v, do = (t[sl].to(torch.float64).numpy() for t in (Q, K, V, dO))
    done, t_total = 0, 0.0
    while t_total < budget_s or done == 0:
        t0 = time.perf_counter()
        oracle.forward_dropout(q, k, v, w.causal, w.scale, w.dropout, w.seed, 0)
        oracle.backward_dropout(q, k, v, do, w.causal, w.scale, w.dropout, w.seed, 0)
        t_total += time.perf_counter() - t0
        done += 1
    per_head = (w.flops_fwd() + w.flops_bwd()) / (w.B * w.Hq)
    return {"value": per_head * done / t_total / 1e12, "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d pass(es) over head 0 of %s (N%d d%d causal, dropout %.2f), fp64 "
                      "forward+backward, %.1f s" % (done, w.name, w.N, w.d, w.dropout, t_total),
            "seconds": t_total}


def cpu_oracle_sample(w, budget_s: float, max_heads: int, inputs=None, first_group: int = 0):
    """Times the fp64 oracle (forward + backward of whole KV groups) on the host cores."""
    import torch

    import oracle
    from exact_attention_89_gb300.inputs import workload_inputs
    if not w.backward:
        return cpu_oracle_rows_sample(w, budget_s, inputs)
    if w.mask:
        return cpu_oracle_masked_sample(w, budget_s, inputs)
    if w.dropout:
        return cpu_oracle_dropout_sample(w, budget_s, inputs)
    Q, K, V, dO = inputs if inputs is not None else workload_inputs(w)
    G = w.Hq // w.Hkv
    heads_done, t_total = 0, 0.0
    while heads_done < max_heads and (t_total < budget_s or heads_done == 0):
        b, hk = divmod((first_group + heads_done // G) % (w.B * w.Hkv), w.Hkv)
        sl = slice(hk * G, (hk + 1) * G)
        q = Q[b:b + 1, sl].to(torch.float64).numpy()
        k = K[b:b + 1, hk:hk + 1].to(torch.float64).numpy()
        v = V[b:b + 1, hk:hk + 1].to(torch.float64).numpy()
        do = dO[b:b + 1, sl].to(torch.float64).numpy()
        t0 = time.perf_counter()
        oracle.forward(q, k, v, w.causal, w.scale)
        oracle.backward(q, k, v, do, w.causal, w.scale)
        t_total += time.perf_counter() - t0
        heads_done += G
    per_head = (w.flops_fwd() + w.flops_bwd()) / (w.B * w.Hq)
    return {"value": per_head * heads_done / t_total / 1e12, "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d whole query head(s) of %s (B%d Hq%d Hkv%d N%d d%d causal), fp64 "
                      "forward+backward, %.1f s" % (heads_done, w.name, w.B, w.Hq, w.Hkv, w.N,
                                                     w.d, t_total),
            "seconds": t_total, "heads": heads_done}


TABLE_CONFIGS = ("tiny_fp32", "fwd_d64", "causal_n4096", "gqa_n8192", "long_n32768")


def oracle_table_rows(names, c5_groups: int = 1):
    """The fp64 oracle timed on the host cores, forward and backward separately, per workload:
    every head / KV group, except the N = 32768 workload, which is timed on whole KV groups and
    extrapolated linearly (groups are independent and equal work).  Its forward runs row by row
    (a whole N x N probability matrix per head would take 8.6 GB); its backward is the row pass
    for dQ plus the key-column pass for dK / dV.  The backward of the full-size functions
    recomputes P, O and D itself, as the oracle's backward does."""
    import numpy as np
    import torch

    import oracle
    from exact_attention_89_gb300.inputs import WORKLOADS, workload_inputs
    rows_out = []
    for name in names:
        w = WORKLOADS[name]
        Q, K, V, dO = workload_inputs(w)
        f = lambda t: t.to(torch.float64).numpy()
        G = w.Hq // w.Hkv
        n_groups = w.B * w.Hkv
        def mean_time(fn):
            # repeated up to half a second, so the small workloads are not timer noise
            n, t = 0, 0.0
            while t < 0.5 or n == 0:
                t0 = time.perf_counter()
                fn()
                t += time.perf_counter() - t0
                n += 1
            return t / n

        if w.N <= 8192:
            q, k, v = f(Q), f(K), f(V)
            t_fwd = mean_time(lambda: oracle.forward(q, k, v, w.causal, w.scale))
            t_bwd = None
            if w.backward:
                do = f(dO)
                t_bwd = mean_time(lambda: oracle.backward(q, k, v, do, w.causal, w.scale))
            timed, extrap = n_groups, 1.0
        else:
            t_fwd, t_bwd = 0.0, 0.0
            timed = min(c5_groups, n_groups)
            for bk in range(timed):
                b, hk = divmod(bk, w.Hkv)
                sl = slice(hk * G, (hk + 1) * G)
                q, k, v = f(Q[b:b + 1, sl]), f(K[b:b + 1, hk:hk + 1]), f(V[b:b + 1, hk:hk + 1])
                do = f(dO[b:b + 1, sl])
                rows = np.arange(G * w.N, dtype=np.int64)
                cols = np.arange(w.N, dtype=np.int64)
                t0 = time.perf_counter()
                oracle.forward_rows(q, k, v, w.causal, w.scale, rows)
                t_fwd += time.perf_counter() - t0
                t0 = time.perf_counter()
                oracle.backward_dq_rows(q, k, v, do, w.causal, w.scale, rows)
                oracle.backward_dkv_cols(q, k, v, do, w.causal, w.scale, cols)
                t_bwd += time.perf_counter() - t0
            extrap = n_groups / timed
            t_fwd *= extrap
            t_bwd *= extrap
        ff, fb = w.flops_fwd(), (w.flops_bwd() if w.backward else None)
        rows_out.append({
            "workload": name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
            "causal": w.causal, "dtype": "fp32 inputs" if w.dtype == torch.float32 else "bf16 inputs",
            "threads": oracle.num_threads(),
            "fwd_s": t_fwd, "fwd_gflops": ff / t_fwd / 1e9,
            "bwd_s": t_bwd, "bwd_gflops": (fb / t_bwd / 1e9) if t_bwd else None,
            "groups_timed": "%d of %d" % (timed, n_groups),
            "extrapolated": extrap != 1.0})
    return rows_out


def run_oracle_table(args):
    """Prints one JSON object: the oracle's forward and backward times per workload on all host
    cores, and on one core for the two small workloads (a child process with
    OMP_NUM_THREADS=1)."""
    names = [n for n in args.oracle_table.split(",") if n] if args.oracle_table != "all" else \
        list(TABLE_CONFIGS)
    out = {"cpu": cpu_info(), "rows": oracle_table_rows(names)}
    if args.oracle_table == "all":
        env = dict(os.environ, OMP_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--impl", "reference",
                            "--oracle-table", "tiny_fp32,fwd_d64"], env=env,
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("single-thread oracle timing failed:\n" + r.stderr[-2000:])
        out["single_thread"] = json.loads(r.stdout.strip().splitlines()[-1])
    print(json.dumps(out))
    return 0


def run_reference(args):
    """The reference arm: the fp64 oracle as it stands, on the host cores, same metric."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from exact_attention_89_gb300.inputs import WORKLOADS, workload_inputs
    w = WORKLOADS[WORKLOAD]
    inputs = workload_inputs(w)
    # one whole KV group (fwd + bwd) per step: a bounded sample of the workload
    for i in range(args.warmup):
        cpu_oracle_sample(w, 0.0, 1, inputs, first_group=i)
    t = 0.0
    heads = 0
    for i in range(args.steps):
        r = cpu_oracle_sample(w, 0.0, 1, inputs, first_group=i)
        t += r["seconds"]
        heads += r["heads"]
    per_head = (w.flops_fwd() + w.flops_bwd()) / (w.B * w.Hq)
    value = per_head * heads / t / 1e12
    import oracle
    line = {"impl": "reference", "metric": "attention TFLOP/s fwd+bwd, bf16 d=128 causal",
            "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N,
                       "d": w.d, "causal": w.causal, "seed": w.seed,
                       "step": "one whole query head, forward + backward (bounded sample)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": "%d step(s) of one whole head each" % args.steps},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for cpu_baseline (0 disables)")
    ap.add_argument("--no-extras", action="store_true",
                    help="only warm-up and timed steps (no clock load, e2e or cpu baseline); "
                         "for profiler runs")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager calls instead of replays of the step captured in a CUDA graph")
    ap.add_argument("--oracle-table", default=None,
                    help="with --impl reference: time the oracle's forward and backward per "
                         "workload ('all' or a comma-separated list) instead of the bench line")
    args = ap.parse_args()
    if args.impl == "reference" and args.oracle_table:
        return run_oracle_table(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        args.warmup = 3

    import torch
    import torch.distributed as dist

    from exact_attention_89_gb300 import build as fbuild
    from exact_attention_89_gb300 import flashattn as fa
    from exact_attention_89_gb300.inputs import WORKLOADS, workload_inputs

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not os.path.exists(fa.LIB_PATH):
        if rank == 0:
            fbuild.build()
        if ws > 1:
            dist.barrier()
    fa.lib()

    w = WORKLOADS[args.workload]
    Qh, Kh, Vh, dOh = workload_inputs(w, seed_offset=replica_seed_offset(rank))
    q, k, v = (t.to(dev) for t in (Qh, Kh, Vh))
    do = dOh.to(dev) if dOh is not None else None
    B, Hq, Hkv, N, d = w.B, w.Hq, w.Hkv, w.N, w.d
    S = w.num_splits
    split = S > 1
    masked = bool(w.mask)
    if masked:
        from exact_attention_89_gb300.inputs import workload_mask
        ql_h, kl_h, bm_h = workload_mask(w)
        mq, mkk, mbm = (None if a is None else torch.from_numpy(a).to(dev)
                        for a in (ql_h, kl_h, bm_h))
    O = torch.empty_like(q)
    LSE = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    if w.backward:
        dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wbytes = (fa.fa_bwd_fp32_tc_workspace_bytes(B, Hq, Hkv, N, d) if w.tensor_fp32 else
                  fa.fa_bwd_workspace_bytes(B, Hq, N, d))
        wsp = torch.empty(wbytes, dtype=torch.uint8, device=dev)
    if split:
        Op = torch.empty(S, B, Hq, N, d, dtype=torch.float32, device=dev)
        Lp = torch.empty(S, B, Hq, N, dtype=torch.float32, device=dev)
    if w.kv_outer:
        kws = torch.empty(fa.fa_fwd_kvouter_workspace_bytes(B, Hq, N, d), dtype=torch.uint8,
                          device=dev)
    if w.tensor_fp32:
        kws = torch.empty(fa.fa_fwd_fp32_tc_workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8,
                          device=dev)
    stream = torch.cuda.current_stream()

    # the tensors a step reads and writes (the end-to-end run swaps in other sets)
    main_set = {"q": q, "k": k, "v": v, "do": do, "O": O, "LSE": LSE}
    if w.backward:
        main_set.update(dQ=dQ, dK=dK, dV=dV)

    def fwd_first(t=main_set):
        # the forward's tensor-core launch
        if split:
            fa.fa_fwd_split(t["q"], t["k"], t["v"], Op, Lp, w.causal, w.scale, S)
        elif masked:
            fa.fa_fwd_masked(t["q"], t["k"], t["v"], t["O"], t["LSE"], w.causal, w.scale, mq, mkk, mbm)
        elif w.dropout:
            fa.fa_fwd_dropout(t["q"], t["k"], t["v"], t["O"], t["LSE"], w.causal, w.scale, w.dropout,
                              w.seed, 0)
        elif w.kv_outer:
            fa.fa_fwd_kvouter(t["q"], t["k"], t["v"], t["O"], t["LSE"], w.causal, w.scale, kws)
        elif w.tensor_fp32:
            fa.fa_fwd_fp32_tc(t["q"], t["k"], t["v"], t["O"], t["LSE"], w.causal, w.scale, kws)
        else:
            fa.fa_fwd(t["q"], t["k"], t["v"], t["O"], t["LSE"], w.causal, w.scale)

    def second(t=main_set):
        # what follows it in a step: the merge of the partials, or the backward
        if split:
            fa.fa_merge(Op, Lp, t["O"], t["LSE"])
            return
        if not w.backward:
            return
        args_b = (t["q"], t["k"], t["v"], t["O"], t["do"], t["LSE"], t["dQ"], t["dK"], t["dV"],
                  w.causal, w.scale)
        if masked:
            fa.fa_bwd_masked(*args_b, wsp, mq, mkk, mbm)
        elif w.dropout:
            fa.fa_bwd_dropout(*args_b, w.dropout, w.seed, 0, wsp)
        elif w.tensor_fp32:
            fa.fa_bwd_fp32_tc(*args_b, wsp)
        else:
            fa.fa_bwd(*args_b, wsp)

    def step():
        fwd_first()
        second()

    def barrier():
        if ws > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = fa.fa_get_device_status()
    if st != fa.FA_OK:
        raise RuntimeError("device status after warm-up: " + fa.fa_status_string(st))

    # One step captured in a CUDA graph: the timed steps replay it, with no host-side launch path
    # between the kernels of a step or between steps (the entry points allocate nothing and never
    # synchronise after their first call).  --no-graph or --no-extras time eager calls instead.
    graph = None
    if not (args.no_graph or args.no_extras):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()

    # ---------------------------------------------------------------- device-timed region
    bus = None
    try:
        bus = getattr(torch.cuda.get_device_properties(dev), "pci_bus_id", None)
    except Exception:
        bus = None
    sampler = ClockSampler(str(bus) if bus is not None else None)
    sampler.start()

    def load_for(seconds):
        # the same steps, untimed, so the clock samples around the short timed region are
        # taken under the same load
        t_end_load = time.perf_counter() + seconds
        while time.perf_counter() < t_end_load:
            for _ in range(20):
                step()
            torch.cuda.synchronize()

    if not args.no_extras:
        load_for(0.8)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for e0, e1, e2 in ev:
        e0.record(stream)
        fwd_first()
        e1.record(stream)
        second()
        e2.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    # the same K steps as replays of the captured graph: the step time `value` reports
    graph_total_ms = None
    step_times = sorted(e0.elapsed_time(e2) for e0, _, e2 in ev)   # the replays' below, if any
    if graph is not None:
        barrier()
        torch.cuda.synchronize()
        g_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        g_ev[0].record(stream)
        for i in range(args.steps):
            graph.replay()
            g_ev[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier()
        graph_total_ms = g_ev[0].elapsed_time(g_ev[-1])
        step_times = sorted(a.elapsed_time(b) for a, b in zip(g_ev[:-1], g_ev[1:]))
    if not args.no_extras:
        load_for(0.6)
    clocks = sampler.stop()
    st = fa.fa_get_device_status()
    if st != fa.FA_OK:
        raise RuntimeError("device status after timed region: " + fa.fa_status_string(st))
    # eager steps: their per-launch events give the split of a step between its kernels
    eager_total_ms = max_over_ranks(t_start.elapsed_time(t_end), ws, dev)
    first_ms = sum(a.elapsed_time(b) for a, b, _ in ev) / args.steps
    second_ms = sum(b.elapsed_time(c) for _, b, c in ev) / args.steps
    total_ms = (max_over_ranks(graph_total_ms, ws, dev) if graph_total_ms is not None
                else eager_total_ms)

    # FLOPs: the formula 4 B Hq N^2 d (/2 causal, x2.5 backward), or under a general mask
    # 4 d per allowed (query, key) pair
    flops_fwd = (4.0 * d * allowed_pairs(w, ql_h, kl_h, bm_h)) if masked else w.flops_fwd()
    flops_bwd = 2.5 * flops_fwd if w.backward else 0.0
    flops_step = flops_fwd + flops_bwd
    value = whole_job_tflops(ws, flops_step, args.steps, total_ms)

    # the one-pass forward on the same inputs, for comparison with the split path
    one_pass_ms = None
    if (split or w.kv_outer or w.tensor_fp32) and not args.no_extras:
        # the comparison forward: the query-outer bf16 one, or the fp32 one on the CUDA cores
        ref_fwd = fa.fa_fwd_fp32 if w.tensor_fp32 else fa.fa_fwd
        for _ in range(3):
            ref_fwd(q, k, v, O, LSE, w.causal, w.scale)
        o_s = torch.cuda.Event(enable_timing=True)
        o_e = torch.cuda.Event(enable_timing=True)
        o_s.record(stream)
        for _ in range(args.steps):
            ref_fwd(q, k, v, O, LSE, w.causal, w.scale)
        o_e.record(stream)
        torch.cuda.synchronize()
        one_pass_ms = o_s.elapsed_time(o_e) / args.steps
    simt_bwd_ms = None
    if w.tensor_fp32 and w.backward and not args.no_extras:
        # the fp32 backward on the CUDA cores, same inputs (it uses the D part of a workspace)
        wsimt = torch.empty(fa.fa_bwd_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device=dev)
        fa.fa_bwd_fp32(q, k, v, O, do, LSE, dQ, dK, dV, w.causal, w.scale, wsimt)
        b_s = torch.cuda.Event(enable_timing=True)
        b_e = torch.cuda.Event(enable_timing=True)
        b_s.record(stream)
        fa.fa_bwd_fp32(q, k, v, O, do, LSE, dQ, dK, dV, w.causal, w.scale, wsimt)
        b_e.record(stream)
        torch.cuda.synchronize()
        simt_bwd_ms = b_s.elapsed_time(b_e)

    # the deterministic backward (dQ reductions in a fixed order) on the same inputs, timed like
    # fa_bwd in the steps above, for its cost against fa_bwd
    det_bwd_ms = None
    if (w.backward and not (masked or w.dropout or w.tensor_fp32 or split)
            and not args.no_extras):
        wdet = torch.empty(fa.fa_bwd_deterministic_workspace_bytes(B, Hq, N, d), dtype=torch.uint8,
                           device=dev)
        det_args = (q, k, v, O, do, LSE, dQ, dK, dV, w.causal, w.scale, wdet)
        for _ in range(3):
            fa.fa_bwd_deterministic(*det_args)
        d_s = torch.cuda.Event(enable_timing=True)
        d_e = torch.cuda.Event(enable_timing=True)
        d_s.record(stream)
        for _ in range(args.steps):
            fa.fa_bwd_deterministic(*det_args)
        d_e.record(stream)
        torch.cuda.synchronize()
        if fa.fa_get_device_status() != fa.FA_OK:
            raise RuntimeError("device status after the deterministic backward")
        det_bwd_ms = d_s.elapsed_time(d_e) / args.steps
        del wdet

    # ---------------------------------------------------------------- end to end (host buffers)
    # Every step copies its inputs from pinned host memory, runs the path through the public
    # entry points and copies its outputs back to pinned host memory.  The copies run on their
    # own streams with two sets of device buffers, so the inputs of step k + 1 and the outputs of
    # step k - 1 move while step k computes, as a training loop fed from host memory would run.
    pin = [t.pin_memory() for t in (Qh, Kh, Vh, dOh) if t is not None]
    out_names = ["O", "LSE", "dQ", "dK", "dV"] if w.backward else ["O", "LSE"]
    outs_h = [torch.empty(main_set[n].shape, dtype=main_set[n].dtype, pin_memory=True)
              for n in out_names]
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    in_names = ["q", "k", "v", "do"][:len(pin)]
    e2e_sets = [main_set]
    if not args.no_extras:
        e2e_sets.append({n: torch.empty_like(main_set[n]) for n in in_names + out_names})
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def e2e_run(nsteps):
        """nsteps pipelined steps; returns their time in ms (events on the compute stream)."""
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        t0.record(stream)
        s_in.wait_event(t0)
        s_out.wait_event(t0)
        for kk in range(nsteps):
            b = kk % 2
            t = e2e_sets[b]
            with torch.cuda.stream(s_in):
                if kk >= 2:
                    s_in.wait_event(done[b])          # step k - 2 has read this input set
                for n, src in zip(in_names, pin):
                    t[n].copy_(src, non_blocking=True)
                ready[b].record(s_in)
            stream.wait_event(ready[b])
            if kk >= 2:
                stream.wait_event(out_done[b])        # step k - 2's outputs have left this set
            fwd_first(t)
            second(t)
            done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[b])
                for hbuf, n in zip(outs_h, out_names):
                    hbuf.copy_(t[n], non_blocking=True)
                out_done[b].record(s_out)
        for e in out_done[:min(nsteps, 2)]:
            stream.wait_event(e)
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    e2e_ms = float("nan")
    if not args.no_extras:
        e2e_run(2)
        barrier()
        e2e_ms = e2e_run(args.steps)
    e2e_ms = max_over_ranks(e2e_ms, ws, dev)
    e2e_value = whole_job_tflops(ws, flops_step, args.steps, e2e_ms)

    # ---------------------------------------------------------------- roofline + cpu baseline
    peaks, peaks_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # the other full-size causal d = 128 workloads, when the main one is the default
    others = None
    if w.name == WORKLOAD and not args.no_extras:
        others = {}
        for name in OTHER_WORKLOADS:
            others[name] = time_plain_workload(name, args.steps, args.warmup, dev, peak)
            torch.cuda.empty_cache()
        if ws > 1:
            for r in others.values():
                for key in ("fwd_ms", "bwd_ms"):
                    r[key] = max_over_ranks(r[key], ws, dev)
    # one exponential per allowed (query, key) pair in each pass
    exps = (allowed_pairs(w, ql_h, kl_h, bm_h) if masked else
            w.B * w.Hq * w.N * w.N / (2.0 if w.causal else 1.0))
    fwd_key = kernel_sources_hash("fa_fwd_sm103a.cu") + ":" + w.name
    bwd_key = kernel_sources_hash("fa_bwd_sm103a.cu") + ":" + w.name
    peak_source = ("%s burst bf16 (MEASURED_PEAKS.json)" % peaks_src if peaks_src == "measured"
                   else "fallback 1.9 PFLOP/s bf16")
    fwd_achieved = flops_fwd / (first_ms * 1e-3) / 1e12
    if split:
        # the merge reads every LSE part and the O parts of rows with an allowed key in that
        # range, and writes O (bf16) and LSE
        rows = B * Hq * N
        live = sum((B * Hq * max(0, N - k0) if w.causal else rows) if k1 > k0 else 0
                   for k0, k1 in split_key_ranges(N, S))
        merge_bytes = S * rows * 4 + live * d * 4 + rows * (d * 2 + 4)
        hbm = float(peaks["hbm_gbs"])
        merge_gbs = merge_bytes / (second_ms * 1e-3) / 1e9
        roofline = {"bound": "tensor", "kernel": "fa_fwd_split", "achieved": fwd_achieved,
                    "peak": peak, "unit": "TFLOP/s", "frac": fwd_achieved / peak,
                    "traffic": NCU_TRAFFIC.get(fwd_key), "peak_source": peak_source,
                    "flops_per_launch": w.flops_fwd(), "ms": first_ms,
                    "merge": {"kernel": "fa_merge", "bound": "hbm", "unit": "GB/s",
                              "bytes_per_launch": merge_bytes, "ms": second_ms,
                              "achieved": merge_gbs, "peak": hbm, "frac": merge_gbs / hbm},
                    "one_pass_fwd_ms": one_pass_ms, "sources": fwd_key}
    elif w.backward and w.tensor_fp32:
        # three TF32 products per product: the TF32 dense peak (bf16 / 2 nominal) x 1/3; the
        # dq pass's recomputed S and dP (7 products instead of 5) count against the kernel
        bwd_achieved = flops_bwd / (second_ms * 1e-3) / 1e12
        tc_key = kernel_sources_hash("fa_bwd_tf32x3_sm103a.cu") + ":" + w.name
        roofline = {"bound": "tensor",
                    "kernel": "fa_bwd_fp32_tc (split + dq pass + dkv pass)",
                    "achieved": bwd_achieved, "peak": peak / 2, "unit": "TFLOP/s",
                    "frac": bwd_achieved * 3 / (peak / 2),
                    "traffic": NCU_TRAFFIC.get(tc_key),
                    "peak_source": peak_source + " x 1/2 (TF32 rate)",
                    "note": "achieved counts the method's FLOPs once; frac counts the three TF32 "
                            "products against the TF32 peak",
                    "flops_per_launch": flops_bwd, "bwd_ms": second_ms,
                    "simt_fp32_fwd_ms": one_pass_ms, "simt_fp32_bwd_ms": simt_bwd_ms,
                    "fwd": {"kernel": "fa_fwd_fp32_tc (split + attn)", "achieved": fwd_achieved,
                            "frac": fwd_achieved * 3 / (peak / 2), "ms": first_ms,
                            "flops_per_launch": flops_fwd},
                    "sources": tc_key}
    elif w.backward:
        bwd_achieved = flops_bwd / (second_ms * 1e-3) / 1e12
        bname, fname = (("fa_bwd_masked", "fa_fwd_masked") if masked else
                        ("fa_bwd_dropout", "fa_fwd_dropout") if w.dropout else ("fa_bwd", "fa_fwd"))
        roofline = {"bound": "tensor",
                    "kernel": "%s (bwd_main + preprocess + dq_convert)" % bname,
                    "achieved": bwd_achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": bwd_achieved / peak,
                    "traffic": NCU_TRAFFIC.get(bwd_key), "peak_source": peak_source,
                    "flops_per_launch": flops_bwd,
                    "fwd": {"kernel": fname, "achieved": fwd_achieved,
                            "frac": fwd_achieved / peak, "ms": first_ms,
                            "flops_per_launch": flops_fwd,
                            "mufu_ex2": ex2_ceiling(exps, flops_fwd, first_ms,
                                                    (clocks or {}).get("sm_mhz"), num_sms)},
                    "mufu_ex2": ex2_ceiling(exps, flops_bwd, second_ms,
                                            (clocks or {}).get("sm_mhz"), num_sms),
                    "bwd_ms": second_ms, "sources": bwd_key}
        if det_bwd_ms is not None:
            roofline["deterministic_bwd"] = {
                "kernel": "fa_bwd_deterministic (dQ reductions in a fixed order)",
                "ms": det_bwd_ms, "achieved": flops_bwd / (det_bwd_ms * 1e-3) / 1e12,
                "time_vs_fa_bwd": det_bwd_ms / second_ms}
    else:
        roofline = {"bound": "tensor",
                    "kernel": ("fa_fwd_kvouter" if w.kv_outer else
                               "fa_fwd_fp32_tc (split + attn)" if w.tensor_fp32 else "fa_fwd"),
                    "achieved": fwd_achieved,
                    "peak": peak, "unit": "TFLOP/s", "frac": fwd_achieved / peak,
                    "traffic": NCU_TRAFFIC.get(fwd_key), "peak_source": peak_source,
                    "flops_per_launch": w.flops_fwd(), "ms": first_ms,
                    "one_pass_fwd_ms": one_pass_ms,
                    "sources": (kernel_sources_hash("fa_fwd_kvouter_sm103a.cu") + ":" + w.name
                                if w.kv_outer else
                                kernel_sources_hash("fa_fwd_tf32x3_sm103a.cu") + ":" + w.name
                                if w.tensor_fp32 else fwd_key)}
        if w.kv_outer or w.tensor_fp32:
            roofline["traffic"] = NCU_TRAFFIC.get(roofline["sources"])
        if w.tensor_fp32:
            # three TF32 products per product: the TF32 dense peak (bf16 / 2 nominal) x 1/3
            roofline.update({"peak": peak / 2, "peak_source": peak_source + " x 1/2 (TF32 rate)",
                             "frac": fwd_achieved * 3 / (peak / 2),
                             "note": "achieved counts the method's FLOPs once; frac counts the "
                                     "three TF32 products against the TF32 peak",
                             "simt_fp32_fwd_ms": one_pass_ms})
    cpu = None
    if rank == 0 and ws == 1 and args.cpu_budget > 0 and not args.no_extras:
        r = cpu_oracle_sample(w, args.cpu_budget, w.B * w.Hq)
        cpu = {k: r[k] for k in ("value", "unit", "cores", "kind", "sample")}
        ci = cpu_info()
        cpu.update(cpu_model=ci["cpu_model"], omp_num_threads=ci["omp_num_threads"])

    if rank == 0:
        if w.backward:
            what = "fwd+bwd" + (" under a general mask (%s)" % w.mask if masked else
                                " with dropout p=%g" % w.dropout if w.dropout else
                                " on tensor cores (3xTF32)" if w.tensor_fp32 else "")
            l2 = ("inputs larger than L2 (Q,K,V,dO,O = 5 x %.0f MB), no flush"
                  % (q.numel() * q.element_size() / 1e6))
        else:
            what = ("fwd (split-KV x%d + merge)" % S if split else
                    "fwd, key/value-outer order" if w.kv_outer else
                    "fwd fp32 on tensor cores (3xTF32)" if w.tensor_fp32 else "fwd")
            l2 = ("Q,K,V,O = 4 x %.0f MB%s; no flush" % (
                q.numel() * q.element_size() / 1e6,
                " + fp32 partials %.0f MB" % (Op.numel() * 4 / 1e6) if split else ""))
        line = {"metric": "attention TFLOP/s %s, %s d=%d %s"
                          % (what, "fp32" if w.tensor_fp32 else "bf16", d,
                             "causal" if w.causal else "non-causal"),
                "value": value,
                "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": total_ms / args.steps, "higher_is_better": True,
                # per-step spread of the timed steps (this rank): median and fastest
                "ms_per_step_median": step_times[len(step_times) // 2],
                "ms_per_step_min": step_times[0],
                "scaling": "weak", "vs_baseline": None,
                "dtype": "f32" if w.tensor_fp32 else "bf16", "data": "synthetic",
                "config": {"workload": w.name, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d,
                           "causal": w.causal, "seed": w.seed, "scale": w.scale,
                           "num_splits": S, "mask": w.mask or None,
                           "flops": ("4 d per allowed pair" if masked else
                                     "4 B Hq N^2 d (/2 causal)") +
                                    (" (x3.5 fwd+bwd)" if w.backward else " (forward)"),
                           "l2": l2, "parallelism": "replicas x%d" % ws},
                "fwd_tflops": fwd_achieved,
                "fwd_frac_of_peak": fwd_achieved / peak,
                "fwd_bwd_frac_of_peak": value / ws / peak if w.backward else None,
                # the same fractions against the nominal dense bf16 rate of the datasheet
                "nominal_peak_tflops": NOMINAL_BF16_TFLOPS,
                "fwd_frac_of_nominal_peak": fwd_achieved / NOMINAL_BF16_TFLOPS,
                "fwd_bwd_frac_of_nominal_peak": (value / ws / NOMINAL_BF16_TFLOPS
                                                 if w.backward else None),
                "other_workloads": others,
                # how the K timed steps ran, and the same steps as eager calls
                "timed_as": ("replays of one step captured in a CUDA graph" if graph is not None
                             else "eager calls"),
                "eager": {"ms_per_step": eager_total_ms / args.steps,
                          "value": whole_job_tflops(ws, flops_step, args.steps, eager_total_ms),
                          "unit": "TFLOP/s"},
                # (not measured under --no-extras: null rather than NaN, which is not JSON)
                "e2e": {"value": None if math.isnan(e2e_ms) else e2e_value, "unit": "TFLOP/s",
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "ms_per_step": None if math.isnan(e2e_ms) else e2e_ms / args.steps,
                        "pipeline": "host-to-device copy of step k+1 and device-to-host copy "
                                    "of step k-1 overlap step k (two device buffer sets, copy "
                                    "streams); first and last copies inside the timed region"},
                "gpu_launches": args.steps * (
                    (2 if split or w.tensor_fp32 else 1) +
                    ((4 if w.tensor_fp32 else 3) if w.backward else 0)),
                "gpu_launches_other_workloads": (4 * args.steps * len(others)) if others else 0,
                "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks}
        print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
