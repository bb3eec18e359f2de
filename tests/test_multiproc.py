"""Multi-rank logic of the benchmark on the CPU: two gloo processes.

The attention path has no data-path exchange; N > 1 runs are replicas on their own seeded
inputs, and the only collective is the MAX over ranks of the timed region.  These tests run
those pieces with world_size 2 on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import bench
    from exact_attention_89_gb300.inputs import make_inputs
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, _ = bench.dist_env()
        ms = 10.0 + 5.0 * rank                       # rank 1 is the slow one
        mx = bench.max_over_ranks(ms, got_ws, torch.device("cpu"))
        q, _, _, _ = make_inputs(1, 2, 1, 16, 8, seed=7 + bench.replica_seed_offset(got_rank))
        val = bench.whole_job_tflops(got_ws, 1e12, 10, mx)
        out[rank] = (got_ws, got_rank, mx, float(q.float().sum()), val)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_and_max_timing():
    ws = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(ws, port, out), nprocs=ws, join=True)
    r0, r1 = out[0], out[1]
    assert (r0[0], r0[1]) == (2, 0) and (r1[0], r1[1]) == (2, 1)
    # every rank sees the slowest rank's time
    assert r0[2] == r1[2] == 15.0
    # replicas draw different inputs, deterministically
    assert r0[3] != r1[3]
    from exact_attention_89_gb300.inputs import make_inputs
    assert float(make_inputs(1, 2, 1, 16, 8, seed=8)[0].float().sum()) == r1[3]
    # whole-job value: 2 ranks x 10 steps x 1 TFLOP in 15 ms
    assert abs(r0[4] - 2 * 10 * 1e12 / 15e-3 / 1e12) < 1e-9


def test_single_rank_helpers():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.replica_seed_offset(3) == 3
    assert abs(bench.whole_job_tflops(1, 2e12, 4, 8.0) - 1000.0) < 1e-9


def test_split_key_ranges_partition_the_keys():
    """The merge-traffic accounting assumes the split forward's ranges: ceil(nb / S) 128-key
    blocks per range, the last ones possibly short or empty, together exactly [0, N)."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    for N in (1, 127, 128, 129, 1000, 4096, 32768):
        for S in (1, 2, 3, 4, 7, 64):
            r = bench.split_key_ranges(N, S)
            assert len(r) == S
            nb = -(-N // 128)
            per = -(-nb // S)
            pos = 0
            for s, (k0, k1) in enumerate(r):
                assert k0 == min(N, s * per * 128) and k1 == min(N, (s + 1) * per * 128)
                assert k0 == pos or k1 == k0
                assert k0 % 128 == 0 or k0 == N
                pos = max(pos, k1)
            assert pos == N


def test_traffic_key_ignores_comments_only():
    """The ncu traffic table is keyed by the kernels' code without comments: a comment edit keeps
    the key (the captured kernel is unchanged), any edit of the code changes it."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    src = 'int f(int a) { // add one\n    return a + 1; /* the result */\n}\n'
    assert bench._code_only(src) == bench._code_only(src.replace('add one', 'increment'))
    assert bench._code_only(src) == bench._code_only(src.replace('/* the result */', '') + '\n\n')
    assert bench._code_only(src) != bench._code_only(src.replace('a + 1', 'a + 2'))
    assert bench._code_only('x = 1; /* a\nb */ y = 2;') == 'x = 1;  y = 2;'
