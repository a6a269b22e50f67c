"""Multi-process host logic on the CPU with the gloo backend, world size 2 (no GPU):
the max-over-ranks timing of bench.py, the all-gather of sequence-parallel partials,
and the reference arm under torchrun (rank 0 prints one line, rank 1 exits at once)."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _max_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    _init(rank, world, port)
    try:
        q.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def _sp_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from decode_attention_05_gb300.sequence_parallel import gather_partials
    _init(rank, world, port)
    try:
        # One long row cut into two contiguous shards; this rank's partial is the
        # oracle's unsplit result over its shard (a one-split partial, as a device
        # would produce), and the gathered partials merge to the full result.
        rng = np.random.default_rng(5)
        B, Hq, Hkv, d, L = 2, 4, 2, 8, 40
        qv = rng.standard_normal((B, Hq, d)).astype(np.float32)
        k = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
        v = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
        cut = [0, 23, L]
        lo, hi = cut[rank], cut[rank + 1]
        o, lse = oracle.decode(qv, np.ascontiguousarray(k[:, :, lo:hi]),
                               np.ascontiguousarray(v[:, :, lo:hi]),
                               np.full(B, hi - lo, np.int32))
        lse_all, o_all = gather_partials(torch.from_numpy(lse)[:, :, None],
                                         torch.from_numpy(o)[:, :, None, :])
        q.put((rank, lse_all.numpy(), o_all.numpy()))
    finally:
        dist.destroy_process_group()


def test_sequence_parallel_gather_gloo():
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_sp_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = {}
    for _ in range(2):
        rank, lse_all, o_all = q.get(timeout=10)
        res[rank] = (lse_all, o_all)
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])
    lse_all, o_all = res[0]
    assert lse_all.shape == (2, 4, 2) and o_all.shape == (2, 4, 2, 8)
    # Rank-major: split 0 is rank 0's shard.  The merged result equals the unsplit one.
    rng = np.random.default_rng(5)
    qv = rng.standard_normal((2, 4, 8)).astype(np.float32)
    k = rng.standard_normal((2, 2, 40, 8)).astype(np.float32)
    v = rng.standard_normal((2, 2, 40, 8)).astype(np.float32)
    ref_o, ref_l = oracle.decode(qv, k, v, np.full(2, 40, np.int32))
    for b in range(2):
        for h in range(4):
            parts = [(o_all[b, h, s].astype(np.float64), float(lse_all[b, h, s])) for s in range(2)]
            mo, ml = oracle.merge_blocks(parts)
            assert np.allclose(mo, ref_o[b, h], rtol=1e-6, atol=1e-6)
            assert abs(ml - ref_l[b, h]) < 1e-5


def test_reference_arm_under_torchrun():
    """`bench.py --impl reference` launched like the multi-GPU runs: only rank 0 works
    and prints one JSON line; the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--config", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"


def _splits_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    from decode_attention_05_gb300 import sequence_parallel as sp
    _init(rank, world, port)
    try:
        # Shards of different capacities resolve different local counts; every rank must
        # use the largest (the gather needs one count everywhere).
        sp.fd.resolve_num_splits = lambda B, Hq, Hkv, d, cap, n: 3 + 5 * rank
        q.put((rank, sp.shard_num_splits(1, 8, 1, 128, 1000 * (rank + 1), 0),
               sp.shard_num_splits(1, 8, 1, 128, 1000, 7)))
    finally:
        dist.destroy_process_group()


def test_shard_split_count_agrees_across_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_splits_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 8, 7), (1, 8, 7)]
