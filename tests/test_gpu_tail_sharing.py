"""Tail sharing on the tcgen05 kernel (FD_SCHEDULE_TAIL_SHARING, opt-in): a CTA
that has finished its own split takes tiles from the back of a split of the same
(b, kv head) still in progress and folds them into its own partial.  Every key must
still land in exactly one partial, so the merged result equals the fp64 oracle within
the bf16 tolerance of test_gpu_parity:
  out: |got - ref| <= 4e-3 + 8e-3 |ref|     lse: |got - ref| <= 1e-4 + 1e-5 |ref|

* parity with and without sharing over contiguous and paged caches, ragged rows and
  multi-token groups, in both merge modes;
* a workload where sharing is certain to happen (one split of a group ends after one
  tile while the others hold 32): that split's LSE_i must grow, because its partial now
  holds stolen keys, while the merged result stays the oracle's;
* claim words left by a larger call in the same workspace, and CUDA-graph replays of
  one call (same epoch every time), must not hand out tiles twice.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")


def _case(Q, G, Hkv, lens, ps, cap, seed):
    Hq = Hkv * G
    if ps:
        w = workloads.paged_case(len(lens), Hq, Hkv, 128, ps, -(-cap // ps), lens, seed=seed,
                                 extra_pages=2, out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(len(lens), Hq, Hkv, 128, cap, lens, seed=seed,
                                      out_dtype=torch.float32)
    q4 = workloads.multi_token_queries(len(lens), Q, Hq, 128, seed=seed + 1)
    _, k, v, lens_np, bt, pg = w.oracle_arrays()
    ref = oracle.decode_causal(workloads.np_storage(q4), k, v, lens_np, block_table=bt,
                               page_size=pg)
    return w, q4, ref


def _check(o, l, ref_o, ref_l):
    o = o.double().cpu().numpy().reshape(ref_o.shape)
    l = l.double().cpu().numpy().reshape(ref_l.shape)
    assert not np.isnan(o).any() and not np.isnan(l).any()
    err = np.abs(o - ref_o)
    assert (err <= 4e-3 + 8e-3 * np.abs(ref_o)).all(), "out max err %.3g" % err.max()
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(l), empty)
    assert (o[empty] == 0).all()
    lerr = np.abs(l[~empty] - ref_l[~empty])
    assert (lerr <= 1e-4 + 1e-5 * np.abs(ref_l[~empty])).all(), "lse max err %.3g" % lerr.max()


def _run(w, q4, S, schedule, merge=fd.FD_MERGE_KERNEL, ws=None):
    B, Q, Hq, d = q4.shape
    wd = w.to("cuda")
    if ws is None:
        ws = torch.zeros(fd.workspace_size(B, Q * Hq, w.Hkv, d, S), dtype=torch.uint8,
                         device="cuda")
    opts = fd.options(path=fd.FD_PATH_TCGEN05, schedule=schedule, merge_mode=merge)
    o, l = fd.decode_attention(q4.cuda(), wd.k, wd.v, wd.seq_lens, wd.block_table, w.page_size,
                               S, workspace=ws, out_dtype=torch.float32, options=opts)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    return o, l, ws


@pytest.mark.parametrize("schedule", [fd.FD_SCHEDULE_TAIL_SHARING, fd.FD_SCHEDULE_GRID])
@pytest.mark.parametrize("merge", [fd.FD_MERGE_KERNEL, fd.FD_MERGE_IN_KERNEL])
@pytest.mark.parametrize("Q,G,Hkv,lens,ps,cap,S", [
    (4, 8, 2, [6000, 1, 2500], 0, 8192, 6),
    (8, 8, 1, [8192, 7000], 0, 8192, 5),
    (2, 16, 2, [3000, 4096, 65], 16, 4096, 7),
    (3, 8, 2, [5000, 333], 64, 6144, 4),
    (1, 32, 1, [7777], 0, 8192, 9),
])
def test_tail_sharing_parity(Q, G, Hkv, lens, ps, cap, S, schedule, merge):
    w, q4, (ref_o, ref_l) = _case(Q, G, Hkv, lens, ps, cap, seed=500 + Q + G + len(lens))
    o, l, _ = _run(w, q4, S, schedule, merge)
    _check(o, l, ref_o, ref_l)


def test_tail_sharing_moves_keys_between_partials():
    # Row length 3 * 2048 + 64 with split_len 2048: splits 0-2 hold 32 tiles each, split 3
    # one tile.  Split 3's CTA is done long before the others and takes tiles from them.
    L = 3 * 2048 + 64
    w, q4, (ref_o, ref_l) = _case(4, 8, 1, [L], 0, 4 * 2048, seed=777)
    S = 4
    B, Q, Hq, d = q4.shape
    lse_parts = {}
    for schedule in (fd.FD_SCHEDULE_GRID, fd.FD_SCHEDULE_TAIL_SHARING):
        o, l, ws = _run(w, q4, S, schedule)
        _check(o, l, ref_o, ref_l)
        lp, _ = fd.workspace_partials(ws, B * Q, Hq, d, S)
        lse_parts[schedule] = lp.double().cpu().numpy().reshape(B * Q * Hq, S)
    grid, shared = lse_parts[fd.FD_SCHEDULE_GRID], lse_parts[fd.FD_SCHEDULE_TAIL_SHARING]
    # More keys in split 3's partial: its LSE (log of a sum of positive terms) grows.
    assert (shared[:, 3] > grid[:, 3] + 1e-3).all()
    # Fewer in at least one of the others.
    assert (shared[:, :3] < grid[:, :3] - 1e-3).any()


def test_tail_sharing_after_a_larger_call_and_in_graph_replays():
    big_w, big_q, (big_o, big_l) = _case(8, 8, 1, [8192], 0, 8192, seed=900)
    w, q4, (ref_o, ref_l) = _case(4, 8, 2, [6000, 2048], 0, 8192, seed=901)
    B, Q, Hq, d = q4.shape
    ws = torch.zeros(fd.workspace_size(1, 8 * 8, 1, 128, 64) + (1 << 20), dtype=torch.uint8,
                     device="cuda")
    # A larger call first: its partials fill the region where the next call's claim words
    # live.
    o, l, _ = _run(big_w, big_q, 64, fd.FD_SCHEDULE_TAIL_SHARING, ws=ws)
    _check(o, l, big_o, big_l)
    o, l, _ = _run(w, q4, 6, fd.FD_SCHEDULE_TAIL_SHARING, ws=ws)
    _check(o, l, ref_o, ref_l)
    # The same call captured once and replayed: the replays share one epoch.
    wd = w.to("cuda")
    qd = q4.cuda()
    out = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(qd.shape[:-1], dtype=torch.float32, device="cuda")
    opts = fd.options(path=fd.FD_PATH_TCGEN05, schedule=fd.FD_SCHEDULE_TAIL_SHARING)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fd.decode_attention(qd, wd.k, wd.v, wd.seq_lens, None, 0, 6, out=out, lse_out=lse,
                            workspace=ws, options=opts)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fd.decode_attention(qd, wd.k, wd.v, wd.seq_lens, None, 0, 6, out=out, lse_out=lse,
                            workspace=ws, options=opts)
    for _ in range(5):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        _check(out, lse, ref_o, ref_l)
    assert fd.read_device_error(ws) == 0
