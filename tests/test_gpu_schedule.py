"""GPU parity of the alternative schedules of the tensor-core partial pass.

Persistent: the same per-item arithmetic as the non-persistent kernel of the same tiling
(the grid kernel, or the head-group kernel where the automatic rule takes head groups),
only assigned differently to CTAs, so every case is checked twice: against the fp64
oracle (the tolerances of test_gpu_parity) and bit for bit against that kernel.  The
queue in the workspace header must also come back clean after each launch (several
calls in a row, stale workspace contents, a replayed CUDA graph).

Head groups: tiles of 16 tokens x 4 kv heads (small pages, contiguous caches); checked against the
oracle and against the grid schedule up to rounding order.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import cached, check, ref_for

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")


@pytest.fixture(autouse=True)
def _restore_schedule():
    yield
    if torch.cuda.is_available():
        fd.set_schedule(fd.FD_SCHEDULE_AUTO)
        fd.set_path(fd.FD_PATH_AUTO)
        fd.set_merge_mode(fd.FD_MERGE_KERNEL)


def _decode(wd, w, S, ws=None, q=None):
    B, Hq, d = w.q.shape
    Qn = 1 if q is None else q.shape[1]
    if ws is None:
        ws = torch.zeros(fd.workspace_size(B, Qn * Hq, w.Hkv, d, S), dtype=torch.uint8,
                         device="cuda")
    o, l = fd.decode_attention(wd.q if q is None else q, wd.k, wd.v, wd.seq_lens,
                               wd.block_table, wd.page_size, S, workspace=ws,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    return o, l


def _both(wd, w, S, q=None):
    """Persistent schedule and the automatic one (the same tiling), bit for bit."""
    fd.set_path(fd.FD_PATH_MMA)
    fd.set_schedule(fd.FD_SCHEDULE_AUTO)
    og, lg = _decode(wd, w, S, q=q)
    fd.set_schedule(fd.FD_SCHEDULE_PERSISTENT)
    op, lp = _decode(wd, w, S, q=q)
    assert torch.equal(og, op), "persistent and non-persistent outputs differ"
    assert torch.equal(lg, lp), "persistent and non-persistent LSE differ"
    return op, lp


CASES = {
    # name: (builder, split counts)
    "gqa8-ragged": (lambda: workloads.contiguous_case(
        6, 32, 4, 128, 5000, [5000, 1, 0, 4097, 2500, 129], seed=401), (1, 7, 64, 300)),
    "mha-d64": (lambda: workloads.contiguous_case(
        3, 16, 16, 64, 3000, [3000, 1000, 17], seed=402), (1, 9, 40)),
    "gqa16": (lambda: workloads.contiguous_case(
        2, 32, 2, 128, 4000, [4000, 3333], seed=403), (3, 100)),
    "paged16": (lambda: workloads.paged_case(
        5, 32, 8, 128, 16, 256, [4096, 1, 0, 2500, 77], seed=404), (1, 6, 40)),
    "paged256": (lambda: workloads.paged_case(
        4, 16, 4, 128, 256, 16, [4096, 300, 2000, 1], seed=405), (2, 16, 64)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_persistent_matches_oracle_and_grid(name):
    build, splits = CASES[name]
    w = build()
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    for S in splits:
        o, l = _both(wd, w, S)
        check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


def test_persistent_full_size_gqa_128k_sampled():
    """The 128K-token GQA workload with a split count that makes thirteen times more
    items than SMs: grid and persistent agree bit for bit and match the oracle."""
    w, wd = cached(3)
    o, l = _both(wd, w, 256)
    ref_o, ref_l = ref_for(w, "c3")
    check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


@pytest.mark.parametrize("Q,G", [(2, 8), (4, 4), (16, 1)])
def test_persistent_multi_token(Q, G):
    Hkv, d = 2, 128
    Hq = Hkv * G
    lens = [1, 65, 300, 1000]
    w = workloads.paged_case(len(lens), Hq, Hkv, d, 16, 64, lens, seed=410 + Q,
                             out_dtype=torch.float32)
    q4 = workloads.multi_token_queries(len(lens), Q, Hq, d, seed=420 + Q)
    _, k, v, lens_np, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_causal(workloads.np_storage(q4), k, v, lens_np,
                                        block_table=bt, page_size=ps)
    wd = w.to("cuda")
    B = len(lens)
    for S in (1, 16, 50):
        o, l = _both(wd, w, S, q=q4.cuda())
        mw = workloads.Workload("mt", q4.reshape(B * Q, Hq, d), w.k, w.v, w.seq_lens)
        check(mw, o.cpu().double().numpy().reshape(B * Q, Hq, d),
              l.cpu().double().numpy().reshape(B * Q, Hq),
              ref_o.reshape(B * Q, Hq, d), ref_l.reshape(B * Q, Hq))


def test_persistent_fp8_kv():
    w = workloads.paged_case(4, 32, 8, 128, 16, 256, [1, 37, 2500, 4096], seed=430)
    kc, vc, ks, vs = workloads.fp8_quantize(w)
    q, _, _, lens, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_kv8(q, kc.view(torch.uint8).numpy(), vc.view(torch.uint8).numpy(),
                                     ks.numpy(), vs.numpy(), lens, block_table=bt, page_size=ps)
    wd = w.to("cuda")
    args = (wd.q, kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda(), wd.seq_lens, wd.block_table, 16)
    res = []
    for sched in (fd.FD_SCHEDULE_GRID, fd.FD_SCHEDULE_PERSISTENT):
        fd.set_schedule(sched)
        ws = torch.zeros(fd.workspace_size(4, 32, 8, 128, 48), dtype=torch.uint8, device="cuda")
        o, l = fd.decode_attention_fp8kv(*args, 48, workspace=ws)
        torch.cuda.synchronize()
        assert fd.read_device_error(ws) == 0
        check(w, o.float().cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)
        res.append((o, l))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


@pytest.mark.parametrize("kind", ["paged16", "contiguous-large-batch", "fp8-paged32"])
def test_persistent_head_groups(kind):
    """The persistent schedule over head-group tiles (where the automatic rule takes
    them): items of 4 kv heads from the queue, a warp per head.  Against the oracle and,
    bit for bit, the head-group kernel, for 1 to 37 splits.  A large batch of short rows
    (at most 256 tokens per split) takes it by default."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hkv, G = 8, 4
    name = lambda B, ps, kv, S: fd.partial_kernel_name_for(
        torch.bfloat16, kv, B, 1, Hkv * G, Hkv, 128, ps, 2048, S,
        options=fd.options(path=fd.FD_PATH_MMA, schedule=fd.FD_SCHEDULE_PERSISTENT))
    if kind == "contiguous-large-batch":
        B = -(-6 * sms * 4 // Hkv)              # 6 head-group items per SM at one split
        import random
        rnd = random.Random(460)
        lens = [0, 1, 16, 17, 200] + [rnd.randint(1, 200) for _ in range(B - 5)]
        w = workloads.contiguous_case(B, Hkv * G, Hkv, 128, 200, lens, seed=461,
                                      out_dtype=torch.float32)
        assert name(B, 0, torch.bfloat16, 1) == "fd_partial_heads_persist_kernel"
        assert name(-(-5 * sms // Hkv) - 1, 0, torch.bfloat16, 1) == "fd_partial_persist_kernel"
        splits = (1, 3)
    else:
        ps = 16 if kind == "paged16" else 32
        w = workloads.paged_case(len(HEAD_LENS), Hkv * G, Hkv, 128, ps, -(-2048 // ps),
                                 HEAD_LENS, seed=462 + ps, extra_pages=1,
                                 out_dtype=torch.float32)
        splits = (1, 6, 37)
    if kind != "fp8-paged32":
        if kind == "paged16":
            assert name(8, 16, torch.bfloat16, 6) == "fd_partial_heads_persist_kernel"
        ref_o, ref_l = ref_for(w)
        wd = w.to("cuda")
        for S in splits:
            oh, lh = _run_sched(wd, w, S, fd.FD_SCHEDULE_HEAD_GROUPS)
            op, lp = _run_sched(wd, w, S, fd.FD_SCHEDULE_PERSISTENT)
            check(w, op.cpu().double().numpy(), lp.cpu().double().numpy(), ref_o, ref_l)
            assert torch.equal(oh, op) and torch.equal(lh, lp)
            if kind == "contiguous-large-batch":      # the automatic choice (200 tokens)
                oa, la = _run_sched(wd, w, S, fd.FD_SCHEDULE_AUTO)
                assert torch.equal(oa, op) and torch.equal(la, lp)
        return
    assert name(8, 32, torch.float8_e4m3fn, 6) == "fd_partial_heads_persist_kernel"
    kc, vc, ks, vs = workloads.fp8_quantize(w)
    q, _, _, lens, bt, ps_ = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_kv8(q, kc.view(torch.uint8).numpy(), vc.view(torch.uint8).numpy(),
                                     ks.numpy(), vs.numpy(), lens, block_table=bt, page_size=ps_)
    wd = w.to("cuda")
    args = (wd.q, kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda(), wd.seq_lens, wd.block_table, 32)
    fd.set_path(fd.FD_PATH_MMA)
    for S in splits:
        res = []
        for sched in (fd.FD_SCHEDULE_HEAD_GROUPS, fd.FD_SCHEDULE_PERSISTENT):
            fd.set_schedule(sched)
            ws = torch.zeros(fd.workspace_size(w.B, 32, 8, 128, S), dtype=torch.uint8,
                             device="cuda")
            o, l = fd.decode_attention_fp8kv(*args, S, workspace=ws, out_dtype=torch.float32)
            torch.cuda.synchronize()
            assert fd.read_device_error(ws) == 0
            check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)
            res.append((o, l))
        assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


@pytest.mark.parametrize("d,paged", [(128, 0), (128, 16), (64, 0), (64, 8)])
def test_persistent_wide_groups(d, paged):
    """The persistent schedule over wide groups (4 query tokens x G 8 = 32 rows per kv
    head, 8 rows a warp): against the multi-token oracle and, bit for bit, the wide
    kernel on the grid, for 1, 3 and 9 splits; rows shorter than the query count leave
    their first queries without keys."""
    Q, G, Hkv = 4, 8, 2
    Hq = Hkv * G
    lens = [1, 3, 65, 300, 1000, 0]
    if paged:
        w = workloads.paged_case(len(lens), Hq, Hkv, d, paged, -(-1024 // paged), lens,
                                 seed=470 + d + paged, out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(len(lens), Hq, Hkv, d, 1024, lens, seed=470 + d,
                                      out_dtype=torch.float32)
    q4 = workloads.multi_token_queries(len(lens), Q, Hq, d, seed=480 + d)
    _, k, v, lens_np, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_causal(workloads.np_storage(q4), k, v, lens_np,
                                        block_table=bt, page_size=ps)
    B = len(lens)
    assert fd.partial_kernel_name_for(torch.bfloat16, torch.bfloat16, B, Q, Hq, Hkv, d, paged,
                                      w.L_cap, 3, options=fd.options(
                                          path=fd.FD_PATH_MMA,
                                          schedule=fd.FD_SCHEDULE_PERSISTENT)) == \
        "fd_partial_wide_persist_kernel"
    wd = w.to("cuda")
    qd = q4.cuda()
    for S in (1, 3, 9):
        og, lg = _run_sched(wd, w, S, fd.FD_SCHEDULE_GRID, q=qd)
        op, lp = _run_sched(wd, w, S, fd.FD_SCHEDULE_PERSISTENT, q=qd)
        assert torch.equal(og, op) and torch.equal(lg, lp)
        mw = workloads.Workload("mt", q4.reshape(B * Q, Hq, d), w.k, w.v, w.seq_lens)
        check(mw, op.cpu().double().numpy().reshape(B * Q, Hq, d),
              lp.cpu().double().numpy().reshape(B * Q, Hq),
              ref_o.reshape(B * Q, Hq, d), ref_l.reshape(B * Q, Hq))


def test_persistent_back_to_back_and_stale_workspace():
    """Calls in a row on one stream with no host sync between them, in a workspace whose
    partial regions start as random bytes: each launch must find a clean queue."""
    fd.set_path(fd.FD_PATH_MMA)
    fd.set_schedule(fd.FD_SCHEDULE_PERSISTENT)
    cases = [workloads.contiguous_case(3, 16, 4, 128, 2000, [2000, 5, 999], seed=440 + i,
                                       out_dtype=torch.float32) for i in range(3)]
    refs = [ref_for(w) for w in cases]
    n = fd.workspace_size(3, 16, 4, 128, 200)
    g = torch.Generator(device="cuda").manual_seed(9)
    ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
    ws[:256] = 0
    outs = []
    for rep in range(3):
        for w, S in zip(cases, (200, 7, 1)):
            wd = w.to("cuda")
            outs.append(fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, num_splits=S,
                                            workspace=ws, out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    for i, (o, l) in enumerate(outs):
        ro, rl = refs[i % 3]
        check(cases[i % 3], o.cpu().double().numpy(), l.cpu().double().numpy(), ro, rl)
    # The queue words are back to zero after the last launch.
    assert int(ws[64:72].view(torch.int64).item()) == 0
    assert int(ws[128:136].view(torch.int64).item()) == 0


def test_persistent_graph_replay():
    """A captured decode replayed several times: the same launch (same queue epoch) runs
    again, so it relies on the last CTA putting the queue back to zero."""
    fd.set_path(fd.FD_PATH_MMA)
    fd.set_schedule(fd.FD_SCHEDULE_PERSISTENT)
    w = workloads.paged_case(4, 32, 8, 128, 16, 128, [2048, 1000, 1, 1500], seed=450,
                             out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    S = 64
    ws = torch.zeros(fd.workspace_size(4, 32, 8, 128, S), dtype=torch.uint8, device="cuda")
    out = torch.empty(4, 32, 128, dtype=torch.float32, device="cuda")
    lse = torch.empty(4, 32, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                     # warm-up outside the capture
        fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, wd.block_table, 16, S,
                            workspace=ws, out=out, lse_out=lse)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, wd.block_table, 16, S,
                            workspace=ws, out=out, lse_out=lse)
    for _ in range(3):
        out.zero_()
        lse.zero_()
        graph.replay()
        torch.cuda.synchronize()
        check(w, out.cpu().double().numpy(), lse.cpu().double().numpy(), ref_o, ref_l)
    assert fd.read_device_error(ws) == 0


# ------------------------------------------------------------------ head-group tiles

def _run_sched(wd, w, S, sched, q=None, out_dtype=torch.float32):
    fd.set_path(fd.FD_PATH_MMA)
    fd.set_schedule(sched)
    B, Hq, d = w.q.shape
    Qn = 1 if q is None else q.shape[1]
    ws = torch.zeros(fd.workspace_size(B, Qn * Hq, w.Hkv, d, S), dtype=torch.uint8, device="cuda")
    o, l = fd.decode_attention(wd.q if q is None else q, wd.k, wd.v, wd.seq_lens,
                               wd.block_table, wd.page_size, S, workspace=ws, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    return o, l


HEAD_LENS = [0, 1, 15, 16, 17, 37, 500, 2048]


@pytest.mark.parametrize("ps,Hkv,G", [(16, 4, 1), (16, 4, 8), (16, 8, 4), (32, 8, 2),
                                      (16, 12, 16), (32, 4, 16), (64, 8, 4), (256, 4, 2)])
def test_head_groups_match_oracle_and_grid(ps, Hkv, G):
    """Tiles of 16 tokens x 4 kv heads (one TMA box), one consumer warp per head: against
    the oracle, and against the one-head-per-CTA grid schedule.  The outputs of the two
    differ by the bf16 rounding of P (each warp's running maximum differs), so only the
    oracle bound applies to them; the LSE (from fp32 sums) must agree closely."""
    w = workloads.paged_case(len(HEAD_LENS), Hkv * G, Hkv, 128, ps, -(-2048 // ps), HEAD_LENS,
                             seed=500 + ps + Hkv + G, extra_pages=2, out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    for S in (1, 5, 33):
        oh, lh = _run_sched(wd, w, S, fd.FD_SCHEDULE_HEAD_GROUPS)
        check(w, oh.cpu().double().numpy(), lh.cpu().double().numpy(), ref_o, ref_l)
        og, lg = _run_sched(wd, w, S, fd.FD_SCHEDULE_GRID)
        assert torch.equal(torch.isneginf(lh), torch.isneginf(lg))
        fin = torch.isfinite(lg)
        assert torch.allclose(lh[fin], lg[fin], atol=1e-5, rtol=1e-6)


@pytest.mark.parametrize("Hkv,G", [(4, 1), (8, 4), (12, 16), (4, 8)])
def test_head_groups_contiguous(Hkv, G):
    """Head-group tiles on a contiguous cache (16 tokens x 4 kv heads of a row, one TMA
    box; stale slots past each length hold NaN; the last box of a row runs past the
    capacity): against the oracle and the grid schedule's LSE, with 1, 5 and 33 splits."""
    w = workloads.contiguous_case(len(HEAD_LENS), Hkv * G, Hkv, 128, 2050, HEAD_LENS,
                                  seed=580 + Hkv + G, out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    for S in (1, 5, 33):
        oh, lh = _run_sched(wd, w, S, fd.FD_SCHEDULE_HEAD_GROUPS)
        check(w, oh.cpu().double().numpy(), lh.cpu().double().numpy(), ref_o, ref_l)
        og, lg = _run_sched(wd, w, S, fd.FD_SCHEDULE_GRID)
        assert torch.equal(torch.isneginf(lh), torch.isneginf(lg))
        fin = torch.isfinite(lg)
        assert torch.allclose(lh[fin], lg[fin], atol=1e-5, rtol=1e-6)


def test_head_groups_contiguous_multi_token():
    Q, G, Hkv, d = 2, 8, 8, 128
    Hq = Hkv * G
    lens = [1, 2, 65, 300, 1000]
    w = workloads.contiguous_case(len(lens), Hq, Hkv, d, 1000, lens, seed=590,
                                  out_dtype=torch.float32)
    q4 = workloads.multi_token_queries(len(lens), Q, Hq, d, seed=591)
    _, k, v, lens_np, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_causal(workloads.np_storage(q4), k, v, lens_np)
    wd = w.to("cuda")
    B = len(lens)
    for S in (1, 3):
        o, l = _run_sched(wd, w, S, fd.FD_SCHEDULE_HEAD_GROUPS, q=q4.cuda())
        mw = workloads.Workload("mt", q4.reshape(B * Q, Hq, d), w.k, w.v, w.seq_lens)
        check(mw, o.cpu().double().numpy().reshape(B * Q, Hq, d),
              l.cpu().double().numpy().reshape(B * Q, Hq),
              ref_o.reshape(B * Q, Hq, d), ref_l.reshape(B * Q, Hq))


@pytest.mark.parametrize("paged", [0, 64])
def test_head_groups_auto_for_large_batches(paged):
    """The default schedule takes head groups on a contiguous cache (or 64-token pages)
    once the batch holds 5 (b, kv head) pairs per SM, and the grid below that: a ragged
    batch of that size against the oracle, and the kernel the sized name query reports
    on both sides of the threshold."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hkv, G = 8, 4
    B = -(-5 * sms // Hkv)
    import random
    rnd = random.Random(600)
    lens = [0, 1, 16, 17, 300] + [rnd.randint(1, 300) for _ in range(B - 5)]
    if paged:
        w = workloads.paged_case(B, Hkv * G, Hkv, 128, paged, 5, lens, seed=601,
                                 out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(B, Hkv * G, Hkv, 128, 300, lens, seed=601,
                                      out_dtype=torch.float32)
    name = lambda b: fd.partial_kernel_name_for(torch.bfloat16, torch.bfloat16, b, 1, Hkv * G,
                                                Hkv, 128, paged, w.L_cap)
    assert name(B) == "fd_partial_heads_kernel"              # 300 tokens a split
    assert name(B - 1) == "fd_partial_mma_kernel"
    short = lambda b, L: fd.partial_kernel_name_for(torch.bfloat16, torch.bfloat16, b, 1,
                                                    Hkv * G, Hkv, 128, paged, L, 1)
    B6 = -(-6 * sms * 4 // Hkv)                 # 6 head-group items per SM
    assert short(B6, 256) == "fd_partial_heads_persist_kernel"
    assert short(B6, 320) == "fd_partial_heads_kernel"
    assert short(B6 - 1, 256) == "fd_partial_heads_kernel"
    assert short(B, 256) == "fd_partial_heads_kernel"
    assert short(B - 1, 128) == "fd_partial_mma_kernel"
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    S = fd.resolve_num_splits(B, Hkv * G, Hkv, 128, w.L_cap, 0)
    o, l = _run_sched(wd, w, S, fd.FD_SCHEDULE_AUTO)
    check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


def _fp8_views(codes):
    return codes.view(torch.uint8).numpy()


@pytest.mark.parametrize("ps,Hkv,G", [(0, 8, 4), (32, 8, 4), (64, 4, 8), (0, 4, 16),
                                      (32, 12, 2), (16, 8, 4)])
def test_head_groups_fp8(ps, Hkv, G):
    """FP8 E4M3 caches with head-group tiles of 32 tokens x 4 kv heads (one 16 KB box; a
    warp per head, per-head scales) against the fp64 FP8 oracle, and the grid schedule's
    LSE.  16-token pages cannot hold a 32-token tile: there the setting runs the grid
    schedule, bit for bit."""
    lens = HEAD_LENS
    if ps:
        w = workloads.paged_case(len(lens), Hkv * G, Hkv, 128, ps, -(-2048 // ps), lens,
                                 seed=610 + ps + G, extra_pages=1, out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(len(lens), Hkv * G, Hkv, 128, 2050, lens, seed=610 + G,
                                      out_dtype=torch.float32)
    kc, vc, ks, vs = workloads.fp8_quantize(w)
    q, _, _, lens_np, bt, ps_ = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_kv8(q, _fp8_views(kc), _fp8_views(vc), ks.numpy(), vs.numpy(),
                                     lens_np, block_table=bt, page_size=ps_)
    wd = w.to("cuda")
    kcd, vcd, ksd, vsd = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
    B, Hq = w.B, w.Hq
    expect = "fd_partial_mma_kernel" if ps == 16 else "fd_partial_heads_kernel"
    assert fd.partial_kernel_name_for(torch.bfloat16, torch.float8_e4m3fn, B, 1, Hq, Hkv, 128,
                                      ps, w.L_cap, 5, options=fd.options(
                                          path=fd.FD_PATH_MMA,
                                          schedule=fd.FD_SCHEDULE_HEAD_GROUPS)) == expect
    fd.set_path(fd.FD_PATH_MMA)
    for S in (1, 5, 33):
        res = {}
        for sched in (fd.FD_SCHEDULE_HEAD_GROUPS, fd.FD_SCHEDULE_GRID):
            fd.set_schedule(sched)
            ws = torch.zeros(fd.workspace_size(B, Hq, Hkv, 128, S), dtype=torch.uint8,
                             device="cuda")
            o, l = fd.decode_attention_fp8kv(wd.q, kcd, vcd, ksd, vsd, wd.seq_lens,
                                             wd.block_table, ps, S, workspace=ws,
                                             out_dtype=torch.float32)
            torch.cuda.synchronize()
            assert fd.read_device_error(ws) == 0
            res[sched] = (o, l)
        oh, lh = res[fd.FD_SCHEDULE_HEAD_GROUPS]
        og, lg = res[fd.FD_SCHEDULE_GRID]
        check(w, oh.cpu().double().numpy(), lh.cpu().double().numpy(), ref_o, ref_l)
        if ps == 16:
            assert torch.equal(oh, og) and torch.equal(lh, lg)
        assert torch.equal(torch.isneginf(lh), torch.isneginf(lg))
        fin = torch.isfinite(lg)
        assert torch.allclose(lh[fin], lg[fin], atol=1e-5, rtol=1e-6)


def test_head_groups_fp8_auto_for_large_batches():
    """FP8 cache, contiguous: the default schedule takes head groups from 5 (b, kv head)
    pairs per SM (and for 32-token pages at any batch); a ragged batch of that size
    against the fp64 FP8 oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hkv, G = 8, 4
    B = -(-5 * sms // Hkv)
    import random
    rnd = random.Random(620)
    lens = [0, 1, 32, 33, 300] + [rnd.randint(1, 300) for _ in range(B - 5)]
    w = workloads.contiguous_case(B, Hkv * G, Hkv, 128, 300, lens, seed=621,
                                  out_dtype=torch.float32)
    name = lambda b, ps: fd.partial_kernel_name_for(torch.bfloat16, torch.float8_e4m3fn, b, 1,
                                                    Hkv * G, Hkv, 128, ps, 320)
    assert name(B, 0) == "fd_partial_heads_kernel"
    assert name(B - 1, 0) == "fd_partial_mma_kernel"
    assert name(1, 32) == "fd_partial_heads_kernel"
    assert name(B - 1, 64) == "fd_partial_mma_kernel"
    kc, vc, ks, vs = workloads.fp8_quantize(w)
    q, _, _, lens_np, _, _ = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_kv8(q, _fp8_views(kc), _fp8_views(vc), ks.numpy(), vs.numpy(),
                                     lens_np)
    wd = w.to("cuda")
    o, l = fd.decode_attention_fp8kv(wd.q, kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda(),
                                     wd.seq_lens, out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


def test_head_groups_bf16_out_and_auto_default():
    """The default schedule takes head groups for a 16-token-page bf16 cache; bf16 out."""
    w = workloads.paged_case(4, 32, 8, 128, 16, 128, [2048, 1000, 1, 1500], seed=520)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    o, l = _run_sched(wd, w, 16, fd.FD_SCHEDULE_AUTO, out_dtype=torch.bfloat16)
    check(w, o.float().cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


@pytest.mark.parametrize("Q,G", [(2, 8), (4, 2), (16, 1)])
def test_head_groups_multi_token(Q, G):
    Hkv, d = 4, 128
    Hq = Hkv * G
    lens = [1, 3, 65, 300, 1000]
    w = workloads.paged_case(len(lens), Hq, Hkv, d, 16, 64, lens, seed=530 + Q,
                             out_dtype=torch.float32)
    q4 = workloads.multi_token_queries(len(lens), Q, Hq, d, seed=540 + Q)
    _, k, v, lens_np, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_causal(workloads.np_storage(q4), k, v, lens_np,
                                        block_table=bt, page_size=ps)
    wd = w.to("cuda")
    B = len(lens)
    for S in (1, 7):
        o, l = _run_sched(wd, w, S, fd.FD_SCHEDULE_HEAD_GROUPS, q=q4.cuda())
        mw = workloads.Workload("mt", q4.reshape(B * Q, Hq, d), w.k, w.v, w.seq_lens)
        check(mw, o.cpu().double().numpy().reshape(B * Q, Hq, d),
              l.cpu().double().numpy().reshape(B * Q, Hq),
              ref_o.reshape(B * Q, Hq, d), ref_l.reshape(B * Q, Hq))


def test_head_groups_bad_page_is_flagged_and_contained():
    """A used table entry outside the pool in row 0: flagged, every output finite, and
    row 1 (a clean table) still equals the oracle."""
    lens = [100, 90]
    w = workloads.paged_case(2, 32, 8, 128, 16, 8, lens, seed=550, out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    bt = wd.block_table.clone()
    bt[0, 2] = 10_000
    fd.set_path(fd.FD_PATH_MMA)
    fd.set_schedule(fd.FD_SCHEDULE_HEAD_GROUPS)
    ws = torch.zeros(fd.workspace_size(2, 32, 8, 128, 3), dtype=torch.uint8, device="cuda")
    o, l = fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, bt, 16, 3, workspace=ws,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 2            # FD_DEVFLAG_PAGE
    assert torch.isfinite(o).all() and torch.isfinite(l).all()
    check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l,
          rows=np.arange(32, 64))


def test_head_groups_partials_and_merge():
    """fd_decode_partial under head groups, then fd_merge_partials, equals the one-call
    decode (both merge with the same kernel)."""
    w = workloads.paged_case(3, 16, 4, 128, 32, 64, [2048, 700, 33], seed=560,
                             out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    fd.set_schedule(fd.FD_SCHEDULE_HEAD_GROUPS)
    S = 9
    ws = torch.zeros(fd.workspace_size(3, 16, 4, 128, S), dtype=torch.uint8, device="cuda")
    fd.decode_partial(wd.q, wd.k, wd.v, wd.seq_lens, ws, wd.block_table, 32, S)
    lp, op = fd.workspace_partials(ws, 3, 16, 128, S)
    o2, l2 = fd.merge_partials(lp, op, out_dtype=torch.float32)
    o1, l1 = _run_sched(wd, w, S, fd.FD_SCHEDULE_HEAD_GROUPS)
    torch.cuda.synchronize()
    check(w, o2.cpu().double().numpy(), l2.cpu().double().numpy(), ref_o, ref_l)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("ps,Hkv", [(16, 2), (8, 4), (0, 6)])
def test_head_groups_fall_back_to_grid(ps, Hkv):
    """Where head groups do not apply (8-token pages, Hkv not a multiple of 4), the
    head-group setting runs the grid schedule: identical results."""
    lens = [700, 1, 129]
    if ps:
        w = workloads.paged_case(3, Hkv * 4, Hkv, 128, ps, -(-1024 // ps), lens, seed=570 + ps,
                                 out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(3, Hkv * 4, Hkv, 128, 1024, lens, seed=570,
                                      out_dtype=torch.float32)
    wd = w.to("cuda")
    oh, lh = _run_sched(wd, w, 5, fd.FD_SCHEDULE_HEAD_GROUPS)
    og, lg = _run_sched(wd, w, 5, fd.FD_SCHEDULE_GRID)
    assert torch.equal(oh, og) and torch.equal(lh, lg)
