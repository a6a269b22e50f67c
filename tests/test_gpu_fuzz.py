"""Seeded random parity cases: shapes, layouts, lengths, split counts, query tokens,
cache formats and schedules drawn together, each checked element by element against
the fp64 oracle with the tolerances of test_gpu_parity.  Sizes stay small, so the
oracle finishes each case in about a second at most; every case prints its draw when
it fails, and the seed of case i is 7000 + i (medium cases: i = 100000 + j)."""
import random

import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import check

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")

N_CASES = 160


@pytest.fixture(autouse=True)
def _restore_settings():
    yield
    if torch.cuda.is_available():
        fd.set_schedule(fd.FD_SCHEDULE_AUTO)
        fd.set_path(fd.FD_PATH_AUTO)
        fd.set_merge_mode(fd.FD_MERGE_KERNEL)


def draw(i, medium=False):
    r = random.Random(7000 + i)
    d = r.choice([64, 128, 128])
    fp8 = d == 128 and r.random() < 0.2
    f32 = not fp8 and r.random() < 0.15
    Q = r.choice([1, 1, 1, 2, 3, 4, 8])
    # above 16 rows: the tensor-core paths only (bf16 up to 64 rows, FP8 up to 32)
    max_rows = 16 if f32 else (32 if fp8 else 64)
    G = r.choice([g for g in (1, 2, 4, 8, 16, 32, 64) if Q * g <= max_rows])
    Hkv = r.choice([1, 2, 3, 4, 8])
    B = r.randint(1, 5)
    paged = r.random() < 0.5
    ps = r.choice([8, 16, 32, 64, 128]) if paged else 0
    cap = r.choice([64, 200, 1000, 2048, 3000])
    if medium:                      # multi-wave grids, page-table windows past 32 pages
        cap = r.choice([8192, 20000, 32768])
        B = r.randint(1, 8)
    if paged:
        cap = -(-cap // ps) * ps
    lens = [r.choice([0, 1, r.randint(1, cap), cap, r.randint(cap // 2, cap)]) for _ in range(B)]
    S = r.choice([0, 1, 2, 5, 16, 64] + ([128, 300, 512] if medium else []))
    sched = r.choice([fd.FD_SCHEDULE_AUTO, fd.FD_SCHEDULE_GRID, fd.FD_SCHEDULE_PERSISTENT,
                      fd.FD_SCHEDULE_HEAD_GROUPS, fd.FD_SCHEDULE_TAIL_SHARING])
    merge = r.choice([fd.FD_MERGE_KERNEL, fd.FD_MERGE_KERNEL, fd.FD_MERGE_IN_KERNEL])
    if f32:     # the tensor-core path takes up to 8 f32 rows
        path = fd.FD_PATH_MMA if Q * G <= 8 and r.random() < 0.7 else fd.FD_PATH_SIMT
    elif not fp8 and Q * G <= 16 and r.random() < 0.2:
        path = fd.FD_PATH_SIMT
    else:       # AUTO runs the tcgen05 kernel for bf16 groups above 16 rows at d = 128
        path = fd.FD_PATH_AUTO if r.random() < 0.5 else fd.FD_PATH_MMA
    return dict(d=d, fp8=fp8, f32=f32, Q=Q, G=G, Hkv=Hkv, B=B, ps=ps, cap=cap, lens=lens, S=S,
                sched=sched, merge=merge, path=path)


N_MEDIUM = 40


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(i):
    run_case(i, draw(i))


@pytest.mark.parametrize("i", range(N_MEDIUM))
def test_random_medium_case(i):
    """Longer caches (8K to 32K tokens), more rows and up to 512 splits."""
    run_case(100000 + i, draw(100000 + i, medium=True))


def run_case(i, c):
    dtype = torch.float32 if c["f32"] else torch.bfloat16
    Hq = c["Hkv"] * c["G"]
    if c["ps"]:
        w = workloads.paged_case(c["B"], Hq, c["Hkv"], c["d"], c["ps"], c["cap"] // c["ps"],
                                 c["lens"], seed=8000 + i, dtype=dtype, extra_pages=1,
                                 out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(c["B"], Hq, c["Hkv"], c["d"], c["cap"], c["lens"],
                                      seed=8000 + i, dtype=dtype, out_dtype=torch.float32)
    fd.set_schedule(c["sched"])
    fd.set_merge_mode(c["merge"])
    fd.set_path(c["path"])
    Q, B, d = c["Q"], c["B"], c["d"]
    q4 = workloads.multi_token_queries(B, Q, Hq, d, seed=9000 + i, dtype=dtype)
    _, k, v, lens, bt, ps = w.oracle_arrays()
    qs = workloads.np_storage(q4)
    wd = w.to("cuda")
    qd = q4.cuda() if Q > 1 else q4[:, 0].contiguous().cuda()
    S_res = fd.resolve_num_splits(B, Hq, c["Hkv"], d, w.L_cap, c["S"])
    ws = torch.zeros(fd.workspace_size(B, Q * Hq, c["Hkv"], d, S_res), dtype=torch.uint8,
                     device="cuda")
    if c["fp8"]:
        kc, vc, ks, vs = workloads.fp8_quantize(w, power_of_two_scales=Q > 1)
        if Q == 1:
            ref_o, ref_l = oracle.decode_kv8(qs[:, 0], kc.view(torch.uint8).numpy(),
                                             vc.view(torch.uint8).numpy(), ks.numpy(),
                                             vs.numpy(), lens, block_table=bt, page_size=ps)
        else:   # power-of-two scales: the dequantised cache is exact in fp32
            deq = lambda t, s: (t.float() * s.view(1, -1, 1, 1)).numpy()
            ref_o, ref_l = oracle.decode_causal(q4.float().numpy(), deq(kc, ks), deq(vc, vs),
                                                lens, block_table=bt, page_size=ps)
        o, l = fd.decode_attention_fp8kv(qd, kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda(),
                                         wd.seq_lens, wd.block_table, w.page_size, c["S"],
                                         workspace=ws, out_dtype=torch.float32)
    else:
        if Q == 1:
            ref_o, ref_l = oracle.decode(qs[:, 0], k, v, lens, block_table=bt, page_size=ps)
        else:
            ref_o, ref_l = oracle.decode_causal(qs, k, v, lens, block_table=bt, page_size=ps)
        o, l = fd.decode_attention(qd, wd.k, wd.v, wd.seq_lens, wd.block_table, w.page_size,
                                   c["S"], workspace=ws, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0, c
    mw = workloads.Workload("fuzz", q4.reshape(B * Q, Hq, d), w.k, w.v, w.seq_lens)
    try:
        check(mw, o.cpu().double().numpy().reshape(B * Q, Hq, d),
              l.cpu().double().numpy().reshape(B * Q, Hq),
              np.asarray(ref_o).reshape(B * Q, Hq, d), np.asarray(ref_l).reshape(B * Q, Hq))
    except AssertionError as e:
        raise AssertionError("case %d %r: %s" % (i, c, e)) from None
