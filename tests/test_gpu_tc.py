"""GPU parity of the tcgen05 kernel (tensor-memory accumulators), the automatic choice
for groups of 17 to 64 query rows per kv head with bf16 q/K/V at d = 128, and available
for any group size through FD_PATH_TCGEN05.  Checked element by element against the
fp64 oracle with the bf16 tolerance of test_gpu_parity, and against the mma.sync wide
kernel on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import check, ref_for, run

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")


@pytest.fixture(autouse=True)
def _restore_settings():
    yield
    if torch.cuda.is_available():
        fd.set_path(fd.FD_PATH_AUTO)
        fd.set_merge_mode(fd.FD_MERGE_KERNEL)
        fd.set_schedule(fd.FD_SCHEDULE_AUTO)


def multi_token(Q, G, Hkv, lens, ps, seed, cap=2048):
    Hq = Hkv * G
    if ps:
        w = workloads.paged_case(len(lens), Hq, Hkv, 128, ps, -(-cap // ps), lens, seed=seed,
                                 extra_pages=2, out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(len(lens), Hq, Hkv, 128, cap, lens, seed=seed,
                                      out_dtype=torch.float32)
    q4 = workloads.multi_token_queries(len(lens), Q, Hq, 128, seed=seed + 1)
    _, k, v, lens_np, bt, pg = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_causal(workloads.np_storage(q4), k, v, lens_np,
                                        block_table=bt, page_size=pg)
    return w, q4, ref_o, ref_l


def decode(w, q4, S):
    B, Q, Hq, d = q4.shape
    wd = w.to("cuda")
    ws = torch.zeros(fd.workspace_size(B, Q * Hq, w.Hkv, d, S), dtype=torch.uint8, device="cuda")
    o, l = fd.decode_attention(q4.cuda(), wd.k, wd.v, wd.seq_lens, wd.block_table, w.page_size,
                               S, workspace=ws, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    return (o.cpu().double().numpy().reshape(B * Q, Hq, d),
            l.cpu().double().numpy().reshape(B * Q, Hq))


@pytest.mark.parametrize("merge", [0, 1])        # merge kernel, merge inside the partial pass
@pytest.mark.parametrize("Q,G,Hkv,ps", [
    (3, 8, 2, 0), (4, 8, 2, 0), (8, 8, 1, 0), (2, 16, 2, 16), (4, 16, 1, 32), (1, 32, 2, 0),
    (1, 64, 1, 64), (5, 4, 2, 128), (3, 16, 1, 0), (8, 8, 2, 16), (6, 4, 2, 0)])
def test_tc_wide_groups(Q, G, Hkv, ps, merge):
    """17 to 64 rows per kv head (the automatic choice there): ragged rows, rows shorter
    than Q (keyless queries), NaN tails, tile and page boundaries, several split
    counts."""
    fd.set_merge_mode(merge)
    fd.set_path(fd.FD_PATH_TCGEN05)
    lens = [1, max(Q - 1, 1), 64, 65, 333, 1500, 2048]
    w, q4, ref_o, ref_l = multi_token(Q, G, Hkv, lens, ps, seed=1200 + Q * 13 + G + ps)
    assert fd.partial_kernel_name(torch.bfloat16, torch.bfloat16, 128, Hkv, ps,
                                  rows=Q * G) == "fd_partial_tc_kernel"
    B, Hq = len(lens), Hkv * G
    mw = workloads.Workload("tc", q4.reshape(B * Q, Hq, 128), w.k, w.v, w.seq_lens)
    for S in (1, 3, 16, 64):
        o, l = decode(w, q4, S)
        check(mw, o, l, ref_o.reshape(B * Q, Hq, 128), ref_l.reshape(B * Q, Hq))


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("ps", [0, 16, 256])
def test_tc_single_token_any_group(G, ps):
    """The explicit tcgen05 path on single-token decode for every group size."""
    fd.set_path(fd.FD_PATH_TCGEN05)
    lens = [0, 1, 63, 64, 65, 700, 2048]
    if ps:
        w = workloads.paged_case(len(lens), 4 * G, 4, 128, ps, -(-2048 // ps), lens,
                                 seed=1300 + G + ps, extra_pages=2, out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(len(lens), 4 * G, 4, 128, 2048, lens, seed=1300 + G,
                                      out_dtype=torch.float32)
    assert fd.partial_kernel_name(torch.bfloat16, torch.bfloat16, 128, 4, ps, rows=G) == \
        "fd_partial_tc_kernel"
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    for S in (1, 5, 32):
        o, l, _, _ = run(w, num_splits=S, path=fd.FD_PATH_TCGEN05, wd=wd)
        check(w, o, l, ref_o, ref_l)


def test_tc_matches_mma_wide_kernel():
    """The same 64-row case through both tensor-core kernels: both within the oracle's
    tolerance, and close to each other (P is rounded to bf16 by both, against running
    maxima that may differ)."""
    Q, G, Hkv = 8, 8, 2
    lens = [4096, 3000, 17]
    w, q4, ref_o, ref_l = multi_token(Q, G, Hkv, lens, 0, seed=1400, cap=4096)
    B, Hq = len(lens), Hkv * G
    mw = workloads.Workload("tc", q4.reshape(B * Q, Hq, 128), w.k, w.v, w.seq_lens)
    outs = []
    for path in (fd.FD_PATH_TCGEN05, fd.FD_PATH_MMA):
        fd.set_path(path)
        o, l = decode(w, q4, 9)
        check(mw, o, l, ref_o.reshape(B * Q, Hq, 128), ref_l.reshape(B * Q, Hq))
        outs.append((o, l))
    assert np.abs(outs[0][0] - outs[1][0]).max() < 8e-3
    assert np.abs(outs[0][1] - outs[1][1]).max() < 1e-4


def test_tc_rescale_on_growing_scores():
    """Scores that grow along the sequence force the running max up many times inside
    one split (each rescale of O in tensor memory): a row of keys k_t = (t / 64) e_0 and
    q = e_0 * 8 sqrt(d), so the score rises by 8 every 64 tokens."""
    L = 4096
    q = torch.zeros(1, 32, 128)
    q[0, :, 0] = 8.0 * 128 ** 0.5 / 64.0 * torch.linspace(0.5, 1.0, 32)
    k = torch.randn(1, 1, L, 128, generator=torch.Generator().manual_seed(3)) * 0.01
    k[0, 0, :, 0] = torch.arange(L, dtype=torch.float32) / 64.0 * 8.0
    v = torch.randn(1, 1, L, 128, generator=torch.Generator().manual_seed(4))
    w = workloads.Workload("grow", q.bfloat16(), k.bfloat16(), v.bfloat16(),
                           torch.tensor([L], dtype=torch.int32), out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    for S in (1, 2):
        o, l, _, _ = run(w, num_splits=S, path=fd.FD_PATH_TCGEN05)
        check(w, o, l, ref_o, ref_l)


def test_tc_refuses_what_it_does_not_take():
    fd.set_path(fd.FD_PATH_TCGEN05)
    seq = torch.tensor([64], dtype=torch.int32, device="cuda")
    for d, dt in ((64, torch.bfloat16), (128, torch.float32)):
        q = torch.zeros(1, 8, d, dtype=dt, device="cuda")
        k = torch.zeros(1, 1, 64, d, dtype=dt, device="cuda")
        with pytest.raises(fd.FdError):
            fd.decode_attention(q, k, k, seq, num_splits=1)


@pytest.mark.parametrize("Q,G", [(8, 8), (4, 8), (1, 8)])
def test_tc_long_splits(Q, G):
    """Hundreds of tiles per split (32K tokens, one or four splits): the pipeline's
    barriers cycle through many phases, with the softmax warps free to run ahead of the
    issuing thread; any lost phase would trip a bounded wait and raise the device flag."""
    fd.set_path(fd.FD_PATH_TCGEN05)
    lens = [32768, 30001]
    w, q4, ref_o, ref_l = multi_token(Q, G, 1, lens, 0, seed=1500 + Q, cap=32768)
    B, Hq = len(lens), G
    mw = workloads.Workload("tc", q4.reshape(B * Q, Hq, 128), w.k, w.v, w.seq_lens)
    for S in (1, 4):
        o, l = decode(w, q4, S)
        check(mw, o, l, ref_o.reshape(B * Q, Hq, 128), ref_l.reshape(B * Q, Hq))


def test_tc_default_split_count():
    """num_splits = 0 on a wide group: one CTA's worth of splits per SM, never more than
    the single-token plan (so workspaces sized by the single-token count suffice), and
    the call with the planned count matches the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    one = fd.resolve_num_splits(1, 64, 8, 128, 131072, 0)
    wide = fd.resolve_num_splits(1, 64, 8, 128, 131072, 0, Q=8)
    assert wide == min(one, max(1, sms // 8)), (one, wide)
    assert fd.resolve_num_splits(1, 64, 8, 128, 131072, 0, Q=2) == one      # 16 rows
    assert fd.resolve_num_splits(1, 64, 8, 128, 131072, 7, Q=8) == 7        # explicit
    lens = [3000, 2047, 5]
    w, q4, ref_o, ref_l = multi_token(4, 8, 2, lens, 0, seed=1600, cap=3072)
    wd = w.to("cuda")
    o, l = fd.decode_attention(q4.cuda(), wd.k, wd.v, wd.seq_lens, out_dtype=torch.float32)
    torch.cuda.synchronize()
    B, Hq = len(lens), 16
    mw = workloads.Workload("tc", q4.reshape(B * 4, Hq, 128), w.k, w.v, w.seq_lens)
    check(mw, o.cpu().double().numpy().reshape(B * 4, Hq, 128),
          l.cpu().double().numpy().reshape(B * 4, Hq), ref_o.reshape(B * 4, Hq, 128),
          ref_l.reshape(B * 4, Hq))


@pytest.mark.parametrize("ps", [16, 64])
def test_tc_bad_page_is_flagged_and_contained(ps):
    """A used table entry outside the pool in row 0 (several pages per tile at 16-token
    pages, one page per tile at 64): flagged, every output finite, and row 1 (a clean
    table) still equals the causal oracle."""
    Q, G, Hkv = 4, 8, 2
    lens = [300, 290]
    w, q4, ref_o, ref_l = multi_token(Q, G, Hkv, lens, ps, seed=1700 + ps, cap=512)
    wd = w.to("cuda")
    bt = wd.block_table.clone()
    bt[0, 1] = 10_000
    fd.set_path(fd.FD_PATH_TCGEN05)
    B, Hq = len(lens), Hkv * G
    ws = torch.zeros(fd.workspace_size(B, Q * Hq, Hkv, 128, 3), dtype=torch.uint8,
                     device="cuda")
    o, l = fd.decode_attention(q4.cuda(), wd.k, wd.v, wd.seq_lens, bt, ps, 3, workspace=ws,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 2            # FD_DEVFLAG_PAGE
    assert torch.isfinite(o).all() and torch.isfinite(l).all()
    mw = workloads.Workload("tc", q4.reshape(B * Q, Hq, 128), w.k, w.v, w.seq_lens)
    check(mw, o.cpu().double().numpy().reshape(B * Q, Hq, 128),
          l.cpu().double().numpy().reshape(B * Q, Hq), ref_o.reshape(B * Q, Hq, 128),
          ref_l.reshape(B * Q, Hq), rows=np.arange(Q * Hq, 2 * Q * Hq))
