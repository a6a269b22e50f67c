"""The failure path on the GPU, without a GPU fault: an in-kernel wait that nothing
completes must give up after its limit, raise FD_DEVFLAG_TIMEOUT in the workspace, and
leave the context usable for the next decode."""
import time

import pytest
import torch

import workloads
from test_gpu_parity import check, ref_for

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")


def test_wait_that_runs_out_reports_and_context_survives():
    ws = torch.zeros(fd.workspace_size(2, 16, 4, 128, 4), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    fd.selftest_bounded_wait(ws, limit_us=50_000)          # 50 ms
    flags = fd.read_device_error(ws)                        # synchronises, then clears
    elapsed = time.perf_counter() - t0
    assert flags == 4                                       # FD_DEVFLAG_TIMEOUT
    assert 0.04 <= elapsed < 5.0                            # it waited, then it returned
    assert fd.read_device_error(ws) == 0                    # cleared by the read
    # The same context and workspace still decode correctly.
    w = workloads.contiguous_case(2, 16, 4, 128, 2000, [2000, 333], seed=801,
                                  out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    o, l = fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, num_splits=4, workspace=ws,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


def test_selftest_argument_checks():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fd.FdError):
        fd.selftest_bounded_wait(ws, limit_us=0)
    with pytest.raises(fd.FdError):
        fd.selftest_bounded_wait(ws, limit_us=3_000_000)


# ------------------------------------------------------------------ the kernels' own waits
# fd_selftest_stalled_decode: the producer of CTA (0, 0, 0) stops before one of its tiles,
# so that CTA's consumers wait on a stage nothing fills.  Their bounded waits (2 s) must
# give up, flag FD_DEVFLAG_TIMEOUT, drain what is in flight and end the CTA normally; the
# same context and workspace must then decode correctly.  One case per kernel family.

def _stalled_case(kind):
    Q = 1
    opts = None
    if kind == "mma":
        w = workloads.contiguous_case(2, 16, 2, 128, 4096, [4096, 2000], seed=811,
                                      out_dtype=torch.float32)
        S, stall = 4, 1
    elif kind == "mma_fused":
        w = workloads.contiguous_case(2, 16, 2, 128, 4096, [4096, 2000], seed=812,
                                      out_dtype=torch.float32)
        S, stall = 4, 2
        opts = fd.options(merge_mode=fd.FD_MERGE_IN_KERNEL)
    elif kind == "heads":
        w = workloads.paged_case(2, 16, 4, 128, 16, 256, [4096, 1000], seed=813,
                                 out_dtype=torch.float32)
        S, stall = 4, 1
    elif kind == "simt":
        w = workloads.contiguous_case(2, 16, 2, 128, 4096, [4096, 2000], seed=814,
                                      out_dtype=torch.float32)
        S, stall = 4, 1
        opts = fd.options(path=fd.FD_PATH_SIMT)
    elif kind in ("tc", "tc_shared"):
        w = workloads.contiguous_case(2, 16, 2, 128, 4096, [4096, 3000], seed=815,
                                      out_dtype=torch.float32)
        Q, S, stall = 4, 3, 2
        opts = fd.options(schedule=fd.FD_SCHEDULE_TAIL_SHARING) if kind == "tc_shared" else None
    elif kind == "wide":                     # d = 64, 32 rows per kv head
        w = workloads.contiguous_case(2, 16, 2, 64, 4096, [4096, 2000], seed=816,
                                      out_dtype=torch.float32)
        Q, S, stall = 4, 4, 1
    elif kind == "persist":
        w = workloads.contiguous_case(2, 16, 2, 128, 4096, [4096, 2000], seed=817,
                                      out_dtype=torch.float32)
        S, stall = 4, 3
        opts = fd.options(path=fd.FD_PATH_MMA, schedule=fd.FD_SCHEDULE_PERSISTENT)
    elif kind == "heads_persist":
        w = workloads.paged_case(2, 16, 4, 128, 16, 256, [4096, 1000], seed=818,
                                 out_dtype=torch.float32)
        S, stall = 4, 5
        opts = fd.options(schedule=fd.FD_SCHEDULE_PERSISTENT)
    elif kind == "heads_contiguous":
        w = workloads.contiguous_case(2, 16, 4, 128, 4096, [4096, 1000], seed=819,
                                      out_dtype=torch.float32)
        S, stall = 4, 1
        opts = fd.options(schedule=fd.FD_SCHEDULE_HEAD_GROUPS)
    elif kind == "wide_persist":             # 32 rows per kv head, persistent
        w = workloads.contiguous_case(2, 16, 2, 128, 4096, [4096, 2000], seed=822,
                                      out_dtype=torch.float32)
        Q, S, stall = 4, 4, 2
        opts = fd.options(path=fd.FD_PATH_MMA, schedule=fd.FD_SCHEDULE_PERSISTENT)
    elif kind == "direct":                   # one split: out written by the partial pass
        w = workloads.contiguous_case(2, 16, 2, 128, 4096, [4096, 2000], seed=821,
                                      out_dtype=torch.float32)
        S, stall = 1, 2
    else:
        raise ValueError(kind)
    return w, Q, S, stall, opts


@pytest.mark.parametrize("kind", ["mma", "mma_fused", "heads", "simt", "tc", "tc_shared", "wide",
                                  "persist", "heads_persist", "heads_contiguous", "direct",
                                  "wide_persist"])
def test_real_kernel_wait_runs_out_and_context_survives(kind):
    import numpy as np
    import oracle
    w, Q, S, stall, opts = _stalled_case(kind)
    wd = w.to("cuda")
    q = wd.q
    if Q > 1:
        q = workloads.multi_token_queries(w.B, Q, w.Hq, w.d, seed=820).cuda()
    expected = {"mma": "fd_partial_mma_kernel", "mma_fused": "fd_partial_mma_kernel",
                "heads": "fd_partial_heads_kernel", "simt": "fd_partial_simt_kernel",
                "tc": "fd_partial_tc_kernel", "tc_shared": "fd_partial_tc_kernel",
                "wide": "fd_partial_wide_kernel", "persist": "fd_partial_persist_kernel",
                "heads_persist": "fd_partial_heads_persist_kernel",
                "heads_contiguous": "fd_partial_heads_kernel",
                "wide_persist": "fd_partial_wide_persist_kernel",
                "direct": "fd_partial_mma_kernel"}[kind]
    assert fd.partial_kernel_name_for(torch.bfloat16, torch.bfloat16, w.B, Q, w.Hq, w.Hkv, w.d,
                                      w.page_size, w.L_cap, S, options=opts) == expected
    ws = torch.zeros(fd.workspace_size(w.B, Q * w.Hq, w.Hkv, w.d, S), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(tuple(q.shape), dtype=torch.float32, device="cuda")
    lse = torch.empty(tuple(q.shape[:-1]), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    fd.selftest_stalled_decode(q, wd.k, wd.v, wd.seq_lens, ws, stall, out, lse,
                               block_table=wd.block_table, page_size=w.page_size,
                               num_splits=S, options=opts)
    flags = fd.read_device_error(ws)                        # synchronises, then clears
    elapsed = time.perf_counter() - t0
    assert flags == 4                                       # FD_DEVFLAG_TIMEOUT
    assert 1.5 <= elapsed < 60.0                            # the 2 s waits ran out, then ended
    # The same context and workspace decode correctly afterwards.
    o, l = fd.decode_attention(q, wd.k, wd.v, wd.seq_lens, wd.block_table, w.page_size, S,
                               workspace=ws, out_dtype=torch.float32, options=opts)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    qn, k, v, lens, bt, ps = w.oracle_arrays()
    if Q > 1:
        ref_o, ref_l = oracle.decode_causal(workloads.np_storage(q.cpu()), k, v, lens,
                                            block_table=bt, page_size=ps)
        o = o.reshape(w.B * Q, w.Hq, w.d)
        l = l.reshape(w.B * Q, w.Hq)
        ref_o = ref_o.reshape(w.B * Q, w.Hq, w.d)
        ref_l = ref_l.reshape(w.B * Q, w.Hq)
    else:
        ref_o, ref_l = oracle.decode(qn, k, v, lens, block_table=bt, page_size=ps)
    check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


def test_stalled_decode_argument_check():
    w = workloads.contiguous_case(1, 8, 1, 128, 256, seed=830).to("cuda")
    ws = torch.zeros(fd.workspace_size(1, 8, 1, 128, 2), dtype=torch.uint8, device="cuda")
    out = torch.empty(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 8, dtype=torch.float32, device="cuda")
    with pytest.raises(fd.FdError):
        fd.selftest_stalled_decode(w.q, w.k, w.v, w.seq_lens, ws, -1, out, lse, num_splits=2)
