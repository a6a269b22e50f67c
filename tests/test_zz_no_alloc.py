"""fd_decode_attention_noalloc, the entry point for callers that cannot allocate device
memory while they run a step (a plugin inside a framework that owns all device memory,
a loop whose memory budget is fixed at start-up).  It keeps its split partials in the
library's built-in scratch instead of a caller workspace.

Checked here through the C ABI, each output against the fp64 oracle and against
fd_decode_attention (caller workspace) on the same inputs, within the parity tolerances
  out: |got - ref| <= 4e-3 + 8e-3 |ref|     lse: |got - ref| <= 1e-4 + 1e-5 |ref|
  * the first call of the process runs on a non-blocking stream with the persistent
    schedule, whose queue words live in the scratch header: the one-time zero-fill must
    be complete before that call's kernels start;
  * two calls in a row on different inputs (what the first left in the shared scratch
    must not leak into the second);
  * multi-token decode (q [B, Q, Hq, d]) on the tcgen05 kernel;
  * a wide group sized with the split count the call itself uses (it fits);
  * requests larger than the scratch, single- and multi-token, refused with
    FD_ERR_UNSUPPORTED.
The file is named so that pytest collects it after every other test file; its first
test is the first no-allocation call of the process whether it runs alone or last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")
from decode_attention_05_gb300._binding import tensor_desc  # noqa: E402

FD_ERR_UNSUPPORTED = 2


@pytest.fixture(autouse=True)
def _restore_settings():
    yield
    if torch.cuda.is_available():
        fd.set_path(fd.FD_PATH_AUTO)
        fd.set_merge_mode(fd.FD_MERGE_KERNEL)
        fd.set_schedule(fd.FD_SCHEDULE_AUTO)


def _call_noalloc(w, q, out, lse, num_splits, stream=None):
    L = fd.lib()
    dq, dk, dv, dbt, do = (tensor_desc(q), tensor_desc(w.k), tensor_desc(w.v),
                           tensor_desc(w.block_table), tensor_desc(out))
    s = stream if stream is not None else torch.cuda.current_stream()
    return L.fd_decode_attention_noalloc(
        ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), w.seq_lens.data_ptr(),
        None if dbt is None else ctypes.byref(dbt), w.page_size, num_splits,
        ctypes.byref(do), lse.data_ptr(), s.cuda_stream or None)


def _oracle(w_cpu, q4=None):
    q, k, v, lens, bt, ps = w_cpu.oracle_arrays()
    if q4 is None:
        return oracle.decode(q, k, v, lens, block_table=bt, page_size=ps)
    return oracle.decode_causal(workloads.np_storage(q4), k, v, lens, block_table=bt,
                                page_size=ps)


def _check(got_o, got_l, ref_o, ref_l):
    go = got_o.double().cpu().numpy().reshape(ref_o.shape)
    gl = got_l.double().cpu().numpy().reshape(ref_l.shape)
    assert not np.isnan(go).any() and not np.isnan(gl).any()
    err = np.abs(go - ref_o)
    assert (err <= 4e-3 + 8e-3 * np.abs(ref_o)).all(), "out max err %.3g" % err.max()
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(gl), empty)
    assert (go[empty] == 0).all()
    lerr = np.abs(gl[~empty] - ref_l[~empty])
    assert (lerr <= 1e-4 + 1e-5 * np.abs(ref_l[~empty])).all(), "lse max err %.3g" % lerr.max()


def _noalloc_vs_both(w_cpu, S, q4=None, stream=None):
    """One no-allocation call, checked against the oracle and fd_decode_attention."""
    w = w_cpu.to("cuda")
    q = w.q if q4 is None else q4.cuda()
    ref_o, ref_l = _oracle(w_cpu, q4)
    out = torch.full(tuple(q.shape), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full(tuple(q.shape[:-1]), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    st = _call_noalloc(w, q, out, lse, S, stream)
    assert st == 0, fd.lib().fd_last_error()
    torch.cuda.synchronize()
    _check(out, lse, ref_o, ref_l)
    wo, wl = fd.decode_attention(q, w.k, w.v, w.seq_lens, w.block_table, w.page_size, S,
                                 out_dtype=torch.float32)
    torch.cuda.synchronize()
    _check(out, lse, wo.double().cpu().numpy().reshape(ref_o.shape),
           wl.double().cpu().numpy().reshape(ref_l.shape))


def test_noalloc_first_call_on_a_non_blocking_stream():
    torch.cuda.set_device(0)
    fd.set_schedule(fd.FD_SCHEDULE_PERSISTENT)
    w = workloads.contiguous_case(3, 32, 4, 128, 4096, [4096, 1, 2500], seed=40,
                                  out_dtype=torch.float32)
    assert fd.partial_kernel_name(torch.bfloat16, torch.bfloat16, 128, 4, 0,
                                  rows=8) == "fd_partial_persist_kernel"
    side = torch.cuda.Stream()                  # created non-blocking by torch
    with torch.cuda.stream(side):
        _noalloc_vs_both(w, 16, stream=side)
    # A second persistent call finds the queue words the first one put back.
    _noalloc_vs_both(workloads.contiguous_case(2, 16, 2, 128, 2048, [2048, 999], seed=44,
                                               out_dtype=torch.float32), 8, stream=side)


def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls_in_a_row():
    fd.set_path(fd.FD_PATH_AUTO)
    # Call 1: a ragged paged GQA batch; call 2: a different contiguous batch, so that
    # anything the first call left in the shared scratch would show up in the second.
    cases = [
        (workloads.paged_case(4, 32, 4, 128, 16, 128, [1, 37, 900, 2048], seed=41,
                              out_dtype=torch.float32), 6),
        (workloads.contiguous_case(2, 16, 2, 128, 3000, [3000, 17], seed=42,
                                   out_dtype=torch.float32), 0),
    ]
    for w_cpu, S in cases:
        _noalloc_vs_both(w_cpu, S)


def test_noalloc_multi_token_decode():
    # 4 query tokens x G = 8 heads = 32 rows per kv head: the tcgen05 kernel.
    w = workloads.contiguous_case(2, 16, 2, 128, 2048, [2048, 301], seed=45,
                                  out_dtype=torch.float32)
    q4 = workloads.multi_token_queries(2, 4, 16, 128, seed=46)
    _noalloc_vs_both(w, 0, q4=q4)
    _noalloc_vs_both(w, 5, q4=q4)


def test_noalloc_sizes_wide_groups_with_the_split_count_they_use():
    # 64 query heads on one kv head over 128K keys: the tcgen05 kernel plans one CTA's
    # worth of splits per SM, whose partials fit the scratch (the single-token count
    # would not).
    w = workloads.contiguous_case(1, 64, 1, 128, 131072, seed=47, poison_tail=False,
                                  out_dtype=torch.float32)
    S = fd.resolve_num_splits(1, 64, 1, 128, 131072, 0)
    assert fd.workspace_size(1, 64, 1, 128, S) <= 8 << 20
    _noalloc_vs_both(w, 0)


def test_noalloc_refuses_requests_beyond_its_scratch():
    # B * Hq * S * (d + 1) * 4 bytes of partials: 64 * 1024 * 129 * 4 > 8 MiB.
    w = workloads.contiguous_case(1, 64, 8, 128, 2048, seed=43, poison_tail=False).to("cuda")
    out = torch.empty(1, 64, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 64, dtype=torch.float32, device="cuda")
    assert _call_noalloc(w, w.q, out, lse, 1024) == FD_ERR_UNSUPPORTED
    assert b"scratch" in fd.lib().fd_last_error()
    # Multi-token: 8 query tokens x 64 heads x 64 splits x 129 floats = 16.9 MB.
    q4 = workloads.multi_token_queries(1, 8, 64, 128, seed=48).cuda()
    out4 = torch.empty(1, 8, 64, 128, dtype=torch.bfloat16, device="cuda")
    lse4 = torch.empty(1, 8, 64, dtype=torch.float32, device="cuda")
    assert _call_noalloc(w, q4, out4, lse4, 64) == FD_ERR_UNSUPPORTED
    assert b"scratch" in fd.lib().fd_last_error()
    torch.cuda.synchronize()
