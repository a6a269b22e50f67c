"""fd_decode_attention_noalloc, the entry point for callers that cannot allocate device
memory while they run a step (a plugin inside a framework that owns all device memory,
a loop whose memory budget is fixed at start-up).  It keeps its split partials in the
library's built-in scratch instead of a caller workspace.

Checked here through the C ABI: two calls in a row, on different inputs, each agree
with fd_decode_attention (caller workspace) within the parity tolerances
  out: |got - ref| <= 4e-3 + 8e-3 |ref|     lse: |got - ref| <= 1e-4 + 1e-5 |ref|
and a request larger than the scratch is refused with FD_ERR_UNSUPPORTED.  The file
is named so that pytest collects it after every other test file.
"""
import ctypes

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")
from decode_attention_05_gb300._binding import tensor_desc  # noqa: E402

FD_ERR_UNSUPPORTED = 2


def _call_noalloc(w, out, lse, num_splits):
    L = fd.lib()
    dq, dk, dv, dbt, do = (tensor_desc(w.q), tensor_desc(w.k), tensor_desc(w.v),
                           tensor_desc(w.block_table), tensor_desc(out))
    return L.fd_decode_attention_noalloc(
        ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), w.seq_lens.data_ptr(),
        None if dbt is None else ctypes.byref(dbt), w.page_size, num_splits,
        ctypes.byref(do), lse.data_ptr(), torch.cuda.current_stream().cuda_stream or None)


def _compare(got_o, got_l, ref_o, ref_l):
    go, ro = got_o.double(), ref_o.double()
    assert torch.isfinite(go).all()
    assert ((go - ro).abs() <= 4e-3 + 8e-3 * ro.abs()).all()
    empty = torch.isneginf(ref_l)
    assert torch.equal(torch.isneginf(got_l), empty)
    fin = ~empty
    gl, rl = got_l[fin].double(), ref_l[fin].double()
    assert ((gl - rl).abs() <= 1e-4 + 1e-5 * rl.abs()).all()


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    torch.cuda.set_device(0)
    fd.set_path(fd.FD_PATH_AUTO)
    # Call 1: a ragged paged GQA batch; call 2: a different contiguous batch, so that
    # anything the first call left in the shared scratch would show up in the second.
    cases = [
        (workloads.paged_case(4, 32, 4, 128, 16, 128, [1, 37, 900, 2048], seed=41), 6),
        (workloads.contiguous_case(2, 16, 2, 128, 3000, [3000, 17], seed=42), 0),
    ]
    for w_cpu, S in cases:
        w = w_cpu.to("cuda")
        ref_o, ref_l = fd.decode_attention(w.q, w.k, w.v, w.seq_lens, w.block_table,
                                           w.page_size, S)
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        st = _call_noalloc(w, out, lse, S)
        assert st == 0, fd.lib().fd_last_error()
        torch.cuda.synchronize()
        _compare(out, lse, ref_o, ref_l)


def test_noalloc_refuses_requests_beyond_its_scratch():
    # B * Hq * S * (d + 1) * 4 bytes of partials: 64 * 64 * 1024 * 129 * 4 > 8 MiB.
    w = workloads.contiguous_case(1, 64, 8, 128, 2048, seed=43, poison_tail=False).to("cuda")
    out = torch.empty(1, 64, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 64, dtype=torch.float32, device="cuda")
    st = _call_noalloc(w, out, lse, 1024)
    assert st == FD_ERR_UNSUPPORTED
    assert b"scratch" in fd.lib().fd_last_error()
