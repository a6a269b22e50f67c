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
