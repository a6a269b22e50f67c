"""Per-call options and the host-side caches of a call, on the GPU.

* Two threads decode at the same time, each with its own fd_options path (CUDA cores
  and mma.sync), while a third thread keeps changing the process-wide path.  Each
  thread's outputs must equal, bit for bit, a single-threaded run of its own path (the
  two paths round differently, so a call that ran the other path would show), and both
  must match the fp64 oracle within the bf16 tolerance of test_gpu_parity.
* A plan with its own options decodes with them, whatever the process setting.
* The TMA descriptors of a KV cache are cached by pointer, shape and strides: a caller
  that swaps between KV buffers of the same shape (and writes new values into one of
  them) still gets the oracle's answer for the buffers it passes on every call.
"""
import dataclasses
import threading

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")


@pytest.fixture(autouse=True)
def _restore_settings():
    yield
    if torch.cuda.is_available():
        fd.set_path(fd.FD_PATH_AUTO)
        fd.set_merge_mode(fd.FD_MERGE_KERNEL)
        fd.set_schedule(fd.FD_SCHEDULE_AUTO)


def _within_oracle(o, l, ref_o, ref_l):
    o = o.double().cpu().numpy()
    l = l.double().cpu().numpy()
    assert not np.isnan(o).any()
    assert (np.abs(o - ref_o) <= 4e-3 + 8e-3 * np.abs(ref_o)).all()
    fin = ~np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(l), ~fin)
    assert (np.abs(l[fin] - ref_l[fin]) <= 1e-4 + 1e-5 * np.abs(ref_l[fin])).all()


def _oracle(w):
    q, k, v, lens, bt, ps = w.oracle_arrays()
    return oracle.decode(q, k, v, lens, block_table=bt, page_size=ps)


def test_two_threads_with_their_own_paths():
    torch.cuda.set_device(0)
    w_cpu = workloads.contiguous_case(2, 16, 2, 128, 4096, [4096, 2999], seed=61,
                                      out_dtype=torch.float32)
    ref_o, ref_l = _oracle(w_cpu)
    w = w_cpu.to("cuda")
    S = 6
    paths = {"simt": fd.FD_PATH_SIMT, "mma": fd.FD_PATH_MMA}

    def one_call(path, stream, ws, out, lse):
        fd.decode_attention(w.q, w.k, w.v, w.seq_lens, None, 0, S, out=out, lse_out=lse,
                            workspace=ws, stream=stream, options=fd.options(path=path))

    def buffers():
        ws = torch.zeros(fd.workspace_size(2, 16, 2, 128, S), dtype=torch.uint8, device="cuda")
        out = torch.empty(2, 16, 128, dtype=torch.float32, device="cuda")
        lse = torch.empty(2, 16, dtype=torch.float32, device="cuda")
        return ws, out, lse

    single = {}
    for name, path in paths.items():
        ws, out, lse = buffers()
        s = torch.cuda.current_stream()
        one_call(path, s, ws, out, lse)
        torch.cuda.synchronize()
        _within_oracle(out, lse, ref_o, ref_l)
        single[name] = (out.clone(), lse.clone())
    assert not torch.equal(single["simt"][0], single["mma"][0])   # the paths are told apart

    stop = threading.Event()
    errors = []

    def toggler():
        order = [fd.FD_PATH_MMA, fd.FD_PATH_SIMT, fd.FD_PATH_TCGEN05, fd.FD_PATH_AUTO]
        i = 0
        while not stop.is_set():
            fd.set_path(order[i % len(order)])
            i += 1

    def worker(name):
        try:
            torch.cuda.set_device(0)
            stream = torch.cuda.Stream()
            ws, out, lse = buffers()
            torch.cuda.synchronize()            # the zero-filled workspace is in place
            for _ in range(40):
                with torch.cuda.stream(stream):
                    out.fill_(float("nan"))
                    one_call(paths[name], stream, ws, out, lse)
                stream.synchronize()
                if not (torch.equal(out, single[name][0]) and torch.equal(lse, single[name][1])):
                    errors.append("%s: outputs differ from its single-threaded run" % name)
                    return
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append("%s: %r" % (name, e))

    threads = [threading.Thread(target=toggler)] + [
        threading.Thread(target=worker, args=(n,)) for n in paths]
    for t in threads[1:]:
        t.start()
    threads[0].start()
    for t in threads[1:]:
        t.join(120)
    stop.set()
    threads[0].join(10)
    assert not errors, errors


def test_plan_options_override_the_process_setting():
    w_cpu = workloads.contiguous_case(1, 8, 1, 128, 2048, [1777], seed=62,
                                      out_dtype=torch.float32)
    ref_o, ref_l = _oracle(w_cpu)
    w = w_cpu.to("cuda")
    plan = fd.Plan(1, 8, 1, 128, 2048, 4)
    try:
        got = {}
        for name, path in (("simt", fd.FD_PATH_SIMT), ("mma", fd.FD_PATH_MMA)):
            plan.set_options(fd.options(path=path))
            fd.set_path(fd.FD_PATH_MMA if name == "simt" else fd.FD_PATH_SIMT)   # the other one
            o, l = plan.decode(w.q, w.k, w.v, w.seq_lens, out_dtype=torch.float32)
            torch.cuda.synchronize()
            _within_oracle(o, l, ref_o, ref_l)
            fd.set_path(path)
            o2, _ = fd.decode_attention(w.q, w.k, w.v, w.seq_lens, None, 0, 4,
                                        out_dtype=torch.float32)
            torch.cuda.synchronize()
            assert torch.equal(o, o2)            # the plan ran its own path
            got[name] = o
        assert not torch.equal(got["simt"], got["mma"])
        with pytest.raises(fd.FdError):
            plan.set_options(fd.options(path=11))
        plan.set_options(None)
    finally:
        plan.close()


def test_swapping_kv_buffers_of_one_shape():
    w_cpu = workloads.contiguous_case(2, 32, 4, 128, 3072, [3072, 1500], seed=63)
    other = dataclasses.replace(
        workloads.contiguous_case(2, 32, 4, 128, 3072, [3072, 1500], seed=64), q=w_cpu.q)
    w = w_cpu.to("cuda")
    k2, v2 = other.k.cuda(), other.v.cuda()
    refs = {"a": _oracle(w_cpu), "b": _oracle(other)}
    ws = torch.zeros(fd.workspace_size(2, 32, 4, 128, 8), dtype=torch.uint8, device="cuda")
    for key, (k, v) in [("a", (w.k, w.v)), ("b", (k2, v2)), ("a", (w.k, w.v)), ("b", (k2, v2))]:
        o, l = fd.decode_attention(w.q, k, v, w.seq_lens, None, 0, 8, workspace=ws,
                                   out_dtype=torch.float32)
        torch.cuda.synchronize()
        _within_oracle(o, l, *refs[key])
    # New values in the same buffers (same pointers, same shapes): the cached descriptors
    # still point at them, and the result follows the new contents.
    k2.copy_(w.k)
    v2.copy_(w.v)
    o, l = fd.decode_attention(w.q, k2, v2, w.seq_lens, None, 0, 8, workspace=ws,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    _within_oracle(o, l, *refs["a"])


def test_plan_for_multi_token_decode_and_resize():
    # 4 query tokens x G = 8 = 32 rows per kv head (the tcgen05 kernel), planned split count.
    w_cpu = workloads.contiguous_case(2, 16, 2, 128, 4096, [4096, 1500], seed=65,
                                      out_dtype=torch.float32)
    q4 = workloads.multi_token_queries(2, 4, 16, 128, seed=66)
    _, k, v, lens, _, _ = w_cpu.oracle_arrays()
    ref_o, ref_l = oracle.decode_causal(workloads.np_storage(q4), k, v, lens)
    w = w_cpu.to("cuda")
    qd = q4.cuda()
    plan = fd.Plan(2, 16, 2, 128, 4096, 0, Q=4)
    try:
        assert plan.num_splits == fd.resolve_num_splits(2, 16, 2, 128, 4096, 0, Q=4)
        assert plan.workspace_bytes >= fd.workspace_size(2, 4 * 16, 2, 128, plan.num_splits)
        for S in (None, 7):
            if S is not None:
                plan.resize(S)
                assert plan.num_splits == 7
            o, l = plan.decode(qd, w.k, w.v, w.seq_lens, out_dtype=torch.float32)
            torch.cuda.synchronize()
            _within_oracle(o.reshape(8, 16, 128), l.reshape(8, 16), ref_o.reshape(8, 16, 128),
                           ref_l.reshape(8, 16))
        with pytest.raises(fd.FdError):                     # a 3-D q does not fit a Q = 4 plan
            plan.decode(w.q, w.k, w.v, w.seq_lens)
    finally:
        plan.close()


def test_plan_over_an_fp8_cache():
    w_cpu = workloads.contiguous_case(2, 32, 4, 128, 3072, [3072, 999], seed=67)
    kc, vc, ks, vs = workloads.fp8_quantize(w_cpu)
    q = workloads.np_storage(w_cpu.q)
    ref_o, ref_l = oracle.decode_kv8(q, kc.view(torch.uint8).numpy(), vc.view(torch.uint8).numpy(),
                                     ks.numpy(), vs.numpy(), w_cpu.seq_lens.numpy())
    plan = fd.Plan(2, 32, 4, 128, 3072, 4)
    try:
        o, l = plan.decode(w_cpu.q.cuda(), kc.cuda(), vc.cuda(), w_cpu.seq_lens.cuda(),
                           k_scale=ks.cuda(), v_scale=vs.cuda(), out_dtype=torch.float32)
        torch.cuda.synchronize()
        _within_oracle(o, l, ref_o, ref_l)
    finally:
        plan.close()
