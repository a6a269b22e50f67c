"""GPU: single-split calls write the output from the partial pass.

With one split the merge is the identity (the one weight is 2^(LSE_1 - LSE_1) = 1), so a
decode call with num_splits = 1 writes out and lse_out from the partial-pass kernel and
launches no merge (the 16-rows-per-warp head-group, wide and persistent kernels write
partials and are merged as before: the cases "heads-g16", "wide-64rows" and
"persistent-g16").  For every partial-pass kernel this checks, on ragged rows (rows with
no key, with one key, and multi-token rows shorter than their query count):
  * the output against the fp64 oracle, with the parity tolerances of test_gpu_parity;
  * every element written: out and lse_out start as NaN;
  * out bit for bit equal to the two-pass result of the same kernel (fd_decode_partial
    with one split, then fd_merge_partials), and lse_out equal to it within 1e-6
    relative (the merge recomputes M + log2(1) in base 2).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")


@pytest.fixture(autouse=True)
def _restore():
    yield
    if torch.cuda.is_available():
        fd.set_path(fd.FD_PATH_AUTO)
        fd.set_merge_mode(fd.FD_MERGE_KERNEL)
        fd.set_schedule(fd.FD_SCHEDULE_AUTO)


def _check(got_o, got_l, ref_o, ref_l):
    assert not np.isnan(got_o).any() and not np.isnan(got_l).any(), "an element was not written"
    bound = 4e-3 + 8e-3 * np.abs(ref_o)
    err = np.abs(got_o - ref_o)
    assert (err <= bound).all(), "max excess %.3g" % (err - bound).max()
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(got_l), empty)
    assert (got_o[empty] == 0).all()
    lerr = np.abs(got_l[~empty] - ref_l[~empty])
    assert (lerr <= 1e-4 + 1e-5 * np.abs(ref_l[~empty])).all(), "lse max err %.3g" % lerr.max()


# name: (builder kwargs, Q, kernel expected, settings)
CASES = {
    "mma-grid": (dict(Hq=32, Hkv=8, d=128, paged=0), 1, "fd_partial_mma_kernel",
                 dict(path=fd.FD_PATH_MMA)),
    "mma-grid-d64": (dict(Hq=16, Hkv=2, d=64, paged=0), 1, "fd_partial_mma_kernel",
                     dict(path=fd.FD_PATH_MMA)),
    "simt": (dict(Hq=16, Hkv=4, d=128, paged=0), 1, "fd_partial_simt_kernel",
             dict(path=fd.FD_PATH_SIMT)),
    "heads-g4": (dict(Hq=32, Hkv=8, d=128, paged=16), 1, "fd_partial_heads_kernel", dict()),
    "heads-g16": (dict(Hq=128, Hkv=8, d=128, paged=32), 1, "fd_partial_heads_kernel", dict()),
    "persistent": (dict(Hq=32, Hkv=8, d=128, paged=0), 1, "fd_partial_persist_kernel",
                   dict(path=fd.FD_PATH_MMA, schedule=fd.FD_SCHEDULE_PERSISTENT)),
    "merge-in-kernel": (dict(Hq=32, Hkv=4, d=128, paged=0), 1, "fd_partial_mma_kernel",
                        dict(merge=fd.FD_MERGE_IN_KERNEL)),
    "wide": (dict(Hq=16, Hkv=2, d=128, paged=0), 4, "fd_partial_wide_kernel",
             dict(path=fd.FD_PATH_MMA)),
    "wide-64rows": (dict(Hq=16, Hkv=2, d=128, paged=0), 8, "fd_partial_wide_kernel",
                    dict(path=fd.FD_PATH_MMA)),
    "persistent-g16": (dict(Hq=64, Hkv=4, d=128, paged=0), 1, "fd_partial_persist_kernel",
                       dict(path=fd.FD_PATH_MMA, schedule=fd.FD_SCHEDULE_PERSISTENT)),
    "tcgen05": (dict(Hq=16, Hkv=2, d=128, paged=0), 4, "fd_partial_tc_kernel", dict()),
    "tcgen05-paged": (dict(Hq=64, Hkv=2, d=128, paged=64), 1, "fd_partial_tc_kernel", dict()),
}


def _workload(Hq, Hkv, d, paged, seed):
    lens = [0, 1, 3, 700, 64, 65, 2]
    if paged:
        return workloads.paged_case(len(lens), Hq, Hkv, d, paged, 1024 // paged, lens, seed=seed)
    return workloads.contiguous_case(len(lens), Hq, Hkv, d, 700, lens, seed=seed)


def _apply(settings):
    fd.set_path(settings.get("path", fd.FD_PATH_AUTO))
    fd.set_schedule(settings.get("schedule", fd.FD_SCHEDULE_AUTO))
    fd.set_merge_mode(settings.get("merge", fd.FD_MERGE_KERNEL))


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_single_split_direct_output(name, out_dtype):
    shape, Q, kernel, settings = CASES[name]
    w = _workload(**shape, seed=1300 + len(name))
    B, Hq, Hkv, d = w.B, w.Hq, w.Hkv, w.d
    rows = Q * Hq // Hkv
    assert fd.partial_kernel_name(torch.bfloat16, torch.bfloat16, d, Hkv, w.page_size,
                                  rows=rows) is not None
    _, k, v, lens, bt, ps = w.oracle_arrays()
    if Q == 1:
        q = w.q
        ref_o, ref_l = oracle.decode(workloads.np_storage(q), k, v, lens, block_table=bt,
                                     page_size=ps)
    else:
        q = workloads.multi_token_queries(B, Q, Hq, d, seed=1400 + len(name))
        ref_o, ref_l = oracle.decode_causal(workloads.np_storage(q), k, v, lens,
                                            block_table=bt, page_size=ps)
    ref_o = ref_o.reshape(B * Q, Hq, d)
    ref_l = ref_l.reshape(B * Q, Hq)
    wd = w.to("cuda")
    qd = q.cuda()
    _apply(settings)
    with_opts = fd.options(path=settings.get("path"), schedule=settings.get("schedule"),
                           merge_mode=settings.get("merge"))
    assert fd.partial_kernel_name(torch.bfloat16, torch.bfloat16, d, Hkv, w.page_size,
                                  rows=rows, options=with_opts) == kernel

    # one decode call, one split: the partial pass writes out and lse_out
    ws = torch.zeros(fd.workspace_size(B, Q * Hq, Hkv, d, 1), dtype=torch.uint8, device="cuda")
    out = torch.full(tuple(qd.shape), float("nan"), dtype=out_dtype, device="cuda")
    lse = torch.full(tuple(qd.shape[:-1]), float("nan"), dtype=torch.float32, device="cuda")
    fd.decode_attention(qd, wd.k, wd.v, wd.seq_lens, wd.block_table, w.page_size, 1,
                        out=out, lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    got_o = out.float().cpu().double().numpy().reshape(B * Q, Hq, d)
    got_l = lse.cpu().double().numpy().reshape(B * Q, Hq)
    _check(got_o, got_l, ref_o, ref_l)

    # the same kernel's partials (one split), merged by the merge pass
    fd.set_merge_mode(fd.FD_MERGE_KERNEL)
    ws2 = torch.zeros(fd.workspace_size(B, Q * Hq, Hkv, d, 1), dtype=torch.uint8, device="cuda")
    fd.decode_partial(qd, wd.k, wd.v, wd.seq_lens, ws2, wd.block_table, w.page_size, 1)
    lp, op = fd.workspace_partials(ws2, B, Q * Hq, d, 1)
    o2, l2 = fd.merge_partials(lp, op, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws2) == 0
    assert torch.equal(out.reshape(B, Q * Hq, d), o2), "direct and two-pass outputs differ"
    l2 = l2.reshape(lse.shape)
    fin = torch.isfinite(l2)
    assert torch.equal(torch.isneginf(lse), torch.isneginf(l2))
    assert torch.allclose(lse[fin], l2[fin], rtol=1e-6, atol=1e-6)


def test_single_split_fp8_cache():
    """FP8 E4M3 cache, one split: the output straight from the partial pass equals the
    fp64 FP8 oracle and, bit for bit, the two-pass result."""
    w = workloads.contiguous_case(5, 32, 8, 128, 900, [900, 0, 1, 450, 64], seed=1500)
    kc, vc, ks, vs = workloads.fp8_quantize(w)
    q, _, _, lens, bt, ps = w.oracle_arrays()
    v8 = lambda c: c.view(torch.uint8).numpy()
    ref_o, ref_l = oracle.decode_kv8(q, v8(kc), v8(vc), ks.numpy(), vs.numpy(), lens)
    wd = w.to("cuda")
    kcd, vcd, ksd, vsd = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
    out = torch.full((5, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((5, 32), float("nan"), dtype=torch.float32, device="cuda")
    fd.decode_attention_fp8kv(wd.q, kcd, vcd, ksd, vsd, wd.seq_lens, None, 0, 1, out=out,
                              lse_out=lse)
    ws2 = torch.zeros(fd.workspace_size(5, 32, 8, 128, 1), dtype=torch.uint8, device="cuda")
    fd.decode_partial_fp8kv(wd.q, kcd, vcd, ksd, vsd, wd.seq_lens, ws2, None, 0, 1)
    lp, op = fd.workspace_partials(ws2, 5, 32, 128, 1)
    o2, _ = fd.merge_partials(lp, op, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    _check(out.float().cpu().double().numpy(), lse.cpu().double().numpy(), ref_o, ref_l)
    assert torch.equal(out, o2)


def test_single_split_f32_inputs():
    """f32 q/K/V on the 3xTF32 tensor-core tile and on the CUDA cores, one split, f32 out."""
    w = workloads.contiguous_case(4, 16, 4, 128, 600, [600, 0, 1, 333], seed=1510,
                                  dtype=torch.float32)
    q, k, v, lens, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode(q, k, v, lens)
    wd = w.to("cuda")
    for path in (fd.FD_PATH_MMA, fd.FD_PATH_SIMT):
        fd.set_path(path)
        out = torch.full((4, 16, 128), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((4, 16), float("nan"), dtype=torch.float32, device="cuda")
        fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, num_splits=1, out=out, lse_out=lse)
        torch.cuda.synchronize()
        got_o, got_l = out.cpu().double().numpy(), lse.cpu().double().numpy()
        assert not np.isnan(got_o).any()
        empty = np.isneginf(ref_l)
        assert np.array_equal(np.isneginf(got_l), empty) and (got_o[empty] == 0).all()
        assert np.abs(got_o - ref_o).max() <= 1e-4
        assert np.abs(got_l[~empty] - ref_l[~empty]).max() <= 1e-4
