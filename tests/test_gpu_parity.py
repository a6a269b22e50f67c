"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by
element, on the same seeded inputs.

Tolerances (written here, applied to every element):
  * bf16 inputs (out bf16 or f32):  |got - ref| <= 4e-3 + 8e-3 |ref|
  * f32 inputs, f32 out:            |got - ref| <= 1e-4
  * lse_out (natural log):          |got - ref| <= 1e-4 + 1e-5 |ref|
  * no NaN anywhere; rows with no key give out = 0 and lse = -inf exactly.
Both kernel paths (CUDA-core and tensor-core) are checked for bf16; the f32 tensor-core
path has its own file (test_gpu_f32.py).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")

PATHS_BF16 = [("simt", 1), ("mma", 2)]


@pytest.fixture(autouse=True)
def _restore_path():
    yield
    if torch.cuda.is_available():
        fd.set_path(fd.FD_PATH_AUTO)
        fd.set_merge_mode(fd.FD_MERGE_KERNEL)
        fd.set_schedule(fd.FD_SCHEDULE_AUTO)


MERGES = [("merge-kernel", 0), ("merge-in-kernel", 1)]


_ORACLE_CACHE = {}
_WORKLOADS = {}


def cached(n):
    """Workload n generated once per session, with its device copy."""
    if n not in _WORKLOADS:
        w = workloads.CONFIGS[n]()
        _WORKLOADS[n] = (w, w.to("cuda"))
    return _WORKLOADS[n]


def ref_for(w, key=None):
    if key is not None and key in _ORACLE_CACHE:
        return _ORACLE_CACHE[key]
    q, k, v, lens, bt, ps = w.oracle_arrays()
    r = oracle.decode(q, k, v, lens, block_table=bt, page_size=ps)
    if key is not None:
        _ORACLE_CACHE[key] = r
    return r


def run(w, num_splits=None, out_dtype=None, path=None, check_flags=True, wd=None):
    wd = wd if wd is not None else w.to("cuda")
    if path is not None:
        fd.set_path(path)
    S = w.num_splits if num_splits is None else num_splits
    B, Hq, d = w.q.shape
    S_res = fd.resolve_num_splits(B, Hq, w.Hkv, d, w.L_cap, S)
    ws = torch.zeros(fd.workspace_size(B, Hq, w.Hkv, d, S_res), dtype=torch.uint8, device="cuda")
    out, lse = fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, wd.block_table, wd.page_size,
                                   S, workspace=ws, out_dtype=out_dtype or w.out_dtype)
    torch.cuda.synchronize()
    if check_flags:
        assert fd.read_device_error(ws) == 0
    return out.float().cpu().double().numpy(), lse.cpu().double().numpy(), ws, S_res


def check(w, got_o, got_l, ref_o, ref_l, rows=None):
    if rows is not None:
        flat_o, flat_l = got_o.reshape(-1, got_o.shape[-1]), got_l.reshape(-1)
        got_o, got_l = flat_o[rows], flat_l[rows]
        ref_o, ref_l = ref_o.reshape(-1, ref_o.shape[-1])[rows], ref_l.reshape(-1)[rows]
    assert not np.isnan(got_o).any(), "NaN in out"
    assert not np.isnan(got_l).any(), "NaN in lse"
    if w.q.dtype == torch.bfloat16:
        bound = 4e-3 + 8e-3 * np.abs(ref_o)
    else:
        bound = np.full(ref_o.shape, 1e-4)
    err = np.abs(got_o - ref_o)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), "max excess %.3g at %s (got %r, ref %r)" % (
        (err - bound)[worst], worst, got_o[worst], ref_o[worst])
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(got_l), empty)
    assert (got_o[empty] == 0).all()
    fin = ~empty
    lerr = np.abs(got_l[fin] - ref_l[fin])
    assert (lerr <= 1e-4 + 1e-5 * np.abs(ref_l[fin])).all(), "lse max err %.3g" % lerr.max()
    return float(err.max()) if err.size else 0.0


# ------------------------------------------------------------------ pages' example

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_worked_example(dtype):
    """Scores [0, 0, 10], values [0, 0, 9], split [2 | 1]: the merged output equals the
    unsplit 9 e^10 / (2 + e^10), and the per-split partials left in the workspace are
    the blocks' (0, ln 2) and (9, 10), whose naive average 4.5 is far off."""
    w = workloads.worked_example()
    if dtype == "bf16":
        w = workloads.Workload(w.name, w.q.bfloat16(), w.k.bfloat16(), w.v.bfloat16(),
                               w.seq_lens, num_splits=2, out_dtype=torch.float32)
    paths = [fd.FD_PATH_SIMT, fd.FD_PATH_MMA]
    exact = 9.0 * math.exp(10.0) / (2.0 + math.exp(10.0))
    for path in paths:
        o, l, ws, S = run(w, path=path)
        assert S == 2
        tol = 1e-5 if dtype == "f32" else 4e-3 + 8e-3 * exact
        assert np.abs(o[0, 0] - exact).max() <= tol
        assert abs(l[0, 0] - math.log(2.0 + math.exp(10.0))) <= 1e-4
        # The per-split partials the step left in its workspace.
        lp, op = fd.workspace_partials(ws, 1, 1, 64, 2)
        lse_parts = lp.cpu().numpy().reshape(2)
        o_parts = op.cpu().numpy().reshape(2, 64)
        assert abs(lse_parts[0] - math.log(2.0)) < 1e-5 and abs(lse_parts[1] - 10.0) < 1e-5
        assert np.abs(o_parts[0]).max() < 1e-6 and np.abs(o_parts[1] - 9.0).max() < 1e-5
        naive = o_parts.mean(axis=0)
        assert np.abs(naive - exact).min() > 1.0


# ------------------------------------------------------------------ the five workloads

def test_config1_tiny_fp32():
    w = workloads.config1()
    ref_o, ref_l = ref_for(w, "c1")
    for path in (fd.FD_PATH_SIMT, fd.FD_PATH_MMA, fd.FD_PATH_AUTO):   # AUTO: tensor cores
        o, l, _, S = run(w, path=path)
        assert S == 4
        check(w, o, l, ref_o, ref_l)


@pytest.mark.parametrize("name,path", PATHS_BF16)
@pytest.mark.parametrize("S", [0, 1, 3, 16, 64])
def test_config2_mha(name, path, S):
    w, wd = cached(2)
    ref_o, ref_l = ref_for(w, "c2")
    o, l, _, _ = run(w, num_splits=S, path=path, wd=wd)
    check(w, o, l, ref_o, ref_l)


@pytest.mark.parametrize("name,path", PATHS_BF16)
def test_config3_gqa_128k(name, path):
    w, wd = cached(3)
    ref_o, ref_l = ref_for(w, "c3")
    o, l, _, S = run(w, path=path, wd=wd)     # heuristic split count, as bench.py runs it
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert S == fd.num_splits_heuristic(1, 64, 8, 128, 131072, sms) and S > 1
    check(w, o, l, ref_o, ref_l)


@pytest.mark.parametrize("name,path", PATHS_BF16)
@pytest.mark.parametrize("S", [0, -1, 7, 64])
def test_config4_ragged_paged(name, path, S):
    w, wd = cached(4)
    ref_o, ref_l = ref_for(w, "c4")
    if S == -1:                                 # the length-aware planner's choice
        S = fd.num_splits_for_lengths(w.B, w.Hq, w.Hkv, w.d, w.L_cap, w.seq_lens,
                                      torch.cuda.get_device_properties(0).multi_processor_count,
                                      page_size=w.page_size)
    o, l, _, S_res = run(w, num_splits=S, path=path, wd=wd)
    check(w, o, l, ref_o, ref_l)
    # Row 1 (37 tokens) is shorter than one split: all its other splits are empty.
    split_len = -(-w.L_cap // S_res)
    assert int(w.seq_lens[1]) < split_len or S_res == 1


@pytest.mark.parametrize("name,path", PATHS_BF16)
def test_config5_adversarial_error_does_not_grow(name, path):
    """Spiky scores (~120) in different splits; error must stay within tolerance at every
    split count and must not grow with it (checked in f32-out mode, no output rounding)."""
    w, wd = cached(5)
    ref_o, ref_l = ref_for(w, "c5")
    errs = {}
    for S in w.split_sweep:
        o, l, _, _ = run(w, num_splits=S, path=path, wd=wd)
        check(w, o, l, ref_o, ref_l)
        of, lf, _, _ = run(w, num_splits=S, path=path, out_dtype=torch.float32, wd=wd)
        errs[S] = check(w, of, lf, ref_o, ref_l)
    for S, e in errs.items():
        assert e <= 2.0 * errs[1] + 1e-5, errs


def test_config5_spikes_dominate():
    """The spike heads really see scores near 120: their lse is ~120 and their output is
    close to the spike token's value row."""
    w, wd = cached(5)
    ref_o, ref_l = ref_for(w, "c5")
    spikes = workloads.config5_spikes()
    G = w.Hq // w.Hkv
    for b in range(w.B):
        for g in range(w.Hkv):
            for j in range(4):
                h = g * G + j
                assert 110.0 < ref_l[b, h] < 130.0
    o, l, _, _ = run(w, num_splits=64, path=fd.FD_PATH_MMA, wd=wd)
    b, g, j = 3, 5, 2
    t = int(spikes[b, g, j])
    vrow = w.v[b, g, t].float().numpy()
    assert np.abs(o[b, g * G + j] - vrow).max() < 0.05


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("name,path", PATHS_BF16 + [("simt-f32", 1)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_shapes_ragged_contiguous(name, path, d, G):
    """Every supported (d, G); ragged rows incl. 0, 1 and tile-boundary lengths; NaN in
    the stale cache slots past each length; several split counts."""
    dtype = torch.float32 if name == "simt-f32" else torch.bfloat16
    Hkv = 2
    lens = [0, 1, 63, 64, 65, 300, 517]
    w = workloads.contiguous_case(len(lens), Hkv * G, Hkv, d, 520, lens, seed=7 + d + G,
                                  dtype=dtype, out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    for S in (1, 3, 8, 33):
        o, l, _, _ = run(w, num_splits=S, path=path)
        check(w, o, l, ref_o, ref_l)


@pytest.mark.parametrize("name,path", PATHS_BF16)
@pytest.mark.parametrize("ps", [8, 16, 32, 64, 128, 256])
def test_paged_page_sizes(name, path, ps):
    lens = [1, 37, 200, 513, 1000, 0, 2048]
    max_pages = -(-2048 // ps)
    w = workloads.paged_case(len(lens), 16, 4, 128, ps, max_pages, lens, seed=ps,
                             extra_pages=3, out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    for S in (1, 5, 16):
        o, l, _, _ = run(w, num_splits=S, path=path)
        check(w, o, l, ref_o, ref_l)


@pytest.mark.parametrize("name,path", PATHS_BF16)
def test_paged_d64(name, path):
    lens = [5, 130, 700]
    w = workloads.paged_case(3, 8, 2, 64, 16, 64, lens, seed=64)
    ref_o, ref_l = ref_for(w)
    o, l, _, _ = run(w, num_splits=6, path=path)
    check(w, o, l, ref_o, ref_l)


@pytest.mark.parametrize("name,path", PATHS_BF16)
def test_many_empty_splits(name, path):
    """More splits than tiles, up to the 4096 maximum: most splits are empty (weight 0)."""
    w = workloads.contiguous_case(2, 8, 2, 128, 4096, [3, 4096], seed=11)
    ref_o, ref_l = ref_for(w)
    for S in (512, 4096):
        o, l, _, _ = run(w, num_splits=S, path=path)
        check(w, o, l, ref_o, ref_l)


@pytest.mark.parametrize("name,path", PATHS_BF16)
def test_strided_views(name, path):
    """q, k, v and out as strided views of larger buffers (16-byte multiple strides)."""
    g = torch.Generator().manual_seed(5)
    big_q = torch.randn(3, 16, 136, generator=g).bfloat16()
    big_k = torch.randn(3, 4, 700, 136, generator=g).bfloat16()
    big_v = torch.randn(3, 4, 700, 136, generator=g).bfloat16()
    q, k, v = big_q[:, ::2, :128], big_k[:, ::2, :600, :128], big_v[:, ::2, :600, :128]
    lens = torch.tensor([600, 77, 333], dtype=torch.int32)
    w = workloads.Workload("strided", q, k, v, lens, out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    fd.set_path(path)
    qd, kd, vd = q.cuda(), None, None
    kd = big_k.cuda()[:, ::2, :600, :128]
    vd = big_v.cuda()[:, ::2, :600, :128]
    qd = big_q.cuda()[:, ::2, :128]
    out_big = torch.zeros(3, 8, 160, dtype=torch.float32, device="cuda")
    out = out_big[:, :, :128]
    fd.decode_attention(qd, kd, vd, lens.cuda(), num_splits=4, out=out)
    torch.cuda.synchronize()
    o = out.cpu().double().numpy()
    assert (out_big[:, :, 128:] == 0).all()
    lse = fd.decode_attention(qd, kd, vd, lens.cuda(), num_splits=4,
                              out_dtype=torch.float32)[1].cpu().double().numpy()
    check(w, o, lse, ref_o, ref_l)


def test_bad_page_and_length_are_flagged():
    """A used block-table entry outside the pool and a length beyond capacity are
    reported through the workspace flags; the outputs stay finite."""
    lens = [40, 50]
    w = workloads.paged_case(2, 8, 2, 128, 16, 4, lens, seed=3)
    wd = w.to("cuda")
    bt = wd.block_table.clone()
    bt[0, 1] = 10_000
    ws = torch.zeros(fd.workspace_size(2, 8, 2, 128, 2), dtype=torch.uint8, device="cuda")
    out, lse = fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, bt, 16, 2, workspace=ws)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 2            # FD_DEVFLAG_PAGE
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    assert fd.read_device_error(ws) == 0            # cleared by the read
    seq = torch.tensor([40, 65], dtype=torch.int32, device="cuda")   # capacity is 64
    fd.decode_attention(wd.q, wd.k, wd.v, seq, wd.block_table, 16, 2, workspace=ws)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) & 1             # FD_DEVFLAG_SEQ_LEN


def test_plan_resize_keeps_results():
    w = workloads.contiguous_case(2, 16, 4, 128, 3000, [3000, 1234], seed=21,
                                  out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    plan = fd.Plan(2, 16, 4, 128, 3000, 4)
    try:
        assert plan.num_splits == 4
        bytes4 = plan.workspace_bytes
        o, l = plan.decode(wd.q, wd.k, wd.v, wd.seq_lens, out_dtype=torch.float32)
        torch.cuda.synchronize()
        check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)
        plan.resize(37)
        assert plan.num_splits == 37 and plan.workspace_bytes > bytes4
        o, l = plan.decode(wd.q, wd.k, wd.v, wd.seq_lens, out_dtype=torch.float32)
        torch.cuda.synchronize()
        check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)
    finally:
        plan.close()


def test_side_stream_and_events():
    """Work issued on a side stream completes before results are read there."""
    w = workloads.contiguous_case(1, 8, 8, 128, 2048, seed=31, out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, l = fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, num_splits=8,
                                   out_dtype=torch.float32)
    s.synchronize()
    check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


@pytest.mark.parametrize("name,path", PATHS_BF16)
def test_single_launch_equals_two_pass(name, path):
    """fd_decode_attention in single-launch mode (partials + in-kernel merge by the last
    CTA of each group) against fd_decode_partial followed by fd_merge_partials, both with
    one kv head per CTA (the same partials, so only the merge order differs)."""
    fd.set_merge_mode(fd.FD_MERGE_IN_KERNEL)
    fd.set_schedule(fd.FD_SCHEDULE_GRID)
    w = workloads.paged_case(5, 32, 8, 128, 16, 256, [4096, 1, 0, 2500, 77], seed=51,
                             out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    fd.set_path(path)
    for S in (1, 6, 40, 64):
        ws = torch.zeros(fd.workspace_size(5, 32, 8, 128, S), dtype=torch.uint8, device="cuda")
        o1, l1 = fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, wd.block_table, 16, S,
                                     workspace=ws, out_dtype=torch.float32)
        fd.decode_partial(wd.q, wd.k, wd.v, wd.seq_lens, ws, wd.block_table, 16, S)
        lp, op = fd.workspace_partials(ws, 5, 32, 128, S)
        o2, l2 = fd.merge_partials(lp, op, out_dtype=torch.float32)
        torch.cuda.synchronize()
        check(w, o1.cpu().double().numpy(), l1.cpu().double().numpy(), ref_o, ref_l)
        check(w, o2.cpu().double().numpy(), l2.cpu().double().numpy(), ref_o, ref_l)
        assert torch.allclose(o1, o2, atol=2e-6, rtol=1e-5)


@pytest.mark.parametrize("merge,mode", MERGES)
@pytest.mark.parametrize("name,path", PATHS_BF16)
def test_workspace_reuse_across_calls(name, path, merge, mode):
    """One workspace, many calls with different inputs and split counts (so the merge
    tickets move around inside it): every call must still merge exactly once."""
    fd.set_path(path)
    fd.set_merge_mode(mode)
    cases = [workloads.contiguous_case(3, 16, 4, 128, 2000, [2000, 5, 999], seed=61 + i,
                                       out_dtype=torch.float32) for i in range(3)]
    refs = [ref_for(w) for w in cases]
    ws = torch.zeros(fd.workspace_size(3, 16, 4, 128, 64), dtype=torch.uint8, device="cuda")
    for rep in range(3):
        for (w, (ro, rl)), S in zip(zip(cases, refs), (64, 7, 1)):
            wd = w.to("cuda")
            o, l = fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, num_splits=S,
                                       workspace=ws, out_dtype=torch.float32)
            torch.cuda.synchronize()
            check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ro, rl)
    assert fd.read_device_error(ws) == 0


@pytest.mark.parametrize("merge,mode", MERGES)
@pytest.mark.parametrize("name,path", PATHS_BF16)
def test_workspace_with_stale_contents(name, path, merge, mode):
    """Apart from its flag header, a workspace may hold anything (left by calls of other
    sizes): the merge tickets of each call start from a fresh epoch."""
    fd.set_path(path)
    fd.set_merge_mode(mode)
    w = workloads.contiguous_case(2, 16, 2, 128, 3000, [3000, 1500], seed=71,
                                  out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    n = fd.workspace_size(2, 16, 2, 128, 48)
    g = torch.Generator(device="cuda").manual_seed(3)
    ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
    ws[:256] = 0
    for S in (48, 5):
        o, l = fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, num_splits=S, workspace=ws,
                                   out_dtype=torch.float32)
        torch.cuda.synchronize()
        check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)
    assert fd.read_device_error(ws) == 0


@pytest.mark.parametrize("name,path", PATHS_BF16)
def test_sequence_sharded_merge(name, path):
    """Context parallelism simulated on one GPU: the KV sequence is cut into 4 shards of
    uneven length (as 4 devices would hold them), each shard's partials come from
    fd_decode_partial on that shard alone, and fd_merge_partials over all of them equals
    the unsharded result -- including a row that ends inside shard 2 and has no key at
    all in shard 3."""
    fd.set_path(path)
    w = workloads.contiguous_case(2, 32, 8, 128, 8192, [8192, 5000], seed=81,
                                  out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    cuts = [0, 3000, 4096, 6500, 8192]
    lse_list, o_list = [], []
    for r in range(4):
        lo, hi = cuts[r], cuts[r + 1]
        k = wd.k[:, :, lo:hi].contiguous()
        v = wd.v[:, :, lo:hi].contiguous()
        lens = (wd.seq_lens - lo).clamp(0, hi - lo).to(torch.int32)
        S = 3
        ws = torch.zeros(fd.workspace_size(2, 32, 8, 128, S), dtype=torch.uint8, device="cuda")
        fd.decode_partial(wd.q, k, v, lens, ws, num_splits=S)
        lp, op = fd.workspace_partials(ws, 2, 32, 128, S)
        lse_list.append(lp.clone())
        o_list.append(op.clone())
    lse_all = torch.cat(lse_list, dim=2).contiguous()
    o_all = torch.cat(o_list, dim=2).contiguous()
    o, l = fd.merge_partials(lse_all, o_all, out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("S", [0, 1, 2, 3, 8, 9])
def test_large_batch_merge(d, S):
    """Batches of 1024 query rows or more with up to 8 splits are merged one warp per row
    (not one CTA per row): 48 rows x 32 heads of ragged lengths -- empty rows, one-key
    rows, rows that end inside a split and splits with no key -- against the oracle, with
    the planner's split count, 2, 3 and 8 splits (one warp per row), 9 (one CTA per row)
    and one split (no merge: the partial pass writes the output)."""
    import random
    rnd = random.Random(1000 + d)
    lens = [0, 1, 600, 599, 65] + [rnd.randint(0, 600) for _ in range(43)]
    w = workloads.contiguous_case(48, 32, 8, d, 600, lens, seed=1000 + d,
                                  out_dtype=torch.float32)
    assert 48 * 32 >= 1024
    ref_o, ref_l = ref_for(w, key=("large-batch", d))
    o, l, ws, S_res = run(w, num_splits=S)
    check(w, o, l, ref_o, ref_l)


def test_large_batch_external_merge():
    """fd_merge_partials over 1280 rows (the warp-per-row merge) of partials computed in
    two sequence shards equals the unsharded oracle."""
    w = workloads.contiguous_case(40, 32, 8, 128, 1000, [1000, 0, 400, 401] + [777] * 36,
                                  seed=1010, out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    wd = w.to("cuda")
    lse_list, o_list = [], []
    for lo, hi in ((0, 400), (400, 1000)):
        k = wd.k[:, :, lo:hi].contiguous()
        v = wd.v[:, :, lo:hi].contiguous()
        lens = (wd.seq_lens - lo).clamp(0, hi - lo).to(torch.int32)
        ws = torch.zeros(fd.workspace_size(40, 32, 8, 128, 2), dtype=torch.uint8, device="cuda")
        fd.decode_partial(wd.q, k, v, lens, ws, num_splits=2)
        lp, op = fd.workspace_partials(ws, 40, 32, 128, 2)
        lse_list.append(lp.clone())
        o_list.append(op.clone())
    o, l = fd.merge_partials(torch.cat(lse_list, dim=2).contiguous(),
                             torch.cat(o_list, dim=2).contiguous(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(w, o.cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


@pytest.mark.parametrize("name,path", PATHS_BF16)
@pytest.mark.parametrize("Q,G", [(1, 8), (2, 8), (3, 4), (4, 4), (4, 2), (16, 1)])
@pytest.mark.parametrize("paged", [False, True])
def test_multi_token_decode(name, path, Q, G, paged):
    """q [B, Q, Hq, d]: query j of row b sees keys t <= L_b - Q + j (the causal mask
    inside each split).  Rows shorter than Q leave their first queries without keys
    (out 0, lse -inf).  Checked against the fp64 multi-token oracle for several S."""
    fd.set_path(path)
    Hkv, d = 2, 128
    Hq = Hkv * G
    lens = [1, Q - 1 if Q > 1 else 2, 65, 300, 1000]
    if paged:
        w = workloads.paged_case(len(lens), Hq, Hkv, d, 16, 64, lens, seed=90 + Q * 7 + G,
                                 out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(len(lens), Hq, Hkv, d, 1024, lens, seed=90 + Q * 7 + G,
                                      out_dtype=torch.float32)
    q4 = workloads.multi_token_queries(len(lens), Q, Hq, d, seed=190 + Q + G)
    _, k, v, lens_np, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_causal(workloads.np_storage(q4), k, v, lens_np,
                                        block_table=bt, page_size=ps)
    wd = w.to("cuda")
    qd = q4.cuda()
    B = len(lens)
    for S in (1, 3, 16):
        ws = torch.zeros(fd.workspace_size(B, Q * Hq, Hkv, d, S), dtype=torch.uint8, device="cuda")
        o, l = fd.decode_attention(qd, wd.k, wd.v, wd.seq_lens, wd.block_table, w.page_size, S,
                                   workspace=ws, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert o.shape == (B, Q, Hq, d) and l.shape == (B, Q, Hq)
        assert fd.read_device_error(ws) == 0
        got_o = o.cpu().double().numpy().reshape(B * Q, Hq, d)
        got_l = l.cpu().double().numpy().reshape(B * Q, Hq)
        mw = workloads.Workload("mt", q4.reshape(B * Q, Hq, d), w.k, w.v, w.seq_lens)
        check(mw, got_o, got_l, ref_o.reshape(B * Q, Hq, d), ref_l.reshape(B * Q, Hq))


def test_multi_token_limits():
    """Up to 64 query rows per kv head on the bf16 tensor-core path, 32 with an FP8
    cache; more rows, or more than 16 on the CUDA-core path, are refused on the host."""
    seq = torch.tensor([64], dtype=torch.int32, device="cuda")
    k = torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(1, 5, 16, 128, dtype=torch.bfloat16, device="cuda")     # 5 x 16 = 80 rows
    with pytest.raises(fd.FdError):
        fd.decode_attention(q, k, k, seq, num_splits=1)
    q = torch.zeros(1, 3, 8, 128, dtype=torch.bfloat16, device="cuda")      # 24 rows
    fd.set_path(fd.FD_PATH_SIMT)
    with pytest.raises(fd.FdError):
        fd.decode_attention(q, k, k, seq, num_splits=1)
    fd.set_path(fd.FD_PATH_AUTO)
    k8 = k.float().to(torch.float8_e4m3fn)
    q40 = torch.zeros(1, 5, 8, 128, dtype=torch.bfloat16, device="cuda")    # 40 rows
    with pytest.raises(fd.FdError):
        fd.decode_attention_fp8kv(q40, k8, k8, None, None, seq, num_splits=1)
    o8, _ = fd.decode_attention_fp8kv(q, k8, k8, None, None, seq, num_splits=1)  # 24: accepted
    o, l = fd.decode_attention(q, k, k, seq, num_splits=1)                   # accepted
    torch.cuda.synchronize()
    assert o8.shape == (1, 3, 8, 128)
    torch.cuda.synchronize()
    assert o.shape == (1, 3, 8, 128)


@pytest.mark.parametrize("merge,mode", MERGES)
@pytest.mark.parametrize("Q,G,Hkv,d,paged", [
    (3, 8, 2, 128, False), (4, 8, 2, 128, True), (8, 8, 1, 128, False), (2, 16, 2, 128, True),
    (4, 16, 1, 128, False), (1, 32, 2, 128, False), (1, 64, 1, 128, True), (5, 4, 2, 128, False),
    (3, 16, 1, 64, False), (8, 8, 2, 64, True)])
def test_wide_groups(Q, G, Hkv, d, paged, merge, mode):
    """17 to 64 query rows per kv head (multi-token decode on GQA groups, or groups of 32
    and 64 heads): the mma.sync wide kernel (FD_PATH_MMA; the tcgen05 kernel has its own
    tests), each warp on its own rows over every token, against the fp64 causal oracle;
    rows shorter than Q leave their first queries keyless."""
    fd.set_merge_mode(mode)
    fd.set_path(fd.FD_PATH_MMA)
    Hq = Hkv * G
    lens = [1, max(Q - 1, 1), 70, 333, 1500, 2048]
    if paged:
        w = workloads.paged_case(len(lens), Hq, Hkv, d, 16, 128, lens, seed=900 + Q * 11 + G + d,
                                 out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(len(lens), Hq, Hkv, d, 2048, lens, seed=900 + Q * 11 + G + d,
                                      out_dtype=torch.float32)
    q4 = workloads.multi_token_queries(len(lens), Q, Hq, d, seed=950 + Q + G + d)
    _, k, v, lens_np, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_causal(workloads.np_storage(q4), k, v, lens_np,
                                        block_table=bt, page_size=ps)
    wd = w.to("cuda")
    B = len(lens)
    qd = q4.cuda() if Q > 1 else q4[:, 0].contiguous().cuda()
    assert fd.partial_kernel_name(torch.bfloat16, torch.bfloat16, d, Hkv, w.page_size,
                                  rows=Q * G) == "fd_partial_wide_kernel"
    for S in (1, 5, 16):
        ws = torch.zeros(fd.workspace_size(B, Q * Hq, Hkv, d, S), dtype=torch.uint8, device="cuda")
        o, l = fd.decode_attention(qd, wd.k, wd.v, wd.seq_lens, wd.block_table, w.page_size, S,
                                   workspace=ws, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert fd.read_device_error(ws) == 0
        mw = workloads.Workload("wide", q4.reshape(B * Q, Hq, d), w.k, w.v, w.seq_lens)
        check(mw, o.cpu().double().numpy().reshape(B * Q, Hq, d),
              l.cpu().double().numpy().reshape(B * Q, Hq),
              ref_o.reshape(B * Q, Hq, d), ref_l.reshape(B * Q, Hq))


def _fp8_views(codes):
    return codes.view(torch.uint8).numpy()


@pytest.mark.parametrize("case", ["contiguous", "paged16", "paged256", "gqa16"])
def test_fp8_kv_cache(case):
    """FP8 E4M3 KV cache with per-kv-head scales against the fp64 FP8 oracle (stale
    slots hold NaN codes), several split counts, both merge modes."""
    if case == "contiguous":
        w = workloads.contiguous_case(4, 32, 8, 128, 3000, [3000, 1, 777, 2048], seed=301)
    elif case == "gqa16":
        w = workloads.contiguous_case(2, 32, 2, 128, 2000, [2000, 1500], seed=302)
    else:
        ps = 16 if case == "paged16" else 256
        w = workloads.paged_case(4, 32, 8, 128, ps, 4096 // ps, [1, 37, 2500, 4096], seed=303)
    kc, vc, ks, vs = workloads.fp8_quantize(w)
    q, _, _, lens, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_kv8(q, _fp8_views(kc), _fp8_views(vc), ks.numpy(), vs.numpy(),
                                     lens, block_table=bt, page_size=ps)
    wd = w.to("cuda")
    kcd, vcd, ksd, vsd = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
    for mode in (fd.FD_MERGE_KERNEL, fd.FD_MERGE_IN_KERNEL):
        fd.set_merge_mode(mode)
        for S in (1, 5, 32):
            ws = torch.zeros(fd.workspace_size(w.B, w.Hq, w.Hkv, 128, S), dtype=torch.uint8,
                             device="cuda")
            o, l = fd.decode_attention_fp8kv(wd.q, kcd, vcd, ksd, vsd, wd.seq_lens,
                                             wd.block_table, w.page_size, S, workspace=ws)
            torch.cuda.synchronize()
            assert fd.read_device_error(ws) == 0
            check(w, o.float().cpu().double().numpy(), l.cpu().double().numpy(), ref_o, ref_l)


def test_fp8_kv_multi_token():
    """FP8 KV with multi-token queries: power-of-two scales make the dequantised cache
    exact in fp32, so the fp64 multi-token oracle over it is the reference."""
    Q = 2
    w = workloads.contiguous_case(3, 32, 4, 128, 1500, [1500, 1, 900], seed=311)
    kc, vc, ks, vs = workloads.fp8_quantize(w, power_of_two_scales=True)
    deq = lambda c, s: (c.float() * s.view(1, -1, 1, 1)).numpy()
    q4 = workloads.multi_token_queries(3, Q, 32, 128, seed=312)
    ref_o, ref_l = oracle.decode_causal(q4.float().numpy(), deq(kc, ks), deq(vc, vs),
                                        w.seq_lens.numpy())      # bf16 q is exact in fp32
    o, l = fd.decode_attention_fp8kv(q4.cuda(), kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda(),
                                     w.seq_lens.cuda(), num_splits=4, out_dtype=torch.float32)
    torch.cuda.synchronize()
    mw = workloads.Workload("mt8", q4.reshape(3 * Q, 32, 128), w.k, w.v, w.seq_lens)
    check(mw, o.cpu().double().numpy().reshape(3 * Q, 32, 128), l.cpu().double().numpy().reshape(3 * Q, 32),
          ref_o.reshape(3 * Q, 32, 128), ref_l.reshape(3 * Q, 32))


@pytest.mark.parametrize("Q,G,paged,sched", [(4, 8, 0, "auto"), (3, 8, 32, "auto"),
                                             (4, 8, 64, "grid"), (2, 16, 0, "persistent"),
                                             (4, 8, 16, "persistent")])
def test_fp8_kv_wide_groups(Q, G, paged, sched):
    """FP8 cache with 17 to 32 query rows per kv head: the mma.sync wide kernel (8 rows a
    warp), on the grid and the persistent schedule, against the fp64 multi-token oracle
    over the dequantised cache (power-of-two scales make it exact in fp32); the
    persistent and grid results agree bit for bit."""
    Hkv = 2
    Hq = Hkv * G
    lens = [1, Q - 1, 65, 300, 1000, 0]
    if paged:
        w = workloads.paged_case(len(lens), Hq, Hkv, 128, paged, -(-1024 // paged), lens,
                                 seed=330 + Q + G + paged, out_dtype=torch.float32)
    else:
        w = workloads.contiguous_case(len(lens), Hq, Hkv, 128, 1024, lens, seed=330 + Q + G,
                                      out_dtype=torch.float32)
    kc, vc, ks, vs = workloads.fp8_quantize(w, power_of_two_scales=True)
    deq = lambda c, s: (c.float() * s.view(1, -1, 1, 1)).numpy()
    q4 = workloads.multi_token_queries(len(lens), Q, Hq, 128, seed=340 + Q + G)
    _, _, _, lens_np, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_causal(q4.float().numpy(), deq(kc, ks), deq(vc, vs), lens_np,
                                        block_table=bt, page_size=ps)
    B = len(lens)
    wd = w.to("cuda")
    kcd, vcd, ksd, vsd, qd = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda(), q4.cuda()
    schedule = {"auto": fd.FD_SCHEDULE_AUTO, "grid": fd.FD_SCHEDULE_GRID,
                "persistent": fd.FD_SCHEDULE_PERSISTENT}[sched]
    res = {}
    for S in (1, 5):
        for sc in {schedule, fd.FD_SCHEDULE_GRID}:
            fd.set_schedule(sc)
            ws = torch.zeros(fd.workspace_size(B, Q * Hq, Hkv, 128, S), dtype=torch.uint8,
                             device="cuda")
            o, l = fd.decode_attention_fp8kv(qd, kcd, vcd, ksd, vsd, wd.seq_lens, wd.block_table,
                                             paged, S, workspace=ws, out_dtype=torch.float32)
            torch.cuda.synchronize()
            assert fd.read_device_error(ws) == 0
            mw = workloads.Workload("mt8", q4.reshape(B * Q, Hq, 128), w.k, w.v, w.seq_lens)
            check(mw, o.cpu().double().numpy().reshape(B * Q, Hq, 128),
                  l.cpu().double().numpy().reshape(B * Q, Hq),
                  ref_o.reshape(B * Q, Hq, 128), ref_l.reshape(B * Q, Hq))
            res[(S, sc)] = (o, l)
        if schedule == fd.FD_SCHEDULE_PERSISTENT:
            a, b = res[(S, schedule)], res[(S, fd.FD_SCHEDULE_GRID)]
            assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    fd.set_schedule(fd.FD_SCHEDULE_AUTO)


def test_fp8_kv_is_refused_by_the_bf16_entry_point():
    w = workloads.contiguous_case(1, 8, 1, 128, 64, seed=5).to("cuda")
    kc = w.k.float().to(torch.float8_e4m3fn)
    with pytest.raises(fd.FdError):
        fd.decode_attention(w.q, kc, kc, w.seq_lens, num_splits=1)
    with pytest.raises(fd.FdError):                   # CUDA-core path has no FP8 tile
        fd.set_path(fd.FD_PATH_SIMT)
        fd.decode_attention_fp8kv(w.q, kc, kc, None, None, w.seq_lens, num_splits=1)


def test_fp8_kv_partials_then_merge():
    """fd_decode_partial_fp8kv followed by fd_merge_partials gives what the one-call FP8
    decode gives (same partial kernel, same merge kernel), and matches the oracle."""
    w = workloads.paged_case(3, 32, 8, 128, 16, 128, [2048, 37, 1500], seed=321)
    kc, vc, ks, vs = workloads.fp8_quantize(w)
    q, _, _, lens, bt, ps = w.oracle_arrays()
    ref_o, ref_l = oracle.decode_kv8(q, _fp8_views(kc), _fp8_views(vc), ks.numpy(), vs.numpy(),
                                     lens, block_table=bt, page_size=ps)
    wd = w.to("cuda")
    kcd, vcd, ksd, vsd = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
    S = 7
    ws = torch.zeros(fd.workspace_size(3, 32, 8, 128, S), dtype=torch.uint8, device="cuda")
    fd.decode_partial_fp8kv(wd.q, kcd, vcd, ksd, vsd, wd.seq_lens, ws, wd.block_table, 16, S)
    lp, op = fd.workspace_partials(ws, 3, 32, 128, S)
    o2, l2 = fd.merge_partials(lp, op, out_dtype=torch.float32)
    o1, l1 = fd.decode_attention_fp8kv(wd.q, kcd, vcd, ksd, vsd, wd.seq_lens, wd.block_table,
                                       16, S, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    check(w, o2.cpu().double().numpy(), l2.cpu().double().numpy(), ref_o, ref_l)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bench_launch_configuration():
    """The 128K GQA workload run the way bench.py times it: planned split count, a CUDA
    graph of back-to-back decode calls (programmatic dependent launch between them)
    replayed several times, then the partial pass alone the same way followed by one
    merge.  Every output against the oracle."""
    w, wd = cached(3)
    ref_o, ref_l = ref_for(w, "c3")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    S = fd.num_splits_for_lengths(1, 64, 8, 128, 131072, w.seq_lens.tolist(), sms)
    ws = torch.zeros(fd.workspace_size(1, 64, 8, 128, S), dtype=torch.uint8, device="cuda")
    out = torch.empty(1, 64, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 64, dtype=torch.float32, device="cuda")
    step = lambda: fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, None, 0, S, out=out,
                                       lse_out=lse, workspace=ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(20):
            step()
    out.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    check(w, out.float().cpu().double().numpy(), lse.cpu().double().numpy(), ref_o, ref_l)
    # partial pass back to back, then the merge of the last one's partials
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        for _ in range(10):
            fd.decode_partial(wd.q, wd.k, wd.v, wd.seq_lens, ws, None, 0, S)
    g2.replay()
    lp, op = fd.workspace_partials(ws, 1, 64, 128, S)
    o2, l2 = fd.merge_partials(lp, op, out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(w, o2.cpu().double().numpy(), l2.cpu().double().numpy(), ref_o, ref_l)
