"""The C-ABI library loads and exports every symbol include/fd.h declares, and its
host-only entry points (sizes, heuristic, validation) behave -- no GPU needed.

Validation tests pass fake, never-dereferenced device addresses: every case below is
rejected on the host before the library touches a pointer or calls CUDA."""
import ctypes
import os
import re

import pytest

import decode_attention_05_gb300 as fd
from decode_attention_05_gb300._binding import FdTensor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fd.h")

INVALID, UNSUPPORTED, WS_SMALL = 1, 2, 3


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^FD_API\s+[\w\s\*]+?\b(fd_\w+)\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fd_decode_attention", "fd_workspace_size", "fd_num_splits_heuristic",
                     "fd_plan_create", "fd_plan_resize", "fd_plan_destroy",
                     "fd_read_device_error", "fd_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = fd.lib()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_exports_nothing_undeclared():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", fd.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted({l.split()[-1] for l in out.splitlines() if " T " in l and "fd_" in l})
    assert exported == declared_functions()


def test_status_strings_and_version():
    lib = fd.lib()
    for code, name in [(0, b"FD_OK"), (1, b"FD_ERR_INVALID_ARG"), (2, b"FD_ERR_UNSUPPORTED"),
                       (3, b"FD_ERR_WORKSPACE_TOO_SMALL"), (4, b"FD_ERR_CUDA"),
                       (5, b"FD_ERR_DEVICE_FLAG")]:
        assert lib.fd_status_string(code) == name
    assert b"sm_103a" in lib.fd_version()


def test_workspace_size_layout():
    # 256-byte header, then LSE_i [B, Hq, S] f32, O_i [B, Hq, S, d] f32, the ticket
    # counters [B, Hkv] (64-bit) of the single-launch merge and the claim words
    # [B, Hkv, S] (16 bytes) of tail sharing, each rounded up to 256 B.
    up = lambda x: (x + 255) // 256 * 256

    def expect(B, Hq, Hkv, d, S):
        o_off = up(256 + B * Hq * S * 4)
        cnt_off = up(o_off + B * Hq * S * d * 4)
        steal_off = up(cnt_off + B * Hkv * 8)
        return up(steal_off + B * Hkv * S * 16)
    for B, Hq, Hkv, d, S in [(1, 64, 8, 128, 38), (4, 32, 32, 128, 3), (1, 1, 1, 64, 4),
                             (16, 32, 8, 128, 256), (3, 6, 3, 64, 4096)]:
        assert fd.workspace_size(B, Hq, Hkv, d, S) == expect(B, Hq, Hkv, d, S)
    assert fd.workspace_size(1, 1, 1, 64, 0) == 0
    assert fd.workspace_size(1, 1, 1, 64, 4097) == 0
    assert fd.workspace_size(0, 1, 1, 64, 1) == 0
    # Where the partials live inside a workspace (host arithmetic only).
    fake = 0x7f0000000000
    lp, op = ctypes.c_void_p(), ctypes.c_void_p()
    assert fd.lib().fd_workspace_partials(fake, 1, 64, 128, 38, ctypes.byref(lp),
                                          ctypes.byref(op)) == 0
    assert lp.value == fake + 256 and op.value == fake + up(256 + 64 * 38 * 4)


def test_heuristic_properties():
    h = fd.num_splits_heuristic
    # Full rows of 128K tokens, 8 (b, kv head) pairs, 152 SMs: one wave of at most two
    # CTAs per SM (S <= 38), and split_len a whole number of 64-token tiles -> 32.
    assert h(1, 64, 8, 128, 131072, 152) == 32
    assert h(4, 32, 32, 128, 4096, 152) == 2           # 128 pairs: two splits fit a wave
    assert h(8, 32, 8, 128, 16384, 152) == 4
    # Never more CTAs than one wave, never splits shorter than 256 tokens.
    for B, Hkv, L in [(1, 8, 131072), (1, 1, 1 << 20), (3, 4, 5000), (2, 8, 300)]:
        S = h(B, 4 * Hkv, Hkv, 128, L, 152)
        assert B * Hkv * S <= 2 * 152 or S == 1
        assert S == 1 or -(-L // S) >= 64
    assert h(1, 32, 8, 128, 256, 152) == 1
    # Enough (b, kv head) pairs already fill the GPU: one split.
    assert h(64, 32, 32, 128, 4096, 152) == 1
    # More SMs -> at least as many splits.
    for L in (1024, 8192, 65536, 1 << 20):
        assert h(1, 64, 8, 128, L, 304) >= h(1, 64, 8, 128, L, 152)
    # Invalid sizes fall back to one split.
    assert h(0, 64, 8, 128, 1000, 152) == 1
    assert h(1, 64, 8, 128, 1000, 0) == 1


def test_length_aware_planner():
    import workloads
    f = fd.num_splits_for_lengths
    # A ragged batch whose capacity is 32K but most rows are far shorter: the planner
    # splits more than the capacity-only heuristic would.
    lens = workloads.config4_lens()
    S = f(16, 32, 8, 128, 32768, lens, 152, page_size=16)
    assert S > fd.num_splits_heuristic(16, 32, 8, 128, 32768, 152)
    assert S == f(16, 32, 8, 128, 32768, lens, 152, page_size=16)             # deterministic
    # Full rows: a single-wave split count, as the capacity-only heuristic plans.

    # The counts measured fastest on GB300 for the uniform workloads (128K GQA, MHA 4K,
    # adversarial 16K) and the ragged paged one.
    assert f(1, 64, 8, 128, 131072, [131072], 152) == 32
    assert f(4, 32, 32, 128, 4096, [4096] * 4, 152) == 2
    assert f(8, 32, 8, 128, 16384, [16384] * 8, 152) == 4
    assert f(16, 32, 8, 128, 32768, lens, 152, page_size=16) == 16
    # Nothing to read, or invalid sizes: one split.
    assert f(4, 8, 8, 128, 4096, [0, 0, 0, 0], 152) == 1
    assert f(0, 8, 8, 128, 4096, [], 152) == 1


def test_merge_mode_round_trip():
    lib = fd.lib()
    try:
        assert fd.get_merge_mode() == fd.FD_MERGE_KERNEL          # the default
        fd.set_merge_mode(fd.FD_MERGE_IN_KERNEL)
        assert fd.get_merge_mode() == fd.FD_MERGE_IN_KERNEL
        with pytest.raises(fd.FdError):
            fd.set_merge_mode(5)
    finally:
        lib.fd_set_merge_mode(fd.FD_MERGE_KERNEL)


def test_schedule_round_trip():
    lib = fd.lib()
    try:
        assert fd.get_schedule() == fd.FD_SCHEDULE_AUTO            # the default
        for sched in (fd.FD_SCHEDULE_GRID, fd.FD_SCHEDULE_PERSISTENT,
                      fd.FD_SCHEDULE_HEAD_GROUPS, fd.FD_SCHEDULE_TAIL_SHARING,
                      fd.FD_SCHEDULE_AUTO):
            fd.set_schedule(sched)
            assert fd.get_schedule() == sched
        with pytest.raises(fd.FdError):
            fd.set_schedule(5)
        assert fd.get_schedule() == fd.FD_SCHEDULE_AUTO            # unchanged on error
    finally:
        lib.fd_set_schedule(fd.FD_SCHEDULE_AUTO)


def test_partial_kernel_name_follows_settings():
    """Which partial kernel a call would launch, from the sizes and process settings."""
    import torch
    bf, f32, f8 = torch.bfloat16, torch.float32, torch.float8_e4m3fn
    name = fd.partial_kernel_name
    lib = fd.lib()
    try:
        assert name(bf, bf, 128, 8) == "fd_partial_mma_kernel"                 # contiguous
        assert name(bf, bf, 128, 8, 16) == "fd_partial_heads_kernel"           # small pages
        assert name(bf, bf, 128, 8, 32) == "fd_partial_heads_kernel"
        assert name(bf, bf, 128, 8, 64) == "fd_partial_mma_kernel"
        assert name(bf, bf, 128, 6, 16) == "fd_partial_mma_kernel"             # Hkv % 4
        assert name(bf, bf, 64, 8, 16) == "fd_partial_mma_kernel"              # d = 64
        assert name(bf, f8, 128, 8, 16) == "fd_partial_mma_kernel"             # FP8 KV
        assert name(bf, f8, 128, 8, 32) == "fd_partial_heads_kernel"           # 32-token tiles
        assert name(bf, f8, 128, 8, 64) == "fd_partial_mma_kernel"
        assert name(f32, f32, 128, 8) == "fd_partial_mma_kernel"               # 3xTF32
        assert name(f32, f32, 64, 8, 16, rows=4) == "fd_partial_mma_kernel"    # grid only
        assert name(f32, f32, 128, 8, rows=16) == "fd_partial_simt_kernel"     # > 8 rows
        assert name(f32, f8, 128, 8) is None
        assert name(bf, bf, 128, 8, rows=16) == "fd_partial_mma_kernel"       # Q x G <= 16
        assert name(bf, bf, 128, 8, rows=17) == "fd_partial_tc_kernel"        # Q x G > 16
        assert name(bf, bf, 128, 8, rows=32) == "fd_partial_tc_kernel"
        assert name(bf, bf, 128, 8, 16, rows=64) == "fd_partial_tc_kernel"
        assert name(bf, bf, 128, 8, 8, rows=64) == "fd_partial_wide_kernel"   # 8-token pages
        assert name(bf, bf, 64, 8, rows=32) == "fd_partial_wide_kernel"       # d = 64
        assert name(bf, f8, 128, 8, rows=32) == "fd_partial_wide_kernel"      # FP8 <= 32
        assert name(bf, f8, 128, 8, rows=33) is None
        assert name(f32, f32, 128, 8, rows=32) is None
        assert name(bf, bf, 128, 8, rows=65) is None
        fd.set_merge_mode(fd.FD_MERGE_IN_KERNEL)                              # single launch
        assert name(bf, bf, 128, 8, 16) == "fd_partial_mma_kernel"
        assert name(bf, bf, 128, 8, 16, with_output=False) == "fd_partial_heads_kernel"
        fd.set_merge_mode(fd.FD_MERGE_KERNEL)
        fd.set_schedule(fd.FD_SCHEDULE_GRID)
        assert name(bf, bf, 128, 8, 16) == "fd_partial_mma_kernel"
        fd.set_schedule(fd.FD_SCHEDULE_PERSISTENT)
        assert name(bf, bf, 128, 8, 16) == "fd_partial_heads_persist_kernel"   # its tiling
        assert name(bf, bf, 128, 8, 64) == "fd_partial_persist_kernel"
        assert name(bf, bf, 128, 8) == "fd_partial_persist_kernel"
        assert name(f32, f32, 128, 8) == "fd_partial_mma_kernel"
        fd.set_path(fd.FD_PATH_MMA)
        assert name(f32, f32, 128, 8, rows=16) is None
        assert name(bf, bf, 128, 8, rows=32) == "fd_partial_wide_persist_kernel"  # 8 a warp
        assert name(bf, bf, 128, 8, rows=64) == "fd_partial_wide_kernel"          # 16 a warp
        fd.set_path(fd.FD_PATH_TCGEN05)
        assert name(bf, bf, 128, 8) == "fd_partial_tc_kernel"                 # any group size
        assert name(bf, bf, 128, 8, 32, rows=64) == "fd_partial_tc_kernel"
        assert name(bf, bf, 128, 8, 8) is None
        assert name(bf, bf, 64, 8) is None
        assert name(f32, f32, 128, 8) is None
        assert name(bf, f8, 128, 8) is None
        fd.set_path(fd.FD_PATH_SIMT)
        assert name(f32, f32, 128, 8) == "fd_partial_simt_kernel"
        assert name(bf, bf, 128, 8) == "fd_partial_simt_kernel"
    finally:
        lib.fd_set_schedule(fd.FD_SCHEDULE_AUTO)
        lib.fd_set_merge_mode(fd.FD_MERGE_KERNEL)
        lib.fd_set_path(fd.FD_PATH_AUTO)


def test_path_setting_round_trip():
    lib = fd.lib()
    try:
        for path in (fd.FD_PATH_SIMT, fd.FD_PATH_MMA, fd.FD_PATH_TCGEN05, fd.FD_PATH_AUTO):
            fd.set_path(path)
            assert fd.get_path() == path
        with pytest.raises(fd.FdError):
            fd.set_path(7)
    finally:
        lib.fd_set_path(fd.FD_PATH_AUTO)


# ---------------------------------------------------------------- host-side validation

FAKE = 0x7f0000000000          # 16-byte aligned, never dereferenced


def desc(shape, dtype=1, stride=None, data=FAKE):
    t = FdTensor()
    t.data = data
    t.dtype = dtype
    t.ndim = len(shape)
    if stride is None:
        stride, acc = [], 1
        for s in reversed(shape):
            stride.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, stride)):
        t.shape[i] = s
        t.stride[i] = st
    return t


def call(q, k, v, out, *, bt=None, page_size=0, S=4, ws_bytes=1 << 24, ws=FAKE,
         seq=FAKE, lse=FAKE):
    lib = fd.lib()
    r = lambda x: None if x is None else ctypes.byref(x)
    return lib.fd_decode_attention(r(q), r(k), r(v), seq, r(bt), page_size, S, r(out), lse, ws,
                                   ws_bytes, None)


def good():
    return (desc([2, 8, 128]), desc([2, 2, 1024, 128]), desc([2, 2, 1024, 128]),
            desc([2, 8, 128]))


def test_fp8_row_limit_on_the_host():
    """An FP8 cache takes up to 32 query rows per kv head: 40 (5 query tokens x G 8) are
    refused before anything touches the device."""
    lib = fd.lib()
    r = ctypes.byref
    for Qn, ok in ((5, False), (4, True)):
        q, out = desc([2, Qn, 16, 128]), desc([2, Qn, 16, 128])
        k, v = desc([2, 2, 1024, 128], dtype=3), desc([2, 2, 1024, 128], dtype=3)
        st = lib.fd_decode_attention_fp8kv(r(q), r(k), r(v), None, None, FAKE, None, 0, 4,
                                           r(out), FAKE, FAKE, 1 << 28, None)
        msg = lib.fd_last_error().decode()
        if not ok:
            assert st == UNSUPPORTED and "32 query rows" in msg, msg
        else:
            assert "query rows" not in msg, msg


@pytest.mark.parametrize("case,expected", [
    ("null_q", INVALID), ("null_seq", INVALID), ("null_ws", INVALID), ("rank", INVALID),
    ("hq_not_multiple", INVALID), ("kv_shape_mismatch", INVALID), ("dtype_mix", INVALID),
    ("head_dim_96", UNSUPPORTED), ("group_3", UNSUPPORTED), ("f32_in_bf16_out", UNSUPPORTED),
    ("neg_splits", INVALID), ("too_many_splits", INVALID), ("noncontig_last", INVALID),
    ("misaligned_k", INVALID), ("odd_stride", INVALID), ("page_size_no_table", INVALID),
    ("page_size_not_pow2", INVALID), ("page_size_small", INVALID), ("table_dtype", INVALID),
    ("ws_small", WS_SMALL), ("ws_misaligned", INVALID), ("out_shape", INVALID),
    ("paged_shape", INVALID),
])
def test_validation(case, expected):
    q, k, v, out = good()
    kw = {}
    if case == "null_q":
        q = None
    elif case == "null_seq":
        kw["seq"] = None
    elif case == "null_ws":
        kw["ws"] = None
    elif case == "rank":
        q = desc([2, 8, 128, 1])
    elif case == "hq_not_multiple":
        q, out = desc([2, 7, 128]), desc([2, 7, 128])
    elif case == "kv_shape_mismatch":
        v = desc([2, 2, 512, 128])
    elif case == "dtype_mix":
        k = desc([2, 2, 1024, 128], dtype=0)
    elif case == "head_dim_96":
        q, k, v, out = desc([2, 8, 96]), desc([2, 2, 64, 96]), desc([2, 2, 64, 96]), desc([2, 8, 96])
    elif case == "group_3":
        q, out = desc([2, 6, 128]), desc([2, 6, 128])
    elif case == "f32_in_bf16_out":
        q, k, v = desc([2, 8, 128], 0), desc([2, 2, 1024, 128], 0), desc([2, 2, 1024, 128], 0)
    elif case == "neg_splits":
        kw["S"] = -1
    elif case == "too_many_splits":
        kw["S"] = 4097
    elif case == "noncontig_last":
        k = desc([2, 2, 1024, 128], stride=[2 * 1024 * 256, 1024 * 256, 256, 2])
    elif case == "misaligned_k":
        k = desc([2, 2, 1024, 128], data=FAKE + 8)
    elif case == "odd_stride":
        k = desc([2, 2, 1024, 128], stride=[2 * 1024 * 130, 1024 * 130, 130, 1])
    elif case == "page_size_no_table":
        kw["page_size"] = 16
    elif case == "page_size_not_pow2":
        kw["bt"], kw["page_size"] = desc([2, 8], dtype=2), 24
        k, v = desc([16, 2, 24, 128]), desc([16, 2, 24, 128])
    elif case == "page_size_small":
        kw["bt"], kw["page_size"] = desc([2, 8], dtype=2), 4
        k, v = desc([16, 2, 4, 128]), desc([16, 2, 4, 128])
    elif case == "table_dtype":
        kw["bt"], kw["page_size"] = desc([2, 8], dtype=0), 16
        k, v = desc([16, 2, 16, 128]), desc([16, 2, 16, 128])
    elif case == "ws_small":
        kw["ws_bytes"] = 1024
    elif case == "ws_misaligned":
        kw["ws"] = FAKE + 16
    elif case == "out_shape":
        out = desc([2, 8, 64])
    elif case == "paged_shape":
        kw["bt"], kw["page_size"] = desc([2, 8], dtype=2), 16
        k, v = desc([16, 2, 32, 128]), desc([16, 2, 32, 128])
    assert call(q, k, v, out, **kw) == expected
    assert fd.lib().fd_last_error()        # a reason is recorded


# ---------------------------------------------------------------- per-call options

def test_partial_kernel_name_for_sized_calls():
    """The kernel of a call with exact sizes: one split with an output never merges
    in-kernel (so small pages keep head groups under FD_MERGE_IN_KERNEL), forced head
    groups take contiguous caches and large pages, and bad sizes give None.  (Without a
    device the SM count is unknown and the large-batch rule never applies.)"""
    import torch
    bf = torch.bfloat16
    name = fd.partial_kernel_name_for
    inkernel = fd.options(merge_mode=fd.FD_MERGE_IN_KERNEL)
    assert name(bf, bf, 4, 1, 32, 8, 128, 16, 4096, 1, options=inkernel) == "fd_partial_heads_kernel"
    assert name(bf, bf, 4, 1, 32, 8, 128, 16, 4096, 4, options=inkernel) == "fd_partial_mma_kernel"
    assert name(bf, bf, 4, 1, 32, 8, 128, 16, 4096, 4, with_output=False,
                options=inkernel) == "fd_partial_heads_kernel"
    heads = fd.options(schedule=fd.FD_SCHEDULE_HEAD_GROUPS)
    assert name(bf, bf, 4, 1, 32, 8, 128, 0, 4096, 4, options=heads) == "fd_partial_heads_kernel"
    assert name(bf, bf, 4, 1, 32, 8, 128, 64, 4096, 4, options=heads) == "fd_partial_heads_kernel"
    assert name(bf, bf, 4, 1, 32, 8, 128, 8, 4096, 4, options=heads) == "fd_partial_mma_kernel"
    assert name(bf, bf, 4, 1, 24, 6, 128, 0, 4096, 4, options=heads) == "fd_partial_mma_kernel"
    assert name(bf, bf, 4, 4, 32, 8, 128, 0, 4096, 4) == "fd_partial_mma_kernel"     # 16 rows
    assert name(bf, bf, 4, 8, 32, 8, 128, 0, 4096, 4) == "fd_partial_tc_kernel"      # 32 rows
    # up to 32 rows with at most 512 tokens a split: the persistent mma.sync wide kernel
    assert name(bf, bf, 4, 8, 32, 8, 128, 0, 2048, 4) == "fd_partial_wide_persist_kernel"
    assert name(bf, bf, 4, 8, 32, 8, 128, 0, 2052, 4) == "fd_partial_tc_kernel"     # 513 a split
    assert name(bf, bf, 4, 8, 64, 8, 128, 0, 1024, 4) == "fd_partial_tc_kernel"     # 64 rows
    grid = fd.options(schedule=fd.FD_SCHEDULE_GRID)
    assert name(bf, bf, 4, 8, 32, 8, 128, 0, 2048, 4, options=grid) == "fd_partial_wide_kernel"
    for bad in ((0, 1, 32, 8), (4, 0, 32, 8), (4, 1, 30, 8), (4, 1, 32, 0), (4, 17, 32, 8)):
        assert name(bf, bf, *bad, 128, 0, 4096, 4) is None
    assert name(bf, bf, 4, 1, 32, 8, 128, 0, 0, 4) is None
    assert name(bf, bf, 4, 1, 32, 8, 128, 0, 4096, -1) is None
    assert name(bf, bf, 4, 1, 32, 8, 128, 0, 4096, 4, options=fd.options(path=9)) is None


def test_options_choose_the_kernel_per_call():
    """fd_options override the process-wide settings for one query (and one call) and
    leave those settings as they were; FD_FROM_PROCESS fields follow them."""
    import torch
    bf = torch.bfloat16
    name = fd.partial_kernel_name
    lib = fd.lib()
    try:
        fd.set_path(fd.FD_PATH_SIMT)
        fd.set_schedule(fd.FD_SCHEDULE_PERSISTENT)
        assert name(bf, bf, 128, 8) == "fd_partial_simt_kernel"
        o = fd.options(path=fd.FD_PATH_MMA, schedule=fd.FD_SCHEDULE_GRID)
        assert name(bf, bf, 128, 8, options=o) == "fd_partial_mma_kernel"
        assert name(bf, bf, 128, 8, options=fd.options(path=fd.FD_PATH_MMA)) == \
            "fd_partial_persist_kernel"                        # schedule from the process
        assert name(bf, bf, 128, 8, options=fd.options()) == "fd_partial_simt_kernel"
        assert name(bf, bf, 128, 8, 16, options=fd.options(
            path=fd.FD_PATH_AUTO, schedule=fd.FD_SCHEDULE_AUTO)) == "fd_partial_heads_kernel"
        assert name(bf, bf, 128, 8, 16, options=fd.options(
            path=fd.FD_PATH_AUTO, schedule=fd.FD_SCHEDULE_AUTO,
            merge_mode=fd.FD_MERGE_IN_KERNEL)) == "fd_partial_mma_kernel"
        assert name(bf, bf, 128, 8, options=fd.options(path=fd.FD_PATH_TCGEN05)) == \
            "fd_partial_tc_kernel"
        for bad in (fd.options(path=9), fd.options(merge_mode=2), fd.options(schedule=-2)):
            assert name(bf, bf, 128, 8, options=bad) is None
        assert fd.get_path() == fd.FD_PATH_SIMT                # process settings untouched
        assert fd.get_schedule() == fd.FD_SCHEDULE_PERSISTENT
    finally:
        lib.fd_set_schedule(fd.FD_SCHEDULE_AUTO)
        lib.fd_set_merge_mode(fd.FD_MERGE_KERNEL)
        lib.fd_set_path(fd.FD_PATH_AUTO)


def call_ex(q, k, v, out, opts, *, k_scale=None, v_scale=None, S=4):
    lib = fd.lib()
    r = lambda x: None if x is None else ctypes.byref(x)
    return lib.fd_decode_attention_ex(r(q), r(k), r(v), k_scale, v_scale, FAKE, None, 0, S,
                                      r(out), FAKE, FAKE, 1 << 24, None, r(opts))


def test_decode_ex_validation():
    q, k, v, out = good()
    assert call_ex(q, k, v, out, fd.options(path=9)) == INVALID
    assert call_ex(q, k, v, out, fd.options(merge_mode=3)) == INVALID
    assert call_ex(q, k, v, out, fd.options(schedule=7)) == INVALID
    # Scales belong to an FP8 cache only.
    assert call_ex(q, k, v, out, None, k_scale=FAKE) == INVALID
    # An FP8 cache takes bf16 q and head dim 128; the checks of the FP8 entry point apply.
    k8, v8 = desc([2, 2, 1024, 64], dtype=3), desc([2, 2, 1024, 64], dtype=3)
    q64, out64 = desc([2, 8, 64]), desc([2, 8, 64])
    assert call_ex(q64, k8, v8, out64, None) == UNSUPPORTED
    # The partial pass alone (out NULL) still validates every input.
    assert call_ex(desc([2, 7, 128]), k, v, None, None) == INVALID
    # An FP8 cache through the plain entry point is refused, as before.
    assert call(q, desc([2, 2, 1024, 128], dtype=3), desc([2, 2, 1024, 128], dtype=3), out) \
        == INVALID


def test_plan_argument_checks():
    """Invalid plan sizes are refused on the host, before any allocation."""
    lib = fd.lib()
    h = ctypes.c_void_p()
    assert lib.fd_plan_create_q(ctypes.byref(h), 1, 0, 8, 1, 128, 1024, 0) == INVALID   # Q = 0
    assert lib.fd_plan_create_q(ctypes.byref(h), 1, 2, 6, 4, 128, 1024, 0) == INVALID   # Hq % Hkv
    assert lib.fd_plan_create_q(ctypes.byref(h), 1, 2, 8, 1, 128, 1024, 4097) == INVALID
    assert lib.fd_plan_create(ctypes.byref(h), 0, 8, 1, 128, 1024, 0) == INVALID
    assert not h.value
    assert lib.fd_plan_decode_ex(None, None, None, None, None, None, None, None, 0, None, None,
                                 None) == INVALID
