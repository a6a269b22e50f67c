"""ctypes binding of libfd (see include/fd.h for the meaning of every argument)."""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

FD_OK = 0
FD_ERR_DEVICE_FLAG = 5
FD_F32, FD_BF16, FD_I32, FD_F8E4M3 = 0, 1, 2, 3
FD_PATH_AUTO, FD_PATH_SIMT, FD_PATH_MMA, FD_PATH_TCGEN05 = 0, 1, 2, 3
FD_MERGE_KERNEL, FD_MERGE_IN_KERNEL = 0, 1
FD_SCHEDULE_AUTO, FD_SCHEDULE_GRID, FD_SCHEDULE_PERSISTENT, FD_SCHEDULE_HEAD_GROUPS = 0, 1, 2, 3
FD_SCHEDULE_TAIL_SHARING = 4
FD_FROM_PROCESS = -1

_STATUS = {0: "FD_OK", 1: "FD_ERR_INVALID_ARG", 2: "FD_ERR_UNSUPPORTED",
           3: "FD_ERR_WORKSPACE_TOO_SMALL", 4: "FD_ERR_CUDA", 5: "FD_ERR_DEVICE_FLAG"}


class FdError(RuntimeError):
    """A libfd call returned a status other than FD_OK."""

    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS.get(status, status), message))
        self.status = status


class FdTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class FdOptions(ctypes.Structure):
    """fd_options: path, merge mode and schedule of one call (FD_FROM_PROCESS = the
    process-wide setting)."""
    _fields_ = [("path", ctypes.c_int32), ("merge_mode", ctypes.c_int32),
                ("schedule", ctypes.c_int32)]


def options(path: Optional[int] = None, merge_mode: Optional[int] = None,
            schedule: Optional[int] = None) -> FdOptions:
    """An fd_options for one call or plan; a field left as None takes the process-wide
    setting at the time of the call."""
    pick = lambda v: FD_FROM_PROCESS if v is None else int(v)
    return FdOptions(pick(path), pick(merge_mode), pick(schedule))


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libfd.so (build it first if it is missing or stale).  Raises if that fails."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise ImportError("libfd.so is missing at %s" % path)
            L = ctypes.CDLL(path)
            _declare(L)
            _lib = L
    return _lib


def _declare(L):
    P = ctypes.POINTER(FdTensor)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    L.fd_decode_attention.restype = ctypes.c_int
    L.fd_decode_attention.argtypes = [P, P, P, vp, P, i32, i32, P, vp, vp, sz, vp]
    O = ctypes.POINTER(FdOptions)
    L.fd_decode_attention_ex.restype = ctypes.c_int
    L.fd_decode_attention_ex.argtypes = [P, P, P, vp, vp, vp, P, i32, i32, P, vp, vp, sz, vp, O]
    L.fd_selftest_stalled_decode.restype = ctypes.c_int
    L.fd_selftest_stalled_decode.argtypes = [P, P, P, vp, vp, vp, P, i32, i32, P, vp, vp, sz,
                                             vp, O, i32]
    L.fd_plan_set_options.restype = ctypes.c_int
    L.fd_plan_set_options.argtypes = [vp, O]
    L.fd_partial_kernel_name_ex.restype = ctypes.c_char_p
    L.fd_partial_kernel_name_ex.argtypes = [O, i32, i32, i32, i32, i32, i32, i32]
    L.fd_partial_kernel_name_for.restype = ctypes.c_char_p
    L.fd_partial_kernel_name_for.argtypes = [O, i32, i32, i32, i32, i32, i32, i32, i32,
                                             ctypes.c_int64, i32, i32]
    L.fd_decode_attention_noalloc.restype = ctypes.c_int
    L.fd_decode_attention_noalloc.argtypes = [P, P, P, vp, P, i32, i32, P, vp, vp]
    L.fd_decode_attention_fp8kv.restype = ctypes.c_int
    L.fd_decode_attention_fp8kv.argtypes = [P, P, P, vp, vp, vp, P, i32, i32, P, vp, vp, sz, vp]
    L.fd_decode_partial.restype = ctypes.c_int
    L.fd_decode_partial.argtypes = [P, P, P, vp, P, i32, i32, vp, sz, vp]
    L.fd_decode_partial_fp8kv.restype = ctypes.c_int
    L.fd_decode_partial_fp8kv.argtypes = [P, P, P, vp, vp, vp, P, i32, i32, vp, sz, vp]
    L.fd_workspace_partials.restype = ctypes.c_int
    L.fd_workspace_partials.argtypes = [vp, i32, i32, i32, i32, ctypes.POINTER(vp),
                                        ctypes.POINTER(vp)]
    L.fd_merge_partials.restype = ctypes.c_int
    L.fd_merge_partials.argtypes = [i32, i32, i32, i32, vp, vp, P, vp, vp]
    L.fd_workspace_size.restype = sz
    L.fd_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.fd_num_splits_heuristic.restype = i32
    L.fd_num_splits_heuristic.argtypes = [i32, i32, i32, i32, i64, i32]
    L.fd_num_splits_for_lengths.restype = i32
    L.fd_num_splits_for_lengths.argtypes = [i32, i32, i32, i32, i64, vp, i32, i32]
    L.fd_resolve_num_splits.restype = i32
    L.fd_resolve_num_splits.argtypes = [i32, i32, i32, i32, i64, i32]
    L.fd_resolve_num_splits_q.restype = i32
    L.fd_resolve_num_splits_q.argtypes = [i32, i32, i32, i32, i32, i64, i32]
    L.fd_workspace_init.restype = ctypes.c_int
    L.fd_workspace_init.argtypes = [vp, sz, vp]
    L.fd_read_device_error.restype = ctypes.c_int
    L.fd_read_device_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    L.fd_plan_create.restype = ctypes.c_int
    L.fd_plan_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i64, i32]
    L.fd_plan_create_q.restype = ctypes.c_int
    L.fd_plan_create_q.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i64, i32]
    L.fd_plan_decode_ex.restype = ctypes.c_int
    L.fd_plan_decode_ex.argtypes = [vp, P, P, P, vp, vp, vp, P, i32, P, vp, vp]
    L.fd_plan_num_splits.restype = i32
    L.fd_plan_num_splits.argtypes = [vp]
    L.fd_plan_workspace_bytes.restype = sz
    L.fd_plan_workspace_bytes.argtypes = [vp]
    L.fd_plan_workspace.restype = vp
    L.fd_plan_workspace.argtypes = [vp]
    L.fd_plan_decode.restype = ctypes.c_int
    L.fd_plan_decode.argtypes = [vp, P, P, P, vp, P, i32, P, vp, vp]
    L.fd_plan_resize.restype = ctypes.c_int
    L.fd_plan_resize.argtypes = [vp, i32]
    L.fd_plan_destroy.restype = None
    L.fd_plan_destroy.argtypes = [vp]
    L.fd_set_path.restype = ctypes.c_int
    L.fd_set_path.argtypes = [i32]
    L.fd_set_merge_mode.restype = ctypes.c_int
    L.fd_set_merge_mode.argtypes = [i32]
    L.fd_get_merge_mode.restype = i32
    L.fd_get_merge_mode.argtypes = []
    L.fd_set_schedule.restype = ctypes.c_int
    L.fd_set_schedule.argtypes = [i32]
    L.fd_get_schedule.restype = i32
    L.fd_get_schedule.argtypes = []
    L.fd_selftest_bounded_wait.restype = ctypes.c_int
    L.fd_selftest_bounded_wait.argtypes = [vp, ctypes.c_uint32, vp]
    L.fd_partial_kernel_name.restype = ctypes.c_char_p
    L.fd_partial_kernel_name.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.fd_get_path.restype = i32
    L.fd_get_path.argtypes = []
    L.fd_status_string.restype = ctypes.c_char_p
    L.fd_status_string.argtypes = [ctypes.c_int]
    L.fd_last_error.restype = ctypes.c_char_p
    L.fd_last_error.argtypes = []
    L.fd_version.restype = ctypes.c_char_p
    L.fd_version.argtypes = []


def _check(status: int):
    if status != FD_OK:
        raise FdError(status, lib().fd_last_error().decode(errors="replace"))


_DTYPES = {torch.float32: FD_F32, torch.bfloat16: FD_BF16, torch.int32: FD_I32,
           torch.float8_e4m3fn: FD_F8E4M3}


def tensor_desc(t: Optional[torch.Tensor]) -> Optional[FdTensor]:
    """Describe a torch tensor (up to 4-D) as an fd_tensor; strides in elements."""
    if t is None:
        return None
    if t.dtype not in _DTYPES:
        raise TypeError("unsupported dtype %s" % t.dtype)
    if t.dim() > 4:
        raise ValueError("fd_tensor holds at most 4 dims")
    d = FdTensor()
    d.data = t.data_ptr()
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _ref(x):
    return None if x is None else ctypes.byref(x)


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    h = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return h or None


def workspace_size(B: int, Hq: int, Hkv: int, d: int, num_splits: int) -> int:
    return int(lib().fd_workspace_size(B, Hq, Hkv, d, num_splits))


def num_splits_heuristic(B: int, Hq: int, Hkv: int, d: int, L_cap: int, num_sms: int) -> int:
    return int(lib().fd_num_splits_heuristic(B, Hq, Hkv, d, L_cap, num_sms))


def num_splits_for_lengths(B: int, Hq: int, Hkv: int, d: int, L_cap: int, seq_lens,
                           num_sms: int, page_size: int = 0) -> int:
    """fd_num_splits_for_lengths over host lengths (a CPU int32 tensor or a sequence)."""
    lens = torch.as_tensor(seq_lens, dtype=torch.int32).cpu().contiguous()
    if lens.numel() != B:
        raise ValueError("need one length per batch row")
    return int(lib().fd_num_splits_for_lengths(B, Hq, Hkv, d, L_cap, lens.data_ptr(), page_size,
                                               num_sms))


def resolve_num_splits(B: int, Hq: int, Hkv: int, d: int, L_cap: int, num_splits: int,
                       Q: int = 1) -> int:
    """Split count a call would use (Q query tokens per row; see fd_resolve_num_splits_q)."""
    return int(lib().fd_resolve_num_splits_q(B, Q, Hq, Hkv, d, L_cap, num_splits))


def set_path(path: int):
    _check(lib().fd_set_path(path))


def get_path() -> int:
    return int(lib().fd_get_path())


def set_merge_mode(mode: int):
    _check(lib().fd_set_merge_mode(mode))


def get_merge_mode() -> int:
    return int(lib().fd_get_merge_mode())


def set_schedule(schedule: int):
    _check(lib().fd_set_schedule(schedule))


def get_schedule() -> int:
    return int(lib().fd_get_schedule())


def selftest_bounded_wait(workspace: torch.Tensor, limit_us: int = 50000, stream=None):
    """fd_selftest_bounded_wait: a kernel whose wait runs out must flag a timeout."""
    _check(lib().fd_selftest_bounded_wait(workspace.data_ptr(), limit_us,
                                          _stream_handle(stream)))


def partial_kernel_name_for(dtype, kv_dtype, B: int, Q: int, Hq: int, Hkv: int, d: int,
                            page_size: int, L_cap: int, num_splits: int = 0,
                            with_output: bool = True,
                            options: Optional[FdOptions] = None) -> Optional[str]:
    """The partial-pass kernel a call with exactly these sizes would launch (torch
    dtypes): fd_partial_kernel_name_for."""
    name = lib().fd_partial_kernel_name_for(
        None if options is None else ctypes.byref(options), _DTYPES[dtype], _DTYPES[kv_dtype],
        B, Q, Hq, Hkv, d, page_size, L_cap, num_splits, 1 if with_output else 0)
    return name.decode() if name else None


def partial_kernel_name(dtype, kv_dtype, d: int, Hkv: int, page_size: int = 0,
                        with_output: bool = True, rows: int = 8,
                        options: Optional[FdOptions] = None) -> Optional[str]:
    """The partial-pass kernel a call with these sizes would launch (torch dtypes);
    rows = query rows per kv head (query tokens x Hq / Hkv); options as for the call."""
    args = (_DTYPES[dtype], _DTYPES[kv_dtype], d, Hkv, page_size, rows, 1 if with_output else 0)
    if options is None:
        name = lib().fd_partial_kernel_name(*args)
    else:
        name = lib().fd_partial_kernel_name_ex(ctypes.byref(options), *args)
    return name.decode() if name else None


def selftest_stalled_decode(q, k_cache, v_cache, seq_lens, workspace: torch.Tensor,
                            stall_tile: int, out: torch.Tensor, lse_out: torch.Tensor,
                            block_table=None, page_size: int = 0, num_splits: int = 0,
                            k_scale=None, v_scale=None, options: Optional["FdOptions"] = None,
                            stream=None):
    """fd_selftest_stalled_decode: a decode whose first CTA's producer stops before tile
    `stall_tile`, so that CTA's bounded waits run out (see include/fd.h)."""
    if q.dim() == 4:
        B, Qn, Hq, d = q.shape
    else:
        (B, Hq, d), Qn = q.shape, 1
    S = resolve_num_splits(B, Hq, k_cache.shape[1], d, _cap(k_cache, block_table, page_size),
                           num_splits, Q=Qn)
    dq, dk, dv, dbt, do = (tensor_desc(q), tensor_desc(k_cache), tensor_desc(v_cache),
                           tensor_desc(block_table), tensor_desc(out))
    ptr = lambda t: None if t is None else t.data_ptr()
    _check(lib().fd_selftest_stalled_decode(
        ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ptr(k_scale), ptr(v_scale),
        seq_lens.data_ptr(), _ref(dbt), page_size, S, ctypes.byref(do), lse_out.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream_handle(stream), None if options is None else ctypes.byref(options), stall_tile))


def workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().fd_workspace_init(ws.data_ptr(), ws.numel() * ws.element_size(),
                                   _stream_handle(stream)))


def read_device_error(ws: torch.Tensor, stream=None) -> int:
    """Synchronise, return the workspace's device error flags and clear them."""
    flags = ctypes.c_uint32(0)
    st = lib().fd_read_device_error(ws.data_ptr(), _stream_handle(stream), ctypes.byref(flags))
    if st not in (FD_OK, FD_ERR_DEVICE_FLAG):
        _check(st)
    return int(flags.value)


def _cap(k_cache, block_table, page_size):
    return k_cache.shape[2] if block_table is None else block_table.shape[1] * page_size


def decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     seq_lens: torch.Tensor, block_table: Optional[torch.Tensor] = None,
                     page_size: int = 0, num_splits: int = 0,
                     out: Optional[torch.Tensor] = None, lse_out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, out_dtype=None,
                     stream=None, options: Optional[FdOptions] = None
                     ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Run fd_decode_attention on the current CUDA stream; returns (out, lse_out).

    Missing ``out``/``lse_out``/``workspace`` buffers are allocated with torch (a
    fresh workspace is zero-filled); the library itself allocates nothing.  With
    ``options`` (see ``options()``) the call goes through fd_decode_attention_ex with
    its own path, merge mode and schedule.
    """
    L = lib()
    if q.dim() == 4:                                   # [B, Q, Hq, d]: multi-token decode
        B, Qn, Hq, d = q.shape
    else:
        (B, Hq, d), Qn = q.shape, 1
    Hkv = k_cache.shape[1]
    S = resolve_num_splits(B, Hq, Hkv, d, _cap(k_cache, block_table, page_size), num_splits,
                           Q=Qn)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    if lse_out is None:
        lse_out = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.zeros(workspace_size(B, Qn * Hq, Hkv, d, S), dtype=torch.uint8,
                                device=q.device)
    if seq_lens.dtype != torch.int32:
        raise TypeError("seq_lens must be int32")
    dq, dk, dv, dbt, do = (tensor_desc(q), tensor_desc(k_cache), tensor_desc(v_cache),
                           tensor_desc(block_table), tensor_desc(out))
    ws_args = (workspace.data_ptr(), workspace.numel() * workspace.element_size(),
               _stream_handle(stream))
    if options is None:
        st = L.fd_decode_attention(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv),
                                   seq_lens.data_ptr(), _ref(dbt), page_size, S,
                                   ctypes.byref(do), lse_out.data_ptr(), *ws_args)
    else:
        st = L.fd_decode_attention_ex(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv),
                                      None, None, seq_lens.data_ptr(), _ref(dbt), page_size, S,
                                      ctypes.byref(do), lse_out.data_ptr(), *ws_args,
                                      ctypes.byref(options))
    _check(st)
    return out, lse_out


def decode_attention_noalloc(q, k_cache, v_cache, seq_lens, out: torch.Tensor,
                             lse_out: Optional[torch.Tensor] = None, block_table=None,
                             page_size: int = 0, num_splits: int = 0, stream=None):
    """fd_decode_attention_noalloc: the caller passes every buffer, the library uses
    its built-in scratch instead of a workspace (see include/fd.h for the limits)."""
    dq, dk, dv, dbt, do = (tensor_desc(q), tensor_desc(k_cache), tensor_desc(v_cache),
                           tensor_desc(block_table), tensor_desc(out))
    _check(lib().fd_decode_attention_noalloc(
        ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), seq_lens.data_ptr(), _ref(dbt),
        page_size, num_splits, ctypes.byref(do), None if lse_out is None else lse_out.data_ptr(),
        _stream_handle(stream)))
    return out, lse_out


def decode_attention_fp8kv(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           k_scale: Optional[torch.Tensor], v_scale: Optional[torch.Tensor],
                           seq_lens: torch.Tensor, block_table: Optional[torch.Tensor] = None,
                           page_size: int = 0, num_splits: int = 0,
                           out: Optional[torch.Tensor] = None,
                           lse_out: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, out_dtype=None,
                           stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """fd_decode_attention_fp8kv: k/v torch.float8_e4m3fn, per-kv-head f32 scales."""
    L = lib()
    if q.dim() == 4:
        B, Qn, Hq, d = q.shape
    else:
        (B, Hq, d), Qn = q.shape, 1
    Hkv = k_cache.shape[1]
    S = resolve_num_splits(B, Hq, Hkv, d, _cap(k_cache, block_table, page_size), num_splits,
                           Q=Qn)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    if lse_out is None:
        lse_out = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.zeros(workspace_size(B, Qn * Hq, Hkv, d, S), dtype=torch.uint8,
                                device=q.device)
    dq, dk, dv, dbt, do = (tensor_desc(q), tensor_desc(k_cache), tensor_desc(v_cache),
                           tensor_desc(block_table), tensor_desc(out))
    ptr = lambda t: None if t is None else t.data_ptr()
    _check(L.fd_decode_attention_fp8kv(
        ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ptr(k_scale), ptr(v_scale),
        seq_lens.data_ptr(), _ref(dbt), page_size, S, ctypes.byref(do), lse_out.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream_handle(stream)))
    return out, lse_out


def decode_partial(q, k_cache, v_cache, seq_lens, workspace: torch.Tensor, block_table=None,
                   page_size: int = 0, num_splits: int = 0, stream=None) -> int:
    """Partial pass only (fd_decode_partial); returns the split count used."""
    B, Hq, d = q.shape[0], q.shape[-2], q.shape[-1]
    S = resolve_num_splits(B, Hq, k_cache.shape[1], d, _cap(k_cache, block_table, page_size),
                           num_splits)
    dq, dk, dv, dbt = tensor_desc(q), tensor_desc(k_cache), tensor_desc(v_cache), tensor_desc(block_table)
    _check(lib().fd_decode_partial(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv),
                                   seq_lens.data_ptr(), _ref(dbt), page_size, S,
                                   workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                   _stream_handle(stream)))
    return S


def decode_partial_fp8kv(q, k_cache, v_cache, k_scale, v_scale, seq_lens,
                         workspace: torch.Tensor, block_table=None, page_size: int = 0,
                         num_splits: int = 0, stream=None) -> int:
    """Partial pass over an FP8 E4M3 cache (fd_decode_partial_fp8kv); returns S."""
    B, Hq, d = q.shape[0], q.shape[-2], q.shape[-1]
    S = resolve_num_splits(B, Hq, k_cache.shape[1], d, _cap(k_cache, block_table, page_size),
                           num_splits)
    dq, dk, dv, dbt = tensor_desc(q), tensor_desc(k_cache), tensor_desc(v_cache), tensor_desc(block_table)
    ptr = lambda t: None if t is None else t.data_ptr()
    _check(lib().fd_decode_partial_fp8kv(
        ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ptr(k_scale), ptr(v_scale),
        seq_lens.data_ptr(), _ref(dbt), page_size, S, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(stream)))
    return S


def workspace_partials(workspace: torch.Tensor, B: int, Hq: int, d: int, num_splits: int):
    """Views (lse_part [B, Hq, S], o_part [B, Hq, S, d]) of the partials in a workspace."""
    lp, op = ctypes.c_void_p(), ctypes.c_void_p()
    _check(lib().fd_workspace_partials(workspace.data_ptr(), B, Hq, d, num_splits,
                                       ctypes.byref(lp), ctypes.byref(op)))
    base = workspace.data_ptr()
    raw = workspace.view(torch.uint8)
    lo = (lp.value - base)
    oo = (op.value - base)
    lse = raw[lo:lo + B * Hq * num_splits * 4].view(torch.float32).view(B, Hq, num_splits)
    o = raw[oo:oo + B * Hq * num_splits * d * 4].view(torch.float32).view(B, Hq, num_splits, d)
    return lse, o


def merge_partials(lse_part: torch.Tensor, o_part: torch.Tensor, out: Optional[torch.Tensor] = None,
                   lse_out: Optional[torch.Tensor] = None, out_dtype=torch.float32, stream=None):
    """Merge pass only (fd_merge_partials) over [B, Hq, S] LSEs and [B, Hq, S, d] outputs."""
    B, Hq, S, d = o_part.shape
    if out is None:
        out = torch.empty((B, Hq, d), dtype=out_dtype, device=o_part.device)
    if lse_out is None:
        lse_out = torch.empty((B, Hq), dtype=torch.float32, device=o_part.device)
    if not (lse_part.is_contiguous() and o_part.is_contiguous()):
        raise ValueError("lse_part and o_part must be contiguous")
    do = tensor_desc(out)
    _check(lib().fd_merge_partials(B, Hq, d, S, lse_part.data_ptr(), o_part.data_ptr(),
                                   ctypes.byref(do), lse_out.data_ptr(), _stream_handle(stream)))
    return out, lse_out


class Plan:
    """fd_plan: fixed sizes and split count, owning its workspace and completion event.
    Q > 1: a plan for multi-token decode (q [B, Q, Hq, d])."""

    def __init__(self, B: int, Hq: int, Hkv: int, d: int, L_cap: int, num_splits: int = 0,
                 Q: int = 1):
        self._h = ctypes.c_void_p()
        self.Q = Q
        if Q == 1:
            _check(lib().fd_plan_create(ctypes.byref(self._h), B, Hq, Hkv, d, L_cap, num_splits))
        else:
            _check(lib().fd_plan_create_q(ctypes.byref(self._h), B, Q, Hq, Hkv, d, L_cap,
                                          num_splits))

    @property
    def num_splits(self) -> int:
        return int(lib().fd_plan_num_splits(self._h))

    @property
    def workspace_bytes(self) -> int:
        return int(lib().fd_plan_workspace_bytes(self._h))

    @property
    def workspace_ptr(self) -> int:
        return int(lib().fd_plan_workspace(self._h) or 0)

    def decode(self, q, k_cache, v_cache, seq_lens, block_table=None, page_size=0, out=None,
               lse_out=None, out_dtype=None, stream=None, k_scale=None, v_scale=None):
        """fd_plan_decode (or fd_plan_decode_ex for a 4-D q or an FP8 cache)."""
        if out is None:
            out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
        if lse_out is None:
            lse_out = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
        dq, dk, dv, dbt, do = (tensor_desc(q), tensor_desc(k_cache), tensor_desc(v_cache),
                               tensor_desc(block_table), tensor_desc(out))
        ptr = lambda t: None if t is None else t.data_ptr()
        if q.dim() == 3 and k_cache.dtype != torch.float8_e4m3fn:
            _check(lib().fd_plan_decode(self._h, ctypes.byref(dq), ctypes.byref(dk),
                                        ctypes.byref(dv), seq_lens.data_ptr(), _ref(dbt),
                                        page_size, ctypes.byref(do), lse_out.data_ptr(),
                                        _stream_handle(stream)))
        else:
            _check(lib().fd_plan_decode_ex(self._h, ctypes.byref(dq), ctypes.byref(dk),
                                           ctypes.byref(dv), ptr(k_scale), ptr(v_scale),
                                           seq_lens.data_ptr(), _ref(dbt), page_size,
                                           ctypes.byref(do), lse_out.data_ptr(),
                                           _stream_handle(stream)))
        return out, lse_out

    def resize(self, num_splits: int):
        _check(lib().fd_plan_resize(self._h, num_splits))

    def set_options(self, opts: Optional[FdOptions]):
        """fd_plan_set_options: path, merge mode and schedule of this plan's decodes
        (None = the process-wide settings)."""
        _check(lib().fd_plan_set_options(self._h, None if opts is None else ctypes.byref(opts)))

    def close(self):
        if self._h:
            lib().fd_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 -- interpreter shutdown
            pass
