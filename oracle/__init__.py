"""fp64 CPU oracle for split-KV decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and it
shares no code with the CUDA library: the two meet only at the seeded input
generators in ``workloads.py``, which hold none of the method's arithmetic.

Two independent pieces live here:

* ``decode`` -- the plain UNSPLIT decode attention in fp64 (C, OpenMP over rows),
  see ``fd_oracle.c``.  Split-KV decoding (Flash-Decoding) reaches exactly this
  result up to rounding order, so it is the reference for every GPU parity test.

* ``block_partial`` / ``merge_blocks`` -- the split-and-merge identity restated in
  pure Python fp64, used to pin the oracle (split-count invariance) and to
  reproduce the worked example of the page "2kiu.com/news/6053916", section
  "weight block results with log-sum-exp": a block turns its scores and values
  into (normalised output, m + log z); the merge takes M = max of the block LSEs,
  weights w_i = exp(LSE_i - M) and returns sum(w_i * o_i) / sum(w_i).
  The same merge is described in "FlashDecoding interview notes"
  (gtnt.cn/news/53829), section three, point 2 (w_i in (0, 1]).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfd_oracle.so")

F32 = 0
BF16 = 1

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP, no -ffast-math).  Returns the .so path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load_library(path: Optional[str] = None):
    """Load (building first if needed) the C oracle and declare its signatures."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    lib.fd_oracle_decode.restype = ctypes.c_int
    lib.fd_oracle_decode.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    lib.fd_oracle_decode_causal.restype = ctypes.c_int
    lib.fd_oracle_decode_causal.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    lib.fd_oracle_e4m3_to_double.restype = ctypes.c_double
    lib.fd_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.fd_oracle_decode_kv8.restype = ctypes.c_int
    lib.fd_oracle_decode_kv8.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    lib.fd_oracle_max_threads.restype = ctypes.c_int
    lib.fd_oracle_max_threads.argtypes = []
    if path is None:
        _lib = lib
    return lib


def max_threads() -> int:
    return int(load_library().fd_oracle_max_threads())


def _as_storage(a: np.ndarray) -> Tuple[np.ndarray, int]:
    """Accept fp32 arrays, or bf16 given as raw uint16 bit patterns."""
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), F32
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), BF16
    raise TypeError("oracle inputs must be float32 or uint16 (bf16 bits), got %s" % a.dtype)


def decode(q: np.ndarray, k: np.ndarray, v: np.ndarray, seq_lens: np.ndarray,
           block_table: Optional[np.ndarray] = None, page_size: int = 0,
           rows: Optional[Iterable[int]] = None, num_threads: int = 0,
           lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Unsplit fp64 decode attention.

    q [B, Hq, d]; k, v contiguous [B, Hkv, L_cap, d] (``block_table`` None) or paged
    [num_pages, Hkv, page_size, d] with ``block_table`` int32 [B, max_pages].
    Returns (out [B, Hq, d] float64, lse [B, Hq] float64, natural log).  Rows not
    listed in ``rows`` (flat ids b * Hq + h) are left as NaN.
    """
    lib = lib or load_library()
    q, dt_q = _as_storage(q)
    k, dt_k = _as_storage(k)
    v, dt_v = _as_storage(v)
    if not (dt_q == dt_k == dt_v):
        raise TypeError("q, k and v must share one storage dtype")
    B, Hq, d = q.shape
    Hkv = k.shape[1]
    if k.shape != v.shape or k.shape[3] != d:
        raise ValueError("k/v shape mismatch")
    seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if block_table is None:
        L_cap = k.shape[2]
        bt_ptr, max_pages, ps, num_pages = None, 0, 0, 0
        bt = None
    else:
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        max_pages = bt.shape[1]
        ps = int(page_size)
        if k.shape[2] != ps:
            raise ValueError("paged k must be [num_pages, Hkv, page_size, d]")
        L_cap = max_pages * ps
        num_pages = k.shape[0]
        bt_ptr = bt.ctypes.data
    out = np.full((B, Hq, d), np.nan, dtype=np.float64)
    lse = np.full((B, Hq), np.nan, dtype=np.float64)
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.fromiter(rows, dtype=np.int64))
        rows_ptr, n_rows = rows_arr.ctypes.data, rows_arr.size
    else:
        rows_arr, rows_ptr, n_rows = None, None, 0
    rc = lib.fd_oracle_decode(B, Hq, Hkv, d, dt_q, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                              seq.ctypes.data, L_cap, bt_ptr, max_pages, ps, num_pages,
                              rows_ptr, n_rows, out.ctypes.data, lse.ctypes.data,
                              int(num_threads))
    if rc != 0:
        raise ValueError("fd_oracle_decode rejected its arguments (code %d)" % rc)
    return out, lse


def decode_causal(q: np.ndarray, k: np.ndarray, v: np.ndarray, seq_lens: np.ndarray,
                  block_table: Optional[np.ndarray] = None, page_size: int = 0,
                  rows: Optional[Iterable[int]] = None, num_threads: int = 0,
                  lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Multi-token decode in fp64: q [B, Q, Hq, d]; query j of row b sees keys
    t < L_b - Q + 1 + j.  Returns (out [B, Q, Hq, d], lse [B, Q, Hq]); rows not listed
    in ``rows`` (flat ids (b * Q + j) * Hq + h) are NaN."""
    lib = lib or load_library()
    q, dt_q = _as_storage(q)
    k, dt_k = _as_storage(k)
    v, dt_v = _as_storage(v)
    if not (dt_q == dt_k == dt_v):
        raise TypeError("q, k and v must share one storage dtype")
    B, Q, Hq, d = q.shape
    Hkv = k.shape[1]
    seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if block_table is None:
        L_cap, bt_ptr, max_pages, ps, num_pages, bt = k.shape[2], None, 0, 0, 0, None
    else:
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        max_pages, ps, num_pages = bt.shape[1], int(page_size), k.shape[0]
        L_cap, bt_ptr = max_pages * ps, bt.ctypes.data
    out = np.full((B, Q, Hq, d), np.nan, dtype=np.float64)
    lse = np.full((B, Q, Hq), np.nan, dtype=np.float64)
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.fromiter(rows, dtype=np.int64))
        rows_ptr, n_rows = rows_arr.ctypes.data, rows_arr.size
    else:
        rows_arr, rows_ptr, n_rows = None, None, 0
    rc = lib.fd_oracle_decode_causal(B, Q, Hq, Hkv, d, dt_q, q.ctypes.data, k.ctypes.data,
                                     v.ctypes.data, seq.ctypes.data, L_cap, bt_ptr, max_pages,
                                     ps, num_pages, rows_ptr, n_rows, out.ctypes.data,
                                     lse.ctypes.data, int(num_threads))
    if rc != 0:
        raise ValueError("fd_oracle_decode_causal rejected its arguments (code %d)" % rc)
    return out, lse


def e4m3_to_double(code: int, lib=None) -> float:
    """One FP8 E4M3 code widened to double by the oracle's definition-based decoder."""
    return float((lib or load_library()).fd_oracle_e4m3_to_double(int(code) & 0xFF))


def decode_kv8(q: np.ndarray, k_codes: np.ndarray, v_codes: np.ndarray, k_scale: np.ndarray,
               v_scale: np.ndarray, seq_lens: np.ndarray, block_table: Optional[np.ndarray] = None,
               page_size: int = 0, rows: Optional[Iterable[int]] = None, num_threads: int = 0,
               lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Decode over an FP8 E4M3 KV cache (uint8 codes) with per-kv-head scales [Hkv]:
    k = code * k_scale[g], v = code * v_scale[g]; q fp32 or bf16 bits.  fp64 results."""
    lib = lib or load_library()
    q, dt_q = _as_storage(q)
    k = np.ascontiguousarray(k_codes, dtype=np.uint8)
    v = np.ascontiguousarray(v_codes, dtype=np.uint8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    B, Hq, d = q.shape
    Hkv = k.shape[1]
    if ks.shape != (Hkv,) or vs.shape != (Hkv,):
        raise ValueError("one scale per kv head")
    seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if block_table is None:
        L_cap, bt_ptr, max_pages, ps, num_pages, bt = k.shape[2], None, 0, 0, 0, None
    else:
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        max_pages, ps, num_pages = bt.shape[1], int(page_size), k.shape[0]
        L_cap, bt_ptr = max_pages * ps, bt.ctypes.data
    out = np.full((B, Hq, d), np.nan, dtype=np.float64)
    lse = np.full((B, Hq), np.nan, dtype=np.float64)
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.fromiter(rows, dtype=np.int64))
        rows_ptr, n_rows = rows_arr.ctypes.data, rows_arr.size
    else:
        rows_arr, rows_ptr, n_rows = None, None, 0
    rc = lib.fd_oracle_decode_kv8(B, Hq, Hkv, d, dt_q, q.ctypes.data, k.ctypes.data,
                                  v.ctypes.data, ks.ctypes.data, vs.ctypes.data, seq.ctypes.data,
                                  L_cap, bt_ptr, max_pages, ps, num_pages, rows_ptr, n_rows,
                                  out.ctypes.data, lse.ctypes.data, int(num_threads))
    if rc != 0:
        raise ValueError("fd_oracle_decode_kv8 rejected its arguments (code %d)" % rc)
    return out, lse


# --------------------------------------------------------------------------------------
# Split / merge identity, pure Python fp64 (scalar or vector values).
# --------------------------------------------------------------------------------------

def block_partial(scores: Sequence[float], values: Sequence) -> Tuple[object, float]:
    """One KV block: (softmax-weighted average of its values, LSE of its scores).

    A block must hold at least one key, and as many values as scores; anything else
    is an error, as on the page's worked example.  Values may be floats or numpy
    vectors.
    """
    if len(scores) == 0 or len(scores) != len(values):
        raise ValueError("a block needs at least one key and one value per key")
    m = max(scores)
    weights = [math.exp(s - m) for s in scores]
    z = math.fsum(weights)
    acc = values[0] * weights[0]
    for w, val in zip(weights[1:], values[1:]):
        acc = acc + val * w
    return acc / z, m + math.log(z)


def merge_blocks(parts: Sequence[Tuple[object, float]]) -> Tuple[object, float]:
    """Merge (output, LSE) pairs of disjoint blocks into the global result.

    M = max_i LSE_i; w_i = exp(LSE_i - M) lies in (0, 1]; the merged output is
    sum_i w_i o_i / sum_i w_i and the merged LSE is M + log(sum_i w_i).  With no
    blocks at all there is nothing to merge and that is an error.
    """
    if len(parts) == 0:
        raise ValueError("no blocks to merge")
    M = max(lse for _, lse in parts)
    w = [math.exp(lse - M) for _, lse in parts]
    den = math.fsum(w)
    acc = parts[0][0] * w[0]
    for wi, (o, _) in zip(w[1:], parts[1:]):
        acc = acc + o * wi
    return acc / den, M + math.log(den)


def merge_weights(lses: Sequence[float]) -> list:
    """The normalised merge weights exp(LSE_i - M) / sum_j exp(LSE_j - M)."""
    M = max(lses)
    w = [math.exp(x - M) for x in lses]
    den = math.fsum(w)
    return [x / den for x in w]


def split_ranges(length: int, num_splits: int, capacity: Optional[int] = None):
    """Token ranges of the splits: split_len = ceil(capacity / S); split i covers
    [i * split_len, min((i + 1) * split_len, length)), and is empty when it starts at or
    beyond ``length``.  Pure index arithmetic, used by the split-invariance pins."""
    cap = length if capacity is None else capacity
    split_len = -(-cap // num_splits) if cap > 0 else 0
    out = []
    for i in range(num_splits):
        lo = i * split_len
        hi = min((i + 1) * split_len, length)
        out.append((lo, hi) if lo < hi else (lo, lo))
    return out
