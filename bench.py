"""Benchmark: one decode step of split-KV attention on the 128K-context GQA workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fd|reference]
                    [--config 1-5] [--kv bf16|fp8] [--num-splits S] [--no-graph]

Workload (default): bf16, B=1, Hq=64, Hkv=8 (G=8), d=128, L=131072, contiguous KV
cache (512 MiB of K+V, four times the L2), split count from the library's length-aware
planner (fd_num_splits_for_lengths).
A step is one full pass of the hot path: the split-KV partial kernel plus the LSE
merge kernel, through the C ABI (fd_decode_attention).

Prints ONE JSON line.  ``value`` is the whole-job KV-read throughput (GB/s) over the
K timed steps (device time, CUDA events, max over ranks); ``ms_per_step`` and
``us_per_step`` give the step time.  The timed loops replay CUDA graphs of 100
back-to-back calls (``--no-graph``: one call at a time from Python); a cache smaller
than three L2s is streamed from two alternating copies.  ``--kv fp8`` runs the same
workload over its FP8 E4M3 quantisation (per-kv-head scales).  Also reported:
  roofline      the partial kernel alone: algorithmic KV bytes per launch / its mean
                CUDA-event duration, against the measured HBM copy bandwidth;
  e2e           the same metric through the public Python API with the step's inputs
                copied from pinned host memory and the result read back every step;
  cpu_baseline  the fp64 oracle timed on the host cores on a bounded sample;
  clocks        SM clocks and throttle reasons sampled during the timed region.

With N > 1 (torchrun) every rank runs its own full replica of the workload (weak
scaling, no collective on the data path).  ``--impl reference`` times the fp64 oracle
instead (rank 0 only; other ranks exit 0 at once).
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import datetime
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode-step µs and KV-read GB/s (% of GB300 HBM peak), GQA 128K ctx"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 << 20          # GB300 L2 as the runtime reports it
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["fd", "reference"], default="fd")
    ap.add_argument("--config", type=int, default=3, help="workload number (1-5)")
    ap.add_argument("--num-splits", type=int, default=0, help="0 = library heuristic")
    ap.add_argument("--path", choices=["auto", "simt", "mma", "tcgen05"], default="auto")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="KV cache storage: the workload's own, or FP8 E4M3 codes with "
                         "per-kv-head scales (decode over the quantised cache)")
    ap.add_argument("--query-tokens", type=int, default=1,
                    help="Q > 1: multi-token decode (speculative verification) of Q query "
                         "tokens per row over the same cache, causal inside the split")
    ap.add_argument("--no-graph", action="store_true",
                    help="issue every timed call from Python instead of replaying CUDA graphs")
    ap.add_argument("--batch", type=int, default=0,
                    help="with --context: a large-batch serving workload of B full rows "
                         "(Hq 32, Hkv 8, d 128) instead of --config")
    ap.add_argument("--context", type=int, default=0, help="tokens per row for --batch")
    return ap.parse_args()


def base_workload(args):
    """The workload the arms run: --config N, or a serving batch (--batch, --context)."""
    if args.batch or args.context:
        if args.batch <= 0 or args.context <= 0:
            raise SystemExit("--batch and --context go together, both > 0")
        return workloads.serving_case(args.batch, args.context)
    return workloads.CONFIGS[args.config]()


# ----------------------------------------------------------------------------- helpers

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device=None) -> float:
    """The maximum of `value` over all ranks (the job is as slow as its slowest rank);
    the value itself when there is no process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy, burst)"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


KERNEL_SOURCES = {
    "fd_partial_mma_kernel": ["fd_partial_mma.cu", "fd_pipeline.cuh", "fd_epilogue.cuh",
                              "fd_device.cuh", "fd_internal.h"],
    "fd_partial_heads_kernel": ["fd_partial_mma.cu", "fd_pipeline.cuh", "fd_epilogue.cuh",
                                "fd_device.cuh", "fd_internal.h"],
    "fd_partial_persist_kernel": ["fd_partial_mma.cu", "fd_pipeline.cuh", "fd_epilogue.cuh",
                                  "fd_device.cuh", "fd_internal.h"],
    "fd_partial_heads_persist_kernel": ["fd_partial_mma.cu", "fd_pipeline.cuh",
                                        "fd_epilogue.cuh", "fd_device.cuh", "fd_internal.h"],
    "fd_partial_wide_persist_kernel": ["fd_partial_mma.cu", "fd_pipeline.cuh",
                                       "fd_epilogue.cuh", "fd_device.cuh", "fd_internal.h"],
    "fd_partial_simt_kernel": ["fd_partial_simt.cu", "fd_partial_simt.cuh", "fd_pipeline.cuh",
                               "fd_epilogue.cuh", "fd_device.cuh", "fd_internal.h"],
    "fd_partial_wide_kernel": ["fd_partial_mma.cu", "fd_pipeline.cuh", "fd_epilogue.cuh",
                               "fd_device.cuh", "fd_internal.h"],
    "fd_partial_tc_kernel": ["fd_partial_tc.cu", "fd_pipeline.cuh", "fd_epilogue.cuh",
                             "fd_device.cuh", "fd_internal.h"],
}


def _code_only(text: str) -> str:
    """C/CUDA source without comments and with whitespace runs collapsed, so that an
    ncu record stays tied to the code and not to its comments."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code of the source files that define `kernel` (ties an ncu record to
    them; comments and layout do not count)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_05_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            rec = json.load(f)
        e = rec["entries"][kernel + "|" + workload]
        if e["source_hash"] != kernel_source_hash(kernel):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:  # noqa: BLE001
        return None


class ClockSampler:
    """nvidia-smi in the background (20 ms period); keeps samples inside a window."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:  # noqa: BLE001
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:  # noqa: BLE001
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = []
        for line in self.out.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.out.name)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        if not inside and rows:                       # region shorter than the period
            inside = sorted(rows, key=lambda r: abs(r[0] - 0.5 * (t0 + t1)))[:3]
        if not inside:
            return None
        mhz = sorted(r[1] for r in inside)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": inside[0][2], "reasons": reasons,
                "samples": len(inside)}


def fp8_variant(w):
    """The workload with its K/V cache quantised to FP8 E4M3 codes (per-kv-head scales);
    returns (workload, k_scale, v_scale)."""
    kc, vc, ks, vs = workloads.fp8_quantize(w)
    w8 = dataclasses.replace(w, name=w.name + ", FP8 E4M3 KV", k=kc, v=vc)
    return w8, ks, vs


def with_query_tokens(w, Q: int):
    """The workload with Q query tokens per row (multi-token decode): q [B, Q, Hq, d]
    drawn from its own seed; the cache is unchanged."""
    if Q <= 1:
        return w
    q4 = workloads.multi_token_queries(w.B, Q, w.Hq, w.d, seed=4242, dtype=w.q.dtype)
    return dataclasses.replace(w, q=q4, name="%s, %d query tokens" % (w.name, Q))


def oracle_decoder(w, scales=None):
    """(decode(seq_lens, rows), seq_lens) running the oracle on the workload's stored
    values: the bf16/f32 decode (causal for multi-token queries), or the FP8 one when
    scales are given."""
    import oracle
    if scales is None:
        q, k, v, lens, bt, ps = w.oracle_arrays()
        fn = oracle.decode_causal if w.Q > 1 else oracle.decode
        return (lambda seq, rows=None: fn(q, k, v, seq, block_table=bt, page_size=ps,
                                          rows=rows)), lens
    q = workloads.np_storage(w.q)
    kc = w.k.view(torch.uint8).numpy()
    vc = w.v.view(torch.uint8).numpy()
    ks, vs = scales[0].numpy(), scales[1].numpy()
    lens = w.seq_lens.numpy()
    bt = None if w.block_table is None else w.block_table.numpy()
    ps = w.page_size
    return (lambda seq, rows=None: oracle.decode_kv8(q, kc, vc, ks, vs, seq, block_table=bt,
                                                      page_size=ps, rows=rows)), lens


def oracle_sample(w, budget_s: float, scales=None):
    """Time the fp64 oracle (as it stands) on a bounded sample of the workload.

    If a whole step fits the budget, whole steps are repeated until about `budget_s`
    seconds of work are done and the median step is kept.  Otherwise the sample is
    every query head over the first `tokens` keys (uniform lengths) or a subset of the
    query heads (ragged lengths), scaled to a step.  Returns (KV GB/s in the step's
    terms, threads used, sample description, seconds of work, step seconds)."""
    import statistics

    import oracle
    run, lens = oracle_decoder(w, scales)
    threads = oracle.max_threads()
    n_rows = w.B * w.Q * w.Hq
    L = int(lens.max())
    uniform = int(lens.min()) == L

    def timed(seq, rows=None):
        t0 = time.perf_counter()
        run(seq, rows)
        return time.perf_counter() - t0

    probe_tokens = min(L, 2048)
    if uniform:
        sl = lens.copy()
        sl[:] = probe_tokens
        est_step = timed(sl) * L / probe_tokens
    else:
        probe_rows = list(range(0, n_rows, max(1, n_rows // threads)))[:threads]
        est_step = timed(lens, probe_rows) * n_rows / len(probe_rows)
    if est_step <= budget_s:
        times = [timed(lens)]
        while sum(times) < budget_s and len(times) < 100000:
            times.append(timed(lens))
        step_s = statistics.median(times)
        work = sum(times)
        desc = "whole step (all %d query heads, all keys) x%d, median; %.1f s of work" % (
            n_rows, len(times), work)
    elif uniform:
        tokens = max(probe_tokens, int(L * budget_s / est_step))
        sl = lens.copy()
        sl[:] = tokens
        work = timed(sl)
        step_s = work * L / tokens
        desc = "all %d query heads x first %d of %d keys, scaled to a step; %.1f s of work" % (
            n_rows, tokens, L, work)
    else:
        keep = max(1, int(n_rows * budget_s / est_step))
        rows = list(range(0, n_rows, max(1, n_rows // keep)))[:keep]
        work = timed(lens, rows)
        step_s = work * n_rows / len(rows)
        desc = "%d of %d query heads, all keys, scaled to a step; %.1f s of work" % (
            len(rows), n_rows, work)
    gbs = w.kv_bytes() / step_s / 1e9
    return gbs, threads, desc, work, step_s


# ----------------------------------------------------------------------------- arms

REFERENCE_BUDGET_S = 240.0     # the whole reference arm (warm-up + timed steps)


def run_reference(args):
    """The oracle as the reference arm: whole steps of the workload (every query row,
    every key) when warm-up + timed steps fit REFERENCE_BUDGET_S, else each step is a
    bounded sample (a subset of the query rows, and of the keys if need be) scaled to a
    step."""
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    w = with_query_tokens(base_workload(args), args.query_tokens)
    scales = None
    if args.kv == "fp8":
        w, ks, vs = fp8_variant(w)
        scales = (ks, vs)
    import oracle
    run, lens = oracle_decoder(w, scales)
    threads = oracle.max_threads()
    n_rows = w.B * w.Q * w.Hq                    # query rows: B x Q x Hq
    L = int(lens.max())
    calls = args.steps + args.warmup
    t0 = time.perf_counter()
    run(lens)                                    # one whole step, also the first warm-up
    est_step = time.perf_counter() - t0
    if calls * est_step <= REFERENCE_BUDGET_S:
        sl, rows, frac = lens, None, 1.0
        sample = "whole step (all %d query rows, all keys)" % n_rows
        same = True
    else:
        per_step = REFERENCE_BUDGET_S / calls
        keep = max(1, min(n_rows, int(n_rows * per_step / est_step)))
        rows = list(range(0, n_rows, max(1, n_rows // keep)))[:keep]
        row_frac = len(rows) / n_rows
        tokens = L
        if est_step * row_frac > per_step:       # even one row per thread is too long
            tokens = int(max(16, min(L, L * per_step / (est_step * row_frac))))
        sl = lens.copy()
        sl[:] = [min(int(x), tokens) for x in lens]
        frac = row_frac * (tokens / L)
        sample = "%d of %d query rows x first %d of %d keys per step (%.5f of a step)" % (
            len(rows), n_rows, tokens, L, frac)
        same = False
    for _ in range(max(0, args.warmup - 1)):
        run(sl, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(sl, rows)
    elapsed = time.perf_counter() - t0
    step_s = elapsed / args.steps / frac
    gbs = w.kv_bytes() / step_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 3), "us_per_step": round(step_s * 1e6, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "sample": sample, "same_config": same},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_fd(args):
    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import decode_attention_05_gb300 as fd
    from decode_attention_05_gb300._binding import tensor_desc
    L = fd.lib()
    fd.set_path({"auto": fd.FD_PATH_AUTO, "simt": fd.FD_PATH_SIMT, "mma": fd.FD_PATH_MMA,
                 "tcgen05": fd.FD_PATH_TCGEN05}[args.path])

    w_cpu = with_query_tokens(base_workload(args), args.query_tokens)
    scales_cpu = None
    if args.kv == "fp8":
        if w_cpu.Q > 1:
            raise SystemExit("--kv fp8 takes single-token decode only")
        w_cpu, ks, vs = fp8_variant(w_cpu)
        scales_cpu = (ks, vs)
    w = w_cpu.to("cuda")
    scales = None if scales_cpu is None else tuple(t.cuda() for t in scales_cpu)
    B, Hq, d, Hkv, Qt = w.B, w.Hq, w.d, w.Hkv, w.Q
    rows = Qt * (Hq // Hkv)                           # query rows per (b, kv head)
    kernel = fd.partial_kernel_name(w.q.dtype, w.k.dtype, d, Hkv, w.page_size, rows=rows)
    S = args.num_splits or w.num_splits
    if S == 0:          # the lengths are known here: plan with them
        sms = torch.cuda.get_device_properties(local).multi_processor_count
        # The planner models the single-token kernels (two CTAs per SM, bound by HBM).  The
        # kernels of wide groups are bound by their tile math and do best with one CTA's
        # worth of splits per SM (the tcgen05 kernel holds one CTA per SM; the mma.sync
        # wide kernel measured 132 us at 19 splits against 156 us at 32 on the 128K cache).
        wide = kernel in ("fd_partial_tc_kernel", "fd_partial_wide_kernel")
        S = fd.num_splits_for_lengths(B, Hq, Hkv, d, w.L_cap, w_cpu.seq_lens,
                                      sms // 2 if wide else sms, page_size=w.page_size)
    # The kernel this call runs, now that the batch and the split count are known (large
    # batches take head groups, short rows the persistent schedule).
    kernel = fd.partial_kernel_name_for(w.q.dtype, w.k.dtype, B, Qt, Hq, Hkv, d, w.page_size,
                                        w.L_cap, S) or kernel
    ws = torch.zeros(fd.workspace_size(B, Qt * Hq, Hkv, d, S), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(tuple(w.q.shape), dtype=w.out_dtype, device="cuda")
    lse = torch.empty(tuple(w.q.shape[:-1]), dtype=torch.float32, device="cuda")
    dq, dk, dv, dbt, do = (tensor_desc(w.q), tensor_desc(w.k), tensor_desc(w.v),
                           tensor_desc(w.block_table), tensor_desc(out))
    bt_ref = None if dbt is None else ctypes.byref(dbt)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream or None
    ws_bytes = ws.numel()
    # A cache smaller than three L2s is streamed from alternating copies, so that no
    # step finds the previous step's KV in L2.
    kv_bytes = w.kv_bytes()
    n_sets = 2 if kv_bytes < 3 * L2_BYTES else 1
    kv_sets = [(w.k, w.v)] + [(w.k.clone(), w.v.clone()) for _ in range(n_sets - 1)]
    kv_descs = [(tensor_desc(k), tensor_desc(v)) for k, v in kv_sets]
    if scales is None:
        decode_fn, partial_fn = L.fd_decode_attention, L.fd_decode_partial
        kv_args = [(ctypes.byref(dq), ctypes.byref(dk_), ctypes.byref(dv_))
                   for dk_, dv_ in kv_descs]
    else:
        decode_fn, partial_fn = L.fd_decode_attention_fp8kv, L.fd_decode_partial_fp8kv
        kv_args = [(ctypes.byref(dq), ctypes.byref(dk_), ctypes.byref(dv_), scales[0].data_ptr(),
                    scales[1].data_ptr()) for dk_, dv_ in kv_descs]
    step_args = [a + (w.seq_lens.data_ptr(), bt_ref, w.page_size, S, ctypes.byref(do),
                      lse.data_ptr(), ws.data_ptr(), ws_bytes) for a in kv_args]
    turn = [0]

    def next_set():
        i = turn[0] % n_sets
        turn[0] += 1
        return i

    def step():
        st = decode_fn(*step_args[next_set()], sh)
        if st:
            raise fd.FdError(st, L.fd_last_error().decode())

    # Timed loops replay a CUDA graph of GRAPH_CHUNK back-to-back calls (as a decode loop
    # would run them), so that the host's per-call cost stays out of the device time;
    # exactly n calls are issued either way.  call(stream_handle) issues one call.
    GRAPH_CHUNK = 100

    def checked(st):
        if st:
            raise fd.FdError(st, L.fd_last_error().decode())

    # A run shorter than GRAPH_CHUNK steps replays one graph of exactly `steps` calls.
    chunk = max(1, min(GRAPH_CHUNK, args.steps))

    def make_graph(call, chunk):
        if args.no_graph:
            return None
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for _ in range(2):
                call(cap.cuda_stream)
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for _ in range(chunk):
                call(cap.cuda_stream)
        torch.cuda.synchronize()
        return g

    def issue(call, graph, n):
        if graph is None:
            for _ in range(n):
                call(sh)
            return
        for _ in range(n // chunk):
            graph.replay()
        for _ in range(n % chunk):
            call(sh)

    def launch_label(n):
        """What issue(call, graph, n) does, in words."""
        if args.no_graph:
            return "%d direct calls from Python (no CUDA graph)" % n
        text = "CUDA graph of %d back-to-back decode calls, replayed %d time%s" % (
            chunk, n // chunk, "" if n // chunk == 1 else "s")
        if n % chunk:
            text += ", then %d direct calls" % (n % chunk)
        return text

    step_call = lambda s: checked(decode_fn(*step_args[next_set()], s))

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        step()
    step_graph = make_graph(step_call, chunk)
    if step_graph is not None:
        step_graph.replay()
    if fd.read_device_error(ws) != 0:
        raise RuntimeError("device error flags set during warm-up")

    sampler = ClockSampler(local)
    time.sleep(0.3)                                   # let nvidia-smi start sampling
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    issue(step_call, step_graph, args.steps)
    e1.record(stream)
    e1.synchronize()
    t_wall1 = time.time()
    barrier()
    ms = e0.elapsed_time(e1)
    clocks = sampler.stop(t_wall0, t_wall1)
    ms = max_over_ranks(ms, device="cuda")
    ms_per_step = ms / args.steps
    value = world * kv_bytes * args.steps / (ms * 1e-3) / 1e9

    # ---- roofline of the dominant kernel: the partial pass alone, K launches
    partial_args = [a + (w.seq_lens.data_ptr(), bt_ref, w.page_size, S, ws.data_ptr(), ws_bytes)
                    for a in kv_args]
    partial_call = lambda s: checked(partial_fn(*partial_args[next_set()], s))
    for _ in range(3):
        partial_call(sh)
    partial_graph = make_graph(partial_call, chunk)
    barrier()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    issue(partial_call, partial_graph, args.steps)
    e3.record(stream)
    e3.synchronize()
    partial_ms = e2.elapsed_time(e3) / args.steps
    merge_ms = 0.0          # one split: the step's partial pass writes the output itself
    if S > 1:
        lse_part, o_part = fd.workspace_partials(ws, B * Qt, Hq, d, S)
        dout = tensor_desc(out.view(B * Qt, Hq, d))
        merge_call = lambda s: checked(L.fd_merge_partials(B * Qt, Hq, d, S, lse_part.data_ptr(),
                                                           o_part.data_ptr(), ctypes.byref(dout),
                                                           lse.data_ptr(), s))
        merge_graph = make_graph(merge_call, chunk)
        barrier()
        e4, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e4.record(stream)
        issue(merge_call, merge_graph, args.steps)
        e5.record(stream)
        e5.synchronize()
        merge_ms = e4.elapsed_time(e5) / args.steps
    peak, peak_src = measured_peak()
    achieved = kv_bytes / (partial_ms * 1e-3) / 1e9
    path_name = {"fd_partial_simt_kernel": "simt", "fd_partial_tc_kernel": "tcgen05"}.get(kernel, "mma")
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(kernel, w.name),
                "kernel": kernel, "peak_source": peak_src,
                "algorithmic_bytes_per_launch": kv_bytes,
                "partial_us": round(partial_ms * 1e3, 2), "merge_us": round(merge_ms * 1e3, 2),
                "launch": launch_label(args.steps)}
    if S == 1:
        roofline["merge"] = ("none in the step: with one split the partial pass writes the "
                             "output; partial_us times the partials-only pass")

    # ---- end to end through the public API, host buffers, copies inside the timed region
    pin = lambda t: t.pin_memory()
    qh, kh, vh, sh_lens = pin(w_cpu.q), pin(w_cpu.k), pin(w_cpu.v), pin(w_cpu.seq_lens)
    scales_h = () if scales_cpu is None else tuple(pin(t) for t in scales_cpu)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh, sh_lens) + scales_h)
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()

    def e2e_step():
        w.q.copy_(qh, non_blocking=True)
        w.k.copy_(kh, non_blocking=True)
        w.v.copy_(vh, non_blocking=True)
        w.seq_lens.copy_(sh_lens, non_blocking=True)
        if scales is None:
            fd.decode_attention(w.q, w.k, w.v, w.seq_lens, w.block_table, w.page_size, S,
                                out=out, lse_out=lse, workspace=ws)
        else:
            for dst, src in zip(scales, scales_h):
                dst.copy_(src, non_blocking=True)
            fd.decode_attention_fp8kv(w.q, w.k, w.v, scales[0], scales[1], w.seq_lens,
                                      w.block_table, w.page_size, S, out=out, lse_out=lse,
                                      workspace=ws)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    barrier()
    e6, e7 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e6.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e7.record(stream)
    e7.synchronize()
    e2e_ms = e6.elapsed_time(e7) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, device="cuda")
    e2e = {"value": round(world * kv_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e2e_ms, 3)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, cores, desc, _, step_s = oracle_sample(w_cpu, args.cpu_budget_s, scales_cpu)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": desc, "step_ms_extrapolated": round(step_s * 1e3, 1)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "us_per_step": round(ms_per_step * 1e3, 2),
            "hbm_frac_step": round(value / world / peak, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("bf16" if w.q.dtype == torch.bfloat16 else "f32") +
                     ("+e4m3 KV" if scales is not None else ""),
            "data": "synthetic",
            "config": {"workload": w.name, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d,
                       "query_tokens": Qt,
                       "L": int(w.seq_lens.max()), "num_splits": S, "path": path_name,
                       "kv_bytes_per_step": kv_bytes,
                       "l2": ("inputs larger than L2 (KV %d MiB vs 126 MiB L2), no flush" %
                              (kv_bytes >> 20) if n_sets == 1 else
                              "KV %d MiB < 3 x 126 MiB L2: steps alternate between %d copies "
                              "of the cache, no flush" % (kv_bytes >> 20, n_sets)),
                       "parallelism": "replicas x%d" % world,
                       "launch": launch_label(args.steps)},
            "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks,
            "gpu_launches": 2 * args.steps,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_fd(args)


if __name__ == "__main__":
    sys.exit(main())
