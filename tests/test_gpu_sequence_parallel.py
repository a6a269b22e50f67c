"""sequence_parallel.sp_decode_attention end to end on one GPU, with a world-size-1
NCCL process group: its split resolution and workspace sizing, the partial pass, the
all-gather of the partials and the merge, against the fp64 oracle ("AI Infra: math and
infra optimisation in large models", section 2.6 "Sequence Parallelism": each shard
hands over only its partial outputs and one LSE per row).  A row whose shard is empty
(length 0) gets weight 0 and out = 0, lse = -inf.  The two-rank exchange itself is
covered by the gloo test in test_multiprocess.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
import workloads

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")
from decode_attention_05_gb300 import sequence_parallel as sp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture
def nccl_group():
    if not dist.is_nccl_available():
        pytest.skip("torch was built without NCCL")
    torch.cuda.set_device(0)
    created = not dist.is_initialized()
    if created:
        dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % _free_port(),
                                rank=0, world_size=1, device_id=torch.device("cuda", 0))
    yield None
    if created:
        dist.destroy_process_group()


@pytest.mark.parametrize("num_splits", [0, 5])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_sp_decode_attention_one_rank(nccl_group, num_splits, out_dtype):
    w_cpu = workloads.contiguous_case(3, 32, 4, 128, 4096, [4096, 0, 1234], seed=71,
                                      out_dtype=out_dtype)
    q, k, v, lens, bt, ps = w_cpu.oracle_arrays()
    ref_o, ref_l = oracle.decode(q, k, v, lens)
    w = w_cpu.to("cuda")
    out, lse = sp.sp_decode_attention(w.q, w.k, w.v, w.seq_lens, num_splits,
                                      group=nccl_group, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert out.dtype == out_dtype
    got_o = out.double().cpu().numpy()
    got_l = lse.double().cpu().numpy()
    assert not np.isnan(got_o).any() and not np.isnan(got_l).any()
    assert (np.abs(got_o - ref_o) <= 4e-3 + 8e-3 * np.abs(ref_o)).all()
    empty = np.isneginf(ref_l)
    assert empty[1].all() and not empty[0].any()          # row 1's shard holds no key
    assert np.array_equal(np.isneginf(got_l), empty)
    assert (got_o[empty] == 0).all()
    assert (np.abs(got_l[~empty] - ref_l[~empty]) <= 1e-4 + 1e-5 * np.abs(ref_l[~empty])).all()


def test_sp_decode_attention_paged_shard(nccl_group):
    w_cpu = workloads.paged_case(2, 16, 2, 128, 64, 40, [2500, 63], seed=72,
                                 out_dtype=torch.float32)
    q, k, v, lens, bt, ps = w_cpu.oracle_arrays()
    ref_o, ref_l = oracle.decode(q, k, v, lens, block_table=bt, page_size=ps)
    w = w_cpu.to("cuda")
    out, lse = sp.sp_decode_attention(w.q, w.k, w.v, w.seq_lens, 0, group=nccl_group,
                                      block_table=w.block_table, page_size=64)
    torch.cuda.synchronize()
    got_o = out.double().cpu().numpy()
    assert (np.abs(got_o - ref_o) <= 4e-3 + 8e-3 * np.abs(ref_o)).all()
    assert (np.abs(lse.double().cpu().numpy() - ref_l) <= 1e-4 + 1e-5 * np.abs(ref_l)).all()
