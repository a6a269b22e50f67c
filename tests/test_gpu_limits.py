"""Parity at the size limits: a million-token row, thousands of batch rows, many kv
heads, the largest page size and the largest split count, each against the fp64
oracle on every output."""
import pytest
import torch

import workloads
from test_gpu_parity import check, ref_for

pytestmark = pytest.mark.gpu

fd = pytest.importorskip("decode_attention_05_gb300")


def _decode(w, S):
    wd = w.to("cuda")
    B, Hq, d = w.q.shape
    S_res = fd.resolve_num_splits(B, Hq, w.Hkv, d, w.L_cap, S)
    ws = torch.zeros(fd.workspace_size(B, Hq, w.Hkv, d, S_res), dtype=torch.uint8, device="cuda")
    o, l = fd.decode_attention(wd.q, wd.k, wd.v, wd.seq_lens, wd.block_table, wd.page_size, S,
                               workspace=ws, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fd.read_device_error(ws) == 0
    return o.cpu().double().numpy(), l.cpu().double().numpy()


def test_million_token_row():
    L = 1 << 20
    w = workloads.contiguous_case(1, 8, 1, 64, L, [L], seed=701, poison_tail=False,
                                  out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    for S in (0, 4096):
        o, l = _decode(w, S)
        check(w, o, l, ref_o, ref_l)


def test_many_batch_rows():
    B = 2048
    g = torch.Generator().manual_seed(702)
    lens = torch.randint(0, 129, (B,), generator=g).tolist()
    w = workloads.contiguous_case(B, 8, 2, 128, 128, lens, seed=702, out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    for S in (1, 3):
        o, l = _decode(w, S)
        check(w, o, l, ref_o, ref_l)


def test_many_kv_heads():
    w = workloads.contiguous_case(2, 64, 64, 128, 1500, [1500, 777], seed=703,
                                  out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    o, l = _decode(w, 0)
    check(w, o, l, ref_o, ref_l)


def test_largest_page_size():
    w = workloads.paged_case(2, 16, 4, 128, 65536, 2, [131072, 70000], seed=704,
                             out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    for S in (0, 3):
        o, l = _decode(w, S)
        check(w, o, l, ref_o, ref_l)


def test_max_splits_with_a_batch():
    w = workloads.contiguous_case(16, 8, 2, 64, 8192, [8192, 1, 0, 4097] * 4, seed=705,
                                  out_dtype=torch.float32)
    ref_o, ref_l = ref_for(w)
    o, l = _decode(w, 4096)
    check(w, o, l, ref_o, ref_l)
