"""Seeded synthetic inputs for decode attention: the five workloads and small cases.

This module only draws and lays out inputs.  It holds none of the method's
arithmetic: it never computes a score, a softmax, an LSE or an output.  Both the
CUDA path and the fp64 oracle read the tensors it returns; neither imports the
other.

Recipe (every workload): values are drawn with ``torch.Generator`` on the CPU in
fp32 from a fixed seed, then cast to the storage dtype (bf16 round-to-nearest-even
or fp32).  The oracle reads the same stored values, widened exactly to fp64.

  1 tiny fp32      B=1 Hq=Hkv=1 d=64 L=257, S=4 (splits 65/65/65/62); N(0,1); seed 1001
  2 MHA bf16       B=4 Hq=Hkv=32 d=128 L=4096 contiguous; N(0,1); seed 1002
  3 GQA 128K bf16  B=1 Hq=64 Hkv=8 d=128 L=131072 contiguous; N(0,1); seed 1003
  4 ragged paged   B=16 Hq=32 Hkv=8 d=128; seq_lens ~ U{1..32768} with two forced short
                   rows (1 and 37 tokens); page_size=16; a pool of exactly
                   sum(ceil(L_b/16)) pages placed by a seeded random permutation;
                   block table int32 [16, 2048] with -1 past each row's pages; the
                   stale slots past L_b in each row's last page hold NaN; seed 1004
  5 adversarial    B=8 Hq=32 Hkv=8 d=128 L=16384 contiguous; K ~ N(0,1) with 4 spike
                   tokens per (b, kv head): t_j = 4096 j + r_j, r_j < 2048, and
                   k[t_j] = 120 sqrt(d) q_h / |q_h|^2 for h = g G + j, so that head's
                   score is ~120 (before bf16 rounding of k); V[t] = N(0,1) + t/L
                   (every row distinct); splits S in {1, 8, 64, 256}; seed 1005
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor                     # [B, Hq, d] (or [B, Q, Hq, d]: Q query tokens) CPU
    k: torch.Tensor                     # contiguous [B, Hkv, L_cap, d] | paged [P, Hkv, ps, d]
    v: torch.Tensor
    seq_lens: torch.Tensor              # int32 [B]
    block_table: Optional[torch.Tensor] = None   # int32 [B, max_pages] (paged only)
    page_size: int = 0
    num_splits: int = 0                 # 0 -> the library's heuristic
    split_sweep: tuple = ()             # extra split counts the parity tests sweep
    out_dtype: torch.dtype = torch.bfloat16

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def Hq(self) -> int:
        return self.q.shape[-2]

    @property
    def d(self) -> int:
        return self.q.shape[-1]

    @property
    def Q(self) -> int:
        """Query tokens per row (multi-token decode), 1 for single-token decode."""
        return self.q.shape[1] if self.q.dim() == 4 else 1

    @property
    def Hkv(self) -> int:
        return self.k.shape[1]

    @property
    def L_cap(self) -> int:
        if self.block_table is None:
            return self.k.shape[2]
        return self.block_table.shape[1] * self.page_size

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one decode step must read: sum_b L_b * Hkv * d * 2 (K, V)."""
        return int(self.seq_lens.to(torch.int64).sum()) * self.Hkv * self.d * 2 * self.k.element_size()

    def oracle_arrays(self):
        """numpy views for the oracle: fp32 as float32, bf16 as raw uint16 bit patterns."""
        def np_view(t):
            t = t.contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
        bt = None if self.block_table is None else self.block_table.numpy()
        return (np_view(self.q), np_view(self.k), np_view(self.v), self.seq_lens.numpy(), bt,
                self.page_size)

    def to(self, device) -> "Workload":
        def mv(t):
            return None if t is None else t.to(device)
        return dataclasses.replace(self, q=mv(self.q), k=mv(self.k), v=mv(self.v),
                                   seq_lens=mv(self.seq_lens), block_table=mv(self.block_table))


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _randn(g, shape, dtype):
    return torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)


def contiguous_case(B, Hq, Hkv, d, L_cap, seq_lens=None, *, seed, dtype=torch.bfloat16,
                    num_splits=0, poison_tail=True, out_dtype=None, name=None) -> Workload:
    """A contiguous-cache case with N(0,1) q, K, V.  Cache slots at or past each row's
    length hold NaN when ``poison_tail`` (stale slots the length mask must exclude)."""
    g = _gen(seed)
    q = _randn(g, (B, Hq, d), dtype)
    k = _randn(g, (B, Hkv, L_cap, d), dtype)
    v = _randn(g, (B, Hkv, L_cap, d), dtype)
    if seq_lens is None:
        seq_lens = [L_cap] * B
    lens = torch.tensor(seq_lens, dtype=torch.int32)
    if poison_tail:
        for b, L in enumerate(seq_lens):
            k[b, :, L:] = float("nan")
            v[b, :, L:] = float("nan")
    return Workload(name or "contiguous", q, k, v, lens, num_splits=num_splits,
                    out_dtype=out_dtype or dtype)


def paged_case(B, Hq, Hkv, d, page_size, max_pages, seq_lens, *, seed, dtype=torch.bfloat16,
               num_splits=0, extra_pages=0, out_dtype=None, name=None) -> Workload:
    """A paged case: a pool of sum(ceil(L_b/ps)) (+ extra) pages in a seeded random
    physical order; block table int32 [B, max_pages], -1 past each row's pages; the
    slots past L_b in a row's last page hold NaN."""
    g = _gen(seed)
    lens = [int(x) for x in seq_lens]
    pages_per_row = [-(-L // page_size) for L in lens]
    P = sum(pages_per_row) + extra_pages
    q = _randn(g, (B, Hq, d), dtype)
    k = _randn(g, (max(P, 1), Hkv, page_size, d), dtype)
    v = _randn(g, (max(P, 1), Hkv, page_size, d), dtype)
    perm = torch.randperm(max(P, 1), generator=g)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    nxt = 0
    for b in range(B):
        for i in range(pages_per_row[b]):
            table[b, i] = int(perm[nxt])
            nxt += 1
        tail = lens[b] % page_size
        if tail and pages_per_row[b]:
            last = int(table[b, pages_per_row[b] - 1])
            k[last, :, tail:] = float("nan")
            v[last, :, tail:] = float("nan")
    return Workload(name or "paged", q, k, v, torch.tensor(lens, dtype=torch.int32), table,
                    page_size, num_splits=num_splits, out_dtype=out_dtype or dtype)


def multi_token_queries(B: int, Q: int, Hq: int, d: int, *, seed: int,
                        dtype=torch.bfloat16) -> torch.Tensor:
    """Queries for multi-token decode: [B, Q, Hq, d], N(0,1), drawn from their own seed."""
    return _randn(_gen(seed), (B, Q, Hq, d), dtype)


def np_storage(t: torch.Tensor) -> np.ndarray:
    """A tensor as the oracle reads it: fp32 as float32, bf16 as raw uint16 bits."""
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def fp8_quantize(w: Workload, power_of_two_scales: bool = False):
    """An FP8 E4M3 copy of a workload's K and V with one scale per kv head for each:
    scale = amax(|x|) of that head / 448 (the largest E4M3 value), codes = x / scale
    rounded to E4M3 by torch.  NaN stale slots stay NaN codes.  With
    `power_of_two_scales` the scales are rounded up to powers of two, so that
    code * scale is exact in fp32.  Returns (k_codes, v_codes, k_scale, v_scale)."""
    def quant(x):
        x = x.float()
        head_dim = 1                                   # [B|P, Hkv, rows, d]
        amax = torch.nan_to_num(x.abs(), nan=0.0).amax(dim=(0, 2, 3)).clamp_min(1e-12)
        scale = amax / 448.0
        if power_of_two_scales:
            scale = torch.exp2(torch.ceil(torch.log2(scale)))
        shape = [1] * x.dim()
        shape[head_dim] = -1
        codes = (x / scale.view(shape)).to(torch.float8_e4m3fn)
        return codes, scale.to(torch.float32)
    kc, ks = quant(w.k)
    vc, vs = quant(w.v)
    return kc, vc, ks, vs


def worked_example(d: int = 64) -> Workload:
    """The pages' counter-example as one fp32 attention row: q = 80 e_0, k_0 = k_1 = 0,
    k_2 = e_0 (scores [0, 0, 10] at scale 1/8); values 0, 0, 9 in every dim; S = 2,
    which splits the three keys [2 | 1]."""
    q = torch.zeros(1, 1, d)
    q[0, 0, 0] = 80.0
    k = torch.zeros(1, 1, 3, d)
    k[0, 0, 2, 0] = 1.0
    v = torch.zeros(1, 1, 3, d)
    v[0, 0, 2, :] = 9.0
    return Workload("worked-example", q, k, v, torch.tensor([3], dtype=torch.int32),
                    num_splits=2, out_dtype=torch.float32)


def config1() -> Workload:
    w = contiguous_case(1, 1, 1, 64, 257, seed=1001, dtype=torch.float32, num_splits=4,
                        poison_tail=False, out_dtype=torch.float32,
                        name="tiny fp32 B1 H1 d64 L257 S4")
    return w


def config2() -> Workload:
    return contiguous_case(4, 32, 32, 128, 4096, seed=1002, poison_tail=False,
                           name="MHA bf16 B4 H32 d128 L4096")


def config3() -> Workload:
    return contiguous_case(1, 64, 8, 128, 131072, seed=1003, poison_tail=False,
                           name="GQA bf16 B1 Hq64 Hkv8 d128 L131072")


def config4_lens(seed: int = 1004, B: int = 16, L_max: int = 32768) -> List[int]:
    g = _gen(seed)
    lens = torch.randint(1, L_max + 1, (B,), generator=g, dtype=torch.int64).tolist()
    lens[0] = 1            # a single-token row
    lens[1] = 37           # shorter than any split: every split but the first is empty
    return lens


def config4() -> Workload:
    lens = config4_lens()
    return paged_case(16, 32, 8, 128, 16, 2048, lens, seed=1004,
                      name="ragged paged GQA bf16 B16 Hq32 Hkv8 d128 ps16 L<=32768")


def serving_case(B: int, L: int, Hq: int = 32, Hkv: int = 8, d: int = 128) -> Workload:
    """A large-batch serving step: B rows of L tokens each (every row full), bf16,
    N(0,1), contiguous cache; seed 2000 + B.  Not one of the five workloads: a shape for
    the many-short-rows regime (bench.py --batch/--context)."""
    return contiguous_case(B, Hq, Hkv, d, L, seed=2000 + B, poison_tail=False,
                           name="serving bf16 B%d Hq%d Hkv%d d%d L%d" % (B, Hq, Hkv, d, L))


def config5(num_splits: int = 8) -> Workload:
    B, Hq, Hkv, d, L = 8, 32, 8, 128, 16384
    G = Hq // Hkv
    g = _gen(1005)
    q32 = torch.randn((B, Hq, d), generator=g, dtype=torch.float32)
    q = q32.to(torch.bfloat16)
    k32 = torch.randn((B, Hkv, L, d), generator=g, dtype=torch.float32)
    v32 = torch.randn((B, Hkv, L, d), generator=g, dtype=torch.float32)
    v32 += (torch.arange(L, dtype=torch.float32) / L).view(1, 1, L, 1)
    r = torch.randint(0, 2048, (B, Hkv, 4), generator=g)
    qb = q.to(torch.float32)       # the stored query the kernel sees
    for b in range(B):
        for kv in range(Hkv):
            for j in range(4):
                h = kv * G + j
                t = 4096 * j + int(r[b, kv, j])
                qh = qb[b, h]
                k32[b, kv, t] = 120.0 * math.sqrt(d) * qh / float(qh.dot(qh))
    return Workload("adversarial bf16 B8 Hq32 Hkv8 d128 L16384", q, k32.to(torch.bfloat16),
                    v32.to(torch.bfloat16), torch.full((B,), L, dtype=torch.int32),
                    num_splits=num_splits, split_sweep=(1, 8, 64, 256))


def config5_spikes(seed: int = 1005):
    """Spike token positions t[b, kv, j] of workload 5 (for tests that look at them)."""
    B, Hq, Hkv, d, L = 8, 32, 8, 128, 16384
    g = _gen(seed)
    torch.randn((B, Hq, d), generator=g)
    torch.randn((B, Hkv, L, d), generator=g)
    torch.randn((B, Hkv, L, d), generator=g)
    r = torch.randint(0, 2048, (B, Hkv, 4), generator=g)
    return torch.arange(4).view(1, 1, 4) * 4096 + r


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}
