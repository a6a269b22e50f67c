"""Pins that tie the fp64 oracle to facts fixed outside the oracle itself.

Each ``pin_*`` function takes a loaded oracle library handle (``oracle.load_library``)
and raises ``AssertionError`` when the oracle disagrees with:

* values the pages print (tests/golden/*.json, each with its citation);
* closed forms (one key, equal scores, a single dominant spike, empty sequence);
* invariants (constant score shift, split count, physical page permutation);
* an independent high-precision evaluation (Python ``decimal``, 40 digits, no
  max shift) on tiny shapes;
* a library special case (torch float64 CPU softmax / logsumexp / SDPA with the
  KV heads repeated per query group).

The pins are chosen so that a plausible slip in the oracle -- a dropped key, a
wrong sign, a wrong head index, a transposed operand, a missing scale or a wrong
log base -- breaks at least one of them; ``test_oracle_mutants.py`` checks that by
planting such slips in copies of the oracle source.
"""
from __future__ import annotations

import decimal
import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (input generation only)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _softmax_via_oracle(lib, logits):
    """Drive the attention oracle with d = 1 so that its softmax weights become outputs.

    Row b has q = [1], keys k_t = [z_t] (score z_t / sqrt(1)), and one-hot values
    v_t = [t == b]: the output of row b is then the weight of token b.
    """
    L = len(logits)
    q = np.ones((L, 1, 1), np.float32)
    k = np.tile(np.asarray(logits, np.float32).reshape(1, 1, L, 1), (L, 1, 1, 1))
    v = np.zeros((L, 1, L, 1), np.float32)
    for b in range(L):
        v[b, 0, b, 0] = 1.0
    out, lse = oracle.decode(q, k, v, np.full(L, L, np.int32), lib=lib)
    return out[:, 0, 0], lse[0, 0]


def pin_softmax_examples(lib):
    g = _golden("softmax_examples.json")
    for case in g["cases"]:
        p, _ = _softmax_via_oracle(lib, case["logits"])
        got = np.round(p, case["decimals"])
        assert np.allclose(got, case["probs"], atol=0.5 * 10.0 ** (-case["decimals"])), (case, p)
        assert abs(p.sum() - 1.0) < 1e-12
        if "equals_softmax_of" in case:
            p2, _ = _softmax_via_oracle(lib, case["equals_softmax_of"])
            assert np.allclose(p, p2, rtol=0, atol=1e-12)
    # A score of 120 must not overflow: the weight stays finite and exact.
    p, lse = _softmax_via_oracle(lib, [120.0, 0.0])
    assert np.all(np.isfinite(p)) and math.isfinite(lse)
    assert abs(math.exp(120.0) - g["exp_120_approx"]) <= g["exp_120_rel_tol"] * g["exp_120_approx"]
    assert math.exp(120.0) > g["fp16_max"]
    assert abs(lse - (120.0 + math.log1p(math.exp(-120.0)))) < 1e-12


def pin_worked_example(lib):
    """The pages' counter-example, as a d = 64 attention row: q = 80 e_0, k_0 = k_1 = 0,
    k_2 = e_0 give scores [0, 0, 10] at scale 1/8; values 0, 0, 9 in every dim."""
    g = _golden("worked_example.json")
    d = 64
    s, vals = g["scores"], g["values"]
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = 8.0 * s[2]
    k = np.zeros((1, 1, 3, d), np.float32)
    k[0, 0, 2, 0] = 1.0
    v = np.zeros((1, 1, 3, d), np.float32)
    for t in range(3):
        v[0, 0, t, :] = vals[t]
    out, lse = oracle.decode(q, k, v, np.array([3], np.int32), lib=lib)
    e10 = math.exp(10.0)
    closed_o = 9.0 * e10 / (2.0 + e10)          # the unsplit softmax average
    closed_lse = math.log(2.0 + e10)
    assert np.allclose(out[0, 0], closed_o, rtol=1e-13, atol=0)
    assert abs(lse[0, 0] - closed_lse) < 1e-12
    # The split [2 | 1] merged with LSE weights equals the unsplit answer ...
    sizes = g["split_sizes"]
    parts, lo = [], 0
    for n in sizes:
        parts.append(oracle.block_partial(s[lo:lo + n], vals[lo:lo + n]))
        lo += n
    assert [p[0] for p in parts] == g["block_outputs"]
    merged, merged_lse = oracle.merge_blocks(parts)
    assert math.isclose(merged, out[0, 0, 0], rel_tol=g["merged_equals_unsplit_rel_tol"])
    assert math.isclose(merged_lse, lse[0, 0], rel_tol=1e-12)
    # ... while the naive average of the block outputs is far off.
    naive = sum(p[0] for p in parts) / len(parts)
    assert naive == g["naive_average"]
    assert abs(naive - out[0, 0, 0]) > g["naive_average_error_exceeds"]


def pin_closed_forms(lib):
    rng = np.random.default_rng(11)
    d = 8
    # One key: o = v_0, lse = s_0.
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    k = rng.standard_normal((1, 1, 5, d)).astype(np.float32)
    v = rng.standard_normal((1, 1, 5, d)).astype(np.float32)
    out, lse = oracle.decode(q, k, v, np.array([1], np.int32), lib=lib)
    s0 = float(np.dot(q[0, 0].astype(np.float64), k[0, 0, 0].astype(np.float64))) / math.sqrt(d)
    assert np.allclose(out[0, 0], v[0, 0, 0], rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - s0) < 1e-12
    # Equal scores: o = mean of the L values, lse = s + ln L.
    L = 7
    kk = np.tile(k[:, :, :1, :], (1, 1, L, 1))
    vv = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    out, lse = oracle.decode(q, kk, vv, np.array([L], np.int32), lib=lib)
    assert np.allclose(out[0, 0], vv[0, 0].astype(np.float64).mean(axis=0), rtol=0, atol=1e-12)
    assert abs(lse[0, 0] - (s0 + math.log(L))) < 1e-12
    # One spike with gap D above every other score: |o - v_spike| <= (L-1) e^-D max|v|.
    L = 6
    qs = np.zeros((1, 1, d), np.float32)
    qs[0, 0, 0] = 1.0
    ks = np.zeros((1, 1, L, d), np.float32)
    ks[0, 0, 3, 0] = 12.0 * math.sqrt(d)          # score 12, all others 0
    vs = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    out, _ = oracle.decode(qs, ks, vs, np.array([L], np.int32), lib=lib)
    bound = (L - 1) * math.exp(-12.0) * np.abs(vs).max()
    err = np.abs(out[0, 0] - vs[0, 0, 3]).max()
    assert err <= bound and err > 0.0
    # Empty sequence: o = 0, lse = -inf (no fake block).
    out, lse = oracle.decode(q, k, v, np.array([0], np.int32), lib=lib)
    assert np.all(out[0, 0] == 0.0) and lse[0, 0] == -math.inf


def pin_shift_invariance(lib):
    """Adding c to every score leaves o unchanged and moves lse by c.  With q_0 = 2 and
    d = 16, adding 2c to component 0 of every key adds exactly c to every score; keys
    on a 1/64 grid keep that addition exact in fp32."""
    rng = np.random.default_rng(12)
    d, L = 16, 33
    q = (np.round(rng.standard_normal((1, 1, d)) * 64.0) / 64.0).astype(np.float32)
    q[0, 0, 0] = 2.0
    k = (np.round(rng.standard_normal((1, 1, L, d)) * 64.0) / 64.0).astype(np.float32)
    v = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    c = 37.5
    k2 = k.copy()
    k2[..., 0] += np.float32(2.0 * c)
    assert np.all(k2[..., 0].astype(np.float64) - k[..., 0].astype(np.float64) == 2.0 * c)
    o1, l1 = oracle.decode(q, k, v, np.array([L], np.int32), lib=lib)
    o2, l2 = oracle.decode(q, k2, v, np.array([L], np.int32), lib=lib)
    assert abs((l2[0, 0] - l1[0, 0]) - c) < 1e-12
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-13)


def pin_split_invariance(lib):
    """The oracle's unsplit row equals the LSE merge of split partials for several S,
    including uneven tails and S = L (one key per block); weights sum to 1."""
    rng = np.random.default_rng(13)
    d, L = 8, 23
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    k = (3.0 * rng.standard_normal((1, 1, L, d))).astype(np.float32)
    v = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    out, lse = oracle.decode(q, k, v, np.array([L], np.int32), lib=lib)
    s = (k[0, 0].astype(np.float64) @ q[0, 0].astype(np.float64)) / math.sqrt(d)
    vals = [v[0, 0, t].astype(np.float64) for t in range(L)]
    for S in (1, 2, 3, 7, L):
        parts = [oracle.block_partial(list(s[a:b]), vals[a:b])
                 for a, b in oracle.split_ranges(L, S) if b > a]
        merged, merged_lse = oracle.merge_blocks(parts)
        assert np.allclose(merged, out[0, 0], rtol=1e-12, atol=1e-13), S
        assert abs(merged_lse - lse[0, 0]) < 1e-12, S
        w = oracle.merge_weights([p[1] for p in parts])
        assert abs(math.fsum(w) - 1.0) < 1e-15
        assert all(0.0 < x <= 1.0 for x in w)


def pin_brute_force_decimal(lib):
    """Tiny shapes against 40-digit decimal arithmetic: exact products of the stored
    inputs, exp and ln in decimal, no max shift -- an evaluation that shares no step
    with the oracle's double-precision loops.  Covers GQA, bf16 storage and ragged
    lengths (including 0 and 1)."""
    ctx = decimal.Context(prec=40)
    rng = np.random.default_rng(14)
    B, Hkv, G, d, Lc = 3, 2, 2, 4, 8
    Hq = Hkv * G
    for storage in ("f32", "bf16"):
        q = rng.standard_normal((B, Hq, d)).astype(np.float32)
        k = (2.0 * rng.standard_normal((B, Hkv, Lc, d))).astype(np.float32)
        v = rng.standard_normal((B, Hkv, Lc, d)).astype(np.float32)
        if storage == "bf16":
            qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
            qf, kf, vf = _bits_to_f64(qb), _bits_to_f64(kb), _bits_to_f64(vb)
            args = (qb, kb, vb)
        else:
            qf, kf, vf = q.astype(np.float64), k.astype(np.float64), v.astype(np.float64)
            args = (q, k, v)
        lens = np.array([Lc, 1, 5], np.int32)
        out, lse = oracle.decode(*args, lens, lib=lib)
        inv_sqrt_d = ctx.divide(decimal.Decimal(1), ctx.sqrt(decimal.Decimal(d)))
        for b in range(B):
            for h in range(Hq):
                g = h // G
                ex, num = [], [decimal.Decimal(0)] * d
                for t in range(int(lens[b])):
                    dot = decimal.Decimal(0)
                    for j in range(d):
                        dot = ctx.add(dot, ctx.multiply(decimal.Decimal(float(qf[b, h, j])),
                                                        decimal.Decimal(float(kf[b, g, t, j]))))
                    e = ctx.exp(ctx.multiply(dot, inv_sqrt_d))
                    ex.append(e)
                    for j in range(d):
                        num[j] = ctx.add(num[j], ctx.multiply(e, decimal.Decimal(float(vf[b, g, t, j]))))
                den = sum(ex, decimal.Decimal(0))
                ref_lse = float(ctx.ln(den))
                ref_o = [float(ctx.divide(x, den)) for x in num]
                assert abs(lse[b, h] - ref_lse) < 1e-12, (storage, b, h)
                assert np.allclose(out[b, h], ref_o, rtol=1e-12, atol=1e-13), (storage, b, h)


def pin_torch_library(lib):
    """torch float64 CPU: softmax(q K^T / sqrt(d)) V, logsumexp, and SDPA, with each KV
    head repeated for its G query heads (the GQA special case of plain attention)."""
    import torch
    rng = np.random.default_rng(15)
    B, Hkv, G, d, Lc = 2, 2, 4, 16, 40
    Hq = Hkv * G
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, Lc, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Lc, d)).astype(np.float32)
    lens = np.array([Lc, 17], np.int32)
    out, lse = oracle.decode(q, k, v, lens, lib=lib)
    for b in range(B):
        L = int(lens[b])
        qt = torch.from_numpy(q[b].astype(np.float64))                     # [Hq, d]
        kt = torch.from_numpy(k[b, :, :L].astype(np.float64)).repeat_interleave(G, dim=0)
        vt = torch.from_numpy(v[b, :, :L].astype(np.float64)).repeat_interleave(G, dim=0)
        scores = torch.einsum("hd,htd->ht", qt, kt) / math.sqrt(d)
        ref = torch.einsum("ht,htd->hd", torch.softmax(scores, dim=-1), vt)
        ref_lse = torch.logsumexp(scores, dim=-1)
        sdpa = torch.nn.functional.scaled_dot_product_attention(
            qt[:, None, :], kt, vt)[:, 0, :]
        assert np.allclose(out[b], ref.numpy(), rtol=1e-12, atol=1e-13)
        assert np.allclose(out[b], sdpa.numpy(), rtol=1e-10, atol=1e-12)
        assert np.allclose(lse[b], ref_lse.numpy(), rtol=1e-13, atol=1e-13)


def pin_paged_permutation(lib):
    """Paging by a block table: logical order follows the table, not the physical page
    number.  A contiguous cache cut into pages, shuffled, with the table pointing at
    the new places, gives the same rows; reading the pages in physical order does not."""
    rng = np.random.default_rng(16)
    B, Hkv, G, d, ps, max_pages = 2, 2, 2, 8, 4, 5
    Hq = Hkv * G
    Lc = ps * max_pages
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, Lc, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Lc, d)).astype(np.float32)
    lens = np.array([Lc - 3, 9], np.int32)
    ref_o, ref_l = oracle.decode(q, k, v, lens, lib=lib)
    P = B * max_pages
    perm = rng.permutation(P)
    kp = np.empty((P, Hkv, ps, d), np.float32)
    vp = np.empty_like(kp)
    table = np.full((B, max_pages), -1, np.int32)
    for b in range(B):
        for i in range(max_pages):
            phys = int(perm[b * max_pages + i])
            kp[phys] = k[b, :, i * ps:(i + 1) * ps]
            vp[phys] = v[b, :, i * ps:(i + 1) * ps]
            if i * ps < lens[b]:
                table[b, i] = phys
    o, l = oracle.decode(q, kp, vp, lens, block_table=table, page_size=ps, lib=lib)
    assert np.allclose(o, ref_o, rtol=1e-13, atol=1e-14)
    assert np.allclose(l, ref_l, rtol=1e-13, atol=1e-14)
    sorted_table = np.full_like(table, -1)
    for b in range(B):
        used = table[b][table[b] >= 0]
        sorted_table[b, :used.size] = np.sort(used)
    assert not np.array_equal(sorted_table, table)
    o2, _ = oracle.decode(q, kp, vp, lens, block_table=sorted_table, page_size=ps, lib=lib)
    assert not np.allclose(o2, ref_o, atol=1e-3)


def pin_gqa_map(lib):
    """kv head = floor(h / G): give KV head g values all equal to 10 g + 1, then every
    query head h must return exactly 10 floor(h / G) + 1."""
    rng = np.random.default_rng(17)
    B, Hkv, G, d, L = 2, 4, 3, 8, 12
    Hq = Hkv * G
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    v = np.empty((B, Hkv, L, d), np.float32)
    for g in range(Hkv):
        v[:, g] = 10.0 * g + 1.0
    out, _ = oracle.decode(q, k, v, np.array([L, 5], np.int32), lib=lib)
    for h in range(Hq):
        assert np.allclose(out[:, h], 10.0 * (h // G) + 1.0, rtol=1e-14, atol=1e-13), h
    # And the batch map: batch b reads only its own cache rows.
    vb = np.zeros((B, Hkv, L, d), np.float32)
    vb[1] = 1.0
    out, _ = oracle.decode(q, k, vb, np.array([L, 5], np.int32), lib=lib)
    assert np.all(out[0] == 0.0) and np.allclose(out[1], 1.0, rtol=1e-14)


def pin_layout_transpose(lib):
    """q is [B, Hq, d]: rows with distinct query vectors give distinct, correctly placed
    results -- a transposed q (read as [Hq, B, d]) would swap them."""
    d, L = 4, 3
    q = np.zeros((2, 3, d), np.float32)
    for b in range(2):
        for h in range(3):
            q[b, h, 0] = 4.0 * (b * 3 + h)           # score of key 1 = 2 (b*3+h)
    k = np.zeros((2, 1, L, d), np.float32)
    k[:, :, 1, 0] = 1.0
    v = np.zeros((2, 1, L, d), np.float32)
    v[:, :, 1, :] = 1.0
    out, lse = oracle.decode(q, k, v, np.array([L, L], np.int32), lib=lib)
    for b in range(2):
        for h in range(3):
            z = 2.0 * (b * 3 + h)
            assert abs(out[b, h, 0] - math.exp(z) / (2.0 + math.exp(z))) < 1e-13
            assert abs(lse[b, h] - math.log(2.0 + math.exp(z))) < 1e-13


def pin_causal_reduces_to_decode(lib):
    """One query token: the multi-token oracle is the single-token one, bit for bit."""
    rng = np.random.default_rng(18)
    B, Hkv, G, d, L = 2, 2, 3, 8, 17
    q = rng.standard_normal((B, 1, Hkv * G, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    lens = np.array([L, 9], np.int32)
    o1, l1 = oracle.decode_causal(q, k, v, lens, lib=lib)
    o2, l2 = oracle.decode(q[:, 0], k, v, lens, lib=lib)
    assert np.array_equal(o1[:, 0], o2) and np.array_equal(l1[:, 0], l2)


def pin_causal_prefix_and_library(lib):
    """Query j of Q sees exactly the first L - Q + 1 + j keys: it equals single-token decode
    over that prefix, and torch float64 SDPA with a bottom-right aligned causal mask
    (keys repeated per query group); queries that see no key give 0 and -inf."""
    import torch
    rng = np.random.default_rng(19)
    B, Q, Hkv, G, d, Lc = 3, 4, 2, 2, 16, 30
    Hq = Hkv * G
    q = rng.standard_normal((B, Q, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, Lc, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Lc, d)).astype(np.float32)
    lens = np.array([30, 11, 2], np.int32)             # row 2: only 2 keys for 4 queries
    o, l = oracle.decode_causal(q, k, v, lens, lib=lib)
    for j in range(Q):
        pre = np.maximum(lens - Q + 1 + j, 0).astype(np.int32)
        oj, lj = oracle.decode(q[:, j], k, v, pre, lib=lib)
        assert np.allclose(o[:, j], oj, rtol=1e-13, atol=1e-14)
        assert np.array_equal(np.isneginf(l[:, j]), np.isneginf(lj))
        fin = ~np.isneginf(lj)
        assert np.allclose(l[:, j][fin], lj[fin], rtol=1e-13, atol=1e-14)
    assert np.all(o[2, :2] == 0.0) and np.all(np.isneginf(l[2, :2]))
    for b in range(B):
        L = int(lens[b])
        qt = torch.from_numpy(q[b].astype(np.float64)).permute(1, 0, 2)          # [Hq, Q, d]
        kt = torch.from_numpy(k[b, :, :L].astype(np.float64)).repeat_interleave(G, dim=0)
        vt = torch.from_numpy(v[b, :, :L].astype(np.float64)).repeat_interleave(G, dim=0)
        pos = torch.arange(Q)[:, None] + (L - Q)                                 # query positions
        mask = torch.arange(L)[None, :] <= pos                                   # [Q, L]
        live = mask.any(dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt[:, live], kt, vt, attn_mask=mask[live])                            # [Hq, Ql, d]
        got = torch.from_numpy(o[b]).permute(1, 0, 2)[:, live]
        assert torch.allclose(got, ref, rtol=1e-10, atol=1e-12)


def pin_causal_decimal(lib):
    """40-digit decimal evaluation of the causal rows on a tiny bf16 case."""
    ctx = decimal.Context(prec=40)
    rng = np.random.default_rng(20)
    B, Q, Hkv, G, d, Lc = 2, 3, 1, 2, 4, 6
    Hq = Hkv * G
    qb = _bf16_bits(rng.standard_normal((B, Q, Hq, d)).astype(np.float32))
    kb = _bf16_bits((2 * rng.standard_normal((B, Hkv, Lc, d))).astype(np.float32))
    vb = _bf16_bits(rng.standard_normal((B, Hkv, Lc, d)).astype(np.float32))
    qf, kf, vf = _bits_to_f64(qb), _bits_to_f64(kb), _bits_to_f64(vb)
    lens = np.array([6, 4], np.int32)
    o, l = oracle.decode_causal(qb, kb, vb, lens, lib=lib)
    inv = ctx.divide(decimal.Decimal(1), ctx.sqrt(decimal.Decimal(d)))
    for b in range(B):
        for j in range(Q):
            for h in range(Hq):
                vis = int(lens[b]) - Q + 1 + j
                ex, num = [], [decimal.Decimal(0)] * d
                for t in range(vis):
                    dot = decimal.Decimal(0)
                    for c in range(d):
                        dot = ctx.add(dot, ctx.multiply(decimal.Decimal(float(qf[b, j, h, c])),
                                                        decimal.Decimal(float(kf[b, h // G, t, c]))))
                    e = ctx.exp(ctx.multiply(dot, inv))
                    ex.append(e)
                    for c in range(d):
                        num[c] = ctx.add(num[c], ctx.multiply(e, decimal.Decimal(float(vf[b, h // G, t, c]))))
                den = sum(ex, decimal.Decimal(0))
                assert abs(l[b, j, h] - float(ctx.ln(den))) < 1e-12
                assert np.allclose(o[b, j, h], [float(ctx.divide(x, den)) for x in num],
                                   rtol=1e-12, atol=1e-13)


def pin_e4m3_decoding(lib):
    """Every FP8 E4M3 code against torch's float8_e4m3fn -> float64 conversion (a library
    routine), plus values fixed by the format: 0x38 = 1, 0x7E = 448 (largest finite),
    0x01 = 2^-9 (smallest subnormal), 0x08 = 2^-6 (smallest normal), 0x7F = NaN."""
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c, lib=lib) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    fixed = {0x38: 1.0, 0x7E: 448.0, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6, 0xB8: -1.0, 0x00: 0.0}
    for c, val in fixed.items():
        assert oracle.e4m3_to_double(c, lib=lib) == val
    assert math.isnan(oracle.e4m3_to_double(0x7F, lib=lib))


def pin_kv8_equals_dequantised(lib):
    """Decode over FP8 codes with per-head scales equals plain decode over the
    dequantised cache (codes widened, times the scale, stored exactly in fp32)."""
    import torch
    rng = np.random.default_rng(21)
    B, Hkv, G, d, L = 2, 2, 2, 16, 23
    Hq = Hkv * G
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    codes_k = rng.integers(0, 256, (B, Hkv, L, d), dtype=np.uint8)
    codes_v = rng.integers(0, 256, (B, Hkv, L, d), dtype=np.uint8)
    for c in (codes_k, codes_v):                       # no NaN codes (0x7F, 0xFF)
        c[(c & 0x7F) == 0x7F] = 0x38
    ks = np.array([0.5, 0.125], np.float32)
    vs = np.array([0.25, 2.0], np.float32)
    lens = np.array([L, 9], np.int32)
    o, l = oracle.decode_kv8(q, codes_k, codes_v, ks, vs, lens, lib=lib)
    deq = lambda c, sc: (torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
                         * sc[None, :, None, None]).astype(np.float32)
    o2, l2 = oracle.decode(q, deq(codes_k, ks), deq(codes_v, vs), lens, lib=lib)
    assert np.allclose(o, o2, rtol=1e-13, atol=1e-13) and np.allclose(l, l2, rtol=1e-13, atol=1e-13)


ALL_PINS = [
    pin_softmax_examples, pin_worked_example, pin_closed_forms, pin_shift_invariance,
    pin_split_invariance, pin_brute_force_decimal, pin_torch_library,
    pin_paged_permutation, pin_gqa_map, pin_layout_transpose,
    pin_causal_reduces_to_decode, pin_causal_prefix_and_library, pin_causal_decimal,
    pin_e4m3_decoding, pin_kv8_equals_dequantised,
]


def failing_pins(lib):
    """Names of the pins that fail (or raise) for a given oracle library."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except Exception:  # noqa: BLE001 -- any failure counts
            bad.append(pin.__name__)
    return bad
