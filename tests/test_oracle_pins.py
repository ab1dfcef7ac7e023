"""Pins for the fp64 oracle, independent of the oracle's own code.

Each test checks the oracle against something it does not compute itself:
a brute-force masked softmax over the whole packed batch (scipy's
logsumexp), closed forms, invariants of the method, or the worked example of
Figure 2(b) in the ByteScale research digest.  A plausible slip in the oracle
(a dropped key, an off-by-one causal edge, a wrong GQA head, a wrong scale, a
leak across documents, a wrong merge weight, a wrong best-fit choice) fails at
least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from packed_varlen_attention_aware_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_qkv(lengths, hq, hkv, d, seed, std=1.0):
    T = int(sum(lengths))
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(T, hq, d, generator=g) * std).to(torch.bfloat16)
    k = (torch.randn(T, hkv, d, generator=g) * std).to(torch.bfloat16)
    v = (torch.randn(T, hkv, d, generator=g) * std).to(torch.bfloat16)
    return wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v)


def _bits_to_f64(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def _bruteforce(q, k, v, lengths, hq, hkv, d, scale):
    """softmax(Q K^T * scale + mask) V over the whole packed batch with an
    explicit T x T mask: same document and key position <= query position."""
    Q, K, V = _bits_to_f64(q), _bits_to_f64(k), _bits_to_f64(v)
    T = Q.shape[0]
    doc = np.repeat(np.arange(len(lengths)), lengths)
    pos = np.arange(T)
    mask = (doc[:, None] == doc[None, :]) & (pos[None, :] <= pos[:, None])
    O = np.zeros((T, hq, d))
    L = np.zeros((hq, T))
    for h in range(hq):
        g = h // (hq // hkv)
        S = Q[:, h, :] @ K[:, g, :].T * scale
        S = np.where(mask, S, -np.inf)
        lse = logsumexp(S, axis=1)
        P = np.exp(S - lse[:, None])
        O[:, h, :] = P @ V[:, g, :]
        L[h] = lse
    return O, L


@pytest.mark.parametrize("lengths,hq,hkv,d,seed", [
    ([1, 5, 17, 40, 3], 4, 2, 16, 0),
    ([33, 1, 64], 2, 1, 32, 1),
    ([7, 9, 2, 30], 3, 3, 8, 2),
    ([50], 4, 4, 64, 3),
])
def test_attention_equals_bruteforce_masked_softmax(lengths, hq, hkv, d, seed):
    q, k, v = _rand_qkv(lengths, hq, hkv, d, seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, _cu(lengths), hq, hkv, d, scale)
    O, L = _bruteforce(q, k, v, lengths, hq, hkv, d, scale)
    assert np.max(np.abs(o - O)) < 1e-12
    assert np.max(np.abs(lse - L)) < 1e-12


def _bruteforce_f64(Q, K, V, lengths, hq, hkv, scale):
    """The same explicit-mask softmax on arbitrary fp64 inputs."""
    T, _, d = Q.shape
    doc = np.repeat(np.arange(len(lengths)), lengths)
    pos = np.arange(T)
    mask = (doc[:, None] == doc[None, :]) & (pos[None, :] <= pos[:, None])
    O = np.zeros((T, hq, d))
    L = np.zeros((hq, T))
    for h in range(hq):
        g = h // (hq // hkv)
        S = np.where(mask, Q[:, h, :] @ K[:, g, :].T * scale, -np.inf)
        L[h] = logsumexp(S, axis=1)
        O[:, h, :] = np.exp(S - L[h][:, None]) @ V[:, g, :]
    return O, L


@pytest.mark.parametrize("lengths,hq,hkv,d,seed", [
    ([1, 6, 13, 2], 4, 2, 8, 0),
    ([21], 3, 1, 5, 1),
    ([9, 9, 1, 30], 2, 2, 16, 2),
])
def test_attention_f64_equals_bruteforce_masked_softmax(lengths, hq, hkv, d, seed):
    """The fp64-input forward (the one the backward's finite differences
    differentiate) against the explicit-mask softmax on inputs that are not
    bf16-representable, and bit for bit against the bf16-input forward on
    bf16 inputs."""
    rng = np.random.default_rng(100 + seed)
    T = sum(lengths)
    Q, K, V = rng.normal(0, 1.3, (T, hq, d)), rng.normal(0, 1.3, (T, hkv, d)), rng.normal(0, 1, (T, hkv, d))
    scale = 0.61
    o, lse = oracle.attention_f64(Q, K, V, _cu(lengths), hq, hkv, d, scale)
    O, L = _bruteforce_f64(Q, K, V, lengths, hq, hkv, scale)
    assert np.max(np.abs(o - O)) < 1e-12
    assert np.max(np.abs(lse - L)) < 1e-12
    q, k, v = _rand_qkv(lengths, hq, hkv, d, seed)
    o16, lse16 = oracle.attention(q, k, v, _cu(lengths), hq, hkv, d, scale)
    o64, lse64 = oracle.attention_f64(q, k, v, _cu(lengths), hq, hkv, d, scale)
    assert np.array_equal(o16, o64) and np.array_equal(lse16, lse64)


def test_zero_keys_closed_form():
    """K = 0: every score is 0, so LSE_p = ln(p+1) and O_p = mean(v_0..v_p)."""
    lengths = [3, 20, 1, 9]
    hq, hkv, d = 2, 1, 8
    q, k, v = _rand_qkv(lengths, hq, hkv, d, 5)
    k[:] = 0
    o, lse = oracle.attention(q, k, v, _cu(lengths), hq, hkv, d, 0.5)
    V = _bits_to_f64(v)
    cu = _cu(lengths)
    for i, s in enumerate(lengths):
        p = np.arange(s)
        for h in range(hq):
            assert np.allclose(lse[h, cu[i]:cu[i + 1]], np.log(p + 1.0), atol=1e-13, rtol=0)
            prefix_mean = np.cumsum(V[cu[i]:cu[i + 1], 0, :], axis=0) / (p + 1.0)[:, None]
            assert np.allclose(o[cu[i]:cu[i + 1], h, :], prefix_mean, atol=1e-13, rtol=0)


def test_constant_values_give_constant_output():
    """V = c on every key: the softmax weights sum to one, so O = c."""
    lengths = [4, 11, 6]
    hq, hkv, d = 4, 2, 16
    q, k, v = _rand_qkv(lengths, hq, hkv, d, 6)
    c = torch.linspace(-3, 3, d).to(torch.bfloat16)
    v[:] = wl.bf16_bits(c)[None, None, :]
    o, _ = oracle.attention(q, k, v, _cu(lengths), hq, hkv, d, 0.25)
    assert np.max(np.abs(o - _bits_to_f64(wl.bf16_bits(c))[None, None, :])) < 1e-13


def test_single_token_documents():
    """s = 1: O = v_0 and LSE = scale * q.k."""
    lengths = [1, 1, 1]
    hq, hkv, d = 2, 2, 32
    q, k, v = _rand_qkv(lengths, hq, hkv, d, 7)
    o, lse = oracle.attention(q, k, v, _cu(lengths), hq, hkv, d, 0.125)
    Q, K, V = _bits_to_f64(q), _bits_to_f64(k), _bits_to_f64(v)
    assert np.array_equal(o, V)
    assert np.allclose(lse.T, 0.125 * np.einsum("thd,thd->th", Q, K), atol=1e-13, rtol=0)


@pytest.mark.parametrize("C", [1, 3, 8, 13, 64])
def test_merged_chunk_partials_equal_unchunked(C):
    """Section 3.2: each query chunk's result is the LSE merge of its partial
    blocks over the causal-prior key chunks."""
    lengths = [29, 5, 40]
    hq, hkv, d = 2, 1, 16
    q, k, v = _rand_qkv(lengths, hq, hkv, d, 8)
    scale = 0.3
    cu = _cu(lengths)
    full_o, full_lse = oracle.attention(q, k, v, cu, hq, hkv, d, scale)
    p = oracle.plan(lengths, C)
    ct = p["chunk_table"]
    for c in range(p["num_chunks"]):
        doc, idx, beg, ln = (int(x) for x in ct[c])
        toks = np.repeat(np.arange(beg, beg + ln), hq)
        heads = np.tile(np.arange(hq), ln)
        parts_o, parts_l = [], []
        for kc in range(idx + 1):
            lo = np.full(len(toks), kc * C, np.int64)
            hi = np.full(len(toks), min((kc + 1) * C, lengths[doc]), np.int64)
            o, l = oracle.attention_rows(q, k, v, cu, hq, hkv, d, scale, toks, heads, lo, hi)
            parts_o.append(o)
            parts_l.append(l)
        mo, ml = oracle.merge(np.stack(parts_o), np.stack(parts_l))
        assert np.max(np.abs(mo - full_o[toks, heads])) < 1e-12
        assert np.max(np.abs(ml - full_lse[heads, toks])) < 1e-12


def test_packing_invariance():
    """A document's output does not depend on what it is packed with."""
    hq, hkv, d = 2, 2, 16
    docs = [5, 12, 1, 7]
    rng = np.random.default_rng(0)
    data = [_rand_qkv([s], hq, hkv, d, 100 + i) for i, s in enumerate(docs)]
    ref = [oracle.attention(*data[i], _cu([s]), hq, hkv, d, 0.2) for i, s in enumerate(docs)]
    for _ in range(3):
        order = rng.permutation(len(docs))
        q = np.concatenate([data[i][0] for i in order])
        k = np.concatenate([data[i][1] for i in order])
        v = np.concatenate([data[i][2] for i in order])
        lens = [docs[i] for i in order]
        o, lse = oracle.attention(q, k, v, _cu(lens), hq, hkv, d, 0.2)
        cu = _cu(lens)
        for j, i in enumerate(order):
            assert np.array_equal(o[cu[j]:cu[j + 1]], ref[i][0])
            assert np.array_equal(lse[:, cu[j]:cu[j + 1]], ref[i][1])


def test_merge_closed_forms():
    rng = np.random.default_rng(1)
    o1 = rng.standard_normal((5, 8))
    o2 = rng.standard_normal((5, 8))
    l1 = rng.standard_normal(5)
    # m = 1 is the identity
    mo, ml = oracle.merge(o1[None], l1[None])
    assert np.array_equal(mo, o1) and np.array_equal(ml, l1)
    # equal LSEs: average of the outputs, LSE + ln 2
    mo, ml = oracle.merge(np.stack([o1, o2]), np.stack([l1, l1]))
    assert np.allclose(mo, (o1 + o2) / 2, atol=1e-15, rtol=0)
    assert np.allclose(ml, l1 + math.log(2.0), atol=1e-15, rtol=0)
    # a -inf partial contributes nothing
    mo, ml = oracle.merge(np.stack([o1, o2]), np.stack([l1, np.full(5, -np.inf)]))
    assert np.array_equal(mo, o1) and np.array_equal(ml, l1)
    # weights follow exp(lse_k - lse): lse2 = lse1 + ln 3 gives weights 1/4, 3/4
    mo, ml = oracle.merge(np.stack([o1, o2]), np.stack([l1, l1 + math.log(3.0)]))
    assert np.allclose(mo, 0.25 * o1 + 0.75 * o2, atol=1e-14, rtol=0)
    assert np.allclose(ml, l1 + math.log(4.0), atol=1e-14, rtol=0)
    # all -inf: lse -inf, o 0
    mo, ml = oracle.merge(np.stack([o1]), np.full((1, 5), -np.inf))
    assert np.all(ml == -np.inf) and np.all(mo == 0)


# ---------------------------------------------------------------- plan pins

def test_figure2b_assignment():
    g = json.load(open(os.path.join(GOLDEN, "fig2b_hdp_assignment.json")))
    p = oracle.plan(g["lengths"], g["capacity"])
    assert p["num_shards"] == g["num_ranks"]
    ct = p["chunk_table"]
    for doc, ranks in enumerate(g["ranks_of_sequence"]):
        got = sorted(int(p["shard_of_chunk"][c]) for c in range(p["num_chunks"]) if ct[c, 0] == doc)
        assert got == sorted(ranks), (doc, got, ranks)


def test_rank_counts_from_pages():
    g = json.load(open(os.path.join(GOLDEN, "rank_counts.json")))
    for case in g["cases"]:
        p = oracle.plan([case["length"]], case["capacity"])
        assert p["num_chunks"] == case["ranks"], case
        assert p["num_shards"] == case["ranks"], case


def test_plan_sizes_of_named_workloads():
    # tiny: 64,128,256 fit in one chunk each, 512 splits in two -> 5 chunks, 1+1+1+3 blocks
    p = oracle.plan([64, 128, 256, 512], 256)
    assert (p["num_chunks"], p["num_blocks"]) == (5, 6)
    p = oracle.plan([131072], 8192)
    assert (p["num_chunks"], p["num_blocks"], p["num_shards"]) == (16, 136, 16)
    nc, nb, tt = oracle.plan_sizes([2097152], 8192)
    assert (nc, nb, tt) == (256, 32896, 2097152)


def test_plan_tables_against_closed_forms():
    """The oracle counts with loops; check it against the closed forms
    ceil(s/C), n(n+1)/2 and (b(b+1) - a(a+1))/2 on random inputs."""
    rng = np.random.default_rng(3)
    for trial in range(30):
        n = int(rng.integers(1, 12))
        lengths = rng.integers(1, 200, n)
        C = int(rng.integers(1, 90))
        p = oracle.plan(lengths, C)
        nchunks = [-(-int(s) // C) for s in lengths]
        assert np.array_equal(p["cu_seqlens"], np.concatenate([[0], np.cumsum(lengths)]))
        assert np.array_equal(p["chunk_offsets"], np.concatenate([[0], np.cumsum(nchunks)]))
        assert np.array_equal(p["block_offsets"],
                              np.concatenate([[0], np.cumsum([c * (c + 1) // 2 for c in nchunks])]))
        c = 0
        b = 0
        for i, s in enumerate(lengths):
            for j in range(nchunks[i]):
                a_, b_ = j * C, min((j + 1) * C, int(s))
                assert tuple(p["chunk_table"][c]) == (i, j, p["cu_seqlens"][i] + a_, b_ - a_)
                assert p["chunk_pairs"][c] == (b_ * (b_ + 1) - a_ * (a_ + 1)) // 2
                c += 1
            first = p["chunk_offsets"][i]
            for qc in range(nchunks[i]):
                for kc in range(qc + 1):
                    assert tuple(p["block_table"][b]) == (first + qc, first + kc)
                    b += 1
        # shard capacity and full-chunk exclusivity
        loads = np.zeros(p["num_shards"], np.int64)
        for cc in range(p["num_chunks"]):
            loads[p["shard_of_chunk"][cc]] += p["chunk_table"][cc, 3]
        assert np.all(loads <= C)
        full = [cc for cc in range(p["num_chunks"]) if p["chunk_table"][cc, 3] == C]
        assert [p["shard_of_chunk"][cc] for cc in full] == list(range(len(full)))


def test_best_fit_decreasing_hand_example():
    """Worked by hand under the best-fit-decreasing reading (C = 6):
    pieces 5,3,3,2,2,1 (docs 0..5).  5 opens shard 0 (1 left); 3 opens shard 1
    (3 left); 3 fits only shard 1 (0 left); 2 fits nowhere, opens shard 2
    (4 left); 2 -> shard 2 (2 left); 1 fits shards 0 (1 left) and 2 (2 left),
    least remaining wins -> shard 0."""
    p = oracle.plan([5, 3, 3, 2, 2, 1], 6)
    assert list(p["shard_of_chunk"]) == [0, 1, 1, 2, 2, 0]
    assert p["num_shards"] == 3
    # ties on remaining capacity go to the lowest shard id; equal lengths go in doc order
    p = oracle.plan([4, 4, 2, 2], 6)
    assert list(p["shard_of_chunk"]) == [0, 1, 0, 1]


def test_tail_chunks_are_packed_like_short_docs():
    # 20 at C=8 -> chunks 8, 8, 4 ; the tail (4) and a short doc (4) share a shard
    p = oracle.plan([20, 4], 8)
    assert list(p["shard_of_chunk"]) == [0, 1, 2, 2]


# ---------------------------------------------------------------- FLOPs pins

def test_flops_closed_form_and_named_values():
    assert oracle.flops_total([64, 128, 256, 512], 64, 4) == 178_749_440
    s = 131072
    assert oracle.flops_total([s], 128, 32) == 4 * 128 * 32 * s * (s + 1) // 2
    rng = np.random.default_rng(4)
    for _ in range(10):
        lengths = rng.integers(1, 5000, int(rng.integers(1, 20)))
        d, h = int(rng.choice([64, 128])), int(rng.integers(1, 33))
        assert oracle.flops_total(lengths, d, h) == sum(4 * d * h * int(x) * (int(x) + 1) // 2 for x in lengths)


def test_flops_per_shard():
    p = oracle.plan([131072], 8192)
    f = oracle.flops_per_shard(p, 128, 32)
    C = 8192
    for j in range(16):
        assert f[j] == 4 * 128 * 32 * (C * C * j + C * (C + 1) // 2)
    assert f[0] == 549_822_922_752
    assert f[15] == 17_042_497_339_392
    assert int(f.sum()) == oracle.flops_total([131072], 128, 32)
    p = oracle.plan([64, 128, 256, 512], 256)
    assert int(oracle.flops_per_shard(p, 64, 4).sum()) == 178_749_440


# ---------------------------------------------------------------- work list pins

@pytest.mark.parametrize("split", [False, True])
def test_tile_worklist_covers_every_causal_pair_once(split):
    """The tiles' (query rows x key range) cover each same-document causal
    pair exactly once, and never a cross-document or future pair."""
    tile = 4
    lengths = [1, 9, 16, 3, 23]
    C = 8
    p = oracle.plan(lengths, C)
    wlst = oracle.tile_worklist(p, tile=tile, split=split)
    T = sum(lengths)
    doc = np.repeat(np.arange(len(lengths)), lengths)
    cover = np.zeros((T, T), np.int32)
    starts = np.concatenate([[0], np.cumsum(lengths)])
    for q0, qrows, kv0, kvlen, blk, off, w, slen in wlst:
        assert w == -(-kvlen // tile)
        # the last column is the query's document length (fused list only)
        d_i = doc[q0]
        assert slen == (0 if split else lengths[d_i])
        if not split:
            assert kv0 == starts[d_i] and off == q0 - starts[d_i]
        for t in range(q0, q0 + qrows):
            for u in range(kv0, kv0 + kvlen):
                if u <= t:
                    cover[t, u] += 1
    want = ((doc[:, None] == doc[None, :]) & (np.arange(T)[None, :] <= np.arange(T)[:, None])).astype(np.int32)
    assert np.array_equal(cover, want)
    assert np.all(np.diff(wlst[:, 6]) <= 0)
