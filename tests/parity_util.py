"""Shared helpers for the GPU parity tests: run the CUDA path through the
C ABI, run the fp64 oracle on the same bytes, compare within the tolerances."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import packed_varlen_attention_aware_gb300 as pkg
from packed_varlen_attention_aware_gb300 import workloads as wl

# Attention tolerances against the fp64 oracle, on the same bf16-rounded
# inputs: the GPU output is bf16 (round to nearest even), so its rounding
# counts toward the error.
TOL_MAX_O = 1.5e-2
TOL_MEAN_O = 1e-3
TOL_MAX_LSE = 2e-3

PLAN_KEYS = ("cu_seqlens", "chunk_offsets", "block_offsets", "chunk_table", "block_table", "chunk_pairs")


def check_plan(lengths, C, with_shards=True, d=128, hq=32):
    """Every plan table, both work lists and the per-shard FLOPs, bit-exact."""
    dl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    flags = pkg.HDP_PLAN_DEFAULT if with_shards else pkg.HDP_PLAN_NO_SHARDS
    with pkg.hdp_plan_create(dl, C, flags=flags) as plan:
        ref = oracle.plan(lengths, C)
        got = plan.tables()
        v = plan.view
        assert v.num_chunks == ref["num_chunks"] and v.num_blocks == ref["num_blocks"]
        assert v.total_tokens == int(ref["cu_seqlens"][-1])
        assert v.max_doc_len == max(lengths)
        for key in PLAN_KEYS:
            assert np.array_equal(got[key], ref[key]), key
        assert np.array_equal(got["tiles_fused"], oracle.tile_worklist(ref, 128, split=False))
        if C % 128 == 0:
            assert np.array_equal(got["tiles_split"], oracle.tile_worklist(ref, 128, split=True))
        if with_shards:
            assert v.num_shards == ref["num_shards"]
            assert np.array_equal(got["shard_of_chunk"], ref["shard_of_chunk"])
            f = torch.empty(max(v.num_shards, 1), dtype=torch.int64, device="cuda")
            pkg.hdp_flops_per_shard(plan, d, hq, f)
            assert np.array_equal(f.cpu().numpy()[: v.num_shards], oracle.flops_per_shard(ref, d, hq))
        return ref


def run_gpu(q, k, v, lengths, C, mode, plan=None):
    dl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    o, lse, plan = pkg.attention(q, k, v, dl, C, mode=mode, plan=plan)
    pkg.hdp_device_status()
    return o, lse, plan


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """o_gpu/lse_gpu: float64 numpy arrays of the CUDA results (same shape as refs).

    The message also counts the reference elements with |O| >= 4, where half
    a bf16 ulp (2^-6 = 0.0156) alone exceeds the 1.5e-2 bar: rows with very
    few keys, where O is about one v value."""
    do = np.abs(o_gpu - o_ref)
    dl = np.abs(lse_gpu - lse_ref)
    big = int(np.count_nonzero(np.abs(o_ref) >= 4.0))
    msg = (f"{what}: max|dO|={do.max():.3e} mean|dO|={do.mean():.3e} max|dLSE|={dl.max():.3e} "
           f"|O|>=4: {big} of {o_ref.size}")
    if os.environ.get("HDP_PARITY_REPORT"):
        print("parity", msg, flush=True)
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all(), msg
    assert do.max() <= TOL_MAX_O, msg
    assert do.mean() <= TOL_MEAN_O, msg
    assert dl.max() <= TOL_MAX_LSE, msg
    return msg


def full_parity(lengths, hq, hkv, d, C, mode, seed=0, std=1.0):
    """Whole-output comparison (small sizes)."""
    w = wl.Workload("case", tuple(lengths), C, hq, hkv, d, std, seed)
    q, k, v = wl.qkv(w, device="cpu")
    o, lse, plan = run_gpu(q.cuda(), k.cuda(), v.cuda(), lengths, C, mode)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    o_ref, lse_ref = oracle.attention(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), cu, hq, hkv, d, w.scale)
    msg = compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref,
                  f"{lengths[:6]} hq={hq} hkv={hkv} d={d} C={C} mode={mode}")
    plan.destroy()
    return msg, o, lse


def sample_rows(lengths, hq, n_random, seed, tile=128):
    """Sampled (token, head) pairs: each document's first and last token, the
    rows around every query-tile edge of the longest document, and random ones."""
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    toks = []
    for i, s in enumerate(lengths):
        toks += [cu[i], cu[i] + s - 1]
    big = int(np.argmax(lengths))
    for e in range(0, lengths[big], max(tile, lengths[big] // 64 // tile * tile)):
        for off in (e - 1, e, e + 127):
            if 0 <= off < lengths[big]:
                toks.append(cu[big] + off)
    toks += list(rng.integers(0, cu[-1], n_random))
    toks = np.array(toks, dtype=np.int64)
    heads = rng.integers(0, hq, len(toks)).astype(np.int32)
    return toks, heads


def sampled_parity(w, q, k, v, o, lse, toks, heads, what=""):
    """Compare sampled rows of the CUDA output against the oracle computed row by row."""
    cu = np.concatenate([[0], np.cumsum(w.lengths)]).astype(np.int32)
    qh = np.zeros((w.total_tokens, w.hq, w.d), np.uint16)
    uniq = np.unique(toks)
    qh[uniq] = wl.bf16_bits(q[torch.as_tensor(uniq, device=q.device)])
    kh, vh = wl.bf16_bits(k), wl.bf16_bits(v)
    o_ref, lse_ref = oracle.attention_rows(qh, kh, vh, cu, w.hq, w.hkv, w.d, w.scale, toks, heads)
    ti = torch.as_tensor(toks, device=o.device)
    hi = torch.as_tensor(heads.astype(np.int64), device=o.device)
    o_gpu = o[ti, hi].double().cpu().numpy()
    lse_gpu = lse[hi, ti].double().cpu().numpy()
    return compare(o_gpu, lse_gpu, o_ref, lse_ref, what)
