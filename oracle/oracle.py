"""ctypes marshalling for the C oracle (``hdp_oracle.c``), plus the tile work
list order, which is integer bookkeeping written out in Python.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hdp_oracle.c")
_LIB = os.path.join(_HERE, "libhdp_oracle.so")
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, IEEE semantics, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_plan_sizes.argtypes = [P, i32, i32, P, P, P]
            lib.oracle_plan.argtypes = [P, i32, i32, P, P, P, P, P, P, P, P]
            lib.oracle_flops_total.argtypes = [P, i32, i32, i32]
            lib.oracle_flops_total.restype = i64
            lib.oracle_flops_per_shard.argtypes = [P, P, i32, i32, i32, i32, P]
            lib.oracle_attention.argtypes = [P, P, P, P, i32, i32, i32, i32, f64, P, P]
            lib.oracle_attention_rows.argtypes = [P, P, P, P, i32, i32, i32, i32, f64, P, P, P, P, i64, P, P]
            lib.oracle_merge.argtypes = [i32, i64, i32, P, P, P, P]
            lib.oracle_attention_f64.argtypes = [P, P, P, P, i32, i32, i32, i32, f64, P, P]
            lib.oracle_attention_bwd.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, P, P, P]
            lib.oracle_attention_bwd_dq_rows.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, P, P, i64, P]
            lib.oracle_attention_bwd_dkv_rows.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, P, P, i64, P, P]
            lib.oracle_attention_bwd_dkv_doc.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, i32, i32, P, i64,
                                                         P, P]
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(x: np.ndarray) -> np.ndarray:
    """bf16 tensors travel as their uint16 bit patterns."""
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("pass bf16 data as uint16 bit patterns")
    return x


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().oracle_num_threads())


def plan_sizes(lengths, C: int):
    lib = _load()
    L = np.ascontiguousarray(lengths, dtype=np.int32)
    nc = np.zeros(1, np.int32)
    nb = np.zeros(1, np.int64)
    tt = np.zeros(1, np.int64)
    rc = lib.oracle_plan_sizes(_ptr(L), len(L), int(C), _ptr(nc), _ptr(nb), _ptr(tt))
    if rc != 0:
        raise ValueError(f"oracle_plan_sizes: invalid input (rc={rc})")
    return int(nc[0]), int(nb[0]), int(tt[0])


def plan(lengths, C: int, shards: bool = True) -> dict:
    """Sharding plan of section 3.1 (see hdp_oracle.c for the tables).
    shards=False skips best-fit packing (quadratic in the number of pieces)."""
    lib = _load()
    L = np.ascontiguousarray(lengths, dtype=np.int32)
    n = len(L)
    nc, nb, _ = plan_sizes(L, C)
    out = dict(
        cu_seqlens=np.zeros(n + 1, np.int32),
        chunk_offsets=np.zeros(n + 1, np.int32),
        block_offsets=np.zeros(n + 1, np.int64),
        chunk_table=np.zeros((max(nc, 1), 4), np.int32),
        block_table=np.zeros((max(nb, 1), 2), np.int32),
        chunk_pairs=np.zeros(max(nc, 1), np.int64),
        shard_of_chunk=np.zeros(max(nc, 1), np.int32),
    )
    ns = np.zeros(1, np.int32)
    rc = lib.oracle_plan(_ptr(L), n, int(C), _ptr(out["cu_seqlens"]), _ptr(out["chunk_offsets"]),
                         _ptr(out["block_offsets"]), _ptr(out["chunk_table"]), _ptr(out["block_table"]),
                         _ptr(out["chunk_pairs"]), _ptr(out["shard_of_chunk"]) if shards else None, _ptr(ns))
    if rc != 0:
        raise ValueError(f"oracle_plan failed (rc={rc})")
    out["chunk_table"] = out["chunk_table"][:nc]
    out["block_table"] = out["block_table"][:nb]
    out["chunk_pairs"] = out["chunk_pairs"][:nc]
    out["shard_of_chunk"] = out["shard_of_chunk"][:nc]
    out["num_chunks"] = nc
    out["num_blocks"] = nb
    out["num_shards"] = int(ns[0])
    out["capacity"] = int(C)
    return out


def flops_total(lengths, d: int, hq: int) -> int:
    lib = _load()
    L = np.ascontiguousarray(lengths, dtype=np.int32)
    return int(lib.oracle_flops_total(_ptr(L), len(L), int(d), int(hq)))


def flops_per_shard(p: dict, d: int, hq: int) -> np.ndarray:
    lib = _load()
    out = np.zeros(max(p["num_shards"], 1), np.int64)
    cp = np.ascontiguousarray(p["chunk_pairs"], np.int64)
    sc = np.ascontiguousarray(p["shard_of_chunk"], np.int32)
    rc = lib.oracle_flops_per_shard(_ptr(cp), _ptr(sc), p["num_chunks"], p["num_shards"], int(d), int(hq), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_flops_per_shard failed")
    return out[: p["num_shards"]]


def attention(q, k, v, cu_seqlens, hq: int, hkv: int, d: int, scale: float):
    """Full attention.  q [T][hq][d], k/v [T][hkv][d] as bf16 bit patterns.
    Returns o [T][hq][d] fp64 and lse [hq][T] fp64."""
    lib = _load()
    q, k, v = _bits(q), _bits(k), _bits(v)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    T = int(cu[-1])
    o = np.zeros((T, hq, d), np.float64)
    lse = np.zeros((hq, T), np.float64)
    rc = lib.oracle_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, hq, hkv, d, float(scale), _ptr(o),
                              _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_attention failed (rc={rc})")
    return o, lse


def attention_rows(q, k, v, cu_seqlens, hq: int, hkv: int, d: int, scale: float, tokens, heads, key_lo=None,
                   key_hi=None):
    """Sampled rows (optionally restricted to doc-local key ranges).
    Returns o [ns][d] and lse [ns] in fp64."""
    lib = _load()
    q, k, v = _bits(q), _bits(k), _bits(v)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    t = np.ascontiguousarray(tokens, np.int64)
    h = np.ascontiguousarray(heads, np.int32)
    ns = len(t)
    lo = None if key_lo is None else np.ascontiguousarray(key_lo, np.int64)
    hi = None if key_hi is None else np.ascontiguousarray(key_hi, np.int64)
    o = np.zeros((ns, d), np.float64)
    lse = np.zeros(ns, np.float64)
    rc = lib.oracle_attention_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, hq, hkv, d, float(scale),
                                   _ptr(t), _ptr(h), None if lo is None else _ptr(lo),
                                   None if hi is None else _ptr(hi), ns, _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_attention_rows failed (rc={rc})")
    return o, lse


def bf16_bits_to_f64(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64, exactly."""
    x = _bits(x)
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _f64(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return np.ascontiguousarray(x, dtype=np.float64)


def attention_f64(q, k, v, cu_seqlens, hq: int, hkv: int, d: int, scale: float):
    """Forward on fp64 inputs (or bf16 bit patterns, converted exactly).
    Returns o [T][hq][d] and lse [hq][T] in fp64."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    T = int(cu[-1])
    o = np.zeros((T, hq, d), np.float64)
    lse = np.zeros((hq, T), np.float64)
    rc = lib.oracle_attention_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, hq, hkv, d, float(scale),
                                  _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_attention_f64 failed (rc={rc})")
    return o, lse


def attention_bwd(q, k, v, dout, cu_seqlens, hq: int, hkv: int, d: int, scale: float):
    """Gradients of sum(O * dout) w.r.t. q, k, v (fp64; bf16 inputs converted
    exactly).  Returns dq [T][hq][d], dk [T][hkv][d], dv [T][hkv][d]."""
    lib = _load()
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    T = int(cu[-1])
    dq = np.zeros((T, hq, d), np.float64)
    dk = np.zeros((T, hkv, d), np.float64)
    dv = np.zeros((T, hkv, d), np.float64)
    rc = lib.oracle_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(cu), len(cu) - 1, hq, hkv, d,
                                  float(scale), _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd failed (rc={rc})")
    return dq, dk, dv


def attention_bwd_dq_rows(q, k, v, dout, cu_seqlens, hq: int, hkv: int, d: int, scale: float, tokens, heads):
    """dq of sampled (token, query head) rows, fp64 [ns][d]."""
    lib = _load()
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    t = np.ascontiguousarray(tokens, np.int64)
    h = np.ascontiguousarray(heads, np.int32)
    out = np.zeros((len(t), d), np.float64)
    rc = lib.oracle_attention_bwd_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(cu), len(cu) - 1, hq, hkv, d,
                                          float(scale), _ptr(t), _ptr(h), len(t), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd_dq_rows failed (rc={rc})")
    return out


def attention_bwd_dkv_rows(q, k, v, dout, cu_seqlens, hq: int, hkv: int, d: int, scale: float, tokens,
                           kv_heads):
    """dk and dv of sampled (key token, kv head) rows, fp64 [ns][d] each."""
    lib = _load()
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    t = np.ascontiguousarray(tokens, np.int64)
    g = np.ascontiguousarray(kv_heads, np.int32)
    dk = np.zeros((len(t), d), np.float64)
    dv = np.zeros((len(t), d), np.float64)
    rc = lib.oracle_attention_bwd_dkv_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(cu), len(cu) - 1, hq, hkv, d,
                                           float(scale), _ptr(t), _ptr(g), len(t), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd_dkv_rows failed (rc={rc})")
    return dk, dv


def attention_bwd_dkv_doc(q, k, v, dout, cu_seqlens, hq: int, hkv: int, d: int, scale: float, doc: int, kv_head: int,
                          keys):
    """dk and dv of selected doc-local keys of one document and kv head,
    fp64 [nk][d] each (each query row computed once for all the keys)."""
    lib = _load()
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    kk = np.ascontiguousarray(keys, np.int64)
    dk = np.zeros((len(kk), d), np.float64)
    dv = np.zeros((len(kk), d), np.float64)
    rc = lib.oracle_attention_bwd_dkv_doc(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(cu), len(cu) - 1, hq, hkv, d,
                                          float(scale), int(doc), int(kv_head), _ptr(kk), len(kk), _ptr(dk),
                                          _ptr(dv))
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd_dkv_doc failed (rc={rc})")
    return dk, dv


def merge(o_parts, lse_parts):
    """o_parts [m][rows][d], lse_parts [m][rows] -> (o [rows][d], lse [rows])."""
    lib = _load()
    o_parts = np.ascontiguousarray(o_parts, np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, np.float64)
    m, rows, d = o_parts.shape
    o = np.zeros((rows, d), np.float64)
    lse = np.zeros(rows, np.float64)
    rc = lib.oracle_merge(m, rows, d, _ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_merge failed")
    return o, lse


def tile_worklist(p: dict, tile: int = 128, split: bool = False) -> np.ndarray:
    """Query-tile work list, heaviest first.

    Tiles: each document (or, with split=True, each causal block (qc, kc)) is
    cut into query tiles of `tile` rows starting at its first query token.  A
    tile's key range is the causal-prior keys of the same document (of chunk kc
    only when split), so tiles that would be fully masked never appear
    (section 3.2: a query attends only to its own sequence).  Weight = number of
    `tile`-row key tiles in that range.  Order: weight descending, then
    enumeration order (doc / block ascending, query tile ascending).

    Each row: q_row0, q_rows, kv_row0, kv_len, block (-1 when not split),
    row offset of the tile inside its query chunk (inside its document when
    not split), weight, document length when not split (0 when split).
    """
    items = []
    ct = p["chunk_table"]
    cu = p["cu_seqlens"]
    if not split:
        n = len(cu) - 1
        for i in range(n):
            start, s = int(cu[i]), int(cu[i + 1] - cu[i])
            for qt in range((s + tile - 1) // tile):
                q0 = start + qt * tile
                qrows = min(tile, s - qt * tile)
                kv_len = qt * tile + qrows
                w = (kv_len + tile - 1) // tile
                items.append((q0, qrows, start, kv_len, -1, qt * tile, w, s))
    else:
        for b, (qc, kc) in enumerate(p["block_table"]):
            qdoc, _, qbeg, qlen = (int(x) for x in ct[qc])
            _, _, kbeg, klen = (int(x) for x in ct[kc])
            for qt in range((qlen + tile - 1) // tile):
                q0 = qbeg + qt * tile
                qrows = min(tile, qlen - qt * tile)
                if qc == kc:
                    kv_len = qt * tile + qrows
                else:
                    kv_len = klen
                w = (kv_len + tile - 1) // tile
                items.append((q0, qrows, kbeg, kv_len, b, qt * tile, w, 0))
    order = sorted(range(len(items)), key=lambda j: (-items[j][6], j))
    return np.array([items[j] for j in order], dtype=np.int32).reshape(-1, 8)
