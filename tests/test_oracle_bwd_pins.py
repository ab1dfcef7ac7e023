"""Pins of the backward oracle (gradients of the document-masked causal
attention) to facts outside its own formulas:

- central finite differences of the oracle's fp64 forward: with
  L = sum O * G, every entry of dq, dk, dv equals dL/dx to ~1e-8;
- closed forms: a one-token document has P = 1, O = v, so dv = dO and
  dq = dk = 0; gradients of sums (sum_b dv_b = sum over the group's query
  heads of sum_a dO_a, because each row of P sums to one; the total of
  dq . q equals the total of dk . k, both being sum dS * S);
- GQA: dk, dv of a kv head equal the sums over its query heads of the
  gradients of the same problem with K, V repeated per query head;
- document independence: a document's gradients do not depend on the other
  documents packed beside it.
"""
import numpy as np
import pytest

import oracle


def _rand(shape, rng, scale=1.0):
    return rng.normal(0, scale, shape)


def _loss(q, k, v, g, cu, hq, hkv, d, scale):
    o, _ = oracle.attention_f64(q, k, v, cu, hq, hkv, d, scale)
    return float(np.sum(o * g))


@pytest.mark.parametrize("lengths,hq,hkv,d", [([5, 3], 4, 2, 8), ([1, 6], 2, 2, 4), ([7], 3, 1, 5)])
def test_finite_differences(lengths, hq, hkv, d):
    rng = np.random.default_rng(sum(lengths) * 10 + hq)
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v = _rand((T, hq, d), rng), _rand((T, hkv, d), rng), _rand((T, hkv, d), rng)
    g = _rand((T, hq, d), rng)
    scale = 0.7
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, cu, hq, hkv, d, scale)
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (_loss(args_p["q"], args_p["k"], args_p["v"], g, cu, hq, hkv, d, scale)
                  - _loss(args_m["q"], args_m["k"], args_m["v"], g, cu, hq, hkv, d, scale)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_single_token_documents():
    rng = np.random.default_rng(1)
    hq, hkv, d = 4, 2, 6
    cu = np.array([0, 1, 2, 3], np.int32)
    q, k, v = _rand((3, hq, d), rng), _rand((3, hkv, d), rng), _rand((3, hkv, d), rng)
    g = _rand((3, hq, d), rng)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, cu, hq, hkv, d, 0.5)
    assert np.all(dq == 0) and np.allclose(dk, 0, atol=1e-15)
    assert np.allclose(dv, g.reshape(3, hkv, hq // hkv, d).sum(axis=2), rtol=1e-14, atol=0)


def test_sum_identities():
    rng = np.random.default_rng(2)
    hq, hkv, d = 4, 2, 8
    lengths = [9, 4, 13]
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v = _rand((T, hq, d), rng), _rand((T, hkv, d), rng), _rand((T, hkv, d), rng)
    g = _rand((T, hq, d), rng)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, cu, hq, hkv, d, 0.3)
    grp = hq // hkv
    for i in range(len(lengths)):
        a, b = cu[i], cu[i + 1]
        for kvh in range(hkv):
            heads = range(kvh * grp, (kvh + 1) * grp)
            assert np.allclose(dv[a:b, kvh].sum(0), sum(g[a:b, h].sum(0) for h in heads), rtol=1e-12, atol=1e-12)
            lhs = sum(np.sum(dq[a:b, h] * q[a:b, h]) for h in heads)
            rhs = np.sum(dk[a:b, kvh] * k[a:b, kvh])
            assert lhs == pytest.approx(rhs, rel=1e-10, abs=1e-12)


def test_gqa_equals_repeated_heads():
    rng = np.random.default_rng(3)
    hq, hkv, d = 6, 2, 4
    lengths = [7, 5]
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v = _rand((T, hq, d), rng), _rand((T, hkv, d), rng), _rand((T, hkv, d), rng)
    g = _rand((T, hq, d), rng)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, cu, hq, hkv, d, 0.4)
    kr, vr = np.repeat(k, hq // hkv, axis=1), np.repeat(v, hq // hkv, axis=1)
    dq2, dk2, dv2 = oracle.attention_bwd(q, kr, vr, g, cu, hq, hq, d, 0.4)
    assert np.allclose(dq, dq2, rtol=1e-13, atol=1e-15)
    assert np.allclose(dk, dk2.reshape(T, hkv, hq // hkv, d).sum(2), rtol=1e-12, atol=1e-14)
    assert np.allclose(dv, dv2.reshape(T, hkv, hq // hkv, d).sum(2), rtol=1e-12, atol=1e-14)


def test_document_independence_and_dq_rows():
    rng = np.random.default_rng(4)
    hq, hkv, d = 4, 1, 8
    docs = [6, 11, 3]
    data = [(_rand((s, hq, d), rng), _rand((s, hkv, d), rng), _rand((s, hkv, d), rng), _rand((s, hq, d), rng))
            for s in docs]
    alone = [oracle.attention_bwd(*x, np.array([0, s], np.int32), hq, hkv, d, 0.35) for x, s in zip(data, docs)]
    packed = [np.concatenate([x[j] for x in data]) for j in range(4)]
    cu = np.concatenate([[0], np.cumsum(docs)]).astype(np.int32)
    dq, dk, dv = oracle.attention_bwd(*packed, cu, hq, hkv, d, 0.35)
    for i, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        assert np.array_equal(dq[a:b], alone[i][0])
        assert np.array_equal(dk[a:b], alone[i][1])
        assert np.array_equal(dv[a:b], alone[i][2])
    toks = np.array([0, 5, 6, 16, 19])
    heads = np.array([0, 3, 1, 2, 0], np.int32)
    rows = oracle.attention_bwd_dq_rows(*packed, cu, hq, hkv, d, 0.35, toks, heads)
    assert np.array_equal(rows, dq[toks, heads])
    kt = np.array([0, 5, 6, 16, 17, 19])
    kh = np.zeros(len(kt), np.int32)
    dk_r, dv_r = oracle.attention_bwd_dkv_rows(*packed, cu, hq, hkv, d, 0.35, kt, kh)
    assert np.allclose(dk_r, dk[kt, 0], rtol=1e-12, atol=1e-14)
    assert np.allclose(dv_r, dv[kt, 0], rtol=1e-12, atol=1e-14)


def test_dkv_of_document_keys_against_finite_differences():
    """dk, dv of chosen keys of one document (the per-document form used on
    long documents) against central differences of the fp64 forward, and
    against the whole-batch gradients."""
    rng = np.random.default_rng(6)
    hq, hkv, d = 4, 2, 3
    lengths = [5, 12, 4]
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v = _rand((T, hq, d), rng), _rand((T, hkv, d), rng), _rand((T, hkv, d), rng)
    g = _rand((T, hq, d), rng)
    scale = 0.45
    keys = np.array([0, 6, 11, 3])
    doc, kvh = 1, 1
    dk, dv = oracle.attention_bwd_dkv_doc(q, k, v, g, cu, hq, hkv, d, scale, doc, kvh, keys)
    eps = 1e-6
    for i, j in enumerate(keys):
        tok = cu[doc] + j
        for name, x, grad in (("k", k, dk), ("v", v, dv)):
            for c in range(d):
                xp, xm = x.copy(), x.copy()
                xp[tok, kvh, c] += eps
                xm[tok, kvh, c] -= eps
                args_p = {"k": k, "v": v}
                args_m = dict(args_p)
                args_p[name], args_m[name] = xp, xm
                fd = (_loss(q, args_p["k"], args_p["v"], g, cu, hq, hkv, d, scale)
                      - _loss(q, args_m["k"], args_m["v"], g, cu, hq, hkv, d, scale)) / (2 * eps)
                assert abs(fd - grad[i, c]) <= 1e-7 * max(1.0, abs(fd)), (name, j, c, fd, grad[i, c])
    _, dk_all, dv_all = oracle.attention_bwd(q, k, v, g, cu, hq, hkv, d, scale)
    assert np.allclose(dk, dk_all[cu[doc] + keys, kvh], rtol=1e-12, atol=1e-14)
    assert np.allclose(dv, dv_all[cu[doc] + keys, kvh], rtol=1e-12, atol=1e-14)
