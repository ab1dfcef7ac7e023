"""GPU parity of the backward pass (dq, dk, dv through the C ABI) against the
fp64 oracle on the same bf16 inputs.

The GPU path runs its own forward (FUSED) for o and lse, then the backward;
the oracle computes the exact gradients from q, k, v and dout alone.

Tolerances, per gradient tensor X with reference R, from the arithmetic:
P and dS enter the tensor-core products rounded to bf16 (relative 2^-8 each,
the unit roundoff of round-to-nearest with 8 significant bits),
D = rowsum(dout * o) uses the bf16 forward output, and the results are
rounded to bf16 (relative 2^-8).  Independent roundings over the summed keys
or queries grow like the square root of their count relative to the largest
term, so we require max|X - R| <= 2e-2 max|R| and mean|X - R| <= 1e-2 mean|R|.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import packed_varlen_attention_aware_gb300 as pkg
from packed_varlen_attention_aware_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_TOL, MEAN_TOL = 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def _inputs(lengths, hq, hkv, d, seed, std=1.0):
    T = sum(lengths)
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(T, hq, d, generator=g) * std).to(torch.bfloat16)
    k = (torch.randn(T, hkv, d, generator=g) * std).to(torch.bfloat16)
    v = (torch.randn(T, hkv, d, generator=g) * std).to(torch.bfloat16)
    do = torch.randn(T, hq, d, generator=g).to(torch.bfloat16)
    return q, k, v, do


def run_bwd(q, k, v, do, lengths, C):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    dl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    o, lse, plan = pkg.attention(qd, kd, vd, dl, C)
    dq, dk, dv = pkg.attention_backward(plan, qd, kd, vd, o, lse, dod)
    st = pkg.hdp_device_status()
    assert st is None or st == pkg.HDP_OK
    torch.cuda.synchronize()
    plan.destroy()
    return dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy()


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def compare(name, got, ref):
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_TOL * float(np.abs(ref).max()) + 1e-6, f"{name}: max err {mx} vs max|ref| {np.abs(ref).max()}"
    assert mean <= MEAN_TOL * float(np.abs(ref).mean()) + 1e-7, f"{name}: mean err {mean} vs mean|ref| {np.abs(ref).mean()}"


def full_bwd_parity(lengths, hq, hkv, d, C, seed=0):
    q, k, v, do = _inputs(lengths, hq, hkv, d, seed)
    dq, dk, dv = run_bwd(q, k, v, do, lengths, C)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    rq, rk, rv = oracle.attention_bwd(_bits(q), _bits(k), _bits(v), _bits(do), cu, hq, hkv, d, 1.0 / math.sqrt(d))
    compare("dq", dq, rq)
    compare("dk", dk, rk)
    compare("dv", dv, rv)


def test_tiny():
    w = wl.workload("tiny")
    full_bwd_parity(list(w.lengths), w.hq, w.hkv, w.d, w.capacity)


@pytest.mark.parametrize("lengths,hq,hkv,d,C", [
    ([1], 2, 1, 64, 128),
    ([1, 2, 3, 127, 128, 129], 4, 2, 128, 128),
    ([300, 1, 255, 513], 8, 2, 128, 256),
    ([1000, 17, 640], 6, 2, 64, 384),     # group of 3
    ([129, 257, 383], 3, 3, 128, 128),    # no GQA
    ([2048, 100, 1500, 33], 32, 8, 128, 512),
])
def test_small_cases(lengths, hq, hkv, d, C):
    full_bwd_parity(lengths, hq, hkv, d, C, seed=len(lengths))


def test_one_token_documents_closed_form():
    """One-token documents: P = 1, so dV is the sum of dO over the GQA group's
    query heads, and dS = P (dP - D) = 0 with dP = D = dO . v: dQ = dK = 0 up to
    the rounding of dP (tensor core) against D (row sum)."""
    n, hq, hkv, d = 1000, 4, 2, 128
    q, k, v, do = _inputs([1] * n, hq, hkv, d, 41)
    dq, dk, dv = run_bwd(q, k, v, do, [1] * n, 128)
    grp = hq // hkv
    ref_dv = do.double().view(n, hkv, grp, d).sum(2).numpy()
    compare("dv", dv, ref_dv)
    assert np.abs(dq).max() <= 1e-2 * float(np.abs(q.float().numpy()).max())
    assert np.abs(dk).max() <= 1e-2 * float(np.abs(k.float().numpy()).max())


def test_many_tiny_documents_and_odd_capacity():
    """200 documents of 1 to 40 tokens (key tiles straddling many document
    boundaries) with C = 100, which the backward does not depend on."""
    rng = np.random.default_rng(17)
    lengths = [int(x) for x in rng.integers(1, 41, 200)]
    full_bwd_parity(lengths, 4, 1, 64, 100, seed=19)


def test_one_kv_head_for_32_query_heads():
    """Multi-query attention: dK and dV sum over a GQA group of 32."""
    full_bwd_parity([700, 300, 129], 32, 1, 128, 256, seed=23)


def test_large_logits():
    """Q and K with standard deviation 3 (scores of standard deviation 9
    nats): sharply peaked rows of P."""
    lengths, hq, hkv, d, C = [1500, 700, 129], 8, 2, 128, 256
    q, k, v, do = _inputs(lengths, hq, hkv, d, 31)
    q = (q.float() * 3).to(torch.bfloat16)
    k = (k.float() * 3).to(torch.bfloat16)
    dq, dk, dv = run_bwd(q, k, v, do, lengths, C)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    rq, rk, rv = oracle.attention_bwd(_bits(q), _bits(k), _bits(v), _bits(do), cu, hq, hkv, d, 1.0 / math.sqrt(d))
    compare("dq", dq, rq)
    compare("dk", dk, rk)
    compare("dv", dv, rv)


def test_deterministic():
    """dq, dk and dv each accumulate in one CTA's TMEM in a fixed order, with
    no atomics: bit-identical across runs."""
    lengths, hq, hkv, d = [700, 1300, 5], 8, 2, 128
    q, k, v, do = _inputs(lengths, hq, hkv, d, 9)
    a = run_bwd(q, k, v, do, lengths, 256)
    b = run_bwd(q, k, v, do, lengths, 256)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def _identities(w, q, k, v, do, dq, dk, dv):
    """Properties that hold at any size: sum_b dv_b = sum over the group's
    heads of sum_a dO_a (rows of P sum to one) and sum dq.q = sum dk.k per
    document and kv head (both equal sum dS * S)."""
    grp = w.hq // w.hkv
    cu = np.concatenate([[0], np.cumsum(w.lengths)])
    qf, kf, dof = q.float(), k.float(), do.float()
    for i in range(len(w.lengths)):
        a, b = int(cu[i]), int(cu[i + 1])
        for g in range(w.hkv):
            want = dof[a:b, g * grp:(g + 1) * grp].sum(dim=(0, 1)).double()
            got = dv[a:b, g].double().sum(0)
            assert torch.allclose(got, want, rtol=2e-2, atol=2e-2 * float(want.abs().max()) + 1e-2)
            lhs = float((dq[a:b, g * grp:(g + 1) * grp].double() * qf[a:b, g * grp:(g + 1) * grp].double()).sum())
            rhs = float((dk[a:b, g].double() * kf[a:b, g].double()).sum())
            scale = float((dq[a:b, g * grp:(g + 1) * grp].double().abs() * qf[a:b, g * grp:(g + 1) * grp].double().abs()).sum())
            assert abs(lhs - rhs) <= 2e-2 * scale + 1e-3


@pytest.mark.parametrize("name", ["mb32k", "seq128k"])
def test_named_workload_sampled(name):
    w = wl.workload(name)
    q, k, v = wl.qkv(w, device="cpu")
    g = torch.Generator().manual_seed(77)
    do = torch.randn(w.total_tokens, w.hq, w.d, generator=g).to(torch.bfloat16)
    lengths = list(w.lengths)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    dl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    o, lse, plan = pkg.attention(qd, kd, vd, dl, w.capacity)
    dq, dk, dv = pkg.attention_backward(plan, qd, kd, vd, o, lse, dod)
    torch.cuda.synchronize()
    plan.destroy()
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    _identities(w, q, k, v, do, dq, dk, dv)
    rng = np.random.default_rng(5)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    scale = 1.0 / math.sqrt(w.d)
    qb, kb, vb, dob = _bits(q), _bits(k), _bits(v), _bits(do)
    # dq rows: starts, ends and random positions of every document
    toks = []
    for i in range(len(lengths)):
        s = lengths[i]
        toks += [cu[i], cu[i] + s - 1] + list(cu[i] + rng.integers(0, s, 3))
    toks = np.array(toks, dtype=np.int64)
    heads = rng.integers(0, w.hq, len(toks)).astype(np.int32)
    ref = oracle.attention_bwd_dq_rows(qb, kb, vb, dob, cu, w.hq, w.hkv, w.d, scale, toks, heads)
    compare(f"{name} dq rows", dq.float().numpy()[toks, heads], ref)
    # dk / dv rows of keys near each document's end (few later queries)
    kt = []
    for i in range(len(lengths)):
        s = lengths[i]
        kt += list(cu[i] + s - 1 - rng.integers(0, min(s, 96), 3))
    kt = np.array(kt, dtype=np.int64)
    kh = rng.integers(0, w.hkv, len(kt)).astype(np.int32)
    rk, rv = oracle.attention_bwd_dkv_rows(qb, kb, vb, dob, cu, w.hq, w.hkv, w.d, scale, kt, kh)
    compare(f"{name} dk rows", dk.float().numpy()[kt, kh], rk)
    compare(f"{name} dv rows", dv.float().numpy()[kt, kh], rv)
    if name == "mb32k":
        # keys at the start, the middle and the end of the longest document:
        # the early ones accumulate over every query tile of the document and
        # every query head of the group inside one CTA's TMEM
        i = int(np.argmax(lengths))
        s, a = lengths[i], int(cu[i])
        mid = s // 2
        keys = np.array([0, 1, int(rng.integers(2, 128)), mid - 1, mid, mid + int(rng.integers(1, 128)),
                         s - 129, s - 2, s - 1], np.int64)
        doc_cu = np.array([0, s], np.int32)  # a document's gradients do not depend on its neighbours
        for g in (0, int(rng.integers(1, w.hkv))):
            rk, rv = oracle.attention_bwd_dkv_doc(qb[a:a + s], kb[a:a + s], vb[a:a + s], dob[a:a + s], doc_cu, w.hq,
                                                  w.hkv, w.d, scale, 0, g, keys)
            compare(f"{name} dk, doc {i} kv head {g}", dk.float().numpy()[a + keys, g], rk)
            compare(f"{name} dv, doc {i} kv head {g}", dv.float().numpy()[a + keys, g], rv)


def test_workspace_and_argument_checks():
    lengths = [300]
    dl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    with pkg.hdp_plan_create(dl, 256) as plan:
        need = pkg.hdp_attention_bwd_workspace_bytes(plan, 4, 128)
        assert need >= 300 * 4 * 4  # D = rowsum(dout * o), fp32 [hq][T]
        q = torch.zeros(300, 4, 128, dtype=torch.bfloat16, device="cuda")
        k = torch.zeros(300, 2, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros(4, 300, dtype=torch.float32, device="cuda")
        small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
        with pytest.raises(pkg.HdpError) as e:
            pkg.hdp_attention_bwd(plan, q, k, k, q, lse, q, 4, 2, 128, 0.1, small, q, k, k)
        assert e.value.status == pkg.HDP_ERR_INVALID_ARGUMENT
        with pytest.raises(pkg.HdpError) as e:
            pkg.hdp_attention_bwd(plan, q, k, k, q, lse, q, 4, 2, 96, 0.1, small, q, k, k)
        assert e.value.status == pkg.HDP_ERR_UNSUPPORTED
