"""Failure detection and memory bounds on the GPU, without a fault.

- Bounded waits: the attention forward's role waits give up after a budget of
  SM clocks.  With the budget set to one clock the first unsatisfied wait of
  a one-CTA launch expires; the kernel must still return (it drains its own
  copies and tensor-core work and frees its tensor memory), the host must
  read HDP_ERR_DEVICE_TIMEOUT from hdp_device_status, the error must clear,
  and the next call must be correct again.
- Guard bands: every output and workspace buffer sits between two 1 MiB
  bands of a known byte pattern; after the call the bands must be unchanged
  bit for bit (no write outside a buffer), and the outputs must still match
  the oracle.  This stands in for a memory checker, which is not available
  on the GPUs these tests run on.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import packed_varlen_attention_aware_gb300 as pkg
from packed_varlen_attention_aware_gb300 import workloads as wl

from parity_util import compare, full_parity, sample_rows, sampled_parity

pytestmark = pytest.mark.gpu

FUSED, SPLIT = pkg.HDP_MODE_FUSED, pkg.HDP_MODE_SPLIT
GUARD = 1 << 20
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


# ---------------------------------------------------------------- bounded waits

def test_expired_wait_reports_timeout_and_the_next_call_recovers():
    lengths, hq, hkv, d, C = [64], 2, 1, 64, 128  # one work unit, so one CTA
    w = wl.Workload("timeout", tuple(lengths), C, hq, hkv, d, 1.0, 3)
    q, k, v = (t.cuda() for t in wl.qkv(w))
    dl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros((hq, 64), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    pkg.hdp_device_status()  # start from a clear error word
    with pkg.hdp_plan_create(dl, C) as plan:
        pkg.hdp_set_wait_budget(1)
        try:
            pkg.hdp_attention_fwd(plan, q, k, v, hq, hkv, d, w.scale, FUSED, None, o, lse)
            torch.cuda.synchronize()  # the kernel returned: no hang, no fault
        finally:
            pkg.hdp_set_wait_budget(0)
        with pytest.raises(pkg.HdpError) as e:
            pkg.hdp_device_status()
        assert e.value.status == pkg.HDP_ERR_DEVICE_TIMEOUT
        assert "bounded wait expired" in str(e.value)
        pkg.hdp_device_status()  # reading the error cleared it
        # the same plan, default budget: correct again
        pkg.hdp_attention_fwd(plan, q, k, v, hq, hkv, d, w.scale, FUSED, None, o, lse)
        pkg.hdp_device_status()
    cu = np.array([0, 64], np.int32)
    o_ref, lse_ref = oracle.attention(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), cu, hq, hkv, d, w.scale)
    compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, "after a timeout")
    full_parity([300, 1, 255, 513], 8, 2, 128, 256, SPLIT)


def test_backward_expired_wait_reports_timeout_and_the_next_call_recovers():
    """The backward's two kernels take the same wait budget: with one clock the
    first unsatisfied wait expires, every role stops and drains, the status
    reads HDP_ERR_DEVICE_TIMEOUT, and the next call is correct."""
    lengths, hq, hkv, d, C = [64], 2, 1, 64, 128
    g = torch.Generator().manual_seed(7)
    q = torch.randn(64, hq, d, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(64, hkv, d, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(64, hkv, d, generator=g).to(torch.bfloat16).cuda()
    do = torch.randn(64, hq, d, generator=g).to(torch.bfloat16).cuda()
    dl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    pkg.hdp_device_status()
    o, lse, plan = pkg.attention(q, k, v, dl, C)
    try:
        pkg.hdp_set_wait_budget(1)
        try:
            pkg.attention_backward(plan, q, k, v, o, lse, do)
            torch.cuda.synchronize()  # both kernels returned
        finally:
            pkg.hdp_set_wait_budget(0)
        with pytest.raises(pkg.HdpError) as e:
            pkg.hdp_device_status()
        assert e.value.status == pkg.HDP_ERR_DEVICE_TIMEOUT
        pkg.hdp_device_status()
        dq, dk, dv = pkg.attention_backward(plan, q, k, v, o, lse, do)
        pkg.hdp_device_status()
    finally:
        plan.destroy()
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    cu = np.array([0, 64], np.int32)
    refs = oracle.attention_bwd(bits(q), bits(k), bits(v), bits(do), cu, hq, hkv, d, 1.0 / d ** 0.5)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        err = np.abs(got.float().cpu().numpy() - ref)
        assert err.max() <= 2e-2 * np.abs(ref).max() + 1e-6, name


# ---------------------------------------------------------------- pacing
# A 327,680-token document: one kv head's K and V rows (168 MB at d = 128)
# exceed L2, so the forward's CTAs pace each other through the library's
# static position table.  Two query heads on one kv head keep it cheap.
LONG = 327680


def _long_case(seed):
    w = wl.Workload("paced", (LONG,), 8192, 2, 1, 128, 1.0, seed)
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", None)
    if l2:
        assert 2 * LONG * w.d * 2 > l2, "the input no longer reaches the paced path"
    q, k, v = wl.qkv(w, device="cuda")
    return w, q, k, v


def test_paced_launch_expired_wait_reports_timeout_and_the_next_call_recovers():
    """A paced launch whose waits expire at once: the pacer warp stops with
    its CTA, the kernel returns, the status reads HDP_ERR_DEVICE_TIMEOUT, and
    the next call on the same plan passes parity."""
    w, q, k, v = _long_case(21)
    dl = torch.tensor(w.lengths, dtype=torch.int32, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros((w.hq, LONG), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    pkg.hdp_device_status()
    with pkg.hdp_plan_create(dl, w.capacity, flags=pkg.HDP_PLAN_NO_SPLIT) as plan:
        pkg.hdp_set_wait_budget(1)
        try:
            pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, FUSED, None, o, lse)
            torch.cuda.synchronize()
        finally:
            pkg.hdp_set_wait_budget(0)
        with pytest.raises(pkg.HdpError) as e:
            pkg.hdp_device_status()
        assert e.value.status == pkg.HDP_ERR_DEVICE_TIMEOUT
        pkg.hdp_device_status()
        pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, FUSED, None, o, lse)
        pkg.hdp_device_status()
    toks, heads = sample_rows(list(w.lengths), w.hq, 40, 21)
    sampled_parity(w, q, k, v, o, lse, toks, heads, "paced, after a timeout")


@pytest.mark.parametrize("mode", [FUSED, SPLIT])
def test_concurrent_paced_launches_match_lone_launches(mode):
    """Launches in flight together on two streams share the pacing table; each
    must give its lone launch's output bit for bit."""
    cases = [_long_case(31), _long_case(32)]
    outs, plans, wss = [], [], []
    for w, q, k, v in cases:
        dl = torch.tensor(w.lengths, dtype=torch.int32, device="cuda")
        plan = pkg.hdp_plan_create(dl, w.capacity, flags=pkg.HDP_PLAN_NO_SPLIT)
        wsb = pkg.hdp_attention_workspace_bytes(plan, w.hq, w.d, mode)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
        plans.append(plan)
        wss.append(ws)
        o = torch.empty_like(q)
        lse = torch.empty((w.hq, LONG), dtype=torch.float32, device="cuda")
        pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, mode, ws, o, lse)
        outs.append((o, lse))
    pkg.hdp_device_status()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    got = []
    torch.cuda.synchronize()
    for (w, q, k, v), plan, st in zip(cases, plans, streams):
        o = torch.empty_like(q)
        lse = torch.empty((w.hq, LONG), dtype=torch.float32, device="cuda")
        got.append((o, lse))
    for rep in range(2):  # two launches per stream, all enqueued before any wait
        for i, ((w, q, k, v), plan, st) in enumerate(zip(cases, plans, streams)):
            # the two streams need separate SPLIT workspaces: each case has its own
            pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, mode, wss[i], got[i][0], got[i][1],
                                  stream=st)
    torch.cuda.synchronize()
    pkg.hdp_device_status()
    for (o, lse), (o2, lse2) in zip(outs, got):
        assert torch.equal(o, o2) and torch.equal(lse, lse2)
    for plan in plans:
        plan.destroy()


# ---------------------------------------------------------------- guard bands

def _guarded(nbytes):
    buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes]


def _bands_intact(buf, nbytes, what):
    lo, hi = buf[:GUARD], buf[GUARD + nbytes:]
    assert bool((lo == PATTERN).all()), f"{what}: write below the buffer"
    assert bool((hi == PATTERN).all()), f"{what}: write above the buffer"


def _run_guarded(w, q, k, v, mode):
    T = w.total_tokens
    o_bytes, lse_bytes = T * w.hq * w.d * 2, w.hq * T * 4
    ob, om = _guarded(o_bytes)
    lb, lm = _guarded(lse_bytes)
    o = om.view(torch.bfloat16).view(T, w.hq, w.d)
    lse = lm.view(torch.float32).view(w.hq, T)
    dl = torch.tensor(w.lengths, dtype=torch.int32, device="cuda")
    with pkg.hdp_plan_create(dl, w.capacity) as plan:
        wsb = pkg.hdp_attention_workspace_bytes(plan, w.hq, w.d, mode)
        wb, wm = _guarded(wsb) if wsb else (None, None)
        pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, mode, wm, o, lse)
        pkg.hdp_device_status()
    _bands_intact(ob, o_bytes, "o")
    _bands_intact(lb, lse_bytes, "lse")
    if wb is not None:
        _bands_intact(wb, wsb, "SPLIT workspace")
    return o, lse


@pytest.mark.parametrize("mode", [FUSED, SPLIT])
@pytest.mark.parametrize("lengths,hq,hkv,d,C", [
    ([64, 128, 256, 512], 4, 4, 64, 256),          # the tiny workload
    ([1, 2, 3, 127, 128, 129], 4, 2, 128, 128),    # ragged tails
    ([1000, 17, 640], 6, 2, 64, 384),              # odd GQA pair
])
def test_guard_bands_small(lengths, hq, hkv, d, C, mode):
    w = wl.Workload("guard", tuple(lengths), C, hq, hkv, d, 1.0, 5)
    q, k, v = wl.qkv(w)
    o, lse = _run_guarded(w, q.cuda(), k.cuda(), v.cuda(), mode)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    o_ref, lse_ref = oracle.attention(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), cu, hq, hkv, d, w.scale)
    compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, f"guarded {lengths} mode {mode}")


@pytest.mark.parametrize("mode", [FUSED, SPLIT])
def test_guard_bands_seq128k(mode):
    w = wl.workload("seq128k")
    q, k, v = wl.qkv(w, device="cuda")
    o, lse = _run_guarded(w, q, k, v, mode)
    toks, heads = sample_rows(list(w.lengths), w.hq, 24, seed=31)
    sampled_parity(w, q, k, v, o, lse, toks, heads, f"guarded seq128k mode {mode}")


def test_guard_bands_backward():
    lengths, hq, hkv, d, C = [1, 2, 3, 127, 128, 129, 700], 8, 2, 128, 256
    T = sum(lengths)
    g = torch.Generator().manual_seed(12)
    q, k, v, do = (torch.randn(T, h, d, generator=g).to(torch.bfloat16) for h in (hq, hkv, hkv, hq))
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    dl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    o, lse, plan = pkg.attention(qd, kd, vd, dl, C)
    bufs = {}
    outs = {}
    for name, heads in (("dq", hq), ("dk", hkv), ("dv", hkv)):
        nbytes = T * heads * d * 2
        b, m = _guarded(nbytes)
        bufs[name] = (b, nbytes)
        outs[name] = m.view(torch.bfloat16).view(T, heads, d)
    wsb = pkg.hdp_attention_bwd_workspace_bytes(plan, hq, d)
    wb, wm = _guarded(wsb)
    pkg.hdp_attention_bwd(plan, qd, kd, vd, o, lse, dod, hq, hkv, d, 1.0 / math.sqrt(d), wm, outs["dq"], outs["dk"],
                          outs["dv"])
    pkg.hdp_device_status()
    plan.destroy()
    for name, (b, nbytes) in bufs.items():
        _bands_intact(b, nbytes, name)
    _bands_intact(wb, wsb, "backward workspace")
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    refs = oracle.attention_bwd(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), wl.bf16_bits(do), cu, hq, hkv, d,
                                1.0 / math.sqrt(d))
    for name, ref in zip(("dq", "dk", "dv"), refs):
        got = outs[name].double().cpu().numpy()
        err = np.abs(got - ref)
        assert err.max() <= 2e-2 * np.abs(ref).max() and err.mean() <= 1e-2 * np.abs(ref).mean(), name
