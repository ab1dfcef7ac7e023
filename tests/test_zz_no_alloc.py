"""SPLIT attention without allocation, against the workspace version.

hdp_attention_fwd_split_noalloc is for callers that cannot allocate device
memory when they run attention (CUDA graph capture, servers that reserve all
memory up front, code that must not trigger the synchronisation an allocation
can imply).  It must give the same result as hdp_attention_fwd in SPLIT mode
with a caller-provided workspace, call after call, although every call reuses
the same fixed scratch area.  This file is collected last on purpose.
"""
import math

import numpy as np
import pytest
import torch

import packed_varlen_attention_aware_gb300 as pkg
from packed_varlen_attention_aware_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_MAX_O, TOL_MEAN_O, TOL_MAX_LSE = 1.5e-2, 1e-3, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def _case(lengths, hq, hkv, d, C, seed):
    w = wl.Workload("noalloc", tuple(lengths), C, hq, hkv, d, 1.0, seed)
    q, k, v = (t.cuda() for t in wl.qkv(w))
    dl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    return w, q, k, v, dl


def _with_workspace(plan, w, q, k, v):
    o = torch.empty_like(q)
    lse = torch.empty((w.hq, w.total_tokens), dtype=torch.float32, device="cuda")
    ws = torch.empty(pkg.hdp_attention_workspace_bytes(plan, w.hq, w.d, pkg.HDP_MODE_SPLIT), dtype=torch.uint8,
                     device="cuda")
    pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, pkg.HDP_MODE_SPLIT, ws, o, lse)
    return o, lse


def _no_alloc(plan, w, q, k, v):
    o = torch.empty_like(q)
    lse = torch.empty((w.hq, w.total_tokens), dtype=torch.float32, device="cuda")
    pkg.hdp_attention_fwd_split_noalloc(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, o, lse)
    return o, lse


def _close(a_o, a_l, b_o, b_l):
    do = (a_o.double() - b_o.double()).abs()
    dl = (a_l.double() - b_l.double()).abs()
    assert torch.isfinite(a_o.float()).all() and torch.isfinite(a_l).all()
    assert do.max().item() <= TOL_MAX_O and do.mean().item() <= TOL_MEAN_O and dl.max().item() <= TOL_MAX_LSE


def test_two_calls_in_a_row_match_the_workspace_version():
    # two different problems back to back: the second call must not see the first one's partials
    cases = [([64, 128, 256, 512], 4, 4, 64, 256, 0), ([700, 1300, 5, 129], 8, 2, 128, 256, 1)]
    for lengths, hq, hkv, d, C, seed in cases:
        w, q, k, v, dl = _case(lengths, hq, hkv, d, C, seed)
        with pkg.hdp_plan_create(dl, C) as plan:
            ref_o, ref_l = _with_workspace(plan, w, q, k, v)
            got_o, got_l = _no_alloc(plan, w, q, k, v)
            pkg.hdp_device_status()
            _close(got_o, got_l, ref_o, ref_l)


def test_rejects_plans_beyond_the_static_maximum():
    # 16 chunks of 8192 tokens: 136 blocks x 8192 rows x 32 heads x 129 x 4 bytes >> 64 MiB
    w, q, k, v, dl = _case([8192 * 4], 32, 8, 128, 8192, 2)
    with pkg.hdp_plan_create(dl, 8192) as plan:
        with pytest.raises(pkg.HdpError) as e:
            _no_alloc(plan, w, q, k, v)
        assert e.value.status == pkg.HDP_ERR_INVALID_ARGUMENT
        assert "static maximum" in str(e.value)
