"""SPLIT attention without allocation, against the workspace version and the
fp64 oracle.

hdp_attention_fwd_split_noalloc serves callers that cannot allocate device
memory when they run attention: serving processes that reserve all device
memory at start-up and forbid allocation on the request path, and callers
that must not take the device-wide synchronisation cudaMalloc/cudaFree can
imply.  Its partials live in one fixed scratch array inside the library.  It
runs the same kernels as hdp_attention_fwd in SPLIT mode with a
caller-provided workspace, so its results must equal that version's bit for
bit, call after call, although every call reuses the same scratch array; and
both must match the oracle within the attention tolerances.  This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import packed_varlen_attention_aware_gb300 as pkg
from packed_varlen_attention_aware_gb300 import workloads as wl

from parity_util import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def _case(lengths, hq, hkv, d, C, seed):
    w = wl.Workload("noalloc", tuple(lengths), C, hq, hkv, d, 1.0, seed)
    q, k, v = wl.qkv(w)  # CPU: the oracle reads the same bytes
    dl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    return w, q, k, v, dl


def _outputs(w):
    o = torch.empty((w.total_tokens, w.hq, w.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.hq, w.total_tokens), dtype=torch.float32, device="cuda")
    return o, lse


def _with_workspace(plan, w, q, k, v):
    o, lse = _outputs(w)
    ws = torch.empty(pkg.hdp_attention_workspace_bytes(plan, w.hq, w.d, pkg.HDP_MODE_SPLIT), dtype=torch.uint8,
                     device="cuda")
    pkg.hdp_attention_fwd(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, pkg.HDP_MODE_SPLIT, ws, o, lse)
    pkg.hdp_device_status()
    return o, lse


def _no_alloc(plan, w, q, k, v):
    o, lse = _outputs(w)
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    pkg.hdp_attention_fwd_split_noalloc(plan, q, k, v, w.hq, w.hkv, w.d, w.scale, o, lse)
    pkg.hdp_device_status()
    assert torch.cuda.memory_allocated() == before
    return o, lse


def test_two_calls_in_a_row_match_the_workspace_version_and_the_oracle():
    # two different problems back to back: the second call must not see the
    # first one's partials in the shared scratch array
    cases = [([64, 128, 256, 512], 4, 4, 64, 256, 0), ([700, 1300, 5, 129], 8, 2, 128, 256, 1)]
    for lengths, hq, hkv, d, C, seed in cases:
        w, q, k, v, dl = _case(lengths, hq, hkv, d, C, seed)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        with pkg.hdp_plan_create(dl, C) as plan:
            assert plan.view.num_blocks > plan.view.num_chunks  # several partials merged per row
            ref_o, ref_l = _with_workspace(plan, w, qd, kd, vd)
            got_o, got_l = _no_alloc(plan, w, qd, kd, vd)
        assert torch.equal(got_o, ref_o) and torch.equal(got_l, ref_l), f"{lengths}: differs from the workspace path"
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        o_ref, lse_ref = oracle.attention(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), cu, hq, hkv, d,
                                          w.scale)
        for name, o, lse in (("no-alloc", got_o, got_l), ("workspace", ref_o, ref_l)):
            compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, f"{name} {lengths}")


def test_rejects_plans_beyond_the_static_maximum():
    # one 32,768-token document at C = 8,192: 4 chunks, 10 causal blocks;
    # 10 x 8192 rows x 32 heads x (128 + 1) x 4 bytes = 1.35 GB > 64 MiB
    w, q, k, v, dl = _case([8192 * 4], 32, 8, 128, 8192, 2)
    with pkg.hdp_plan_create(dl, 8192) as plan:
        assert plan.view.num_chunks == 4 and plan.view.num_blocks == 10
        with pytest.raises(pkg.HdpError) as e:
            _no_alloc(plan, w, q.cuda(), k.cuda(), v.cuda())
        assert e.value.status == pkg.HDP_ERR_INVALID_ARGUMENT
        assert "static maximum" in str(e.value)
