"""GB300 (sm_103a) document-masked causal attention over packed, chunked
micro-batches -- the local attention step of ByteScale's hybrid data
parallelism ("ByteScale: Communication-Efficient Scaling of LLM Training with
a 2048K Context Length on 16384 GPUs", research digest, sections 3.1-3.2).

The compute path is libhdpattn.so (include/hdpattn.h); this package is its
ctypes binding plus seeded workload generators.  Importing the package does
not load the library; the first call does, and fails loudly if it is absent.
"""
from __future__ import annotations

import math

from .binding import (  # noqa: F401
    EXPORTED,
    HDP_BALANCE_DP,
    HDP_BALANCE_PP,
    HDP_ERR_CUDA,
    HDP_ERR_DEVICE_TIMEOUT,
    HDP_ERR_INVALID_ARGUMENT,
    HDP_ERR_OUT_OF_MEMORY,
    HDP_ERR_UNSUPPORTED,
    HDP_MODE_FUSED,
    HDP_MODE_SPLIT,
    HDP_OK,
    HDP_PLAN_DEFAULT,
    HDP_PLAN_NO_SHARDS,
    HDP_PLAN_NO_SPLIT,
    HdpError,
    OffloadModel,
    Plan,
    hdp_attention_bwd,
    hdp_attention_bwd_workspace_bytes,
    hdp_attention_fwd,
    hdp_attention_fwd_split_noalloc,
    hdp_balance_schedule,
    hdp_attention_workspace_bytes,
    hdp_device_status,
    hdp_fit_cost_model,
    hdp_flops_per_shard,
    hdp_kernel_launch_count,
    hdp_host_sync_count,
    hdp_set_wait_budget,
    hdp_last_error_message,
    hdp_lse_merge,
    hdp_lse_merge_rows,
    hdp_offload_ranks,
    hdp_plan_create,
    hdp_plan_create_ex,
    hdp_plan_destroy,
    hdp_plan_view,
    hdp_ring_attention_time,
    hdp_ring_step_compute,
    hdp_status_string,
    load,
)


def attention(q, k, v, d_lengths, capacity: int, mode: int = HDP_MODE_FUSED, scale: float | None = None,
              plan: Plan | None = None, stream=None):
    """Convenience wrapper: plan (unless given), attention, and (in SPLIT mode)
    the merge.  q [T][hq][d], k/v [T][hkv][d] bf16 CUDA tensors; returns
    (o bf16 [T][hq][d], lse fp32 [hq][T], plan)."""
    import torch

    T, hq, d = q.shape
    hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if plan is None:
        plan = hdp_plan_create(d_lengths, capacity, stream=stream)
    o = torch.empty_like(q)
    lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    ws = None
    nbytes = hdp_attention_workspace_bytes(plan, hq, d, mode)
    if nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    hdp_attention_fwd(plan, q, k, v, hq, hkv, d, scale, mode, ws, o, lse, stream=stream)
    return o, lse, plan


def attention_backward(plan: Plan, q, k, v, o, lse, dout, scale: float | None = None, stream=None):
    """Gradients (dq, dk, dv) of sum(o * dout) for the forward that produced
    (o, lse) with this plan.  bf16 CUDA tensors in the forward's layouts."""
    import torch

    T, hq, d = q.shape
    hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    nbytes = hdp_attention_bwd_workspace_bytes(plan, hq, d)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    hdp_attention_bwd(plan, q, k, v, o, lse, dout, hq, hkv, d, scale, ws, dq, dk, dv, stream=stream)
    return dq, dk, dv
