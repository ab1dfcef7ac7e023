"""ctypes binding of libhdpattn.so with the C ABI's names (include/hdpattn.h).

Argument marshalling only: torch tensors are passed as device pointers and
every step runs in the library's CUDA kernels.  There is no fallback: if the
shared library is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libhdpattn.so")

HDP_OK = 0
HDP_ERR_INVALID_ARGUMENT = 1
HDP_ERR_UNSUPPORTED = 2
HDP_ERR_OUT_OF_MEMORY = 3
HDP_ERR_CUDA = 4
HDP_ERR_DEVICE_TIMEOUT = 5
HDP_MODE_FUSED = 0
HDP_MODE_SPLIT = 1
HDP_PLAN_DEFAULT = 0
HDP_PLAN_NO_SHARDS = 1
HDP_PLAN_NO_SPLIT = 2
HDP_BALANCE_DP = 0
HDP_BALANCE_PP = 1

# Every symbol include/hdpattn.h declares.
EXPORTED = (
    "hdp_plan_create", "hdp_plan_create_ex", "hdp_plan_view", "hdp_plan_destroy",
    "hdp_attention_workspace_bytes", "hdp_attention_fwd", "hdp_lse_merge", "hdp_lse_merge_rows",
    "hdp_flops_per_shard", "hdp_device_status", "hdp_status_string", "hdp_last_error_message",
    "hdp_kernel_launch_count", "hdp_host_sync_count", "hdp_set_wait_budget", "hdp_attention_fwd_split_noalloc",
    "hdp_ring_step_compute", "hdp_ring_attention_time", "hdp_offload_ranks", "hdp_fit_cost_model",
    "hdp_balance_schedule", "hdp_attention_bwd_workspace_bytes", "hdp_attention_bwd",
)


class OffloadModel(ctypes.Structure):
    """hdp_offload_model_t: T(s) = alpha1 s^2 + beta1 s + gamma, Act(s) = alpha2 s + beta2."""
    _fields_ = [("alpha1", ctypes.c_double), ("beta1", ctypes.c_double), ("gamma", ctypes.c_double),
                ("alpha2", ctypes.c_double), ("beta2", ctypes.c_double), ("bw_d2h", ctypes.c_double),
                ("bw_h2d", ctypes.c_double), ("layers", ctypes.c_int32)]


class HdpError(RuntimeError):
    def __init__(self, status: int, call: str, message: str):
        self.status = status
        super().__init__(f"{call} failed: status {status} ({message})")


class PlanView(ctypes.Structure):
    _fields_ = [
        ("num_docs", ctypes.c_int32), ("capacity", ctypes.c_int32), ("num_chunks", ctypes.c_int32),
        ("num_shards", ctypes.c_int32), ("num_blocks", ctypes.c_int64), ("total_tokens", ctypes.c_int64),
        ("max_doc_len", ctypes.c_int32), ("tile", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p), ("chunk_offsets", ctypes.c_void_p), ("block_offsets", ctypes.c_void_p),
        ("chunk_table", ctypes.c_void_p), ("block_table", ctypes.c_void_p), ("chunk_pairs", ctypes.c_void_p),
        ("shard_of_chunk", ctypes.c_void_p), ("tiles_fused", ctypes.c_void_p), ("num_tiles_fused", ctypes.c_int64),
        ("tiles_split", ctypes.c_void_p), ("num_tiles_split", ctypes.c_int64),
    ]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load (once) and return the ctypes handle; raises if the library is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with packed_varlen_attention_aware_gb300.build.build()")
        lib = ctypes.CDLL(p)
        V, I32, I64, U32, F32, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                     ctypes.c_float, ctypes.c_size_t)
        sig = {
            "hdp_plan_create": [V, I32, I32, V, V],
            "hdp_plan_create_ex": [V, I32, I32, U32, V, V],
            "hdp_plan_view": [V, ctypes.POINTER(PlanView)],
            "hdp_plan_destroy": [V],
            "hdp_attention_workspace_bytes": [V, I32, I32, I32, ctypes.POINTER(SZ)],
            "hdp_attention_fwd": [V, V, V, V, I32, I32, I32, F32, I32, V, SZ, V, V, V],
            "hdp_attention_fwd_split_noalloc": [V, V, V, V, I32, I32, I32, F32, V, V, V],
            "hdp_lse_merge": [V, V, V, I32, I32, V, V, V],
            "hdp_lse_merge_rows": [I32, I64, I32, V, V, V, V, V],
            "hdp_flops_per_shard": [V, I32, I32, V, V],
            "hdp_device_status": [V],
            "hdp_set_wait_budget": [I64],
            "hdp_status_string": [ctypes.c_int],
            "hdp_last_error_message": [],
            "hdp_ring_step_compute": [V, I32, I32, I32, ctypes.c_double, ctypes.POINTER(ctypes.c_double)],
            "hdp_ring_attention_time": [I32, ctypes.c_double, ctypes.c_double, ctypes.POINTER(ctypes.c_double)],
            "hdp_offload_ranks": [ctypes.POINTER(OffloadModel), I64, I64, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(I64)],
            "hdp_fit_cost_model": [V, V, V, I32, I32, V],
            "hdp_balance_schedule": [V, I32, I32, I32, I64, I32, V, V, V],
            "hdp_attention_bwd_workspace_bytes": [V, I32, I32, ctypes.POINTER(SZ)],
            "hdp_attention_bwd": [V, V, V, V, V, V, V, I32, I32, I32, F32, V, SZ, V, V, V, V],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        lib.hdp_kernel_launch_count.argtypes = []
        lib.hdp_kernel_launch_count.restype = ctypes.c_uint64
        lib.hdp_host_sync_count.argtypes = []
        lib.hdp_host_sync_count.restype = ctypes.c_uint64
        lib.hdp_status_string.restype = ctypes.c_char_p
        lib.hdp_last_error_message.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int, call: str):
    if status != HDP_OK:
        msg = load().hdp_last_error_message().decode(errors="replace")
        raise HdpError(status, call, msg)


def _stream(stream):
    import torch

    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class _DeviceArray:
    """Zero-copy view of plan-owned device memory for torch.as_tensor."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


class Plan:
    """Owner of an hdp_plan_t; tables are exposed as torch views (valid while the plan lives)."""

    def __init__(self, handle: ctypes.c_void_p):
        self._h = handle
        v = PlanView()
        _check(load().hdp_plan_view(self._h, ctypes.byref(v)), "hdp_plan_view")
        self.view = v

    @property
    def handle(self):
        return self._h

    def _table(self, name, shape, typestr):
        import torch

        ptr = getattr(self.view, name)
        if not ptr or 0 in shape:
            dt = {"<i4": torch.int32, "<i8": torch.int64}[typestr]
            return torch.zeros(shape, dtype=dt, device="cuda")
        return torch.as_tensor(_DeviceArray(ptr, shape, typestr), device="cuda")

    def tables(self) -> dict:
        """Host copies (numpy) of every table of the plan."""
        v = self.view
        n, nc, nb = v.num_docs, v.num_chunks, v.num_blocks
        out = {
            "cu_seqlens": self._table("cu_seqlens", (n + 1,), "<i4"),
            "chunk_offsets": self._table("chunk_offsets", (n + 1,), "<i4"),
            "block_offsets": self._table("block_offsets", (n + 1,), "<i8"),
            "chunk_table": self._table("chunk_table", (nc, 4), "<i4"),
            "block_table": self._table("block_table", (nb, 2), "<i4"),
            "chunk_pairs": self._table("chunk_pairs", (nc,), "<i8"),
            "tiles_fused": self._table("tiles_fused", (v.num_tiles_fused, 8), "<i4"),
        }
        if v.shard_of_chunk:
            out["shard_of_chunk"] = self._table("shard_of_chunk", (nc,), "<i4")
        if v.tiles_split:
            out["tiles_split"] = self._table("tiles_split", (v.num_tiles_split, 8), "<i4")
        return {k: t.cpu().numpy() for k, t in out.items()}

    def destroy(self):
        if self._h:
            h, self._h = self._h, None
            _check(load().hdp_plan_destroy(h), "hdp_plan_destroy")

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def hdp_plan_create(d_lengths, capacity: int, flags: int = HDP_PLAN_DEFAULT, stream=None) -> Plan:
    """d_lengths: int32 CUDA tensor of document lengths."""
    import torch

    if d_lengths.dtype != torch.int32 or not d_lengths.is_cuda or not d_lengths.is_contiguous():
        raise TypeError("d_lengths must be a contiguous int32 CUDA tensor")
    h = ctypes.c_void_p()
    _check(load().hdp_plan_create_ex(_ptr(d_lengths), d_lengths.numel(), int(capacity), int(flags),
                                     _stream(stream), ctypes.byref(h)), "hdp_plan_create")
    return Plan(h)


def hdp_plan_create_ex(d_lengths, capacity: int, flags: int, stream=None) -> Plan:
    return hdp_plan_create(d_lengths, capacity, flags=flags, stream=stream)


def hdp_plan_view(plan: Plan) -> PlanView:
    return plan.view


def hdp_plan_destroy(plan: Plan):
    plan.destroy()


def hdp_attention_workspace_bytes(plan: Plan, hq: int, d: int, mode: int) -> int:
    n = ctypes.c_size_t()
    _check(load().hdp_attention_workspace_bytes(plan.handle, hq, d, mode, ctypes.byref(n)),
           "hdp_attention_workspace_bytes")
    return int(n.value)


def hdp_attention_fwd(plan: Plan, q, k, v, hq: int, hkv: int, d: int, scale: float, mode: int, workspace, o, lse,
                      stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().hdp_attention_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), hq, hkv, d, float(scale), mode,
                                    _ptr(workspace), ws_bytes, _ptr(o), _ptr(lse), _stream(stream)),
           "hdp_attention_fwd")


def hdp_attention_fwd_split_noalloc(plan: Plan, q, k, v, hq: int, hkv: int, d: int, scale: float, o, lse,
                                    stream=None):
    """SPLIT attention using the library's fixed scratch area (no allocation)."""
    _check(load().hdp_attention_fwd_split_noalloc(plan.handle, _ptr(q), _ptr(k), _ptr(v), hq, hkv, d, float(scale),
                                                  _ptr(o), _ptr(lse), _stream(stream)),
           "hdp_attention_fwd_split_noalloc")


def hdp_attention_bwd_workspace_bytes(plan: Plan, hq: int, d: int) -> int:
    out = ctypes.c_size_t()
    _check(load().hdp_attention_bwd_workspace_bytes(plan.handle, hq, d, ctypes.byref(out)),
           "hdp_attention_bwd_workspace_bytes")
    return out.value


def hdp_attention_bwd(plan: Plan, q, k, v, o, lse, dout, hq: int, hkv: int, d: int, scale: float, workspace, dq, dk,
                      dv, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().hdp_attention_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), hq, hkv,
                                    d, float(scale), _ptr(workspace), ws_bytes, _ptr(dq), _ptr(dk), _ptr(dv),
                                    _stream(stream)),
           "hdp_attention_bwd")


def hdp_lse_merge(plan: Plan, o_part, lse_part, hq: int, d: int, o, lse, stream=None):
    _check(load().hdp_lse_merge(plan.handle, _ptr(o_part), _ptr(lse_part), hq, d, _ptr(o), _ptr(lse),
                                _stream(stream)), "hdp_lse_merge")


def hdp_lse_merge_rows(o_parts, lse_parts, o, lse, stream=None):
    m, rows, d = o_parts.shape
    _check(load().hdp_lse_merge_rows(m, rows, d, _ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse),
                                     _stream(stream)), "hdp_lse_merge_rows")


def hdp_flops_per_shard(plan: Plan, d: int, hq: int, d_out, stream=None):
    _check(load().hdp_flops_per_shard(plan.handle, d, hq, _ptr(d_out), _stream(stream)), "hdp_flops_per_shard")


def hdp_device_status(stream=None):
    _check(load().hdp_device_status(_stream(stream)), "hdp_device_status")


def hdp_status_string(status: int) -> str:
    return load().hdp_status_string(status).decode()


def hdp_kernel_launch_count() -> int:
    return int(load().hdp_kernel_launch_count())


def hdp_host_sync_count() -> int:
    return int(load().hdp_host_sync_count())


def hdp_set_wait_budget(clocks: int) -> None:
    _check(load().hdp_set_wait_budget(int(clocks)), "hdp_set_wait_budget")


def hdp_last_error_message() -> str:
    return load().hdp_last_error_message().decode(errors="replace")


# ---------------------------------------------------------------- cost models (host arithmetic)

def hdp_ring_step_compute(lengths, num_ranks: int, capacity: int, t_blk: float) -> float:
    """t_c = t_blk * sum_i (s_i / (N C))^2 for a pack on a ring of N ranks."""
    import numpy as np

    a = np.ascontiguousarray(lengths, dtype=np.int32)
    out = ctypes.c_double()
    _check(load().hdp_ring_step_compute(a.ctypes.data_as(ctypes.c_void_p), int(a.size), int(num_ranks),
                                        int(capacity), float(t_blk), ctypes.byref(out)), "hdp_ring_step_compute")
    return out.value


def hdp_ring_attention_time(num_ranks: int, t_c: float, t_x: float) -> float:
    """T_attn = (N - 1) * max(t_c, t_x) + t_c."""
    out = ctypes.c_double()
    _check(load().hdp_ring_attention_time(int(num_ranks), float(t_c), float(t_x), ctypes.byref(out)),
           "hdp_ring_attention_time")
    return out.value


def hdp_offload_ranks(model: dict, s: int, capacity: int):
    """Eq. 3: (offload ratio r, rank count D) for a sequence of s tokens."""
    m = OffloadModel(**{k: model[k] for k in ("alpha1", "beta1", "gamma", "alpha2", "beta2", "bw_d2h", "bw_h2d",
                                              "layers")})
    r, d = ctypes.c_double(), ctypes.c_int64()
    _check(load().hdp_offload_ranks(ctypes.byref(m), int(s), int(capacity), ctypes.byref(r), ctypes.byref(d)),
           "hdp_offload_ranks")
    return r.value, int(d.value)


def hdp_fit_cost_model(x, y, degree: int, w=None):
    """Weighted least-squares polynomial coefficients (of x^0 .. x^degree)
    through (x, y); w None = unweighted."""
    import numpy as np

    xa = np.ascontiguousarray(x, dtype=np.float64)
    ya = np.ascontiguousarray(y, dtype=np.float64)
    if xa.shape != ya.shape:
        raise ValueError("x and y differ in length")
    wa = None if w is None else np.ascontiguousarray(w, dtype=np.float64)
    if wa is not None and wa.shape != xa.shape:
        raise ValueError("w and x differ in length")
    coef = np.zeros(int(degree) + 1, dtype=np.float64)
    vp = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    _check(load().hdp_fit_cost_model(vp(xa), vp(ya), vp(wa), int(xa.size), int(degree), vp(coef)),
           "hdp_fit_cost_model")
    return coef


# ---------------------------------------------------------------- balance scheduler (host)

def hdp_balance_schedule(costs, workers: int, buckets: int, delta: int, mode: int = HDP_BALANCE_DP):
    """Section 3.4 balance scheduler.  Returns numpy arrays
    (worker of each micro-batch int32[m], load of each worker int64[workers],
    bucket of each micro-batch int32[m])."""
    import numpy as np

    c = np.ascontiguousarray(costs, dtype=np.int64)
    m = int(c.size)
    w = np.empty(m, dtype=np.int32)
    load = np.empty(int(workers), dtype=np.int64)
    b = np.empty(m, dtype=np.int32)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(load_lib().hdp_balance_schedule(vp(c), m, int(workers), int(buckets), int(delta), int(mode), vp(w),
                                           vp(load), vp(b)), "hdp_balance_schedule")
    return w, load, b


load_lib = load
