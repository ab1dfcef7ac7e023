"""Seeded synthetic workloads: document lengths and bf16 Q/K/V.

This module only draws inputs; it holds none of the attention, plan or merge
arithmetic, so both the CUDA path and the CPU oracle's tests may use it.

The pages measure on ByteDance's production data and on GitHub data, neither of
which is available here; these draws stand in for their shapes
("ByteScale: Communication-Efficient Scaling of LLM Training with a 2048K
Context Length on 16384 GPUs", section 2, Figure 1: skewed lengths where 1% of
samples, at 128K and longer, hold about 44% of the tokens; ~32K-token packed
micro-batches).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    lengths: tuple
    capacity: int
    hq: int
    hkv: int
    d: int
    std: float = 1.0
    seed: int = 0
    info: dict = field(default_factory=dict, compare=False)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def lengths_mb32k(seed: int = 0, total: int = 32768):
    """floor(2^U), U ~ Uniform(8, 15), drawn until the pack holds `total`
    tokens; the last document is truncated to fit."""
    rng = np.random.default_rng(seed)
    out, t = [], 0
    while t < total:
        s = int(math.floor(2.0 ** rng.uniform(8.0, 15.0)))
        s = min(s, total - t)
        out.append(s)
        t += s
    return out


def lengths_mix1m(seed: int = 0, total: int = 1 << 20, lo_share: float = 0.40, hi_share: float = 0.45):
    """Skewed mixture: 80% uniform in [256, 4096], 19% log-uniform in
    [4K, 128K), 1% log-uniform in [128K, 512K); lengths are floor(e^u) for the
    log-uniform parts.  Drawn until `total` tokens, the last truncated; the
    whole batch is redrawn from the same stream until the tokens of sequences
    of 128K and longer (judged after truncation) make up [lo_share, hi_share].
    Returns (lengths, attempts)."""
    rng = np.random.default_rng(seed)
    attempts = 0
    while True:
        attempts += 1
        out, t = [], 0
        while t < total:
            r = rng.uniform()
            if r < 0.80:
                s = int(rng.integers(256, 4096, endpoint=True))
            elif r < 0.99:
                s = int(math.floor(math.exp(rng.uniform(math.log(4096), math.log(131072)))))
            else:
                s = int(math.floor(math.exp(rng.uniform(math.log(131072), math.log(524288)))))
            s = min(s, total - t)
            out.append(s)
            t += s
        long_tokens = sum(s for s in out if s >= 131072)
        share = long_tokens / total
        if lo_share <= share <= hi_share:
            return out, attempts


def workload(name: str, seed: int = 0) -> Workload:
    """The five named workloads."""
    if name == "tiny":
        return Workload("tiny", (64, 128, 256, 512), 256, 4, 4, 64, 1.0, seed)
    if name == "mb32k":
        return Workload("mb32k", tuple(lengths_mb32k(seed)), 32768, 32, 8, 128, 1.0, seed)
    if name == "seq128k":
        return Workload("seq128k", (131072,), 8192, 32, 8, 128, 1.0, seed)
    if name == "mix1m":
        lens, attempts = lengths_mix1m(seed)
        return Workload("mix1m", tuple(lens), 8192, 32, 8, 128, 1.0, seed, {"attempts": attempts})
    if name == "seq2m":
        return Workload("seq2m", (2097152,), 8192, 32, 8, 128, 0.5, seed)
    raise KeyError(name)


NAMES = ("tiny", "mb32k", "seq128k", "mix1m", "seq2m")


def qkv(w: Workload, device: str = "cpu", seed: int | None = None):
    """bf16 Q [T][hq][d], K and V [T][hkv][d] drawn as fp32 N(0, std^2) and
    rounded to bf16 (round to nearest even).  Returns torch tensors on
    `device`; the same seed on the same device gives the same bytes."""
    import torch

    s = w.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(1_000_003 * s + 17)
    T = w.total_tokens
    out = []
    for shape in ((T, w.hq, w.d), (T, w.hkv, w.d), (T, w.hkv, w.d)):
        x = torch.empty(shape, dtype=torch.bfloat16, device=device)
        # fill in slabs to bound the fp32 staging buffer
        flat = x.view(-1)
        step = 1 << 26
        for a in range(0, flat.numel(), step):
            b = min(flat.numel(), a + step)
            flat[a:b] = (torch.randn(b - a, generator=g, device=device, dtype=torch.float32) * w.std).to(
                torch.bfloat16)
        out.append(x)
    return tuple(out)


def bf16_bits(t) -> np.ndarray:
    """A bf16 torch tensor's bit patterns as a uint16 numpy array (host)."""
    import torch

    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
