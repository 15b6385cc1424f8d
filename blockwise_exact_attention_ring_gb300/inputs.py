"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only draws random tensors and
names shapes, so that the CUDA path, the oracle, the tests and the benchmark
all see the same bits.  Nothing here is a stand-in for a dataset; every input
is synthetic, with the shapes of the workloads the ring-attention pages
describe (a 32K-token sequence over 4 devices, 256K-token causal striped
training, a 1M-token Llama-3-8B-shaped layer, and the pages' own 4-device toy
simulation).
"""
from __future__ import annotations

from dataclasses import dataclass, asdict
from typing import Dict, Optional

import torch

LAYOUT_CONTIGUOUS = 0
LAYOUT_STRIPED = 1


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    S: int
    d: int
    n_blocks: int
    layout: int
    causal: bool
    dtype: str          # "f32" or "bf16"
    seed: int
    std: float = 1.0
    spike_frac: float = 0.0   # fraction of key rows scaled by spike_scale
    spike_scale: float = 8.0

    @property
    def L(self) -> int:
        return self.S // self.n_blocks

    def as_config(self) -> Dict:
        c = asdict(self)
        c["workload"] = c.pop("name")
        c["layout"] = "striped" if self.layout == LAYOUT_STRIPED else "contiguous"
        return c


WORKLOADS: Dict[str, Workload] = {w.name: w for w in [
    # the pages' 4-device simulation: 4 ranks x block 8, dim 16, fp32, seed 0
    Workload("ring4-s32-d16-f32-example", 1, 1, 1, 32, 16, 4, LAYOUT_CONTIGUOUS,
             False, "f32", 0),
    # PyTorch context-parallel example shape, non-causal, over 2 ranks
    Workload("ring2-s4k-h4-d64-bf16", 1, 4, 4, 4096, 64, 2, LAYOUT_CONTIGUOUS,
             False, "bf16", 1002),
    # 32K tokens over 4 ranks, causal, grouped-query heads
    Workload("ring4-s32k-h32kv8-d128-causal-contiguous", 1, 32, 8, 32768, 128, 4,
             LAYOUT_CONTIGUOUS, True, "bf16", 1003),
    # 256K-token causal training sequence over 8 ranks, both layouts
    Workload("ring8-s256k-h32kv8-d128-causal-contiguous", 1, 32, 8, 262144, 128, 8,
             LAYOUT_CONTIGUOUS, True, "bf16", 1004),
    Workload("ring8-s256k-h32kv8-d128-causal-striped", 1, 32, 8, 262144, 128, 8,
             LAYOUT_STRIPED, True, "bf16", 1004),
    # 1M-token Llama-3-8B-shaped layer, striped over 32 ranks, N(0, 0.5^2)
    # with 1 % of key rows scaled by 8 to stress the running max
    Workload("ring32-s1m-h32kv8-d128-causal-striped", 1, 32, 8, 1048576, 128, 32,
             LAYOUT_STRIPED, True, "bf16", 1005, std=0.5, spike_frac=0.01,
             spike_scale=8.0),
    # profiling proxies of the 256K shape (memory-counter captures stay a few
    # GB on the device): the same heads and ranks at 64K and 128K tokens, whose
    # K and V (268 MB, 537 MB) already exceed the 126 MB L2
    Workload("ring8-s64k-h32kv8-d128-causal-striped", 1, 32, 8, 65536, 128, 8,
             LAYOUT_STRIPED, True, "bf16", 1006),
    Workload("ring8-s128k-h32kv8-d128-causal-striped", 1, 32, 8, 131072, 128, 8,
             LAYOUT_STRIPED, True, "bf16", 1007),
    # one kv head of the 256K striped workload (its four query heads): the
    # 256K workload runs one launch per kv head, each exactly this problem,
    # so one capture of this launch times eight is a 256K step (~1.5 GB on
    # the device)
    Workload("ring8-s256k-h4kv1-d128-causal-striped", 1, 4, 1, 262144, 128, 8,
             LAYOUT_STRIPED, True, "bf16", 1008),
]}


def page_example_qkv():
    """The pages' toy inputs: torch.manual_seed(0), one randn draw of shape
    (3, 32, 16) split into q, k, v; returned as [1, 1, 32, 16] fp32 on CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(0)
    x = torch.randn(3, 32, 16, generator=g, dtype=torch.float32)
    return tuple(t.reshape(1, 1, 32, 16).contiguous() for t in x)


def make_qkv(B: int, H: int, Hkv: int, S: int, d: int, *, seed: int,
             dtype: torch.dtype = torch.bfloat16, device="cpu", std: float = 1.0,
             spike_frac: float = 0.0, spike_scale: float = 8.0):
    """q [B,H,S,d], k and v [B,Hkv,S,d]: i.i.d. N(0, std^2) drawn in fp32 from
    a seeded generator on `device`, then rounded to `dtype` (round to nearest
    even).  With spike_frac > 0, a seeded Bernoulli(spike_frac) choice of
    (b, kv-head, token) key rows is multiplied by spike_scale before rounding
    (a power of two keeps the bf16 values exact multiples)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    q = torch.randn(B, H, S, d, generator=g, device=dev, dtype=torch.float32)
    k = torch.randn(B, Hkv, S, d, generator=g, device=dev, dtype=torch.float32)
    v = torch.randn(B, Hkv, S, d, generator=g, device=dev, dtype=torch.float32)
    if std != 1.0:
        q.mul_(std), k.mul_(std), v.mul_(std)
    if spike_frac > 0.0:
        pick = torch.rand(B, Hkv, S, 1, generator=g, device=dev) < spike_frac
        k = torch.where(pick, k * spike_scale, k)
    return q.to(dtype), k.to(dtype), v.to(dtype)


def workload_qkv(w: Workload, device="cpu"):
    if w.name == "ring4-s32-d16-f32-example":
        return tuple(t.to(device) for t in page_example_qkv())
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    return make_qkv(w.B, w.H, w.Hkv, w.S, w.d, seed=w.seed, dtype=dt, device=device,
                    std=w.std, spike_frac=w.spike_frac, spike_scale=w.spike_scale)


def sample_rows(B: int, H: int, S: int, n_blocks: int, n: int = 1024,
                seed: int = 7) -> torch.Tensor:
    """Seeded sample of query rows over the flattened (b, h, t) axis, drawn
    without replacement, always holding the block and stripe edges
    t in {0, 1, L-1, L, S-1} of head 0.  Returns sorted int64 row ids."""
    total = B * H * S
    L = S // n_blocks
    edges = sorted({t for t in (0, 1, L - 1, L, S - 1) if 0 <= t < S})
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    n = min(n, total)
    perm = torch.randperm(total, generator=g)[: max(0, n - len(edges))]
    # an edge that was also drawn at random appears once, so at most n rows
    return torch.unique(torch.cat([perm, torch.tensor(edges, dtype=torch.int64)]))
