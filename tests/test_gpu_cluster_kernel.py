"""Kernel variant 3: the single-CTA tensor-core kernel launched as clusters of
two CTAs that share each key/value tile load by TMA multicast.  Every unit
runs the same instructions on the same data as in variant 1, only placed on a
CTA pair, so the two variants must agree bit for bit; and both reproduce the
fp64 oracle."""
import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import inputs

from test_gpu_parity import _check, _dev

pytestmark = pytest.mark.gpu


def _both(q, k, v, **kw):
    prev = ra.set_kernel_variant(1)
    try:
        a = ra.forward(q, k, v, **kw)
        ra.set_kernel_variant(3)
        b = ra.forward(q, k, v, **kw)
        ra.check()
    finally:
        ra.set_kernel_variant(prev)
    return a, b


CLUSTER_SHAPES = [
    # B, H, Hkv, S, d, N      (four or more query heads per kv head take clusters)
    (1, 8, 2, 1000, 128, 2),    # group 4, ragged L = 500
    (2, 8, 2, 1024, 128, 8),    # one tile per rank
    (1, 16, 2, 768, 64, 3),     # group 8, d = 64, L = 256
    (1, 8, 1, 32, 128, 4),      # L = 8, far below a tile
    (3, 8, 2, 260, 128, 4),     # odd batch, L = 65
    (1, 4, 1, 2304, 128, 1),    # one rank, 18 tiles
    (1, 4, 2, 1024, 128, 4),    # group 2: falls back to single CTAs
]


@pytest.mark.parametrize("shape", CLUSTER_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("mode", ["fused", "per_step"])
def test_cluster_kernel_matches_oracle_and_single_cta(shape, causal, layout, mode):
    B, H, Hkv, S, d, N = shape
    q, k, v = _dev(*inputs.make_qkv(B, H, Hkv, S, d, seed=13 * S + N + d))
    (a, la), (b, lb) = _both(q, k, v, n_blocks=N, layout=layout, causal=causal, mode=mode)
    assert torch.equal(a, b) and torch.equal(la, lb)
    _check(b, lb, q, k, v, causal)


def test_cluster_kernel_running_max_stress():
    q, k, v = inputs.make_qkv(1, 4, 1, 1024, 128, seed=17, spike_frac=0.05, spike_scale=16.0)
    q, k, v = _dev(q * 6, k, v)
    for layout in ("contiguous", "striped"):
        (a, la), (b, lb) = _both(q, k, v, n_blocks=4, layout=layout, causal=True)
        assert torch.equal(a, b) and torch.equal(la, lb)
        _check(b, lb, q, k, v, True)


@pytest.mark.parametrize("name", ["ring4-s32k-h32kv8-d128-causal-contiguous",
                                  "ring8-s256k-h32kv8-d128-causal-striped"])
def test_cluster_kernel_workloads(name):
    """Full-size workloads: bitwise equal to variant 1, and the oracle's
    sampled rows."""
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.workload_qkv(w, device="cuda")
    layout = "striped" if w.layout == inputs.LAYOUT_STRIPED else "contiguous"
    (a, la), (b, lb) = _both(q, k, v, n_blocks=w.n_blocks, layout=layout, causal=w.causal)
    assert torch.equal(a, b) and torch.equal(la, lb)
    rows = inputs.sample_rows(w.B, w.H, w.S, w.n_blocks).numpy()
    _check(b, lb, q, k, v, w.causal, rows=rows)


def test_cluster_kernel_block_partials():
    """One device's ring step (ra_forward_block) on clusters: the units of one
    rank still pair up, and the partials equal variant 1's bit for bit."""
    B, H, Hkv, S, d, N = 1, 8, 2, 2048, 128, 4
    q, k, v = _dev(*inputs.make_qkv(B, H, Hkv, S, d, seed=71))
    for layout in ("contiguous", "striped"):
        outs = []
        for variant in (1, 3):
            prev = ra.set_kernel_variant(variant)
            try:
                o = torch.zeros(B, H, S, d, device="cuda", dtype=torch.float32)
                l = torch.full((B, H, S), float("-inf"), device="cuda", dtype=torch.float32)
                for rank in range(N):
                    ra.forward_block(q, k, v, o, l, N, rank, (rank + 1) % N, layout=layout, causal=True)
                ra.check()
            finally:
                ra.set_kernel_variant(prev)
            outs.append((o, l))
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
