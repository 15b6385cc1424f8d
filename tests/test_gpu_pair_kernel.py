"""Parity of the CTA-pair tensor-core kernel (tcgen05 cta_group::2, d = 128)
with the fp64 oracle, through the C ABI, on the same cases as the single-CTA
kernel; and agreement of the two kernels with each other."""
import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import inputs

from test_gpu_parity import _check, _dev

pytestmark = pytest.mark.gpu


@pytest.fixture
def pair_kernel():
    prev = ra.set_kernel_variant(2)
    yield
    ra.set_kernel_variant(prev)


PAIR_SHAPES = [
    (1, 4, 2, 1000, 128, 2),    # GQA head pairs, ragged L = 500
    (1, 3, 1, 800, 128, 4),     # odd group: tile pairs, L = 200
    (2, 8, 2, 1024, 128, 8),    # one tile per rank
    (1, 2, 1, 32, 128, 4),      # L = 8
    (3, 6, 3, 260, 128, 4),     # odd batch, L = 65
    (1, 2, 2, 4, 128, 4),       # one token per rank
    (1, 4, 4, 2304, 128, 1),    # one rank, 18 tiles
]


@pytest.mark.parametrize("shape", PAIR_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("mode", ["fused", "per_step"])
def test_pair_kernel_small(pair_kernel, shape, causal, layout, mode):
    B, H, Hkv, S, d, N = shape
    q, k, v = _dev(*inputs.make_qkv(B, H, Hkv, S, d, seed=11 * S + N))
    out, lse = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=causal, mode=mode)
    ra.check()
    _check(out, lse, q, k, v, causal)


def test_pair_kernel_running_max_stress(pair_kernel):
    q, k, v = inputs.make_qkv(1, 2, 1, 1024, 128, seed=11, spike_frac=0.05, spike_scale=16.0)
    q, k, v = _dev(q * 2, k, v)
    for layout in ("contiguous", "striped"):
        out, lse = ra.forward(q, k, v, n_blocks=4, layout=layout, causal=True)
        _check(out, lse, q, k, v, True)
    ra.check()


@pytest.mark.parametrize("name", ["ring4-s32k-h32kv8-d128-causal-contiguous",
                                  "ring8-s256k-h32kv8-d128-causal-striped"])
def test_pair_kernel_workloads(pair_kernel, name):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.workload_qkv(w, device="cuda")
    layout = "striped" if w.layout == inputs.LAYOUT_STRIPED else "contiguous"
    out, lse = ra.forward(q, k, v, n_blocks=w.n_blocks, layout=layout, causal=w.causal)
    ra.check()
    rows = inputs.sample_rows(w.B, w.H, w.S, w.n_blocks).numpy()
    _check(out, lse, q, k, v, w.causal, rows=rows)


def test_pair_and_single_kernels_agree():
    q, k, v = _dev(*inputs.make_qkv(1, 8, 2, 4096, 128, seed=123))
    prev = ra.set_kernel_variant(1)
    try:
        a, la = ra.forward(q, k, v, n_blocks=4, layout="striped", causal=True)
        ra.set_kernel_variant(2)
        b, lb = ra.forward(q, k, v, n_blocks=4, layout="striped", causal=True)
        ra.check()
    finally:
        ra.set_kernel_variant(prev)
    assert (a.float() - b.float()).abs().max().item() < 2e-2
    assert (la - lb).abs().max().item() < 1e-3
