"""Small problems: the fused kernel cuts every unit's ring walk into pieces.

When the work units cannot fill half the SMs, each unit's walk over its key
tiles (in ring order) is split into up to sm / units contiguous pieces,
computed by different CTAs as independent normalised partials, which a
second kernel folds together by the running-softmax merge ("Ring Attention"
page, section "Halka Dikkati Nasil Calisir": partial results of the blocks
are merged through the running max and sum).  These tests check that the
split is taken where the rule says
(the workspace holds the pieces' partials), that the result matches the fp64
oracle at the bf16 tolerances, including pieces that see no key at all
(contiguous causal ranks with short walks), and that it agrees with the
per-step ring, which never splits."""
import numpy as np
import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import inputs

from test_gpu_parity import _check, _dev

pytestmark = pytest.mark.gpu


def _expected_split(B, H, Hkv, S, N, layout, causal):
    """The split rule, restated from the host enumeration of the units."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    units = ra.schedule_units(B, H, Hkv, S, N, layout, causal)
    n = len(units)
    if n == 0 or 2 * n > sm:
        return 1
    return max(1, min(sm // n, 16, int(units[:, 5].max())))


def _align(x):
    return (x + 255) // 256 * 256


SPLIT_SHAPES = [
    # B, H, Hkv, S, d, N, layout, causal
    (1, 4, 4, 4096, 64, 2, "contiguous", False),     # the pages' context-parallel example shape
    (1, 4, 2, 1000, 128, 2, "contiguous", True),     # ragged L = 500; short walks leave empty pieces
    (1, 8, 2, 512, 128, 4, "contiguous", True),      # group 4: CTA clusters over the pieces
    (1, 8, 2, 2048, 128, 4, "striped", True),
    (2, 2, 1, 768, 64, 3, "striped", False),         # L = 256, d = 64
    (1, 2, 1, 4, 128, 4, "striped", True),           # one token per rank
    (1, 3, 1, 390, 128, 3, "contiguous", True),      # odd group: tile pairs of one head
]


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=lambda c: "B{}H{}kv{}S{}d{}N{}-{}-{}".format(*c))
def test_split_walks_match_the_oracle(shape):
    B, H, Hkv, S, d, N, layout, causal = shape
    q, k, v = _dev(*inputs.make_qkv(B, H, Hkv, S, d, seed=3 * S + N + d))
    out, lse = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=causal)
    ra.check()
    _check(out, lse, q, k, v, causal)


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=lambda c: "B{}H{}kv{}S{}d{}N{}-{}-{}".format(*c))
def test_workspace_holds_the_pieces(shape):
    """ra_workspace_bytes includes nsplit fp32 partials of out and lse exactly
    when the rule splits (and then no striped out/lse copies)."""
    B, H, Hkv, S, d, N, layout, causal = shape
    ns = _expected_split(B, H, Hkv, S, N, layout, causal)
    got = ra.workspace_bytes(B, H, Hkv, S, d, N, layout, causal, "fused")
    q_elems, kv_elems, rows = B * H * S * d, B * Hkv * S * d, B * H * S
    want = 0
    if layout == "striped":
        want += _align(q_elems * 2) + 2 * _align(kv_elems * 2)
        if ns == 1:
            want += _align(q_elems * 2) + _align(rows * 4)
    if ns > 1:
        want += _align(ns * q_elems * 4) + _align(ns * rows * 4)
    assert got == want, (ns, got, want)


def test_the_pages_example_shape_is_split():
    assert _expected_split(1, 4, 4, 4096, 2, "contiguous", False) > 1


@pytest.mark.parametrize("layout,causal", [("contiguous", True), ("striped", True), ("contiguous", False)])
def test_split_agrees_with_the_per_step_ring(layout, causal):
    B, H, Hkv, S, d, N = 1, 8, 2, 1536, 128, 3
    q, k, v = _dev(*inputs.make_qkv(B, H, Hkv, S, d, seed=91))
    a, la = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=causal)
    b, lb = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=causal, mode="per_step")
    ra.check()
    assert (a.float() - b.float()).abs().max().item() < 2e-2
    assert (la - lb).abs().max().item() < 1e-3


def test_split_is_deterministic_and_variant_independent():
    """The pieces and their combination do not depend on the kernel variant
    (one CTA or K/V-sharing clusters): bit-identical results, call after call."""
    B, H, Hkv, S, d, N = 1, 8, 2, 1024, 128, 4
    q, k, v = _dev(*inputs.make_qkv(B, H, Hkv, S, d, seed=5))
    res = []
    prev = ra.set_kernel_variant(1)
    try:
        for variant in (1, 3, 3):
            ra.set_kernel_variant(variant)
            res.append(ra.forward(q, k, v, n_blocks=N, layout="striped", causal=True))
        ra.check()
    finally:
        ra.set_kernel_variant(prev)
    for o, l in res[1:]:
        assert torch.equal(o, res[0][0]) and torch.equal(l, res[0][1])
