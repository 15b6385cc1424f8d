"""ra_forward_noalloc: the entry point for callers that cannot allocate device
memory (a framework or server that owns the whole memory budget, or a
latency-critical loop that must not allocate).  It keeps all its scratch in a
fixed array inside the library, so this file runs last: it must pass both on
its own in a fresh process and after every other test.

Each case calls the new entry point twice in a row through the C ABI.  It
enqueues the same kernels as ra_forward, so both results must equal
ra_forward's bit for bit, under the default kernel (K/V-sharing CTA clusters)
and under the one-CTA kernel; they are also compared with the fp64 oracle at
the bf16 tolerances the parity tests use (out 2e-2, lse 1e-3 max-abs)."""
import ctypes

import numpy as np
import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import binding as rb
from blockwise_exact_attention_ring_gb300 import inputs

pytestmark = pytest.mark.gpu


def _call(fn, q, k, v, out, lse, N, layout, causal):
    B, H, S, d = q.shape
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = rb._p
    return fn(P(q), P(k), P(v), P(out), P(lse), B, H, k.shape[1], S, d, N, layout, int(causal), st)


@pytest.mark.parametrize("variant", [0, 1], ids=["clusters", "one-cta"])
@pytest.mark.parametrize("B,H,Hkv,S,d,N,layout,causal", [
    (1, 8, 2, 2048, 128, 4, 1, True),    # striped: striped copies and split-walk partials; CTA clusters
    (1, 4, 2, 1000, 128, 2, 0, True),    # contiguous, ragged block: split-walk partials only
    (2, 2, 2, 1536, 64, 3, 1, False),    # d = 64, tile pairs, non-causal striped
])
def test_noalloc_matches_ra_forward_twice(B, H, Hkv, S, d, N, layout, causal, variant):
    import oracle
    L = ra.lib()
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=S + 31 * d))
    prev = ra.set_kernel_variant(variant)
    try:
        ref_o = torch.empty_like(q)
        ref_l = torch.empty(B, H, S, device="cuda", dtype=torch.float32)
        assert _call(L.ra_forward, q, k, v, ref_o, ref_l, N, layout, causal) == rb.RA_OK
        for _ in range(2):
            out = torch.full_like(q, float("nan"))
            lse = torch.full((B, H, S), float("nan"), device="cuda", dtype=torch.float32)
            assert _call(L.ra_forward_noalloc, q, k, v, out, lse, N, layout, causal) == rb.RA_OK
            ra.check()
            assert torch.equal(out, ref_o)
            assert torch.equal(lse, ref_l)
    finally:
        ra.set_kernel_variant(prev)
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal)
    assert np.abs(out.float().cpu().numpy() - ro).max() < 2e-2
    assert np.abs(lse.cpu().numpy() - rl).max() < 1e-3


def test_noalloc_runs_a_large_contiguous_problem_without_scratch():
    """A contiguous problem large enough to fill the GPU needs no scratch at
    all (no striped copies, no split walks): it runs with the array untouched
    and equals ra_forward bit for bit."""
    B, H, Hkv, S, d, N = 1, 16, 4, 8192, 128, 4
    assert ra.workspace_bytes(B, H, Hkv, S, d, N, "contiguous", True, "fused") == 0
    L = ra.lib()
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=12))
    ref_o, ref_l = ra.forward(q, k, v, n_blocks=N, causal=True)
    out = torch.empty_like(q)
    lse = torch.empty(B, H, S, device="cuda", dtype=torch.float32)
    assert _call(L.ra_forward_noalloc, q, k, v, out, lse, N, 0, True) == rb.RA_OK
    ra.check()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = ra.lib()
    # fake, aligned, disjoint pointers: the size check fails before any launch
    Q, K, V, O, LS = (ctypes.c_void_p(0x10000000 * (i + 1)) for i in range(5))
    # striped 8 heads x 64K tokens x 128: q' alone is 128 MiB > 64 MiB
    rc = L.ra_forward_noalloc(Q, K, V, O, LS, 1, 8, 8, 65536, 128, 4, 1, 1, None)
    assert rc == rb.RA_ERR_SCRATCH_LIMIT
    assert ra.status_string(rc) == "RA_ERR_SCRATCH_LIMIT"


RAGGED = [
    # B, H, Hkv, S, d, N
    (1, 8, 2, 600, 128, 3),    # L = 200: a full tile and a 72-row tail; group 4 (CTA clusters)
    (1, 4, 2, 260, 64, 4),     # L = 65, d = 64
    (2, 8, 2, 32, 128, 4),     # L = 8, far below a tile
    (1, 4, 1, 4, 128, 4),      # L = 1: one token per rank
    (1, 3, 1, 390, 128, 3),    # odd group: tile pairs of one head, L = 130
]


@pytest.mark.parametrize("shape", RAGGED)
@pytest.mark.parametrize("layout", [0, 1], ids=["contiguous", "striped"])
def test_noalloc_writes_only_its_outputs(shape, layout):
    """Guard bands of a sentinel byte around out and lse (a memory checker is
    closed on this pool) on ragged tails, where the striped path writes its
    results back from the library's array through the inverse permutation."""
    B, H, Hkv, S, d, N = shape
    guard, sentinel = 4096, 0x5A
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=2 * S + N))
    ob, lb = B * H * S * d * 2, B * H * S * 4
    obuf = torch.full((guard + ob + guard,), sentinel, dtype=torch.uint8, device="cuda")
    lbuf = torch.full((guard + lb + guard,), sentinel, dtype=torch.uint8, device="cuda")
    out = obuf[guard:guard + ob].view(torch.bfloat16).view(B, H, S, d)
    lse = lbuf[guard:guard + lb].view(torch.float32).view(B, H, S)
    L = ra.lib()
    assert _call(L.ra_forward_noalloc, q, k, v, out, lse, N, layout, True) == rb.RA_OK
    ra.check()
    torch.cuda.synchronize()
    for buf, n in ((obuf, ob), (lbuf, lb)):
        assert bool((buf[:guard] == sentinel).all()) and bool((buf[guard + n:] == sentinel).all())
    ref_o, ref_l = ra.forward(q, k, v, n_blocks=N, layout="striped" if layout else "contiguous", causal=True)
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
