"""ra_forward_noalloc: the entry point for callers that cannot allocate device
memory (a framework or server that owns the whole memory budget, or a
latency-critical loop that must not allocate).  It keeps all its scratch in a
fixed array inside the library, so this file runs last: it must pass both on
its own in a fresh process and after every other test.

Each case calls the new entry point twice in a row through the C ABI and
compares both results with ra_forward's, at the bf16 tolerances the parity
tests use (out 2e-2, lse 1e-3 max-abs)."""
import ctypes

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


@pytest.mark.parametrize("B,H,Hkv,S,d,N,layout,causal", [
    (1, 4, 2, 2048, 128, 4, 1, True),    # striped: work list + striped copies in the array
    (1, 4, 2, 1000, 128, 2, 0, True),    # contiguous, ragged block: work list only
    (2, 2, 2, 1536, 64, 3, 1, False),    # d = 64, tile pairs, non-causal striped
])
def test_noalloc_matches_ra_forward_twice(B, H, Hkv, S, d, N, layout, causal):
    L = ra.lib()
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=S + 31 * d))
    ref_o = torch.empty_like(q)
    ref_l = torch.empty(B, H, S, device="cuda", dtype=torch.float32)
    assert _call(L.ra_forward, q, k, v, ref_o, ref_l, N, layout, causal) == rb.RA_OK
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, S), float("nan"), device="cuda", dtype=torch.float32)
        assert _call(L.ra_forward_noalloc, q, k, v, out, lse, N, layout, causal) == rb.RA_OK
        ra.check()
        assert (out.float() - ref_o.float()).abs().max().item() < 2e-2
        assert (lse - ref_l).abs().max().item() < 1e-3


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = ra.lib()
    # fake, aligned, disjoint pointers: the size check fails before any launch
    Q, K, V, O, LS = (ctypes.c_void_p(0x10000000 * (i + 1)) for i in range(5))
    # striped 8 heads x 64K tokens x 128: q' alone is 128 MiB > 64 MiB
    rc = L.ra_forward_noalloc(Q, K, V, O, LS, 1, 8, 8, 65536, 128, 4, 1, 1, None)
    assert rc == rb.RA_ERR_SCRATCH_LIMIT
    assert ra.status_string(rc) == "RA_ERR_SCRATCH_LIMIT"
