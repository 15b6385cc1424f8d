"""Failure detection without faulting or hanging a GPU.

On the GPU: every mbarrier wait of the tensor-core kernel is bounded; a probe
kernel runs the same bounded wait on a barrier nothing arrives at, with a
50 ms limit, and the host must read RA_ERR_TIMEOUT from ra_check() while the
context stays usable.  On the host: invalid requests are refused before any
launch (see also test_library.py)."""
import ctypes

import numpy as np
import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import binding as rb
from blockwise_exact_attention_ring_gb300 import inputs
import oracle


def test_wait_probe_rejects_out_of_range_limits():
    L = ra.lib()
    assert L.ra_wait_probe(10, None) == rb.RA_ERR_INVALID_ARG              # < 1 ms
    assert L.ra_wait_probe(20_000_000_000, None) == rb.RA_ERR_INVALID_ARG  # > 10 s


@pytest.mark.gpu
def test_bounded_wait_runs_out_and_is_reported():
    L = ra.lib()
    ra.check()                                    # start from a clean error word
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.ra_wait_probe(50_000_000, st) == rb.RA_OK
    with pytest.raises(rb.RaError) as err:
        ra.check()
    assert err.value.status == rb.RA_ERR_TIMEOUT
    ra.check()                                    # the word was cleared
    # the context is still usable: a forward afterwards is exact
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 2, 1, 512, 128, seed=77))
    out, lse = ra.forward(q, k, v, n_blocks=2, layout="striped", causal=True)
    ra.check()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True)
    assert np.abs(out.float().cpu().numpy() - ro).max() < 2e-2
    assert np.abs(lse.cpu().numpy() - rl).max() < 1e-3


@pytest.mark.gpu
def test_short_wait_limit_does_not_trip_a_healthy_run():
    """A 100 ms limit on every wait is far above any single wait of a healthy
    run, so a normal forward still completes with RA_OK."""
    L = ra.lib()
    L.ra_set_wait_timeout_ns(100_000_000)
    try:
        # group 2 runs one CTA per unit; group 4 runs CTA pairs whose waits
        # include the peer's multicast copies and stage releases; the short
        # sequences split every unit's walk into pieces (empty pieces skip
        # every wait)
        for H, Hkv, S in ((4, 2, 4096), (8, 2, 4096), (4, 2, 1024), (8, 2, 512)):
            q, k, v = (t.cuda() for t in inputs.make_qkv(1, H, Hkv, S, 128, seed=78))
            ra.forward(q, k, v, n_blocks=4, causal=True)
            ra.check()
    finally:
        L.ra_set_wait_timeout_ns(0)
