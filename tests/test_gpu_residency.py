"""Buffers the library refuses: every tensor an entry point reads or writes
must be device memory of the current GPU.  The attention kernels copy tiles
with TMA, and the default forward launch multicasts each key/value tile to
both CTAs of a cluster; such copies must only ever cover this GPU's own
memory.  Pinned host memory and plain malloc'ed host memory, passed as any
one of q, k, v, out or lse, get RA_ERR_INVALID_ARG and nothing is enqueued
(the library's launch counter does not move)."""
import ctypes

import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import binding as rb
from blockwise_exact_attention_ring_gb300 import inputs

pytestmark = pytest.mark.gpu

B, H, Hkv, S, d, N = 1, 4, 2, 512, 128, 2


@pytest.fixture(scope="module")
def libc():
    c = ctypes.CDLL(None)
    c.malloc.restype = ctypes.c_void_p
    c.malloc.argtypes = [ctypes.c_size_t]
    c.free.argtypes = [ctypes.c_void_p]
    return c


def _device_set():
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=5))
    out = torch.empty_like(q)
    lse = torch.empty(B, H, S, device="cuda", dtype=torch.float32)
    return [q, k, v, out, lse]


def _ptrs(ts):
    return [ctypes.c_void_p(t.data_ptr()) for t in ts]


def _calls(L, p, layout):
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (*p, B, H, Hkv, S, d, N, layout, 1)
    return {
        "ra_forward": lambda: L.ra_forward(*args, st),
        "ra_forward_noalloc": lambda: L.ra_forward_noalloc(*args, st),
    }


@pytest.mark.parametrize("which", range(5), ids=["q", "k", "v", "out", "lse"])
@pytest.mark.parametrize("host_kind", ["pinned", "malloc"])
@pytest.mark.parametrize("layout", [0, 1], ids=["contiguous", "striped"])
def test_host_buffers_are_refused_before_any_launch(libc, which, host_kind, layout):
    L = ra.lib()
    L.ra_launch_count.restype = ctypes.c_ulonglong
    ts = _device_set()
    nbytes = ts[which].numel() * ts[which].element_size()
    raw = None
    if host_kind == "pinned":
        host = torch.empty(ts[which].shape, dtype=ts[which].dtype, pin_memory=True)
        p_host = ctypes.c_void_p(host.data_ptr())
    else:
        raw = libc.malloc(nbytes + 16)
        assert raw
        p_host = ctypes.c_void_p((raw + 15) & ~15)
    try:
        p = _ptrs(ts)
        p[which] = p_host
        torch.cuda.synchronize()
        for name, call in _calls(L, p, layout).items():
            n0 = L.ra_launch_count()
            rc = call()
            assert rc == rb.RA_ERR_INVALID_ARG, (name, ra.status_string(rc))
            assert L.ra_launch_count() == n0, name
        torch.cuda.synchronize()
        ra.check()
    finally:
        if raw:
            libc.free(raw)


def test_device_buffers_still_run():
    """The same call with every buffer on the device runs (and matches the
    one-CTA launch, which needs no cluster)."""
    L = ra.lib()
    ts = _device_set()
    rc = _calls(L, _ptrs(ts), 1)["ra_forward"]()
    assert rc == rb.RA_OK
    ra.check()
    assert torch.isfinite(ts[3].float()).all() and torch.isfinite(ts[4]).all()


def test_host_buffers_refused_by_permute_merge_and_backward(libc):
    L = ra.lib()
    L.ra_launch_count.restype = ctypes.c_ulonglong
    q, k, v, out, lse = _device_set()
    host = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    n0 = L.ra_launch_count()
    P = rb._p
    assert L.ra_permute(P(q), P(host), B, H, S, d, 2, N, 0, st) == rb.RA_ERR_INVALID_ARG
    rows = B * H * S
    o_run = torch.zeros(rows, d, device="cuda")
    l_run = torch.zeros(rows, device="cuda")
    l_host = torch.zeros(rows, pin_memory=True)
    o_s = torch.zeros_like(o_run)
    assert L.ra_merge(P(o_run), P(l_run), P(o_s), P(l_host), rows, d, st) == rb.RA_ERR_INVALID_ARG
    dout = torch.randn_like(q.float()).to(q.dtype)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nb = ra.backward_workspace_bytes(B, H, Hkv, S, d, N, "contiguous", True)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    rc = L.ra_backward_ws(P(q), P(k), P(v), P(out), P(lse), P(host), P(dq), P(dk), P(dv), B, H, Hkv, S, d,
                          N, 0, 1, P(ws), nb, st)
    assert rc == rb.RA_ERR_INVALID_ARG
    assert L.ra_launch_count() == n0
    ra.check()
