"""Guard bands around every output: each output buffer is the middle of a
larger allocation whose head and tail hold a sentinel pattern, and after the
call the sentinels must be intact bit for bit.  This stands in for a memory
checker (closed on this pool) on the paths with ragged tails, where an
off-by-one tile bound would write past the end: L not a multiple of 128,
blocks shorter than a tile, one token per rank; both layouts, all forward
modes, both dtypes, every forward kernel variant (K/V-sharing clusters, one
CTA), the backward and the permutation.  The no-alloc entry
point has its own guarded cases in the file that runs last."""
import ctypes

import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import binding as rb
from blockwise_exact_attention_ring_gb300 import inputs

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side (a multiple of 16, so the interior stays 16-byte aligned)
SENTINEL = 0x5A


class Guarded:
    """A CUDA byte buffer with guard bands; `t` is the interior viewed as a tensor."""

    def __init__(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        self.nbytes = n * torch.empty(0, dtype=dtype).element_size()
        self.buf = torch.full((GUARD + self.nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self):
        torch.cuda.synchronize()
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.nbytes:]
        return bool((head == SENTINEL).all()) and bool((tail == SENTINEL).all())


RAGGED = [
    # B, H, Hkv, S, d, N
    (1, 8, 2, 600, 128, 3),    # L = 200: a full tile and a 72-row tail; group 4 (CTA clusters)
    (1, 4, 2, 260, 64, 4),     # L = 65, d = 64, group 2
    (2, 8, 2, 32, 128, 4),     # L = 8, far below a tile
    (1, 4, 1, 4, 128, 4),      # L = 1: one token per rank
    (1, 3, 1, 390, 128, 3),    # odd group: tile pairs of one head, L = 130
]


# bf16 in every forward mode; the exact fp32 path has the fused mode only
MODE_DTYPE = [("fused", torch.bfloat16), ("per_step", torch.bfloat16), ("ring", torch.bfloat16),
              ("fused", torch.float32)]


@pytest.mark.parametrize("shape", RAGGED)
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("mode,dtype", MODE_DTYPE, ids=lambda x: str(x).replace("torch.", ""))
def test_forward_writes_only_its_outputs(shape, layout, mode, dtype):
    B, H, Hkv, S, d, N = shape
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=S + N, dtype=dtype))
    out = Guarded((B, H, S, d), dtype)
    lse = Guarded((B, H, S), torch.float32)
    ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True, mode=mode, out=out.t, lse=lse.t)
    ra.check()
    assert out.intact() and lse.intact()
    assert torch.isfinite(out.t.float()).all() and torch.isfinite(lse.t).all()


@pytest.mark.parametrize("variant", [0, 1, 3])
@pytest.mark.parametrize("shape", RAGGED)
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_every_forward_kernel_variant_writes_only_its_outputs(shape, layout, variant):
    B, H, Hkv, S, d, N = shape
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=S + N + 17 * variant))
    out = Guarded((B, H, S, d), torch.bfloat16)
    lse = Guarded((B, H, S), torch.float32)
    prev = ra.set_kernel_variant(variant)
    try:
        ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True, out=out.t, lse=lse.t)
        ra.check()
    finally:
        ra.set_kernel_variant(prev)
    assert out.intact() and lse.intact()
    assert torch.isfinite(out.t.float()).all() and torch.isfinite(lse.t).all()


@pytest.mark.parametrize("shape", [(1, 2, 1, 600, 128, 3),    # L = 200
                                   (1, 6, 2, 768, 64, 2),     # d = 64, group 3
                                   (1, 4, 2, 1024, 128, 4)])  # whole tiles
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_backward_writes_only_its_gradients(shape, layout):
    B, H, Hkv, S, d, N = shape
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=3 * S + N))
    out, lse = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True)
    dout = torch.randn_like(q.float()).to(q.dtype)
    dq, dk, dv = Guarded(q.shape, q.dtype), Guarded(k.shape, k.dtype), Guarded(v.shape, v.dtype)
    L = ra.lib()
    P = rb._p
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.ra_backward(P(q), P(k), P(v), P(out), P(lse), P(dout), P(dq.t), P(dk.t), P(dv.t),
                       B, H, Hkv, S, d, N, rb.LAYOUTS[layout], 1, st)
    assert rc == rb.RA_OK
    ra.check()
    assert dq.intact() and dk.intact() and dv.intact()


@pytest.mark.parametrize("N", [3, 4, 8])
def test_permute_writes_only_its_output(N):
    S = 8 * N + N  # L = 9
    x = torch.randn(2, 3, S, 64, device="cuda").to(torch.bfloat16)
    y = Guarded(x.shape, x.dtype)
    ra.permute(x, N, out=y.t)
    z = Guarded(x.shape, x.dtype)
    ra.permute(y.t, N, inverse=True, out=z.t)
    ra.check()
    assert y.intact() and z.intact()
    assert torch.equal(z.t, x)
