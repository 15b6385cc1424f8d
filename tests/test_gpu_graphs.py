"""The library's calls are stream-ordered and allocation-free with a caller
workspace, so they can be captured into a CUDA graph and replayed: the replay
gives the same bits as the eager calls (fused, per-step and ring forward,
with the ring's second stream forked and joined inside the capture; the
backward)."""
import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["fused", "per_step", "ring"])
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_forward_graph_replay_is_bitwise(mode, layout):
    B, H, Hkv, S, d, N = 1, 4, 2, 2048, 128, 4
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=91))
    nb = ra.workspace_bytes(B, H, Hkv, S, d, N, layout, True, mode, q.dtype)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    out, lse = torch.empty_like(q), torch.empty(B, H, S, device="cuda")
    ref = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True, mode=mode)
    ra.check()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm the path on a side stream, as capture requires
        ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True, mode=mode, out=out, lse=lse, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True, mode=mode, out=out, lse=lse, workspace=ws)
    out.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    ra.check()
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])
    # new inputs in the same buffers flow through the replay
    q.copy_(torch.flip(q, dims=[2]))
    ref2 = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True, mode=mode)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref2[0]) and torch.equal(lse, ref2[1])


def test_backward_graph_replay_is_bitwise():
    B, H, Hkv, S, d, N = 1, 4, 2, 1024, 128, 4
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=92))
    dout = torch.randn_like(q)
    out, lse = ra.forward(q, k, v, n_blocks=N, layout="striped", causal=True)
    ref = ra.backward(q, k, v, out, lse, dout, N, layout="striped", causal=True)
    nb = ra.backward_workspace_bytes(B, H, Hkv, S, d, N, "striped", True)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    L = ra.lib()
    P = lambda t: t.data_ptr()

    def call(stream):
        st = L.ra_backward_ws(P(q), P(k), P(v), P(out), P(lse), P(dout), P(dq), P(dk), P(dv), B, H, Hkv, S, d, N,
                              1, 1, P(ws), ws.numel(), stream.cuda_stream)
        assert st == 0

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    call(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        call(torch.cuda.current_stream())
    for t in (dq, dk, dv):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    ra.check()
    assert torch.equal(dq, ref[0]) and torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
