"""Backward pass (ra_backward) against the fp64 oracle of the gradients of
exact attention.

Tolerance: every gradient is a sum of products in which one factor (P, dS,
and out through delta) is rounded to bf16 (relative 2^-9) before an fp32
accumulation, and the result is rounded to bf16 again; with cancellation in
dS = P (dP - delta) the error is bounded relative to the tensor's largest
entry, not entrywise.  The bar is max |got - ref| <= 2e-2 max |ref| per
tensor (the bf16 output bar of the forward, scaled to the gradient's size),
and the mean error <= 2e-3 max |ref|.
"""
import numpy as np
import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import inputs
from oracle.backward import attention_backward, dkdv_rows, dq_rows

pytestmark = pytest.mark.gpu

REL_MAX, REL_MEAN = 2e-2, 2e-3


def _dout(B, H, S, d, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, H, S, d, generator=g).to(torch.bfloat16)


def _check(got, ref, what):
    got = got.float().cpu().double().numpy()
    scale = np.abs(ref).max()
    err = np.abs(got - ref)
    assert err.max() <= REL_MAX * scale, f"{what}: max err {err.max():.3g} vs scale {scale:.3g}"
    assert err.mean() <= REL_MEAN * scale, f"{what}: mean err {err.mean():.3g} vs scale {scale:.3g}"


CASES = [
    # B, H, Hkv, S, d, N, layout, causal
    (1, 2, 1, 256, 64, 2, "contiguous", True),
    (1, 4, 2, 1024, 128, 4, "striped", True),
    (1, 4, 2, 1024, 128, 4, "contiguous", True),
    (2, 2, 2, 512, 64, 1, "contiguous", False),
    (1, 2, 1, 600, 128, 3, "striped", True),      # L = 200: ragged tiles
    (1, 4, 4, 384, 128, 3, "contiguous", False),
    (1, 6, 2, 768, 64, 2, "striped", False),
    (1, 4, 4, 4096, 64, 2, "contiguous", False),  # the pages' context-parallel example shape
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}kv{}S{}d{}N{}-{}-{}".format(*c))
def test_backward_matches_oracle(case):
    B, H, Hkv, S, d, N, layout, causal = case
    q, k, v = inputs.make_qkv(B, H, Hkv, S, d, seed=S + 3 * d + N)
    dout = _dout(B, H, S, d, seed=S + 1)
    qd, kd, vd, dod = (t.cuda().contiguous() for t in (q, k, v, dout))
    out, lse = ra.forward(qd, kd, vd, n_blocks=N, layout=layout, causal=causal)
    dq, dk, dv = ra.backward(qd, kd, vd, out, lse, dod, N, layout=layout, causal=causal)
    ra.check()
    rq, rk, rv = attention_backward(q, k, v, dout, causal)
    _check(dq, rq, "dq")
    _check(dk, rk, "dk")
    _check(dv, rv, "dv")


def test_backward_independent_of_ring_size_and_layout():
    """Same tokens, any N and layout: the same gradients up to rounding."""
    B, H, Hkv, S, d = 1, 4, 2, 1536, 128
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, S, d, seed=8))
    dout = _dout(B, H, S, d, seed=9).cuda()
    base = None
    for N, layout in [(1, "contiguous"), (3, "contiguous"), (4, "striped"), (6, "striped")]:
        out, lse = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True)
        g = ra.backward(q, k, v, out, lse, dout, N, layout=layout, causal=True)
        ra.check()
        if base is None:
            base = g
            continue
        for a, b in zip(base, g):
            scale = a.float().abs().max().item()
            assert (a.float() - b.float()).abs().max().item() <= 2e-2 * scale


def test_backward_deterministic():
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 4, 2, 1024, 128, seed=4))
    dout = _dout(1, 4, 1024, 128, seed=5).cuda()
    out, lse = ra.forward(q, k, v, n_blocks=4, layout="striped", causal=True)
    a = ra.backward(q, k, v, out, lse, dout, 4, layout="striped", causal=True)
    b = ra.backward(q, k, v, out, lse, dout, 4, layout="striped", causal=True)
    ra.check()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# Key rows compared element by element with the oracle at each workload size,
# as (kv head, natural position) with S the sequence length.  Under the causal
# mask key u is seen by the queries t >= u: early keys gather gradient from
# the whole sequence (every ring step of every later block), late keys from a
# few rows only (under striping the last positions belong to every rank).
KEY_ROWS = {
    "ring4-s32k-h32kv8-d128-causal-contiguous":
        lambda S: [(0, 0), (0, 1), (0, 127), (0, 128), (0, 8191), (0, 8192),
                   (5, S - 1), (5, S - 2), (5, S - 128), (5, S - 1000)],
    "ring8-s256k-h32kv8-d128-causal-striped":
        lambda S: [(g, S - o) for g in (0, 7) for o in (1, 2, 8, 9, 100, 257, 511, 512)],
    # the other lines whose backward the bench measures: late keys only (an
    # early key's oracle would recompute hundreds of thousands of softmax rows)
    "ring8-s256k-h32kv8-d128-causal-contiguous":
        lambda S: [(g, S - o) for g in (0, 7) for o in (1, 2, 8, 9, 100, 257, 511, 512)],
    "ring32-s1m-h32kv8-d128-causal-striped":
        lambda S: [(g, S - o) for g in (0, 7) for o in (1, 2, 33, 100, 257, 512)],
}


@pytest.mark.parametrize("name", list(KEY_ROWS))
def test_backward_workload_sampled_rows(name):
    """A workload's full shape, in its own layout (32K tokens over 4
    contiguous blocks; 256K tokens over 8, striped and contiguous; 1M tokens
    over 32, striped: every line whose backward the bench measures): dq on
    sampled query rows and dk, dv on sampled key rows
    against the fp64 oracle row by row, each at the per-tensor bar
    2e-2 * max |ref| over the compared rows; and over all keys the identities
    sum_u dV = sum_t dO (per kv head) and sum_u dK = 0, which the whole dK
    and dV must satisfy."""
    w = inputs.WORKLOADS[name]
    layout = "striped" if w.layout == inputs.LAYOUT_STRIPED else "contiguous"
    q, k, v = inputs.workload_qkv(w, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(77)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    out, lse = ra.forward(q, k, v, n_blocks=w.n_blocks, layout=layout, causal=True)
    dq, dk, dv = ra.backward(q, k, v, out, lse, dout, w.n_blocks, layout=layout, causal=True)
    ra.check()
    def picked(x, rows):  # the selected rows only, gathered on the device
        idx = torch.as_tensor(np.asarray(rows), device=x.device)
        return x.reshape(-1, w.d)[idx].double().cpu().numpy()

    qc, kc, vc, dc = (t.cpu() for t in (q, k, v, dout))
    rows = inputs.sample_rows(w.B, w.H, w.S, w.n_blocks, n=48 if w.S > 65536 else 96, seed=7)
    ref = dq_rows(qc, kc, vc, dc, rows, causal=True)
    got = picked(dq, rows)
    assert np.abs(got - ref).max() <= REL_MAX * np.abs(ref).max()
    key_rows = np.array([gg * w.S + u for gg, u in KEY_ROWS[name](w.S)])  # B = 1
    ref_k, ref_v = dkdv_rows(qc, kc, vc, dc, key_rows, causal=True)
    got_k, got_v = picked(dk, key_rows), picked(dv, key_rows)
    assert np.abs(got_k - ref_k).max() <= REL_MAX * np.abs(ref_k).max()
    assert np.abs(got_v - ref_v).max() <= REL_MAX * np.abs(ref_v).max()
    del qc, kc, vc, dc
    grp = w.H // w.Hkv
    f64 = torch.float64
    dv_sum = dv.sum(dim=2, dtype=f64)
    do_sum = dout.reshape(w.B, w.Hkv, grp, w.S, w.d).sum(dim=(2, 3), dtype=f64)
    assert (dv_sum - do_sum).abs().max().item() <= 1e-2 * dout.abs().sum(dim=2, dtype=f64).max().item()
    dk_sum = dk.sum(dim=2, dtype=f64)
    assert dk_sum.abs().max().item() <= 1e-2 * dk.abs().sum(dim=2, dtype=f64).max().item()


F32_CASES = [
    # B, H, Hkv, S, d, N, layout, causal
    (1, 1, 1, 32, 16, 4, "contiguous", False),   # the pages' 4-device example shape
    (1, 2, 1, 96, 32, 3, "striped", True),
    (2, 2, 2, 64, 16, 4, "contiguous", True),
    (1, 4, 2, 128, 64, 2, "contiguous", False),
    (1, 3, 1, 90, 40, 3, "striped", False),      # d not a multiple of 32
]


@pytest.mark.parametrize("case", F32_CASES, ids=lambda c: "B{}H{}kv{}S{}d{}N{}-{}-{}".format(*c))
def test_backward_f32_exact(case):
    """The fp32 path (ra_backward_f32) against the fp64 oracle at fp32
    precision: max error <= 1e-5 of max(1, max |ref|)."""
    B, H, Hkv, S, d, N, layout, causal = case
    if (B, H, S, d) == (1, 1, 32, 16):
        q, k, v = inputs.page_example_qkv()
    else:
        q, k, v = inputs.make_qkv(B, H, Hkv, S, d, seed=S * d, dtype=torch.float32)
    g = torch.Generator().manual_seed(S + d)
    dout = torch.randn(B, H, S, d, generator=g)
    qd, kd, vd, dod = (t.cuda().contiguous() for t in (q, k, v, dout))
    out, lse = ra.forward(qd, kd, vd, n_blocks=N, layout=layout, causal=causal)
    grads = ra.backward(qd, kd, vd, out, lse, dod, N, layout=layout, causal=causal)
    ra.check()
    for name, got, ref in zip(("dq", "dk", "dv"), grads, attention_backward(q, k, v, dout, causal)):
        err = np.abs(got.cpu().double().numpy() - ref).max()
        assert err <= 1e-5 * max(1.0, np.abs(ref).max()), f"{name}: {err:.3g}"


def test_backward_rejects_bad_arguments():
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 2, 1, 256, 64, seed=1))
    out, lse = ra.forward(q, k, v, n_blocks=2, causal=True)
    dout = torch.zeros_like(q)
    L = ra.lib()
    P = lambda t: t.data_ptr()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    # dq aliasing q
    assert L.ra_backward(P(q), P(k), P(v), P(out), P(lse), P(dout), P(q), P(dk), P(dv),
                         1, 2, 1, 256, 64, 2, 0, 1, None) == 1
    # d = 32 is not a tensor-core head dimension
    assert L.ra_backward(P(q), P(k), P(v), P(out), P(lse), P(dout), P(dq), P(dk), P(dv),
                         1, 2, 1, 512, 32, 2, 0, 1, None) == 2
    ra.check()
