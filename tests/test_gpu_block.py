"""ra_forward_block, one device's work at one ring step, against the fp64
oracle restricted to that step's key block; merging a rank's partials over
the ring gives its rows of the full result."""

import numpy as np
import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-5, 1e-5), torch.bfloat16: (2e-2, 1e-3)}


def _positions(layout, S, N):
    """pos[rank, a]: natural token at local row a of rank's block."""
    order = oracle.stripe_order(S, N) if layout == "striped" else np.arange(S)
    return order.reshape(N, S // N)


def _rank_major(x, layout, N):
    return ra.permute(x, N) if layout == "striped" else x


CASES = [
    # B, H, Hkv, S, d, N, dtype
    (1, 4, 2, 1024, 128, 4, torch.bfloat16),
    (1, 2, 1, 600, 64, 3, torch.bfloat16),      # L = 200: ragged tiles
    (2, 3, 3, 96, 32, 3, torch.float32),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}kv{c[2]}S{c[3]}d{c[4]}N{c[5]}-{c[6]}")
@pytest.mark.parametrize("layout,causal", [("contiguous", True), ("striped", True), ("contiguous", False)])
def test_block_partials_and_their_merge(case, layout, causal):
    B, H, Hkv, S, d, N, dtype = case
    L = S // N
    q, k, v = inputs.make_qkv(B, H, Hkv, S, d, seed=31, dtype=dtype)
    qd, kd, vd = (_rank_major(t.cuda().contiguous(), layout, N) for t in (q, k, v))
    pos = _positions(layout, S, N)
    tol_o, tol_l = TOL[dtype]
    run = run_l = None
    for i in range(N):
        rows_nat = (np.arange(B * H)[:, None] * S + pos[i][None, :]).reshape(-1)
        for s in range(N):
            j = (i - s) % N
            out_s = torch.full((B, H, S, d), float("nan"), device="cuda")
            lse_s = torch.full((B, H, S), float("nan"), device="cuda")
            ra.forward_block(qd, kd, vd, out_s, lse_s, N, rank=i, step=s, layout=layout, causal=causal)
            ra.check()
            got_o = out_s[:, :, i * L:(i + 1) * L].reshape(-1, d).cpu().double().numpy()
            got_l = lse_s[:, :, i * L:(i + 1) * L].reshape(-1).cpu().double().numpy()
            # rows of the other ranks are not written
            others = torch.ones(S, dtype=torch.bool)
            others[i * L:(i + 1) * L] = False
            assert torch.isnan(lse_s[:, :, others.cuda()]).all()
            key_mask = np.zeros(S, np.uint8)
            key_mask[pos[j]] = 1
            ref_o, ref_l = oracle.attention(q, k, v, causal=causal, rows=rows_nat, key_mask=key_mask)
            empty = np.isneginf(ref_l)
            assert np.array_equal(np.isneginf(got_l), empty), (i, s)
            assert np.all(got_o[empty] == 0)
            if (~empty).any():
                assert np.abs(got_o[~empty] - ref_o[~empty]).max() < tol_o, (i, s)
                assert np.abs(got_l[~empty] - ref_l[~empty]).max() < tol_l, (i, s)
            # fold this step into the running result of every rank's rows
            if run is None:
                run = torch.zeros(B, H, S, d, device="cuda")
                run_l = torch.full((B, H, S), float("-inf"), device="cuda")
            part = torch.zeros(B, H, S, d, device="cuda")
            part_l = torch.full((B, H, S), float("-inf"), device="cuda")
            part[:, :, i * L:(i + 1) * L] = out_s[:, :, i * L:(i + 1) * L]
            part_l[:, :, i * L:(i + 1) * L] = lse_s[:, :, i * L:(i + 1) * L]
            ra.merge(run.view(-1, d), run_l.view(-1), part.view(-1, d), part_l.view(-1))
    ra.check()
    # the merged partials are the full attention (rows back in natural order)
    if layout == "striped":
        run = ra.permute(run, N, inverse=True)
        run_l = ra.permute(run_l, N, inverse=True)
    ref_o, ref_l = oracle.attention(q, k, v, causal=causal)
    assert np.abs(run.cpu().double().numpy() - ref_o).max() < tol_o
    assert np.abs(run_l.cpu().double().numpy() - ref_l).max() < tol_l


def test_block_rejects_bad_arguments():
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 2, 1, 256, 64, seed=1))
    out_s = torch.empty(1, 2, 256, 64, device="cuda")
    lse_s = torch.empty(1, 2, 256, device="cuda")
    for rank, step in [(-1, 0), (2, 0), (0, 2), (0, -1)]:
        with pytest.raises(ra.RaError):
            ra.forward_block(q, k, v, out_s, lse_s, 2, rank=rank, step=step)
    with pytest.raises(ra.RaError):   # d = 64 bf16 but S % N != 0
        ra.forward_block(q, k, v, out_s, lse_s, 3, rank=0, step=0)
    ra.check()


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_merge_is_step_order_invariant(layout):
    """The ring's partials merged in ring order, reversed, and in a seeded
    random order give the same attention (up to fp32 rounding of the merge),
    and each matches the oracle: the result does not depend on the order in
    which blocks arrive."""
    B, H, Hkv, S, d, N = 1, 8, 2, 1536, 128, 6
    L = S // N
    q, k, v = inputs.make_qkv(B, H, Hkv, S, d, seed=41)
    qd, kd, vd = (_rank_major(t.cuda().contiguous(), layout, N) for t in (q, k, v))
    parts = {}
    for i in range(N):
        for s in range(N):
            o = torch.zeros(B, H, S, d, device="cuda")
            l = torch.full((B, H, S), float("-inf"), device="cuda")
            ra.forward_block(qd, kd, vd, o, l, N, rank=i, step=s, layout=layout, causal=True)
            parts[(i, s)] = (o, l)
    ra.check()
    rng = np.random.default_rng(5)
    orders = [list(range(N)), list(reversed(range(N))), list(rng.permutation(N))]
    results = []
    for order in orders:
        run = torch.zeros(B, H, S, d, device="cuda")
        run_l = torch.full((B, H, S), float("-inf"), device="cuda")
        for s in order:
            part = torch.zeros_like(run)
            part_l = torch.full_like(run_l, float("-inf"))
            for i in range(N):
                o, l = parts[(i, s)]
                part[:, :, i * L:(i + 1) * L] = o[:, :, i * L:(i + 1) * L]
                part_l[:, :, i * L:(i + 1) * L] = l[:, :, i * L:(i + 1) * L]
            ra.merge(run.view(-1, d), run_l.view(-1), part.view(-1, d), part_l.view(-1))
        ra.check()
        if layout == "striped":
            run = ra.permute(run, N, inverse=True)
            run_l = ra.permute(run_l, N, inverse=True)
        results.append((run, run_l))
    ref_o, ref_l = oracle.attention(q, k, v, causal=True)
    for run, run_l in results:
        assert np.abs(run.cpu().double().numpy() - ref_o).max() < 2e-2
        assert np.abs(run_l.cpu().double().numpy() - ref_l).max() < 1e-3
    for run, run_l in results[1:]:
        assert (run - results[0][0]).abs().max().item() < 1e-5
        assert (run_l - results[0][1]).abs().max().item() < 1e-5
