"""The Ulysses alternative on one GPU: the all-to-all relayout (bit-exact
against the oracle's definition) and the attention it feeds (against the fp64
oracle on the whole sequence)."""
import numpy as np
import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-5, 1e-5), torch.bfloat16: (2e-2, 1e-3)}


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.uint8])
@pytest.mark.parametrize("n,B,Hn,S,d", [(2, 1, 4, 256, 64), (4, 2, 8, 96, 128), (8, 1, 8, 1024, 16),
                                        (3, 1, 6, 30, 5), (1, 1, 2, 64, 32)])
def test_all_to_all_bit_exact(dtype, n, B, Hn, S, d):
    g = torch.Generator().manual_seed(S + d)
    x = torch.randint(0, 255, (B, Hn, S, d), generator=g, dtype=torch.uint8)
    x = x.to(dtype) if dtype != torch.uint8 else x
    shards = torch.from_numpy(np.ascontiguousarray(oracle.shard_sequence(x.numpy() if dtype != torch.bfloat16
                                                                         else x.float().numpy(), n)))
    shards = shards.to(dtype).cuda().contiguous()
    heads = ra.all_to_all(shards, n)
    ref = oracle.heads_of(shards.cpu().float().numpy() if dtype == torch.bfloat16 else shards.cpu().numpy())
    got = heads.cpu().float().numpy() if dtype == torch.bfloat16 else heads.cpu().numpy()
    assert np.array_equal(got, ref)
    back = ra.all_to_all(heads, n, inverse=True)
    assert torch.equal(back, shards)
    # per-row values (lse): no trailing d axis
    rows = shards[..., 0].contiguous().float()
    rh = ra.all_to_all(rows, n)
    assert np.array_equal(rh.cpu().numpy(), oracle.heads_of(rows.cpu().numpy()))
    assert torch.equal(ra.all_to_all(rh, n, inverse=True), rows)


CASES = [
    # n, B, H, Hkv, S, d, dtype
    (4, 1, 8, 4, 1024, 128, torch.bfloat16),
    (2, 2, 4, 2, 640, 64, torch.bfloat16),
    (8, 1, 32, 8, 2048, 128, torch.bfloat16),
    (3, 1, 6, 3, 96, 32, torch.float32),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"n{c[0]}B{c[1]}H{c[2]}kv{c[3]}S{c[4]}d{c[5]}-{c[6]}")
@pytest.mark.parametrize("causal", [True, False])
def test_ulysses_matches_oracle(case, causal):
    n, B, H, Hkv, S, d, dtype = case
    q, k, v = inputs.make_qkv(B, H, Hkv, S, d, seed=11 * n + S, dtype=dtype)
    sh = [torch.from_numpy(np.ascontiguousarray(oracle.shard_sequence(t.float().numpy(), n))).to(dtype)
          .cuda().contiguous() for t in (q, k, v)]
    out, lse = ra.forward_ulysses(*sh, n, causal=causal)
    ra.check()
    got_o = oracle.gather_sequence(out.cpu().double().numpy())
    got_l = oracle.gather_sequence(lse.cpu().double().numpy()[..., None])[..., 0]
    ref_o, ref_l = oracle.attention(q, k, v, causal=causal)
    tol_o, tol_l = TOL[dtype]
    assert np.abs(got_o - ref_o).max() < tol_o
    assert np.abs(got_l - ref_l).max() < tol_l
    if dtype == torch.bfloat16:
        # same tokens through the ring: the two alternatives agree
        o2, l2 = ra.forward(q.cuda(), k.cuda(), v.cuda(), n_blocks=n, layout="striped", causal=causal)
        assert np.abs(o2.float().cpu().numpy() - got_o).max() < 2 * tol_o
        assert np.abs(l2.cpu().numpy() - got_l).max() < 2 * tol_l


def test_ulysses_needs_whole_kv_heads_per_device():
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 8, 2, 256, 64, seed=3))
    sh = [t.reshape(1, *t.shape).contiguous() for t in (q, k, v)]
    # n = 4 devices but 2 kv heads
    sh4 = [torch.zeros(4, 1, t.shape[2], 64, 64, dtype=t.dtype, device="cuda") for t in sh]
    with pytest.raises(ra.RaError):
        ra.forward_ulysses(*sh4, 4, causal=True)
    ra.check()
