"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Tolerances (max-abs over every compared element): fp32 path 1e-5 on out and
lse; bf16 path 2e-2 on out (bf16 output rounding plus bf16 P operands) and
1e-3 on lse.  The layout permutation is checked bit-exact."""
import itertools

import numpy as np
import pytest
import torch

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-5, 1e-5), torch.bfloat16: (2e-2, 1e-3)}


def _dev(*ts):
    return [t.cuda().contiguous() for t in ts]


def _compare(out, lse, q, k, v, causal, rows=None):
    """Max-abs differences of the GPU (out, lse) against the oracle."""
    qc, kc, vc = (t.cpu() for t in (q, k, v))
    o_ref, l_ref = oracle.attention(qc, kc, vc, causal=causal, rows=rows)
    d = q.shape[-1]
    o = out.float().cpu().reshape(-1, d).numpy().astype(np.float64)
    l = lse.cpu().reshape(-1).numpy().astype(np.float64)
    if rows is not None:
        r = np.asarray(rows)
        o, l = o[r], l[r]
    o_ref = o_ref.reshape(-1, d)
    l_ref = l_ref.reshape(-1)
    return float(np.abs(o - o_ref).max()), float(np.abs(l - l_ref).max())


def _check(out, lse, q, k, v, causal, rows=None):
    eo, el = _compare(out, lse, q, k, v, causal, rows)
    to, tl = TOL[q.dtype]
    assert eo < to and el < tl, f"max-abs out {eo:.3g} (tol {to}), lse {el:.3g} (tol {tl})"
    return eo, el


# ---------------------------------------------------------------- fp32 path

@pytest.mark.parametrize("layout,mode", list(itertools.product(["contiguous", "striped"],
                                                                ["fused", "per_step", "ring"])))
def test_page_example_fp32(layout, mode):
    """The pages' 4-device, block-8, dim-16 simulation on the seed-0 inputs."""
    q, k, v = _dev(*inputs.page_example_qkv())
    out, lse = ra.forward(q, k, v, n_blocks=4, layout=layout, causal=False, mode=mode)
    ra.check()
    _check(out, lse, q, k, v, False)


@pytest.mark.parametrize("B,H,Hkv,S,d,N", [(1, 2, 1, 96, 16, 3), (2, 3, 3, 70, 7, 5),
                                           (1, 4, 2, 300, 64, 4), (1, 2, 2, 256, 128, 1)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_fp32_small(B, H, Hkv, S, d, N, causal, layout):
    q, k, v = _dev(*inputs.make_qkv(B, H, Hkv, S, d, seed=S + d, dtype=torch.float32))
    out, lse = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=causal)
    _check(out, lse, q, k, v, causal)
    if d % 4 == 0:
        out2, lse2 = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=causal, mode="per_step")
        _check(out2, lse2, q, k, v, causal)
    ra.check()


# ---------------------------------------------------------------- bf16 tensor-core path

BF16_SHAPES = [
    # B, H, Hkv, S, d, N        (L = S / N; tiles of 128, ragged tails)
    (1, 4, 2, 1000, 128, 2),    # GQA head pairs, L = 500 = 3*128 + 116
    (1, 2, 2, 1152, 64, 3),     # no GQA: tile pairs, L = 384 (3 tiles, odd)
    (1, 3, 1, 800, 128, 4),     # odd group: tile pairs, L = 200
    (2, 8, 2, 1024, 128, 8),    # L = 128, one tile per rank
    (1, 2, 1, 32, 64, 4),       # L = 8: a block far smaller than a tile
    (1, 4, 4, 512, 64, 1),      # one rank: plain attention
    (3, 6, 3, 260, 128, 4),     # odd batch, group 2, L = 65
    (1, 2, 2, 4, 64, 4),        # L = 1: one token per rank
    (1, 1, 1, 1, 128, 1),       # a single token
]


@pytest.mark.parametrize("shape", BF16_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("mode", ["fused", "per_step", "ring"])
def test_bf16_small(shape, causal, layout, mode):
    B, H, Hkv, S, d, N = shape
    q, k, v = _dev(*inputs.make_qkv(B, H, Hkv, S, d, seed=7 * S + d + N))
    out, lse = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=causal, mode=mode)
    ra.check()
    _check(out, lse, q, k, v, causal)


@pytest.mark.parametrize("layout,causal,N", [("striped", True, 4), ("contiguous", True, 5),
                                             ("contiguous", False, 2), ("striped", True, 1)])
def test_ring_rotation_is_bitwise_per_step(layout, causal, N):
    """RA_MODE_RING reads every step's key/value blocks from the copies the
    copy stream rotated into place; the kernels and their order are those of
    the per-step mode, so the results are identical bit for bit."""
    q, k, v = _dev(*inputs.make_qkv(1, 4, 2, 640 * N, 128, seed=50 + N))
    a = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=causal, mode="per_step")
    b = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=causal, mode="ring")
    ra.check()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    _check(b[0], b[1], q, k, v, causal)


def test_bf16_result_independent_of_ring_size():
    """Invariance to N (and so to the ring order of blocks), causal striped and
    contiguous: every N reproduces the oracle, and the runs agree closely."""
    q, k, v = _dev(*inputs.make_qkv(1, 4, 2, 2048, 128, seed=99))
    outs = []
    for N, layout in itertools.product([1, 2, 4, 8, 16], ["contiguous", "striped"]):
        out, lse = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True)
        _check(out, lse, q, k, v, True)
        outs.append(out.float())
    ra.check()
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() < 2e-2


def test_bf16_deterministic():
    q, k, v = _dev(*inputs.make_qkv(1, 4, 2, 1536, 128, seed=5))
    a = ra.forward(q, k, v, n_blocks=3, layout="striped", causal=True)
    b = ra.forward(q, k, v, n_blocks=3, layout="striped", causal=True)
    ra.check()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_bf16_large_scores_stress_running_max():
    """Keys scaled so the running max jumps far beyond the lazy-rescale
    threshold, several times along a row."""
    q, k, v = inputs.make_qkv(1, 2, 1, 1024, 128, seed=11, spike_frac=0.05, spike_scale=16.0)
    q, k, v = _dev(q * 2, k, v)
    for layout in ("contiguous", "striped"):
        out, lse = ra.forward(q, k, v, n_blocks=4, layout=layout, causal=True)
        _check(out, lse, q, k, v, True)
    ra.check()


def test_bf16_huge_scores_need_the_true_row_max():
    """Scores spanning about +-600 in the log2 domain: 2^(s - m) stays
    finite only if m is at least the tile's true row maximum, so a row max
    taken from the wrong columns or rows overflows to inf / NaN here (the
    unmasked tiles take it from the tensor-memory load's own reduction)."""
    q, k, v = inputs.make_qkv(1, 2, 1, 1024, 128, seed=12, spike_frac=0.05, spike_scale=16.0)
    q, k, v = _dev(q * 6, k, v)
    for layout in ("contiguous", "striped"):
        out, lse = ra.forward(q, k, v, n_blocks=4, layout=layout, causal=True)
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        _check(out, lse, q, k, v, True)
    ra.check()


# ---------------------------------------------------------------- named workloads

def _workload(name):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.workload_qkv(w, device="cuda")
    return w, q, k, v


def test_workload_ring2_s4k_full_oracle():
    w, q, k, v = _workload("ring2-s4k-h4-d64-bf16")
    out, lse = ra.forward(q, k, v, n_blocks=w.n_blocks, layout="contiguous", causal=w.causal)
    ra.check()
    _check(out, lse, q, k, v, w.causal)


@pytest.mark.parametrize("name", ["ring4-s32k-h32kv8-d128-causal-contiguous",
                                  "ring8-s256k-h32kv8-d128-causal-contiguous",
                                  "ring8-s256k-h32kv8-d128-causal-striped",
                                  "ring32-s1m-h32kv8-d128-causal-striped"])
def test_workload_sampled_rows(name):
    w, q, k, v = _workload(name)
    layout = "striped" if w.layout == inputs.LAYOUT_STRIPED else "contiguous"
    out, lse = ra.forward(q, k, v, n_blocks=w.n_blocks, layout=layout, causal=w.causal)
    ra.check()
    rows = inputs.sample_rows(w.B, w.H, w.S, w.n_blocks).numpy()
    _check(out, lse, q, k, v, w.causal, rows=rows)


def test_workload_256k_layouts_agree():
    """Contiguous and striped runs of the same 256K causal problem agree after
    the striped output is put back in natural order."""
    w, q, k, v = _workload("ring8-s256k-h32kv8-d128-causal-striped")
    a, la = ra.forward(q, k, v, n_blocks=8, layout="contiguous", causal=True)
    b, lb = ra.forward(q, k, v, n_blocks=8, layout="striped", causal=True)
    ra.check()
    assert (a.float() - b.float()).abs().max().item() < 2e-2
    assert (la - lb).abs().max().item() < 1e-3


# ---------------------------------------------------------------- permute / merge kernels

@pytest.mark.parametrize("dtype,shape,N", [(torch.bfloat16, (1, 3, 96, 128), 4),
                                            (torch.float32, (2, 5, 60, 16), 6),
                                            (torch.float32, (1, 7, 64, 1), 8),
                                            (torch.bfloat16, (1, 1, 21, 3), 7),
                                            (torch.float32, (1, 2, 40, 64), 1)])
def test_permute_bit_exact(dtype, shape, N):
    x = torch.randn(*shape, generator=torch.Generator().manual_seed(3)).to(dtype)
    xd = x.cuda()
    y = ra.permute(xd if shape[-1] != 1 else xd[..., 0].contiguous(), N)
    ref = oracle.permute(x.float().numpy(), N)
    got = y.float().cpu().numpy()
    if shape[-1] == 1:
        ref = ref[..., 0]
    assert np.array_equal(got, ref)
    back = ra.permute(y, N, inverse=True)
    assert torch.equal(back, xd if shape[-1] != 1 else xd[..., 0])


def test_merge_of_partials_equals_union_attention():
    """merge(oracle over keys A, oracle over keys B) on the GPU equals the
    oracle over A u B; rows where one side or both sides see no key included."""
    S, d = 64, 32
    q, k, v = (t.double() for t in inputs.make_qkv(1, 2, 2, S, d, seed=21, dtype=torch.float32))
    ma = np.zeros(S, np.uint8)
    ma[:20] = 1
    mb = 1 - ma
    oa, la = oracle.attention(q, k, v, causal=True, key_mask=ma)
    ob, lb = oracle.attention(q, k, v, causal=True, key_mask=mb)
    ou, lu = oracle.attention(q, k, v, causal=True)
    # rows t < 20 see no key of B: lse_b = -inf there; add a row empty on both
    la[0, 0, 5], oa[0, 0, 5] = -np.inf, 0.0
    lb[0, 0, 5], ob[0, 0, 5] = -np.inf, 0.0
    run = torch.tensor(oa, dtype=torch.float32).cuda().reshape(-1, d).contiguous()
    run_l = torch.tensor(la, dtype=torch.float32).cuda().reshape(-1).contiguous()
    part = torch.tensor(ob, dtype=torch.float32).cuda().reshape(-1, d).contiguous()
    part_l = torch.tensor(lb, dtype=torch.float32).cuda().reshape(-1).contiguous()
    ra.merge(run, run_l, part, part_l)
    ra.check()
    got_o, got_l = run.cpu().double().numpy(), run_l.cpu().double().numpy()
    ou, lu = ou.reshape(-1, d), lu.reshape(-1)
    ou[5], lu[5] = 0.0, -np.inf
    assert np.isneginf(got_l[5]) and np.all(got_o[5] == 0)
    fin = np.isfinite(lu)
    assert np.abs(got_o - ou).max() < 1e-5
    assert np.abs(got_l[fin] - lu[fin]).max() < 1e-5
    ref_o, ref_l = oracle.merge(oa.reshape(-1, d), la.reshape(-1), ob.reshape(-1, d), lb.reshape(-1))
    assert np.abs(got_o - ref_o).max() < 1e-5


def test_check_reports_ok_after_clean_runs():
    q, k, v = _dev(*inputs.make_qkv(1, 2, 1, 256, 64, seed=1))
    ra.forward(q, k, v, n_blocks=2, causal=True)
    ra.check()   # raises on a device-side timeout


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("spikes", [False, True])
def test_bf16_d64_long_walks(layout, spikes):
    """Head dimension 64 rotates three S/P buffers between the two query
    tiles of a CTA (the S product of a tile's next key tile is issued before
    that tile's P V).  A problem large enough for many units per CTA and long
    ring walks (no split), causal, against the oracle on 1024 sampled rows;
    with spikes, 5 % of the keys scaled by 16 move the running max often."""
    B, H, Hkv, S, d, N = 1, 16, 4, 16384, 64, 4
    kw = dict(spike_frac=0.05, spike_scale=16.0) if spikes else {}
    q, k, v = _dev(*inputs.make_qkv(B, H, Hkv, S, d, seed=640 + spikes, **kw))
    assert ra.workspace_bytes(B, H, Hkv, S, d, N, "contiguous", True, "fused") == 0  # no split
    out, lse = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True)
    ra.check()
    rows = inputs.sample_rows(B, H, S, N, n=1024, seed=11).numpy()
    _check(out, lse, q, k, v, True, rows=rows)


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_per_kv_head_launches_with_batch(layout):
    """From 2^19 key/value rows the library launches the kernel once per
    (batch, kv head) on slices of q, k, v, out and lse.  B = 2 and four kv
    heads (2 x 4 x 65536 = 2^19 rows) take that path with slices that start
    in the second batch entry: sampled rows against the oracle, and the whole
    output bit for bit against the same problem computed head by head below
    the threshold (one kv head per call: B = 1, Hkv = 1, a single launch)."""
    B, H, Hkv, S, d, N = 2, 8, 4, 65536, 64, 8
    assert B * Hkv * S >= 1 << 19
    q, k, v = _dev(*inputs.make_qkv(B, H, Hkv, S, d, seed=77))
    out, lse = ra.forward(q, k, v, n_blocks=N, layout=layout, causal=True)
    ra.check()
    rows = inputs.sample_rows(B, H, S, N, n=512, seed=13).numpy()
    _check(out, lse, q, k, v, True, rows=rows)
    g = H // Hkv
    for b in range(B):
        for h in range(Hkv):
            o1, l1 = ra.forward(q[b:b + 1, h * g:(h + 1) * g].contiguous(), k[b:b + 1, h:h + 1].contiguous(),
                                v[b:b + 1, h:h + 1].contiguous(), n_blocks=N, layout=layout, causal=True)
            assert torch.equal(o1, out[b:b + 1, h * g:(h + 1) * g])
            assert torch.equal(l1, lse[b:b + 1, h * g:(h + 1) * g])
    ra.check()
