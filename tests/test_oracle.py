"""Pins for the fp64 CPU oracle: the pages' worked example, a library special
case, closed forms, brute force, the merge identity and the striped index map.
A final test plants known mistakes in the oracle and checks that some pin
catches each of them."""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from blockwise_exact_attention_ring_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    facts = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split("=", 1)
                facts[key] = val
    return facts


def _rand(shape, seed, dtype=torch.float64):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64).to(dtype)


# --------------------------------------------------------------------------
# the pages' worked example
# --------------------------------------------------------------------------

def _ring_by_blocks(q, k, v, n_dev, dtype):
    """The pages' ring, restated: every device keeps its query block, meets the
    key/value block j = (i - step) mod N at each step, accumulates the sum of
    exponentiated scaled scores and the score-weighted values, and divides the
    two at the end.  q, k, v: [S, d].  Returns ([S, d], largest score block)."""
    S, d = q.shape
    L = S // n_dev
    q, k, v = (x.to(dtype) for x in (q, k, v))
    result = torch.empty(S, d, dtype=dtype)
    biggest = (0, 0)
    for dev in range(n_dev):
        rows = slice(dev * L, (dev + 1) * L)
        weighted = torch.zeros(L, d, dtype=dtype)
        total = torch.zeros(L, 1, dtype=dtype)
        for step in range(n_dev):
            src = (dev - step) % n_dev
            cols = slice(src * L, (src + 1) * L)
            scores = q[rows] @ k[cols].transpose(0, 1) / math.sqrt(d)
            biggest = max(biggest, tuple(scores.shape))
            e = torch.exp(scores)
            weighted += e @ v[cols]
            total += e.sum(dim=1, keepdim=True)
        result[rows] = weighted / total
    return result, biggest


def test_page_example_ring_matches_full_attention():
    facts = _golden("page_example.txt")
    n_dev, block, dim = int(facts["n_devices"]), int(facts["block"]), int(facts["dim"])
    q, k, v = (x[0, 0] for x in inputs.page_example_qkv())
    assert q.shape == (n_dev * block, dim)

    ring32, biggest = _ring_by_blocks(q, k, v, n_dev, torch.float32)
    full32 = torch.softmax(q @ k.T / math.sqrt(dim), dim=-1) @ v
    atol = float(facts["allclose_atol"])
    same = torch.allclose(ring32, full32, atol=atol)
    assert str(same) == facts["matches_full_attention"]
    assert f"{biggest[0]}x{biggest[1]}" == facts["score_block_per_device"]
    assert f"{q.shape[0]}x{k.shape[0]}" == facts["full_score_matrix"]

    out, lse = oracle.attention(*inputs.page_example_qkv(), causal=False)
    ring64, _ = _ring_by_blocks(q, k, v, n_dev, torch.float64)
    assert np.abs(out[0, 0] - ring64.numpy()).max() < 1e-12
    assert np.abs(out[0, 0] - ring32.double().numpy()).max() < atol
    assert np.abs(out[0, 0] - full32.double().numpy()).max() < atol
    # lse against the log-sum-exp of the full scaled score matrix
    s64 = (q.double() @ k.double().T) / math.sqrt(dim)
    assert np.abs(lse[0, 0] - torch.logsumexp(s64, dim=-1).numpy()).max() < 1e-12


# --------------------------------------------------------------------------
# pin helpers (each returns True when the oracle passes the pin); the planted
# fault test reuses them
# --------------------------------------------------------------------------

def _pin_sdpa(causal, fault=0, B=2, H=4, Hkv=2, S=37, d=8, seed=11):
    q = _rand((B, H, S, d), seed)
    k = _rand((B, Hkv, S, d), seed + 1)
    v = _rand((B, Hkv, S, d), seed + 2)
    out, lse = oracle.attention(q, k, v, causal=causal, fault=fault)
    ke = k.repeat_interleave(H // Hkv, dim=1)
    ve = v.repeat_interleave(H // Hkv, dim=1)
    ref = F.scaled_dot_product_attention(q, ke, ve, is_causal=causal)
    s = q @ ke.transpose(-1, -2) / math.sqrt(d)
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    ref_lse = torch.logsumexp(s, dim=-1)
    return (np.abs(out - ref.numpy()).max() < 1e-12
            and np.abs(lse - ref_lse.numpy()).max() < 1e-12)


def _pin_zero_queries(causal, fault=0, S=23, d=4):
    q = torch.zeros(1, 2, S, d, dtype=torch.float64)
    k = _rand((1, 1, S, d), 3)
    v = _rand((1, 1, S, d), 4)
    out, lse = oracle.attention(q, k, v, causal=causal, fault=fault)
    ok = True
    for t in range(S):
        n = t + 1 if causal else S
        ok &= np.abs(out[0, :, t] - v[0, 0, :n].mean(dim=0).numpy()).max() < 1e-13
        ok &= np.abs(lse[0, :, t] - math.log(n)).max() < 1e-13
    return bool(ok)


def _pin_constant_values(causal, fault=0, S=19, d=5):
    q = _rand((1, 3, S, d), 5)
    k = _rand((1, 3, S, d), 6)
    v = torch.full((1, 3, S, d), 0.375, dtype=torch.float64)
    out, _ = oracle.attention(q, k, v, causal=causal, fault=fault)
    return bool(np.abs(out - 0.375).max() < 1e-14)


def _pin_causal_first_row(fault=0, S=17, d=6):
    q = _rand((1, 2, S, d), 7)
    k = _rand((1, 2, S, d), 8)
    v = _rand((1, 2, S, d), 9)
    out, lse = oracle.attention(q, k, v, causal=True, fault=fault)
    s00 = (q[0, :, 0] * k[0, :, 0]).sum(-1) / math.sqrt(d)
    return bool(np.abs(out[0, :, 0] - v[0, :, 0].numpy()).max() < 1e-14
                and np.abs(lse[0, :, 0] - s00.numpy()).max() < 1e-13)


def _pin_identical_keys(causal, fault=0, S=21, d=4):
    q = _rand((1, 1, S, d), 10)
    k = _rand((1, 1, 1, d), 12).expand(1, 1, S, d).contiguous()
    v = _rand((1, 1, S, d), 13)
    out, lse = oracle.attention(q, k, v, causal=causal, fault=fault)
    ok = True
    for t in range(S):
        n = t + 1 if causal else S
        s = float((q[0, 0, t] * k[0, 0, 0]).sum()) / math.sqrt(d)
        ok &= np.abs(out[0, 0, t] - v[0, 0, :n].mean(dim=0).numpy()).max() < 1e-13
        ok &= abs(lse[0, 0, t] - (s + math.log(n))) < 1e-12
    return bool(ok)


def _brute_force(q, k, v, causal):
    """Triple loop over python floats: the definition with nothing factored."""
    B, H, S, d = q.shape
    Hkv = k.shape[1]
    out = np.zeros((B, H, S, d))
    lse = np.zeros((B, H, S))
    for b in range(B):
        for h in range(H):
            g = h // (H // Hkv)
            for t in range(S):
                keys = range(t + 1) if causal else range(S)
                scores = [sum(float(q[b, h, t, c]) * float(k[b, g, u, c]) for c in range(d))
                          / math.sqrt(d) for u in keys]
                top = max(scores)
                w = [math.exp(s - top) for s in scores]
                den = math.fsum(w)
                for c in range(d):
                    out[b, h, t, c] = math.fsum(wi * float(v[b, g, u, c])
                                                for wi, u in zip(w, keys)) / den
                lse[b, h, t] = top + math.log(den)
    return out, lse


def _pin_brute_force(causal, fault=0, B=1, H=4, Hkv=2, S=9, d=3, seed=21):
    q = _rand((B, H, S, d), seed)
    k = _rand((B, Hkv, S, d), seed + 1)
    v = _rand((B, Hkv, S, d), seed + 2)
    out, lse = oracle.attention(q, k, v, causal=causal, fault=fault)
    ro, rl = _brute_force(q, k, v, causal)
    return bool(np.abs(out - ro).max() < 1e-12 and np.abs(lse - rl).max() < 1e-12)


def _pin_merge_identity(causal, n_blocks=4, fault=0, S=24, d=4):
    """Attention over the union of disjoint key sets equals the running-softmax
    merge of attention over each set (the pages' ring merge)."""
    q = _rand((1, 2, S, d), 30)
    k = _rand((1, 2, S, d), 31)
    v = _rand((1, 2, S, d), 32)
    full_o, full_l = oracle.attention(q, k, v, causal=causal, fault=fault)
    L = S // n_blocks
    acc_o = np.zeros_like(full_o)
    acc_l = np.full(full_l.shape, -np.inf)
    for j in range(n_blocks):
        mask = np.zeros(S, dtype=np.uint8)
        mask[j * L:(j + 1) * L] = 1
        o, l = oracle.attention(q, k, v, causal=causal, key_mask=mask, fault=fault)
        acc_o, acc_l = oracle.merge(acc_o, acc_l, o, l)
    with np.errstate(invalid="ignore"):
        return bool(np.abs(acc_o - full_o).max() < 1e-12
                    and np.abs(acc_l - full_l).max() < 1e-12)


ALL_PINS = [
    lambda f: _pin_sdpa(False, f), lambda f: _pin_sdpa(True, f),
    lambda f: _pin_zero_queries(False, f), lambda f: _pin_zero_queries(True, f),
    lambda f: _pin_constant_values(True, f), lambda f: _pin_causal_first_row(f),
    lambda f: _pin_identical_keys(True, f), lambda f: _pin_brute_force(False, f),
    lambda f: _pin_brute_force(True, f), lambda f: _pin_merge_identity(True, 4, f),
]


@pytest.mark.parametrize("causal", [False, True])
def test_oracle_matches_sdpa_float64(causal):
    assert _pin_sdpa(causal)
    assert _pin_sdpa(causal, B=1, H=3, Hkv=3, S=50, d=16, seed=99)   # no GQA
    assert _pin_sdpa(causal, B=1, H=8, Hkv=1, S=7, d=2, seed=5)      # one kv head


@pytest.mark.parametrize("causal", [False, True])
def test_closed_forms(causal):
    assert _pin_zero_queries(causal)
    assert _pin_constant_values(causal)
    assert _pin_identical_keys(causal)


def test_causal_first_row_is_its_own_value():
    assert _pin_causal_first_row()


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(causal):
    assert _pin_brute_force(causal)
    assert _pin_brute_force(causal, B=2, H=2, Hkv=1, S=5, d=2, seed=44)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n_blocks", [1, 2, 3, 4])
def test_merge_of_ring_steps_is_full_attention(causal, n_blocks):
    assert _pin_merge_identity(causal, n_blocks=n_blocks, S=24)


def test_merge_empty_rows_stay_empty():
    o = np.ones((3, 2))
    l = np.array([-np.inf, 0.5, -np.inf])
    z = np.zeros((3, 2))
    zl = np.array([-np.inf, -np.inf, -np.inf])
    mo, ml = oracle.merge(z, zl, o * np.array([[0], [1], [0]]), l)
    assert np.isneginf(ml[0]) and np.isneginf(ml[2]) and ml[1] == 0.5
    assert np.all(mo[0] == 0) and np.all(mo[2] == 0) and np.all(mo[1] == 1)
    # equal lse on both sides: equal weights
    mo, ml = oracle.merge(np.full((1, 2), 2.0), np.array([1.0]), np.full((1, 2), 4.0), np.array([1.0]))
    assert abs(ml[0] - (1.0 + math.log(2.0))) < 1e-15 and np.allclose(mo, 3.0, atol=0, rtol=1e-15)


def test_empty_key_set_row():
    q = _rand((1, 1, 8, 4), 1)
    k = _rand((1, 1, 8, 4), 2)
    v = _rand((1, 1, 8, 4), 3)
    mask = np.zeros(8, dtype=np.uint8)
    mask[5:] = 1
    out, lse = oracle.attention(q, k, v, causal=True, key_mask=mask)
    assert np.all(np.isneginf(lse[0, 0, :5])) and np.all(out[0, 0, :5] == 0)
    assert np.all(np.isfinite(lse[0, 0, 5:]))


def test_bf16_inputs_are_widened_exactly():
    q, k, v = inputs.make_qkv(1, 4, 2, 40, 8, seed=3, dtype=torch.bfloat16)
    o16, l16 = oracle.attention(q, k, v, causal=True)
    o64, l64 = oracle.attention(q.double(), k.double(), v.double(), causal=True)
    assert np.array_equal(o16, o64) and np.array_equal(l16, l64)
    o32, l32 = oracle.attention(q.float(), k.float(), v.float(), causal=True)
    assert np.array_equal(o32, o64) and np.array_equal(l32, l64)


def test_row_subset_matches_full():
    q, k, v = inputs.make_qkv(2, 4, 2, 33, 8, seed=4, dtype=torch.float32)
    full_o, full_l = oracle.attention(q, k, v, causal=True)
    rows = np.array([0, 5, 32, 33, 100, 2 * 4 * 33 - 1], dtype=np.int64)
    o, l = oracle.attention(q, k, v, causal=True, rows=rows)
    assert np.array_equal(o, full_o.reshape(-1, 8)[rows])
    assert np.array_equal(l, full_l.reshape(-1)[rows])


@pytest.mark.parametrize("S,N", [(32, 4), (12, 3), (8, 8), (10, 1), (64, 16)])
def test_stripe_order_definition(S, N):
    order = oracle.stripe_order(S, N)
    L = S // N
    # brute force: list rank 0's tokens, then rank 1's, ... each in increasing t
    expect = [t for r in range(N) for t in range(S) if t % N == r]
    assert order.tolist() == expect
    assert sorted(order.tolist()) == list(range(S))
    x = np.arange(2 * 3 * S * 2).reshape(2, 3, S, 2)
    y = oracle.permute(x, N)
    if N > 1:
        # row L of the striped order is rank 1's first token, t = 1
        assert np.array_equal(y[:, :, L], x[:, :, 1])
        with pytest.raises(ValueError):
            oracle.stripe_order(S + 1, N)
    else:
        assert np.array_equal(y, x)
        with pytest.raises(ValueError):
            oracle.stripe_order(S, 0)
    assert np.array_equal(oracle.permute(y, N, inverse=True), x)


@pytest.mark.parametrize("B,Hn,S,n", [(1, 4, 8, 2), (2, 6, 12, 3), (1, 8, 16, 8), (2, 2, 6, 1)])
def test_ulysses_relayout_definition(B, Hn, S, n):
    """Brute force over every element: after the all-to-all, device g's local
    head h' at token t is head g Hg + h' of the device that held token t
    (device t // L, local row t % L)."""
    L, Hg = S // n, Hn // n
    x = np.arange(B * Hn * S * 3).reshape(B, Hn, S, 3)
    shards = oracle.shard_sequence(x, n)
    assert shards.shape == (n, B, Hn, L, 3)
    heads = oracle.heads_of(shards)
    assert heads.shape == (n, B, Hg, S, 3)
    for g in range(n):
        for b in range(B):
            for hl in range(Hg):
                for t in range(S):
                    assert np.array_equal(heads[g, b, hl, t], shards[t // L, b, g * Hg + hl, t % L])
    assert np.array_equal(oracle.gather_sequence(shards), x)
    # every element moved exactly once
    assert sorted(heads.reshape(-1).tolist()) == list(range(x.size))
    with pytest.raises(ValueError):
        oracle.shard_sequence(x, S + 1)


def test_oracle_rejects_bad_arguments():
    q = torch.zeros(1, 3, 4, 2, dtype=torch.float64)
    k = torch.zeros(1, 2, 4, 2, dtype=torch.float64)
    with pytest.raises(ValueError):
        oracle.attention(q, k, k)            # H % Hkv != 0
    with pytest.raises(ValueError):
        oracle.attention(q, q, q, rows=[12])  # row out of range
    with pytest.raises(TypeError):
        oracle.attention(q.float(), q, q)     # mixed dtypes


def test_every_pin_passes():
    assert all(pin(0) for pin in ALL_PINS)


@pytest.mark.parametrize("fault", [1, 2, 3, 4, 5, 6])
def test_planted_oracle_faults_are_caught(fault):
    """Each deliberate mistake planted in the oracle fails at least one pin."""
    results = [pin(fault) for pin in ALL_PINS]
    assert not all(results), f"fault {fault} slipped through every pin"
