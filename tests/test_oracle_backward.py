"""Pins of the fp64 backward oracle against things other than itself: torch
autograd of the textbook formula, central finite differences, and two
identities of the softmax gradient.  The sampled-key-row oracle dkdv_rows
(used at workload sizes) is pinned against autograd directly, in chunks
smaller than a row block so that the chunking is exercised too."""
import numpy as np
import pytest
import torch

from oracle.backward import attention_backward, dkdv_rows, dq_rows


def _inputs(B, H, Hkv, S, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, S, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, S, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, S, d, generator=g, dtype=torch.float64)
    do = torch.randn(B, H, S, d, generator=g, dtype=torch.float64)
    return q, k, v, do


def _textbook_out(q, k, v, causal):
    """softmax(q k^T / sqrt(d)) v with the kv heads repeated over their group."""
    grp = q.shape[1] // k.shape[1]
    kk = k.repeat_interleave(grp, dim=1)
    vv = v.repeat_interleave(grp, dim=1)
    s = q @ kk.transpose(-1, -2) / q.shape[-1] ** 0.5
    if causal:
        S = q.shape[2]
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    return torch.softmax(s, dim=-1) @ vv


def pin_autograd(fault):
    ok = True
    for (B, H, Hkv, S, d), causal in [((1, 2, 1, 6, 4), True), ((2, 4, 2, 5, 3), False), ((1, 3, 3, 7, 8), True)]:
        q, k, v, do = _inputs(B, H, Hkv, S, d, seed=S * d + H)
        qs, ks, vs = (t.clone().requires_grad_(True) for t in (q, k, v))
        (_textbook_out(qs, ks, vs, causal) * do).sum().backward()
        dq, dk, dv = attention_backward(q, k, v, do, causal, fault=fault)
        for got, ref in ((dq, qs.grad), (dk, ks.grad), (dv, vs.grad)):
            ok &= bool(np.abs(got - ref.numpy()).max() < 1e-10)
    return ok


def pin_finite_differences(fault):
    """d/dx sum(dO * O) by central differences for a few entries of q, k, v."""
    B, H, Hkv, S, d = 1, 2, 1, 5, 3
    q, k, v, do = _inputs(B, H, Hkv, S, d, seed=99)
    grads = attention_backward(q, k, v, do, True, fault=fault)
    eps = 1e-6
    ok = True
    for which, idx in [(0, (0, 1, 3, 2)), (1, (0, 0, 1, 0)), (1, (0, 0, 4, 2)), (2, (0, 0, 2, 1)), (0, (0, 0, 4, 0))]:
        args = [q.clone(), k.clone(), v.clone()]
        args[which][idx] += eps
        up = (_textbook_out(*args, True) * do).sum().item()
        args[which][idx] -= 2 * eps
        dn = (_textbook_out(*args, True) * do).sum().item()
        fd = (up - dn) / (2 * eps)
        ok &= abs(fd - grads[which][idx]) < 1e-6
    return ok


def pin_identities(fault):
    """Rows of P sum to one and rows of dS sum to zero, so per kv head
    sum_u dV[u] = sum over the group's queries of dO, and sum_u dK[u] = 0."""
    ok = True
    for causal in (False, True):
        B, H, Hkv, S, d = 2, 4, 2, 9, 5
        q, k, v, do = _inputs(B, H, Hkv, S, d, seed=5 + causal)
        dq, dk, dv = attention_backward(q, k, v, do, causal, fault=fault)
        grp = H // Hkv
        dosum = do.numpy().reshape(B, Hkv, grp, S, d).sum(axis=(2, 3))
        ok &= bool(np.abs(dv.sum(axis=2) - dosum).max() < 1e-10)
        ok &= bool(np.abs(dk.sum(axis=2)).max() < 1e-10)
    return ok


ALL_PINS = [pin_autograd, pin_finite_differences, pin_identities]


def test_backward_pins_pass():
    for pin in ALL_PINS:
        assert pin(0), pin.__name__


@pytest.mark.parametrize("fault", [1, 2, 3, 4, 5])
def test_planted_backward_faults_are_caught(fault):
    assert not all(pin(fault) for pin in ALL_PINS), f"fault {fault} slipped through"


def pin_rows_autograd(fault):
    """dkdv_rows on chosen key rows (first, last, block edges, every kv head)
    against torch autograd of the textbook formula."""
    ok = True
    for (B, H, Hkv, S, d), causal in [((1, 2, 1, 6, 4), True), ((2, 4, 2, 5, 3), False),
                                      ((1, 4, 2, 9, 8), True), ((1, 3, 1, 11, 5), False)]:
        q, k, v, do = _inputs(B, H, Hkv, S, d, seed=7 * S + d)
        ks, vs = (t.clone().requires_grad_(True) for t in (k, v))
        (_textbook_out(q, ks, vs, causal) * do).sum().backward()
        rows = np.unique(np.array([0, 1, S // 2, S - 1, S, 2 * S - 1, B * Hkv * S - 1]) % (B * Hkv * S))
        gk, gv = dkdv_rows(q, k, v, do, rows, causal, fault=fault, chunk_elems=2 * S)
        ok &= bool(np.abs(gk - ks.grad.numpy().reshape(-1, d)[rows]).max() < 1e-10)
        ok &= bool(np.abs(gv - vs.grad.numpy().reshape(-1, d)[rows]).max() < 1e-10)
    return ok


def test_dkdv_rows_pin_passes():
    assert pin_rows_autograd(0)


@pytest.mark.parametrize("fault", [1, 2, 3, 4, 5])
def test_planted_dkdv_rows_faults_are_caught(fault):
    assert not pin_rows_autograd(fault), f"fault {fault} slipped through"


def test_dkdv_rows_match_full_oracle():
    q, k, v, do = _inputs(2, 4, 2, 37, 8, seed=11)
    for causal in (False, True):
        _, dk, dv = attention_backward(q, k, v, do, causal)
        rows = np.array([0, 3, 36, 37 + 5, 2 * 37 + 36, 3 * 37 + 17, 3 * 37 + 18])
        gk, gv = dkdv_rows(q, k, v, do, rows, causal, chunk_elems=37 * 5)
        assert np.abs(gk - dk.reshape(-1, 8)[rows]).max() < 1e-12
        assert np.abs(gv - dv.reshape(-1, 8)[rows]).max() < 1e-12


def test_dq_rows_match_full():
    q, k, v, do = _inputs(1, 4, 2, 33, 8, seed=3)
    for causal in (False, True):
        dq, _, _ = attention_backward(q, k, v, do, causal)
        rows = np.array([0, 5, 32, 33 + 7, 2 * 33 + 32, 3 * 33])
        got = dq_rows(q, k, v, do, rows, causal)
        assert np.abs(got - dq.reshape(-1, 8)[rows]).max() < 1e-12


def test_backward_rejects_bad_shapes():
    q, k, v, do = _inputs(1, 3, 2, 4, 2, seed=1)
    with pytest.raises(ValueError):
        attention_backward(q, k, v, do)
