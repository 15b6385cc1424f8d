"""fp64 CPU oracle of the backward pass of exact attention (test infrastructure).

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.

The pages train through ring attention (the "Context Parallelism" glossary
page, section "Pratik Kullanim ve Odunlesimler", calls backward on the
attention output), and the ring is exact, so its gradients are those of
exact attention.  Written out from the definition, per query head h with kv
head g = h // (H / Hkv), scale c = 1 / sqrt(d), causal keys u <= t:

    P = softmax(c Q K^T)             (rows over visible keys)
    dV_g += P^T dO                   dP = dO V^T
    delta_t = sum_u P[t,u] dP[t,u]   dS = P * (dP - delta)
    dQ = c dS K                      dK_g += c dS^T Q

Matrix products are numpy float64 matmuls; nothing is blocked or reordered.
``fault`` plants one deliberate mistake (for the pin tests only):
    1 drops delta, 2 uses dS instead of dS^T for dK (transposed operand),
    3 drops the scale of dK, 4 keeps only the first head of a GQA group in
    dK and dV, 5 masks keys u < t instead of u <= t.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np


def _f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _probs(qh: np.ndarray, kg: np.ndarray, c: float, causal: bool, fault: int) -> np.ndarray:
    """Softmax rows of c q k^T over the visible keys (fp64)."""
    s = (qh @ kg.T) * c
    if causal:
        S = s.shape[0]
        t = np.arange(S)[:, None]
        u = np.arange(S)[None, :]
        hidden = (u >= t) if fault == 5 else (u > t)
        if fault == 5:
            hidden[0, 0] = False  # keep row 0 defined
        s = np.where(hidden, -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    return p / p.sum(axis=1, keepdims=True)


def attention_backward(q, k, v, dout, causal: bool = False,
                       fault: int = 0) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(dq [B,H,S,d], dk [B,Hkv,S,d], dv [B,Hkv,S,d]) in fp64 for the loss
    sum(dout * attention(q, k, v)); inputs [B,H,S,d] / [B,Hkv,S,d] in natural
    token order (torch or numpy, any float dtype)."""
    qa, ka, va, da = (_f64(t) for t in (q, k, v, dout))
    if qa.ndim != 4 or ka.ndim != 4 or va.shape != ka.shape or da.shape != qa.shape:
        raise ValueError("expected q, dout [B,H,S,d] and k, v [B,Hkv,S,d]")
    B, H, S, d = qa.shape
    Hkv = ka.shape[1]
    if H % Hkv != 0 or ka.shape[0] != B or ka.shape[2] != S or ka.shape[3] != d:
        raise ValueError("k/v shape does not match q")
    grp = H // Hkv
    c = 1.0 / np.sqrt(d)
    dq = np.zeros_like(qa)
    dk = np.zeros_like(ka)
    dv = np.zeros_like(va)
    for b in range(B):
        for h in range(H):
            g = h // grp
            p = _probs(qa[b, h], ka[b, g], c, causal, fault)
            dp = da[b, h] @ va[b, g].T
            delta = 0.0 if fault == 1 else (p * dp).sum(axis=1, keepdims=True)
            ds = p * (dp - delta)
            dq[b, h] = c * (ds @ ka[b, g])
            if fault == 4 and h % grp != 0:
                continue
            dk_part = (ds @ qa[b, h]) if fault == 2 else (ds.T @ qa[b, h])
            dk[b, g] += dk_part if fault == 3 else c * dk_part
            dv[b, g] += p.T @ da[b, h]
    return dq, dk, dv


def dq_rows(q, k, v, dout, rows, causal: bool = False) -> np.ndarray:
    """dq for selected flattened (b, h, t) rows only: each row needs its own
    softmax row, dO row and the keys and values, O(S d) per row.  Only the
    kv heads the rows use are widened to fp64."""
    B, H, S, d = q.shape
    grp = H // k.shape[1]
    c = 1.0 / np.sqrt(d)
    rows = np.asarray(rows, dtype=np.int64).ravel()
    out = np.empty((rows.size, d))
    heads = {}
    for n, r in enumerate(rows):
        b, h, t = int(r // (H * S)), int(r // S % H), int(r % S)
        g = h // grp
        if (b, g) not in heads:
            heads[(b, g)] = (_f64(k[b, g]), _f64(v[b, g]))
        kg, vg = heads[(b, g)]
        kk = kg[:t + 1] if causal else kg
        vv = vg[:t + 1] if causal else vg
        qt, dt = _f64(q[b, h, t]), _f64(dout[b, h, t])
        s = (kk @ qt) * c
        p = np.exp(s - s.max())
        p /= p.sum()
        dp = vv @ dt
        ds = p * (dp - (p * dp).sum())
        out[n] = c * (ds @ kk)
    return out
