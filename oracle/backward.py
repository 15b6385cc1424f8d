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

``dkdv_rows`` gives dK and dV for selected key rows only (the large
workloads, where the full gradients do not fit a CPU check): for each key u
it sums over the query rows t that see it, with every such row's softmax
recomputed from scratch over all its visible keys.
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


def dkdv_rows(q, k, v, dout, key_rows, causal: bool = False, fault: int = 0,
              chunk_elems: int = 1 << 24) -> Tuple[np.ndarray, np.ndarray]:
    """(dk, dv) [n, d] in fp64 for selected flattened (b, g, u) key rows of
    the [B, Hkv, S, d] key/value tensors.  From the definition, per kv head g
    and each query row (h, t) of its group that sees any selected key
    (t >= u under the causal mask):

        P[t, :]   = softmax over the visible keys of c q_t . k_u'
        dP[t, u'] = dO_t . v_u'            delta_t = sum_u' P[t, u'] dP[t, u']
        dV_u     += P[t, u] dO_t           dK_u   += c P[t, u] (dP[t, u] - delta_t) q_t

    The query rows are taken in chunks of at most ``chunk_elems`` scores;
    every chunk recomputes its rows' full softmax.  The arithmetic is plain
    float64 PyTorch CPU ops (matmul, exp, sums), which use every host core.
    ``fault`` plants the same kinds of mistakes as in ``attention_backward``
    (pin tests only): 1 drops delta, 2 takes the query row at the key's
    position (u) instead of t for dK, 3 drops the scale of dK, 4 keeps only
    the first head of a GQA group, 5 hides key u from query u under the
    causal mask."""
    import torch

    def f64(x):
        return x.detach().cpu().double() if isinstance(x, torch.Tensor) else torch.from_numpy(_f64(x))

    B, H, S, d = q.shape
    Hkv = k.shape[1]
    grp = H // Hkv
    c = 1.0 / np.sqrt(d)
    key_rows = np.asarray(key_rows, dtype=np.int64).ravel()
    dk = torch.zeros(key_rows.size, d, dtype=torch.float64)
    dv = torch.zeros(key_rows.size, d, dtype=torch.float64)
    by_head = {}
    for n, r in enumerate(key_rows):
        b, g, u = int(r // (Hkv * S)), int(r // S % Hkv), int(r % S)
        by_head.setdefault((b, g), []).append((n, u))
    for (b, g), sel in by_head.items():
        idx = torch.tensor([n for n, _ in sel])
        us = torch.tensor([u for _, u in sel])
        t_lo = int(us.min()) if causal else 0
        kg, vg = f64(k[b, g]), f64(v[b, g])
        vu = vg[us]
        heads = range(grp) if fault != 4 else range(1)
        step = max(1, chunk_elems // S)
        for hh in heads:
            h = g * grp + hh
            qh, dh = f64(q[b, h]), f64(dout[b, h])
            for t0 in range(t_lo, S, step):
                t1 = min(S, t0 + step)
                nk = t1 if causal else S          # keys any row of the chunk can see
                qt, dt = qh[t0:t1], dh[t0:t1]
                s = (qt @ kg[:nk].T) * c
                if causal:
                    t = torch.arange(t0, t1)[:, None]
                    u_all = torch.arange(nk)[None, :]
                    hidden = (u_all >= t) if fault == 5 else (u_all > t)
                    if fault == 5:
                        hidden[:, 0] = False      # keep every row defined
                    s.masked_fill_(hidden, float("-inf"))
                p = torch.softmax(s, dim=1)
                dp = dt @ vg[:nk].T
                delta = 0.0 if fault == 1 else (p * dp).sum(dim=1, keepdim=True)
                vis = us < nk                     # selected keys inside the chunk's key range
                pu = torch.zeros(t1 - t0, us.numel(), dtype=torch.float64)
                pu[:, vis] = p[:, us[vis]]
                dsu = pu * (dt @ vu.T - delta)
                dv[idx] += pu.T @ dt
                if fault == 2:
                    part = dsu.sum(dim=0)[:, None] * qh[us]
                else:
                    part = dsu.T @ qt
                dk[idx] += part if fault == 3 else c * part
    return dk.numpy(), dv.numpy()
