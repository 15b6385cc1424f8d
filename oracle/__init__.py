"""Plain, slow, fp64 CPU oracle for blockwise exact (ring) attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package.  The CUDA library and
its Python binding never import, link or execute anything here, and this
package imports nothing from them.

Contents
--------
``attention``      the definition of exact attention, fp64, in C (ra_oracle.c);
                   see that file's header for the formula and its sources.
``merge``          the definition of combining two partial softmax results.
``stripe_order``   the striped token layout as a plain index map.
``permute``        apply that index map to the sequence axis (numpy indexing).
``shard_sequence`` / ``gather_sequence``  natural [B, Hn, S, d] <-> the
                   sequence shards of n devices [n, B, Hn, S/n, d].
``heads_of``       what each device holds after the Ulysses all-to-all: all
                   tokens of its heads, [n, B, Hn/n, S, d].
``backward.attention_backward`` / ``backward.dq_rows``  fp64 gradients of
                   exact attention (oracle/backward.py), pinned in
                   tests/test_oracle_backward.py.

Sources (web pages on ring attention):
  * "Ring Attention" glossary page (ultralytics.com/tr), section
    "Halka Dikkati Nasil Calisir": exact full attention as the target of the
    ring, the running sums of exponentiated scores and weighted values that are
    divided at the end, and striped attention, which hands every device tokens
    spread evenly along the sequence.
  * "Ring Attention" page, section on ring attention and other kinds of
    parallelism: DeepSpeed Ulysses, where an all-to-all exchange gives every
    device all tokens of a subset of the attention heads.
  * "Context Parallelism" glossary page (ultralytics.com/tr), section
    "Pratik Kullanim ve Odunlesimler": [batch, heads, sequence, dim] layout,
    sequence on dim 2, causal scaled-dot-product attention.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ra_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_ra_oracle.so")
_lib = None

F32, BF16, F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ra_oracle.c with gcc (-O2, OpenMP, no fast-math) in place."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-Wextra", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_attention_rows.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_threads.restype = None
        _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle runs on (OMP_NUM_THREADS or all cores)."""
    return int(_load().oracle_num_threads())


def set_threads(n: int) -> None:
    """Run the oracle on n threads from now on (0: all cores)."""
    _load().oracle_set_threads(int(n))


def _as_host_array(x) -> Tuple[np.ndarray, int]:
    """Return a C-contiguous host array and the oracle dtype code.

    Accepts numpy float32/float64 arrays and CPU torch tensors of dtype
    bfloat16/float32/float64.  bf16 travels as its raw 16-bit patterns, which
    the C side widens exactly.
    """
    if isinstance(x, np.ndarray):
        if x.dtype == np.float32:
            return np.ascontiguousarray(x), F32
        if x.dtype == np.float64:
            return np.ascontiguousarray(x), F64
        raise TypeError(f"unsupported numpy dtype {x.dtype}")
    import torch  # local: the oracle itself needs only numpy
    if not isinstance(x, torch.Tensor):
        raise TypeError(type(x))
    x = x.detach()
    if x.device.type != "cpu":
        raise ValueError("the oracle runs on host memory; copy the tensor to CPU first")
    x = x.contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16), BF16
    if x.dtype == torch.float32:
        return x.numpy(), F32
    if x.dtype == torch.float64:
        return x.numpy(), F64
    raise TypeError(f"unsupported torch dtype {x.dtype}")


def attention(q, k, v, causal: bool = False, rows=None, key_mask=None,
              fault: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Exact attention in fp64 for the requested query rows.

    q: [B, H, S, d]; k, v: [B, Hkv, S, d] (same dtype), natural token order.
    rows: None for every row, else int64 indices into the flattened (b, h, t)
          axis, i.e. (b*H + h)*S + t.
    key_mask: None, or a length-S array; only keys u with key_mask[u] != 0 are
          attended (the key set of one ring step).
    Returns (out, lse) as float64: out [B, H, S, d] and lse [B, H, S] when rows
    is None, else out [n_rows, d] and lse [n_rows].
    """
    qa, dt = _as_host_array(q)
    ka, dtk = _as_host_array(k)
    va, dtv = _as_host_array(v)
    if not (dt == dtk == dtv):
        raise TypeError("q, k, v must share a dtype")
    if qa.ndim != 4 or ka.ndim != 4 or va.shape != ka.shape:
        raise ValueError("expected q [B,H,S,d] and k, v [B,Hkv,S,d]")
    B, H, S, d = qa.shape
    Hkv = ka.shape[1]
    if ka.shape[0] != B or ka.shape[2] != S or ka.shape[3] != d:
        raise ValueError("k/v shape does not match q")
    full = rows is None
    if full:
        row_ids = np.arange(B * H * S, dtype=np.int64)
    else:
        row_ids = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).ravel())
    n = row_ids.size
    out = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    mask_ptr = None
    if key_mask is not None:
        km = np.ascontiguousarray(np.asarray(key_mask).astype(np.uint8).ravel())
        if km.size != S:
            raise ValueError("key_mask must have length S")
        mask_ptr = km.ctypes.data
    rc = _load().oracle_attention_rows(
        qa.ctypes.data, ka.ctypes.data, va.ctypes.data, dt,
        B, H, Hkv, S, d, int(bool(causal)), mask_ptr,
        row_ids.ctypes.data, n, out.ctypes.data, lse.ctypes.data, int(fault))
    if rc != 0:
        raise ValueError(f"oracle_attention_rows failed with code {rc}")
    if full:
        return out.reshape(B, H, S, d), lse.reshape(B, H, S)
    return out, lse


def merge(out_a, lse_a, out_b, lse_b) -> Tuple[np.ndarray, np.ndarray]:
    """Combine two softmax-normalised partial results over disjoint key sets.

    The running-softmax merge of the "Ring Attention" page (section "Halka
    Dikkati Nasil Calisir"): each side is (out = numerator / denominator,
    lse = ln denominator); the union has denominator e^lse_a + e^lse_b and
    numerator e^lse_a out_a + e^lse_b out_b.  Rows where both sides are empty
    (lse = -inf) stay empty: out 0, lse -inf.
    """
    out_a = np.asarray(out_a, dtype=np.float64)
    out_b = np.asarray(out_b, dtype=np.float64)
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    lse = np.logaddexp(lse_a, lse_b)
    empty = np.isneginf(lse)
    safe = np.where(empty, 0.0, lse)
    wa = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - safe))
    wb = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - safe))
    out = wa[..., None] * out_a + wb[..., None] * out_b
    return out, lse


def stripe_order(S: int, n_blocks: int) -> np.ndarray:
    """Natural token index held at each row of the striped (rank-major) order.

    Striped attention gives every ring rank tokens spread evenly along the
    sequence ("Ring Attention" page, section "Halka Dikkati Nasil Calisir");
    the mapping read here is token t -> rank t mod N, kept in increasing t
    within a rank, ranks stored one after another.  Row p = r*L + a of the
    striped order therefore holds token t = a*N + r, with L = S / N.
    """
    if n_blocks < 1 or S % n_blocks != 0:
        raise ValueError("S must be a multiple of n_blocks")
    L = S // n_blocks
    p = np.arange(S, dtype=np.int64)
    r, a = p // L, p % L
    return a * n_blocks + r


def permute(x: np.ndarray, n_blocks: int, inverse: bool = False, seq_dim: int = 2) -> np.ndarray:
    """Move the sequence axis of x between natural and striped order.

    Forward: dst[..., p, ...] = src[..., stripe_order[p], ...].
    Inverse: dst[..., stripe_order[p], ...] = src[..., p, ...].
    """
    x = np.asarray(x)
    order = stripe_order(x.shape[seq_dim], n_blocks)
    if not inverse:
        return np.take(x, order, axis=seq_dim)
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size, dtype=np.int64)
    return np.take(x, inv, axis=seq_dim)


def shard_sequence(x: np.ndarray, n_dev: int) -> np.ndarray:
    """Split the sequence axis (dim 2) of x [B, Hn, S, ...] into n_dev
    consecutive blocks and stack them in front: out[i] = x[:, :, iL:(i+1)L]."""
    x = np.asarray(x)
    S = x.shape[2]
    if n_dev < 1 or S % n_dev != 0:
        raise ValueError("S must be a multiple of n_dev")
    L = S // n_dev
    return np.stack([x[:, :, i * L:(i + 1) * L] for i in range(n_dev)])


def gather_sequence(shards: np.ndarray) -> np.ndarray:
    """Inverse of shard_sequence: concatenate the device blocks along the
    sequence axis."""
    shards = np.asarray(shards)
    return np.concatenate(list(shards), axis=2)


def heads_of(shards: np.ndarray) -> np.ndarray:
    """After the Ulysses all-to-all, device g holds every token of heads
    [g Hg, (g + 1) Hg), Hg = Hn / n: out[g] = full[:, g Hg:(g + 1) Hg] of the
    sequence put back together from the shards [n, B, Hn, L, ...]."""
    shards = np.asarray(shards)
    n, Hn = shards.shape[0], shards.shape[2]
    if Hn % n != 0:
        raise ValueError("the head count must be a multiple of the device count")
    full = gather_sequence(shards)
    Hg = Hn // n
    return np.stack([full[:, g * Hg:(g + 1) * Hg] for g in range(n)])


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(force="--force" in sys.argv))
