"""ctypes binding of libra.so: argument marshalling only.

Every computation runs in the library's CUDA kernels; this module converts
torch tensors to device pointers and streams, allocates outputs with torch's
caching allocator, and turns status codes into exceptions.  If libra.so has
not been built, the first call raises: there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libra.so")
HEADER = os.path.join(HERE, "..", "include", "ra.h")

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA = 0, 1, 2, 3
RA_ERR_NO_MEMORY, RA_ERR_TIMEOUT, RA_ERR_WORKSPACE, RA_ERR_SCRATCH_LIMIT = 4, 5, 6, 7
LAYOUTS = {"contiguous": 0, "striped": 1}
MODES = {"fused": 0, "per_step": 1, "ring": 2}
DTYPES = {torch.bfloat16: 0, torch.float32: 1}

_lib = None


class RaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: {status_string(status)} ({status})")


def _p(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def lib():
    """Load libra.so once; raise if it is missing (build it first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with blockwise_exact_attention_ring_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, ll, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
    L.ra_forward.argtypes = [vp] * 5 + [i] * 8 + [vp]
    L.ra_forward_f32.argtypes = [vp] * 5 + [i] * 8 + [vp]
    L.ra_forward_noalloc.argtypes = [vp] * 5 + [i] * 8 + [vp]
    L.ra_workspace_bytes.argtypes = [i] * 10
    L.ra_workspace_bytes.restype = sz
    L.ra_forward_ws.argtypes = [vp] * 5 + [i] * 10 + [vp, sz, vp]
    L.ra_forward_rank_major.argtypes = [vp] * 5 + [i] * 10 + [vp, sz, vp]
    L.ra_forward_block.argtypes = [vp] * 5 + [i] * 11 + [vp]
    L.ra_all_to_all.argtypes = [vp, vp] + [i] * 7 + [vp]
    L.ra_backward.argtypes = [vp] * 9 + [i] * 8 + [vp]
    L.ra_backward_ws.argtypes = [vp] * 9 + [i] * 8 + [vp, sz, vp]
    L.ra_backward_f32.argtypes = [vp] * 9 + [i] * 8 + [vp]
    L.ra_backward_workspace_bytes.argtypes = [i] * 8
    L.ra_backward_workspace_bytes.restype = sz
    L.ra_backward_tile_pairs.argtypes = [i] * 8 + [vp, ll]
    L.ra_backward_tile_pairs.restype = ll
    L.ra_ulysses_workspace_bytes.argtypes = [i] * 8
    L.ra_ulysses_workspace_bytes.restype = sz
    L.ra_forward_ulysses.argtypes = [vp] * 5 + [i] * 8 + [vp, sz, vp]
    L.ra_permute.argtypes = [vp, vp] + [i] * 7 + [vp]
    L.ra_merge.argtypes = [vp] * 4 + [ll, i, vp]
    L.ra_check.argtypes = [vp]
    L.ra_status_string.argtypes = [i]
    L.ra_status_string.restype = ctypes.c_char_p
    L.ra_version.restype = ctypes.c_char_p
    L.ra_set_kernel_variant.argtypes = [i]
    L.ra_set_kernel_variant.restype = i
    L.ra_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
    L.ra_set_wait_timeout_ns.restype = None
    L.ra_wait_probe.argtypes = [ctypes.c_ulonglong, vp]
    L.ra_wait_probe.restype = i
    L.ra_launch_count.restype = ctypes.c_ulonglong
    L.ra_schedule_units.argtypes = [i] * 9 + [vp, ll]
    L.ra_schedule_units.restype = ll
    L.ra_schedule_block_units.argtypes = [i] * 9 + [vp, ll]
    L.ra_schedule_block_units.restype = ll
    L.ra_schedule_stats.argtypes = [i, i, i, i, vp, vp]
    L.ra_schedule_stats.restype = ll
    for fn in ("ra_forward", "ra_forward_f32", "ra_forward_noalloc", "ra_forward_ws",
               "ra_forward_rank_major", "ra_forward_block", "ra_all_to_all", "ra_forward_ulysses",
               "ra_backward", "ra_backward_ws", "ra_backward_f32", "ra_permute", "ra_merge", "ra_check"):
        getattr(L, fn).restype = i
    _lib = L
    return L


def header_functions():
    """Names of the functions include/ra.h declares."""
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z0-9_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return lib().ra_status_string(int(status)).decode()


def version() -> str:
    return lib().ra_version().decode()


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int, what: str):
    if status != RA_OK:
        raise RaError(status, what)


def _dims(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,H,S,d] and k, v [B,Hkv,S,d]")
    B, H, S, d = q.shape
    if k.shape[0] != B or k.shape[2] != S or k.shape[3] != d:
        raise ValueError("k/v shape does not match q")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
        if t.dtype != q.dtype:
            raise ValueError("q, k, v must share a dtype")
    if q.dtype not in DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    return B, H, k.shape[1], S, d


def workspace_bytes(B, H, Hkv, S, d, n_blocks, layout="contiguous", causal=False,
                    mode="fused", dtype=torch.bfloat16) -> int:
    return int(lib().ra_workspace_bytes(B, H, Hkv, S, d, n_blocks, LAYOUTS[layout], int(causal),
                                        MODES[mode], DTYPES[dtype]))


def forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_blocks: int,
            layout: str = "contiguous", causal: bool = False, mode: str = "fused",
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None, stream=None
            ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Ring-ordered blockwise exact attention: returns (out, lse).

    q [B,H,S,d], k/v [B,Hkv,S,d] bf16 or fp32 CUDA tensors in natural token
    order; out has q's dtype, lse is fp32 [B,H,S].  With mode="fused" and no
    workspace the library allocates its scratch stream-ordered (ra_forward /
    ra_forward_f32); otherwise ra_forward_ws runs on `workspace` (a uint8 CUDA
    tensor, allocated here when None)."""
    B, H, Hkv, S, d = _dims(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, S, device=q.device, dtype=torch.float32)
    st = _stream(stream)
    lay, cz = LAYOUTS[layout], int(bool(causal))
    L = lib()
    if mode == "fused" and workspace is None:
        fn = L.ra_forward if q.dtype == torch.bfloat16 else L.ra_forward_f32
        _check(fn(_p(q), _p(k), _p(v), _p(out), _p(lse), B, H, Hkv, S, d, n_blocks, lay, cz, st),
               fn.__name__)
        return out, lse
    nbytes = workspace_bytes(B, H, Hkv, S, d, n_blocks, layout, causal, mode, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(L.ra_forward_ws(_p(q), _p(k), _p(v), _p(out), _p(lse), B, H, Hkv, S, d, n_blocks, lay,
                           cz, DTYPES[q.dtype], MODES[mode], _p(workspace),
                           workspace.numel() * workspace.element_size(), st), "ra_forward_ws")
    return out, lse


def permute(x: torch.Tensor, n_blocks: int, inverse: bool = False,
            out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Natural <-> striped order along dim 2 of a [B, Hn, S, d] CUDA tensor
    (or dim 2 of [B, Hn, S] for per-row values such as lse)."""
    if not x.is_cuda or not x.is_contiguous() or x.dim() not in (3, 4):
        raise ValueError("x must be a contiguous CUDA tensor [B, Hn, S, d] or [B, Hn, S]")
    B, Hn, S = x.shape[:3]
    d = x.shape[3] if x.dim() == 4 else 1
    if out is None:
        out = torch.empty_like(x)
    _check(lib().ra_permute(_p(x), _p(out), B, Hn, S, d, x.element_size(), n_blocks,
                            int(bool(inverse)), _stream(stream)), "ra_permute")
    return out


def merge(out_run: torch.Tensor, lse_run: torch.Tensor, out_s: torch.Tensor,
          lse_s: torch.Tensor, stream=None) -> None:
    """In place: fold (out_s, lse_s) into (out_run, lse_run); fp32 [rows, d]."""
    d = out_run.shape[-1]
    rows = out_run.numel() // d
    for t in (out_run, lse_run, out_s, lse_s):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32:
            raise ValueError("merge takes contiguous fp32 CUDA tensors")
    _check(lib().ra_merge(_p(out_run), _p(lse_run), _p(out_s), _p(lse_s), rows, d,
                          _stream(stream)), "ra_merge")


def check(stream=None) -> None:
    """Synchronise the stream and raise if a device-side wait ran out."""
    _check(lib().ra_check(_stream(stream)), "ra_check")


def schedule_stats(layout: str, causal: bool, n_blocks: int, L: int):
    """(total visible pairs, pairs[i, s], tiles[i, s]) from the host scheduler."""
    pairs = np.zeros((n_blocks, n_blocks), dtype=np.int64)
    tiles = np.zeros((n_blocks, n_blocks), dtype=np.int64)
    total = lib().ra_schedule_stats(LAYOUTS[layout], int(bool(causal)), n_blocks, L,
                                    pairs.ctypes.data, tiles.ctypes.data)
    if total < 0:
        raise ValueError("invalid schedule request")
    return int(total), pairs, tiles


def schedule_units(B, H, Hkv, S, n_blocks, layout="contiguous", causal=False, steps=None):
    """Work units of the tensor-core kernel in dealing order: int array [n, 8]
    of (bh0, ta0, bh1, ta1, rank, cost, tile1_valid, 0).  steps: None for the
    whole ring, or a single step index."""
    s0, s1 = (0, n_blocks) if steps is None else (steps, steps + 1)
    L = lib()
    n = L.ra_schedule_units(B, H, Hkv, S, n_blocks, LAYOUTS[layout], int(bool(causal)), s0, s1, None, 0)
    if n < 0:
        raise ValueError("invalid schedule request")
    out = np.zeros((n, 8), dtype=np.int32)
    L.ra_schedule_units(B, H, Hkv, S, n_blocks, LAYOUTS[layout], int(bool(causal)), s0, s1,
                        out.ctypes.data, n)
    return out


def block_units(B, H, Hkv, S, n_blocks, layout, causal, rank, step):
    """Work units ra_forward_block launches for (rank, step), same format as
    schedule_units."""
    L = lib()
    args = (B, H, Hkv, S, n_blocks, LAYOUTS[layout], int(bool(causal)), rank, step)
    n = L.ra_schedule_block_units(*args, None, 0)
    if n < 0:
        raise ValueError("invalid schedule request")
    out = np.zeros((n, 8), dtype=np.int32)
    L.ra_schedule_block_units(*args, out.ctypes.data, n)
    return out


def forward_block(q, k, v, out_s, lse_s, n_blocks, rank, step, layout="contiguous", causal=False,
                  stream=None):
    """One device's ring step (ra_forward_block): writes the fp32 partial of
    query block `rank` against key/value block (rank - step) mod n_blocks into
    the rows of that block in out_s [B,H,S,d] and lse_s [B,H,S].  q, k, v are
    in the layout's rank-major order."""
    B, H, Hkv, S, d = _dims(q, k, v)
    if out_s.dtype != torch.float32 or lse_s.dtype != torch.float32:
        raise ValueError("out_s and lse_s must be float32")
    if tuple(out_s.shape) != (B, H, S, d) or tuple(lse_s.shape) != (B, H, S):
        raise ValueError("out_s must be [B,H,S,d] and lse_s [B,H,S]")
    if not (out_s.is_contiguous() and lse_s.is_contiguous()):
        raise ValueError("out_s and lse_s must be contiguous")
    st = lib().ra_forward_block(_p(q), _p(k), _p(v), _p(out_s), _p(lse_s), B, H, Hkv, S, d, n_blocks,
                                LAYOUTS[layout], int(bool(causal)), DTYPES[q.dtype], int(rank),
                                int(step), _stream(stream))
    _check(st, "ra_forward_block")


def backward(q, k, v, out, lse, dout, n_blocks: int, layout: str = "contiguous", causal: bool = False,
             workspace=None, stream=None):
    """Gradients (dq, dk, dv) of sum(dout * out) for (out, lse) = forward(q, k,
    v, ...) with the same n_blocks, layout and causal (ra_backward / ra_backward_ws
    for bf16, ra_backward_f32 for fp32).  CUDA tensors in natural token order;
    lse fp32 [B,H,S]."""
    B, H, Hkv, S, d = _dims(q, k, v)
    for t, shape in ((out, q.shape), (dout, q.shape)):
        if t.shape != shape or t.dtype != q.dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError("out and dout must be contiguous CUDA tensors shaped like q, of q's dtype")
    if lse.shape != (B, H, S) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B,H,S] tensor")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    L = lib()
    args = [_p(q), _p(k), _p(v), _p(out), _p(lse), _p(dout), _p(dq), _p(dk), _p(dv), B, H, Hkv, S, d,
            n_blocks, LAYOUTS[layout], int(bool(causal))]
    if q.dtype == torch.float32:
        if workspace is not None:
            raise ValueError("the fp32 backward allocates its own scratch")
        _check(L.ra_backward_f32(*args, _stream(stream)), "ra_backward_f32")
    elif workspace is None:
        _check(L.ra_backward(*args, _stream(stream)), "ra_backward")
    else:
        _check(L.ra_backward_ws(*args, _p(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream)), "ra_backward_ws")
    return dq, dk, dv


def backward_tile_pairs(B, H, Hkv, S, n_blocks, layout, causal, which):
    """(query tile, key tile) pairs of the backward kernels in visiting order:
    int array [n, 8] of (unit, bh, i, ta, j, tb, position, 0); which 0 = dK/dV
    kernel, 1 = dQ kernel."""
    L = lib()
    args = (B, H, Hkv, S, n_blocks, LAYOUTS[layout], int(bool(causal)), int(which))
    n = L.ra_backward_tile_pairs(*args, None, 0)
    if n < 0:
        raise ValueError("invalid schedule request")
    out = np.zeros((n, 8), dtype=np.int32)
    L.ra_backward_tile_pairs(*args, out.ctypes.data, n)
    return out


def backward_workspace_bytes(B, H, Hkv, S, d, n_blocks, layout="contiguous", causal=False) -> int:
    return int(lib().ra_backward_workspace_bytes(B, H, Hkv, S, d, n_blocks, LAYOUTS[layout], int(causal)))


def all_to_all(x: torch.Tensor, n_dev: int, inverse: bool = False,
               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Ulysses all-to-all (ra_all_to_all): sequence-sharded [n_dev, B, Hn, L, d]
    -> head-sharded [n_dev, B, Hn/n_dev, S, d], or back with inverse=True.
    Per-row values (lse) drop the trailing d axis."""
    if not x.is_cuda or not x.is_contiguous() or x.dim() not in (4, 5):
        raise ValueError("x must be a contiguous CUDA tensor of 5 (or 4, for per-row values) dims")
    per_row = x.dim() == 4
    n, B = x.shape[0], x.shape[1]
    d = 1 if per_row else x.shape[4]
    if n != n_dev:
        raise ValueError("dim 0 must be n_dev")
    if not inverse:
        Hn, S = x.shape[2], x.shape[3] * n_dev
        shape = (n_dev, B, Hn // n_dev, S) + (() if per_row else (d,))
    else:
        Hn, S = x.shape[2] * n_dev, x.shape[3]
        shape = (n_dev, B, Hn, S // n_dev) + (() if per_row else (d,))
    if out is None:
        out = torch.empty(shape, dtype=x.dtype, device=x.device)
    _check(lib().ra_all_to_all(_p(x), _p(out), B, Hn, S, d, x.element_size(), n_dev, int(bool(inverse)),
                               _stream(stream)), "ra_all_to_all")
    return out


def forward_ulysses(q, k, v, n_dev: int, causal: bool = False, workspace=None, stream=None):
    """Ulysses attention over n_dev emulated devices (ra_forward_ulysses).
    q [n_dev, B, H, L, d], k/v [n_dev, B, Hkv, L, d] sequence shards; returns
    (out [n_dev, B, H, L, d], lse fp32 [n_dev, B, H, L])."""
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 5:
            raise ValueError("q, k, v must be contiguous CUDA tensors [n_dev, B, heads, L, d]")
    n, B, H, Ls, d = q.shape
    Hkv = k.shape[2]
    if n != n_dev or v.shape != k.shape or k.shape[0] != n or k.shape[1] != B or k.shape[3:] != q.shape[3:]:
        raise ValueError("shard shapes do not match")
    if q.dtype not in DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share a supported dtype")
    S = Ls * n_dev
    L = lib()
    nbytes = int(L.ra_ulysses_workspace_bytes(B, H, Hkv, S, d, n_dev, int(bool(causal)), DTYPES[q.dtype]))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q)
    lse = torch.empty(n_dev, B, H, Ls, device=q.device, dtype=torch.float32)
    _check(L.ra_forward_ulysses(_p(q), _p(k), _p(v), _p(out), _p(lse), B, H, Hkv, S, d, n_dev,
                                int(bool(causal)), DTYPES[q.dtype], _p(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
           "ra_forward_ulysses")
    return out, lse


def set_kernel_variant(variant: int) -> int:
    """0 automatic (= 3), 1 single-CTA tensor-core kernel, 3 single-CTA
    kernel in clusters of two sharing each key/value load where the heads
    allow it; returns the previous setting."""
    prev = lib().ra_set_kernel_variant(int(variant))
    if prev < 0:
        raise ValueError(f"invalid kernel variant {variant}")
    return prev
