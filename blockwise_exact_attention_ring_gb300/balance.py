"""Load balance of the ring schedule across devices.

On a ring of N devices every device computes one (query block, key/value
block) pair per ring step and then passes its key/value block on, so a step
ends when its slowest device ends.  The time of the whole ring is therefore
the critical path sum_s max_i w(i, s) over the work w(i, s) of device i at
step s, against an ideal of sum_{i,s} w(i, s) / N.  With a causal mask and
contiguous blocks the devices that hold early query blocks see mostly masked
key blocks and wait; striping the tokens over the devices evens the work
("Ring Attention" page, ultralytics.com/tr, section "Halka Dikkati Nasil
Calisir", its closing paragraph on causal masks and striped attention, which
reports up to 1.45x end-to-end training throughput at 256K tokens).

``model`` takes w from the host scheduler (visible query-key pairs or
128 x 128 tiles per device and step, ra_schedule_stats); ``measured`` takes
per-(device, step) kernel times, e.g. of ra_forward_block launches.  Both
return the same summary, so the model can be checked against the GPU.
"""
from __future__ import annotations

import numpy as np

from .binding import schedule_stats


def summarize(w: np.ndarray) -> dict:
    """Critical path of a lock-step ring for work w[i, s] (device i, step s)."""
    w = np.asarray(w, dtype=np.float64)
    if w.ndim != 2 or w.shape[0] != w.shape[1] or w.shape[0] < 1:
        raise ValueError("w must be a square [device, step] array")
    n = w.shape[0]
    step_max = w.max(axis=0)
    total = float(w.sum())
    cp = float(step_max.sum())
    ideal = total / n
    return {
        "n_blocks": n,
        "total": total,
        "critical_path": cp,
        "ideal": ideal,
        "imbalance": cp / ideal if ideal > 0 else float("nan"),
        "step_max": step_max.tolist(),
        "busy_fraction": ideal / cp if cp > 0 else float("nan"),
    }


def model(layout: str, causal: bool, n_blocks: int, L: int, unit: str = "pairs") -> dict:
    """Critical-path summary from the scheduler's work counts; unit is
    'pairs' (visible query-key pairs) or 'tiles' (128 x 128 tiles launched,
    which includes the masked half of diagonal tiles)."""
    _, pairs, tiles = schedule_stats(layout, causal, n_blocks, L)
    if unit not in ("pairs", "tiles"):
        raise ValueError("unit must be 'pairs' or 'tiles'")
    out = summarize(pairs if unit == "pairs" else tiles)
    out.update({"layout": layout, "causal": bool(causal), "L": L, "unit": unit})
    return out


def measured(times: np.ndarray) -> dict:
    """Critical-path summary of measured per-(device, step) times."""
    out = summarize(times)
    out["unit"] = "time"
    return out
