"""Helpers shared by the GPU parity tests: comparison rules and seeded setups.

Matching rules of the workload: FP4 codes and scales
bit-exact; top-K sets exact except for positions whose oracle score lies within
1e-4 relative of the K-th score; attention outputs within 2e-3 relative
(per (sequence, head) row: max|o - r| / max|r|)."""
from __future__ import annotations

import numpy as np
import torch

TOPK_REL = 1e-4
ATTN_REL = 2e-3


def check_topk(gpu_idx, ora_idx, ora_scores, rel=TOPK_REL, n_valid=None):
    """gpu_idx / ora_idx: int arrays [k] ascending with -1 padding; ora_scores:
    oracle score of each candidate index (dict-like or array)."""
    g = np.asarray(gpu_idx)
    o = np.asarray(ora_idx)
    gv, ov = g[g >= 0], o[o >= 0]
    assert np.all(g[len(gv):] == -1), "padding must follow the selected indices"
    assert np.all(np.diff(gv) > 0), "selected indices must be strictly ascending"
    assert len(gv) == len(ov), f"selected {len(gv)} vs oracle {len(ov)}"
    if n_valid is not None:
        assert np.all((gv >= 0) & (gv < n_valid))
    diff = set(gv.tolist()) ^ set(ov.tolist())
    if not diff:
        return 0
    s = np.asarray(ora_scores, dtype=np.float64)
    sk = s[ov].min()
    for i in diff:
        assert abs(s[i] - sk) <= rel * abs(sk), f"index {i}: score {s[i]} vs K-th {sk}"
    return len(diff)


def check_attn(out_gpu, out_ora, rel=ATTN_REL):
    o = np.asarray(out_gpu, dtype=np.float64)
    r = np.asarray(out_ora, dtype=np.float64)
    num = np.abs(o - r).max(axis=-1)
    den = np.abs(r).max(axis=-1)
    ok = (num <= rel * den) | ((den == 0) & (num == 0))
    worst = float((num / np.where(den > 0, den, 1)).max())
    assert ok.all(), f"attention rows off: worst normwise rel {worst}"
    return worst


def check_lse(lse_gpu, lse_ora, rel=ATTN_REL):
    g = np.asarray(lse_gpu, dtype=np.float64)
    r = np.asarray(lse_ora, dtype=np.float64)
    both_inf = np.isneginf(g) & np.isneginf(r)
    err = np.where(both_inf, 0.0, np.abs(g - r))
    assert np.all(err <= rel * np.maximum(np.abs(r), 1.0)), f"lse off by {err.max()}"


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
