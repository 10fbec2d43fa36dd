"""Shared helpers for the GPU parity tests (comparison rules, oracle plumbing)."""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_layer_permute_gb300 import workloads as wl

# float tolerances: rel_rms = ||got - ref|| / ||ref|| and max|got - ref| / max|ref| must both hold
TOL_F32 = 1e-5
TOL_BF16 = 2e-2


def rel_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    den = np.linalg.norm(ref)
    rel_rms = np.linalg.norm(got - ref) / den if den > 0 else np.linalg.norm(got)
    m = np.abs(ref).max() if ref.size else 0.0
    max_rel = np.abs(got - ref).max() / m if m > 0 else (np.abs(got).max() if got.size else 0.0)
    return rel_rms, max_rel


def assert_close(got, ref, tol, what=""):
    rel_rms, max_rel = rel_errors(got, ref)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite values"
    assert rel_rms <= tol and max_rel <= tol, f"{what}: rel_rms={rel_rms:.3e} max_rel={max_rel:.3e} tol={tol}"


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def compact_experts(ids: np.ndarray, W1: torch.Tensor, W2: torch.Tensor, S1=None, S2=None):
    """Host copies of only the experts that `ids` uses, and ids remapped to them (for sampled oracle runs)."""
    used = sorted({int(e) for e in ids.reshape(-1) if e >= 0})
    remap = np.full(max(used, default=0) + 2, -1, np.int64)
    for n, e in enumerate(used):
        remap[e] = n
    new_ids = np.where(ids >= 0, remap[np.where(ids >= 0, ids, len(remap) - 1)], -1).astype(np.int32)
    sel = torch.tensor(used, dtype=torch.long, device=W1.device)
    out = [wl.to_numpy(W1.index_select(0, sel)), wl.to_numpy(W2.index_select(0, sel))]
    out.append(None if S1 is None else wl.to_numpy(S1.index_select(0, sel)))
    out.append(None if S2 is None else wl.to_numpy(S2.index_select(0, sel)))
    return new_ids, out


def oracle_map(fn, tasks, workers=None):
    """Runs fn(task) for every task on a thread pool and returns the results in task order.

    The oracle's C calls release the GIL (ctypes), so one oracle call per token runs on every host core at
    once, sharing the host arrays without copies; the oracle itself is unchanged (one plain call per task)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    n = workers or max(1, os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=n) as ex:
        return list(ex.map(fn, tasks))
