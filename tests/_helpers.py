"""Shared test helpers: run the library on a workload and compare with the
oracle under the tolerances the method fixes."""
from __future__ import annotations

import numpy as np
import torch

import oracle.dsa_oracle as O
from dsa_inputs import make_inputs, to_f64

# output tolerances (relative L2 over the whole output tensor)
TOL_16BIT = 2e-3
TOL_INT8 = 5e-3
# selected sets may differ only where a score lies this close (relative) to
# the k-th score
SEL_REL = 1e-5


def f64_inputs(cpu: dict) -> dict:
    out = {}
    for k, v in cpu.items():
        out[k] = to_f64(v) if isinstance(v, torch.Tensor) else v
    out["total_len"] = cpu["total_len"].numpy().astype(np.int64)
    return out


def to_device(cpu: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def score_error_bound(qI_s, w_s, kI_rows, score):
    """Forward-error bound of an fp32-accumulated indexer score (two times
    the classic gamma_n bound of the 64-term dot products, plus the head sum)."""
    u = 2.0 ** -24
    absdots = np.abs(kI_rows) @ np.abs(qI_s).T            # [n, HI]
    return 2.0 * (absdots @ w_s) * (64 * u) * 1.01 + np.abs(score) * 40 * u + 1e-30


def check_index_row(gpu_row, qI_s, w_s, kI_b, n):
    ref = O.index_scores_row(qI_s, w_s, kI_b, n)
    bound = score_error_bound(qI_s, w_s, kI_b[:n], ref)
    err = np.abs(gpu_row[:n].astype(np.float64) - ref)
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, (f"{bad.size} scores outside the fp32 error bound; first t={bad[0]} "
                           f"gpu={gpu_row[bad[0]]} ref={ref[bad[0]]} bound={bound[bad[0]]}")
    return ref


def check_selection(ref_scores_row: np.ndarray, gpu_idx_row: np.ndarray, k: int):
    """The GPU's selected set must be a valid top-k of the oracle scores up to
    the tie band: elements of the symmetric difference with the oracle's set
    all score within SEL_REL (relative) of the oracle's k-th score."""
    n = ref_scores_row.shape[0]
    keff = min(k, n)
    g = np.asarray(gpu_idx_row, dtype=np.int64)
    assert (g[keff:] == -1).all(), "padding after k_eff must be -1"
    sel = g[:keff]
    assert (sel >= 0).all() and (sel < n).all(), "selected index out of range"
    assert keff <= 1 or (np.diff(sel) > 0).all(), "selected indices must ascend"
    oref = O.topk_select_row(ref_scores_row, k)[:keff]
    diff = np.setxor1d(sel, oref)
    if diff.size == 0:
        return 0
    order = np.sort(ref_scores_row)[::-1]
    kth = order[keff - 1]
    tol = SEL_REL * max(abs(kth), 1e-30)
    far = diff[np.abs(ref_scores_row[diff] - kth) > tol]
    assert far.size == 0, (f"{far.size} selection differences away from the k-th score "
                           f"{kth}: e.g. t={far[0]} score={ref_scores_row[far[0]]}")
    return diff.size
