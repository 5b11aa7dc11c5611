"""Match criteria of the CUDA path against the oracle.

* top-k: the selected sets must be equal, except that an element on either
  side of the difference is tolerated (reported) when its oracle score lies
  within 1e-4 relative of the k-th oracle score (accumulation order decides
  near-ties); sizes, range, uniqueness and the -1 tail are exact.
* indexer scores: |I_gpu - I_or| <= 1e-2 * max(|I_or|, 1e-3 * max_s |I_or|).
* attention: ||o_gpu - o_or||_2 / ||o_or||_2 <= 2e-2 per row (bf16), 1e-4 (float32).
"""
from __future__ import annotations

import numpy as np

from oracle import topk as otopk

TIE_BAND = 1e-4
SCORE_RTOL = 1e-2
ATT_TOL_BF16 = 2e-2
ATT_TOL_F32 = 1e-4


def check_topk_row(gpu_row: np.ndarray, scores: np.ndarray, k: int) -> int:
    """Returns the number of tolerated (near-tie) differences; raises on a real one."""
    gpu_row = np.asarray(gpu_row, dtype=np.int64)
    V = len(scores)
    n = min(k, V)
    valid = gpu_row[gpu_row >= 0]
    assert len(valid) == n, f"selected {len(valid)} positions, expected {n}"
    assert np.all(gpu_row[:n] >= 0) and np.all(gpu_row[n:] == -1), "padding must be a -1 tail"
    assert len(np.unique(valid)) == n, "duplicate positions"
    assert valid.min() >= 0 and valid.max() < V, "position outside the visible range"
    want = otopk.topk_select(scores, k)
    want = set(int(x) for x in want if x >= 0)
    got = set(int(x) for x in valid)
    diff = want.symmetric_difference(got)
    if not diff:
        return 0
    Ik = otopk.kth_score(scores, k)
    for s in diff:
        assert abs(scores[s] - Ik) <= TIE_BAND * abs(Ik), \
            f"position {s} (score {scores[s]!r}) differs but is not within the tie band of the k-th score {Ik!r}"
    return len(diff)


def check_scores_row(gpu: np.ndarray, ref: np.ndarray):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    floor = 1e-3 * np.max(np.abs(ref)) if len(ref) else 0.0
    tol = SCORE_RTOL * np.maximum(np.abs(ref), floor)
    bad = np.abs(gpu - ref) > tol
    assert not bad.any(), f"{bad.sum()} scores out of tolerance, worst {np.max(np.abs(gpu - ref) - tol)}"


def rel_l2(gpu: np.ndarray, ref: np.ndarray) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nrm = np.linalg.norm(ref)
    return float(np.linalg.norm(gpu - ref) / (nrm if nrm > 0 else 1.0))


def check_attention_row(gpu_o, ref_o, tol):
    e = rel_l2(gpu_o, ref_o)
    assert e <= tol, f"relative L2 error {e} > {tol}"
    return e
