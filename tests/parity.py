"""Parity checks of GPU results against the oracle.

Scores: |gpu - oracle| <= 1e-6 * max_b |oracle[i][b]| per row (the FP64
gate floored at 1e-6 of the score scale, "#337 gfx12 QSA select", What
item 2 and the bench paragraph).

Ids, two ways:
- exact: the GPU top-k of the GPU's own fp32 scores equals the oracle's
  top-k of those same fp32 scores, bit for bit (ties to lower ids);
- near-tie rule against the FP64 oracle: where the k-th and (k+1)-th
  oracle scores differ by more than 4x the row tolerance the ids are equal;
  otherwise every id in the symmetric difference lies within 4x the
  tolerance of the k-th score.
"""

from __future__ import annotations

import numpy as np

SCORE_REL_TOL = 1e-6


def row_tol(S_ref: np.ndarray) -> np.ndarray:
    return SCORE_REL_TOL * np.abs(S_ref).max(axis=1)


def check_scores(S_gpu: np.ndarray, S_ref: np.ndarray) -> float:
    """Asserts the score gate; returns the worst error in units of tol."""
    assert S_gpu.shape == S_ref.shape, (S_gpu.shape, S_ref.shape)
    assert S_gpu.dtype == np.float32
    assert not np.isnan(S_gpu).any(), "NaN in GPU scores"
    tol = row_tol(S_ref)[:, None]
    err = np.abs(S_gpu.astype(np.float64) - S_ref)
    ratio = err / np.maximum(tol, np.finfo(np.float64).tiny)
    worst = float(ratio.max()) if ratio.size else 0.0
    assert np.all(err <= tol), f"score error {worst:.3g} x tolerance (row, col) {np.unravel_index(ratio.argmax(), ratio.shape)}"
    return worst


def check_ids_valid(ids: np.ndarray, active: int, k: int) -> None:
    m = min(k, active)
    assert ids.shape[1] == k
    assert np.all(ids[:, m:] == -1)
    sel = ids[:, :m]
    assert np.all(sel >= 0) and np.all(sel < active)
    if m > 1:
        assert np.all(np.diff(sel, axis=1) > 0), "ids not strictly ascending (duplicates or order)"


def check_ids_near_tie(ids_gpu: np.ndarray, S_ref: np.ndarray, ids_ref: np.ndarray, k: int) -> int:
    """Returns the number of rows exempted as near-ties."""
    nq, active = S_ref.shape
    check_ids_valid(ids_gpu, active, k)
    if k >= active:
        assert np.array_equal(ids_gpu, ids_ref)
        return 0
    tol = row_tol(S_ref)
    exempt = 0
    for i in range(nq):
        if np.array_equal(ids_gpu[i], ids_ref[i]):
            continue
        srt = np.sort(S_ref[i])[::-1]
        sk, sk1 = srt[k - 1], srt[k]
        assert sk - sk1 <= 4 * tol[i], f"row {i}: ids differ with a clear gap {sk - sk1:.3g} > 4 tol"
        diff = np.setxor1d(ids_gpu[i], ids_ref[i])
        assert np.all(np.abs(S_ref[i][diff] - sk) <= 4 * tol[i]), f"row {i}: differing id not a near-tie"
        exempt += 1
    return exempt
