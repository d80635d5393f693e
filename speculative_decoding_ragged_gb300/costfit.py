"""Least-squares fit of the additive step-cost model the confidence scheduler maximises against.

"DSpark in SGLang" (LMSYS blog summary), A2 method details, cost-table profiling and modelling
(Fig. 6): the scheduler's estimate of one decode step is T(bs, K) = bias + alpha(bs) + theta(M)
with M = bs + K, where alpha(bs) is the per-request floor (draft pass, part of attention) and
theta(M) the target's cost of verifying M tokens. The pages fit this model to recorded step
times and compare the fit's predictions with measured steps; they do not print the fitting
procedure, so this module takes the plainest reading: ordinary least squares over table
entries.

* Parameters: one bias, one alpha per distinct recorded batch size, one theta per distinct
  recorded key of M. The key is M itself, or the capture tier M is padded to when `tiers` is
  given (a graph replayed at a tier costs the same for every M it holds).
* Gauge: bias, alpha and theta are only defined up to constants moved between them, so the
  first (smallest) alpha and theta entries are pinned to zero and the bias carries the level.
* Full tables for dspark_schedule (alpha[0..B], theta[0..B*gamma]) interpolate linearly between
  recorded knots in bs and in the key, and hold the end values outside the recorded range.

Host-side numpy only; the fitted tables are plain float64 arrays the caller hands to
dspark_schedule (through CostTable).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np


def tier_key(M, tiers: Optional[Sequence[int]]) -> np.ndarray:
    """The theta key of each M: M itself, or the smallest tier >= M (M when no tier holds it),
    the row count dspark_pack pads to."""
    M = np.asarray(M, dtype=np.int64)
    if tiers is None or len(tiers) == 0:
        return M.copy()
    t = np.sort(np.asarray(tiers, dtype=np.int64))
    i = np.searchsorted(t, M, side="left")
    out = M.copy()
    ok = i < t.size
    out[ok] = t[i[ok]]
    return out


def _interp(x, knots, values) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    if knots.size == 1:
        return np.full(x.shape, values[0], dtype=np.float64)
    return np.interp(x, knots.astype(np.float64), values)


@dataclass
class AdditiveFit:
    bias: float
    bs_knots: np.ndarray       # recorded batch sizes, ascending
    alpha_knots: np.ndarray    # alpha at those sizes; alpha_knots[0] == 0 (gauge)
    key_knots: np.ndarray      # recorded theta keys (M or tier), ascending
    theta_knots: np.ndarray    # theta at those keys; theta_knots[0] == 0 (gauge)
    tiers: Optional[tuple]
    residual_rms: float        # root mean square of the training residuals
    n_samples: int

    def alpha(self, bs) -> np.ndarray:
        return _interp(bs, self.bs_knots, self.alpha_knots)

    def theta(self, M) -> np.ndarray:
        return _interp(tier_key(M, self.tiers), self.key_knots, self.theta_knots)

    def predict(self, bs, M) -> np.ndarray:
        return self.bias + self.alpha(bs) + self.theta(M)

    def tables(self, B: int, gamma: int):
        """(bias, alpha[0..B], theta[0..B*gamma]) as float64 arrays for dspark_schedule."""
        alpha = self.alpha(np.arange(B + 1))
        theta = self.theta(np.arange(B * gamma + 1))
        return float(self.bias), alpha, theta


def fit_additive(bs, M, T, tiers: Optional[Sequence[int]] = None) -> AdditiveFit:
    """Fit bias, alpha(bs) and theta(key(M)) to step times T by ordinary least squares.

    bs, M, T: equal-length 1-D sequences of recorded samples (batch size, verified tokens
    M = bs + K, step time in any unit). Raises ValueError when the samples do not determine
    the tables: a batch size and a key that never share a chain of samples (the bipartite
    graph of recorded (bs, key) pairs is disconnected)."""
    bs = np.asarray(bs, dtype=np.int64).ravel()
    M = np.asarray(M, dtype=np.int64).ravel()
    T = np.asarray(T, dtype=np.float64).ravel()
    if not (bs.size == M.size == T.size) or bs.size == 0:
        raise ValueError("bs, M and T must be non-empty and of equal length")
    if (bs < 0).any() or (M < bs).any():
        raise ValueError("need 0 <= bs <= M for every sample")
    if not np.isfinite(T).all():
        raise ValueError("step times must be finite")
    tiers_t = None if tiers is None else tuple(int(t) for t in tiers)
    key = tier_key(M, tiers_t)
    bs_knots, bs_idx = np.unique(bs, return_inverse=True)
    key_knots, key_idx = np.unique(key, return_inverse=True)
    na, nt = bs_knots.size, key_knots.size
    n_col = 1 + (na - 1) + (nt - 1)
    X = np.zeros((T.size, n_col), dtype=np.float64)
    X[:, 0] = 1.0
    rows = np.arange(T.size)
    a = bs_idx > 0
    X[rows[a], bs_idx[a]] = 1.0
    t = key_idx > 0
    X[rows[t], (na - 1) + key_idx[t]] = 1.0
    coef, _, rank, _ = np.linalg.lstsq(X, T, rcond=None)
    if rank < n_col:
        raise ValueError("the samples do not determine the additive tables: some batch sizes "
                         "and keys of M never occur linked through common samples")
    alpha = np.concatenate([[0.0], coef[1:na]])
    theta = np.concatenate([[0.0], coef[na:]])
    resid = T - X @ coef
    return AdditiveFit(bias=float(coef[0]), bs_knots=bs_knots, alpha_knots=alpha,
                       key_knots=key_knots, theta_knots=theta, tiers=tiers_t,
                       residual_rms=float(np.sqrt(np.mean(resid * resid))), n_samples=int(T.size))


def compare(fit: AdditiveFit, bs, M, T) -> dict:
    """Predicted against measured step times: mean and max relative error, R^2, samples."""
    T = np.asarray(T, dtype=np.float64).ravel()
    P = fit.predict(bs, M)
    rel = np.abs(P - T) / np.abs(T)
    ss_res = float(np.sum((T - P) ** 2))
    ss_tot = float(np.sum((T - T.mean()) ** 2))
    return dict(n=int(T.size), mean_abs_rel=float(rel.mean()), max_abs_rel=float(rel.max()),
                r2=(1.0 - ss_res / ss_tot) if ss_tot > 0 else float("nan"))
