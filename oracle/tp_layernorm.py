"""Plain fp64 CPU oracle of LayerNorm with the hidden dimension split over the shards.

TEST INFRASTRUCTURE ONLY: slow on purpose and written for reading. It shares no code with the
CUDA library and imports nothing from it.

Page this follows (cited by title and section):

* [Intelli] "Tensor Parallelism: principle and practice", section 4.2 (how each layer type is
  split): for layer normalisation each device computes the mean and variance on its own
  part, and the statistics are then synchronised with an All-Reduce.

Reading taken where the page is silent:

* R9  Each shard holds a block of columns of every token row (the hidden dimension is split),
      with its slice of gamma and beta. The statistics that the All-Reduce combines are those
      of the whole row: the mean and the biased variance (divided by the hidden size), with
      eps added to the variance inside the square root, as in the usual LayerNorm
      y = (x - mean) / sqrt(var + eps) * gamma + beta. Combining the shards' statistics
      reaches exactly (up to rounding) the statistics of the concatenated row, so the oracle
      is that plain definition written out on the concatenated row; its outputs are cut back
      into the shards' column blocks. The backward is the plain gradient of that definition;
      its per-row sums (of dY * gamma and of dY * gamma * xhat) are the same kind of
      all-shard statistics.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np

__all__ = ["layernorm_forward", "layernorm_backward", "split_hidden"]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def split_hidden(M, n: int) -> List[np.ndarray]:
    """Column blocks of [T, H] (or of a vector [H]) for n shards; H must divide by n."""
    M = _f64(M)
    H = M.shape[-1]
    if H % n != 0:
        raise ValueError(f"hidden {H} is not divisible by {n} shards")
    s = H // n
    return [M[..., i * s:(i + 1) * s] for i in range(n)]


def _concat(parts: Sequence[np.ndarray]) -> np.ndarray:
    return np.concatenate([_f64(p) for p in parts], axis=-1)


def layernorm_forward(X_shards, gamma_shards=None, beta_shards=None, eps: float = 1e-5):
    """[Intelli] section 4.2, reading R9. X_shards: n arrays [T, H/n] (column blocks of every
    token row); gamma_shards, beta_shards: n arrays [H/n] or None (1 and 0).

    Returns {"Y": n arrays [T, H/n], "mean": [T], "rstd": [T], "xhat": [T, H]}."""
    n = len(X_shards)
    X = _concat(X_shards)
    T, H = X.shape
    gamma = np.ones(H) if gamma_shards is None else _concat(gamma_shards)
    beta = np.zeros(H) if beta_shards is None else _concat(beta_shards)
    mean = X.mean(axis=1)                                   # the row's mean
    var = ((X - mean[:, None]) ** 2).mean(axis=1)           # biased variance of the row
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (X - mean[:, None]) * rstd[:, None]
    Y = xhat * gamma[None, :] + beta[None, :]
    return {"Y": split_hidden(Y, n), "mean": mean, "rstd": rstd, "xhat": xhat}


def layernorm_backward(X_shards, gamma_shards, dY_shards, eps: float = 1e-5, fwd=None):
    """Gradient of layernorm_forward. With g = dY * gamma and row means over the whole hidden
    dimension:  dX = rstd * (g - mean(g) - xhat * mean(g * xhat));  dgamma = sum_t dY * xhat;
    dbeta = sum_t dY (column sums over the tokens, per shard).

    Returns {"dX": n arrays [T, H/n], "dgamma": n arrays [H/n], "dbeta": n arrays [H/n]}."""
    n = len(X_shards)
    if fwd is None:
        fwd = layernorm_forward(X_shards, gamma_shards, None, eps)
    xhat, rstd = fwd["xhat"], fwd["rstd"]
    H = xhat.shape[1]
    gamma = np.ones(H) if gamma_shards is None else _concat(gamma_shards)
    dY = _concat(dY_shards)
    g = dY * gamma[None, :]
    m1 = g.mean(axis=1)                    # statistic 1 of the row
    m2 = (g * xhat).mean(axis=1)           # statistic 2 of the row
    dX = rstd[:, None] * (g - m1[:, None] - xhat * m2[:, None])
    dgamma = (dY * xhat).sum(axis=0)
    dbeta = dY.sum(axis=0)
    return {"dX": split_hidden(dX, n), "dgamma": split_hidden(dgamma, n),
            "dbeta": split_hidden(dbeta, n)}
