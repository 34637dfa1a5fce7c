"""Float64 oracle of the offline rotation calibration.

TEST INFRASTRUCTURE ONLY: imported by tests/ and by the CPU leg of
``bench.py``; the product library never imports it.

Source: "卓绝TurboQuant：Together AI把2-bit KV Cache推向实在行状", section
"OSCAR 把旋转瞄准 attention": the orthogonal factor U of the rotation
R = U . Hadamard . bit-reversal is fixed offline per layer and KV head, for K
from the covariance of the queries that read the keys, for V from the
covariance of the values as weighted by the attention scores.  The pages give
no formula; the plainest reading, taken here:

  - U_K[kv] = eigenvectors of C_K = mean over calibration samples of q q^T,
    the samples being every calibration query token of every query head that
    uses KV head kv (query head h uses KV head h // G);
  - U_V[kv] = eigenvectors of C_V = mean of o o^T over the same samples, o the
    attention output of that query head over the calibration tokens (full,
    non-causal attention, scale sm_scale): with S the attention-probability
    matrix, sum o o^T = (S V)^T (S V) = V^T S^T S V, the score-weighted
    value covariance;
  - U's columns are the eigenvectors sorted by decreasing eigenvalue, each
    with its entry of largest magnitude positive (first such entry on ties),
    so that y = x . U projects x on the principal directions in order.

Everything is float64 with numpy; ``numpy.linalg.eigh`` serves as the
symmetric eigensolver (a library primitive).
"""
from __future__ import annotations

import numpy as np


def query_covariance(q: np.ndarray, num_kv_heads: int) -> np.ndarray:
    """C_K: q [n][Hq][d] -> [Hk][d][d], mean of q q^T over (token, head of the group)."""
    n, hq, d = q.shape
    g = hq // num_kv_heads
    x = np.asarray(q, np.float64).reshape(n, num_kv_heads, g, d)
    out = np.empty((num_kv_heads, d, d))
    for kv in range(num_kv_heads):
        s = x[:, kv].reshape(n * g, d)
        out[kv] = s.T @ s / (n * g)
    return out


def attention_outputs(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float) -> np.ndarray:
    """o [n][Hq][d]: full softmax attention of every query head over the
    calibration tokens of its KV head (k, v: [t][Hk][d])."""
    n, hq, d = q.shape
    hk = k.shape[1]
    g = hq // hk
    q64, k64, v64 = (np.asarray(a, np.float64) for a in (q, k, v))
    out = np.empty((n, hq, d))
    for h in range(hq):
        kv = h // g
        logits = (q64[:, h, :] @ k64[:, kv, :].T) * sm_scale          # [n][t]
        logits -= logits.max(axis=1, keepdims=True)
        p = np.exp(logits)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v64[:, kv, :]
    return out


def value_covariance(o: np.ndarray, num_kv_heads: int) -> np.ndarray:
    """C_V: the same mean of outer products as query_covariance, over the outputs."""
    return query_covariance(o, num_kv_heads)


def rotation_from_covariance(c: np.ndarray):
    """(U, eigenvalues) of a symmetric matrix: columns sorted by decreasing
    eigenvalue, largest-magnitude entry of each column positive."""
    w, u = np.linalg.eigh(np.asarray(c, np.float64))
    order = np.argsort(-w, kind="stable")
    w, u = w[order], u[:, order]
    for j in range(u.shape[1]):
        i = int(np.argmax(np.abs(u[:, j])))
        if u[i, j] < 0:
            u[:, j] = -u[:, j]
    return u, w


def calibrate(q: np.ndarray, kv: np.ndarray, sm_scale: float):
    """U [Hk][2][d][d] (K, V) and eigenvalues [Hk][2][d] from calibration
    queries q [n][Hq][d] and tokens kv [t][Hk][2][d]."""
    hk = kv.shape[1]
    d = q.shape[2]
    ck = query_covariance(q, hk)
    cv = value_covariance(attention_outputs(q, kv[:, :, 0, :], kv[:, :, 1, :], sm_scale), hk)
    U = np.empty((hk, 2, d, d))
    lam = np.empty((hk, 2, d))
    for h in range(hk):
        U[h, 0], lam[h, 0] = rotation_from_covariance(ck[h])
        U[h, 1], lam[h, 1] = rotation_from_covariance(cv[h])
    return U, lam


def clip_search(kv: np.ndarray, U: np.ndarray, grid, group: int = 32):
    """Clip ratios chosen offline with U ([NEWS] sec. B fixes the clip
    thresholds offline together with U; the criterion is a reading): for
    each (KV head, K/V) the candidate c with the least mean squared error
    sum (y - y^)^2 / (n_t d) over the calibration tokens, y = x . R the rotated
    vector (float64) and y^ its dequantised value under the eviction's
    quantiser (the C oracle's quantize_vec / dequantize_vec) with clip c,
    measured against the unclipped y; ties go to the larger c.

    kv: float64 [n_t][Hk][2][d]; U: [Hk][2][d][d].  Returns (clip [Hk][2],
    mse [Hk][2][len(grid)])."""
    from oracle import get
    orc = get()
    n_t, hk, _, d = kv.shape
    grid = [float(c) for c in grid]
    mse = np.zeros((hk, 2, len(grid)))
    clip = np.zeros((hk, 2))
    for h in range(hk):
        for w in range(2):
            Y = np.asarray(kv[:, h, w, :], np.float64) @ orc.build_R(U[h, w])
            for ci, c in enumerate(grid):
                err = 0.0
                for y in Y:
                    codes, s16, z16 = orc.quantize_vec(y, group, c)[:3]
                    err += float(((y - orc.dequantize_vec(codes, s16, z16, group)) ** 2).sum())
                mse[h, w, ci] = err / (n_t * d)
            best = 0
            for ci in range(1, len(grid)):
                if mse[h, w, ci] < mse[h, w, best] or (mse[h, w, ci] == mse[h, w, best] and grid[ci] > grid[best]):
                    best = ci
            clip[h, w] = grid[best]
    return clip, mse
