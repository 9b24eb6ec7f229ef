"""fp64 reference gradients of causal, GQA-aware attention (the backward pass).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages describe the backward pass only by what it reuses: it rebuilds the
score blocks from Q, K and the small saved row statistics instead of storing
the L x L table ("Long-Context Attention Explained" (sevydevy), "What
FlashAttention does not change"; "Memory-bound vs compute-bound" lesson
(Pranay), "Attention itself": recomputation in the backward pass is close to
free). What it computes is fixed by the forward definition (oracle.attention):
the gradients of O = softmax(scale * Q K^T + mask) V with respect to Q, K and V
for an upstream gradient dO, written out by the chain rule:

    P_ij   = softmax_j(scale * s_ij)                (masked entries 0)
    dV_j   = sum_{h in group(j)} sum_i P_ij dO_i
    dP_ij  = dO_i . V_j
    D_i    = sum_j P_ij dP_ij                       (= dO_i . O_i)
    dS_ij  = P_ij (dP_ij - D_i)
    dQ_i   = scale * sum_j dS_ij K_j
    dK_j   = scale * sum_{h in group(j)} sum_i dS_ij Q_i

K/V head j of a GQA group collects the gradients of all g query heads that
read it. Everything is float64; P is rebuilt from the scores row block by row
block, exactly as the forward oracle builds it.
"""

from __future__ import annotations

import math

import numpy as np

_MAX_SCORE_ELEMS = 1 << 24


def attention_backward(q, k, v, do, *, causal: bool = True, scale: float | None = None):
    """Gradients (dq, dk, dv) of the attention forward for upstream gradient ``do``.

    q, do: [B, L, n_q, d]; k, v: [B, L, n_kv, d] (square prefill). Returns
    float64 arrays shaped like q, k, v.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, L, n_q, d = q.shape
    n_kv = k.shape[2]
    if k.shape != (B, L, n_kv, d) or v.shape != k.shape or do.shape != q.shape:
        raise ValueError("q, do: [B, L, n_q, d]; k, v: [B, L, n_kv, d]")
    if n_q % n_kv:
        raise ValueError("n_q must be a multiple of n_kv")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    scale = float(scale)
    g = n_q // n_kv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    step = max(1, min(256, _MAX_SCORE_ELEMS // max(L, 1)))
    keys = np.arange(L)
    for b in range(B):
        for h in range(n_q):
            kvh = h // g
            kmat, vmat = k[b, :, kvh, :], v[b, :, kvh, :]
            for i0 in range(0, L, step):
                rows = np.arange(i0, min(L, i0 + step))
                lv = int(rows[-1]) + 1 if causal else L
                qb, dob = q[b, rows, h, :], do[b, rows, h, :]
                s = scale * (qb @ kmat[:lv].T)
                if causal:
                    s = np.where(keys[None, :lv] <= rows[:, None], s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                p = np.exp(s - m)
                p /= p.sum(axis=1, keepdims=True)            # P, masked entries 0
                dp = dob @ vmat[:lv].T                       # dP = dO V^T
                dd = (p * dp).sum(axis=1, keepdims=True)     # D_i
                ds = p * (dp - dd)                           # dS
                dq[b, rows, h, :] = scale * (ds @ kmat[:lv])
                dk[b, :lv, kvh, :] += scale * (ds.T @ qb)
                dv[b, :lv, kvh, :] += p.T @ dob
    return dq, dk, dv


def softmax_rowdot(o, do):
    """D_i = dO_i . O_i per (b, h, i), [B, n_q, L]: the row statistic the
    backward pass needs besides the log-sum-exp."""
    o = np.asarray(o, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    return np.einsum("blhd,blhd->bhl", o, do)
