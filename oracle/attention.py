"""fp64 reference for causal, GQA-aware scaled dot-product attention (forward).

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the CPU
baseline of the benchmark, never by the CUDA product path.

What it computes (the plain definition, no tiling, no online softmax):

    kv(h)  = h // g,  g = n_q / n_kv               (contiguous head groups)
    s_ij   = scale * sum_d Q[b,i,h,d] * K[b,j,kv(h),d]     for j in J(i)
    J(i)   = {0..i+Lk-Lq} if causal else {0..Lk-1}
    m_i    = max_j s_ij
    p_ij   = exp(s_ij - m_i),   l_i = sum_j p_ij
    O[b,i,h,:]  = sum_j p_ij * V[b,j,kv(h),:] / l_i
    LSE[b,h,i]  = m_i + ln(l_i)

Sources:
  * "Why Attention Scaling Breaks" (shivam2003), section "The O(n^2) problem":
    S = Q K^T, A = softmax(S / sqrt(d)), O = A V.
  * "Long-Context Attention Explained: Quadratic Cost, KV Cache and
    FlashAttention" (sevydevy): softmax of Q K^T over sqrt(head size) times V;
    softmax turns a row of scores into weights that add up to 1; a
    text-generating model lets each token look only backwards (its own
    position included, as in the class-room picture); subtracting the row
    maximum is the safe-softmax step that keeps exp from overflowing.
  * "prefill-attention" flop record (phantomic12), "Arithmetic intensity"
    and "Workarounds": GQA shares each K/V head among g = n_q/n_kv query
    heads.

Q may be a chunk of Lq query rows at the end of a longer sequence whose
Lk >= Lq keys and values are all present (chunked prefill: the
"prefill-attention" flop record (phantomic12), "Workarounds", splits a long
prompt into pieces; each piece attends to every earlier token and to itself).
Row i of the chunk sits at absolute position i + Lk - Lq. With Lq = Lk this is
ordinary square prefill.

Readings where the pages are silent (each listed in the design notes):
  * the mask keeps key j <= the query's absolute position (diagonal included);
  * a chunk is aligned to the end of the key range (bottom-right);
  * query head h reads K/V head h // g;
  * the log-sum-exp is the natural-log LSE of the *scaled* scores;
  * the scale multiplies the dot product; any finite value is allowed.

Inputs are whatever real arrays the caller passes (typically the exact bf16
values the GPU consumes, upcast); everything is computed in float64. Scores
are materialised one block of query rows at a time: a block of rows against
every key that row block can see, then masked, max-subtracted, exponentiated,
summed and applied to V with a library matmul. That blocking only bounds the
memory of the materialised scores; each row's arithmetic is the definition
above.
"""

from __future__ import annotations

import math

import numpy as np

# Largest number of float64 score entries materialised at once (128 MiB).
_MAX_SCORE_ELEMS = 1 << 24


def kv_head_of(h: int, n_q: int, n_kv: int) -> int:
    """K/V head read by query head ``h``: contiguous groups of g = n_q/n_kv."""
    if n_q % n_kv:
        raise ValueError("n_q must be a multiple of n_kv")
    return h // (n_q // n_kv)


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, L, H, d_h]")
    B, Lq, n_q, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k and v must be [B, Lk, n_kv, d_h] matching q")
    Lk, n_kv = k.shape[1], k.shape[2]
    if Lk < Lq:
        raise ValueError("k and v must hold at least as many positions as q")
    if n_q % n_kv:
        raise ValueError("n_q must be a multiple of n_kv")
    return B, Lq, Lk, n_q, n_kv, d


def _rows_block(qrows, krows, vrows, pos, causal, scale):
    """Definition applied to a set of query rows of one (b, h).

    qrows: [R, d] float64, the query vectors; pos: [R] their absolute
    positions. krows, vrows: [Lv, d] float64, every key/value the rows may
    see (Lv = max(pos)+1 when causal, else every key).
    Returns (o [R, d], lse [R]).
    """
    s = scale * (qrows @ krows.T)                     # [R, Lv] scores
    if causal:
        keys = np.arange(krows.shape[0])
        s = np.where(keys[None, :] <= pos[:, None], s, -np.inf)
    m = s.max(axis=1)                                 # row maximum
    m_safe = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - m_safe[:, None])                   # masked entries -> 0
    l = p.sum(axis=1)
    o = (p @ vrows) / l[:, None]
    lse = m_safe + np.log(l)
    return o, lse


def attention_rows(q, k, v, rows, *, causal: bool = True, scale: float | None = None,
                   n_q: int | None = None, lq: int | None = None):
    """Attention output for selected query rows only.

    ``rows``: integer array [R, 3] of (b, h, i), i a row of the query chunk.
    ``q`` is either the full [B, Lq, n_q, d] query tensor or just the R query
    vectors [R, d] of the listed rows, in the order of ``rows`` (then ``n_q``
    and ``lq`` (the chunk length, default Lk) must be given).
    k, v: [B, Lk, n_kv, d].
    Returns (o [R, d] float64, lse [R] float64) in the order of ``rows``.
    """
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    if q.ndim == 4:
        B, L, Lk, n_q, n_kv, d = _check_shapes(q, k, v)
        q_vec = None
    else:
        if n_q is None:
            raise ValueError("n_q is required when q holds only the selected rows")
        if q.ndim != 2 or q.shape[0] != rows.shape[0] or k.ndim != 4 or k.shape != v.shape:
            raise ValueError("q must be [R, d] matching rows; k, v [B, Lk, n_kv, d]")
        B, Lk, n_kv, d = k.shape
        L = Lk if lq is None else int(lq)
        if q.shape[1] != d or n_q % n_kv or not 0 < L <= Lk:
            raise ValueError("head dim mismatch, n_q not a multiple of n_kv, or bad chunk length")
        q_vec = q
    offset = Lk - L
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    scale = float(scale)
    if rows.size and (rows.min(axis=0) < 0).any():
        raise ValueError("negative row index")
    if rows.size and ((rows[:, 0] >= B).any() or (rows[:, 1] >= n_q).any() or (rows[:, 2] >= L).any()):
        raise ValueError("row index out of range")
    out_o = np.zeros((rows.shape[0], d), dtype=np.float64)
    out_lse = np.zeros(rows.shape[0], dtype=np.float64)
    # Group the requested rows by (b, h); each group shares one K/V head.
    order = np.lexsort((rows[:, 2], rows[:, 1], rows[:, 0]))
    srt = rows[order]
    bounds = np.flatnonzero(np.diff(srt[:, 0] * n_q + srt[:, 1])) + 1
    for grp in np.split(np.arange(srt.shape[0]), bounds):
        if grp.size == 0:
            continue
        b, h = int(srt[grp[0], 0]), int(srt[grp[0], 1])
        kvh = kv_head_of(h, n_q, n_kv)
        kmat = np.asarray(k[b, :, kvh, :], dtype=np.float64)
        vmat = np.asarray(v[b, :, kvh, :], dtype=np.float64)
        idx = srt[grp, 2]
        step = max(1, min(256, _MAX_SCORE_ELEMS // max(Lk, 1)))
        for s0 in range(0, idx.size, step):
            sel = idx[s0:s0 + step]
            dest = order[grp[s0:s0 + step]]
            pos = sel + offset
            lv = int(pos.max()) + 1 if causal else Lk
            if q_vec is None:
                qrows = np.asarray(q[b, sel, h, :], dtype=np.float64)
            else:
                qrows = np.asarray(q_vec[dest], dtype=np.float64)
            o, lse = _rows_block(qrows, kmat[:lv], vmat[:lv], pos, causal, scale)
            out_o[dest] = o
            out_lse[dest] = lse
    return out_o, out_lse


def attention(q, k, v, *, causal: bool = True, scale: float | None = None):
    """Full attention forward.

    q: [B, Lq, n_q, d]; k, v: [B, Lk, n_kv, d] with Lk >= Lq (the query rows
    are the last Lq positions); any real dtype (upcast to fp64).
    Returns (o [B, Lq, n_q, d] float64, lse [B, n_q, Lq] float64).
    """
    B, L, Lk, n_q, n_kv, d = _check_shapes(q, k, v)
    offset = Lk - L
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    scale = float(scale)
    o = np.zeros((B, L, n_q, d), dtype=np.float64)
    lse = np.zeros((B, n_q, L), dtype=np.float64)
    step = max(1, min(256, _MAX_SCORE_ELEMS // max(Lk, 1)))
    for b in range(B):
        for h in range(n_q):
            kvh = kv_head_of(h, n_q, n_kv)
            kmat = np.asarray(k[b, :, kvh, :], dtype=np.float64)
            vmat = np.asarray(v[b, :, kvh, :], dtype=np.float64)
            for i0 in range(0, L, step):
                sel = np.arange(i0, min(L, i0 + step))
                pos = sel + offset
                lv = int(pos[-1]) + 1 if causal else Lk
                qrows = np.asarray(q[b, i0:i0 + sel.size, h, :], dtype=np.float64)
                ob, lb = _rows_block(qrows, kmat[:lv], vmat[:lv], pos, causal, scale)
                o[b, i0:i0 + sel.size, h, :] = ob
                lse[b, h, i0:i0 + sel.size] = lb
    return o, lse
