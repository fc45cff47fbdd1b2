"""Exact softmax attention and its gradient in float64 -- TEST INFRASTRUCTURE.

Sources (page title, then section):

* "FlashAttention-3: Hopper Asynchrony and FP8 Attention", "Symbol Map": the
  score tile is Q K^T, the output is normalised by the softmax sum, and the
  stored log-sum-exp is L = m + log(l) with m the row maximum and l the
  max-subtracted exponential sum.  "Putting It Together", step 7: only O and L
  are written.
* "FlashAttention 3 Hardware Acceleration: Hopper GPU Strategies for
  Long-Context Enterprise Inference Optimization", "Quadratic Attention
  Complexity" and "Intermediate Attention Matrix Storage": standard attention
  forms S = Q K^T, P = softmax(S) row-wise, then O = P V.  This oracle is that
  standard, materialised computation.
* The backward pass is the chain rule applied to that definition (the pages
  say only that S and P are recomputed from L, in "Backward warp
  specialization" of the first page).  With dP = dO V^T the softmax Jacobian
  gives dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik).  The row term is computed here
  directly from P and dP, not through the dO . O shortcut the GPU uses, so the
  two share no derivation.

Readings where the pages are silent:
* ``scale`` multiplies Q K^T before masking and softmax; L is the natural log
  of the sum over the scaled, masked scores.
* The causal mask is lower-triangular with top-left alignment: query i sees
  keys j <= i (queries and keys have the same length N).
"""
from __future__ import annotations

import numpy as np


def _scores(q, k, scale, causal):
    """Scaled scores of one head, with masked entries set to -inf."""
    s = (q @ k.T) * scale
    if causal:
        n_q, n_k = s.shape
        mask = np.arange(n_k)[None, :] > np.arange(n_q)[:, None]
        s = np.where(mask, -np.inf, s)
    return s


def attention_probs(q, k, scale, causal=False):
    """Row-softmax of the scaled, masked scores of one head ([N, d] inputs).

    Returns (P, m, l): P = exp(S - m) / l with m the row max of S and l the
    sum of exp(S - m) over the row.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    s = _scores(q, k, scale, causal)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    return e / l, m[:, 0], l[:, 0]


def attention_forward_head(q, k, v, scale, causal=False):
    """O = softmax(scale * q k^T [+ causal mask]) v and L = m + log(l) for one head."""
    p, m, l = attention_probs(q, k, scale, causal)
    o = p @ np.asarray(v, dtype=np.float64)
    lse = m + np.log(l)
    return o, lse


def attention_forward(q, k, v, scale, causal=False):
    """Batched oracle forward.

    q, k, v: arrays [B, H, N, d] (any float dtype; computed in float64).
    Returns O [B, H, N, d] and LSE [B, H, N], both float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, d = q.shape
    o = np.empty((B, H, N, v.shape[-1]), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = attention_forward_head(q[b, h], k[b, h], v[b, h],
                                                        scale, causal)
    return o, lse


def attention_backward_head(q, k, v, do, scale, causal=False):
    """Gradients (dQ, dK, dV) of sum(O * dO) for one head, by the chain rule.

    S = scale * q k^T, P = softmax(S), O = P v:
      dV = P^T dO
      dP = dO v^T
      dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)      (softmax Jacobian)
      dQ = scale * dS k
      dK = scale * dS^T q
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    p, _, _ = attention_probs(q, k, scale, causal)
    dv = p.T @ do
    dp = do @ v.T
    row = (p * dp).sum(axis=1, keepdims=True)
    ds = p * (dp - row)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


def attention_backward(q, k, v, do, scale, causal=False):
    """Batched oracle backward; inputs [B, H, N, d]; returns float64 dQ, dK, dV."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = attention_backward_head(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
    return dq, dk, dv


def attention_forward_rows(q, k, v, scale, causal, rows):
    """O and L of selected query rows of one head ([N, d] inputs).

    Row i of exact attention depends only on q_i and all of k, v, so the
    selected rows are computed one at a time from the same definition; this is
    how outputs of very large problems are spot-checked.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    o = np.empty((rows.size, v.shape[1]))
    lse = np.empty(rows.size)
    for n, i in enumerate(rows):
        s = (k @ q[i]) * scale
        if causal:
            s[i + 1:] = -np.inf
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        o[n] = (e / l) @ v
        lse[n] = m + np.log(l)
    return o, lse
