"""Grouped-query attention and packed variable-length batches -- TEST INFRASTRUCTURE.

Sources (page title, then section):

* "FlashAttention 3 Hardware Acceleration: Hopper GPU Strategies for
  Long-Context Enterprise Inference Optimization", "Runtime Kernel Selection":
  grouped query attention patterns are supported; "GPU Compatibility and
  Enablement Matrix": variable-length sequence handling.

The pages name both features without defining them, so the plain readings
are used (each is listed in the design notes):

* Grouped-query attention: H query heads share H_kv key/value heads
  (H % H_kv == 0); query head h uses key/value head h // (H / H_kv), i.e. the
  G = H / H_kv consecutive query heads of a group share one key/value head.
  The gradient of a shared key/value head is the sum over its group.
* Variable length: B sequences packed back to back, token-major [total, heads,
  d]; sequence b is tokens cu_seqlens[b] .. cu_seqlens[b+1] - 1.  Attention (and
  the causal mask) acts within each sequence only.  LSE is laid out [H, total].

Each function below applies the exact single-head definitions of
``attention.py`` to every (sequence, head) pair: no blocking or fusion.
"""
from __future__ import annotations

import numpy as np

from .attention import attention_backward_head, attention_forward_head


def _group(H: int, H_kv: int) -> int:
    if H_kv < 1 or H % H_kv:
        raise ValueError("H_kv must divide H")
    return H // H_kv


def attention_forward_gqa(q, k, v, scale, causal=False):
    """q [B, H, N, d]; k, v [B, H_kv, N, d] -> O [B, H, N, d], LSE [B, H, N] (float64)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, d = q.shape
    G = _group(H, k.shape[1])
    o = np.empty((B, H, N, v.shape[-1]))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = attention_forward_head(q[b, h], k[b, h // G], v[b, h // G],
                                                        scale, causal)
    return o, lse


def attention_backward_gqa(q, k, v, do, scale, causal=False):
    """Gradients of sum(O * dO): dQ [B, H, N, d]; dK, dV [B, H_kv, N, d] summed over each group."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, H, N, d = q.shape
    G = _group(H, k.shape[1])
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            g_q, g_k, g_v = attention_backward_head(q[b, h], k[b, h // G], v[b, h // G], do[b, h],
                                                    scale, causal)
            dq[b, h] = g_q
            dk[b, h // G] += g_k
            dv[b, h // G] += g_v
    return dq, dk, dv


def _sequences(cu_seqlens):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    if cu.ndim != 1 or cu.size < 2 or cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0 and be non-decreasing")
    return [(int(cu[i]), int(cu[i + 1])) for i in range(cu.size - 1)]


def attention_forward_varlen(q, k, v, cu_seqlens, scale, causal=False):
    """Packed batch: q [total, H, d]; k, v [total, H_kv, d] -> O [total, H, d], LSE [H, total]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    total, H, d = q.shape
    G = _group(H, k.shape[1])
    o = np.zeros((total, H, v.shape[-1]))
    lse = np.zeros((H, total))
    for s, e in _sequences(cu_seqlens):
        if e == s:
            continue
        for h in range(H):
            o[s:e, h], lse[h, s:e] = attention_forward_head(q[s:e, h], k[s:e, h // G],
                                                            v[s:e, h // G], scale, causal)
    return o, lse


def attention_backward_varlen(q, k, v, do, cu_seqlens, scale, causal=False):
    """Packed batch gradients: dQ [total, H, d]; dK, dV [total, H_kv, d]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    total, H, d = q.shape
    G = _group(H, k.shape[1])
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for s, e in _sequences(cu_seqlens):
        if e == s:
            continue
        for h in range(H):
            g_q, g_k, g_v = attention_backward_head(q[s:e, h], k[s:e, h // G], v[s:e, h // G],
                                                    do[s:e, h], scale, causal)
            dq[s:e, h] = g_q
            dk[s:e, h // G] += g_k
            dv[s:e, h // G] += g_v
    return dq, dk, dv
