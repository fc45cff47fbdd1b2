"""Decode attention over a paged key/value cache -- TEST INFRASTRUCTURE.

Sources (page title, then section): "FlashAttention-3: Hopper Asynchrony and
FP8 Attention", "Where It Breaks" (a decode-focused kernel is open work) and
"Symbol Map" (exact attention, L = m + log l); "FlashAttention 3 Hardware
Acceleration: Hopper GPU Strategies for Long-Context Enterprise Inference
Optimization", "Memory Fragmentation" (the cache held in fixed-size blocks).

Readings (listed in the design notes): the cache is [num_pages, page_size,
H_kv, d]; logical page p of sequence b is physical page block_table[b][p]; the
n_q query tokens of sequence b are its last n_q positions (their keys and values
are already in the cache), so with the causal mask query t sees keys
0 .. seq_lens[b] - n_q + t; grouped query heads as in varlen.py.  A row that
sees no key gets O = 0 and L = -inf.

The function gathers each sequence's keys and values page by page and applies
the plain attention definition row by row.
"""
from __future__ import annotations

import numpy as np


def attention_decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale, causal=False):
    """q [B, H, n_q, d]; caches [num_pages, page_size, H_kv, d] -> O [B, H, n_q, d],
    LSE [B, H, n_q] (float64)."""
    q = np.asarray(q, dtype=np.float64)
    kc = np.asarray(k_cache, dtype=np.float64)
    vc = np.asarray(v_cache, dtype=np.float64)
    table = np.asarray(block_table)
    lens = np.asarray(seq_lens)
    B, H, n_q, d = q.shape
    page_size, H_kv = kc.shape[1], kc.shape[2]
    if H % H_kv:
        raise ValueError("H_kv must divide H")
    G = H // H_kv
    o = np.zeros((B, H, n_q, vc.shape[-1]))
    lse = np.full((B, H, n_q), -np.inf)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        npages = -(-L // page_size)
        K = np.concatenate([kc[table[b, p]] for p in range(npages)], axis=0)[:L]   # [L, H_kv, d]
        V = np.concatenate([vc[table[b, p]] for p in range(npages)], axis=0)[:L]
        for h in range(H):
            for t in range(n_q):
                visible = min(L, L - n_q + t + 1) if causal else L
                if visible <= 0:
                    continue
                s = (K[:visible, h // G] @ q[b, h, t]) * scale
                m = s.max()
                e = np.exp(s - m)
                o[b, h, t] = (e / e.sum()) @ V[:visible, h // G]
                lse[b, h, t] = m + np.log(e.sum())
    return o, lse
