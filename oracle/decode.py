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

FP8 cache (the e4m3 key/value cache a decode kernel reads; "FP8 accuracy
controls" for the block scaling and the incoherent transform).  Readings:
a block is one physical page of one key/value head (page_size x d values), with
one float32 descale per block, quantised as in fp8.py; when a sign vector is
given, keys are stored transformed (K M), and the query is transformed by the
same M, since (q M)(K M)^T = q K^T; values are never transformed.  The result
of an FP8 decode is exact attention over the values the cache represents
(code x descale), with the query transformed when the keys were.
"""
from __future__ import annotations

import numpy as np

from .fp8 import e4m3_decode, incoherent_transform, quantize_e4m3_blocks


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


def quantize_paged_cache(cache, signs=None):
    """e4m3 codes [num_pages, page_size, H_kv, d] (uint8) and float32 descales
    [num_pages, H_kv] of a float32 cache, one block per (page, head); keys pass
    the sign vector of the incoherent transform, values pass None."""
    c = np.asarray(cache, dtype=np.float32)
    per_head = np.transpose(c, (0, 2, 1, 3))          # [pages, H_kv, page_size, d]
    codes, descale = quantize_e4m3_blocks(per_head, block_rows=per_head.shape[2], signs=signs)
    return np.ascontiguousarray(np.transpose(codes, (0, 2, 1, 3))), descale[:, :, 0]


def dequantize_paged_cache(codes, descale) -> np.ndarray:
    """float64 values code x descale of a cache quantised per (page, head)."""
    return e4m3_decode(codes) * np.asarray(descale, np.float64)[:, None, :, None]


def attention_decode_paged_fp8(q, k_codes, v_codes, k_descale, v_descale, block_table, seq_lens,
                               scale, causal=False, signs=None):
    """Decode against an e4m3 paged cache: exact attention of q (transformed by
    M when `signs` is given) over the dequantised keys and values."""
    qq = np.asarray(q, dtype=np.float64)
    if signs is not None:
        qq = incoherent_transform(qq, signs)
    return attention_decode_paged(qq, dequantize_paged_cache(k_codes, k_descale),
                                  dequantize_paged_cache(v_codes, v_descale), block_table,
                                  seq_lens, scale, causal)
