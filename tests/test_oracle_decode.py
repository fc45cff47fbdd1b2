"""Pins for the paged decode oracle: torch float64 SDPA on the keys and values
gathered with torch indexing (an independent route), page-permutation
invariance, the last rows of full causal attention, and closed forms."""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _gather(kc, table, L, page_size):
    idx = torch.as_tensor(table)[torch.arange(L) // page_size].long()
    return torch.as_tensor(kc)[idx, torch.arange(L) % page_size]          # [L, H_kv, d]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("page_size,n_q,H,H_kv", [(8, 1, 4, 2), (16, 3, 6, 3), (32, 2, 2, 2)])
def test_decode_equals_sdpa_on_gathered_cache(causal, page_size, n_q, H, H_kv):
    lens = [5, 40, 1, 77]
    d = 8
    kc, vc, table = workloads.paged_cache(51, lens, page_size, H_kv, d)
    q = workloads.normal(52, (len(lens), H, n_q, d))
    o, lse = oracle.attention_decode_paged(q, kc, vc, table, lens, 0.35, causal)
    G = H // H_kv
    for b, L in enumerate(lens):
        K = _gather(kc, table[b], L, page_size).double().repeat_interleave(G, dim=1).permute(1, 0, 2)
        V = _gather(vc, table[b], L, page_size).double().repeat_interleave(G, dim=1).permute(1, 0, 2)
        tq = torch.from_numpy(q[b]).double()                               # [H, n_q, d]
        pos = torch.arange(L - n_q, L)
        mask = torch.arange(L)[None, :] <= pos[:, None] if causal else torch.ones(n_q, L, dtype=torch.bool)
        for h in range(H):
            rows = mask.any(1)
            if rows.any():
                ref = torch.nn.functional.scaled_dot_product_attention(
                    tq[h][rows][None], K[h][None], V[h][None], attn_mask=mask[rows][None], scale=0.35)[0]
                np.testing.assert_allclose(o[b, h][rows.numpy()], ref.numpy(), atol=1e-12)
                s = (tq[h] @ K[h].T * 0.35).masked_fill(~mask, float("-inf"))
                np.testing.assert_allclose(lse[b, h][rows.numpy()], torch.logsumexp(s, -1)[rows].numpy(),
                                           atol=1e-12)
            assert np.all(o[b, h][~rows.numpy()] == 0) and np.all(np.isneginf(lse[b, h][~rows.numpy()]))


def test_page_permutation_changes_nothing():
    lens = [30, 17]
    kc, vc, table = workloads.paged_cache(53, lens, 8, 2, 4, spare_pages=5)
    q = workloads.normal(54, (2, 4, 2, 4))
    o1, l1 = oracle.attention_decode_paged(q, kc, vc, table, lens, 0.5, True)
    perm = np.random.default_rng(55).permutation(kc.shape[0])
    inv = np.argsort(perm)
    table2 = np.where(table >= 0, inv[np.maximum(table, 0)], -1)
    o2, l2 = oracle.attention_decode_paged(q, kc[perm], vc[perm], table2, lens, 0.5, True)
    np.testing.assert_allclose(o1, o2, atol=0)
    np.testing.assert_allclose(l1, l2, atol=0)


def test_decode_rows_are_the_last_rows_of_causal_attention():
    L, page_size, d = 23, 8, 4
    kc, vc, table = workloads.paged_cache(56, [L], page_size, 1, d, spare_pages=0)
    K = np.concatenate([kc[p] for p in table[0]], 0)[:L, 0]
    V = np.concatenate([vc[p] for p in table[0]], 0)[:L, 0]
    Q = workloads.normal(57, (L, d))
    full_o, full_l = oracle.attention_forward_head(Q, K, V, 0.6, True)
    n_q = 5
    o, lse = oracle.attention_decode_paged(Q[None, None, L - n_q:], kc, vc, table, [L], 0.6, True)
    np.testing.assert_allclose(o[0, 0], full_o[L - n_q:], atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], full_l[L - n_q:], atol=1e-12)


def test_zero_query_and_empty_sequence():
    lens = [9, 0]
    kc, vc, table = workloads.paged_cache(58, lens, 8, 1, 4)
    q = np.zeros((2, 1, 1, 4))
    o, lse = oracle.attention_decode_paged(q, kc, vc, table, lens, 1.0, False)
    V = np.concatenate([vc[p] for p in table[0, :2]], 0)[:9, 0].astype(np.float64)
    np.testing.assert_allclose(o[0, 0, 0], V.mean(0), atol=1e-14)
    assert abs(lse[0, 0, 0] - np.log(9)) < 1e-14
    assert np.all(o[1] == 0) and np.isneginf(lse[1, 0, 0])
