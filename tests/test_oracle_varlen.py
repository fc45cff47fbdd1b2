"""Pins for the grouped-query and packed-batch oracle.  Each check uses a route
that shares nothing with the oracle's loops: torch's float64 SDPA with the
key/value heads repeated (and its autograd, which sums a shared head's
gradient over its group), one SDPA call over the whole packed batch with a
block-diagonal mask, and closed forms."""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _sdpa64(q, k, v, causal, scale, mask=None):
    return torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=mask, is_causal=causal if mask is None else False, scale=scale)


@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 2), (6, 3), (4, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_forward_equals_sdpa_with_repeated_heads(H, H_kv, causal):
    B, N, d = 2, 19, 8
    q = workloads.normal(21, (B, H, N, d))
    k, v = workloads.normal(22, (B, H_kv, N, d), 2)
    o, lse = oracle.attention_forward_gqa(q, k, v, 0.4, causal)
    G = H // H_kv
    tq = torch.from_numpy(q).double()
    tk = torch.from_numpy(k).double().repeat_interleave(G, dim=1)
    tv = torch.from_numpy(v).double().repeat_interleave(G, dim=1)
    np.testing.assert_allclose(o, _sdpa64(tq, tk, tv, causal, 0.4).numpy(), atol=1e-12)
    s = torch.einsum("bhqd,bhkd->bhqk", tq, tk) * 0.4
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), atol=1e-12)


@pytest.mark.parametrize("H,H_kv", [(4, 2), (3, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_backward_equals_autograd_through_repeated_heads(H, H_kv, causal):
    B, N, d = 1, 13, 4
    q, do = workloads.normal(23, (B, H, N, d), 2)
    k, v = workloads.normal(24, (B, H_kv, N, d), 2)
    dq, dk, dv = oracle.attention_backward_gqa(q, k, v, do, 0.7, causal)
    G = H // H_kv
    tq, tk, tv = (torch.from_numpy(x).double().requires_grad_() for x in (q, k, v))
    out = _sdpa64(tq, tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1), causal, 0.7)
    out.backward(torch.from_numpy(do).double())
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


def test_gqa_head_mapping_is_consecutive_groups():
    """Query heads 0..G-1 share key/value head 0 (h // G), not h % H_kv: a
    planted interleaved mapping disagrees with the oracle."""
    B, H, H_kv, N, d = 1, 4, 2, 7, 4
    q = workloads.normal(25, (B, H, N, d))
    k, v = workloads.normal(26, (B, H_kv, N, d), 2)
    o, _ = oracle.attention_forward_gqa(q, k, v, 0.5)
    tq = torch.from_numpy(q).double()
    interleaved = _sdpa64(tq, torch.from_numpy(k).double().repeat(1, 2, 1, 1),
                          torch.from_numpy(v).double().repeat(1, 2, 1, 1), False, 0.5)
    assert not np.allclose(o, interleaved.numpy(), atol=1e-6)


def _block_mask(cu, causal):
    """Boolean [total, total] mask: True where query i may see key j."""
    total = int(cu[-1])
    seq = np.zeros(total, dtype=np.int64)
    for b in range(len(cu) - 1):
        seq[cu[b]:cu[b + 1]] = b
    same = seq[:, None] == seq[None, :]
    if causal:
        same &= np.arange(total)[None, :] <= np.arange(total)[:, None]
    return torch.from_numpy(same)


def _packed_cases():
    return [np.array([0, 5, 5, 17, 18, 40], dtype=np.int32),   # with an empty and a length-1 sequence
            np.array([0, 33], dtype=np.int32)]


@pytest.mark.parametrize("cu", _packed_cases())
@pytest.mark.parametrize("H,H_kv", [(2, 2), (4, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_forward_equals_block_diagonal_sdpa(cu, H, H_kv, causal):
    total, d = int(cu[-1]), 8
    q = workloads.normal(27, (total, H, d))
    k, v = workloads.normal(28, (total, H_kv, d), 2)
    o, lse = oracle.attention_forward_varlen(q, k, v, cu, 0.3, causal)
    G = H // H_kv
    # heads first: [1, H, total, d]
    tq = torch.from_numpy(q).double().permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).double().permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    tv = torch.from_numpy(v).double().permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    mask = _block_mask(cu, causal)
    ref = _sdpa64(tq, tk, tv, False, 0.3, mask)[0].permute(1, 0, 2)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)
    s = torch.einsum("hqd,hkd->hqk", tq[0], tk[0]) * 0.3
    s = s.masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_equals_autograd_with_block_diagonal_mask(causal):
    cu = np.array([0, 4, 4, 11, 12], dtype=np.int32)
    total, H, H_kv, d = int(cu[-1]), 4, 2, 4
    q, do = workloads.normal(29, (total, H, d), 2)
    k, v = workloads.normal(30, (total, H_kv, d), 2)
    dq, dk, dv = oracle.attention_backward_varlen(q, k, v, do, cu, 0.6, causal)
    G = H // H_kv
    tq, tk, tv = (torch.from_numpy(x).double().requires_grad_() for x in (q, k, v))
    hq = tq.permute(1, 0, 2)[None]
    hk = tk.permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    hv = tv.permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    out = _sdpa64(hq, hk, hv, False, 0.6, _block_mask(cu, causal))[0].permute(1, 0, 2)
    out.backward(torch.from_numpy(do).double())
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


def test_varlen_closed_forms():
    """A length-1 sequence outputs its own value row with LSE = its one scaled
    score; with Q = 0 every output row is the mean of its sequence's values."""
    cu = np.array([0, 1, 4], dtype=np.int32)
    rng = np.random.default_rng(31)
    q = rng.standard_normal((4, 1, 3))
    k = rng.standard_normal((4, 1, 3))
    v = rng.standard_normal((4, 1, 3))
    o, lse = oracle.attention_forward_varlen(q, k, v, cu, 0.9)
    np.testing.assert_allclose(o[0, 0], v[0, 0], atol=1e-14)
    assert abs(lse[0, 0] - 0.9 * q[0, 0] @ k[0, 0]) < 1e-13
    o0, lse0 = oracle.attention_forward_varlen(np.zeros_like(q), k, v, cu, 0.9)
    np.testing.assert_allclose(o0[1:, 0], np.repeat(v[1:, 0].mean(0)[None], 3, 0), atol=1e-14)
    np.testing.assert_allclose(lse0[0, 1:], np.log(3.0), atol=1e-14)


def test_varlen_rejects_bad_offsets():
    q = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle.attention_forward_varlen(q, q, q, np.array([0, 3, 2, 4]), 1.0)
    with pytest.raises(ValueError):
        oracle.attention_forward_varlen(q, q, q, np.array([1, 4]), 1.0)
