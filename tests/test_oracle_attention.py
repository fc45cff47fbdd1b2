"""Pins for the attention oracle: every check here comes from something other
than the oracle itself -- hand-derived values, closed forms, invariants of the
softmax definition, independent library routines (torch SDPA and autograd in
float64) and central finite differences."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case_idx", [0, 1, 2])
def test_hand_cases_forward(golden_dir, case_idx):
    case = _load(golden_dir, "hand_attention.json")["cases"][case_idx]
    o, lse = oracle.attention_forward_head(np.array(case["q"]), np.array(case["k"]),
                                           np.array(case["v"]), case["scale"], case["causal"])
    np.testing.assert_allclose(o, np.array(case["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(case["lse"]), rtol=0, atol=1e-12)


def test_hand_case_backward(golden_dir):
    case = _load(golden_dir, "hand_attention.json")["cases"][0]
    dq, dk, dv = oracle.attention_backward_head(np.array(case["q"]), np.array(case["k"]),
                                                np.array(case["v"]), np.array(case["do"]),
                                                case["scale"], case["causal"])
    np.testing.assert_allclose(dq, case["dq"], atol=1e-12)
    np.testing.assert_allclose(dk, case["dk"], atol=1e-12)
    np.testing.assert_allclose(dv, case["dv"], atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_visible_values(causal):
    rng = np.random.default_rng(0)
    N, d = 37, 8
    q = np.zeros((N, d))
    k = rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    o, lse = oracle.attention_forward_head(q, k, v, 0.3, causal)
    for i in range(N):
        visible = i + 1 if causal else N
        np.testing.assert_allclose(o[i], v[:visible].mean(axis=0), atol=1e-12)
        assert abs(lse[i] - math.log(visible)) < 1e-12


def test_causal_row0_is_v0():
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal((19, 16)) for _ in range(3))
    o, lse = oracle.attention_forward_head(q, k, v, 0.25, True)
    np.testing.assert_allclose(o[0], v[0], atol=1e-13)
    assert abs(lse[0] - 0.25 * q[0] @ k[0]) < 1e-12


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(2)
    N, d = 24, 16
    q = rng.standard_normal((N, d))
    k = rng.standard_normal((N, d)) * 0.1
    v = rng.standard_normal((N, d))
    jstar = 7
    # make key jstar score 60 above any other for every query with q . k positive
    k[jstar] = 0.0
    q_all = q / np.linalg.norm(q, axis=1, keepdims=True)
    # single query row: k_jstar aligned with it
    k[jstar] = 60.0 * q_all[3] / 1.0
    o, lse = oracle.attention_forward_head(q[3:4], k, v, 1.0 / np.linalg.norm(q[3]), False)
    np.testing.assert_allclose(o[0], v[jstar], atol=1e-15 + 1e-20)
    s = (q[3] @ k.T) / np.linalg.norm(q[3])
    assert abs(lse[0] - s[jstar]) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one_and_lse_bounds(causal):
    rng = np.random.default_rng(3)
    N, d = 50, 32
    q, k = rng.standard_normal((N, d)) * 2, rng.standard_normal((N, d)) * 2
    p, m, l = oracle.attention_probs(q, k, 0.2, causal)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-13)
    assert np.all(p >= 0)
    if causal:
        assert np.all(np.triu(p, 1) == 0)
    _, lse = oracle.attention_forward_head(q, k, rng.standard_normal((N, d)), 0.2, causal)
    visible = np.arange(1, N + 1) if causal else np.full(N, N)
    assert np.all(lse >= m - 1e-12)
    assert np.all(lse <= m + np.log(visible) + 1e-12)


def test_permuting_keys_and_values_together_changes_nothing():
    rng = np.random.default_rng(4)
    N, d = 41, 16
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    perm = rng.permutation(N)
    o1, l1 = oracle.attention_forward_head(q, k, v, 0.25, False)
    o2, l2 = oracle.attention_forward_head(q, k[perm], v[perm], 0.25, False)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(causal):
    """Independent library routine: torch's math SDPA in float64 on the CPU."""
    B, H, N, d = 2, 3, 45, 16
    q, k, v = workloads.normal(11, (B, H, N, d), 3)
    scale = 0.37
    o, lse = oracle.attention_forward(q, k, v, scale, causal)
    tq, tk, tv = (torch.from_numpy(x).double() for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                           scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)
    s = torch.einsum("bhqd,bhkd->bhqk", tq, tk) * scale
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(causal):
    B, H, N, d = 1, 2, 33, 8
    q, k, v, do = workloads.normal(12, (B, H, N, d), 4)
    scale = 0.41
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.from_numpy(x).double().requires_grad_() for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                           scale=scale)
    out.backward(torch.from_numpy(do).double())
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_central_finite_differences(causal):
    rng = np.random.default_rng(5)
    N, d = 6, 3
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    scale = 0.8
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, scale, causal)

    def loss(q_, k_, v_):
        o, _ = oracle.attention_forward_head(q_, k_, v_, scale, causal)
        return float((o * do).sum())

    h = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros((N, d))
        for i in range(N):
            for j in range(d):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][i, j] += h
                args_m[which][i, j] -= h
                num[i, j] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    rng = np.random.default_rng(6)
    N, d = 29, 8
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, 0.5, causal)
    # rows of P sum to one  =>  sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)
    # rows of dS sum to zero  =>  sum_j dK_j = 0
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    if causal:
        # causal row 0 only sees key 0, so its query gradient is zero
        np.testing.assert_allclose(dq[0], 0.0, atol=1e-13)


def test_row_term_equals_do_dot_o():
    """The GPU uses D_i = dO_i . O_i for the softmax-Jacobian row term; the
    oracle computes sum_k P_ik dP_ik.  They agree because sum_k P_ik dP_ik =
    sum_k P_ik (dO_i . V_k) = dO_i . (P V)_i."""
    rng = np.random.default_rng(7)
    N, d = 21, 8
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    p, _, _ = oracle.attention_probs(q, k, 0.3, True)
    o, _ = oracle.attention_forward_head(q, k, v, 0.3, True)
    np.testing.assert_allclose((p * (do @ v.T)).sum(axis=1), (do * o).sum(axis=1), atol=1e-12)


def test_planted_mistakes_are_caught():
    """Sensitivity check: plausible slips in the oracle formulas must fail a pin."""
    rng = np.random.default_rng(8)
    N, d = 5, 3
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=0.6)
    out.backward(torch.from_numpy(do))
    p, _, _ = oracle.attention_probs(q, k, 0.6, True)
    dp = do @ v.T
    # a dropped softmax-Jacobian row term
    bad_ds = p * dp
    assert not np.allclose(0.6 * bad_ds @ k, tq.grad.numpy(), atol=1e-6)
    # a missing scale on dK
    row = (p * dp).sum(1, keepdims=True)
    assert not np.allclose((p * (dp - row)).T @ q, tk.grad.numpy(), atol=1e-6)
    # a transposed P in dV
    assert not np.allclose(p @ do, tv.grad.numpy(), atol=1e-6)


@pytest.mark.parametrize("causal", [False, True])
def test_row_sampler_matches_full_head(causal):
    """The row-by-row oracle used for spot checks equals the batched one and
    torch SDPA on every row."""
    rng = np.random.default_rng(9)
    N, d = 70, 16
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    rows = np.array([0, 1, 33, 69])
    o_r, l_r = oracle.attention_forward_rows(q, k, v, 0.3, causal, rows)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(x)[None, None] for x in (q, k, v)), is_causal=causal, scale=0.3)[0, 0]
    np.testing.assert_allclose(o_r, ref.numpy()[rows], atol=1e-12)
    _, l_full = oracle.attention_forward_head(q, k, v, 0.3, causal)
    np.testing.assert_allclose(l_r, l_full[rows], atol=1e-12)
