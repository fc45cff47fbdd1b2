"""Backward parity for grouped-query attention and packed variable-length
batches: CUDA path (through the C ABI) vs the float64 chain-rule oracle.  O and
LSE come from the library's own forward pass."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import GRAD_REL_RMSE, check_status, dev, guarded, lib, rel_rmse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    return lib()


def _r(seed, shape, count, dtype="bf16"):
    xs = workloads.normal(seed, shape, count)
    xs = xs if count > 1 else [xs]
    return [workloads.round_to(x, dtype) for x in xs]


def _assert_rel(pairs):
    errs = {name: rel_rmse(g, r) for name, g, r in pairs}
    for name, e in errs.items():
        assert e <= GRAD_REL_RMSE, errs


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(4, 2), (6, 1), (3, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_backward(attn, d, H, H_kv, causal):
    B, N = 2, 300
    tq, tdo = _r(90 + d + H_kv, (B, H, N, d), 2)
    tk, tv = _r(91 + d + H_kv, (B, H_kv, N, d), 2)
    scale = 1 / np.sqrt(d)
    g = [t.to(dev()) for t in (tq, tk, tv, tdo)]
    o, lse = attn.attn_fwd_gqa(g[0], g[1], g[2], causal=causal, softmax_scale=scale)
    dq, cq = guarded((B, H, N, d), tq.dtype, 3.0)
    dk, ck = guarded((B, H_kv, N, d), tq.dtype, 3.0)
    dv, cv = guarded((B, H_kv, N, d), tq.dtype, 3.0)
    attn.attn_bwd_gqa(g[0], g[1], g[2], o, g[3], lse, causal=causal, softmax_scale=scale,
                      dq=dq, dk=dk, dv=dv)
    check_status(attn)
    for c in (cq, ck, cv):
        c()
    rq, rk, rv = oracle.attention_backward_gqa(*(workloads.as_f64(t) for t in (tq, tk, tv, tdo)),
                                               scale, causal)
    _assert_rel([("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)])


def _cu(name):
    if name == "mixed":       # empty, length 1, tile-ragged and multi-tile sequences
        return np.array([0, 0, 1, 128, 257, 300, 815], dtype=np.int32)
    if name == "random":
        cu, _ = workloads.varlen_lengths(62, 5, 600)
        return cu
    raise ValueError(name)


def _varlen_bwd(attn, cu, H, H_kv, d, causal, dtype="bf16", seed=95):
    total = int(cu[-1])
    max_len = max(int(np.max(np.diff(cu))), 1)
    tq, tdo = _r(seed, (total, H, d), 2, dtype)
    tk, tv = _r(seed + 1, (total, H_kv, d), 2, dtype)
    scale = 1 / np.sqrt(d)
    g = [t.to(dev()) for t in (tq, tk, tv, tdo)]
    cu_d = torch.from_numpy(cu).to(dev())
    o, lse = attn.attn_fwd_varlen(g[0], g[1], g[2], cu_d, max_len, causal=causal,
                                  softmax_scale=scale)
    dq, cq = guarded((total, H, d), tq.dtype, 3.0)
    dk, ck = guarded((total, H_kv, d), tq.dtype, 3.0)
    dv, cv = guarded((total, H_kv, d), tq.dtype, 3.0)
    attn.attn_bwd_varlen(g[0], g[1], g[2], o, g[3], lse, cu_d, max_len, causal=causal,
                         softmax_scale=scale, dq=dq, dk=dk, dv=dv)
    check_status(attn)
    for c in (cq, ck, cv):
        c()
    rq, rk, rv = oracle.attention_backward_varlen(*(workloads.as_f64(t) for t in (tq, tk, tv, tdo)),
                                                  cu, scale, causal)
    _assert_rel([("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)])


@pytest.mark.parametrize("case", ["mixed", "random"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward(attn, case, d, causal):
    _varlen_bwd(attn, _cu(case), 4, 2, d, causal)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_varlen_backward_dtypes_mqa(attn, dtype):
    _varlen_bwd(attn, _cu("mixed"), 3, 1, 128, True, dtype)


def test_varlen_backward_single_sequence_matches_fixed_length(attn):
    """One packed sequence is the fixed-length problem with B = 1: both paths
    give the same gradients to float32 rounding of the dQ sums."""
    N, H, d = 384, 2, 128
    tq, tk, tv, tdo = _r(97, (N, H, d), 4)
    scale = 1 / np.sqrt(d)
    g = [t.to(dev()) for t in (tq, tk, tv, tdo)]
    cu_d = torch.tensor([0, N], dtype=torch.int32, device=dev())
    o, lse = attn.attn_fwd_varlen(g[0], g[1], g[2], cu_d, N, causal=True, softmax_scale=scale)
    pq, pk, pv = attn.attn_bwd_varlen(g[0], g[1], g[2], o, g[3], lse, cu_d, N, causal=True,
                                      softmax_scale=scale)
    bhnd = [t.permute(1, 0, 2).unsqueeze(0).contiguous() for t in g]
    o2, lse2 = attn.attn_fwd(bhnd[0], bhnd[1], bhnd[2], causal=True, softmax_scale=scale)
    fq, fk, fv = attn.attn_bwd(bhnd[0], bhnd[1], bhnd[2], o2, bhnd[3], lse2, causal=True,
                               softmax_scale=scale)
    check_status(attn)
    for a, b in ((pq, fq), (pk, fk), (pv, fv)):
        b = b[0].permute(1, 0, 2)
        assert torch.allclose(a.float(), b.float(), atol=2e-2, rtol=2e-2)
    assert torch.equal(o, o2[0].permute(1, 0, 2))
    assert torch.equal(lse, lse2[0])
