"""Backward parity: CUDA path (through the C ABI) vs the float64 chain-rule oracle.
O and LSE come from the library's own forward pass."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import GRAD_REL_RMSE, check_status, dev, guarded, lib, rel_rmse, timed_step_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    return lib()


def _run(attn, tq, tk, tv, tdo, causal, scale=None, heads=None):
    B, H, N, d = tq.shape
    scale = 1 / np.sqrt(d) if scale is None else scale
    g = [t.to(dev()) for t in (tq, tk, tv, tdo)]
    o, lse = attn.attn_fwd(g[0], g[1], g[2], causal=causal, softmax_scale=scale)
    dq, cq = guarded((B, H, N, d), tq.dtype, 3.0)
    dk, ck = guarded((B, H, N, d), tq.dtype, 3.0)
    dv, cv = guarded((B, H, N, d), tq.dtype, 3.0)
    attn.attn_bwd(g[0], g[1], g[2], o, g[3], lse, causal=causal, softmax_scale=scale,
                  dq=dq, dk=dk, dv=dv)
    check_status(attn)
    for c in (cq, ck, cv):
        c()
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    out = []
    for b, h in heads:
        ref = oracle.attention_backward_head(*(workloads.as_f64(t[b, h]) for t in (tq, tk, tv, tdo)),
                                             scale, causal)
        out.append([(name, rel_rmse(x[b, h], r)) for name, x, r in
                    (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2]))])
    return dq, dk, dv, out


def _inputs(seed, B, H, N, d, dtype="bf16"):
    return tuple(workloads.round_to(x, dtype) for x in workloads.normal(seed, (B, H, N, d), 4))


def _assert(errs):
    for head in errs:
        for name, e in head:
            assert e <= GRAD_REL_RMSE, (name, e, errs)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 128, 129, 200, 256, 300, 520])
def test_ragged_shapes(attn, N, d, causal):
    *_, errs = _run(attn, *_inputs(200 + N + d, 1, 2, N, d), causal)
    _assert(errs)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_dtypes_multi_head(attn, dtype, causal):
    *_, errs = _run(attn, *_inputs(9, 2, 3, 640, 128, dtype), causal)
    _assert(errs)


def test_larger_scores(attn):
    """Scores with a wider spread (scale 0.25 at d=64) give peaked rows."""
    tq, tk, tv, tdo = _inputs(17, 1, 2, 700, 64)
    *_, errs = _run(attn, tq, tk, tv, tdo, True, scale=0.25)
    _assert(errs)


@pytest.mark.parametrize("w", [workloads.BWD_D128, workloads.BWD_D64], ids=lambda w: w.name)
def test_full_config_sampled_heads(attn, w):
    """The full backward problem (B=2, H=16, N=4096, causal); the oracle checks
    whole heads (every dQ, dK, dV entry of those heads), and two invariants are
    checked on every head: sum_j dV_j = sum_i dO_i and sum_j dK_j = 0."""
    tq, tk, tv, tdo = _inputs(w.seed, w.B, w.H, w.N, w.d)
    dq, dk, dv, errs = _run(attn, tq, tk, tv, tdo, w.causal,
                            heads=[(0, 0), (1, 15), (1, 7)])
    _assert(errs)
    sdv = dv.double().sum(dim=2).cpu().numpy()
    sdo = workloads.as_f64(tdo).sum(axis=2)
    assert np.abs(sdv - sdo).max() <= 2e-2 * np.abs(sdo).max() + 0.5
    sdk = dk.double().sum(dim=2).cpu().numpy()
    assert np.abs(sdk).max() <= 2e-2 * dk.double().abs().sum(dim=2).max().item()


def test_workspace_is_reusable_and_results_repeat(attn):
    """Calling twice with the same workspace gives the same gradients up to
    the ordering of the float32 dQ reductions."""
    tq, tk, tv, tdo = (t.to(dev()) for t in _inputs(5, 1, 4, 512, 128))
    o, lse = attn.attn_fwd(tq, tk, tv, causal=True)
    ws = torch.empty(attn.attn_bwd_workspace_size(1, 4, 512, 128), dtype=torch.uint8,
                     device=dev())
    ws.fill_(0x7F)
    a = attn.attn_bwd(tq, tk, tv, o, tdo, lse, causal=True, workspace=ws)
    b = attn.attn_bwd(tq, tk, tv, o, tdo, lse, causal=True, workspace=ws)
    check_status(attn)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])     # dK, dV: no atomics
    assert (a[0].float() - b[0].float()).abs().max().item() <= 1e-2


def test_timed_config_noncausal_whole_heads(attn):
    """The backward exactly as the benchmark times it: B=2, H=16, N=8192,
    d=128, non-causal -- every CTA walks 64 query tiles and 64 CTAs add into
    each dQ row.  Whole heads (every dQ, dK, dV entry) of three heads against
    the oracle, and on every head sum_j dV_j = sum_i dO_i and sum_j dK_j = 0."""
    w = workloads.LONG_FWD
    assert (w.B, w.H, w.N, w.d, w.causal) == (2, 16, 8192, 128, False)
    tq, tk, tv, tdo = (t.cpu() for t in timed_step_inputs(w.seed, (w.B, w.H, w.N, w.d))[:4])
    dq, dk, dv, errs = _run(attn, tq, tk, tv, tdo, w.causal,
                            heads=[(0, 0), (1, 15), (1, 7)])
    _assert(errs)
    sdv = dv.double().sum(dim=2).cpu().numpy()
    sdo = workloads.as_f64(tdo).sum(axis=2)
    assert np.abs(sdv - sdo).max() <= 2e-2 * np.abs(sdo).max() + 0.5
    sdk = dk.double().sum(dim=2).cpu().numpy()
    assert np.abs(sdk).max() <= 2e-2 * dk.double().abs().sum(dim=2).max().item()
