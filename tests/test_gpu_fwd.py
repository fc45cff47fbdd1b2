"""Forward parity: CUDA path (through the C ABI) vs the float64 CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import (assert_fwd_close, check_status, dev, guarded, lib, FWD_MAX_ABS,
                      FWD_RMSE, LSE_ABS)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    return lib()


def _inputs(seed, B, H, N, d, dtype="bf16", mult=1.0):
    q, k, v = workloads.normal(seed, (B, H, N, d), 3)
    q = q * np.float32(mult)
    k = k * np.float32(mult)
    return tuple(workloads.round_to(x, dtype) for x in (q, k, v))


def _run(attn, tq, tk, tv, causal, scale=None):
    B, H, N, d = tq.shape
    scale = 1 / np.sqrt(d) if scale is None else scale
    o, co = guarded((B, H, N, d), tq.dtype, -7.0)
    lse, cl = guarded((B, H, N), torch.float32, -7.0)
    attn.attn_fwd(tq.to(dev()), tk.to(dev()), tv.to(dev()), causal=causal, softmax_scale=scale,
                  o=o, lse=lse)
    check_status(attn)
    co()
    cl()
    ref_o, ref_l = oracle.attention_forward(*(workloads.as_f64(t) for t in (tq, tk, tv)),
                                            scale, causal)
    return o, lse, ref_o, ref_l


def test_tiny_config(attn):
    w = workloads.TINY_FWD
    tq, tk, tv = _inputs(w.seed, w.B, w.H, w.N, w.d)
    assert_fwd_close(*_run(attn, tq, tk, tv, w.causal))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 256, 300, 513])
def test_ragged_shapes(attn, N, d, causal):
    tq, tk, tv = _inputs(100 + N + d, 1, 2, N, d)
    assert_fwd_close(*_run(attn, tq, tk, tv, causal))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_dtypes_multi_head(attn, dtype, causal):
    tq, tk, tv = _inputs(7, 2, 3, 700, 128, dtype)
    assert_fwd_close(*_run(attn, tq, tk, tv, causal))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_large_scores_force_rescaling(attn, d, causal):
    """Scores with a standard deviation near 9 make the running max jump
    often, exercising the output rescale; keys grow along the sequence so
    late tiles hold the largest scores."""
    B, H, N = 1, 2, 1024
    q, k, v = workloads.normal(21, (B, H, N, d), 3)
    ramp = (1.0 + 3.0 * np.arange(N, dtype=np.float32) / N)[None, None, :, None]
    tq, tk, tv = (workloads.round_to(x, "bf16") for x in (3 * q, 3 * k * ramp, v))
    assert_fwd_close(*_run(attn, tq, tk, tv, causal))


def test_dominant_key_in_last_tile(attn):
    """One key (in the last, ragged tile) outscores all others by a wide margin:
    every output row must equal that key's value row."""
    B, H, N, d = 1, 1, 333, 64
    q, k, v = workloads.normal(31, (B, H, N, d), 3)
    q = np.abs(q)
    k = np.abs(k) * 0.01
    k[0, 0, 320] = 4.0
    tq, tk, tv = (workloads.round_to(x, "bf16") for x in (q, k, v))
    o, lse, ref_o, ref_l = _run(attn, tq, tk, tv, False)
    assert_fwd_close(o, lse, ref_o, ref_l)
    np.testing.assert_allclose(o.float().cpu().numpy()[0, 0],
                               np.broadcast_to(workloads.as_f64(tv)[0, 0, 320], (N, d)),
                               atol=2e-2)


def test_zero_queries_average_values(attn):
    B, H, N, d = 1, 2, 300, 128
    _, tk, tv = _inputs(41, B, H, N, d)
    tq = torch.zeros_like(tk)
    o, lse, ref_o, ref_l = _run(attn, tq, tk, tv, True)
    assert_fwd_close(o, lse, ref_o, ref_l)
    np.testing.assert_allclose(lse.cpu().numpy()[0, 0], np.log(np.arange(1, N + 1)), atol=1e-3)


@pytest.mark.parametrize("causal", [False, True])
def test_mid_config(attn, causal):
    """B=4, H=16, N=2048, d=128 against the full oracle."""
    w = workloads.MID_FWD_CAUSAL if causal else workloads.MID_FWD
    tq, tk, tv = _inputs(w.seed, w.B, w.H, w.N, w.d)
    assert_fwd_close(*_run(attn, tq, tk, tv, causal))


@pytest.mark.parametrize("w", [workloads.LONG_FWD, workloads.LONG_FWD_CAUSAL,
                               workloads.LONG_FWD_D64, workloads.LONG_FWD_D256],
                         ids=lambda w: w.name)
def test_long_config_sampled_rows(attn, w):
    """Full-size long-context problems (the timed shape and the head-dim
    sweep); the oracle checks sampled rows of sampled heads, one at a time."""
    gen = torch.Generator(device=dev()).manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    q, k, v = (torch.randn(shape, generator=gen, device=dev(), dtype=torch.float32)
               .to(torch.bfloat16) for _ in range(3))
    o, lse = attn.attn_fwd(q, k, v, causal=w.causal, softmax_scale=w.scale)
    check_status(attn)
    rng = np.random.default_rng(w.seed)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 129, w.N - 1],
                                     rng.integers(0, w.N, 26)]))
    for (b, h) in [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 3)]:
        qh, kh, vh = (t[b, h].double().cpu().numpy() for t in (q, k, v))
        ref_o, ref_l = oracle.attention_forward_rows(qh, kh, vh, w.scale, w.causal, rows)
        got_o = o[b, h, rows].double().cpu().numpy()
        got_l = lse[b, h, rows].double().cpu().numpy()
        diff = got_o - ref_o
        assert np.abs(diff).max() <= FWD_MAX_ABS
        assert np.sqrt(np.mean(diff ** 2)) <= FWD_RMSE
        assert np.abs(got_l - ref_l).max() <= LSE_ABS


@pytest.mark.parametrize("sched", [1, 2, 3], ids=["one_tile", "eager", "one_tile_eager"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 300, 1000])
def test_schedule_variants(attn, sched, d, causal, N):
    """The measurement variants of the forward (one query tile per CTA, eager
    rescaling) compute the same attention: parity with the oracle, on scores
    spread wide enough that the running max moves often."""
    q, k, v = workloads.normal(500 + N + d, (1, 2, N, d), 3)
    tq, tk, tv = (workloads.round_to(x, "bf16") for x in (2 * q, 2 * k, v))
    scale = 1 / np.sqrt(d)
    o, lse = attn.attn_fwd_schedule(tq.to(dev()), tk.to(dev()), tv.to(dev()), sched,
                                    causal=causal, softmax_scale=scale)
    check_status(attn)
    ref_o, ref_l = oracle.attention_forward(*(workloads.as_f64(t) for t in (tq, tk, tv)),
                                            scale, causal)
    assert_fwd_close(o, lse, ref_o, ref_l)


@pytest.mark.parametrize("sched", [1, 2], ids=["one_tile", "eager"])
@pytest.mark.parametrize("causal", [False, True])
def test_schedule_variants_timed_shape(attn, sched, causal):
    """The variants at the shape the benchmark times them (B=2, H=16, N=8192,
    d=128): sampled rows against the oracle, and whole tensors against the
    default schedule's output."""
    w = workloads.LONG_FWD_CAUSAL if causal else workloads.LONG_FWD
    gen = torch.Generator(device=dev()).manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    q, k, v = (torch.randn(shape, generator=gen, device=dev(), dtype=torch.float32)
               .to(torch.bfloat16) for _ in range(3))
    o, lse = attn.attn_fwd_schedule(q, k, v, sched, causal=causal, softmax_scale=w.scale)
    o0, lse0 = attn.attn_fwd(q, k, v, causal=causal, softmax_scale=w.scale)
    check_status(attn)
    # Eager rescaling rounds P to bfloat16 against another exponent reference
    # (not a power of two apart), so outputs differ by P rounding: whole tensors
    # agree within the forward tolerances.
    diff = (o.float() - o0.float())
    assert diff.abs().max().item() <= FWD_MAX_ABS
    assert diff.pow(2).mean().sqrt().item() <= FWD_RMSE
    assert (lse - lse0).abs().max().item() <= 1e-4
    if sched == 1:       # the same per-row arithmetic in the same order: same bits
        assert torch.equal(o, o0) and torch.equal(lse, lse0)
    rows = np.array([0, 1, 127, 128, 4097, w.N - 1])
    for (b, h) in [(0, 0), (1, 15)]:
        qh, kh, vh = (t[b, h].double().cpu().numpy() for t in (q, k, v))
        ref_o, ref_l = oracle.attention_forward_rows(qh, kh, vh, w.scale, causal, rows)
        diff = o[b, h, rows].double().cpu().numpy() - ref_o
        assert np.abs(diff).max() <= FWD_MAX_ABS and np.sqrt(np.mean(diff ** 2)) <= FWD_RMSE
        assert np.abs(lse[b, h, rows].double().cpu().numpy() - ref_l).max() <= LSE_ABS
