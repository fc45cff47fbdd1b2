"""FP8 path parity: the e4m3 pre-pass against the oracle quantiser, and the FP8
forward against exact float64 attention (on the original float32 inputs and on
the dequantised inputs)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import FP8_RMSE, check_status, dev, lib, timed_step_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    return lib()


def _quant(attn, xs, signs=None, per_tensor=False):
    g = [torch.from_numpy(x).to(dev()) for x in xs]
    s = None if signs is None else torch.from_numpy(signs).to(dev())
    codes, desc = attn.attn_fp8_quantize(*g, hadamard_signs=s, per_tensor=per_tensor)
    check_status(attn)
    return [c.cpu().numpy() for c in codes], [d.cpu().numpy() for d in desc]


@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (2, 3, 256, 128), (1, 1, 1, 128)])
@pytest.mark.parametrize("per_tensor", [False, True])
def test_quantiser_bit_exact_without_hadamard(attn, shape, per_tensor):
    xs = workloads.normal_with_outliers(11, shape, 3)
    codes, desc = _quant(attn, xs, per_tensor=per_tensor)
    for x, c, d in zip(xs, codes, desc):
        rc, rd = oracle.quantize_e4m3_blocks(x, per_tensor=per_tensor)
        np.testing.assert_array_equal(d, rd)
        np.testing.assert_array_equal(c, rc)


def test_quantiser_with_hadamard(attn):
    """The GPU transform runs in float32, the oracle's in float64: descales agree
    to float32 rounding and codes differ by at most one e4m3 step, rarely."""
    shape = (1, 4, 700, 128)
    xs = workloads.normal_with_outliers(12, shape, 3)
    signs = workloads.random_signs(5, 128)
    codes, desc = _quant(attn, xs, signs)
    for which, (x, c, d) in enumerate(zip(xs, codes, desc)):
        rc, rd = oracle.quantize_e4m3_blocks(x, signs=signs if which < 2 else None)
        np.testing.assert_allclose(d, rd, rtol=2e-6)
        if which == 2:
            np.testing.assert_array_equal(c, rc)          # V is not transformed
            continue
        got = oracle.e4m3_decode(c)
        ref = oracle.e4m3_decode(rc)
        diff = np.abs(got - ref)
        step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -6))) - 3)
        assert np.all(diff <= step * 1.0001)
        assert np.mean(c != rc) < 1e-3


def _fp8_forward(attn, q, k, v, signs, per_tensor, causal):
    gq, gk, gv = (torch.from_numpy(x).to(dev()) for x in (q, k, v))
    s = None if signs is None else torch.from_numpy(signs).to(dev())
    (q8, k8, v8), (qd, kd, vd) = attn.attn_fp8_quantize(gq, gk, gv, hadamard_signs=s,
                                                        per_tensor=per_tensor)
    o, lse = attn.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=causal,
                               softmax_scale=1 / np.sqrt(q.shape[-1]))
    check_status(attn)
    return (o, lse), [t.cpu().numpy() for t in (q8, k8, v8, qd, kd, vd)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 129, 300, 640])
def test_fp8_forward_matches_dequantised_oracle(attn, N, causal):
    """Against exact attention on the dequantised e4m3 inputs, the only error
    left is the kernel's own: P rounded to e4m3 for the P V product and float32
    accumulation."""
    B, H, d = 1, 2, 128
    q, k, v = workloads.normal_with_outliers(40 + N, (B, H, N, d), 3)
    signs = workloads.random_signs(5, d)
    (o, lse), (q8, k8, v8, qd, kd, vd) = _fp8_forward(attn, q, k, v, signs, False, causal)
    dq_, dk_, dv_ = (oracle.dequantize_e4m3_blocks(c, s) for c, s in ((q8, qd), (k8, kd), (v8, vd)))
    ref_o, ref_l = oracle.attention_forward(dq_, dk_, dv_, 1 / np.sqrt(d), causal)
    got = o.float().cpu().numpy()
    diff = got - ref_o
    assert np.sqrt(np.mean(diff ** 2)) <= 1e-2 * max(1.0, np.sqrt(np.mean(ref_o ** 2)))
    assert np.abs(diff).max() <= 0.25 * max(1.0, np.abs(ref_o).max())
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=2e-3)


def test_fp8_outlier_config_rmse(attn):
    """The outlier-stress problem at full size (B=2, H=16, N=4096, d=128): RMSE
    of the FP8 output against exact float64 attention on the original float32
    inputs, on sampled heads, for per-tensor, block, and block + Hadamard."""
    w = workloads.FP8_FWD
    q, k, v = workloads.normal_with_outliers(w.seed, (w.B, w.H, w.N, w.d), 3)
    signs = workloads.random_signs(workloads.FP8_HADAMARD_SIGN_SEED, w.d)
    heads = [(0, 0), (1, 9), (0, 15)]
    refs = {bh: oracle.attention_forward_head(q[bh], k[bh], v[bh], w.scale, w.causal)[0]
            for bh in heads}
    rmse = {}
    for name, sg, pt in (("per_tensor", None, True), ("block", None, False),
                         ("block_hadamard", signs, False)):
        (o, _), _ = _fp8_forward(attn, q, k, v, sg, pt, w.causal)
        got = o.float().cpu().numpy()
        err = np.concatenate([(got[bh] - refs[bh]).ravel() for bh in heads])
        rmse[name] = float(np.sqrt(np.mean(err ** 2)))
    print("fp8 rmse", rmse)
    assert rmse["block"] <= FP8_RMSE and rmse["block_hadamard"] <= FP8_RMSE
    # the ordering the oracle's own quantiser gives on this workload
    assert rmse["block_hadamard"] < rmse["block"] < rmse["per_tensor"]


@pytest.mark.parametrize("with_hadamard", [False, True])
@pytest.mark.parametrize("N", [1, 300, 1024])
def test_quantiser_with_rope(attn, N, with_hadamard):
    """Rotary embedding fused in front of the Hadamard: the GPU rotates and
    transforms in float32, the oracle in float64, so descales agree to float32
    rounding and codes differ by at most one e4m3 step, rarely."""
    shape = (2, 2, N, 128)
    xs = workloads.normal_with_outliers(13 + N, shape, 3)
    signs = workloads.random_signs(5, 128) if with_hadamard else None
    cos, sin = workloads.rope_tables(N, 128)
    g = [torch.from_numpy(x).to(dev()) for x in xs]
    s = None if signs is None else torch.from_numpy(signs).to(dev())
    codes, desc = attn.attn_fp8_quantize_rope(*g, torch.from_numpy(cos).to(dev()),
                                              torch.from_numpy(sin).to(dev()), hadamard_signs=s)
    check_status(attn)
    for which, (x, c, d) in enumerate(zip(xs, codes, desc)):
        c, d = c.cpu().numpy(), d.cpu().numpy()
        rc, rd = oracle.quantize_e4m3_blocks(x, signs=signs if which < 2 else None,
                                             rope=(cos, sin) if which < 2 else None)
        if which == 2:                                 # V is neither rotated nor transformed
            np.testing.assert_array_equal(d, rd)
            np.testing.assert_array_equal(c, rc)
            continue
        np.testing.assert_allclose(d, rd, rtol=4e-6)
        got, ref = oracle.e4m3_decode(c), oracle.e4m3_decode(rc)
        step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -6))) - 3)
        assert np.all(np.abs(got - ref) <= step * 1.0001)
        assert np.mean(c != rc) < 2e-3


def test_fp8_forward_with_rope_matches_rotated_attention(attn):
    """Scores of the rotated Q, K: the FP8 forward on the fused pre-pass output
    against exact float64 attention on the rotated float32 inputs."""
    B, H, N, d = 1, 2, 640, 128
    q, k, v = workloads.normal_with_outliers(44, (B, H, N, d), 3)
    signs = workloads.random_signs(5, d)
    cos, sin = workloads.rope_tables(N, d)
    g = [torch.from_numpy(x).to(dev()) for x in (q, k, v)]
    (q8, k8, v8), (qd, kd, vd) = attn.attn_fp8_quantize_rope(
        *g, torch.from_numpy(cos).to(dev()), torch.from_numpy(sin).to(dev()),
        hadamard_signs=torch.from_numpy(signs).to(dev()))
    o, lse = attn.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=True, softmax_scale=1 / np.sqrt(d))
    check_status(attn)
    rq, rk = oracle.rotary_embed(q, cos, sin), oracle.rotary_embed(k, cos, sin)
    ref_o, _ = oracle.attention_forward(rq, rk, v, 1 / np.sqrt(d), True)
    err = o.float().cpu().numpy() - ref_o
    assert np.sqrt(np.mean(err ** 2)) <= FP8_RMSE


def _bf16_inputs(seed, shapes):
    """Seeded float32 arrays rounded to bfloat16: torch tensors and their exact
    float32 values."""
    xs = [workloads.round_to(x, "bf16") for x in
          (workloads.normal_with_outliers(seed + i, s, 1) for i, s in enumerate(shapes))]
    return xs, [x.float().numpy() for x in xs]


@pytest.mark.parametrize("H_kv", [4, 2])
@pytest.mark.parametrize("per_tensor", [False, True])
def test_bf16_quantiser_bit_exact(attn, H_kv, per_tensor):
    """bfloat16 inputs are quantised exactly as their float32 values are."""
    ts, xs = _bf16_inputs(31, [(2, 4, 300, 128), (2, H_kv, 300, 128), (2, H_kv, 300, 128)])
    codes, desc = attn.attn_fp8_quantize_bf16(*(t.to(dev()) for t in ts), per_tensor=per_tensor)
    check_status(attn)
    for x, c, d in zip(xs, codes, desc):
        rc, rd = oracle.quantize_e4m3_blocks(x, per_tensor=per_tensor)
        np.testing.assert_array_equal(d.cpu().numpy(), rd)
        np.testing.assert_array_equal(c.cpu().numpy(), rc)


def test_bf16_prepass_matches_float32_prepass(attn):
    """With the transform, the bfloat16 pre-pass gives the float32 pre-pass's bits
    on the same values (both widen to float32 before the transform)."""
    ts, xs = _bf16_inputs(32, [(1, 4, 700, 128)] * 3)
    signs = torch.from_numpy(workloads.random_signs(5, 128)).to(dev())
    a = attn.attn_fp8_quantize_bf16(*(t.to(dev()) for t in ts), hadamard_signs=signs)
    b = attn.attn_fp8_quantize(*(torch.from_numpy(x).to(dev()) for x in xs), hadamard_signs=signs)
    check_status(attn)
    for ta, tb in zip(a[0] + a[1], b[0] + b[1]):
        assert torch.equal(ta, tb)


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_prepass_forward_matches_dequantised_oracle(attn, causal):
    ts, xs = _bf16_inputs(33, [(1, 2, 384, 128)] * 3)
    signs = workloads.random_signs(6, 128)
    (q8, k8, v8), (qd, kd, vd) = attn.attn_fp8_quantize_bf16(
        *(t.to(dev()) for t in ts), hadamard_signs=torch.from_numpy(signs).to(dev()))
    o, lse = attn.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=causal, softmax_scale=1 / np.sqrt(128))
    check_status(attn)
    deq = [oracle.dequantize_e4m3_blocks(c.cpu().numpy(), s.cpu().numpy())
           for c, s in ((q8, qd), (k8, kd), (v8, vd))]
    ref_o, ref_l = oracle.attention_forward(*deq, 1 / np.sqrt(128), causal)
    diff = o.float().cpu().numpy() - ref_o
    assert np.sqrt(np.mean(diff ** 2)) <= 1e-2 * max(1.0, np.sqrt(np.mean(ref_o ** 2)))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=2e-3)
    # total error against exact attention of the bfloat16 inputs
    exact, _ = oracle.attention_forward(*(x.astype(np.float64) for x in xs), 1 / np.sqrt(128), causal)
    assert np.sqrt(np.mean((o.float().cpu().numpy() - exact) ** 2)) <= FP8_RMSE


@pytest.mark.parametrize("causal", [False, True])
def test_timed_fp8_chain_full_size(attn, causal):
    """The FP8 stages exactly as the benchmark times them, at B=2, H=16,
    N=8192, d=128 on the same seeded bfloat16 inputs: the bfloat16 pre-pass
    (block scales, Hadamard on Q and K) then the FP8 forward.
    * Sampled rows of three heads against exact attention on the dequantised
      codes (the forward kernel's own error: e4m3 P and float32 sums).
    * The same rows against exact attention of the bfloat16 inputs: RMSE within
      the FP8 bar.
    * The sampled heads' codes against the oracle quantiser (at most one e4m3
      step apart, rarely: the transform runs in float32 on the GPU)."""
    w = workloads.LONG_FWD
    *gs, _, gsigns = timed_step_inputs(w.seed, (w.B, w.H, w.N, w.d))
    (q8, k8, v8), (qd, kd, vd) = attn.attn_fp8_quantize_bf16(*gs, hadamard_signs=gsigns)
    o, lse = attn.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=causal, softmax_scale=w.scale)
    check_status(attn)
    rng = np.random.default_rng(99)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 129, 4095, 8190, 8191],
                                     rng.integers(0, w.N, 40)]))
    got_o = o.float().cpu().numpy()
    got_l = lse.cpu().numpy()
    ts = [t.cpu() for t in gs]
    signs = gsigns.cpu().numpy()
    codes = [c.cpu().numpy() for c in (q8, k8, v8)]
    descs = [d.cpu().numpy() for d in (qd, kd, vd)]
    err_deq, err_exact = [], []
    for b, h in ((0, 0), (1, 15), (0, 7)):
        deq = [oracle.dequantize_e4m3_blocks(c[b:b + 1, h:h + 1], d[b:b + 1, h:h + 1])[0, 0]
               for c, d in zip(codes, descs)]
        ref_o, ref_l = oracle.attention_forward_rows(*deq, w.scale, causal, rows)
        err_deq.append(got_o[b, h, rows] - ref_o)
        np.testing.assert_allclose(got_l[b, h, rows], ref_l, atol=2e-3)
        x = [workloads.as_f64(t[b, h]) for t in ts]
        ex_o, _ = oracle.attention_forward_rows(*x, w.scale, causal, rows)
        err_exact.append(got_o[b, h, rows] - ex_o)
        # the quantiser on this head
        for which in range(3):
            xi = workloads.as_f64(ts[which][b:b + 1, h:h + 1]).astype(np.float32)
            rc, rd = oracle.quantize_e4m3_blocks(xi, signs=signs if which < 2 else None)
            np.testing.assert_allclose(descs[which][b:b + 1, h:h + 1], rd, rtol=2e-6)
            c = codes[which][b:b + 1, h:h + 1]
            if which == 2:
                np.testing.assert_array_equal(c, rc)
                continue
            gv, rv = oracle.e4m3_decode(c), oracle.e4m3_decode(rc)
            step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(rv), 2.0 ** -6))) - 3)
            assert np.all(np.abs(gv - rv) <= step * 1.0001)
            assert np.mean(c != rc) < 1e-3
    e = np.concatenate([x.ravel() for x in err_deq])
    assert np.sqrt(np.mean(e ** 2)) <= 1e-2 and np.abs(e).max() <= 0.25, \
        (np.sqrt(np.mean(e ** 2)), np.abs(e).max())
    e = np.concatenate([x.ravel() for x in err_exact])
    assert np.sqrt(np.mean(e ** 2)) <= FP8_RMSE, np.sqrt(np.mean(e ** 2))


def test_exp2_polynomial_error_on_the_gpu(attn):
    """The FMA-pipe exponential of the ATTN_SCHED_EXP2_POLY variant against the
    exact 2^x (float64) and against the MUFU ex2.approx on the GPU: relative
    error <= 1.1e-4 over the softmax's range, exactly 0 at and below -127 and
    at -inf, and 1 at 0."""
    xs = np.concatenate([np.linspace(-126.0, 8.0, 2_000_001), np.arange(-126, 9, dtype=np.float64),
                         np.arange(-126, 8, dtype=np.float64) + 0.5,
                         [-np.inf, -1e30, -200.0, -127.0, -127.0 + 1e-3, -126.75, 0.0, -0.0]])
    x = torch.from_numpy(xs.astype(np.float32)).to(dev())
    y_poly, y_mufu = attn.attn_selftest_exp2(x)
    check_status(attn)
    xf = x.double().cpu().numpy()
    yp = y_poly.double().cpu().numpy()
    ym = y_mufu.double().cpu().numpy()
    exact = np.exp2(xf)
    normal = (xf >= -126.0) & (xf <= 8.0)
    rel = np.abs(yp[normal] / exact[normal] - 1.0)
    assert rel.max() <= 1.1e-4, rel.max()
    # the MUFU path as the kernels use it, for reference: far tighter
    assert np.abs(ym[normal & (xf >= -125.0)] / exact[normal & (xf >= -125.0)] - 1.0).max() <= 1e-6
    assert np.all(yp[xf <= -127.0] == 0.0)
    tiny = (xf > -127.0) & (xf < -126.0)
    assert np.all((yp[tiny] >= 0.0) & (yp[tiny] <= 2.0 ** -126))
    assert np.all(yp[xf == 0.0] == 1.0)


@pytest.mark.parametrize("eighths", ["none", 0, 1, 3, 4])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [129, 640])
def test_fp8_exp2_poly_variant_matches_dequantised_oracle(attn, N, causal, eighths):
    """The forward with none or part of its exponentials on the FMA pipe (a quarter
    for ATTN_SCHED_EXP2_POLY alone, else k eighths) computes the same attention as
    the library's default (the polynomial's error is far below the e4m3 rounding of P)."""
    B, H, d = 1, 2, 128
    q, k, v = workloads.normal_with_outliers(60 + N, (B, H, N, d), 3)
    signs = workloads.random_signs(5, d)
    gq, gk, gv = (torch.from_numpy(x).to(dev()) for x in (q, k, v))
    (q8, k8, v8), (qd, kd, vd) = attn.attn_fp8_quantize(gq, gk, gv,
                                                        hadamard_signs=torch.from_numpy(signs).to(dev()))
    sched = (attn.ATTN_SCHED_EXP2_NONE if eighths == "none" else
             attn.ATTN_SCHED_EXP2_POLY if eighths == 0 else attn.ATTN_SCHED_EXP2_EIGHTHS(eighths))
    o, lse = attn.attn_fwd_fp8_schedule(q8, k8, v8, qd, kd, vd, sched,
                                        causal=causal, softmax_scale=1 / np.sqrt(d))
    o0, _ = attn.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=causal, softmax_scale=1 / np.sqrt(d))
    check_status(attn)
    deq = [oracle.dequantize_e4m3_blocks(c.cpu().numpy(), s.cpu().numpy())
           for c, s in ((q8, qd), (k8, kd), (v8, vd))]
    ref_o, ref_l = oracle.attention_forward(*deq, 1 / np.sqrt(d), causal)
    diff = o.float().cpu().numpy() - ref_o
    assert np.sqrt(np.mean(diff ** 2)) <= 1e-2 * max(1.0, np.sqrt(np.mean(ref_o ** 2)))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=2e-3)
    # and close to the MUFU-only forward
    assert (o.float() - o0.float()).pow(2).mean().sqrt().item() <= 2e-3
