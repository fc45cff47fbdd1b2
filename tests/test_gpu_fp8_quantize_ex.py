"""The general FP8 pre-pass (attn_fp8_quantize_ex): rotary embedding on
bfloat16 and float32 inputs, grouped-query heads and packed batches, against
the oracle quantiser (which rotates and transforms in float64), and the FP8
forward on its output against exact attention of the rotated inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import FP8_RMSE, check_status, dev, lib

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def attn():
    return lib()


def _close_codes(c, rc, frac):
    """GPU codes within one e4m3 step of the oracle's, and rarely different
    (the rotation and transform run in float32 on the GPU, float64 in the oracle)."""
    got, ref = oracle.e4m3_decode(c), oracle.e4m3_decode(rc)
    step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -6))) - 3)
    assert np.all(np.abs(got - ref) <= step * 1.0001)
    assert np.mean(c != rc) < frac


def _bf16(seed, shape):
    t = workloads.round_to(workloads.normal_with_outliers(seed, shape, 1), "bf16")
    return t, t.float().numpy()


@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("H,H_kv", [(4, 2), (2, 2)])
@pytest.mark.parametrize("N", [1, 300, 1024])
def test_bf16_rope_fixed_length(attn, N, H, H_kv, hadamard):
    B = 2
    tq, q = _bf16(70 + N, (B, H, N, D))
    tk, k = _bf16(71 + N, (B, H_kv, N, D))
    tv, v = _bf16(72 + N, (B, H_kv, N, D))
    cos, sin = workloads.rope_tables(N, D)
    signs = workloads.random_signs(5, D) if hadamard else None
    codes, desc = attn.attn_fp8_quantize_ex(
        *(t.to(dev()) for t in (tq, tk, tv)), torch.from_numpy(cos).to(dev()),
        torch.from_numpy(sin).to(dev()),
        hadamard_signs=None if signs is None else torch.from_numpy(signs).to(dev()))
    check_status(attn)
    for which, (x, c, d) in enumerate(zip((q, k, v), codes, desc)):
        c, d = c.cpu().numpy(), d.cpu().numpy()
        rc, rd = oracle.quantize_e4m3_blocks(x, signs=signs if which < 2 else None,
                                             rope=(cos, sin) if which < 2 else None)
        if which == 2:                     # V is neither rotated nor transformed: bit-exact
            np.testing.assert_array_equal(d, rd)
            np.testing.assert_array_equal(c, rc)
            continue
        np.testing.assert_allclose(d, rd, rtol=4e-6)
        _close_codes(c, rc, 2e-3)


def test_bf16_rope_equals_float32_rope_bitwise(attn):
    """bfloat16 inputs are rotated exactly as their float32 values are: the
    register-staged bf16 kernel gives the staged float32 kernel's bits."""
    B, H, N = 1, 4, 700
    ts, xs = zip(*(_bf16(80 + i, (B, H, N, D)) for i in range(3)))
    cos, sin = (torch.from_numpy(t).to(dev()) for t in workloads.rope_tables(N, D))
    signs = torch.from_numpy(workloads.random_signs(5, D)).to(dev())
    a = attn.attn_fp8_quantize_ex(*(t.to(dev()) for t in ts), cos, sin, hadamard_signs=signs)
    b = attn.attn_fp8_quantize_ex(*(torch.from_numpy(x).to(dev()) for x in xs), cos, sin,
                                  hadamard_signs=signs)
    check_status(attn)
    for ta, tb in zip(a[0] + a[1], b[0] + b[1]):
        assert torch.equal(ta, tb)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_packed_rope_gqa(attn, dtype):
    """A packed batch (empty, one-token, tile-ragged and multi-tile sequences),
    H = 4 query heads on H_kv = 2: each sequence is rotated from position 0."""
    cu = np.array([0, 0, 1, 128, 257, 300, 815], dtype=np.int32)
    total, H, H_kv = int(cu[-1]), 4, 2
    lens = np.diff(cu)
    max_len = int(lens.max())
    xs = [workloads.normal_with_outliers(90 + i, (total, h, D), 1) for i, h in enumerate((H, H_kv, H_kv))]
    if dtype == "bf16":
        ts = [workloads.round_to(x, "bf16") for x in xs]
        xs = [t.float().numpy() for t in ts]
    else:
        ts = [torch.from_numpy(x) for x in xs]
    cos, sin = workloads.rope_tables(max_len, D)
    signs = workloads.random_signs(5, D)
    codes, desc = attn.attn_fp8_quantize_ex(
        *(t.to(dev()) for t in ts), torch.from_numpy(cos).to(dev()), torch.from_numpy(sin).to(dev()),
        hadamard_signs=torch.from_numpy(signs).to(dev()), cu_seqlens=torch.from_numpy(cu).to(dev()),
        max_seqlen=max_len)
    check_status(attn)
    nblk = (max_len + 127) // 128
    for which, (x, c, d) in enumerate(zip(xs, codes, desc)):
        c, d = c.cpu().numpy(), d.cpu().numpy()
        for b in range(len(lens)):
            s0, s1 = int(cu[b]), int(cu[b + 1])
            if s1 == s0:
                assert np.all(d[b] == 1.0)
                continue
            seq = np.transpose(x[s0:s1], (1, 0, 2))[None]
            rc, rd = oracle.quantize_e4m3_blocks(
                seq, signs=signs if which < 2 else None,
                rope=(cos[:s1 - s0], sin[:s1 - s0]) if which < 2 else None)
            got = np.transpose(c[s0:s1], (1, 0, 2))[None]
            nb = rd.shape[2]
            np.testing.assert_allclose(d[b:b + 1, :, :nb], rd, rtol=4e-6)
            assert np.all(d[b, :, nb:nblk] == 1.0)
            if which == 2:
                np.testing.assert_array_equal(got, rc)
            else:
                _close_codes(got, rc, 3e-3)


def test_fp8_forward_on_rotated_bf16_inputs(attn):
    """The FP8 forward on the rotated bfloat16 pre-pass output against exact
    float64 attention of the rotated inputs (causal, grouped-query heads)."""
    B, H, H_kv, N = 1, 4, 2, 1024
    tq, q = _bf16(100, (B, H, N, D))
    tk, k = _bf16(101, (B, H_kv, N, D))
    tv, v = _bf16(102, (B, H_kv, N, D))
    cos, sin = workloads.rope_tables(N, D)
    signs = workloads.random_signs(5, D)
    (q8, k8, v8), (qd, kd, vd) = attn.attn_fp8_quantize_ex(
        *(t.to(dev()) for t in (tq, tk, tv)), torch.from_numpy(cos).to(dev()),
        torch.from_numpy(sin).to(dev()), hadamard_signs=torch.from_numpy(signs).to(dev()))
    o, _ = attn.attn_fwd_fp8_gqa(q8, k8, v8, qd, kd, vd, causal=True, softmax_scale=1 / np.sqrt(D))
    check_status(attn)
    rq, rk = oracle.rotary_embed(q, cos, sin), oracle.rotary_embed(k, cos, sin)
    ref_o, _ = oracle.attention_forward_gqa(rq, rk, v, 1 / np.sqrt(D), True)
    err = o.float().cpu().numpy() - ref_o
    assert np.sqrt(np.mean(err ** 2)) <= FP8_RMSE
