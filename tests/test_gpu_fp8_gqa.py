"""FP8 path with grouped-query heads (K and V with H_kv < H heads): the pre-pass
against the oracle quantiser per tensor, the forward against exact float64
attention of the dequantised inputs with shared key/value heads, and the
grouped call against the same call with the key/value heads repeated."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import check_status, dev, lib

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def attn():
    return lib()


def _inputs(seed, B, H, H_kv, N):
    (q,) = [workloads.normal_with_outliers(seed, (B, H, N, D), 1)]
    k, v = workloads.normal_with_outliers(seed + 1, (B, H_kv, N, D), 2)
    return q, k, v


@pytest.mark.parametrize("H,H_kv", [(4, 2), (6, 1)])
@pytest.mark.parametrize("per_tensor", [False, True])
def test_quantiser_bit_exact(attn, H, H_kv, per_tensor):
    q, k, v = _inputs(21, 2, H, H_kv, 300)
    codes, desc = attn.attn_fp8_quantize_gqa(*(torch.from_numpy(x).to(dev()) for x in (q, k, v)),
                                             per_tensor=per_tensor)
    check_status(attn)
    for x, c, d in zip((q, k, v), codes, desc):
        rc, rd = oracle.quantize_e4m3_blocks(x, per_tensor=per_tensor)
        np.testing.assert_array_equal(d.cpu().numpy(), rd)
        np.testing.assert_array_equal(c.cpu().numpy(), rc)


def _fp8_gqa(attn, q, k, v, causal, signs=None):
    s = None if signs is None else torch.from_numpy(signs).to(dev())
    (q8, k8, v8), (qd, kd, vd) = attn.attn_fp8_quantize_gqa(
        *(torch.from_numpy(x).to(dev()) for x in (q, k, v)), hadamard_signs=s)
    o, lse = attn.attn_fwd_fp8_gqa(q8, k8, v8, qd, kd, vd, causal=causal,
                                   softmax_scale=1 / np.sqrt(D))
    check_status(attn)
    return (o, lse), (q8, k8, v8, qd, kd, vd)


@pytest.mark.parametrize("H,H_kv", [(4, 2), (6, 1), (4, 4)])
@pytest.mark.parametrize("N", [100, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_dequantised_oracle(attn, H, H_kv, N, causal):
    """Against exact grouped-query attention on the dequantised e4m3 inputs, the
    only error left is the kernel's own (P rounded to e4m3, float32 sums)."""
    q, k, v = _inputs(30 + N + H_kv, 2, H, H_kv, N)
    signs = workloads.random_signs(6, D)
    (o, lse), t = _fp8_gqa(attn, q, k, v, causal, signs)
    q8, k8, v8, qd, kd, vd = (x.cpu().numpy() for x in t)
    deq = [oracle.dequantize_e4m3_blocks(c, s) for c, s in ((q8, qd), (k8, kd), (v8, vd))]
    ref_o, ref_l = oracle.attention_forward_gqa(*deq, 1 / np.sqrt(D), causal)
    got = o.float().cpu().numpy()
    diff = got - ref_o
    assert np.sqrt(np.mean(diff ** 2)) <= 1e-2 * max(1.0, np.sqrt(np.mean(ref_o ** 2)))
    assert np.abs(diff).max() <= 0.25 * max(1.0, np.abs(ref_o).max())
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=2e-3)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_equals_repeated_heads(attn, causal):
    """Sharing a key/value head is the same arithmetic as repeating it: the
    grouped call and the plain call on repeated codes and descales agree bit
    for bit."""
    H, H_kv, N = 8, 2, 513
    q, k, v = _inputs(40, 1, H, H_kv, N)
    (o, lse), (q8, k8, v8, qd, kd, vd) = _fp8_gqa(attn, q, k, v, causal)
    rep = lambda t: t.repeat_interleave(H // H_kv, dim=1).contiguous()
    o2, lse2 = attn.attn_fwd_fp8(q8, rep(k8), rep(v8), qd, rep(kd), rep(vd), causal=causal,
                                 softmax_scale=1 / np.sqrt(D))
    check_status(attn)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
