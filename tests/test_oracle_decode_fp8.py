"""Pins for the FP8 paged-cache oracle: the e4m3 rounding bound and the
saturation point of every (page, head) block, block independence, the
orthogonality of the key transform, closed forms of a one-key cache, the exact
scaling laws of the descales, physical-page permutation, and the identity
(q M)(K M)^T = q K^T that the transformed cache relies on."""
import numpy as np
import pytest

import oracle
import workloads


def _cache(seed, pages=5, page_size=16, H_kv=2, d=16):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((pages, page_size, H_kv, d), dtype=np.float32)
            * rng.uniform(0.1, 4.0, (pages, 1, H_kv, 1)).astype(np.float32))


def test_block_rounding_bound_and_saturation():
    """Each value lies within half an e4m3 step of code x descale (relative
    2^-4 for normals, 2^-10 x descale below 2^-6 x descale), and the largest
    magnitude of every (page, head) block is coded as exactly +-448."""
    x = _cache(1)
    codes, desc = oracle.quantize_paged_cache(x)
    assert codes.shape == x.shape and codes.dtype == np.uint8 and desc.shape == (5, 2)
    deq = oracle.dequantize_paged_cache(codes, desc)
    d64 = np.asarray(desc, np.float64)[:, None, :, None]
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * d64) * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)
    for p in range(x.shape[0]):
        for h in range(x.shape[2]):
            blk = x[p, :, h]
            i = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert abs(oracle.e4m3_decode(codes[p, :, h][i])) == 448.0
            assert desc[p, h] == np.float32(np.abs(blk).max()) / np.float32(448.0)


def test_blocks_are_independent_and_zero_block_has_unit_descale():
    x = _cache(2)
    y = x.copy()
    y[3, :, 1] *= 10.0
    y[1, :, 0] = 0.0
    c1, d1 = oracle.quantize_paged_cache(x)
    c2, d2 = oracle.quantize_paged_cache(y)
    same = np.ones((5, 2), bool)
    same[3, 1] = same[1, 0] = False
    for p in range(5):
        for h in range(2):
            if same[p, h]:
                assert np.array_equal(c1[p, :, h], c2[p, :, h]) and d1[p, h] == d2[p, h]
    assert d2[1, 0] == 1.0 and np.all(c2[1, :, 0] == 0)
    assert np.isclose(d2[3, 1], 10.0 * d1[3, 1], rtol=1e-6)


def test_key_transform_is_orthogonal():
    """Codes of K M, mapped back with M^T, recover K within the rounding bound."""
    x = _cache(3)
    signs = workloads.random_signs(4, 16)
    codes, desc = oracle.quantize_paged_cache(x, signs)
    m = signs[:, None] * oracle.sylvester_hadamard(16) / 4.0
    back = oracle.dequantize_paged_cache(codes, desc) @ m.T
    err = np.sqrt(np.mean((back - x) ** 2))
    assert err <= 2.0 ** -4 * np.sqrt(np.mean(x ** 2))
    plain = oracle.dequantize_paged_cache(codes, desc)
    assert np.sqrt(np.mean((plain - x) ** 2)) > 0.5 * np.sqrt(np.mean(x ** 2))


def test_one_key_closed_form():
    """With one cached token, O is its dequantised value row and LSE the scaled
    score q . k."""
    rng = np.random.default_rng(5)
    kc = np.zeros((2, 16, 1, 8), np.float32)
    vc = np.zeros_like(kc)
    kc[1, 0, 0] = rng.standard_normal(8)
    vc[1, 0, 0] = rng.standard_normal(8)
    k8, kd = oracle.quantize_paged_cache(kc)
    v8, vd = oracle.quantize_paged_cache(vc)
    table = np.array([[1]], np.int32)
    q = rng.standard_normal((1, 3, 1, 8))
    o, lse = oracle.attention_decode_paged_fp8(q, k8, v8, kd, vd, table, [1], 0.7, True)
    kv = oracle.e4m3_decode(k8[1, 0, 0]) * np.float64(kd[1, 0])
    vv = oracle.e4m3_decode(v8[1, 0, 0]) * np.float64(vd[1, 0])
    for h in range(3):
        np.testing.assert_allclose(o[0, h, 0], vv, rtol=1e-14)
        np.testing.assert_allclose(lse[0, h, 0], 0.7 * q[0, h, 0] @ kv, rtol=1e-13)


def _fp8_case(seed, lens=(37, 70), page_size=16, H=4, H_kv=2, d=16, n_q=2):
    kc, vc, table = workloads.paged_cache(seed, list(lens), page_size, H_kv, d, spare_pages=4)
    k8, kd = oracle.quantize_paged_cache(kc)
    v8, vd = oracle.quantize_paged_cache(vc)
    q = workloads.normal(seed + 1, (len(lens), H, n_q, d))
    return q, k8, v8, kd, vd, table, list(lens)


def test_descale_scaling_laws():
    """Doubling every K descale equals doubling the softmax scale; doubling the
    V descale of every page doubles O and leaves LSE unchanged."""
    q, k8, v8, kd, vd, table, lens = _fp8_case(6)
    o, l = oracle.attention_decode_paged_fp8(q, k8, v8, kd, vd, table, lens, 0.25, True)
    o2, l2 = oracle.attention_decode_paged_fp8(q, k8, v8, 2 * kd, vd, table, lens, 0.125, True)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l2, l, rtol=1e-12)
    o3, l3 = oracle.attention_decode_paged_fp8(q, k8, v8, kd, 2 * vd, table, lens, 0.25, True)
    np.testing.assert_allclose(o3, 2 * o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l3, l, rtol=0)


def test_descales_follow_physical_pages():
    """Moving pages (codes and descales together) and rewriting the block table
    changes nothing; moving the codes alone does."""
    q, k8, v8, kd, vd, table, lens = _fp8_case(7)
    o, l = oracle.attention_decode_paged_fp8(q, k8, v8, kd, vd, table, lens, 0.3, False)
    perm = np.random.default_rng(8).permutation(k8.shape[0])
    inv = np.argsort(perm)
    t2 = np.where(table >= 0, inv[np.maximum(table, 0)], -1)
    o2, l2 = oracle.attention_decode_paged_fp8(q, k8[perm], v8[perm], kd[perm], vd[perm], t2, lens,
                                               0.3, False)
    np.testing.assert_allclose(o2, o, atol=0)
    np.testing.assert_allclose(l2, l, atol=0)
    o3, _ = oracle.attention_decode_paged_fp8(q, k8[perm], v8[perm], kd, vd, t2, lens, 0.3, False)
    assert np.abs(o3 - o).max() > 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_transformed_cache_matches_plain_attention(causal):
    """Keys stored as K M with the query transformed by the same M give the
    attention of the original q, K within e4m3 error (about 2.5% of the RMS of O
    here); the opposite sign vector, or no transform of the query, does not."""
    d = 32
    kc, vc, table = workloads.paged_cache(9, [50, 90], 16, 2, d)
    q = workloads.normal(10, (2, 4, 2, d))
    signs = workloads.random_signs(11, d)
    k8, kd = oracle.quantize_paged_cache(kc, signs)
    v8, vd = oracle.quantize_paged_cache(vc)
    vdq = oracle.dequantize_paged_cache(v8, vd)
    exact, _ = oracle.attention_decode_paged(q, kc, vdq, table, [50, 90], 1 / np.sqrt(d), causal)
    o, _ = oracle.attention_decode_paged_fp8(q, k8, v8, kd, vd, table, [50, 90], 1 / np.sqrt(d),
                                             causal, signs)
    rms = np.sqrt(np.mean(exact ** 2))
    assert np.sqrt(np.mean((o - exact) ** 2)) <= 5e-2 * rms
    for bad in (-signs, None):      # another M, or the query left untransformed
        o_bad, _ = oracle.attention_decode_paged_fp8(q, k8, v8, kd, vd, table, [50, 90],
                                                     1 / np.sqrt(d), causal, bad)
        assert np.sqrt(np.mean((o_bad - exact) ** 2)) > 0.5 * rms
