"""Pins for the FP8 quantiser and incoherent-processing oracle."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads


def test_e4m3_hand_codes(golden_dir):
    with open(os.path.join(golden_dir, "e4m3_codes.json")) as f:
        cases = json.load(f)["cases"]
    xs = np.array([c["x"] for c in cases])
    codes = np.array([c["code"] for c in cases], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e4m3_encode(xs), codes)


def test_e4m3_every_code_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    nan = np.isnan(vals)
    assert nan.sum() == 2 and set(codes[nan]) == {0x7F, 0xFF}
    back = oracle.e4m3_encode(vals[~nan])
    # +0 and -0 are distinct codes with equal value; encode keeps the sign bit
    np.testing.assert_array_equal(back, codes[~nan])
    assert np.nanmax(vals) == 448.0 and np.nanmin(vals) == -448.0


def test_e4m3_matches_torch_after_clamp():
    """Independent library cross-check: torch.float8_e4m3fn (round to nearest
    even).  torch gives NaN rather than saturating above 448, so clamp first."""
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1, 30, 300)])
    x = np.concatenate([x, [0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 1e-12]])
    x = x.astype(np.float32)
    xc = np.clip(x, -448.0, 448.0)
    ref = torch.from_numpy(xc).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = oracle.e4m3_encode(x)
    np.testing.assert_array_equal(mine, ref)


def test_e4m3_rounding_error_bound():
    """Round to nearest: |x - q(x)| <= half a step of the e4m3 grid."""
    rng = np.random.default_rng(1)
    x = rng.uniform(-448, 448, 50000)
    q = oracle.e4m3_decode(oracle.e4m3_encode(x))
    a = np.maximum(np.abs(x), 2.0 ** -6)
    step = 2.0 ** (np.floor(np.log2(a)) - 3)
    assert np.all(np.abs(x - q) <= step / 2 + 1e-15)


def test_hadamard_orthogonality_and_fast_transform():
    for d in (1, 2, 4, 64, 128, 256):
        h = oracle.sylvester_hadamard(d)
        np.testing.assert_array_equal(h @ h.T, d * np.eye(d))
        assert set(np.unique(h)) <= {-1.0, 1.0}
    # Sylvester order: entry (i, j) = (-1)^popcount(i & j)
    d = 128
    h = oracle.sylvester_hadamard(d)
    i, j = np.meshgrid(np.arange(d), np.arange(d), indexing="ij")
    pop = np.vectorize(lambda t: bin(t).count("1"))(i & j)
    np.testing.assert_array_equal(h, (-1.0) ** pop)


def test_incoherent_transform_preserves_scores():
    """(QM)(KM)^T = QK^T for the orthogonal M = diag(s) H / sqrt(d)."""
    B, H, N, d = 1, 2, 40, 128
    q, k = workloads.normal(3, (B, H, N, d), 2)
    s = workloads.random_signs(5, d)
    qm = oracle.incoherent_transform(q, s)
    km = oracle.incoherent_transform(k, s)
    ref = np.einsum("bhqd,bhkd->bhqk", q.astype(np.float64), k.astype(np.float64))
    got = np.einsum("bhqd,bhkd->bhqk", qm, km)
    np.testing.assert_allclose(got, ref, atol=1e-11)
    # and it is not the identity: a single spike is spread over all coordinates
    e = np.zeros(d)
    e[3] = 1.0
    t = oracle.incoherent_transform(e[None], s)[0]
    np.testing.assert_allclose(np.abs(t), 1 / np.sqrt(d), atol=1e-15)


def test_block_quantiser_scales_and_codes():
    rng = np.random.default_rng(2)
    B, H, N, d = 1, 2, 300, 64
    x = (rng.standard_normal((B, H, N, d)) * 3).astype(np.float32)
    x[0, 1, 130:140] = 0.0
    x[0, 1, 256:] = 0.0                       # an all-zero last block
    codes, desc = oracle.quantize_e4m3_blocks(x)
    assert desc.shape == (1, 2, 3) and desc.dtype == np.float32
    assert desc[0, 1, 2] == 1.0               # amax 0 -> descale 1
    blk = np.abs(x[0, 0, :128]).max()
    assert desc[0, 0, 0] == np.float32(blk) / np.float32(448.0)
    deq = oracle.dequantize_e4m3_blocks(codes, desc)
    # the largest entry of each nonzero block maps to +-448 exactly
    for h in range(2):
        for bi in range(2):
            rows = slice(bi * 128, min(N, bi * 128 + 128))
            assert np.abs(oracle.e4m3_decode(codes[0, h, rows])).max() == 448.0
    # relative error per element bounded by the e4m3 grid (2^-4) away from subnormals
    big = np.abs(x) > 0.1
    rel = np.abs(deq - x)[big] / np.abs(x)[big]
    assert rel.max() <= 2.0 ** -4 + 1e-7


def test_per_tensor_mode_uses_one_scale():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 2, 200, 32)).astype(np.float32)
    _, desc = oracle.quantize_e4m3_blocks(x, per_tensor=True)
    assert np.all(desc == np.float32(np.abs(x).max()) / np.float32(448.0))


def test_fp8_error_ordering_on_outlier_workload():
    """RMSE of FP8 attention against exact attention: block+Hadamard < block <
    per-tensor on the outlier-stress inputs (the ordering the first page's 'FP8
    accuracy controls' section reports)."""
    B, H, N, d = 1, 4, 512, 128
    q, k, v = workloads.normal_with_outliers(4, (B, H, N, d), 3)
    s = workloads.random_signs(5, d)
    scale = 1 / np.sqrt(d)
    o_ref, _ = oracle.attention_forward(q, k, v, scale)

    def rmse_for(per_tensor, signs):
        qc, qd = oracle.quantize_e4m3_blocks(q, per_tensor=per_tensor, signs=signs)
        kc, kd = oracle.quantize_e4m3_blocks(k, per_tensor=per_tensor, signs=signs)
        vc, vd = oracle.quantize_e4m3_blocks(v, per_tensor=per_tensor)
        o, _ = oracle.attention_forward(oracle.dequantize_e4m3_blocks(qc, qd),
                                        oracle.dequantize_e4m3_blocks(kc, kd),
                                        oracle.dequantize_e4m3_blocks(vc, vd), scale)
        return float(np.sqrt(np.mean((o - o_ref) ** 2)))

    r_tensor = rmse_for(True, None)
    r_block = rmse_for(False, None)
    r_had = rmse_for(False, s)
    assert r_had < r_block < r_tensor, (r_had, r_block, r_tensor)
    assert r_had < 3e-2
