"""Pins for the oracle's rotary embedding (the rotation fused into the FP8
pre-pass): complex multiplication as an independent route, a hand case,
norm preservation, the relative-position property, and planted slips."""
import numpy as np

import oracle
import workloads


def test_rotation_equals_complex_multiplication():
    rng = np.random.default_rng(41)
    N, d = 9, 16
    x = rng.standard_normal((2, 3, N, d))
    c, s = workloads.rope_tables(N, d)
    got = oracle.rotary_embed(x, c, s)
    z = (x[..., : d // 2] + 1j * x[..., d // 2:]) * (c.astype(np.float64) + 1j * s.astype(np.float64))
    np.testing.assert_allclose(got, np.concatenate([z.real, z.imag], axis=-1), atol=1e-14)


def test_hand_quarter_turn():
    x = np.array([[1.0, 0.0], [0.0, 1.0]])          # two positions, d = 2
    c = np.array([[0.0], [0.0]])
    s = np.array([[1.0], [1.0]])
    np.testing.assert_allclose(oracle.rotary_embed(x, c, s), [[0.0, 1.0], [-1.0, 0.0]], atol=0)


def test_norm_preserved_and_relative_position():
    rng = np.random.default_rng(42)
    N, d = 64, 128
    c, s = workloads.rope_tables(N, d)
    c64, s64 = c.astype(np.float64), s.astype(np.float64)
    # the float32 tables hold cos^2 + sin^2 = 1 to float32 rounding
    q = rng.standard_normal((N, d))
    k = rng.standard_normal((N, d))
    rq = oracle.rotary_embed(q, c, s)
    np.testing.assert_allclose(np.linalg.norm(rq, axis=1), np.linalg.norm(q, axis=1), rtol=1e-6)
    # <R_p q, R_p' k> depends on p - p' only: shift both positions by t
    qv, kv = q[0], k[0]
    rot = lambda v, n: oracle.rotary_embed(v[None], c64[n:n + 1], s64[n:n + 1])[0]
    for p, pp, t in ((5, 2, 7), (30, 10, 20), (3, 3, 50)):
        a = rot(qv, p) @ rot(kv, pp)
        b = rot(qv, p + t) @ rot(kv, pp + t)
        assert abs(a - b) < 1e-4 * (1 + abs(a))


def test_identity_tables_leave_the_quantiser_unchanged():
    x = workloads.normal(43, (1, 2, 200, 128))
    c = np.ones((200, 64), np.float32)
    s = np.zeros((200, 64), np.float32)
    a_codes, a_desc = oracle.quantize_e4m3_blocks(x, rope=(c, s))
    b_codes, b_desc = oracle.quantize_e4m3_blocks(x)
    np.testing.assert_array_equal(a_codes, b_codes)
    np.testing.assert_array_equal(a_desc, b_desc)


def test_planted_interleaved_pairing_differs():
    """Rotating adjacent pairs (x_{2i}, x_{2i+1}) instead of (x_i, x_{i+d/2})
    must not agree with the oracle."""
    rng = np.random.default_rng(44)
    N, d = 5, 8
    x = rng.standard_normal((N, d))
    c, s = workloads.rope_tables(N, d)
    ev, od = x[:, 0::2], x[:, 1::2]
    inter = np.empty_like(x)
    inter[:, 0::2] = ev * c - od * s
    inter[:, 1::2] = od * c + ev * s
    assert not np.allclose(oracle.rotary_embed(x, c, s), inter, atol=1e-6)
