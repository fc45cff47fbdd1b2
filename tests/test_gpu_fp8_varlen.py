"""FP8 path on packed variable-length batches: the packed pre-pass against the
oracle quantiser applied sequence by sequence, the forward against exact float64
attention of the dequantised packed inputs, and a one-sequence batch against the
fixed-length FP8 path."""
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


def _cu(name):
    if name == "mixed":       # empty, length 1, tile-ragged and multi-tile sequences
        return np.array([0, 0, 1, 128, 257, 300, 815], dtype=np.int32)
    if name == "random":
        cu, _ = workloads.varlen_lengths(63, 5, 700)
        return cu
    raise ValueError(name)


def _packed(seed, cu, H, H_kv):
    total = int(cu[-1])
    (q,) = [workloads.normal_with_outliers(seed, (total, H, D), 1)]
    k, v = workloads.normal_with_outliers(seed + 1, (total, H_kv, D), 2)
    return q, k, v


def _oracle_quant(x, cu, signs=None):
    """Per-sequence block quantisation by the oracle: codes [total, heads, d] and
    descales [B, heads, ceil(max_len / 128)] (1 past each sequence's end)."""
    total, heads, _ = x.shape
    lens = np.diff(cu)
    nblk = (int(lens.max()) + 127) // 128
    codes = np.zeros(x.shape, np.uint8)
    desc = np.ones((len(lens), heads, nblk), np.float32)
    for b in range(len(lens)):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        seq = np.transpose(x[s0:s1], (1, 0, 2))[None]          # [1, heads, len, d]
        c, d = oracle.quantize_e4m3_blocks(seq, signs=signs)
        codes[s0:s1] = np.transpose(c[0], (1, 0, 2))
        desc[b, :, :d.shape[2]] = d[0]
    return codes, desc


def _dequant(codes, desc, cu):
    out = np.zeros(codes.shape)
    for b in range(len(cu) - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        seq = np.transpose(codes[s0:s1], (1, 0, 2))[None]
        nb = (s1 - s0 + 127) // 128
        out[s0:s1] = np.transpose(oracle.dequantize_e4m3_blocks(seq, desc[b:b + 1, :, :nb])[0], (1, 0, 2))
    return out


def _quant_gpu(attn, q, k, v, cu, signs=None):
    s = None if signs is None else torch.from_numpy(signs).to(dev())
    max_len = max(int(np.diff(cu).max()), 1)
    codes, desc = attn.attn_fp8_quantize_varlen(*(torch.from_numpy(x).to(dev()) for x in (q, k, v)),
                                                torch.from_numpy(cu).to(dev()), max_len,
                                                hadamard_signs=s)
    check_status(attn)
    return codes, desc, max_len


@pytest.mark.parametrize("case", ["mixed", "random"])
def test_packed_quantiser_bit_exact(attn, case):
    cu = _cu(case)
    q, k, v = _packed(71, cu, 4, 2)
    codes, desc, _ = _quant_gpu(attn, q, k, v, cu)
    for x, c, d in zip((q, k, v), codes, desc):
        rc, rd = _oracle_quant(x, cu)
        np.testing.assert_array_equal(d.cpu().numpy(), rd)
        np.testing.assert_array_equal(c.cpu().numpy(), rc)


@pytest.mark.parametrize("case", ["mixed", "random"])
@pytest.mark.parametrize("H,H_kv", [(4, 2), (3, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_forward_matches_dequantised_oracle(attn, case, H, H_kv, causal):
    cu = _cu(case)
    q, k, v = _packed(72 + H_kv, cu, H, H_kv)
    signs = workloads.random_signs(8, D)
    (q8, k8, v8), (qd, kd, vd), max_len = _quant_gpu(attn, q, k, v, cu, signs)
    o, lse = attn.attn_fwd_fp8_varlen(q8, k8, v8, qd, kd, vd, torch.from_numpy(cu).to(dev()),
                                      max_len, causal=causal, softmax_scale=1 / np.sqrt(D))
    check_status(attn)
    deq = [_dequant(c.cpu().numpy(), s.cpu().numpy(), cu)
           for c, s in ((q8, qd), (k8, kd), (v8, vd))]
    ref_o, ref_l = oracle.attention_forward_varlen(*deq, cu, 1 / np.sqrt(D), causal)
    got = o.float().cpu().numpy()
    diff = got - ref_o
    assert np.sqrt(np.mean(diff ** 2)) <= 1e-2 * max(1.0, np.sqrt(np.mean(ref_o ** 2)))
    assert np.abs(diff).max() <= 0.25 * max(1.0, np.abs(ref_o).max())
    lse_c = lse.cpu().numpy()
    np.testing.assert_allclose(lse_c, ref_l, atol=2e-3)


@pytest.mark.parametrize("causal", [False, True])
def test_single_sequence_equals_fixed_length(attn, causal):
    """One packed sequence is the fixed-length problem with B = 1: the packed
    and the fixed-length FP8 paths give identical bits."""
    N, H = 640, 2
    cu = np.array([0, N], dtype=np.int32)
    q, k, v = _packed(74, cu, H, H)
    (q8, k8, v8), (qd, kd, vd), _ = _quant_gpu(attn, q, k, v, cu)
    o, lse = attn.attn_fwd_fp8_varlen(q8, k8, v8, qd, kd, vd, torch.from_numpy(cu).to(dev()), N,
                                      causal=causal)
    bhnd = [t.permute(1, 0, 2).unsqueeze(0).contiguous() for t in (q8, k8, v8)]
    o2, lse2 = attn.attn_fwd_fp8(*bhnd, qd, kd, vd, causal=causal)
    check_status(attn)
    assert torch.equal(o, o2[0].permute(1, 0, 2))
    assert torch.equal(lse, lse2[0])


def test_inconsistent_offsets_are_reported(attn):
    cu = np.array([0, 100, 400], dtype=np.int32)       # second sequence: 300 > max_seqlen
    q, k, v = _packed(75, cu, 2, 2)
    attn.attn_fp8_quantize_varlen(*(torch.from_numpy(x).to(dev()) for x in (q, k, v)),
                                  torch.from_numpy(cu).to(dev()), 200)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_get_device_status() == 0
