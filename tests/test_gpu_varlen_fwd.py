"""Forward parity for grouped-query attention and packed variable-length
batches: CUDA path (through the C ABI) vs the float64 CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_fwd_close, check_status, dev, guarded, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    return lib()


def _bf16(seed, shape, count, dtype="bf16"):
    xs = workloads.normal(seed, shape, count)
    xs = xs if count > 1 else [xs]
    return [workloads.round_to(x, dtype) for x in xs]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("H,H_kv", [(4, 2), (6, 1), (8, 8)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_forward(attn, d, H, H_kv, causal):
    B, N = 2, 300
    (tq,) = _bf16(40 + d + H_kv, (B, H, N, d), 1)
    tk, tv = _bf16(50 + d + H_kv, (B, H_kv, N, d), 2)
    scale = 1 / np.sqrt(d)
    o, co = guarded((B, H, N, d), tq.dtype, -7.0)
    lse, cl = guarded((B, H, N), torch.float32, -7.0)
    attn.attn_fwd_gqa(tq.to(dev()), tk.to(dev()), tv.to(dev()), causal=causal,
                      softmax_scale=scale, o=o, lse=lse)
    check_status(attn)
    co()
    cl()
    ref_o, ref_l = oracle.attention_forward_gqa(*(workloads.as_f64(t) for t in (tq, tk, tv)),
                                                scale, causal)
    assert_fwd_close(o, lse, ref_o, ref_l)


def _varlen_case(name):
    """cu_seqlens of the named packed batch (int32 numpy)."""
    if name == "mixed":       # empty, length 1, tile-ragged and multi-tile sequences
        return np.array([0, 0, 1, 128, 257, 300, 815], dtype=np.int32)
    if name == "single":
        return np.array([0, 640], dtype=np.int32)
    if name == "random":
        cu, _ = workloads.varlen_lengths(61, 6, 700)
        return cu
    raise ValueError(name)


def _run_varlen(attn, cu, H, H_kv, d, causal, dtype="bf16", seed=70):
    total = int(cu[-1])
    (tq,) = _bf16(seed, (total, H, d), 1, dtype)
    tk, tv = _bf16(seed + 1, (total, H_kv, d), 2, dtype)
    scale = 1 / np.sqrt(d)
    max_len = int(np.max(np.diff(cu))) if len(cu) > 1 else 1
    o, co = guarded((total, H, d), tq.dtype, -7.0)
    lse, cl = guarded((H, total), torch.float32, -7.0)
    attn.attn_fwd_varlen(tq.to(dev()), tk.to(dev()), tv.to(dev()),
                         torch.from_numpy(cu).to(dev()), max(max_len, 1), causal=causal,
                         softmax_scale=scale, o=o, lse=lse)
    check_status(attn)
    co()
    cl()
    ref_o, ref_l = oracle.attention_forward_varlen(*(workloads.as_f64(t) for t in (tq, tk, tv)),
                                                   cu, scale, causal)
    return o, lse, ref_o, ref_l


@pytest.mark.parametrize("case", ["mixed", "single", "random"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_forward(attn, case, d, causal):
    cu = _varlen_case(case)
    assert_fwd_close(*_run_varlen(attn, cu, 4, 2, d, causal))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_varlen_forward_dtypes_mqa(attn, dtype):
    cu = _varlen_case("mixed")
    assert_fwd_close(*_run_varlen(attn, cu, 3, 1, 128, True, dtype))


def test_varlen_larger_max_seqlen_is_allowed(attn):
    """max_seqlen above the true longest sequence only enlarges the grid."""
    cu = _varlen_case("mixed")
    total, H, d = int(cu[-1]), 2, 128
    (tq,) = _bf16(80, (total, H, d), 1)
    tk, tv = _bf16(81, (total, H, d), 2)
    o, lse = attn.attn_fwd_varlen(tq.to(dev()), tk.to(dev()), tv.to(dev()),
                                  torch.from_numpy(cu).to(dev()), 2000, causal=False)
    check_status(attn)
    ref_o, ref_l = oracle.attention_forward_varlen(*(workloads.as_f64(t) for t in (tq, tk, tv)),
                                                   cu, 1 / np.sqrt(d), False)
    assert_fwd_close(o, lse, ref_o, ref_l)


def test_varlen_inconsistent_offsets_are_reported(attn):
    """A sequence longer than max_seqlen is skipped on the device and reported
    as an invalid argument; nothing is written outside the outputs."""
    cu = np.array([0, 100, 400], dtype=np.int32)     # second sequence has 300 tokens
    total, H, d = 400, 2, 64
    (tq,) = _bf16(82, (total, H, d), 1)
    tk, tv = _bf16(83, (total, H, d), 2)
    o, co = guarded((total, H, d), tq.dtype, -7.0)
    lse, cl = guarded((H, total), torch.float32, -7.0)
    attn.attn_fwd_varlen(tq.to(dev()), tk.to(dev()), tv.to(dev()),
                         torch.from_numpy(cu).to(dev()), 200, causal=False, o=o, lse=lse)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_ERR_INVALID_ARG
    assert "cu_seqlens" in attn.attn_last_error()
    co()
    cl()
    assert attn.attn_get_device_status() == 0    # the status word was cleared
