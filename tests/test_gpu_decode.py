"""Paged decode parity: CUDA path (through the C ABI) vs the float64 oracle on
the same bf16/fp16 bits."""
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


def _run(attn, lens, page_size, H, H_kv, n_q, d, causal, dtype="bf16", seed=60, max_seqlen=None):
    kc, vc, table = workloads.paged_cache(seed, lens, page_size, H_kv, d)
    q = workloads.normal(seed + 1, (len(lens), H, n_q, d))
    tq, tk, tv = (workloads.round_to(x, dtype) for x in (q, kc, vc))
    B = len(lens)
    scale = 1 / np.sqrt(d)
    o, co = guarded((B, H, n_q, d), tq.dtype, -7.0)
    lse, cl = guarded((B, H, n_q), torch.float32, -7.0)
    mx = max(max(lens), 1) if max_seqlen is None else max_seqlen
    attn.attn_decode_paged(tq.to(dev()), tk.to(dev()), tv.to(dev()),
                           torch.from_numpy(table).to(dev()),
                           torch.tensor(lens, dtype=torch.int32, device=dev()), mx, causal=causal,
                           softmax_scale=scale, o=o, lse=lse)
    check_status(attn)
    co()
    cl()
    ref_o, ref_l = oracle.attention_decode_paged(*(workloads.as_f64(t) for t in (tq, tk, tv)),
                                                 table, lens, scale, causal)
    return o, lse, ref_o, ref_l


def _close(o, lse, ref_o, ref_l):
    lse_c = lse.cpu().numpy().astype(np.float64)
    seen = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lse_c), seen)
    ref_l = np.where(seen, ref_l, 0.0)
    lse_t = torch.from_numpy(np.where(seen, lse_c, 0.0)).float()
    assert_fwd_close(o, lse_t, ref_o, ref_l)


@pytest.mark.parametrize("page_size", [8, 16, 64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_page_sizes(attn, page_size, causal):
    _close(*_run(attn, [1, 127, 128, 129, 700], page_size, 8, 2, 2, 128, causal))


@pytest.mark.parametrize("H,H_kv,n_q", [(32, 8, 1), (8, 1, 4), (4, 4, 1), (16, 2, 16)])
@pytest.mark.parametrize("d", [64, 128])
def test_heads_and_query_tokens(attn, H, H_kv, n_q, d):
    _close(*_run(attn, [300, 1025, 64], 32, H, H_kv, n_q, d, True, seed=61))


def test_long_sequences_split(attn):
    """Long contexts take several key-range splits, merged by the combine kernel."""
    _close(*_run(attn, [9000, 20000], 64, 8, 2, 1, 128, True, seed=62))


def test_fp16_and_empty_sequence(attn):
    _close(*_run(attn, [0, 513, 2], 16, 4, 2, 3, 128, True, dtype="fp16", seed=63))


def test_larger_max_seqlen_and_more_queries_than_keys(attn):
    # n_q = 4 > len = 2: the first two query rows see no key (O = 0, L = -inf)
    _close(*_run(attn, [2, 300], 16, 4, 4, 4, 64, True, seed=64, max_seqlen=5000))


def test_bad_page_is_reported(attn):
    lens = [200]
    kc, vc, table = workloads.paged_cache(65, lens, 64, 2, 128)
    table[0, 1] = kc.shape[0] + 7                       # out of the cache
    q = workloads.normal(66, (1, 4, 1, 128))
    tq, tk, tv = (workloads.round_to(x, "bf16") for x in (q, kc, vc))
    attn.attn_decode_paged(tq.to(dev()), tk.to(dev()), tv.to(dev()), torch.from_numpy(table).to(dev()),
                           torch.tensor(lens, dtype=torch.int32, device=dev()), 200)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_get_device_status() == 0
