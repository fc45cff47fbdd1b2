"""Paged decode over an e4m3 cache: CUDA path (through the C ABI) vs the float64
oracle on the same codes and descales.

Two comparisons per case:
* against exact attention of the query the kernel actually multiplies (each
  row transformed when keys were, then quantised to e4m3 with its own descale,
  by the oracle's quantiser): what is left is the kernel's own error, P rounded
  to e4m3 for the P V product and float32 accumulation.  The RMSE bar is the
  RMS error of rounding every weight independently with a relative error
  uniform within the e4m3 half step (|delta| <= 2^-4, RMS 2^-4 / sqrt(3)):
  2^-4 / sqrt(3) * sqrt(mean_i sum_j P_ij^2 V_j^2), with sum_j P_ij^2 V_j^2
  taken from the oracle as exact attention with doubled scores over squared
  values, times exp(LSE(2 s) - 2 LSE(s)); LSE does not depend on that rounding;
* against exact attention of the unquantised query over the cache: the query
  is rounded to the relative precision of the cached keys (e4m3, with a finer
  per-row scale), so the kernel's total error is of the order of the error of
  storing the cache in e4m3 (exact attention over the cache vs over the
  float32 keys and values it was quantised from; 0.6 to 1.2 times it on these
  cases, computed with the oracle); the bar is 1.5 times that storage error,
  and on unscaled N(0, 1) caches also the FP8 RMSE bar of the forward."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import FP8_RMSE, check_status, dev, guarded, lib

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def attn():
    return lib()


def _cache(seed, lens, page_size, H_kv, spread=True):
    kc, vc, table = workloads.paged_cache(seed, lens, page_size, H_kv, D)
    if spread:   # a different magnitude per (page, head), so descales differ
        rng = np.random.default_rng(seed + 100)
        kc = kc * rng.uniform(0.25, 4.0, (kc.shape[0], 1, H_kv, 1)).astype(np.float32)
        vc = vc * rng.uniform(0.25, 4.0, (vc.shape[0], 1, H_kv, 1)).astype(np.float32)
    return kc, vc, table


def _run(attn, lens, page_size, H, H_kv, n_q, causal, signs=None, dtype="bf16", seed=80,
         max_seqlen=None, spread=True, light=False):
    kc, vc, table = _cache(seed, lens, page_size, H_kv, spread)
    k8, kd = oracle.quantize_paged_cache(kc, signs)
    v8, vd = oracle.quantize_paged_cache(vc)
    B = len(lens)
    tq = workloads.round_to(workloads.normal(seed + 1, (B, H, n_q, D)), dtype)
    scale = 1 / np.sqrt(D)
    o, co = guarded((B, H, n_q, D), tq.dtype, -7.0)
    lse, cl = guarded((B, H, n_q), torch.float32, -7.0)
    mx = max(max(lens), 1) if max_seqlen is None else max_seqlen
    ts = None if signs is None else torch.from_numpy(signs.astype(np.float32)).to(dev())
    attn.attn_decode_paged_fp8(tq.to(dev()), torch.from_numpy(k8).to(dev()),
                               torch.from_numpy(v8).to(dev()), torch.from_numpy(kd).to(dev()),
                               torch.from_numpy(vd).to(dev()), torch.from_numpy(table).to(dev()),
                               torch.tensor(lens, dtype=torch.int32, device=dev()), mx,
                               causal=causal, softmax_scale=scale, hadamard_signs=ts, o=o, lse=lse)
    check_status(attn)
    co()
    cl()
    q64 = workloads.as_f64(tq)
    # the query the kernel multiplies: transformed, then e4m3 per row
    qt = q64 if signs is None else oracle.incoherent_transform(q64, signs)
    q8, qd = oracle.quantize_e4m3_blocks(qt, block_rows=1)
    q_used = oracle.dequantize_e4m3_blocks(q8, qd, block_rows=1)
    ref_used = oracle.attention_decode_paged_fp8(q_used, k8, v8, kd, vd, table, lens, scale, causal)
    ref_exact = ref_float = None
    if not light:
        ref_exact = oracle.attention_decode_paged_fp8(q64, k8, v8, kd, vd, table, lens, scale, causal,
                                                      signs)
        ref_float, _ = oracle.attention_decode_paged(q64, kc, vc, table, lens, scale, causal)
    # sum_j P_ij^2 V_j^2 of the query the kernel multiplies
    kdq = oracle.dequantize_paged_cache(k8, kd)
    vdq = oracle.dequantize_paged_cache(v8, vd)
    o2, l2 = oracle.attention_decode_paged(q_used, kdq, vdq ** 2, table, lens, 2 * scale, causal)
    l1 = ref_used[1]
    seen = np.isfinite(l1)
    expo = np.subtract(l2, 2 * l1, out=np.zeros_like(l1), where=seen)
    p2v2 = o2 * np.where(seen, np.exp(expo), 0.0)[..., None]
    bar = 2.0 ** -4 / np.sqrt(3) * np.sqrt(np.mean(p2v2))
    return o, lse, ref_used, ref_exact, ref_float, spread, bar


def _check(o, lse, ref_used, ref_exact, ref_float, spread, bar):
    got = o.float().cpu().numpy().astype(np.float64)
    lse_c = lse.cpu().numpy().astype(np.float64)
    ro, rl = ref_used
    seen = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lse_c), seen)
    assert np.all(np.isfinite(got))
    diff = got - ro
    assert np.sqrt(np.mean(diff ** 2)) <= bar, (np.sqrt(np.mean(diff ** 2)), bar)
    assert np.abs(diff).max() <= 0.25 * max(1.0, float(np.abs(ro).max()))
    np.testing.assert_allclose(lse_c[seen], rl[seen], atol=2e-3)
    assert np.all(got[~seen] == 0)
    if ref_exact is None:
        return
    eo = ref_exact[0]
    total = np.sqrt(np.mean((got - eo) ** 2))
    storage = np.sqrt(np.mean((eo - ref_float) ** 2))
    assert total <= 1.5 * storage, (total, storage)
    if not spread:
        assert total <= FP8_RMSE


@pytest.mark.parametrize("page_size", [16, 64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_page_sizes(attn, page_size, causal):
    _check(*_run(attn, [1, 127, 128, 129, 700], page_size, 8, 2, 2, causal))


@pytest.mark.parametrize("H,H_kv,n_q", [(32, 8, 1), (8, 1, 4), (4, 4, 1), (16, 2, 16)])
def test_heads_and_query_tokens(attn, H, H_kv, n_q):
    _check(*_run(attn, [300, 1025, 64], 32, H, H_kv, n_q, True, seed=81))


@pytest.mark.parametrize("H,H_kv,n_q", [(32, 2, 1), (12, 2, 2), (6, 2, 5), (34, 2, 1), (40, 2, 1),
                                         (64, 2, 1), (16, 2, 4), (66, 2, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_query_rows_per_head(attn, H, H_kv, n_q, causal):
    # G n_q = 16, 12 and 15 query rows per key/value head run with the keys on
    # the MMA's M side and N = 16; 17, 20, 32 (as 16 query heads x 2 tokens and
    # as 8 x 4) and 33 rows with the query rows on M
    _check(*_run(attn, [300, 1025, 64], 64, H, H_kv, n_q, causal, seed=92))


def test_transformed_keys_sixteen_rows(attn):
    signs = workloads.random_signs(8, D)
    _check(*_run(attn, [200, 700], 128, 32, 2, 1, True, signs=signs, seed=93))


def test_timed_config_full_size(attn):
    """The benchmark's decode step at full size: 16 sequences of 8192 cached
    tokens, H = 32 query heads on H_kv = 8 (4 query rows per key/value head),
    pages of 256 in a seeded random order, one query token, causal: every
    output row and LSE against the oracle, within the kernel's own error bar."""
    _check(*_run(attn, [8192] * 16, 256, 32, 8, 1, True, seed=94, light=True))


@pytest.mark.parametrize("page_size", [16, 256])
def test_transformed_keys(attn, page_size):
    signs = workloads.random_signs(7, D)
    _check(*_run(attn, [200, 513], page_size, 8, 2, 2, True, signs=signs, seed=82))


def test_long_sequences_split(attn):
    _check(*_run(attn, [9000, 20000], 64, 8, 2, 1, True, seed=83))


def test_long_splits_reuse_every_ring_slot(attn):
    # 19 sequences x 8 key/value heads fill the 152 SMs once, so each CTA takes
    # a whole sequence: 16 tiles, 32 ring items, every slot used two or three times
    _check(*_run(attn, [2048] * 19, 64, 8, 8, 1, True, seed=89))


def test_fp16_and_empty_sequence(attn):
    _check(*_run(attn, [0, 513, 2], 16, 4, 2, 3, True, dtype="fp16", seed=84))


def test_more_queries_than_keys_and_larger_max_seqlen(attn):
    _check(*_run(attn, [2, 300], 16, 4, 4, 4, True, seed=85, max_seqlen=5000))


def test_uniform_descales(attn):
    _check(*_run(attn, [640, 77], 128, 8, 2, 1, False, seed=86, spread=False))


def test_bad_page_is_reported(attn):
    lens = [200]
    kc, vc, table = _cache(87, lens, 64, 2)
    table[0, 1] = kc.shape[0] + 7                       # out of the cache
    k8, kd = oracle.quantize_paged_cache(kc)
    v8, vd = oracle.quantize_paged_cache(vc)
    tq = workloads.round_to(workloads.normal(88, (1, 4, 1, D)), "bf16")
    attn.attn_decode_paged_fp8(tq.to(dev()), torch.from_numpy(k8).to(dev()),
                               torch.from_numpy(v8).to(dev()), torch.from_numpy(kd).to(dev()),
                               torch.from_numpy(vd).to(dev()), torch.from_numpy(table).to(dev()),
                               torch.tensor(lens, dtype=torch.int32, device=dev()), 200)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_get_device_status() == 0
