"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and rounds them to the storage dtype
the kernels read.  It holds none of the attention arithmetic, so both the
CPU oracle (``oracle/``) and the CUDA path (``exact_tiled_attention_25_gb300``)
can take their inputs from it without sharing any computation.

Shapes follow the benchmark setup of "FlashAttention-3: Hopper Asynchrony and
FP8 Attention" (section "How we know: H100 attention benchmarks": random
inputs, 16K total tokens, head dimensions 64/128/256) and the FP8
outlier-stress test of the same page (section "FP8 accuracy controls").  The
page does not give the outlier distribution; the one used here is N(0, 1) on
every entry plus an independent N(0, sigma^2) draw (sigma = 10) on a random
0.1 % of entries.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    """One attention problem: tensors are [B, H, N, d], d fastest."""
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def fwd_flop(self) -> float:
        """4*B*H*N^2*d for the two contractions, halved under the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f


# The five problem families.  Each is a parity case; the long-context one is
# also the timed workload.
TINY_FWD = Workload("tiny_fwd_b1h2n256d64", 1, 2, 256, 64, False, 1)
MID_FWD = Workload("mid_fwd_b4h16n2048d128", 4, 16, 2048, 128, False, 2)
MID_FWD_CAUSAL = Workload("mid_fwd_causal_b4h16n2048d128", 4, 16, 2048, 128, True, 2)
LONG_FWD = Workload("long_fwd_b2h16n8192d128", 2, 16, 8192, 128, False, 3)
LONG_FWD_CAUSAL = Workload("long_fwd_causal_b2h16n8192d128", 2, 16, 8192, 128, True, 3)
# head-dim sweep at 16K tokens and H*d = 2048
LONG_FWD_D64 = Workload("long_fwd_b2h32n8192d64", 2, 32, 8192, 64, False, 3)
LONG_FWD_D256 = Workload("long_fwd_b2h8n8192d256", 2, 8, 8192, 256, False, 3)
FP8_FWD = Workload("fp8_fwd_outlier_b2h16n4096d128", 2, 16, 4096, 128, False, 4)
FP8_HADAMARD_SIGN_SEED = 5
BWD_D128 = Workload("bwd_causal_b2h16n4096d128", 2, 16, 4096, 128, True, 6)
BWD_D64 = Workload("bwd_causal_b2h16n4096d64", 2, 16, 4096, 64, True, 6)


def normal(seed: int, shape, count: int = 1):
    """``count`` float32 arrays of i.i.d. N(0, 1), drawn in order from one generator."""
    rng = np.random.default_rng(seed)
    out = [rng.standard_normal(shape, dtype=np.float32) for _ in range(count)]
    return out if count > 1 else out[0]


def normal_with_outliers(seed: int, shape, count: int = 3, p: float = 1e-3,
                         sigma: float = 10.0):
    """``count`` float32 arrays: N(0,1) everywhere plus N(0, sigma^2) on a
    Bernoulli(p) subset of entries (independent per entry and per array)."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        x = rng.standard_normal(shape, dtype=np.float32)
        hit = rng.random(shape, dtype=np.float32) < p
        extra = rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma)
        out.append(np.where(hit, x + extra, x).astype(np.float32))
    return out if count > 1 else out[0]


def random_signs(seed: int, d: int) -> np.ndarray:
    """d independent +1/-1 entries (float32), equal probability."""
    rng = np.random.default_rng(seed)
    return np.where(rng.random(d) < 0.5, -1.0, 1.0).astype(np.float32)


def round_to(x: np.ndarray, dtype: str):
    """Round float32 values to the 16-bit storage type (round to nearest even).

    Returns a CPU torch tensor of that dtype; its exact values, upcast, are what
    the oracle sees, and its bits are what the GPU reads.
    """
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    if dtype == "fp16":
        return t.to(torch.float16)
    raise ValueError(f"unknown 16-bit dtype {dtype!r}")


def as_f64(t) -> np.ndarray:
    """Exact float64 copy of a CPU torch tensor (any float dtype)."""
    return t.double().numpy()


def varlen_lengths(seed: int, B: int, max_len: int, min_len: int = 0):
    """B sequence lengths drawn uniformly from [min_len, max_len] (int32 offsets
    cu_seqlens [B + 1] and the lengths)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(min_len, max_len + 1, size=B).astype(np.int64)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return cu, lens


def rope_tables(N: int, d: int, base: float = 10000.0):
    """float32 rotary tables cos, sin [N, d/2] of the common frequency ladder
    theta_i = base^(-2i/d) at positions 0..N-1 (an input, like the Hadamard
    signs: the kernels and the oracle both take the tables as given)."""
    i = np.arange(d // 2, dtype=np.float64)
    ang = np.arange(N, dtype=np.float64)[:, None] * base ** (-2.0 * i / d)[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def paged_cache(seed: int, seq_lens, page_size: int, H_kv: int, d: int, spare_pages: int = 3):
    """A paged key/value cache holding sequences of the given lengths: float32
    caches [num_pages, page_size, H_kv, d] of N(0,1) values and an int32 block
    table [B, max_pages] whose pages are a seeded random permutation (plus
    unused spare pages); unused table entries are -1."""
    rng = np.random.default_rng(seed)
    need = [-(-int(n) // page_size) for n in seq_lens]
    max_pages = max(max(need), 1)
    num_pages = sum(need) + spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((len(seq_lens), max_pages), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    kc = rng.standard_normal((num_pages, page_size, H_kv, d), dtype=np.float32)
    vc = rng.standard_normal((num_pages, page_size, H_kv, d), dtype=np.float32)
    return kc, vc, table
