"""CPU oracle for exact tiled attention -- TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 NumPy restatements of what the GPU path computes, written
from the pages on FlashAttention-3 and from the definition of softmax
attention.  There is no tiling, no online softmax and no fusion here: every
function forms the full N x N score matrix, exactly as standard (materialised)
attention does.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The CUDA library never calls it,
and it imports nothing from the CUDA package.

Every function here is pinned by ``tests/test_oracle_*.py`` against closed
forms, invariants, independent library routines, finite differences or
hand-derived fixtures under ``tests/golden/``.  No function is parity-unpinned.
"""
from .attention import (attention_forward, attention_backward, attention_probs,
                        attention_forward_rows,
                        attention_forward_head, attention_backward_head)
from .fp8 import (E4M3_MAX, e4m3_encode, e4m3_decode, sylvester_hadamard,
                  incoherent_transform, quantize_e4m3_blocks, dequantize_e4m3_blocks,
                  rotary_embed)
from .varlen import (attention_forward_gqa, attention_backward_gqa,
                     attention_forward_varlen, attention_backward_varlen)
from .decode import (attention_decode_paged, attention_decode_paged_fp8,
                     dequantize_paged_cache, quantize_paged_cache)

__all__ = [
    "attention_forward", "attention_backward", "attention_probs", "attention_forward_rows",
    "attention_forward_head", "attention_backward_head",
    "E4M3_MAX", "e4m3_encode", "e4m3_decode", "sylvester_hadamard",
    "incoherent_transform", "quantize_e4m3_blocks", "dequantize_e4m3_blocks", "rotary_embed",
    "attention_forward_gqa", "attention_backward_gqa",
    "attention_forward_varlen", "attention_backward_varlen", "attention_decode_paged",
    "attention_decode_paged_fp8", "quantize_paged_cache", "dequantize_paged_cache",
]
