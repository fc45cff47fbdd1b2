"""FP8 (e4m3) block quantisation and incoherent processing -- TEST INFRASTRUCTURE.

Sources (page title, then section):

* "FlashAttention-3: Hopper Asynchrony and FP8 Attention", "FP8 accuracy
  controls": block quantisation keeps one scale per Q, K or V block;
  incoherent processing multiplies Q and K by the same orthogonal matrix M
  before quantisation, so (QM)(KM)^T = QK^T; M is a product of random sign
  diagonals and a Hadamard matrix (O(d log d) to apply).
* "FlashAttention 3 Hardware Acceleration: ...", "FP8 Accumulation": the
  scaling factors are FP32.

The e4m3 encoder below is written from the OCP 8-bit floating point format
definition (E4M3, "fn" variant): 1 sign bit, 4 exponent bits with bias 7,
3 mantissa bits, no infinities, the all-ones pattern S.1111.111 is NaN, the
largest finite magnitude is 1.75 * 2^8 = 448, the smallest normal is 2^-6 and
subnormals are m/8 * 2^-6 (down to 2^-9).

Readings where the pages are silent (each one is listed in the design notes):
* A block is one (b, h) head and 128 consecutive rows, over all d columns.
  One scale per block fits one descale per tile of the score contraction.
* descale = float32(amax) / 448 in float32; amax = 0 gives descale = 1.
* code = e4m3(round-to-nearest-even(x / descale)), with x / descale an
  IEEE float32 division and magnitudes >= 448 saturated to 448.
* M = diag(s) H_d / sqrt(d): s is one +-1 vector shared by Q and K and by all
  heads; H_d is the Sylvester Hadamard matrix in natural order.  V is not
  transformed.
* Per-tensor mode (the comparator in the outlier test) uses one scale for the
  whole tensor and no transform.
* Rotary embedding (the pages say only that the Hadamard transform can be
  fused with it): applied to Q and K before the transform, from caller tables
  cos, sin [N, d/2]; the pair (x_i, x_{i+d/2}) at position n is rotated by the
  angle whose cosine and sine are cos[n, i], sin[n, i].  V is not rotated.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_MIN_SUBNORMAL = 2.0 ** -9
E4M3_NAN = 0x7F


def e4m3_encode(x) -> np.ndarray:
    """Round values to e4m3 codes (uint8): nearest, ties to even, saturating."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.uint8) << 7
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, E4M3_MAX))
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < E4M3_MIN_NORMAL
    # subnormal range: multiples of 2^-9; a count of 8 is exactly the smallest
    # normal, whose code is also 8 (exponent field 1, mantissa 0)
    code = np.where(sub, np.rint(a / E4M3_MIN_SUBNORMAL).astype(np.int64), code)
    # normal range: a = 2^e * (1 + f/8)
    frac, ex = np.frexp(np.where(sub, 1.0, a))     # a = frac * 2^ex, frac in [0.5, 1)
    e = ex.astype(np.int64) - 1
    mant = np.rint((frac * 2.0 - 1.0) * 8.0).astype(np.int64)
    carry = mant == 8
    e = np.where(carry, e + 1, e)
    mant = np.where(carry, 0, mant)
    normal_code = ((e + 7) << 3) | mant
    code = np.where(sub, code, normal_code)
    code = code.astype(np.uint8) | sign
    return np.where(nan, np.uint8(E4M3_NAN) | sign, code).astype(np.uint8)


def e4m3_decode(code) -> np.ndarray:
    """Value (float64) of e4m3 codes; NaN for the S.1111.111 patterns."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6,
                   (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return s * val


def sylvester_hadamard(d: int) -> np.ndarray:
    """The d x d Hadamard matrix of Sylvester's construction (d a power of 2)."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def incoherent_transform(x, signs) -> np.ndarray:
    """x M with M = diag(signs) H_d / sqrt(d), applied to the last axis (float64)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    m = np.asarray(signs, dtype=np.float64)[:, None] * sylvester_hadamard(d) / np.sqrt(d)
    return x @ m


def rotary_embed(x, cos, sin) -> np.ndarray:
    """Rotate pairs (x_i, x_{i+d/2}) of every row of a [..., N, d] array by the
    per-position tables cos, sin [N, d/2] (float64)."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(cos, dtype=np.float64)
    s = np.asarray(sin, dtype=np.float64)
    h = x.shape[-1] // 2
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def quantize_e4m3_blocks(x, block_rows: int = 128, per_tensor: bool = False,
                         signs=None, rope=None):
    """Quantise a [B, H, N, d] tensor to e4m3 codes with float32 descales.

    Steps, in order: optional rotary embedding (rope = (cos, sin) tables) and
    incoherent transform (float64, then rounded to float32, the precision the
    GPU pre-pass holds its values in); amax per
    block (or per tensor); descale = amax / 448 in float32 (1 when amax is 0);
    code = e4m3(x / descale) with a float32 division.

    Returns (codes uint8 [B, H, N, d], descale float32 [B, H, ceil(N/block_rows)]).
    In per-tensor mode every descale entry holds the same value.
    """
    x = np.asarray(x)
    if rope is not None:
        x = rotary_embed(x, *rope)
    if signs is not None:
        x = incoherent_transform(x, signs)
    x = x.astype(np.float32)
    B, H, N, d = x.shape
    nblk = -(-N // block_rows)
    pad = nblk * block_rows - N
    absx = np.abs(x)
    if per_tensor:
        amax = np.full((B, H, nblk), absx.max() if absx.size else 0.0, dtype=np.float32)
    else:
        padded = np.concatenate([absx, np.zeros((B, H, pad, d), np.float32)], axis=2)
        amax = padded.reshape(B, H, nblk, block_rows * d).max(axis=3).astype(np.float32)
    descale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    rows_descale = np.repeat(descale, block_rows, axis=2)[:, :, :N, None]
    scaled = (x / rows_descale).astype(np.float32)           # IEEE float32 division
    return e4m3_encode(scaled), descale


def dequantize_e4m3_blocks(codes, descale, block_rows: int = 128) -> np.ndarray:
    """float64 values code * descale of a block-quantised [B, H, N, d] tensor."""
    codes = np.asarray(codes)
    N = codes.shape[2]
    rows_descale = np.repeat(np.asarray(descale, np.float64), block_rows, axis=2)[:, :, :N, None]
    return e4m3_decode(codes) * rows_descale
