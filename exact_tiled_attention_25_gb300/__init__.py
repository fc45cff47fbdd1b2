"""Exact tiled softmax attention for NVIDIA GB300 (sm_103a).

A thin Python binding over the C ABI of ``libattn_gb300.so``.  Each function
here has the name of the C entry point it calls and only marshals arguments:
it checks tensor metadata, allocates outputs with PyTorch (device memory and
streams are PyTorch's job) and passes raw pointers.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback, and a missing library raises.

Tensors are [B, H, N, d], contiguous; the ``*_varlen`` calls take a packed
batch [total, H, d] with int32 sequence offsets ``cu_seqlens`` [B + 1].  Inputs
on the CPU are accepted: they are copied to the current CUDA device on the
current stream, and the outputs are copied back to the CPU.
"""
from __future__ import annotations

import math

import torch

from . import _lib

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_ARCH = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5

_DTYPES = {torch.bfloat16: 0, torch.float16: 1}

ATTN_SCHED_DEFAULT = 0
ATTN_SCHED_ONE_TILE = 1
ATTN_SCHED_EAGER_RESCALE = 2
ATTN_SCHED_EXP2_POLY = 4
ATTN_SCHED_EXP2_NONE = 8


def ATTN_SCHED_EXP2_EIGHTHS(k: int) -> int:
    """Schedule value for k of every 8 FP8-forward exponentials on the FMA pipe (k = 1..4)."""
    return ATTN_SCHED_EXP2_POLY | (int(k) << 8)


__all__ = ["AttnError", "attn_fwd", "attn_fwd_schedule", "attn_fwd_gqa", "attn_fwd_varlen", "attn_bwd",
           "attn_bwd_gqa", "attn_bwd_varlen", "attn_bwd_varlen_workspace_size",
           "attn_bwd_workspace_size",
           "attn_fp8_quantize", "attn_fp8_quantize_gqa", "attn_fp8_quantize_rope", "attn_fwd_fp8",
           "attn_fwd_fp8_gqa", "attn_fwd_fp8_schedule", "attn_selftest_exp2", "attn_fp8_quantize_varlen", "attn_fwd_fp8_varlen",
           "attn_fp8_quantize_bf16", "attn_fp8_quantize_ex",
           "attn_decode_paged", "attn_decode_paged_fp8", "attn_decode_workspace_size",
           "attn_get_device_status",
           "attn_status_string", "attn_last_error", "load_library"]


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = _lib.load()
        detail = lib.attn_last_error().decode()
        super().__init__(f"{where}: {lib.attn_status_string(code).decode()} ({code})"
                         + (f": {detail}" if detail else ""))
        self.code = code


def load_library():
    """Load libattn_gb300.so (raises if it is not built)."""
    return _lib.load()


def _check(code: int, where: str):
    if code != ATTN_OK:
        raise AttnError(code, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _shape4(t, name):
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, H, N, d]")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return tuple(t.shape)


def _to_device(ts):
    """Copy CPU inputs to the current device; report whether results go back."""
    on_host = all(t.device.type == "cpu" for t in ts)
    if on_host:
        dev = torch.device("cuda", torch.cuda.current_device())
        ts = [t.to(dev, non_blocking=True) for t in ts]
    return ts, on_host


def attn_status_string(code: int) -> str:
    return _lib.load().attn_status_string(code).decode()


def attn_last_error() -> str:
    return _lib.load().attn_last_error().decode()


def attn_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return _lib.load().attn_get_device_status(_stream(stream))


def attn_fwd(q, k, v, causal: bool = False, softmax_scale: float | None = None,
             o=None, lse=None, stream=None):
    """O, LSE = attention(q, k, v) in bf16/fp16; LSE is float32 [B, H, N]."""
    lib = _lib.load()
    (q, k, v), host = _to_device([q, k, v])
    B, H, N, d = _shape4(q, "q")
    if _shape4(k, "k") != (B, H, N, d) or _shape4(v, "v") != (B, H, N, d):
        raise ValueError("q, k, v must have the same shape")
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must all be bfloat16 or all float16")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    code = lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                        int(bool(causal)), scale, _DTYPES[q.dtype], _stream(stream))
    _check(code, "attn_fwd")
    if host:
        return o.cpu(), lse.cpu()
    return o, lse


def attn_fwd_schedule(q, k, v, schedule: int, causal: bool = False,
                      softmax_scale: float | None = None, o=None, lse=None, stream=None):
    """attn_fwd with a schedule variant (ATTN_SCHED_* flags), for measurement."""
    lib = _lib.load()
    (q, k, v), host = _to_device([q, k, v])
    B, H, N, d = _shape4(q, "q")
    if _shape4(k, "k") != (B, H, N, d) or _shape4(v, "v") != (B, H, N, d):
        raise ValueError("q, k, v must have the same shape")
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must all be bfloat16 or all float16")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    code = lib.attn_fwd_schedule(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                 int(bool(causal)), scale, _DTYPES[q.dtype], int(schedule),
                                 _stream(stream))
    _check(code, "attn_fwd_schedule")
    if host:
        return o.cpu(), lse.cpu()
    return o, lse


def attn_fwd_gqa(q, k, v, causal: bool = False, softmax_scale: float | None = None,
                 o=None, lse=None, stream=None):
    """attn_fwd with H_kv = k.shape[1] key/value heads shared by the H query heads."""
    lib = _lib.load()
    (q, k, v), host = _to_device([q, k, v])
    B, H, N, d = _shape4(q, "q")
    Hkv = k.shape[1] if k.dim() == 4 else -1
    if _shape4(k, "k") != (B, Hkv, N, d) or _shape4(v, "v") != (B, Hkv, N, d):
        raise ValueError("k and v must be [B, H_kv, N, d] with q's B, N, d")
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must all be bfloat16 or all float16")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    code = lib.attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                            int(bool(causal)), scale, _DTYPES[q.dtype], _stream(stream))
    _check(code, "attn_fwd_gqa")
    if host:
        return o.cpu(), lse.cpu()
    return o, lse


def _shape3(t, name):
    if t.dim() != 3:
        raise ValueError(f"{name} must be [total, heads, d]")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return tuple(t.shape)


def _cu_seqlens(cu, total):
    if cu.dtype != torch.int32 or cu.dim() != 1 or cu.numel() < 2 or not cu.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int32 vector [B + 1]")
    return cu.numel() - 1


def attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False,
                    softmax_scale: float | None = None, o=None, lse=None, stream=None):
    """Forward over a packed batch: q [total, H, d], k, v [total, H_kv, d],
    cu_seqlens int32 [B + 1]; returns O [total, H, d] and LSE float32 [H, total]."""
    lib = _lib.load()
    (q, k, v, cu_seqlens), host = _to_device([q, k, v, cu_seqlens])
    total, H, d = _shape3(q, "q")
    Hkv = k.shape[1] if k.dim() == 3 else -1
    if _shape3(k, "k") != (total, Hkv, d) or _shape3(v, "v") != (total, Hkv, d):
        raise ValueError("k and v must be [total, H_kv, d] with q's total and d")
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must all be bfloat16 or all float16")
    B = _cu_seqlens(cu_seqlens, total)
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, total), dtype=torch.float32, device=q.device)
    code = lib.attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens),
                               B, int(max_seqlen), total, H, Hkv, d, int(bool(causal)), scale,
                               _DTYPES[q.dtype], _stream(stream))
    _check(code, "attn_fwd_varlen")
    if host:
        return o.cpu(), lse.cpu()
    return o, lse


def attn_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(_lib.load().attn_bwd_workspace_size(B, H, N, d))


def attn_bwd(q, k, v, o, dout, lse, causal: bool = False, softmax_scale: float | None = None,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV of sum(O * dO); o and lse come from attn_fwd."""
    lib = _lib.load()
    (q, k, v, o, dout, lse), host = _to_device([q, k, v, o, dout, lse])
    B, H, N, d = _shape4(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        if _shape4(t, n) != (B, H, N, d) or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    if q.dtype not in _DTYPES:
        raise ValueError("tensors must be bfloat16 or float16")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, H, N]")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = attn_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    code = lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                        workspace.numel() * workspace.element_size(),
                        B, H, N, d, int(bool(causal)), scale, _DTYPES[q.dtype], _stream(stream))
    _check(code, "attn_bwd")
    if host:
        return dq.cpu(), dk.cpu(), dv.cpu()
    return dq, dk, dv


def attn_bwd_gqa(q, k, v, o, dout, lse, causal: bool = False,
                 softmax_scale: float | None = None, dq=None, dk=None, dv=None,
                 workspace=None, stream=None):
    """attn_bwd with k, v (and dk, dv) of H_kv = k.shape[1] heads."""
    lib = _lib.load()
    (q, k, v, o, dout, lse), host = _to_device([q, k, v, o, dout, lse])
    B, H, N, d = _shape4(q, "q")
    Hkv = k.shape[1] if k.dim() == 4 else -1
    for t, n, hh in ((k, "k", Hkv), (v, "v", Hkv), (o, "o", H), (dout, "dout", H)):
        if _shape4(t, n) != (B, hh, N, d) or t.dtype != q.dtype:
            raise ValueError(f"{n} must be [B, {hh}, N, d] in q's dtype")
    if q.dtype not in _DTYPES:
        raise ValueError("tensors must be bfloat16 or float16")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, H, N]")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(attn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8,
                                device=q.device)
    code = lib.attn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                            workspace.numel() * workspace.element_size(),
                            B, H, Hkv, N, d, int(bool(causal)), scale, _DTYPES[q.dtype],
                            _stream(stream))
    _check(code, "attn_bwd_gqa")
    if host:
        return dq.cpu(), dk.cpu(), dv.cpu()
    return dq, dk, dv


def attn_bwd_varlen_workspace_size(B: int, max_seqlen: int, total: int, H: int, d: int) -> int:
    return int(_lib.load().attn_bwd_varlen_workspace_size(B, max_seqlen, total, H, d))


def attn_bwd_varlen(q, k, v, o, dout, lse, cu_seqlens, max_seqlen: int, causal: bool = False,
                    softmax_scale: float | None = None, dq=None, dk=None, dv=None,
                    workspace=None, stream=None):
    """Backward of attn_fwd_varlen: q, o, dout [total, H, d]; k, v [total, H_kv, d];
    lse float32 [H, total]; returns dQ, dK, dV in the inputs' layouts."""
    lib = _lib.load()
    (q, k, v, o, dout, lse, cu_seqlens), host = _to_device([q, k, v, o, dout, lse, cu_seqlens])
    total, H, d = _shape3(q, "q")
    Hkv = k.shape[1] if k.dim() == 3 else -1
    for t, n, hh in ((k, "k", Hkv), (v, "v", Hkv), (o, "o", H), (dout, "dout", H)):
        if _shape3(t, n) != (total, hh, d) or t.dtype != q.dtype:
            raise ValueError(f"{n} must be [total, {hh}, d] in q's dtype")
    if q.dtype not in _DTYPES:
        raise ValueError("tensors must be bfloat16 or float16")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, total) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [H, total]")
    B = _cu_seqlens(cu_seqlens, total)
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(attn_bwd_varlen_workspace_size(B, int(max_seqlen), total, H, d),
                                dtype=torch.uint8, device=q.device)
    code = lib.attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                               _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _ptr(cu_seqlens),
                               B, int(max_seqlen), total, H, Hkv, d, int(bool(causal)), scale,
                               _DTYPES[q.dtype], _stream(stream))
    _check(code, "attn_bwd_varlen")
    if host:
        return dq.cpu(), dk.cpu(), dv.cpu()
    return dq, dk, dv


def attn_fp8_quantize(q, k, v, hadamard_signs=None, per_tensor: bool = False, stream=None):
    """float32 Q, K, V -> (q8, k8, v8) uint8 e4m3 codes and float32 descales."""
    lib = _lib.load()
    ins = [q, k, v] + ([hadamard_signs] if hadamard_signs is not None else [])
    ins, host = _to_device(ins)
    q, k, v = ins[:3]
    signs = ins[3] if hadamard_signs is not None else None
    B, H, N, d = _shape4(q, "q")
    for t, n in ((k, "k"), (v, "v")):
        if _shape4(t, n) != (B, H, N, d) or t.dtype != torch.float32:
            raise ValueError(f"{n} must match q")
    if q.dtype != torch.float32:
        raise ValueError("FP8 pre-pass inputs are float32")
    if signs is not None and (signs.dtype != torch.float32 or signs.numel() != d):
        raise ValueError("hadamard_signs must be d float32 values")
    nblk = (N + 127) // 128
    outs = [torch.empty((B, H, N, d), dtype=torch.uint8, device=q.device) for _ in range(3)]
    desc = [torch.empty((B, H, nblk), dtype=torch.float32, device=q.device) for _ in range(3)]
    code = lib.attn_fp8_quantize(_ptr(q), _ptr(k), _ptr(v), _ptr(signs),
                                 *[_ptr(t) for t in outs], *[_ptr(t) for t in desc],
                                 B, H, N, d, int(bool(per_tensor)), _stream(stream))
    _check(code, "attn_fp8_quantize")
    if host:
        return tuple(t.cpu() for t in outs), tuple(t.cpu() for t in desc)
    return tuple(outs), tuple(desc)


def attn_fp8_quantize_gqa(q, k, v, hadamard_signs=None, per_tensor: bool = False, stream=None):
    """float32 Q [B, H, N, d] and K, V [B, H_kv, N, d] -> e4m3 codes (q8, k8, v8)
    and float32 block descales."""
    lib = _lib.load()
    ins = [q, k, v] + ([hadamard_signs] if hadamard_signs is not None else [])
    ins, host = _to_device(ins)
    q, k, v = ins[:3]
    signs = ins[3] if hadamard_signs is not None else None
    B, H, N, d = _shape4(q, "q")
    _, Hkv, _, _ = _shape4(k, "k")
    for t, n in ((k, "k"), (v, "v")):
        if _shape4(t, n) != (B, Hkv, N, d) or t.dtype != torch.float32:
            raise ValueError("k and v must be float32 [B, H_kv, N, d] with q's B, N, d")
    if q.dtype != torch.float32:
        raise ValueError("FP8 pre-pass inputs are float32")
    if signs is not None and (signs.dtype != torch.float32 or signs.numel() != d):
        raise ValueError("hadamard_signs must be d float32 values")
    nblk = (N + 127) // 128
    outs = [torch.empty((B, h, N, d), dtype=torch.uint8, device=q.device) for h in (H, Hkv, Hkv)]
    desc = [torch.empty((B, h, nblk), dtype=torch.float32, device=q.device) for h in (H, Hkv, Hkv)]
    code = lib.attn_fp8_quantize_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(signs),
                                     *[_ptr(t) for t in outs], *[_ptr(t) for t in desc],
                                     B, H, Hkv, N, d, int(bool(per_tensor)), _stream(stream))
    _check(code, "attn_fp8_quantize_gqa")
    if host:
        return tuple(t.cpu() for t in outs), tuple(t.cpu() for t in desc)
    return tuple(outs), tuple(desc)


def attn_fp8_quantize_rope(q, k, v, rope_cos, rope_sin, hadamard_signs=None, stream=None):
    """attn_fp8_quantize (block mode) with Q and K rotated by the tables
    rope_cos, rope_sin (float32 [N, d/2]) before the Hadamard transform."""
    lib = _lib.load()
    ins = [q, k, v, rope_cos, rope_sin] + ([hadamard_signs] if hadamard_signs is not None else [])
    ins, host = _to_device(ins)
    q, k, v, rc, rs = ins[:5]
    signs = ins[5] if hadamard_signs is not None else None
    B, H, N, d = _shape4(q, "q")
    for t, n in ((k, "k"), (v, "v")):
        if _shape4(t, n) != (B, H, N, d) or t.dtype != torch.float32:
            raise ValueError(f"{n} must match q")
    if q.dtype != torch.float32:
        raise ValueError("FP8 pre-pass inputs are float32")
    for t, n in ((rc, "rope_cos"), (rs, "rope_sin")):
        if t.dtype != torch.float32 or tuple(t.shape) != (N, d // 2) or not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous float32 [N, d/2]")
    if signs is not None and (signs.dtype != torch.float32 or signs.numel() != d):
        raise ValueError("hadamard_signs must be d float32 values")
    nblk = (N + 127) // 128
    outs = [torch.empty((B, H, N, d), dtype=torch.uint8, device=q.device) for _ in range(3)]
    desc = [torch.empty((B, H, nblk), dtype=torch.float32, device=q.device) for _ in range(3)]
    code = lib.attn_fp8_quantize_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(rc), _ptr(rs), _ptr(signs),
                                      *[_ptr(t) for t in outs], *[_ptr(t) for t in desc],
                                      B, H, N, d, _stream(stream))
    _check(code, "attn_fp8_quantize_rope")
    if host:
        return tuple(t.cpu() for t in outs), tuple(t.cpu() for t in desc)
    return tuple(outs), tuple(desc)


def attn_decode_workspace_size(B: int, H: int, H_kv: int, n_q: int, d: int, max_seqlen: int) -> int:
    return int(_lib.load().attn_decode_workspace_size(B, H, H_kv, n_q, d, max_seqlen))


def attn_decode_paged(q, k_cache, v_cache, block_table, seq_lens, max_seqlen: int,
                      causal: bool = True, softmax_scale: float | None = None, o=None, lse=None,
                      workspace=None, stream=None):
    """Decode step: q [B, H, n_q, d] against a paged cache [num_pages, page_size, H_kv, d]
    with an int32 block table [B, max_pages] and int32 seq_lens [B];
    returns O [B, H, n_q, d] and LSE float32 [B, H, n_q]."""
    lib = _lib.load()
    (q, k_cache, v_cache, block_table, seq_lens), host = _to_device(
        [q, k_cache, v_cache, block_table, seq_lens])
    B, H, n_q, d = _shape4(q, "q")
    num_pages, page_size, Hkv, dk = _shape4(k_cache, "k_cache")
    if tuple(v_cache.shape) != (num_pages, page_size, Hkv, dk) or not v_cache.is_contiguous():
        raise ValueError("v_cache must match k_cache")
    if dk != d or q.dtype not in _DTYPES or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise ValueError("q and the caches must share d and dtype (bfloat16 or float16)")
    for t, n, shp in ((block_table, "block_table", 2), (seq_lens, "seq_lens", 1)):
        if t.dtype != torch.int32 or t.dim() != shp or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 tensor of rank {shp}")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table and seq_lens need one entry per sequence")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, n_q), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(attn_decode_workspace_size(B, H, Hkv, n_q, d, int(max_seqlen)),
                                dtype=torch.uint8, device=q.device)
    code = lib.attn_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                 _ptr(seq_lens), _ptr(o), _ptr(lse), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), B, H, Hkv, n_q, d,
                                 num_pages, page_size, block_table.shape[1], int(max_seqlen),
                                 int(bool(causal)), scale, _DTYPES[q.dtype], _stream(stream))
    _check(code, "attn_decode_paged")
    if host:
        return o.cpu(), lse.cpu()
    return o, lse


def attn_decode_paged_fp8(q, k_cache, v_cache, k_descale, v_descale, block_table, seq_lens,
                          max_seqlen: int, causal: bool = True, softmax_scale: float | None = None,
                          hadamard_signs=None, o=None, lse=None, workspace=None, stream=None):
    """Decode step against an e4m3 paged cache: q [B, H, n_q, 128] bf16/fp16,
    caches uint8 [num_pages, page_size, H_kv, 128] with float32 descales
    [num_pages, H_kv]; hadamard_signs (float32 [128]) when the keys were stored
    transformed.  Returns O (q's dtype) and LSE float32 [B, H, n_q]."""
    lib = _lib.load()
    ins = [q, k_cache, v_cache, k_descale, v_descale, block_table, seq_lens]
    if hadamard_signs is not None:
        ins.append(hadamard_signs)
    ins, host = _to_device(ins)
    q, k_cache, v_cache, k_descale, v_descale, block_table, seq_lens = ins[:7]
    signs = ins[7] if hadamard_signs is not None else None
    B, H, n_q, d = _shape4(q, "q")
    num_pages, page_size, Hkv, dk = _shape4(k_cache, "k_cache")
    if tuple(v_cache.shape) != (num_pages, page_size, Hkv, dk) or not v_cache.is_contiguous():
        raise ValueError("v_cache must match k_cache")
    if dk != d or q.dtype not in _DTYPES:
        raise ValueError("q must be bfloat16 or float16 with the caches' d")
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise ValueError("the caches hold uint8 e4m3 codes")
    for t, n in ((k_descale, "k_descale"), (v_descale, "v_descale")):
        if t.dtype != torch.float32 or tuple(t.shape) != (num_pages, Hkv) or not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous float32 [num_pages, H_kv]")
    if signs is not None and (signs.dtype != torch.float32 or signs.numel() != d):
        raise ValueError("hadamard_signs must be d float32 values")
    for t, n, shp in ((block_table, "block_table", 2), (seq_lens, "seq_lens", 1)):
        if t.dtype != torch.int32 or t.dim() != shp or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 tensor of rank {shp}")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table and seq_lens need one entry per sequence")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, n_q), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(attn_decode_workspace_size(B, H, Hkv, n_q, d, int(max_seqlen)),
                                dtype=torch.uint8, device=q.device)
    code = lib.attn_decode_paged_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_descale),
                                     _ptr(v_descale), _ptr(signs), _ptr(block_table),
                                     _ptr(seq_lens), _ptr(o), _ptr(lse), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), B, H, Hkv, n_q,
                                     d, num_pages, page_size, block_table.shape[1],
                                     int(max_seqlen), int(bool(causal)), scale, _DTYPES[q.dtype],
                                     _stream(stream))
    _check(code, "attn_decode_paged_fp8")
    if host:
        return o.cpu(), lse.cpu()
    return o, lse


def attn_fwd_fp8(q8, k8, v8, q_descale, k_descale, v_descale, causal: bool = False,
                 softmax_scale: float | None = None, o=None, lse=None, stream=None):
    """FP8 forward: e4m3 inputs with block descales -> O (bfloat16), LSE (float32)."""
    lib = _lib.load()
    (q8, k8, v8, q_descale, k_descale, v_descale), host = _to_device(
        [q8, k8, v8, q_descale, k_descale, v_descale])
    B, H, N, d = _shape4(q8, "q8")
    for t, n in ((k8, "k8"), (v8, "v8")):
        if _shape4(t, n) != (B, H, N, d) or t.dtype != torch.uint8:
            raise ValueError(f"{n} must match q8 (uint8 e4m3 codes)")
    nblk = (N + 127) // 128
    for t in (q_descale, k_descale, v_descale):
        if t.dtype != torch.float32 or tuple(t.shape) != (B, H, nblk) or not t.is_contiguous():
            raise ValueError("descales must be contiguous float32 [B, H, ceil(N/128)]")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    code = lib.attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_descale), _ptr(k_descale),
                            _ptr(v_descale), _ptr(o), _ptr(lse), B, H, N, d,
                            int(bool(causal)), scale, _stream(stream))
    _check(code, "attn_fwd_fp8")
    if host:
        return o.cpu(), lse.cpu()
    return o, lse


def attn_fwd_fp8_schedule(q8, k8, v8, q_descale, k_descale, v_descale, schedule: int,
                          causal: bool = False, softmax_scale: float | None = None, o=None,
                          lse=None, stream=None):
    """attn_fwd_fp8 with a schedule variant (0 = attn_fwd_fp8, ATTN_SCHED_EXP2_NONE,
    ATTN_SCHED_EXP2_POLY or ATTN_SCHED_EXP2_EIGHTHS(k)), for measurement."""
    lib = _lib.load()
    B, H, N, d = _shape4(q8, "q8")
    for t, n in ((k8, "k8"), (v8, "v8")):
        if _shape4(t, n) != (B, H, N, d):
            raise ValueError("q8, k8, v8 must have the same shape")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    code = lib.attn_fwd_fp8_schedule(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_descale),
                                     _ptr(k_descale), _ptr(v_descale), _ptr(o), _ptr(lse), B, H, N,
                                     d, int(bool(causal)), scale, int(schedule), _stream(stream))
    _check(code, "attn_fwd_fp8_schedule")
    return o, lse


def attn_selftest_exp2(x, stream=None):
    """(2^x by the FMA-pipe polynomial, 2^x by ex2.approx) for a float32 device tensor x."""
    lib = _lib.load()
    if x.dtype != torch.float32 or not x.is_contiguous() or x.device.type != "cuda":
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    y_poly, y_mufu = torch.empty_like(x), torch.empty_like(x)
    code = lib.attn_selftest_exp2(_ptr(x), _ptr(y_poly), _ptr(y_mufu), x.numel(), _stream(stream))
    _check(code, "attn_selftest_exp2")
    return y_poly, y_mufu


def attn_fwd_fp8_gqa(q8, k8, v8, q_descale, k_descale, v_descale, causal: bool = False,
                     softmax_scale: float | None = None, o=None, lse=None, stream=None):
    """FP8 forward with grouped-query heads: q8 [B, H, N, d], k8 and v8
    [B, H_kv, N, d] (uint8 e4m3) with their block descales -> O (bfloat16), LSE."""
    lib = _lib.load()
    (q8, k8, v8, q_descale, k_descale, v_descale), host = _to_device(
        [q8, k8, v8, q_descale, k_descale, v_descale])
    B, H, N, d = _shape4(q8, "q8")
    _, Hkv, _, _ = _shape4(k8, "k8")
    for t, n in ((k8, "k8"), (v8, "v8")):
        if _shape4(t, n) != (B, Hkv, N, d) or t.dtype != torch.uint8:
            raise ValueError(f"{n} must be uint8 e4m3 codes [B, H_kv, N, d]")
    if q8.dtype != torch.uint8:
        raise ValueError("q8 must be uint8 e4m3 codes")
    nblk = (N + 127) // 128
    for t, h in ((q_descale, H), (k_descale, Hkv), (v_descale, Hkv)):
        if t.dtype != torch.float32 or tuple(t.shape) != (B, h, nblk) or not t.is_contiguous():
            raise ValueError("descales must be contiguous float32 [B, heads, ceil(N/128)]")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    code = lib.attn_fwd_fp8_gqa(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_descale), _ptr(k_descale),
                                _ptr(v_descale), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                int(bool(causal)), scale, _stream(stream))
    _check(code, "attn_fwd_fp8_gqa")
    if host:
        return o.cpu(), lse.cpu()
    return o, lse


def attn_fp8_quantize_varlen(q, k, v, cu_seqlens, max_seqlen: int, hadamard_signs=None,
                             stream=None):
    """Block pre-pass of a packed batch: float32 q [total, H, d], k, v
    [total, H_kv, d], int32 cu_seqlens [B + 1] -> e4m3 codes of the same shapes
    and float32 descales [B, heads, ceil(max_seqlen / 128)]."""
    lib = _lib.load()
    ins = [q, k, v, cu_seqlens] + ([hadamard_signs] if hadamard_signs is not None else [])
    ins, host = _to_device(ins)
    q, k, v, cu_seqlens = ins[:4]
    signs = ins[4] if hadamard_signs is not None else None
    total, H, d = _shape3(q, "q")
    Hkv = k.shape[1] if k.dim() == 3 else -1
    if _shape3(k, "k") != (total, Hkv, d) or _shape3(v, "v") != (total, Hkv, d):
        raise ValueError("k and v must be [total, H_kv, d] with q's total and d")
    if any(t.dtype != torch.float32 for t in (q, k, v)):
        raise ValueError("FP8 pre-pass inputs are float32")
    if signs is not None and (signs.dtype != torch.float32 or signs.numel() != d):
        raise ValueError("hadamard_signs must be d float32 values")
    B = _cu_seqlens(cu_seqlens, total)
    nblk = (int(max_seqlen) + 127) // 128
    outs = [torch.empty((total, h, d), dtype=torch.uint8, device=q.device) for h in (H, Hkv, Hkv)]
    desc = [torch.empty((B, h, nblk), dtype=torch.float32, device=q.device) for h in (H, Hkv, Hkv)]
    code = lib.attn_fp8_quantize_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(signs),
                                        *[_ptr(t) for t in outs], *[_ptr(t) for t in desc],
                                        _ptr(cu_seqlens), B, int(max_seqlen), total, H, Hkv, d,
                                        _stream(stream))
    _check(code, "attn_fp8_quantize_varlen")
    if host:
        return tuple(t.cpu() for t in outs), tuple(t.cpu() for t in desc)
    return tuple(outs), tuple(desc)


def attn_fwd_fp8_varlen(q8, k8, v8, q_descale, k_descale, v_descale, cu_seqlens,
                        max_seqlen: int, causal: bool = False,
                        softmax_scale: float | None = None, o=None, lse=None, stream=None):
    """FP8 forward over a packed batch (the output of attn_fp8_quantize_varlen):
    returns O [total, H, d] bfloat16 and LSE float32 [H, total]."""
    lib = _lib.load()
    (q8, k8, v8, q_descale, k_descale, v_descale, cu_seqlens), host = _to_device(
        [q8, k8, v8, q_descale, k_descale, v_descale, cu_seqlens])
    total, H, d = _shape3(q8, "q8")
    Hkv = k8.shape[1] if k8.dim() == 3 else -1
    if _shape3(k8, "k8") != (total, Hkv, d) or _shape3(v8, "v8") != (total, Hkv, d):
        raise ValueError("k8 and v8 must be [total, H_kv, d] with q8's total and d")
    if any(t.dtype != torch.uint8 for t in (q8, k8, v8)):
        raise ValueError("q8, k8, v8 must be uint8 e4m3 codes")
    B = _cu_seqlens(cu_seqlens, total)
    nblk = (int(max_seqlen) + 127) // 128
    for t, h in ((q_descale, H), (k_descale, Hkv), (v_descale, Hkv)):
        if t.dtype != torch.float32 or tuple(t.shape) != (B, h, nblk) or not t.is_contiguous():
            raise ValueError("descales must be contiguous float32 [B, heads, ceil(max_seqlen/128)]")
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    if o is None:
        o = torch.empty((total, H, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((H, total), dtype=torch.float32, device=q8.device)
    code = lib.attn_fwd_fp8_varlen(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_descale),
                                   _ptr(k_descale), _ptr(v_descale), _ptr(o), _ptr(lse),
                                   _ptr(cu_seqlens), B, int(max_seqlen), total, H, Hkv, d,
                                   int(bool(causal)), scale, _stream(stream))
    _check(code, "attn_fwd_fp8_varlen")
    if host:
        return o.cpu(), lse.cpu()
    return o, lse


def attn_fp8_quantize_bf16(q, k, v, hadamard_signs=None, per_tensor: bool = False, stream=None):
    """The pre-pass on bfloat16 q [B, H, N, d] and k, v [B, H_kv, N, d]:
    e4m3 codes (q8, k8, v8) and float32 block descales."""
    lib = _lib.load()
    ins = [q, k, v] + ([hadamard_signs] if hadamard_signs is not None else [])
    ins, host = _to_device(ins)
    q, k, v = ins[:3]
    signs = ins[3] if hadamard_signs is not None else None
    B, H, N, d = _shape4(q, "q")
    _, Hkv, _, _ = _shape4(k, "k")
    for t, n in ((k, "k"), (v, "v")):
        if _shape4(t, n) != (B, Hkv, N, d):
            raise ValueError("k and v must be [B, H_kv, N, d] with q's B, N, d")
    if any(t.dtype != torch.bfloat16 for t in (q, k, v)):
        raise ValueError("inputs must be bfloat16")
    if signs is not None and (signs.dtype != torch.float32 or signs.numel() != d):
        raise ValueError("hadamard_signs must be d float32 values")
    nblk = (N + 127) // 128
    outs = [torch.empty((B, h, N, d), dtype=torch.uint8, device=q.device) for h in (H, Hkv, Hkv)]
    desc = [torch.empty((B, h, nblk), dtype=torch.float32, device=q.device) for h in (H, Hkv, Hkv)]
    code = lib.attn_fp8_quantize_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(signs),
                                      *[_ptr(t) for t in outs], *[_ptr(t) for t in desc],
                                      B, H, Hkv, N, d, int(bool(per_tensor)), _stream(stream))
    _check(code, "attn_fp8_quantize_bf16")
    if host:
        return tuple(t.cpu() for t in outs), tuple(t.cpu() for t in desc)
    return tuple(outs), tuple(desc)


def attn_fp8_quantize_ex(q, k, v, rope_cos=None, rope_sin=None, hadamard_signs=None,
                         cu_seqlens=None, max_seqlen: int | None = None, per_tensor: bool = False,
                         stream=None):
    """The FP8 pre-pass with every option: float32 or bfloat16 inputs (from the
    tensors' dtype), optional rotary tables [N, d/2], optional Hadamard signs,
    grouped-query heads (k, v with fewer heads), and fixed-length [B, H, N, d]
    or packed [total, H, d] batches (with int32 cu_seqlens [B + 1] and
    max_seqlen).  Returns (q8, k8, v8), (q_descale, k_descale, v_descale)."""
    lib = _lib.load()
    if q.dtype not in (torch.float32, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must all be float32 or all bfloat16")
    for t in (q, k, v, rope_cos, rope_sin, hadamard_signs, cu_seqlens):
        if t is not None and (t.device.type != "cuda" or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")
    if cu_seqlens is None:
        B, H, N, d = _shape4(q, "q")
        Hkv = k.shape[1]
        total = 0
        nblk = (N + 127) // 128
        shapes = [(B, H, N, d), (B, Hkv, N, d), (B, Hkv, N, d)]
        dshapes = [(B, H, nblk), (B, Hkv, nblk), (B, Hkv, nblk)]
    else:
        if max_seqlen is None:
            raise ValueError("a packed batch needs max_seqlen")
        total, H, d = _shape3(q, "q")
        Hkv = k.shape[1]
        B, N = cu_seqlens.numel() - 1, int(max_seqlen)
        nblk = (N + 127) // 128
        shapes = [(total, H, d), (total, Hkv, d), (total, Hkv, d)]
        dshapes = [(B, H, nblk), (B, Hkv, nblk), (B, Hkv, nblk)]
    for t, shp, n in ((q, shapes[0], "q"), (k, shapes[1], "k"), (v, shapes[2], "v")):
        if tuple(t.shape) != shp:
            raise ValueError(f"{n} has shape {tuple(t.shape)}, expected {shp}")
    outs = [torch.empty(shp, dtype=torch.uint8, device=q.device) for shp in shapes]
    desc = [torch.empty(shp, dtype=torch.float32, device=q.device) for shp in dshapes]
    code = lib.attn_fp8_quantize_ex(_ptr(q), _ptr(k), _ptr(v), int(q.dtype == torch.bfloat16),
                                    _ptr(rope_cos), _ptr(rope_sin), _ptr(hadamard_signs),
                                    *[_ptr(t) for t in outs], *[_ptr(t) for t in desc],
                                    _ptr(cu_seqlens), B, N, total, H, Hkv, d,
                                    int(bool(per_tensor)), _stream(stream))
    _check(code, "attn_fp8_quantize_ex")
    return tuple(outs), tuple(desc)
