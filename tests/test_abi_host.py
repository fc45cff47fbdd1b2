"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_25_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for expected in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_fp8_quantize",
                     "attn_fwd_fp8", "attn_get_device_status", "attn_status_string",
                     "attn_last_error"):
        assert expected in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(6):
        assert lib.attn_status_string(code)
    assert lib.attn_status_string(99) == b"unknown status"


def test_workspace_size(lib):
    up = lambda x: -(-x // 256) * 256
    for B, H, N, d in ((2, 16, 4096, 128), (1, 3, 300, 64)):
        rows = B * H * N
        rows_pad = B * H * (-(-N // 128) * 128)
        # float32 dQ accumulator + two float32 row vectors padded to 128 rows per head
        expect = up(rows * d * 4) + 2 * up(rows_pad * 4)
        assert lib.attn_bwd_workspace_size(B, H, N, d) == expect
    assert lib.attn_bwd_workspace_size(0, 1, 1, 64) == 0


def _fwd(lib, q=16, k=16, v=16, o=16, l=16, B=1, H=1, N=128, d=128, causal=0, scale=0.1, dt=0):
    return lib.attn_fwd(q, k, v, o, l, B, H, N, d, causal, scale, dt, None)


@pytest.mark.parametrize("kwargs,why", [
    (dict(d=96), "d"),
    (dict(d=0), "d"),
    (dict(N=0), "N"),
    (dict(B=-1), "B"),
    (dict(causal=2), "causal"),
    (dict(scale=0.0), "scale"),
    (dict(scale=float("inf")), "scale"),
    (dict(q=0), "null"),
    (dict(v=8), "aligned"),
    (dict(dt=7), "dtype"),
    (dict(B=65536, H=256, N=256, d=128), "2^31"),
])
def test_fwd_rejects_bad_arguments_without_a_gpu(lib, kwargs, why):
    assert _fwd(lib, **kwargs) == 1          # ATTN_ERR_INVALID_ARG
    assert why.lower() in lib.attn_last_error().decode().lower()


def test_bwd_rejects_small_workspace(lib):
    ws = lib.attn_bwd_workspace_size(1, 1, 128, 64)
    code = lib.attn_bwd(16, 16, 16, 16, 16, 16, 16, 16, 16, 256, ws - 1,
                        1, 1, 128, 64, 0, 0.125, 0, None)
    assert code == 1 and b"workspace" in lib.attn_last_error()
    code = lib.attn_bwd(16, 16, 16, 16, 16, 16, 16, 16, 16, 16, ws,
                        1, 1, 128, 64, 0, 0.125, 0, None)
    assert code == 1 and b"256-byte" in lib.attn_last_error()


def test_fp8_quantize_rejects_bad_modes(lib):
    code = lib.attn_fp8_quantize(16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 1, 128, 128, 1, None)
    assert code == 1 and b"per-tensor" in lib.attn_last_error()
    code = lib.attn_fp8_quantize(16, 16, 16, None, 16, 16, 16, 16, 16, 16, 1, 1, 128, 128, 3, None)
    assert code == 1


def test_unsupported_shapes_are_reported(lib):
    ws = lib.attn_bwd_workspace_size(1, 1, 128, 256)
    code = lib.attn_bwd(16, 16, 16, 16, 16, 16, 16, 16, 16, 256, ws,
                        1, 1, 128, 256, 0, 0.1, 0, None)
    assert code == 2                          # ATTN_ERR_UNSUPPORTED
    code = lib.attn_fwd_fp8(16, 16, 16, 16, 16, 16, 16, 16, 1, 1, 128, 64, 0, 0.1, None)
    assert code == 2


def test_device_check_fails_loudly_without_a_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid arguments reach the device check, which must fail, not fall back
    code = _fwd(lib)
    assert code in (3, 4)


def test_selftest_rejects_bad_limits(lib):
    assert lib.attn_selftest_wait_timeout(0, None) == 1
    assert lib.attn_selftest_wait_timeout(2000000, None) == 1


def test_gqa_and_varlen_entry_points_are_declared():
    names = declared_functions()
    for expected in ("attn_fwd_gqa", "attn_fwd_varlen", "attn_bwd_gqa", "attn_bwd_varlen",
                     "attn_bwd_varlen_workspace_size"):
        assert expected in names


@pytest.mark.parametrize("H,H_kv", [(4, 3), (4, 0), (2, 4)])
def test_gqa_rejects_heads_that_do_not_group(lib, H, H_kv):
    assert lib.attn_fwd_gqa(16, 16, 16, 16, 16, 1, H, H_kv, 128, 128, 0, 0.1, 0, None) == 1
    assert b"H_kv" in lib.attn_last_error()
    ws = lib.attn_bwd_workspace_size(1, H, 128, 128)
    assert lib.attn_bwd_gqa(16, 16, 16, 16, 16, 16, 16, 16, 16, 256, ws,
                            1, H, H_kv, 128, 128, 0, 0.1, 0, None) == 1


def _fwd_varlen(lib, cu=16, B=2, max_len=128, total=200, H=2, H_kv=1, d=128, causal=0):
    return lib.attn_fwd_varlen(16, 16, 16, 16, 16, cu, B, max_len, total, H, H_kv, d, causal, 0.1,
                               0, None)


@pytest.mark.parametrize("kwargs,why", [
    (dict(cu=0), "cu_seqlens"),
    (dict(cu=18), "cu_seqlens"),
    (dict(total=0), "total"),
    (dict(max_len=0), "max_seqlen"),
    (dict(B=0), "B"),
    (dict(d=80), "d"),
    (dict(H_kv=3), "H_kv"),
    (dict(total=1 << 30, H=16), "2^31"),
])
def test_varlen_rejects_bad_arguments_without_a_gpu(lib, kwargs, why):
    assert _fwd_varlen(lib, **kwargs) == 1
    assert why.lower() in lib.attn_last_error().decode().lower()


def test_varlen_workspace_size(lib):
    up = lambda x: -(-x // 256) * 256
    B, max_len, total, H, d = 3, 300, 700, 4, 64
    rows_pad = B * H * (-(-max_len // 128) * 128)
    expect = up(total * H * d * 4) + 2 * up(rows_pad * 4)
    assert lib.attn_bwd_varlen_workspace_size(B, max_len, total, H, d) == expect
    assert lib.attn_bwd_varlen_workspace_size(0, max_len, total, H, d) == 0
    ws = lib.attn_bwd_varlen_workspace_size(2, 128, 200, 2, 64)
    code = lib.attn_bwd_varlen(16, 16, 16, 16, 16, 16, 16, 16, 16, 256, ws - 1, 16,
                               2, 128, 200, 2, 1, 64, 0, 0.1, 0, None)
    assert code == 1 and b"workspace" in lib.attn_last_error()


def test_decode_is_declared_and_validates(lib):
    names = declared_functions()
    assert "attn_decode_paged" in names and "attn_decode_workspace_size" in names
    ws = lib.attn_decode_workspace_size(2, 8, 2, 1, 128, 1000)
    assert ws > 0 and lib.attn_decode_workspace_size(0, 8, 2, 1, 128, 1000) == 0

    def call(**kw):
        a = dict(B=2, H=8, H_kv=2, n_q=1, d=128, num_pages=10, page_size=64, max_pages=5,
                 max_seqlen=1000, causal=1, scale=0.1, ws=ws)
        a.update(kw)
        return lib.attn_decode_paged(16, 16, 16, 16, 16, 16, 16, 256, a["ws"], a["B"], a["H"],
                                     a["H_kv"], a["n_q"], a["d"], a["num_pages"], a["page_size"],
                                     a["max_pages"], a["max_seqlen"], a["causal"], a["scale"], 0, None)
    for kw, code, why in ((dict(page_size=48), 1, "page_size"), (dict(page_size=4), 1, "page_size"),
                          (dict(d=256), 1, "d ="), (dict(H_kv=3), 1, "H_kv"),
                          (dict(H=64, H_kv=1, n_q=4), 2, "128"), (dict(ws=ws - 1), 1, "workspace"),
                          (dict(causal=2), 1, "causal")):
        assert call(**kw) == code, kw
        assert why.lower() in lib.attn_last_error().decode().lower(), (kw, lib.attn_last_error())


def test_fp8_decode_is_declared_and_validates(lib):
    assert "attn_decode_paged_fp8" in declared_functions()
    ws = lib.attn_decode_workspace_size(2, 8, 2, 1, 128, 1000)

    def call(signs=None, **kw):
        a = dict(B=2, H=8, H_kv=2, n_q=1, d=128, num_pages=10, page_size=64, max_pages=5,
                 max_seqlen=1000, causal=1, scale=0.1, ws=ws, kd=16, vd=16)
        a.update(kw)
        return lib.attn_decode_paged_fp8(16, 16, 16, a["kd"], a["vd"], signs, 16, 16, 16, 16, 256,
                                         a["ws"], a["B"], a["H"], a["H_kv"], a["n_q"], a["d"],
                                         a["num_pages"], a["page_size"], a["max_pages"],
                                         a["max_seqlen"], a["causal"], a["scale"], 0, None)
    for kw, code, why in ((dict(page_size=8), 1, "page_size"), (dict(page_size=96), 1, "page_size"),
                          (dict(d=64), 2, "d = 128"), (dict(H_kv=3), 1, "H_kv"),
                          (dict(H=64, H_kv=1, n_q=4), 2, "128"), (dict(ws=ws - 1), 1, "workspace"),
                          (dict(kd=0), 1, "null"), (dict(vd=8), 1, "aligned"),
                          (dict(signs=8), 1, "hadamard_signs"), (dict(scale=0.0), 1, "softmax_scale")):
        assert call(**kw) == code, kw
        assert why.lower() in lib.attn_last_error().decode().lower(), (kw, lib.attn_last_error())


def test_fp8_gqa_is_declared_and_validates(lib):
    names = declared_functions()
    assert "attn_fp8_quantize_gqa" in names and "attn_fwd_fp8_gqa" in names
    for H_kv, why in ((3, "H_kv"), (0, "H_kv"), (8, "H_kv")):
        code = lib.attn_fwd_fp8_gqa(16, 16, 16, 16, 16, 16, 16, 16, 1, 4, H_kv, 256, 128, 0, 0.1,
                                    None)
        assert code == 1 and why.encode() in lib.attn_last_error()
        code = lib.attn_fp8_quantize_gqa(16, 16, 16, None, 16, 16, 16, 16, 16, 16, 1, 4, H_kv,
                                         256, 128, 0, None)
        assert code == 1 and why.encode() in lib.attn_last_error()
    assert lib.attn_fwd_fp8_gqa(16, 16, 16, 16, 16, 16, 16, 16, 1, 4, 2, 256, 64, 0, 0.1,
                                None) == 2                     # d = 128 only


def test_fp8_varlen_is_declared_and_validates(lib):
    names = declared_functions()
    assert "attn_fp8_quantize_varlen" in names and "attn_fwd_fp8_varlen" in names
    # (cu_seqlens, B, max_seqlen, total, H, H_kv, d)
    for args, code, why in (((None, 2, 100, 200, 4, 2, 128), 1, "cu_seqlens"),
                            ((16, 2, 100, 200, 4, 3, 128), 1, "H_kv"),
                            ((16, 0, 100, 200, 4, 2, 128), 1, ">= 1"),
                            ((16, 2, 100, 200, 4, 2, 64), 2, "d = 128")):
        got = lib.attn_fwd_fp8_varlen(16, 16, 16, 16, 16, 16, 16, 16, *args, 0, 0.1, None)
        assert got == code and why.encode() in lib.attn_last_error(), (args, lib.attn_last_error())
        got = lib.attn_fp8_quantize_varlen(16, 16, 16, None, 16, 16, 16, 16, 16, 16, *args, None)
        assert got == code and why.encode() in lib.attn_last_error(), (args, lib.attn_last_error())


def test_fp8_bf16_prepass_is_declared_and_validates(lib):
    assert "attn_fp8_quantize_bf16" in declared_functions()
    code = lib.attn_fp8_quantize_bf16(16, 16, 16, None, 16, 16, 16, 16, 16, 16, 1, 4, 3, 256, 128,
                                      0, None)
    assert code == 1 and b"H_kv" in lib.attn_last_error()
    code = lib.attn_fp8_quantize_bf16(16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 4, 2, 256, 128,
                                      1, None)
    assert code == 1 and b"Hadamard" in lib.attn_last_error()


def test_noalloc_refuses_oversized_problems_before_any_cuda_call(lib):
    """attn_bwd_noalloc checks the problem against its built-in scratch first,
    so the refusal needs no GPU and names the limit."""
    assert "attn_bwd_noalloc" in declared_functions()
    B, H, N, d = 2, 16, 4096, 128
    assert lib.attn_bwd_workspace_size(B, H, N, d) > 64 << 20
    code = lib.attn_bwd_noalloc(16, 16, 16, 16, 16, 16, 16, 16, 16, B, H, N, d, 1, 0.1, 0, None)
    assert code == 1                          # ATTN_ERR_INVALID_ARG
    assert b"built-in scratch" in lib.attn_last_error()


def test_noalloc_reaches_the_device_check_without_a_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # a problem that fits: the device check comes before the symbol lookup
    code = lib.attn_bwd_noalloc(16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 2, 256, 64, 0, 0.1, 0, None)
    assert code in (3, 4)


def test_fp8_quantize_ex_validates(lib):
    assert "attn_fp8_quantize_ex" in declared_functions()

    def call(bf=1, cos=16, sin=16, signs=None, cu=None, B=1, N=256, total=0, H=4, H_kv=2, d=128, pt=0):
        return lib.attn_fp8_quantize_ex(16, 16, 16, bf, cos, sin, signs, 16, 16, 16, 16, 16, 16, cu,
                                        B, N, total, H, H_kv, d, pt, None)
    for kw, code, why in ((dict(bf=2), 1, "input_bf16"), (dict(sin=None), 1, "rope_sin"),
                          (dict(cos=8), 1, "16-byte"), (dict(pt=1), 1, "per-tensor"),
                          (dict(H_kv=3), 1, "H_kv"), (dict(d=64), 2, "d = 128"),
                          (dict(cu=18, total=300), 1, "cu_seqlens"), (dict(cu=16, total=0), 1, ">= 1")):
        assert call(**kw) == code, kw
        assert why.lower() in lib.attn_last_error().decode().lower(), (kw, lib.attn_last_error())


def test_fp8_schedule_validates_the_exp2_share(lib):
    """attn_fwd_fp8_schedule takes 0, ATTN_SCHED_EXP2_NONE, ATTN_SCHED_EXP2_POLY or
    ATTN_SCHED_EXP2_EIGHTHS(1..4) and rejects anything else before touching the GPU."""
    import exact_tiled_attention_25_gb300 as attn
    args = (16, 16, 16, 16, 16, 16, 16, 16, 1, 1, 128, 128, 0, 0.1)
    for bad in (1, 2, 12, attn.ATTN_SCHED_EXP2_NONE | (1 << 8), attn.ATTN_SCHED_EXP2_EIGHTHS(5),
                attn.ATTN_SCHED_EXP2_EIGHTHS(15), attn.ATTN_SCHED_EXP2_POLY | (1 << 12)):
        assert lib.attn_fwd_fp8_schedule(*args, bad, None) == 1, bad
        assert b"schedule" in lib.attn_last_error()
    assert attn.ATTN_SCHED_EXP2_EIGHTHS(2) == attn.ATTN_SCHED_EXP2_POLY | (2 << 8)
