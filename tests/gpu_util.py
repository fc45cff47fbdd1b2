"""Helpers shared by the GPU parity tests (CUDA path vs the CPU oracle)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances of the forward, LSE and gradient comparisons.
FWD_MAX_ABS = 2e-2
FWD_RMSE = 2e-3
LSE_ABS = 1e-3
GRAD_REL_RMSE = 5e-3
FP8_RMSE = 3e-2


def lib():
    import exact_tiled_attention_25_gb300 as attn
    from exact_tiled_attention_25_gb300 import build
    build.build()
    attn.load_library()
    return attn


def dev():
    return torch.device("cuda", torch.cuda.current_device())


def check_status(attn):
    torch.cuda.synchronize()
    code = attn.attn_get_device_status()
    assert code == 0, f"device status {code}: {attn.attn_last_error()}"


def fwd_errors(o_gpu, lse_gpu, o_ref, lse_ref):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    diff = o - o_ref
    return (float(np.abs(diff).max()), float(np.sqrt(np.mean(diff ** 2))),
            float(np.abs(lse - lse_ref).max()))


def assert_fwd_close(o_gpu, lse_gpu, o_ref, lse_ref, max_abs=FWD_MAX_ABS, rmse=FWD_RMSE,
                     lse_abs=LSE_ABS):
    e_max, e_rmse, e_lse = fwd_errors(o_gpu, lse_gpu, o_ref, lse_ref)
    assert e_max <= max_abs and e_rmse <= rmse and e_lse <= lse_abs, (e_max, e_rmse, e_lse)
    return e_max, e_rmse, e_lse


def rel_rmse(g_gpu, g_ref, floor=1e-4):
    """RMSE(g - g_ref) / RMS(g_ref).  The denominator is floored at `floor`
    because some gradients are exactly zero (e.g. dQ and dK with a single key),
    where only float32 rounding residue remains on the GPU.  The floor applies
    only there: a reference with RMS below it must be zero up to float64
    rounding (RMS < 1e-9), otherwise the floor could hide a real error and the
    call fails."""
    g = g_gpu.float().cpu().numpy().astype(np.float64) if hasattr(g_gpu, "float") else np.asarray(
        g_gpu, dtype=np.float64)
    assert np.all(np.isfinite(g))
    rms_ref = float(np.sqrt(np.mean(g_ref ** 2)))
    assert rms_ref >= floor or rms_ref < 1e-9, (
        f"reference RMS {rms_ref:.3g} is below the floor {floor:g} but not zero")
    return float(np.sqrt(np.mean((g - g_ref) ** 2)) / max(rms_ref, floor))


def guarded(shape, dtype, fill):
    """A tensor view with sentinel bands of 4096 bytes before and after it;
    returns (view, check) where check() asserts the bands are untouched."""
    n = int(np.prod(shape))
    esize = torch.empty((), dtype=dtype).element_size()
    pad = 4096 // esize
    buf = torch.full((n + 2 * pad,), fill, dtype=dtype, device=dev())
    view = buf[pad:pad + n].view(shape)

    def check():
        torch.cuda.synchronize()
        head = buf[:pad]
        tail = buf[pad + n:]
        same = (lambda t: torch.all(t == fill).item()) if dtype != torch.uint8 else \
            (lambda t: torch.all(t == fill).item())
        assert same(head) and same(tail), "write outside the output tensor"
    return view, check


def timed_step_inputs(seed=3, shape=(2, 16, 8192, 128)):
    """The benchmark's own inputs for the timed step, drawn the same way on the
    device: Q, K, V, dO i.i.d. N(0, 1) float32 from one seeded torch generator,
    rounded to bfloat16, then the Hadamard signs from the same generator."""
    g = torch.Generator(device=dev()).manual_seed(seed)
    q, k, v, do = (torch.randn(shape, generator=g, device=dev(), dtype=torch.float32)
                   for _ in range(4))
    signs = torch.where(torch.rand(shape[-1], generator=g, device=dev()) < 0.5, -1.0, 1.0).float()
    return tuple(t.to(torch.bfloat16) for t in (q, k, v, do)) + (signs,)
