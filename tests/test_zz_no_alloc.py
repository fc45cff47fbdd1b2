"""attn_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (for example a runtime with no device allocator of its own).  Its
scratch is an array built into the library, so this test checks, through the C
ABI, that two calls in a row match the ordinary attn_bwd (which takes a
caller-allocated workspace), and that problems too large for the built-in
scratch are refused.  The file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_util import GRAD_REL_RMSE, check_status, dev, lib, rel_rmse

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20


def _noalloc(c, tensors, dq, dk, dv, B, H, N, d, causal, scale):
    q, k, v, o, do, lse = tensors
    stream = torch.cuda.current_stream().cuda_stream
    return c.attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H, N, d, int(causal), ctypes.c_float(scale), 0,
                              stream)


def test_noalloc_backward_matches_workspace_backward():
    attn = lib()
    c = attn.load_library()
    B, H, N, d, causal = 1, 4, 1000, 128, True
    scale = 1 / np.sqrt(d)
    q, k, v, do = (workloads.round_to(x, "bf16").to(dev())
                   for x in workloads.normal(77, (B, H, N, d), 4))
    o, lse = attn.attn_fwd(q, k, v, causal=causal, softmax_scale=scale)
    ref = attn.attn_bwd(q, k, v, o, do, lse, causal=causal, softmax_scale=scale)
    check_status(attn)
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        code = _noalloc(c, (q, k, v, o, do, lse), dq, dk, dv, B, H, N, d, causal, scale)
        assert code == 0, attn.attn_last_error()
        check_status(attn)
        for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            err = rel_rmse(got, want.double().cpu().numpy())
            assert err <= GRAD_REL_RMSE, (call, name, err)
        # dK and dV involve no reductions across CTAs: identical bits
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])


def test_noalloc_rejects_problems_beyond_its_scratch():
    attn = lib()
    c = attn.load_library()
    B, H, N, d = 2, 16, 4096, 128          # needs about 68 MB of scratch
    assert attn.attn_bwd_workspace_size(B, H, N, d) > SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.bfloat16, device=dev())
    lse = torch.empty(4, dtype=torch.float32, device=dev())
    code = _noalloc(c, (dummy, dummy, dummy, dummy, dummy, lse), dummy, dummy, dummy,
                    B, H, N, d, True, 0.1)
    assert code == 1                        # ATTN_ERR_INVALID_ARG, nothing launched
    assert "built-in scratch" in attn.attn_last_error()
