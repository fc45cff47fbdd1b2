"""Failure path shared by every kernel: a barrier wait that runs out.

Nothing here faults or traps the GPU: the self-test kernel waits on a barrier
that nothing arrives on, through the same bounded wait the attention kernels
use; the wait gives up after a short limit, records the timeout in the device
status word and returns.  The host must see ATTN_ERR_TIMEOUT once, and the
context must stay usable."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_fwd_close, check_status, dev, lib

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    attn = lib()
    c = attn.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    check_status(attn)                                      # clean to start with
    assert c.attn_selftest_wait_timeout(20000, stream) == 0   # 20 ms limit
    code = attn.attn_get_device_status()
    assert code == attn.ATTN_ERR_TIMEOUT
    assert "self-test" in attn.attn_last_error()
    assert attn.attn_get_device_status() == 0               # the word was cleared
    # the context still works: a small forward matches the oracle
    tq, tk, tv = (workloads.round_to(x, "bf16") for x in workloads.normal(3, (1, 2, 200, 64), 3))
    o, lse = attn.attn_fwd(tq.to(dev()), tk.to(dev()), tv.to(dev()), causal=True)
    check_status(attn)
    ref_o, ref_l = oracle.attention_forward(*(workloads.as_f64(t) for t in (tq, tk, tv)),
                                            1 / np.sqrt(64), True)
    assert_fwd_close(o, lse, ref_o, ref_l)
