"""Failure detection on the GPU without a fault: a device-side wait that can never be
satisfied gives up after its limit, the kernel records the timeout in the status word
and returns, the host reads SP_ERR_TIMEOUT, and the context keeps working."""
import pytest
import torch

import oracle
from gpu_util import check_out, f64, need_gpu
from sequence_head_attention_seq_b300 import sp_attn_fwd, sp_get_device_status, workloads
from sequence_head_attention_seq_b300.binding import sp_selftest_wait_timeout

pytestmark = pytest.mark.gpu

SP_OK, SP_ERR_TIMEOUT = 0, 5


def test_wait_timeout_reported_and_context_usable():
    need_gpu()
    assert sp_get_device_status() == SP_OK
    sp_selftest_wait_timeout()
    assert sp_get_device_status() == SP_ERR_TIMEOUT
    assert sp_get_device_status() == SP_OK            # reading the word clears it
    # the same context still computes attention correctly
    q, k, v = (workloads.randn_bf16((1, 256, 2, 64), 940 + t, 1.0, device="cuda")
               for t in range(3))
    o, _ = sp_attn_fwd(q, k, v, True)
    torch.cuda.synchronize()
    assert sp_get_device_status() == SP_OK
    ro, _ = oracle.default().attn_fwd(f64(q), f64(k), f64(v), True)
    check_out(f64(o), ro, "out after a timed-out wait")
