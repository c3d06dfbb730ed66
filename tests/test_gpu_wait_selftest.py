"""The bounded on-chip waits of the tensor-core kernels, made to expire on purpose.

retention_chunkwise_wait_selftest launches the pair-of-SMs chunkwise kernel on a tiny
shape with every wait limited to 1 ms and a TMA producer that issues no load: nothing ever
completes the barriers, so every wait gives up, the kernel unwinds with no copy or MMA in
flight and frees its tensor memory.  The error must surface as RET_ERR_TIMEOUT, and the
device must stay usable: a normal call right after it still matches the oracle.
"""
import ctypes

import pytest
import torch

import oracle
from linear_recurrence_sequence_chunkwise_b300 import binding as rb
from linear_recurrence_sequence_chunkwise_b300 import build, inputs

from _util import TOL_BF16, err_bf16

DEV = "cuda"


def test_selftest_rejects_bad_pointers_on_the_host():
    build.build()
    L = rb.lib()
    A = ctypes.c_void_p(0x100000)
    assert L.retention_chunkwise_wait_selftest(None, A, A, A, None) == rb.RET_ERR_NULL
    assert L.retention_chunkwise_wait_selftest(ctypes.c_void_p(0x100008), A, A, A,
                                               None) == rb.RET_ERR_ALIGN


@pytest.mark.gpu
def test_expired_waits_report_timeout_and_the_device_stays_usable():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    q = torch.zeros(256, 256, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros_like(q)
    v = torch.zeros(256, 128, dtype=torch.bfloat16, device=DEV)
    o = torch.full((256, 128), 7.0, dtype=torch.float32, device=DEV)
    rb.check_device_error()                      # start from a clear error word
    for _ in range(2):
        assert rb.chunkwise_wait_selftest(q, k, v, o) == rb.RET_OK
        with pytest.raises(rb.RetentionError) as e:
            rb.check_device_error()
        assert e.value.status == rb.RET_ERR_TIMEOUT
    assert bool((o == 7.0).all())                # the output was never written
    # the error word is cleared and the device works: a normal pair-kernel call
    rb.check_device_error()
    b, H, N, dk, dv = 1, 2, 512, 256, 128
    qq = inputs.randn((b, H, N, dk), 430, 1 / 16, "bf16", DEV)
    kk = inputs.randn((b, H, N, dk), 431, 1 / 16, "bf16", DEV)
    vv = inputs.randn((b, H, N, dv), 432, 1 / 16, "bf16", DEV)
    g = inputs.gammas(H)
    got = rb.retention_chunkwise(qq, kk, vv, g, 256)
    assert rb.last_kernel() == "chunkwise_tc_pair"
    assert err_bf16(got, oracle.chunkwise(qq, kk, vv, g, 256)) < TOL_BF16
    rb.check_device_error()
