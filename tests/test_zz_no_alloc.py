"""retention_chunkwise_host_noalloc: the host-streamed chunkwise call on the library's
static device scratch instead of a caller workspace.

The entry point is for callers that cannot call cudaMalloc: code hosted inside a framework
whose caching allocator has already reserved the device memory (a cudaMalloc behind its back
can fail with out-of-memory, or fragment the framework's pool), and latency-critical loops
where cudaMalloc/cudaFree would synchronise the device.  They pass only inputs and outputs.

Host-side checks (no GPU): the entry is exported, the scratch size is reported, and a
call whose workspace would not fit, or with a bad segment length, is rejected before any
device access.  On a GPU: two calls in a row each equal retention_chunkwise_host with a
caller workspace and the fp64 oracle (the scratch keeps the previous call's contents, so
the second call checks that nothing stale leaks into it), and the final state is handed
back.  This file is collected last so that a failure here leaves every other test run.
"""
import ctypes

import pytest
import torch

from linear_recurrence_sequence_chunkwise_b300 import binding as rb
from linear_recurrence_sequence_chunkwise_b300 import build, inputs

A = ctypes.c_void_p(0x100000)
S = ctypes.c_void_p(0)
MIB = 1 << 20


def G(*vals):
    return (ctypes.c_double * len(vals))(*vals)


@pytest.fixture(scope="module")
def L():
    build.build()
    return rb.lib()


def call(L, b=1, H=2, N=512, dk=64, dv=64, chunk=64, seg=128, it=1, ot=0, q=A):
    return L.retention_chunkwise_host_noalloc(q, A, A, A, it, ot, b, H, N, dk, dv, chunk,
                                              G(*([0.9] * H)), None, None, seg, S, S, S)


def test_scratch_size_and_export(L):
    assert L.retention_chunkwise_host_static_scratch_bytes() == 48 * MIB
    assert "retention_chunkwise_host_noalloc" in rb.header_functions()


def test_rejections_before_any_device_access(L):
    # b1 H16 dk256 dv512, 4096-token segments: ~520 MB of workspace, far above the scratch
    need = L.retention_chunkwise_host_workspace_bytes(1, 0, 1, 16, 256, 512, 4096)
    assert need > 48 * MIB
    assert call(L, H=16, N=8192, dk=256, dv=512, chunk=256, seg=4096) == rb.RET_ERR_SHAPE
    assert call(L, seg=96) == rb.RET_ERR_SHAPE
    assert call(L, it=9) == rb.RET_ERR_DTYPE
    assert call(L, q=ctypes.c_void_p(0x100008)) == rb.RET_ERR_ALIGN
    assert call(L, b=0) == rb.RET_OK


@pytest.mark.gpu
def test_noalloc_matches_caller_workspace_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import oracle
    from _util import TOL_BF16, err_bf16
    b, H, N, dk, dv, chunk, seg = 1, 4, 1024, 256, 256, 256, 256
    assert rb.chunkwise_host_workspace_bytes(torch.bfloat16, torch.float32, b, H, dk, dv,
                                             seg) <= rb.chunkwise_host_static_scratch_bytes()
    g = inputs.gammas(H)
    for call_no in range(2):
        base = 9100 + 10 * call_no
        q, k, v = (inputs.randn((b, H, N, d), base + i, 1 / 16, "bf16", "cpu").pin_memory()
                   for i, d in enumerate((dk, dk, dv)))
        s0 = inputs.randn((b, H, dk, dv), base + 5, 0.05, "f32", "cuda")
        o1 = torch.empty((b, H, N, dv), dtype=torch.float32, pin_memory=True)
        o2 = torch.empty_like(o1, pin_memory=True)
        o2.fill_(float("nan"))
        s1, s2 = s0.clone(), s0.clone()
        rb.retention_chunkwise_host(q, k, v, g, chunk, o1, seg, state_in=s1, state_out=s1)
        rb.retention_chunkwise_host_noalloc(q, k, v, g, chunk, o2, seg, state_in=s2,
                                            state_out=s2)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2), f"call {call_no}"
        assert torch.equal(s1, s2), f"call {call_no}"
        want, want_state = oracle.chunkwise(q, k, v, g, chunk, state_in=s0, return_state=True)
        assert err_bf16(o2, want) < TOL_BF16, f"call {call_no}"
        assert err_bf16(s2, want_state) < TOL_BF16, f"call {call_no}"
    rb.check_device_error()
