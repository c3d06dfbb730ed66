"""retention_chunkwise_host: chunkwise retention over pinned host buffers, streamed through
the device in segments with the copies on their own streams.

The streamed result must equal one chunkwise call over the whole sequence: the state
handed from segment to segment is the exact fp32 state of the chunkwise form, so the
only difference allowed is fp32 rounding of the carried state.  Both are also checked
against the oracle.
"""
import pytest
import torch

import oracle
from linear_recurrence_sequence_chunkwise_b300 import binding as rb
from linear_recurrence_sequence_chunkwise_b300 import inputs

from _util import TOL_BF16, chunkwise_tc_name, err_bf16, err_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    rb.lib()


def host_qkv(b, H, N, dk, dv, seed, dtype="bf16"):
    q = inputs.randn((b, H, N, dk), seed, 1 / 16, dtype, "cpu").pin_memory()
    k = inputs.randn((b, H, N, dk), seed + 1, 1 / 16, dtype, "cpu").pin_memory()
    v = inputs.randn((b, H, N, dv), seed + 2, 1 / 16, dtype, "cpu").pin_memory()
    return q, k, v


@pytest.mark.parametrize("dk,dv,chunk,seg", [(256, 512, 256, 512), (128, 128, 128, 256),
                                             (128, 64, 128, 128), (256, 256, 256, 1024)])
def test_streamed_equals_single_call(dk, dv, chunk, seg):
    b, H, N = 2, 3, 1024
    hq, hk, hv = host_qkv(b, H, N, dk, dv, 8000 + dk + dv + seg)
    g = inputs.gammas(H)
    ho = torch.empty((b, H, N, dv), dtype=torch.float32, pin_memory=True)
    ho.fill_(float("nan"))
    rb.retention_chunkwise_host(hq, hk, hv, g, chunk, ho, seg)
    torch.cuda.synchronize()
    assert rb.last_kernel() == chunkwise_tc_name(dk, dv, chunk, seg)
    one = rb.retention_chunkwise(hq.to(DEV), hk.to(DEV), hv.to(DEV), g, chunk).cpu()
    assert not torch.isnan(ho).any()
    assert err_f32(ho, one) < 1e-5
    assert err_bf16(ho, oracle.chunkwise(hq, hk, hv, g, chunk)) < TOL_BF16
    rb.check_device_error()


def test_streamed_carries_incoming_state_and_returns_final_state():
    b, H, N, dk, dv, chunk = 1, 2, 768, 128, 128, 128
    hq, hk, hv = host_qkv(b, H, N, dk, dv, 8100)
    g = [0.97, 0.999]
    s0 = inputs.randn((b, H, dk, dv), 8103, 0.1, "f32", DEV)
    st = s0.clone()
    ho = torch.empty((b, H, N, dv), dtype=torch.float32, pin_memory=True)
    rb.retention_chunkwise_host(hq, hk, hv, g, chunk, ho, 256, state_in=st, state_out=st)
    torch.cuda.synchronize()
    want_o, want_s = oracle.chunkwise(hq, hk, hv, g, chunk, state_in=s0.cpu(),
                                      return_state=True)
    assert err_bf16(ho, want_o) < TOL_BF16
    assert err_bf16(st, want_s) < TOL_BF16


def test_streamed_bf16_output_and_fp32_inputs():
    """fp32 inputs take the CUDA-core kernel; bf16 output halves the D2H bytes."""
    b, H, N, dk, dv, chunk = 1, 2, 512, 64, 64, 64
    hq, hk, hv = host_qkv(b, H, N, dk, dv, 8200, dtype="f32")
    g = [0.9, 0.99]
    ho = torch.empty((b, H, N, dv), dtype=torch.bfloat16, pin_memory=True)
    rb.retention_chunkwise_host(hq, hk, hv, g, chunk, ho, 128)
    torch.cuda.synchronize()
    assert err_bf16(ho, oracle.chunkwise(hq, hk, hv, g, chunk)) < TOL_BF16


def test_streamed_one_segment():
    """A single segment (seg_len = N); completion is ordered on the calling stream."""
    b, H, N, dk, dv, chunk = 1, 1, 256, 128, 128, 128
    hq, hk, hv = host_qkv(b, H, N, dk, dv, 8300)
    g = [0.95]
    ho = torch.empty((b, H, N, dv), dtype=torch.float32, pin_memory=True)
    rb.retention_chunkwise_host(hq, hk, hv, g, chunk, ho, N)
    torch.cuda.current_stream().synchronize()
    assert err_bf16(ho, oracle.chunkwise(hq, hk, hv, g, chunk)) < TOL_BF16


def test_streamed_rejects_segment_not_multiple_of_chunk():
    hq, hk, hv = host_qkv(1, 1, 512, 64, 64, 8400)
    ho = torch.empty((1, 1, 512, 64), dtype=torch.float32, pin_memory=True)
    with pytest.raises(rb.RetentionError) as ei:
        rb.retention_chunkwise_host(hq, hk, hv, [0.9], 128, ho, 192)
    assert ei.value.status == rb.RET_ERR_SHAPE


def test_owned_workspace_outlives_a_non_current_stream():
    """The binding allocates the workspace on the current stream while the copies and
    kernels run on `stream` and the copy streams: memory allocated (and overwritten) on the
    current stream right after the call must not be the workspace block still in use."""
    b, H, N, dk, dv, chunk, seg = 1, 4, 4096, 256, 512, 256, 1024
    hq, hk, hv = host_qkv(b, H, N, dk, dv, 8300)
    g = inputs.gammas(H)
    nbytes = rb.chunkwise_host_workspace_bytes(hq.dtype, torch.float32, b, H, dk, dv, seg)
    s = torch.cuda.Stream()
    ho = torch.empty((b, H, N, dv), dtype=torch.float32, pin_memory=True)
    rb.retention_chunkwise_host(hq, hk, hv, g, chunk, ho, seg, stream=s)
    junk = [torch.full((nbytes // 4 + 1,), float("nan"), device=DEV) for _ in range(3)]
    s.synchronize()
    torch.cuda.synchronize()
    del junk
    assert not torch.isnan(ho).any()
    one = rb.retention_chunkwise(hq.to(DEV), hk.to(DEV), hv.to(DEV), g, chunk).cpu()
    assert err_f32(ho, one) < 1e-5
    rb.check_device_error()
