"""Tensor-core (tcgen05) parallel-form kernel against the oracle.

Shapes the tensor-core kernel takes: bf16 inputs, dk in {128, 256}, dv a multiple
of 128, any N >= 128 (a partial last query/key tile is masked), any gamma in [0, 1], all
normalisation flags.  Each test also checks that this kernel, not the CUDA-core
one, ran.  Tolerance: bf16 inputs with fp32 accumulation, 2e-2 of the output RMS
(bf16 outputs add their own rounding), as in tests/_util.py.
"""
import pytest
import torch

import oracle
from linear_recurrence_sequence_chunkwise_b300 import binding as rb
from linear_recurrence_sequence_chunkwise_b300 import inputs

from _util import TOL_BF16, err_bf16, err_bf16_out, guarded, guards_intact, parallel_tc_name

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    rb.lib()


def mk(b, H, N, dk, dv, seed, std=1.0):
    q = inputs.randn((b, H, N, dk), seed, std, "bf16", DEV)
    k = inputs.randn((b, H, N, dk), seed + 1, std, "bf16", DEV)
    v = inputs.randn((b, H, N, dv), seed + 2, std, "bf16", DEV)
    return q, k, v


@pytest.mark.parametrize("flags", [0, 1, 2, 4, 7])
@pytest.mark.parametrize("dk,dv", [(256, 512), (128, 128), (256, 384), (128, 256)])
@pytest.mark.parametrize("N", [384, 512])
def test_tc_parallel_shapes_and_flags(dk, dv, flags, N):
    """N = 512 with dk 256 and dv 512 runs on pairs of SMs; the rest on one SM."""
    b, H = 1, 2
    q, k, v = mk(b, H, N, dk, dv, 1000 + dk + dv + flags + N)
    g = [0.96875, 0.9990234375]
    got = rb.retention_parallel(q, k, v, g, flags)
    assert rb.last_kernel() == parallel_tc_name(dk, dv, N)
    assert err_bf16(got, oracle.parallel(q, k, v, g, flags)) < TOL_BF16
    rb.check_device_error()


@pytest.mark.parametrize("N", [1, 77, 128, 129, 200, 256, 520, 768])
def test_tc_parallel_ragged_sequence(N):
    """N not a multiple of the 128-row tile: the partial tiles are masked (N < 128
    goes to the CUDA-core kernel); multiples of 256 run on pairs of SMs."""
    b, H, dk, dv = 2, 2, 256, 256
    q, k, v = mk(b, H, N, dk, dv, 2000 + N)
    g = [0.9, 0.99]
    got = rb.retention_parallel(q, k, v, g, 7)
    assert rb.last_kernel() == (parallel_tc_name(dk, dv, N) if N >= 128 else "parallel_simt")
    assert err_bf16(got, oracle.parallel(q, k, v, g, 7)) < TOL_BF16


def test_tc_parallel_special_decays():
    """gamma = 0 (diagonal only) and gamma = 1 (causal linear attention)."""
    b, H, N, dk, dv = 1, 2, 300, 128, 128
    q, k, v = mk(b, H, N, dk, dv, 3000, std=0.25)
    g = [0.0, 1.0]
    for flags in (0, 2, 7):
        got = rb.retention_parallel(q, k, v, g, flags)
        assert rb.last_kernel() == "parallel_tc"
        assert err_bf16(got, oracle.parallel(q, k, v, g, flags)) < TOL_BF16, flags


@pytest.mark.parametrize("N", [260, 512])
def test_tc_parallel_bf16_output_guarded_and_repeatable(N):
    b, H, dk, dv = 2, 3, 256, 512
    q, k, v = mk(b, H, N, dk, dv, 4000 + N)
    g = inputs.gammas(H)
    buf, o = guarded((b, H, N, dv), torch.bfloat16, DEV)
    rb.retention_parallel(q, k, v, g, 7, out=o)
    first = o.clone()
    rb.retention_parallel(q, k, v, g, 7, out=o)
    torch.cuda.synchronize()
    assert rb.last_kernel() == parallel_tc_name(dk, dv, N)
    assert torch.equal(first, o)
    assert guards_intact(buf)
    assert err_bf16_out(o, oracle.parallel(q, k, v, g, 7)) < 1.0


def test_tc_parallel_matches_cuda_core_kernel_on_fp32_copy():
    """The same inputs held in fp32 take the CUDA-core kernel; both agree with the oracle."""
    b, H, N, dk, dv = 1, 2, 256, 128, 128
    q, k, v = mk(b, H, N, dk, dv, 5000)
    g = [0.95, 0.999]
    a = rb.retention_parallel(q, k, v, g, 7)
    assert rb.last_kernel() == "parallel_tc"
    c = rb.retention_parallel(q.float(), k.float(), v.float(), g, 7)
    assert rb.last_kernel() == "parallel_simt"
    want = oracle.parallel(q, k, v, g, 7)
    assert err_bf16(a, want) < TOL_BF16
    assert err_bf16(c, want) < 1e-4


# ---------------------------------------------------------------- fused gated epilogue
@pytest.mark.parametrize("dk,dv,N", [(256, 512, 256), (128, 256, 200), (256, 384, 384),
                                     (128, 128, 130), (256, 256, 512), (256, 512, 768)])
@pytest.mark.parametrize("flags", [0, 7])
def test_tc_parallel_gated_matches_oracle(dk, dv, N, flags):
    """GroupNorm over each (token, head) spans the value-column blocks of a cluster."""
    b, H = 2, 2
    q, k, v = mk(b, H, N, dk, dv, 6000 + dk + dv + N + flags)
    gate = inputs.randn((b, N, H * dv), 6100 + N, 1.0, "bf16", DEV)
    g = [0.96875, 0.999]
    got = rb.retention_parallel_gated(q, k, v, gate, g, flags, 1e-5)
    assert rb.last_kernel() == parallel_tc_name(dk, dv, N, gated=True)
    want = oracle.msr_epilogue(oracle.parallel(q, k, v, g, flags), gate, 1e-5)
    assert err_bf16(got, want) < TOL_BF16
    rb.check_device_error()


@pytest.mark.parametrize("g_dtype,out_dtype", [(torch.float32, torch.float32),
                                               (torch.bfloat16, torch.bfloat16),
                                               (torch.float32, torch.bfloat16)])
@pytest.mark.parametrize("N", [260, 512])
def test_tc_parallel_gated_affine_dtypes_guarded(g_dtype, out_dtype, N):
    b, H, dk, dv = 1, 3, 256, 512
    q, k, v = mk(b, H, N, dk, dv, 6500)
    gate = inputs.randn((b, N, H * dv), 6501, 1.0, "f32", DEV).to(g_dtype)
    w = inputs.randn((H * dv,), 6502, 1.0, "f32", DEV)
    bias = inputs.randn((H * dv,), 6503, 1.0, "f32", DEV)
    g = inputs.gammas(H)
    buf, out = guarded((b, N, H * dv), out_dtype, DEV)
    rb.retention_parallel_gated(q, k, v, gate, g, 7, 1e-5, w, bias, out=out)
    torch.cuda.synchronize()
    assert rb.last_kernel() == parallel_tc_name(dk, dv, N, gated=True)
    assert guards_intact(buf)
    want = oracle.msr_epilogue(oracle.parallel(q, k, v, g, 7), gate, 1e-5, w, bias)
    if out_dtype == torch.bfloat16:
        assert err_bf16_out(out, want) < 1.0
    else:
        assert err_bf16(out, want) < TOL_BF16


@pytest.mark.parametrize("N", [384, 512])
def test_tc_parallel_gated_equals_two_call_path(N):
    """One pass equals retention_parallel followed by msr_epilogue on the GPU."""
    b, H, dk, dv = 2, 2, 256, 512
    q, k, v = mk(b, H, N, dk, dv, 6600 + N)
    gate = inputs.randn((b, N, H * dv), 6601 + N, 1.0, "bf16", DEV)
    g = [0.9, 0.995]
    fused = rb.retention_parallel_gated(q, k, v, gate, g, 7, 1e-5)
    two = rb.msr_epilogue(rb.retention_parallel(q, k, v, g, 7), gate, 1e-5)
    assert err_bf16(fused, two.cpu().double().numpy()) < 5e-3


def test_tc_parallel_gated_unsupported_shape_is_rejected():
    q, k, v = mk(1, 1, 256, 64, 64, 6700)
    gate = inputs.randn((1, 256, 64), 6701, 1.0, "bf16", DEV)
    with pytest.raises(rb.RetentionError) as ei:
        rb.retention_parallel_gated(q, k, v, gate, [0.9], 7)
    assert ei.value.status == rb.RET_ERR_UNSUPPORTED


# ---------------------------------------------------------------- pairs of SMs: fp16 format
@pytest.mark.parametrize("gated", [False, True])
def test_pair_fp16_no_rerun_at_unit_scale(gated):
    """N(0,1) inputs: P and V stay inside fp16's range, no unit re-runs."""
    b, H, N, dk, dv = 1, 2, 512, 256, 512
    q, k, v = mk(b, H, N, dk, dv, 7000)
    g = [0.96875, 0.999]
    rb.parallel_format_reruns()
    if gated:
        gate = inputs.randn((b, N, H * dv), 7001, 1.0, "bf16", DEV)
        got = rb.retention_parallel_gated(q, k, v, gate, g, 7, 1e-5)
        want = oracle.msr_epilogue(oracle.parallel(q, k, v, g, 7), gate, 1e-5)
    else:
        got = rb.retention_parallel(q, k, v, g, 7)
        want = oracle.parallel(q, k, v, g, 7)
    assert rb.last_kernel() == parallel_tc_name(dk, dv, N, gated)
    assert rb.parallel_format_reruns() == 0
    assert err_bf16(got, want) < TOL_BF16
    rb.check_device_error()


@pytest.mark.parametrize("what", ["scores_beyond_fp16", "v_beyond_fp16", "v_below_fp16"])
@pytest.mark.parametrize("gated", [False, True])
def test_pair_reruns_units_outside_fp16(what, gated):
    """A head whose scores (|P| > 65504), V (|v| > 65504) or V scale (max |v| < 2^-6) does not
    suit fp16 is recomputed with hi/lo bf16 P inside the launch; the result still matches."""
    b, H, N, dk, dv = 1, 2, 512, 256, 512
    q, k, v = mk(b, H, N, dk, dv, 7100)
    if what == "scores_beyond_fp16":
        q[:, 1] *= 64.0
        k[:, 1] *= 64.0            # |q.k| up to ~1e5 (flags 0: no score scale)
    elif what == "v_beyond_fp16":
        v[:, 1] *= 2.0 ** 17
    else:
        v[:, 1] *= 2.0 ** -12
    g = [0.96875, 0.999]
    rb.parallel_format_reruns()
    if gated:
        gate = inputs.randn((b, N, H * dv), 7101, 1.0, "bf16", DEV)
        got = rb.retention_parallel_gated(q, k, v, gate, g, 0, 1e-5)
        want = oracle.msr_epilogue(oracle.parallel(q, k, v, g, 0), gate, 1e-5)
    else:
        got = rb.retention_parallel(q, k, v, g, 0)
        want = oracle.parallel(q, k, v, g, 0)
    assert rb.last_kernel() == parallel_tc_name(dk, dv, N, gated)
    assert rb.parallel_format_reruns() > 0
    for h in range(H):
        sl = (slice(None), slice(None), slice(h * dv, (h + 1) * dv)) if gated else (slice(None), h)
        assert err_bf16(got[sl], want[sl]) < TOL_BF16, h
    rb.check_device_error()
