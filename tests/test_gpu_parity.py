"""GPU parity: the CUDA kernels, called through the C ABI, against the fp64 oracle.

Sizes here finish in seconds on the oracle and still span several tiles and a
ragged tail.  Full-size workloads are in test_gpu_fullsize.py.
Tolerances and metrics: tests/_util.py (fp32 1e-4 relative, bf16 2e-2 of RMS).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_sequence_chunkwise_b300 import binding as rb
from linear_recurrence_sequence_chunkwise_b300 import inputs

from _util import TOL_BF16, TOL_F32, err_bf16, err_bf16_out, err_f32, guarded, guards_intact

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    rb.lib()


def mk(b, H, N, dk, dv, dtype, seed, std=1.0):
    q = inputs.randn((b, H, N, dk), seed, std, dtype, DEV)
    k = inputs.randn((b, H, N, dk), seed + 1, std, dtype, DEV)
    v = inputs.randn((b, H, N, dv), seed + 2, std, dtype, DEV)
    return q, k, v


def tol(dtype):
    return (err_f32, TOL_F32) if dtype == "f32" else (err_bf16, TOL_BF16)


# ---------------------------------------------------------------- tiny workload
def test_tiny_workload_all_forms():
    """b1 H2 d16 N64 chunk16 fp32: every GPU form matches the oracle to 1e-4."""
    w = inputs.TINY
    q, k, v = inputs.qkv(w, DEV)
    want = oracle.parallel(q, k, v, w.gamma, 0)
    for flags in (0, 7):
        got = rb.retention_parallel(q, k, v, w.gamma, flags)
        assert err_f32(got, oracle.parallel(q, k, v, w.gamma, flags)) < TOL_F32
    got = rb.retention_chunkwise(q, k, v, w.gamma, w.chunk)
    assert err_f32(got, want) < TOL_F32
    state = torch.zeros(w.b, w.H, w.dk, w.dv, device=DEV)
    outs = []
    for n in range(w.N):
        outs.append(rb.retention_recurrent_step(q[:, :, n].contiguous(), k[:, :, n].contiguous(),
                                                v[:, :, n].contiguous(), state, w.gamma))
    assert err_f32(torch.stack(outs, dim=2), want) < TOL_F32


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_tiny_chunk_sizes(chunk):
    w = inputs.TINY
    q, k, v = inputs.qkv(w, DEV)
    got = rb.retention_chunkwise(q, k, v, w.gamma, chunk)
    assert err_f32(got, oracle.parallel(q, k, v, w.gamma, 0)) < TOL_F32


# ---------------------------------------------------------------- parallel form
@pytest.mark.parametrize("dtype,out_dtype", [("f32", torch.float32), ("bf16", torch.float32),
                                             ("bf16", torch.bfloat16)])
@pytest.mark.parametrize("flags", [0, 1, 2, 4, 7])
def test_parallel_ragged(dtype, out_dtype, flags):
    """N=77 (not a tile multiple), dk != dv, three heads with distinct decays."""
    b, H, N, dk, dv = 2, 3, 77, 32, 48
    q, k, v = mk(b, H, N, dk, dv, dtype, 10)
    g = [0.97, 0.8, 0.5]
    got = rb.retention_parallel(q, k, v, g, flags, out_dtype=out_dtype)
    fn, t = tol(dtype)
    if out_dtype == torch.bfloat16:
        fn, t = err_bf16_out, 1.0
    assert fn(got, oracle.parallel(q, k, v, g, flags)) < t


@pytest.mark.parametrize("flags", [0, 7])
@pytest.mark.parametrize("N", [384, 520])
def test_parallel_bf16_full_dims(flags, N):
    """dk=256, dv=512 (the workload's head dims), several 128-row tiles; N=520 ragged."""
    b, H = 1, 2
    q, k, v = mk(b, H, N, 256, 512, "bf16", 20)
    g = inputs.gammas(H)
    got = rb.retention_parallel(q, k, v, g, flags)
    assert err_bf16(got, oracle.parallel(q, k, v, g, flags)) < TOL_BF16


def test_parallel_special_decays():
    """gamma = 0 (diagonal only) and gamma = 1 (plain causal linear attention)."""
    q, k, v = mk(1, 2, 40, 16, 16, "f32", 30)
    g = [0.0, 1.0]
    for flags in (0, 2, 7):
        got = rb.retention_parallel(q, k, v, g, flags)
        assert err_f32(got, oracle.parallel(q, k, v, g, flags)) < TOL_F32


# ---------------------------------------------------------------- chunkwise form
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [16, 64, 128, 256])
def test_chunkwise_vs_oracle(dtype, chunk):
    b, H, N, dk, dv = 1, 2, 512, 64, 128
    q, k, v = mk(b, H, N, dk, dv, dtype, 40, std=0.25)
    g = inputs.gammas(H)
    got = rb.retention_chunkwise(q, k, v, g, chunk)
    fn, t = tol(dtype)
    assert fn(got, oracle.chunkwise(q, k, v, g, chunk)) < t


@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_chunkwise_bf16_full_dims(chunk):
    b, H, N = 1, 2, 768
    q, k, v = mk(b, H, N, 256, 512, "bf16", 50, std=1 / 16)
    g = [inputs.gammas(16)[0], inputs.gammas(16)[15]]
    want = oracle.chunkwise(q, k, v, g, chunk)
    got = rb.retention_chunkwise(q, k, v, g, chunk, out_dtype=torch.float32)
    assert err_bf16(got, want) < TOL_BF16
    got = rb.retention_chunkwise(q, k, v, g, chunk, out_dtype=torch.bfloat16)
    assert err_bf16_out(got, want) < 1.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunkwise_state_in_out(dtype):
    """Prefix with state_out, continuation with state_in, equal to the whole run;
    state_in and state_out may alias."""
    b, H, N, dk, dv, B = 2, 2, 256, 64, 64, 64
    q, k, v = mk(b, H, N, dk, dv, dtype, 60, std=0.3)
    g = [0.95, 0.7]
    want, s_end = oracle.chunkwise(q, k, v, g, B, return_state=True)
    st = torch.empty(b, H, dk, dv, device=DEV)
    h1 = rb.retention_chunkwise(q[:, :, :128].contiguous(), k[:, :, :128].contiguous(),
                                v[:, :, :128].contiguous(), g, B, state_out=st)
    h2 = rb.retention_chunkwise(q[:, :, 128:].contiguous(), k[:, :, 128:].contiguous(),
                                v[:, :, 128:].contiguous(), g, B, state_in=st, state_out=st)
    fn, t = tol(dtype)
    assert fn(torch.cat([h1, h2], dim=2), want) < t
    assert err_f32(st, s_end) < (TOL_F32 if dtype == "f32" else TOL_BF16)


def test_chunkwise_then_decode_steps():
    """Prefill with chunkwise (state_out), then recurrent steps continue the sequence."""
    b, H, N, extra, dk, dv = 1, 2, 128, 6, 64, 128
    q, k, v = mk(b, H, N + extra, dk, dv, "f32", 70, std=0.3)
    g = [0.9, 0.99]
    want = oracle.recurrent(q, k, v, g)
    st = torch.empty(b, H, dk, dv, device=DEV)
    pre = rb.retention_chunkwise(q[:, :, :N].contiguous(), k[:, :, :N].contiguous(),
                                 v[:, :, :N].contiguous(), g, 32, state_out=st)
    assert err_f32(pre, want[:, :, :N]) < TOL_F32
    for t in range(N, N + extra):
        o = rb.retention_recurrent_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                        v[:, :, t].contiguous(), st, g)
        assert err_f32(o, want[:, :, t]) < TOL_F32


def test_chunkwise_empty_sequence_copies_state():
    b, H, dk, dv = 1, 2, 16, 32
    si = torch.randn(b, H, dk, dv, device=DEV)
    so = torch.zeros_like(si)
    e = torch.empty(b, H, 0, dk, device=DEV)
    ev = torch.empty(b, H, 0, dv, device=DEV)
    rb.retention_chunkwise(e, e, ev, [0.5, 0.6], 16, state_in=si, state_out=so)
    torch.cuda.synchronize()
    assert torch.equal(si, so)
    rb.retention_chunkwise(e, e, ev, [0.5, 0.6], 16, state_out=so)
    torch.cuda.synchronize()
    assert float(so.abs().max()) == 0.0


# ---------------------------------------------------------------- decode step
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dims", [(256, 512), (64, 48), (16, 16)])
def test_decode_steps(dtype, dims):
    dk, dv = dims
    b, H, steps = 3, 4, 5
    g = inputs.gammas(H)
    s0 = inputs.randn((b, H, dk, dv), 80, 0.1, "f32", DEV)
    st = s0.clone()
    ref = oracle._f64(s0)
    for t in range(steps):
        q = inputs.randn((b, H, dk), 81 + 3 * t, 1 / 16, dtype, DEV)
        k = inputs.randn((b, H, dk), 82 + 3 * t, 1 / 16, dtype, DEV)
        v = inputs.randn((b, H, dv), 83 + 3 * t, 1 / 16, dtype, DEV)
        o = rb.retention_recurrent_step(q, k, v, st, g)
        o_ref, ref = oracle.recurrent_step(q, k, v, ref, g)
        assert err_f32(o, o_ref) < TOL_F32
        assert err_f32(st, ref) < TOL_F32


def test_decode_bf16_output_and_guards():
    b, H, dk, dv = 2, 2, 256, 512
    g = [0.9, 0.99]
    st = inputs.randn((b, H, dk, dv), 90, 0.1, "f32", DEV)
    ref = oracle._f64(st)
    q, k, v = (inputs.randn((b, H, d), 91 + i, 1 / 16, "bf16", DEV)
               for i, d in enumerate((dk, dk, dv)))
    buf, o = guarded((b, H, dv), torch.bfloat16, DEV)
    rb.retention_recurrent_step(q, k, v, st, g, out=o)
    o_ref, _ = oracle.recurrent_step(q, k, v, ref, g)
    torch.cuda.synchronize()
    assert err_bf16_out(o, o_ref) < 1.0
    assert guards_intact(buf)


# ---------------------------------------------------------------- epilogue
@pytest.mark.parametrize("y_dtype,g_dtype,out_dtype", [
    (torch.float32, torch.float32, torch.float32),
    (torch.float32, torch.bfloat16, torch.float32),
    (torch.bfloat16, torch.bfloat16, torch.bfloat16),
])
@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("dv", [16, 128, 512])
def test_epilogue(y_dtype, g_dtype, out_dtype, affine, dv):
    b, H, N = 2, 3, 33
    y = (torch.randn(b, H, N, dv, device=DEV) * 3 + 0.5).to(y_dtype)
    gt = torch.randn(b, N, H * dv, device=DEV).to(g_dtype)
    w = torch.randn(H * dv, device=DEV) if affine else None
    bias = torch.randn(H * dv, device=DEV) if affine else None
    buf, out = guarded((b, N, H * dv), out_dtype, DEV)
    rb.msr_epilogue(y, gt, 1e-5, w, bias, out=out)
    want = oracle.msr_epilogue(y, gt, 1e-5, w, bias)
    torch.cuda.synchronize()
    if y_dtype == torch.float32 and out_dtype == torch.float32:
        assert err_f32(out, want) < TOL_F32
    elif out_dtype == torch.bfloat16:
        assert err_bf16_out(out, want) < 1.0
    else:
        assert err_bf16(out, want) < TOL_BF16
    assert guards_intact(buf)


def test_parallel_then_epilogue_is_normalisation_invariant():
    """The pages' claim: the three score normalisations do not change the gated
    output (GroupNorm scale invariance), here through the GPU kernels."""
    b, H, N, dk, dv = 1, 2, 256, 64, 64
    q, k, v = mk(b, H, N, dk, dv, "f32", 95)
    g = [0.97, 0.9]
    gate = torch.randn(b, N, H * dv, device=DEV)
    a = rb.msr_epilogue(rb.retention_parallel(q, k, v, g, 0), gate, 0.0)
    c = rb.msr_epilogue(rb.retention_parallel(q, k, v, g, 7), gate, 0.0)
    assert err_bf16(c, a) < 1e-3


# ---------------------------------------------------------------- ABI on device
def test_misaligned_device_pointer_rejected():
    q, k, v = mk(1, 1, 64, 16, 16, "bf16", 99)
    flat = torch.zeros(1 * 1 * 64 * 16 + 8, dtype=torch.bfloat16, device=DEV)
    bad = flat[1:1 + 64 * 16].view(1, 1, 64, 16)   # 2-byte offset
    with pytest.raises(rb.RetentionError) as ei:
        rb.retention_parallel(bad, k, v, [0.5])
    assert ei.value.status == rb.RET_ERR_ALIGN


def test_outputs_untouched_on_rejected_call():
    q, k, v = mk(1, 1, 64, 16, 16, "f32", 98)
    buf, o = guarded((1, 1, 64, 16), torch.float32, DEV)
    with pytest.raises(rb.RetentionError):
        rb.retention_chunkwise(q, k, v, [0.5], 24, out=o)
    torch.cuda.synchronize()
    assert torch.isnan(buf).all()


def test_no_device_error_pending():
    rb.check_device_error()
