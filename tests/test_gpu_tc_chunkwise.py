"""Tensor-core (tcgen05) chunkwise kernel against the oracle.

Shapes the tensor-core kernel takes: bf16 inputs, dk in {128, 256}, dv a
multiple of 64, chunk in {128, 256}, every gamma with gamma^(-chunk) <= 2^64
(gamma >= 2^-0.5 at chunk 128, >= 2^-0.25 at chunk 256).  Each test also
checks that this kernel, not the CUDA-core one, ran.
"""
import pytest
import torch

import oracle
from linear_recurrence_sequence_chunkwise_b300 import binding as rb
from linear_recurrence_sequence_chunkwise_b300 import inputs

from _util import TOL_BF16, chunkwise_tc_name, err_bf16, err_bf16_out, err_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    rb.lib()


def mk(b, H, N, dk, dv, seed, std=1 / 16):
    q = inputs.randn((b, H, N, dk), seed, std, "bf16", DEV)
    k = inputs.randn((b, H, N, dk), seed + 1, std, "bf16", DEV)
    v = inputs.randn((b, H, N, dv), seed + 2, std, "bf16", DEV)
    return q, k, v


@pytest.mark.parametrize("chunk", [128, 256])
@pytest.mark.parametrize("dk,dv", [(256, 512), (128, 64), (256, 192), (128, 128), (256, 128),
                                   (256, 384)])
def test_tc_chunkwise_shapes(chunk, dk, dv):
    b, H, N = 2, 2, 1024
    q, k, v = mk(b, H, N, dk, dv, 100 + dk + dv)
    g = [0.96875, 0.9990234375]
    got = rb.retention_chunkwise(q, k, v, g, chunk)
    assert rb.last_kernel() == chunkwise_tc_name(dk, dv, chunk, N)
    assert err_bf16(got, oracle.chunkwise(q, k, v, g, chunk)) < TOL_BF16
    rb.check_device_error()


@pytest.mark.parametrize("dv", [128, 512])
def test_one_sm_kernel_at_dk256_when_n_has_no_256_split(dv):
    """chunk 128 with N = 384 (no 256-token split): the one-SM tensor-core kernel, dk 256,
    with incoming and final states."""
    b, H, N, dk = 2, 2, 384, 256
    q, k, v = mk(b, H, N, dk, dv, 150 + dv)
    g = [0.96875, 0.9990234375]
    s0 = inputs.randn((b, H, dk, dv), 151, 0.05, "f32", DEV)
    so = torch.empty_like(s0)
    got = rb.retention_chunkwise(q, k, v, g, 128, state_in=s0, state_out=so)
    assert rb.last_kernel() == "chunkwise_tc"
    want, s_end = oracle.chunkwise(q, k, v, g, 128, state_in=s0, return_state=True)
    assert err_bf16(got, want) < TOL_BF16
    assert err_f32(so, s_end) < TOL_BF16
    rb.check_device_error()


@pytest.mark.parametrize("chunk", [128, 256])
def test_tc_chunkwise_decay_range(chunk):
    """From the smallest decay the folded factors allow to almost 1."""
    b, H, N, dk, dv = 1, 4, 768, 128, 64
    q, k, v = mk(b, H, N, dk, dv, 200)
    g = [0.71 if chunk == 128 else 0.845, 0.9, 0.999, 1.0 - 2.0 ** -20]
    got = rb.retention_chunkwise(q, k, v, g, chunk)
    assert rb.last_kernel() == chunkwise_tc_name(dk, dv, chunk, N)
    assert err_bf16(got, oracle.chunkwise(q, k, v, g, chunk)) < TOL_BF16


@pytest.mark.parametrize("dv", [128, 512])
def test_tc_chunkwise_pair_decay_range(dv):
    """The pair kernel from the smallest decay the folded factors allow to almost 1."""
    b, H, N, dk = 1, 4, 768, 256
    q, k, v = mk(b, H, N, dk, dv, 250 + dv)
    g = [0.845, 0.9, 0.999, 1.0 - 2.0 ** -20]
    got = rb.retention_chunkwise(q, k, v, g, 256)
    assert rb.last_kernel() == "chunkwise_tc_pair"
    assert err_bf16(got, oracle.chunkwise(q, k, v, g, 256)) < TOL_BF16
    rb.check_device_error()


def test_tc_chunkwise_unit_scale_inputs():
    """N(0,1) inputs (outputs far from unit scale) still match to 2e-2 of RMS."""
    b, H, N, dk, dv = 1, 2, 512, 256, 128
    q, k, v = mk(b, H, N, dk, dv, 300, std=1.0)
    g = inputs.gammas(H)
    got = rb.retention_chunkwise(q, k, v, g, 256)
    assert err_bf16(got, oracle.chunkwise(q, k, v, g, 256)) < TOL_BF16


@pytest.mark.parametrize("chunk", [128, 256])
def test_tc_chunkwise_states_and_bf16_out(chunk):
    """state_in/state_out (aliased) continue a sequence exactly like one long call."""
    b, H, N, dk, dv = 2, 3, 1024, 256, 128
    q, k, v = mk(b, H, N, dk, dv, 400)
    g = [0.98, 0.995, 0.9999]
    want, s_end = oracle.chunkwise(q, k, v, g, chunk, return_state=True)
    st = torch.zeros(b, H, dk, dv, device=DEV)
    half = N // 2
    parts = []
    for lo in (0, half):
        sl = slice(lo, lo + half)
        parts.append(rb.retention_chunkwise(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(),
                                            v[:, :, sl].contiguous(), g, chunk,
                                            state_in=st if lo else None, state_out=st,
                                            out_dtype=torch.bfloat16))
        assert rb.last_kernel() == chunkwise_tc_name(dk, dv, chunk, half)
    assert err_bf16_out(torch.cat(parts, dim=2), want) < 1.0
    assert err_f32(st, s_end) < TOL_BF16


def test_tc_chunkwise_nonzero_state_in():
    b, H, N, dk, dv = 1, 2, 512, 128, 128
    q, k, v = mk(b, H, N, dk, dv, 500)
    g = [0.97, 0.995]
    s0 = inputs.randn((b, H, dk, dv), 501, 0.1, "f32", DEV)
    so = torch.empty_like(s0)
    got = rb.retention_chunkwise(q, k, v, g, 256, state_in=s0, state_out=so)
    want, s_end = oracle.chunkwise(q, k, v, g, 256, state_in=s0, return_state=True)
    assert err_bf16(got, want) < TOL_BF16
    assert err_f32(so, s_end) < TOL_BF16


@pytest.mark.parametrize("chunk,gmin,kernel", [(128, 0.70, "chunkwise_simt"),
                                              (256, 0.70, "chunkwise_simt"),
                                              (256, 0.84, "chunkwise_tc")])
def test_small_decay_schedule(chunk, gmin, kernel):
    """gamma^(-256) above 2^64 leaves the folded-factor range at 256-token chunks; 128-token
    chunks on the one-SM kernel still hold it down to gamma ~ 0.71 (the same function), and
    below that the CUDA-core kernel takes the call."""
    b, H, N, dk, dv = 1, 2, 512, 128, 64
    q, k, v = mk(b, H, N, dk, dv, 600)
    g = [gmin, 0.9]
    got = rb.retention_chunkwise(q, k, v, g, chunk)
    assert rb.last_kernel() == kernel
    assert err_bf16(got, oracle.chunkwise(q, k, v, g, chunk)) < TOL_BF16


@pytest.mark.parametrize("chunk,dv", [(128, 192), (256, 192), (256, 384)])
def test_tc_chunkwise_repeatable_and_guarded(chunk, dv):
    """Two calls give bit-identical results; guard bands around O stay intact."""
    from _util import guarded, guards_intact
    b, H, N, dk = 1, 3, 512, 256
    q, k, v = mk(b, H, N, dk, dv, 700)
    g = inputs.gammas(H)
    buf, o = guarded((b, H, N, dv), torch.float32, DEV)
    rb.retention_chunkwise(q, k, v, g, chunk, out=o)
    first = o.clone()
    rb.retention_chunkwise(q, k, v, g, chunk, out=o)
    torch.cuda.synchronize()
    assert rb.last_kernel() == chunkwise_tc_name(dk, dv, chunk, N)
    assert torch.equal(first, o)
    assert guards_intact(buf)
    assert err_bf16(o, oracle.chunkwise(q, k, v, g, chunk)) < TOL_BF16


@pytest.mark.parametrize("b,H,N,dv", [(3, 5, 256, 256), (1, 1, 512, 384), (2, 3, 768, 128)])
def test_tc_chunkwise_pair_edges(b, H, N, dv):
    """The pair kernel with one 256-token chunk, odd batch and head counts, one to three
    128-column value blocks, and an incoming state carried to the final state."""
    dk, chunk = 256, 256
    q, k, v = mk(b, H, N, dk, dv, 900 + N + dv + H)
    g = inputs.gammas(H)
    s0 = inputs.randn((b, H, dk, dv), 901 + N, 0.05, "f32", DEV)
    st = s0.clone()
    got = rb.retention_chunkwise(q, k, v, g, chunk, state_in=st, state_out=st)
    assert rb.last_kernel() == "chunkwise_tc_pair"
    want, s_end = oracle.chunkwise(q, k, v, g, chunk, state_in=s0.cpu(), return_state=True)
    assert err_bf16(got, want) < TOL_BF16
    assert err_f32(st, s_end) < TOL_BF16
    rb.check_device_error()


def test_pair_fp16_format_no_rerun_at_unit_scale_inputs():
    """The pair kernel's fp16 operands hold N(0,1)/16 inputs without re-running any unit."""
    b, H, N, dk, dv = 1, 4, 1024, 256, 512
    q, k, v = mk(b, H, N, dk, dv, 400)
    g = inputs.gammas(H)
    rb.chunkwise_format_reruns()
    got = rb.retention_chunkwise(q, k, v, g, 256)
    assert rb.last_kernel() == "chunkwise_tc_pair"
    assert rb.chunkwise_format_reruns() == 0
    assert err_bf16(got, oracle.chunkwise(q, k, v, g, 256)) < TOL_BF16
    rb.check_device_error()


@pytest.mark.parametrize("what", ["q_beyond_fp16", "scores_beyond_fp16", "v_beyond_fp16"])
def test_pair_reruns_units_that_leave_fp16_range(what):
    """A head whose Q (|q| > 65504), scores (|q.k| > 65504) or V (|v| > 65504) leave fp16's
    range re-runs its units in the bf16 hi/lo format inside the same launch: the result
    still matches the oracle, only that head's dv/128 units re-run, and an aliased incoming
    state (state_in == state_out) is still read intact by the re-run."""
    b, H, N, dk, dv = 1, 3, 768, 256, 256
    q, k, v = mk(b, H, N, dk, dv, 410)
    if what == "q_beyond_fp16":
        q[:, 1] *= 2.0 ** 21          # |q| up to ~5e5
    elif what == "scores_beyond_fp16":
        q[:, 1] *= 2.0 ** 10
        k[:, 1] *= 2.0 ** 10          # |q| below ~400, |q.k| up to ~3e5
    else:
        v[:, 1] *= 2.0 ** 21
    g = inputs.gammas(H)
    s0 = inputs.randn((b, H, dk, dv), 415, 0.05, "f32", DEV)
    st = s0.clone()
    rb.chunkwise_format_reruns()
    got = rb.retention_chunkwise(q, k, v, g, 256, state_in=st, state_out=st)
    assert rb.last_kernel() == "chunkwise_tc_pair"
    assert rb.chunkwise_format_reruns() == b * (dv // 128)
    want, want_state = oracle.chunkwise(q, k, v, g, 256, state_in=s0, return_state=True)
    for h in range(H):
        assert err_bf16(got[:, h], want[:, h]) < TOL_BF16, h
        assert err_bf16(st[:, h], want_state[:, h]) < TOL_BF16, h
    rb.check_device_error()


def test_pair_hilo_format_from_the_start_for_small_decays():
    """Decays with g^(-256) > 4096 take the bf16 hi/lo format from the first pass."""
    b, H, N, dk, dv = 1, 2, 768, 256, 128
    q, k, v = mk(b, H, N, dk, dv, 420)
    g = [0.96, 0.999]
    rb.chunkwise_format_reruns()
    got = rb.retention_chunkwise(q, k, v, g, 256)
    assert rb.last_kernel() == "chunkwise_tc_pair"
    assert rb.chunkwise_format_reruns() == 0
    assert err_bf16(got, oracle.chunkwise(q, k, v, g, 256)) < TOL_BF16
    rb.check_device_error()
