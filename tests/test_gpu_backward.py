"""retention_chunkwise_backward against the oracle's gradient (exact per-entry sums).

The oracle's gradient is pinned in test_oracle_backward.py by exact central
differences of the forward oracle.  Here the CUDA kernel is compared with it element
by element: fp32 inputs at the 1e-4 relative metric, bf16 inputs at 2e-2 of the RMS
(fp32 accumulation), over several chunks, ragged 64-column slices (dk or dv not a
multiple of 64), both states, gamma 0 and 1, and the full-size training-sweep shape
on sampled (batch, head) units.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_sequence_chunkwise_b300 import binding as rb
from linear_recurrence_sequence_chunkwise_b300 import inputs

from _util import TOL_BF16, TOL_F32, err_bf16, err_bf16_out, err_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    rb.lib()


def make(b, H, N, dk, dv, seed, dtype="f32", std=1.0, states=True):
    q = inputs.randn((b, H, N, dk), seed, std, dtype, DEV)
    k = inputs.randn((b, H, N, dk), seed + 1, std, dtype, DEV)
    v = inputs.randn((b, H, N, dv), seed + 2, std, dtype, DEV)
    do = inputs.randn((b, H, N, dv), seed + 3, std, dtype, DEV)
    s0 = inputs.randn((b, H, dk, dv), seed + 4, 0.1, "f32", DEV) if states else None
    ds = inputs.randn((b, H, dk, dv), seed + 5, 0.1, "f32", DEV) if states else None
    return q, k, v, do, s0, ds


def tc_applies(q, gamma, dk, dv, N):
    """The shapes retention_chunkwise_backward_ws runs as tensor-core passes."""
    return (q.dtype == torch.bfloat16 and dk == 256 and dv % 256 == 0 and N % 256 == 0
            and all(0.0 < g and g ** -256 <= 2.0 ** 64 for g in gamma))


def run(q, k, v, do, gamma, chunk, s0=None, ds=None, out_dtype=torch.float32, cuda_cores=False):
    b, H, N, dk = q.shape
    dv = v.shape[-1]
    di = torch.full((b, H, dk, dv), float("nan"), device=DEV)
    gq, gk, gv, di = rb.retention_chunkwise_backward(q, k, v, do, gamma, chunk, state_in=s0,
                                                     dstate_out=ds, dstate_in=di,
                                                     out_dtype=out_dtype, cuda_cores=cuda_cores)
    torch.cuda.synchronize()
    tc = not cuda_cores and tc_applies(q, gamma, dk, dv, N)
    assert rb.last_kernel() == ("chunkwise_backward_tc" if tc else "chunkwise_backward_simt")
    return gq, gk, gv, di


# N a multiple of 64 takes the register-blocked kernel (64-token chunks whatever the
# chunk argument); other N the 16-row kernel with the caller's chunk.
@pytest.mark.parametrize("b,H,N,dk,dv,chunk", [(1, 2, 128, 64, 128, 32), (2, 3, 256, 48, 80, 64),
                                               (1, 2, 96, 256, 512, 16), (1, 1, 512, 128, 64, 256),
                                               (1, 2, 80, 64, 48, 16), (2, 1, 160, 32, 96, 32),
                                               (1, 1, 192, 256, 512, 48)])
def test_fp32_parity(b, H, N, dk, dv, chunk):
    gamma = [0.97, 0.6, 0.999][:H]
    q, k, v, do, s0, ds = make(b, H, N, dk, dv, 100 + dk + dv + chunk)
    got = run(q, k, v, do, gamma, chunk, s0, ds)
    want = oracle.chunkwise_backward(q, k, v, do, gamma, state_in=s0, dstate_out=ds)
    for name, g, w in zip(("dq", "dk", "dv", "dstate_in"), got, want):
        assert err_f32(g, w) < TOL_F32, name


@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_bf16_parity_training_dims(chunk):
    """dk 256, dv 512 as in the training sweep, decays of the sweep's fastest and
    slowest heads, N spanning several chunks."""
    b, H, N, dk, dv = 1, 2, 512, 256, 512
    gamma = [inputs.gammas(16)[0], inputs.gammas(16)[15]]
    q, k, v, do, s0, ds = make(b, H, N, dk, dv, 300 + chunk, "bf16", 1 / 16)
    got = run(q, k, v, do, gamma, chunk, s0, ds)
    want = oracle.chunkwise_backward(q, k, v, do, gamma, state_in=s0, dstate_out=ds)
    for name, g, w in zip(("dq", "dk", "dv", "dstate_in"), got, want):
        assert err_bf16(g, w) < TOL_BF16, name


def test_bf16_outputs():
    b, H, N, dk, dv, chunk = 1, 2, 256, 128, 128, 64
    q, k, v, do, s0, ds = make(b, H, N, dk, dv, 400, "bf16", 1 / 16)
    gq, gk, gv, di = run(q, k, v, do, [0.9, 0.99], chunk, s0, ds, out_dtype=torch.bfloat16)
    want = oracle.chunkwise_backward(q, k, v, do, [0.9, 0.99], state_in=s0, dstate_out=ds)
    for g, w in zip((gq, gk, gv), want[:3]):
        assert g.dtype == torch.bfloat16
        assert err_bf16_out(g, w) <= 1.0
    assert err_bf16(di, want[3]) < TOL_BF16


def test_no_states_and_extreme_decays():
    """gamma 0 (only the diagonal term), 1 (plain prefix sums) and a mid value; no
    incoming state and no state gradient."""
    b, H, N, dk, dv, chunk = 1, 3, 192, 64, 64, 64
    gamma = [0.0, 1.0, 0.5]
    q, k, v, do, _, _ = make(b, H, N, dk, dv, 500, states=False)
    got = run(q, k, v, do, gamma, chunk)
    want = oracle.chunkwise_backward(q, k, v, do, gamma)
    for name, g, w in zip(("dq", "dk", "dv", "dstate_in"), got, want):
        assert err_f32(g, w) < TOL_F32, name


def test_both_kernels_agree_on_the_causal_prefix():
    """dq_n depends on tokens m <= n only, so dq of a 192-token sequence (register-blocked
    kernel, 64-token chunks) equals the first 192 rows of dq of the same sequence extended
    to 208 tokens (16-row kernel, chunk 16)."""
    b, H, dk, dv = 1, 2, 64, 128
    q, k, v, do, s0, _ = make(b, H, 208, dk, dv, 600)
    short = [t[:, :, :192].contiguous() for t in (q, k, v, do)]
    dq_long = run(q, k, v, do, [0.95, 0.8], 16, s0)[0]
    dq_short = run(*short, [0.95, 0.8], 16, s0)[0]
    assert err_f32(dq_short, dq_long[:, :, :192]) < 1e-5


def test_empty_sequence_passes_the_state_gradient_through():
    b, H, dk, dv = 2, 2, 64, 64
    e = torch.empty((b, H, 0, dk), device=DEV)
    ev = torch.empty((b, H, 0, dv), device=DEV)
    ds = inputs.randn((b, H, dk, dv), 700, 1.0, "f32", DEV)
    di = torch.full_like(ds, float("nan"))
    rb.retention_chunkwise_backward(e, e, ev, ev, [0.9, 0.5], 64, dstate_out=ds, dstate_in=di)
    torch.cuda.synchronize()
    assert torch.equal(di, ds)
    rb.retention_chunkwise_backward(e, e, ev, ev, [0.9, 0.5], 64, dstate_in=di)
    torch.cuda.synchronize()
    assert torch.count_nonzero(di) == 0


def test_full_size_training_shape_sampled():
    """b4 H16 N2048 dk256 dv512 chunk 64 (the shape bench.py times): the GPU computes all
    64 (batch, head) units; the oracle recomputes two of them (fastest and slowest decay)."""
    w = inputs.BACKWARD
    q, k, v = inputs.qkv(w, DEV)
    do = inputs.dout(w, DEV)
    gq, gk, gv, _ = rb.retention_chunkwise_backward(q, k, v, do, w.gamma, w.chunk)
    torch.cuda.synchronize()
    assert rb.last_kernel() == "chunkwise_backward_tc"
    idx = [(0, 0), (3, 15)]
    us = [(bi, h) + tuple(t[bi:bi + 1, h:h + 1].cpu() for t in (q, k, v, do)) for bi, h in idx]
    outs = oracle.map_units(
        lambda u: oracle.chunkwise_backward(u[2], u[3], u[4], u[5], [w.gamma[u[1]]]),
        us, threads=len(us))
    for (bi, h, *_), want in zip(us, outs):
        for name, g, wnt in zip(("dq", "dk", "dv"), (gq, gk, gv), want[:3]):
            assert err_bf16(g[bi:bi + 1, h:h + 1], wnt) < TOL_BF16, (bi, h, name)


# Tensor-core passes (retention_chunkwise_backward_ws): bf16, dk 256, dv 256 or 512.
@pytest.mark.parametrize("dv,N,states", [(512, 512, True), (256, 768, True), (512, 256, False)])
def test_tensor_core_passes_against_the_oracle(dv, N, states):
    b, H, dk = 2, 2, 256
    gamma = [inputs.gammas(16)[0], 1.0 - 2.0 ** -12]
    q, k, v, do, s0, ds = make(b, H, N, dk, dv, 800 + dv + N, "bf16", 1 / 16, states=states)
    got = run(q, k, v, do, gamma, 64, s0, ds)
    want = oracle.chunkwise_backward(q, k, v, do, gamma, state_in=s0, dstate_out=ds)
    for name, g, w in zip(("dq", "dk", "dv", "dstate_in"), got, want):
        assert err_bf16(g, w) < TOL_BF16, name
    rb.check_device_error()


def test_tensor_core_passes_match_the_cuda_core_kernel_and_bf16_grads():
    b, H, N, dk, dv = 1, 2, 512, 256, 512
    gamma = [0.97, 0.995]
    q, k, v, do, s0, ds = make(b, H, N, dk, dv, 850, "bf16", 1 / 16)
    tc = run(q, k, v, do, gamma, 128, s0, ds)
    cc = run(q, k, v, do, gamma, 128, s0, ds, cuda_cores=True)
    for name, a, c in zip(("dq", "dk", "dv", "dstate_in"), tc, cc):
        assert err_bf16(a, c) < TOL_BF16, name
    want = oracle.chunkwise_backward(q, k, v, do, gamma, state_in=s0, dstate_out=ds)
    g16 = run(q, k, v, do, gamma, 128, s0, ds, out_dtype=torch.bfloat16)
    for g, w in zip(g16[:3], want[:3]):
        assert g.dtype == torch.bfloat16
        assert err_bf16_out(g, w) <= 1.0
    rb.check_device_error()


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tensor_core_passes_with_operands_beyond_fp16(out_dtype):
    """dout of head 0 scaled by 2^20 (|dout| up to ~2^18): the passes that read dout as Q,
    as keys or as values leave fp16's range and run their units in the hi/lo format.  The
    second half of dq and dk adds to the first half's output, so a re-run must not add twice.
    The gradient is linear in dout: each head is compared with the oracle at its own scale."""
    b, H, N, dk, dv = 1, 2, 512, 256, 512
    gamma = [0.97, 0.995]
    q, k, v, do, s0, ds = make(b, H, N, dk, dv, 900, "bf16", 1 / 16)
    do[:, 0] *= 2.0 ** 20
    rb.chunkwise_format_reruns()
    got = run(q, k, v, do, gamma, 64, s0, ds, out_dtype=out_dtype)
    reruns = rb.chunkwise_format_reruns()
    assert reruns > 0
    want = oracle.chunkwise_backward(q, k, v, do, gamma, state_in=s0, dstate_out=ds)
    for name, g, w in zip(("dq", "dk", "dv", "dstate_in"), got, want):
        for h in range(H):
            gh, wh = g[:, h:h + 1], np.asarray(w)[:, h:h + 1]
            if out_dtype == torch.bfloat16 and name != "dstate_in":
                assert err_bf16_out(gh, wh) <= 1.0, (name, h)
            else:
                assert err_bf16(gh, wh) < TOL_BF16, (name, h)
    rb.check_device_error()
