"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

The GPU computes the whole workload; the oracle recomputes sampled (batch,
head) units in full (each unit is independent of the others), on host threads.
Workloads: parallel_norm (b8 H8 N2048), chunkwise_long (b1 H16 N32768 chunk 256),
the chunkwise sweep (b4 H16, N x chunk grid) and decode (b128 H16, 512 steps).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_sequence_chunkwise_b300 import binding as rb
from linear_recurrence_sequence_chunkwise_b300 import inputs

from _util import TOL_BF16, TOL_F32, err_bf16, err_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    rb.lib()


def units_of(q, k, v, idx):
    """Host copies of the (b, h) units in idx."""
    return [(bi, h, q[bi:bi + 1, h:h + 1].cpu(), k[bi:bi + 1, h:h + 1].cpu(),
             v[bi:bi + 1, h:h + 1].cpu()) for bi, h in idx]


def test_chunkwise_long_full():
    w = inputs.CHUNKWISE_LONG
    q, k, v = inputs.qkv(w, DEV)
    out = rb.retention_chunkwise(q, k, v, w.gamma, w.chunk)
    kern = rb.last_kernel()
    rb.check_device_error()
    assert kern == "chunkwise_tc_pair"
    assert torch.isfinite(out).all()
    idx = [(0, 0), (0, 15)]
    us = units_of(q, k, v, idx)
    outs = oracle.map_units(lambda u: oracle.chunkwise(u[2], u[3], u[4], [w.gamma[u[1]]], w.chunk),
                            us, threads=len(us))
    for (bi, h, *_), want in zip(us, outs):
        assert err_bf16(out[bi:bi + 1, h:h + 1], want) < TOL_BF16, (bi, h)


@pytest.mark.parametrize("N,chunk", [(2048, 64), (2048, 128), (2048, 256), (8192, 64),
                                     (8192, 128), (8192, 256), (16384, 64), (16384, 128),
                                     (16384, 256)])
def test_sweep_point(N, chunk):
    w = [x for x in inputs.SWEEP if x.N == N and x.chunk == chunk][0]
    q, k, v = inputs.qkv(w, DEV)
    out = rb.retention_chunkwise(q, k, v, w.gamma, w.chunk, out_dtype=torch.bfloat16)
    rb.check_device_error()
    # every point on tensor cores, with the 256-token schedule (the same function)
    assert rb.last_kernel() == "chunkwise_tc_pair"
    idx = [(3, 0), (1, 9)]
    us = units_of(q, k, v, idx)
    outs = oracle.map_units(lambda u: oracle.chunkwise(u[2], u[3], u[4], [w.gamma[u[1]]], w.chunk),
                            us, threads=len(us))
    for (bi, h, *_), want in zip(us, outs):
        got = out[bi:bi + 1, h:h + 1].float()
        rms = float(np.sqrt(np.mean(want ** 2)))
        diff = np.abs(got.cpu().double().numpy() - want)
        assert float(np.max(diff / (TOL_BF16 * rms + 2.0 ** -8 * np.abs(want)))) < 1.0, (bi, h)


def test_parallel_norm_full_with_epilogue():
    w = inputs.PARALLEL_NORM
    q, k, v = inputs.qkv(w, DEV)
    g = inputs.gate(w, DEV)
    y = rb.retention_parallel(q, k, v, w.gamma, w.flags)
    out = rb.msr_epilogue(y, g, w.eps)
    rb.check_device_error()
    idx = [(0, 0), (7, 7), (3, 4)]
    us = units_of(q, k, v, idx)
    ys = oracle.map_units(lambda u: oracle.parallel(u[2], u[3], u[4], [w.gamma[u[1]]], w.flags),
                          us, threads=len(us))
    for (bi, h, *_), want in zip(us, ys):
        assert err_bf16(y[bi:bi + 1, h:h + 1], want) < TOL_BF16, (bi, h)
        gu = g[bi:bi + 1, :, h * w.dv:(h + 1) * w.dv].cpu()
        want_o = oracle.msr_epilogue(want, gu, w.eps)
        got_o = out[bi:bi + 1, :, h * w.dv:(h + 1) * w.dv]
        assert err_bf16(got_o, want_o) < TOL_BF16, (bi, h)


def test_parallel_norm_full_fused_gated():
    """The one-pass parallel + gated epilogue call bench.py times, at full size."""
    w = inputs.PARALLEL_NORM
    q, k, v = inputs.qkv(w, DEV)
    g = inputs.gate(w, DEV)
    out = rb.retention_parallel_gated(q, k, v, g, w.gamma, w.flags, w.eps)
    assert rb.last_kernel() == "parallel_gated_tc_pair"
    rb.check_device_error()
    idx = [(0, 0), (7, 7), (5, 2)]
    us = units_of(q, k, v, idx)
    ys = oracle.map_units(lambda u: oracle.parallel(u[2], u[3], u[4], [w.gamma[u[1]]], w.flags),
                          us, threads=len(us))
    for (bi, h, *_), y in zip(us, ys):
        gu = g[bi:bi + 1, :, h * w.dv:(h + 1) * w.dv].cpu()
        want = oracle.msr_epilogue(y, gu, w.eps)
        assert err_bf16(out[bi:bi + 1, :, h * w.dv:(h + 1) * w.dv], want) < TOL_BF16, (bi, h)


def test_decode_full_512_steps():
    w = inputs.DECODE
    s0 = inputs.decode_state(w, DEV)
    st = s0.clone()
    qs, ks, vs = inputs.decode_all_inputs(w, DEV)
    outs = torch.empty(w.steps, w.b, w.H, w.dv, device=DEV)
    for t in range(w.steps):
        rb.retention_recurrent_step(qs[t], ks[t], vs[t], st, w.gamma, out=outs[t])
    rb.check_device_error()
    idx = [(0, 0), (127, 15), (64, 7), (5, 11)]

    def unit(bh):
        bi, h = bh
        # 512 decode steps of one unit == the recurrent form over 512 tokens from S0
        qq = qs[:, bi, h].cpu()[None, None]
        kk = ks[:, bi, h].cpu()[None, None]
        vv = vs[:, bi, h].cpu()[None, None]
        return oracle.recurrent(qq, kk, vv, [w.gamma[h]], state_in=s0[bi:bi + 1, h:h + 1].cpu(),
                                return_state=True)

    res = oracle.map_units(unit, idx, threads=len(idx))
    for (bi, h), (o_ref, s_ref) in zip(idx, res):
        assert err_f32(outs[:, bi, h], o_ref[0, 0]) < TOL_F32, (bi, h)
        assert err_f32(st[bi:bi + 1, h:h + 1], s_ref) < TOL_F32, (bi, h)
