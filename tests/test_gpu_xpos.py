"""retention_xpos_rotate (xPos of [RN2] "Retention" eqs.(2)-(3)) against the oracle.

fp32 at the 1e-4 relative metric (the phase is reduced in fp64, so positions near
10^6 keep fp32 accuracy), bf16 inputs and outputs at their rounding, in place, q only,
theta = 0 exactly the identity, the relative-position property of the rotated scores
on the GPU path, and the chunkwise_long shapes on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_sequence_chunkwise_b300 import binding as rb
from linear_recurrence_sequence_chunkwise_b300 import inputs

from _util import TOL_F32, err_bf16, err_bf16_out, err_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    rb.lib()


def thetas(d):
    return list(10000.0 ** (-np.arange(d // 2) / (d // 2)))


@pytest.mark.parametrize("b,H,N,dk,pos0", [(2, 3, 100, 64, 0), (1, 2, 33, 16, 12345),
                                           (1, 1, 64, 256, 999_000), (2, 1, 7, 128, 5)])
def test_fp32_parity(b, H, N, dk, pos0):
    q = inputs.randn((b, H, N, dk), 10 + dk, 1.0, "f32", DEV)
    k = inputs.randn((b, H, N, dk), 11 + dk, 1.0, "f32", DEV)
    th = thetas(dk)
    qo, ko = rb.retention_xpos_rotate(q, k, th, pos0)
    torch.cuda.synchronize()
    assert rb.last_kernel() == "xpos"
    assert err_f32(qo, oracle.xpos_rotate(q, th, pos0)) < TOL_F32
    assert err_f32(ko, oracle.xpos_rotate(k, th, pos0)) < TOL_F32


def test_bf16_in_place_and_q_only():
    b, H, N, dk = 1, 4, 300, 256
    q = inputs.randn((b, H, N, dk), 20, 1 / 16, "bf16", DEV)
    k = inputs.randn((b, H, N, dk), 21, 1 / 16, "bf16", DEV)
    th = thetas(dk)
    want_q, want_k = oracle.xpos_rotate(q, th, 77), oracle.xpos_rotate(k, th, 77)
    q2, k2 = q.clone(), k.clone()
    rb.retention_xpos_rotate(q2, k2, th, 77, q_out=q2, k_out=k2)
    qf, _ = rb.retention_xpos_rotate(q, None, th, 77, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert err_bf16_out(q2, want_q) <= 1.0 and err_bf16_out(k2, want_k) <= 1.0
    assert err_f32(qf, want_q) < TOL_F32


def test_zero_theta_is_exactly_the_identity():
    q = inputs.randn((1, 2, 50, 64), 30, 1.0, "f32", DEV)
    qo, _ = rb.retention_xpos_rotate(q, None, [0.0] * 32, 123456)
    torch.cuda.synchronize()
    assert torch.equal(qo, q)


def test_rotated_retention_depends_on_relative_position():
    """Retention over rotated Q, K (parallel form, fp32) equals the oracle's parallel
    form over the oracle's rotation, and shifting every position leaves it unchanged."""
    b, H, N, dk, dv = 1, 2, 96, 64, 32
    q = inputs.randn((b, H, N, dk), 40, 1.0, "f32", DEV)
    k = inputs.randn((b, H, N, dk), 41, 1.0, "f32", DEV)
    v = inputs.randn((b, H, N, dv), 42, 1.0, "f32", DEV)
    th, g = thetas(dk), [0.97, 0.9]
    outs = []
    for pos0 in (0, 4096):
        qr, kr = rb.retention_xpos_rotate(q, k, th, pos0)
        outs.append(rb.retention_parallel(qr, kr, v, g))
    torch.cuda.synchronize()
    want = oracle.parallel(oracle.xpos_rotate(q, th, 0), oracle.xpos_rotate(k, th, 0), v, g)
    assert err_f32(outs[0], want) < TOL_F32
    assert err_f32(outs[1], want) < TOL_F32


def test_chunkwise_long_shapes_sampled():
    w = inputs.CHUNKWISE_LONG
    q, k, _ = inputs.qkv(w, DEV)
    th = thetas(w.dk)
    qo, ko = rb.retention_xpos_rotate(q, k, th, 0)
    torch.cuda.synchronize()
    for h, n0 in ((0, 0), (15, w.N - 64)):
        sl = (slice(0, 1), slice(h, h + 1), slice(n0, n0 + 64))
        want = oracle.xpos_rotate(q[sl].contiguous(), th, n0)
        assert err_bf16_out(qo[sl], want) <= 1.0, (h, n0)
        want = oracle.xpos_rotate(k[sl].contiguous(), th, n0)
        assert err_bf16_out(ko[sl], want) <= 1.0, (h, n0)
