"""The gated multi-scale retention layer on the GPU, [RN2] "門控多尺度 Retention".

  * retention_gemm (C = A W on tensor cores) against an fp64 matrix product of the same
    bf16 operands, at ragged and multi-tile shapes, fp32 and bf16 outputs;
  * retention_project_heads (head-major projection with the xPos rotation in the GEMM
    epilogue) against oracle.xpos_rotate of the fp64 projection, including positions near
    10^6 (the phase is reduced exactly as fixed-point turns);
  * retention_msr_layer against oracle.msr_layer at d_model 4096 (H16 dk256 dv512), with the
    parallel form (all three normalisations) and with the chunkwise form.

Tolerances.  The GEMM's only error is fp32 accumulation of exact bf16 products: max error
over max(|c|, rms(c)) <= 1e-4.  The projection adds its bf16 output rounding (the
bf16-output bound of the core tests).  The layer rounds five intermediates to bf16 (Q, K,
V, G and the gated rows that enter W_O, each 2^-9 relative) on top of the core's own 2e-2
budget; the bound used is 3e-2 of the output RMS (measured errors are printed).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_sequence_chunkwise_b300 import binding as rb
from linear_recurrence_sequence_chunkwise_b300 import inputs

from _util import err_bf16, err_bf16_out, err_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_LAYER = 3e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    rb.lib()


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("M,Nc,K", [(128, 256, 64), (300, 512, 512), (1024, 768, 4096),
                                    (77, 256, 320)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_against_fp64_product(M, Nc, K, out_dtype):
    a = inputs.randn((M, K), 500 + M, 1.0, "bf16", DEV)
    w = inputs.randn((K, Nc), 501 + Nc, K ** -0.5, "bf16", DEV)
    c = rb.retention_gemm(a, w, out_dtype=out_dtype)
    assert rb.last_kernel() == "gemm_tc"
    want = f64(a) @ f64(w)
    if out_dtype == torch.float32:
        assert err_f32(c, want) < 1e-4
    else:
        assert err_bf16_out(c, want) < 1.0
    rb.check_device_error()


@pytest.mark.parametrize("d,H,pos0", [(256, 2, 0), (128, 4, 1_000_003), (64, 8, 77)])
def test_project_heads_with_fused_xpos(d, H, pos0):
    b, N, d_in = 2, 256, 512
    x = inputs.randn((b, N, d_in), 510, 1.0, "bf16", DEV)
    w = inputs.randn((d_in, H * d), 511, d_in ** -0.5, "bf16", DEV)
    theta = [10000.0 ** (-j / (d // 2)) for j in range(d // 2)]
    got = rb.retention_project_heads(x, w, H, d, theta, pos0)
    assert rb.last_kernel() == "gemm_tc"
    heads = (f64(x) @ f64(w)).reshape(b, N, H, d).transpose(0, 2, 1, 3)
    want = oracle.xpos_rotate(np.ascontiguousarray(heads), theta, pos0)
    assert err_bf16_out(got, want) < 1.0
    plain = rb.retention_project_heads(x, w, H, d)           # no rotation
    assert err_bf16_out(plain, heads) < 1.0
    rb.check_device_error()


def layer_inputs(b, N, D, H, dk, dv, Dout, seed):
    x = inputs.randn((b, N, D), seed, 1.0, "bf16", DEV)
    s = D ** -0.5
    wq = inputs.randn((D, H * dk), seed + 1, s, "bf16", DEV)
    wk = inputs.randn((D, H * dk), seed + 2, s, "bf16", DEV)
    wv = inputs.randn((D, H * dv), seed + 3, s, "bf16", DEV)
    wg = inputs.randn((D, H * dv), seed + 4, s, "bf16", DEV)
    wo = inputs.randn((H * dv, Dout), seed + 5, (H * dv) ** -0.5, "bf16", DEV)
    return x, wq, wk, wv, wg, wo


@pytest.mark.parametrize("form", ["parallel", "chunkwise"])
def test_msr_layer_d_model_4096(form):
    b, N, D, H, dk, dv, Dout = 1, 256, 4096, 16, 256, 512, 4096
    x, wq, wk, wv, wg, wo = layer_inputs(b, N, D, H, dk, dv, Dout, 520)
    gamma = inputs.gammas(H)
    theta = [10000.0 ** (-j / (dk // 2)) for j in range(dk // 2)]
    flags, chunk = (7, 0) if form == "parallel" else (0, 128)
    got = rb.retention_msr_layer(x, wq, wk, wv, wg, wo, gamma, theta, pos0=5, flags=flags,
                                 eps=1e-5, chunk=chunk)
    rb.check_device_error()
    assert rb.last_kernel() == "gemm_tc"
    want = oracle.msr_layer(x, wq, wk, wv, wg, wo, gamma, theta, flags=flags, eps=1e-5, pos0=5,
                            chunk=chunk or None)
    e = err_bf16(got, want)
    print(f"msr_layer {form}: max error / rms = {e:.4f}")
    assert e < TOL_LAYER


def test_msr_layer_bf16_out_and_small_shape():
    b, N, D, H, dk, dv, Dout = 2, 128, 512, 2, 128, 128, 256
    x, wq, wk, wv, wg, wo = layer_inputs(b, N, D, H, dk, dv, Dout, 530)
    gamma = [0.9, 0.99]
    got = rb.retention_msr_layer(x, wq, wk, wv, wg, wo, gamma, None, out_dtype=torch.bfloat16)
    want = oracle.msr_layer(x, wq, wk, wv, wg, wo, gamma, None)
    assert err_bf16(got, want) < TOL_LAYER
    rb.check_device_error()
