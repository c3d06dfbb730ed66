"""rglru_scan (RG-LRU of the Griffin page) against the oracle.

fp32 inputs at the 1e-4 relative metric, bf16 inputs at 2e-2 of the RMS; T not a
multiple of the kernel's segment or tile, several 64-channel blocks per row, the
incoming and final states, gates driven to their limits, and the full-size workload
(b8 T4096 D4096) on sampled channels.
"""
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


def make(b, T, D, seed, dtype="f32"):
    x = inputs.randn((b, T, D), seed, 1.0, dtype, DEV)
    ga = inputs.randn((b, T, D), seed + 1, 1.0, dtype, DEV)
    gx = inputs.randn((b, T, D), seed + 2, 1.0, dtype, DEV)
    lam = inputs.rglru_lambda(D, seed + 3, 8.0, DEV)
    h0 = inputs.randn((b, D), seed + 4, 1.0, "f32", DEV)
    return x, ga, gx, lam, h0


@pytest.mark.parametrize("b,T,D", [(2, 100, 64), (1, 257, 192), (3, 16, 64), (2, 1, 128),
                                   (1, 1000, 64)])
def test_fp32_parity(b, T, D):
    x, ga, gx, lam, h0 = make(b, T, D, 100 + T + D)
    hl = torch.full((b, D), float("nan"), device=DEV)
    y = rb.rglru_scan(x, ga, gx, lam, h0, 8.0, h_last=hl)
    torch.cuda.synchronize()
    assert rb.last_kernel() == "rglru"
    want, want_h = oracle.rglru(x, ga, gx, lam, h0, 8.0, return_state=True)
    assert err_f32(y, want) < TOL_F32
    assert err_f32(hl, want_h) < TOL_F32


def test_bf16_parity_and_bf16_output():
    b, T, D = 2, 1000, 256
    x, ga, gx, lam, _ = make(b, T, D, 200, "bf16")
    y = rb.rglru_scan(x, ga, gx, lam)
    yb = rb.rglru_scan(x, ga, gx, lam, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    want = oracle.rglru(x, ga, gx, lam)
    assert err_bf16(y, want) < TOL_BF16
    assert err_bf16_out(yb, want) <= 1.0


@pytest.mark.parametrize("T", [1, 63, 65, 130])
def test_bf16_states_gate_limits_and_ragged_tiles(T):
    """bf16 inputs (the TMA-fed kernel, 64-step tiles): incoming and final states, T below,
    just above and across tile boundaries, the recurrence gate closed on 8 channels, a = 0
    and a = 1 on 8 channels each."""
    b, D = 3, 128
    x, ga, gx, lam, h0 = make(b, T, D, 500 + T, "bf16")
    ga[:, :, :8] = -1e4
    lam[8:16] = -1e4
    lam[16:24] = 1e4
    hl = torch.full((b, D), float("nan"), device=DEV)
    y = rb.rglru_scan(x, ga, gx, lam, h0, 8.0, h_last=hl)
    torch.cuda.synchronize()
    assert rb.last_kernel() == "rglru"
    want, want_h = oracle.rglru(x, ga, gx, lam, h0, 8.0, return_state=True)
    assert err_bf16(y, want) < TOL_BF16
    assert err_bf16(hl, want_h) < TOL_BF16
    # r = 0 gives a_t = 1 and a zero input weight exactly: the state passes unchanged
    assert torch.equal(y[:, :, :8], h0[:, None, :8].expand(b, T, 8))
    assert torch.equal(hl[:, :8], h0[:, :8])
    rb.check_device_error()


def test_gate_limits_and_other_c():
    """Recurrence gate closed (r = 0: h stays h0), decay a = 0 (h = i x), a = 1, and
    c = 1 and 3.5 besides the page's 8."""
    b, T, D = 2, 40, 64
    x, ga, gx, lam, h0 = make(b, T, D, 300)
    ga[:, :, :8] = -1e4
    lam[8:16] = -1e4
    lam[16:24] = 1e4
    for c in (8.0, 1.0, 3.5):
        y = rb.rglru_scan(x, ga, gx, lam, h0, c)
        torch.cuda.synchronize()
        assert err_f32(y, oracle.rglru(x, ga, gx, lam, h0, c)) < TOL_F32, c
    assert torch.equal(y[:, :, :8], h0[:, None, :8].expand(b, T, 8))


def test_empty_sequence_copies_the_state():
    b, D = 2, 64
    e = torch.empty((b, 0, D), device=DEV)
    lam = torch.zeros(D, device=DEV)
    h0 = inputs.randn((b, D), 400, 1.0, "f32", DEV)
    hl = torch.full_like(h0, float("nan"))
    rb.rglru_scan(e, e, e, lam, h0, h_last=hl)
    torch.cuda.synchronize()
    assert torch.equal(hl, h0)
    rb.rglru_scan(e, e, e, lam, h_last=hl)
    torch.cuda.synchronize()
    assert torch.count_nonzero(hl) == 0


def test_full_size_sampled_channels():
    """b8 T4096 D4096 (the shape bench.py times): the GPU scans all channels; the oracle
    recomputes 64 channels of two batch rows (channels are independent)."""
    w = inputs.RGLRU
    x, ga, gx, lam = inputs.rglru_inputs(w, DEV)
    y = rb.rglru_scan(x, ga, gx, lam)
    torch.cuda.synchronize()
    for bi, d0 in ((0, 0), (7, 4032)):
        sl = (slice(bi, bi + 1), slice(None), slice(d0, d0 + 64))
        want = oracle.rglru(*(t[sl].contiguous() for t in (x, ga, gx)), lam[d0:d0 + 64])
        assert err_bf16(y[sl], want) < TOL_BF16, (bi, d0)
