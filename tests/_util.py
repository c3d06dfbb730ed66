"""Error metrics and helpers shared by the GPU parity tests.

Tolerances (the error metrics the tests apply):
  fp32 inputs:  max_i |g_i - o_i| / max(|o_i|, rms(o)) <= 1e-4
  bf16 inputs (fp32 accumulation): max_i |g_i - o_i| / rms(o) <= 2e-2
  bf16 outputs additionally allow their own rounding: |g - o| <= 2e-2 rms(o)
  + 2^-8 |o| (an output stored in bf16 cannot be closer than half an ulp,
  2^-9 relative, and a result near a rounding boundary may take one more).
where o is the fp64 oracle and g the CUDA result.  The fp32 metric is a
relative error with the output RMS as the floor of the denominator, so that
entries that cancel to ~0 do not turn rounding noise into huge ratios.
"""
import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def as64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def err_f32(got, want):
    g, w = as64(got), as64(want)
    rms = float(np.sqrt(np.mean(w * w)))
    den = np.maximum(np.abs(w), max(rms, 1e-30))
    return float(np.max(np.abs(g - w) / den))


def err_bf16(got, want):
    g, w = as64(got), as64(want)
    rms = max(float(np.sqrt(np.mean(w * w))), 1e-30)
    return float(np.max(np.abs(g - w)) / rms)


def err_bf16_out(got, want):
    """Ratio to the bf16-output bound; <= 1 passes."""
    g, w = as64(got), as64(want)
    rms = max(float(np.sqrt(np.mean(w * w))), 1e-30)
    return float(np.max(np.abs(g - w) / (TOL_BF16 * rms + 2.0 ** -8 * np.abs(w))))


def chunkwise_tc_name(dk, dv, chunk, N):
    """Tensor-core chunkwise kernel the library picks for bf16 inputs of this shape (decays
    within the pair kernel's range): the pair-of-SMs kernel, with 256-token chunks, for
    dk 256 and dv a multiple of 128 when N is a multiple of 256 (the function does not
    depend on the chunk length); the one-SM kernel otherwise."""
    pair = dk == 256 and dv % 128 == 0 and (chunk == 256 or N % 256 == 0)
    return "chunkwise_tc_pair" if pair else "chunkwise_tc"


def parallel_tc_name(dk, dv, N, gated=False):
    """Tensor-core parallel kernel the library picks for bf16 inputs of this shape: the
    pair-of-SMs kernel for dk 256 with dv and N multiples of 256, the one-SM kernel for
    the other tensor-core shapes."""
    pair = dk == 256 and dv % 256 == 0 and N % 256 == 0 and N >= 256
    return ("parallel_gated_tc" if gated else "parallel_tc") + ("_pair" if pair else "")


def guarded(shape, dtype, device, pad=64):
    """A tensor view with `pad` sentinel elements on each side (canary guard bands)."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * pad, dtype=dtype, device=device)
    buf.fill_(float("nan")) if dtype.is_floating_point else buf.fill_(-1)
    return buf, buf[pad:pad + n].view(*shape)


def guards_intact(buf, pad=64):
    head, tail = buf[:pad], buf[-pad:]
    return bool(torch.isnan(head).all() and torch.isnan(tail).all())
