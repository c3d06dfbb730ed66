"""Host-side checks of the C ABI (no GPU needed; no call here reaches a launch).

The library must load, export every function include/retention.h declares,
and reject bad arguments with the documented status codes before touching the
GPU.  Fake pointers are never dereferenced: every call below fails validation.
"""
import ctypes
import subprocess

import pytest

from linear_recurrence_sequence_chunkwise_b300 import binding, build

A = ctypes.c_void_p(0x100000)       # 16-byte aligned, never dereferenced
A2 = ctypes.c_void_p(0x200000)
MIS = ctypes.c_void_p(0x100004)     # not 16-byte aligned
NUL = None
S = ctypes.c_void_p(0)              # default stream handle, never used here


def G(*vals):
    return (ctypes.c_double * len(vals))(*vals)


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def test_exports_every_declared_function(L):
    names = binding.header_functions()
    assert set(names) == {"retention_parallel", "retention_chunkwise", "retention_recurrent_step",
                          "msr_epilogue", "retention_status_string",
                          "retention_check_device_error", "retention_kernel_launches",
                          "retention_last_kernel", "retention_last_cuda_error",
                          "retention_cuda_error_string", "retention_parallel_gated",
                          "retention_chunkwise_host", "retention_chunkwise_host_workspace_bytes",
                          "retention_chunkwise_host_noalloc",
                          "retention_chunkwise_host_static_scratch_bytes",
                          "retention_chunkwise_backward", "rglru_scan",
                          "retention_xpos_rotate", "retention_chunkwise_format_reruns",
                          "retention_parallel_format_reruns",
                          "retention_chunkwise_wait_selftest", "retention_msr_layer",
                          "retention_msr_layer_workspace_bytes", "retention_gemm",
                          "retention_project_heads", "retention_chunkwise_backward_ws",
                          "retention_chunkwise_backward_workspace_bytes"}
    for n in names:
        assert getattr(L, n) is not None
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


def test_launch_counter_starts_at_zero_and_rejections_do_not_count(L):
    before = binding.kernel_launches()
    assert par(L, dk=24) == binding.RET_ERR_UNSUPPORTED
    assert binding.kernel_launches() == before


def test_cuda_error_query(L):
    assert L.retention_last_cuda_error() == 0          # nothing has failed on this thread
    assert binding.lib().retention_cuda_error_string(0).startswith(b"cudaSuccess")
    assert b"cudaErrorLaunchOutOfResources" in binding.lib().retention_cuda_error_string(701)


def test_status_strings(L):
    for code in range(8):
        assert binding.status_string(code)
    assert binding.status_string(99) == "unknown status"
    assert binding.status_string(0) == "ok"


def par(L, q=A, k=A, v=A, o=A2, it=1, ot=0, b=1, H=2, N=64, dk=64, dv=64, g=None, flags=0):
    g = G(0.9, 0.5) if g is None else g
    return L.retention_parallel(q, k, v, o, it, ot, b, H, N, dk, dv, g, flags, S)


def chk(L, q=A, k=A, v=A, o=A2, it=1, ot=0, b=1, H=2, N=64, dk=64, dv=64, chunk=16, g=None,
        si=None, so=None):
    g = G(0.9, 0.5) if g is None else g
    return L.retention_chunkwise(q, k, v, o, it, ot, b, H, N, dk, dv, chunk, g, si, so, S)


def dec(L, q=A, k=A, v=A, st=A2, o=A2, it=1, ot=0, b=1, H=2, dk=64, dv=64, g=None):
    g = G(0.9, 0.5) if g is None else g
    return L.retention_recurrent_step(q, k, v, st, o, it, ot, b, H, dk, dv, g, S)


def epi(L, y=A, g=A, o=A2, yt=0, gt=1, ot=0, b=1, H=2, N=8, dv=64, eps=1e-5, w=None, bias=None):
    return L.msr_epilogue(y, g, o, yt, gt, ot, b, H, N, dv, ctypes.c_float(eps), w, bias, S)


def test_parallel_rejections(L):
    assert par(L, b=-1) == binding.RET_ERR_SHAPE
    assert par(L, N=-3) == binding.RET_ERR_SHAPE
    assert par(L, it=2) == binding.RET_ERR_DTYPE
    assert par(L, ot=-1) == binding.RET_ERR_DTYPE
    assert par(L, flags=8) == binding.RET_ERR_UNSUPPORTED
    assert par(L, dk=24) == binding.RET_ERR_UNSUPPORTED
    assert par(L, dk=512) == binding.RET_ERR_UNSUPPORTED
    assert par(L, dv=528) == binding.RET_ERR_UNSUPPORTED
    assert par(L, q=NUL) == binding.RET_ERR_NULL
    assert par(L, g=ctypes.POINTER(ctypes.c_double)()) == binding.RET_ERR_NULL
    assert par(L, v=MIS) == binding.RET_ERR_ALIGN
    assert par(L, o=MIS) == binding.RET_ERR_ALIGN
    assert par(L, g=G(0.9, 1.5)) == binding.RET_ERR_UNSUPPORTED
    assert par(L, g=G(-0.1, 0.5)) == binding.RET_ERR_UNSUPPORTED
    assert par(L, g=G(float("nan"), 0.5)) == binding.RET_ERR_UNSUPPORTED
    assert par(L, H=129, g=G(*([0.5] * 129))) == binding.RET_ERR_UNSUPPORTED


def test_empty_inputs_launch_nothing(L):
    assert par(L, b=0, q=NUL, k=NUL, v=NUL, o=NUL) == binding.RET_OK
    assert par(L, N=0, q=NUL, k=NUL, v=NUL, o=NUL) == binding.RET_OK
    assert par(L, H=0, q=NUL, k=NUL, v=NUL, o=NUL, g=G(0.5)) == binding.RET_OK
    assert chk(L, b=0, q=NUL, k=NUL, v=NUL, o=NUL) == binding.RET_OK
    assert chk(L, N=0, q=NUL, k=NUL, v=NUL, o=NUL) == binding.RET_OK   # no state_out: nothing to do
    assert dec(L, b=0, q=NUL, k=NUL, v=NUL, st=NUL, o=NUL) == binding.RET_OK
    assert epi(L, N=0, y=NUL, g=NUL, o=NUL) == binding.RET_OK


def test_chunkwise_rejections(L):
    assert chk(L, chunk=8) == binding.RET_ERR_SHAPE
    assert chk(L, chunk=24) == binding.RET_ERR_SHAPE
    assert chk(L, chunk=512, N=512) == binding.RET_ERR_SHAPE
    assert chk(L, N=100) == binding.RET_ERR_SHAPE
    assert chk(L, N=64, chunk=48) == binding.RET_ERR_SHAPE
    assert chk(L, it=5) == binding.RET_ERR_DTYPE
    assert chk(L, dv=8) == binding.RET_ERR_UNSUPPORTED
    assert chk(L, k=NUL) == binding.RET_ERR_NULL
    assert chk(L, si=MIS) == binding.RET_ERR_ALIGN
    assert chk(L, so=MIS) == binding.RET_ERR_ALIGN
    assert chk(L, g=G(0.9, 1.01)) == binding.RET_ERR_UNSUPPORTED


def bwd(L, q=A, k=A, v=A, do=A, gq=A2, gk=A2, gv=A2, it=1, ot=0, b=1, H=2, N=64, dk=64, dv=64,
        chunk=16, g=None, si=None, ds=None, di=None):
    g = G(0.9, 0.5) if g is None else g
    return L.retention_chunkwise_backward(q, k, v, do, gq, gk, gv, it, ot, b, H, N, dk, dv, chunk,
                                          g, si, ds, di, S)


def test_chunkwise_backward_rejections(L):
    before = binding.kernel_launches()
    assert bwd(L, b=-1) == binding.RET_ERR_SHAPE
    assert bwd(L, chunk=8) == binding.RET_ERR_SHAPE
    assert bwd(L, N=100) == binding.RET_ERR_SHAPE
    assert bwd(L, it=2) == binding.RET_ERR_DTYPE
    assert bwd(L, ot=7) == binding.RET_ERR_DTYPE
    assert bwd(L, dk=24) == binding.RET_ERR_UNSUPPORTED
    assert bwd(L, dv=528) == binding.RET_ERR_UNSUPPORTED
    assert bwd(L, do=NUL) == binding.RET_ERR_NULL
    assert bwd(L, gv=NUL) == binding.RET_ERR_NULL
    assert bwd(L, g=ctypes.POINTER(ctypes.c_double)()) == binding.RET_ERR_NULL
    assert bwd(L, gk=MIS) == binding.RET_ERR_ALIGN
    assert bwd(L, do=MIS) == binding.RET_ERR_ALIGN
    assert bwd(L, di=MIS) == binding.RET_ERR_ALIGN
    assert bwd(L, ds=MIS) == binding.RET_ERR_ALIGN
    assert bwd(L, g=G(0.9, 1.5)) == binding.RET_ERR_UNSUPPORTED
    assert bwd(L, H=129, g=G(*([0.5] * 129))) == binding.RET_ERR_UNSUPPORTED
    # empty inputs: nothing to compute (no dstate_in requested)
    assert bwd(L, b=0, q=NUL, k=NUL, v=NUL, do=NUL, gq=NUL, gk=NUL, gv=NUL) == binding.RET_OK
    assert bwd(L, N=0, q=NUL, k=NUL, v=NUL, do=NUL, gq=NUL, gk=NUL, gv=NUL) == binding.RET_OK
    assert binding.kernel_launches() == before


def rg(L, x=A, ga=A, gx=A, lam=A, h0=None, y=A2, hl=None, it=1, ot=0, b=2, T=64, D=64, c=8.0):
    return L.rglru_scan(x, ga, gx, lam, h0, y, hl, it, ot, b, T, D, ctypes.c_float(c), S)


def test_rglru_rejections(L):
    before = binding.kernel_launches()
    assert rg(L, b=-1) == binding.RET_ERR_SHAPE
    assert rg(L, T=-1) == binding.RET_ERR_SHAPE
    assert rg(L, it=2) == binding.RET_ERR_DTYPE
    assert rg(L, D=12) == binding.RET_ERR_UNSUPPORTED
    assert rg(L, c=-1.0) == binding.RET_ERR_UNSUPPORTED
    assert rg(L, c=float("inf")) == binding.RET_ERR_UNSUPPORTED
    assert rg(L, c=float("nan")) == binding.RET_ERR_UNSUPPORTED
    assert rg(L, x=NUL) == binding.RET_ERR_NULL
    assert rg(L, lam=NUL) == binding.RET_ERR_NULL
    assert rg(L, gx=MIS) == binding.RET_ERR_ALIGN
    assert rg(L, h0=MIS) == binding.RET_ERR_ALIGN
    assert rg(L, hl=MIS) == binding.RET_ERR_ALIGN
    assert rg(L, b=0, x=NUL, ga=NUL, gx=NUL, lam=NUL, y=NUL) == binding.RET_OK
    assert rg(L, T=0, x=NUL, ga=NUL, gx=NUL, lam=NUL, y=NUL) == binding.RET_OK
    assert binding.kernel_launches() == before


def xp(L, q=A, k=A, qo=A2, ko=A2, it=1, ot=1, b=1, H=2, N=64, dk=64, th=None, pos0=0):
    th = (ctypes.c_double * 32)(*([0.1] * 32)) if th is None else th
    return L.retention_xpos_rotate(q, k, qo, ko, it, ot, b, H, N, dk, th,
                                   ctypes.c_longlong(pos0), S)


def test_xpos_rejections(L):
    before = binding.kernel_launches()
    assert xp(L, N=-1) == binding.RET_ERR_SHAPE
    assert xp(L, it=3) == binding.RET_ERR_DTYPE
    assert xp(L, dk=24) == binding.RET_ERR_UNSUPPORTED
    assert xp(L, dk=512) == binding.RET_ERR_UNSUPPORTED
    assert xp(L, q=NUL) == binding.RET_ERR_NULL
    assert xp(L, ko=NUL) == binding.RET_ERR_NULL
    assert xp(L, th=ctypes.POINTER(ctypes.c_double)()) == binding.RET_ERR_NULL
    assert xp(L, qo=MIS) == binding.RET_ERR_ALIGN
    assert xp(L, k=MIS) == binding.RET_ERR_ALIGN
    assert xp(L, qo=A, ot=0) == binding.RET_ERR_DTYPE        # in place across dtypes
    bad = (ctypes.c_double * 32)(*([0.1] * 31 + [float("inf")]))
    assert xp(L, th=bad) == binding.RET_ERR_UNSUPPORTED
    assert xp(L, b=0, q=NUL, k=NUL, qo=NUL, ko=NUL) == binding.RET_OK
    assert binding.kernel_launches() == before


def test_recurrent_step_rejections(L):
    assert dec(L, st=NUL) == binding.RET_ERR_NULL
    assert dec(L, o=MIS) == binding.RET_ERR_ALIGN
    assert dec(L, dk=0) == binding.RET_ERR_UNSUPPORTED
    assert dec(L, dk=-16) == binding.RET_ERR_SHAPE
    assert dec(L, it=3) == binding.RET_ERR_DTYPE
    assert dec(L, g=G(0.5, 2.0)) == binding.RET_ERR_UNSUPPORTED


def test_epilogue_rejections(L):
    assert epi(L, eps=-1.0) == binding.RET_ERR_UNSUPPORTED
    assert epi(L, eps=float("inf")) == binding.RET_ERR_UNSUPPORTED
    assert epi(L, eps=float("nan")) == binding.RET_ERR_UNSUPPORTED
    assert epi(L, dv=520) == binding.RET_ERR_UNSUPPORTED
    assert epi(L, dv=24) == binding.RET_ERR_UNSUPPORTED
    assert epi(L, gt=9) == binding.RET_ERR_DTYPE
    assert epi(L, y=NUL) == binding.RET_ERR_NULL
    assert epi(L, w=MIS) == binding.RET_ERR_ALIGN
    assert epi(L, H=200) == binding.RET_ERR_UNSUPPORTED
    assert epi(L, b=-2) == binding.RET_ERR_SHAPE


def gated(L, q=A, k=A, v=A, g=A, o=A2, it=1, gt=1, ot=0, b=1, H=2, N=256, dk=256, dv=512,
          gam=None, flags=7, eps=1e-5, w=None, bias=None):
    gam = G(0.9, 0.5) if gam is None else gam
    return L.retention_parallel_gated(q, k, v, g, o, it, gt, ot, b, H, N, dk, dv, gam, flags,
                                      ctypes.c_float(eps), w, bias, S)


def test_parallel_gated_rejections(L):
    assert gated(L, b=-1) == binding.RET_ERR_SHAPE
    assert gated(L, gt=4) == binding.RET_ERR_DTYPE
    assert gated(L, flags=16) == binding.RET_ERR_UNSUPPORTED
    assert gated(L, eps=-1.0) == binding.RET_ERR_UNSUPPORTED
    assert gated(L, g=NUL) == binding.RET_ERR_NULL
    assert gated(L, g=MIS) == binding.RET_ERR_ALIGN
    assert gated(L, bias=MIS) == binding.RET_ERR_ALIGN
    # shapes outside the tensor-core kernel: documented as unsupported, nothing launched
    before = binding.kernel_launches()
    assert gated(L, it=0) == binding.RET_ERR_UNSUPPORTED          # fp32 inputs
    assert gated(L, dk=64) == binding.RET_ERR_UNSUPPORTED
    assert gated(L, dv=192) == binding.RET_ERR_UNSUPPORTED
    assert gated(L, N=100) == binding.RET_ERR_UNSUPPORTED
    assert gated(L, N=0, q=NUL, k=NUL, v=NUL, g=NUL, o=NUL) == binding.RET_OK
    assert binding.kernel_launches() == before


def test_binding_refuses_cpu_tensors(L):
    import torch
    q = torch.zeros(1, 1, 16, 16)
    with pytest.raises(ValueError):
        binding.retention_parallel(q, q, q, [0.5])


WS = ctypes.c_void_p(0x400000)      # 256-byte aligned device workspace, never dereferenced


def hst(L, q=A, k=A, v=A, o=A2, it=1, ot=0, b=1, H=2, N=256, dk=64, dv=64, chunk=64, g=None,
        si=None, so=None, seg=128, ws=WS, wsb=None):
    g = G(0.9, 0.5) if g is None else g
    if wsb is None:
        wsb = L.retention_chunkwise_host_workspace_bytes(it, ot, b, H, dk, dv, seg)
    return L.retention_chunkwise_host(q, k, v, o, it, ot, b, H, N, dk, dv, chunk, g, si, so, seg,
                                      ws, wsb, S, S, S)


def test_chunkwise_host_workspace_size(L):
    f = L.retention_chunkwise_host_workspace_bytes
    # fp32 state 2*64*64*4 = 32 KB, then per buffer set q, k (bf16 2*128*64*2 = 32 KB each),
    # v (32 KB) and o (fp32, 64 KB), two sets
    assert f(1, 0, 1, 2, 64, 64, 128) == 32768 + 2 * (32768 * 3 + 65536)
    assert f(1, 1, 1, 2, 64, 64, 128) == 32768 + 2 * (32768 * 4)
    assert f(1, 0, 1, 3, 16, 16, 16) % 256 == 0                       # every part 256-aligned
    assert f(7, 0, 1, 2, 64, 64, 128) == 0
    assert f(1, 0, -1, 2, 64, 64, 128) == 0


def test_chunkwise_backward_ws_rejections(L):
    """The tensor-core shape (bf16, dk 256, dv 512, N 512): a missing, misaligned or short
    workspace is refused before any launch; other shapes keep the CUDA-core checks."""
    W256 = ctypes.c_void_p(0x300000)          # 256-byte aligned, never dereferenced
    W16 = ctypes.c_void_p(0x300010)           # 16-byte but not 256-byte aligned
    need = L.retention_chunkwise_backward_workspace_bytes(0, 1, 2, 512, 256, 512)
    assert need > 0

    def ws(w=W256, nbytes=None, dk=256, dv=512, N=512, it=1, gq=A2):
        return L.retention_chunkwise_backward_ws(A, A, A, A, gq, A2, A2, it, 0, 1, 2, N, dk, dv,
                                                 256 if N % 256 == 0 else 64, G(0.97, 0.99),
                                                 None, None, None, w,
                                                 ctypes.c_size_t(need if nbytes is None else nbytes), S)

    before = binding.kernel_launches()
    assert ws(w=NUL) == binding.RET_ERR_NULL
    assert ws(w=W16) == binding.RET_ERR_ALIGN
    assert ws(nbytes=need - 1) == binding.RET_ERR_SHAPE
    assert ws(gq=MIS) == binding.RET_ERR_ALIGN
    assert ws(gq=NUL) == binding.RET_ERR_NULL
    assert ws(dk=24, w=NUL) == binding.RET_ERR_UNSUPPORTED     # CUDA-core checks, no workspace
    assert ws(it=5) == binding.RET_ERR_DTYPE
    assert binding.kernel_launches() == before


def test_chunkwise_backward_workspace_size(L):
    f = L.retention_chunkwise_backward_workspace_bytes
    f.restype = ctypes.c_size_t
    b, H, N, dk, dv = 2, 3, 512, 256, 512
    st = b * H * dk * dv * 4                 # one fp32 state set: 6 MiB, 256-aligned
    scales = 3 * 128 * 4                     # per-head scales, 1536 bytes (256-aligned)
    # fp32 gradients: S0^T halves, dS^T halves, dS / g, the dv pass's final state, scales
    assert f(0, b, H, N, dk, dv) == 4 * st + scales
    # bf16 gradients add the fp32 partial sums of dq and dk over the halves
    assert f(1, b, H, N, dk, dv) == 4 * st + scales + 2 * (b * H * N * dk * 4)
    # one half (dv 256): no partial sums
    assert f(1, b, H, N, dk, 256) == f(0, b, H, N, dk, 256)
    assert f(0, b, H, N, 128, dv) == 0      # not a tensor-core shape
    assert f(0, b, H, N, dk, 384) == 0
    assert f(0, -1, H, N, dk, dv) == 0


def test_chunkwise_host_rejections(L):
    before = binding.kernel_launches()
    assert hst(L, seg=96) == binding.RET_ERR_SHAPE                    # not a multiple of chunk
    assert hst(L, seg=192) == binding.RET_ERR_SHAPE                   # does not divide N
    assert hst(L, seg=0) == binding.RET_ERR_SHAPE
    assert hst(L, wsb=1024) == binding.RET_ERR_SHAPE                  # workspace too small
    assert hst(L, ws=ctypes.c_void_p(0x400010)) == binding.RET_ERR_ALIGN
    assert hst(L, q=MIS) == binding.RET_ERR_ALIGN
    assert hst(L, si=MIS) == binding.RET_ERR_ALIGN
    assert hst(L, ws=NUL) == binding.RET_ERR_NULL
    assert hst(L, o=NUL) == binding.RET_ERR_NULL
    assert hst(L, it=4) == binding.RET_ERR_DTYPE
    assert hst(L, dk=24) == binding.RET_ERR_UNSUPPORTED
    assert hst(L, g=G(0.9, 1.2)) == binding.RET_ERR_UNSUPPORTED
    assert hst(L, N=200) == binding.RET_ERR_SHAPE                     # N % chunk
    assert hst(L, b=0, q=NUL, k=NUL, v=NUL, o=NUL) == binding.RET_OK
    assert binding.kernel_launches() == before
