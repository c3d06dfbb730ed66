"""Thin ctypes binding of include/retention.h (argument marshalling only).

Every step of the computation runs in the CUDA kernels of libretention_b300.so;
this module only turns torch tensors into device pointers, sizes, dtype codes
and a stream handle, and turns non-zero status codes into exceptions.  It
fails loudly if the library is missing: there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libretention_b300.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "retention.h")

RET_OK, RET_ERR_NULL, RET_ERR_SHAPE, RET_ERR_DTYPE, RET_ERR_ALIGN = 0, 1, 2, 3, 4
RET_ERR_UNSUPPORTED, RET_ERR_CUDA, RET_ERR_TIMEOUT = 5, 6, 7
RET_F32, RET_BF16 = 0, 1
NORM_SCALE, NORM_DECAY, NORM_ROWSUM = 1, 2, 4
NORM_ALL = 7
KERNEL_NAMES = {0: "none", 1: "parallel_simt", 2: "chunkwise_simt", 3: "decode", 4: "epilogue",
                5: "chunkwise_tc", 6: "parallel_tc", 7: "parallel_gated_tc", 8: "chunkwise_tc_pair",
                9: "chunkwise_backward_simt", 10: "rglru", 11: "xpos", 12: "gemm_tc",
                13: "chunkwise_backward_tc", 14: "parallel_tc_pair", 15: "parallel_gated_tc_pair"}

_lib = None
_lock = threading.Lock()


class RetentionError(RuntimeError):
    def __init__(self, func: str, status: int, text: str):
        super().__init__(f"{func}: status {status} ({text})")
        self.status = status


def header_functions() -> list[str]:
    """Names of the functions include/retention.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decl = r"^(?:const\s+)?(?:unsigned\s+)?(?:long\s+)*\w+\s*\**\s+\**(\w+)\s*\("
    return re.findall(decl, text, flags=re.M)


def lib() -> ctypes.CDLL:
    """Load libretention_b300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python linear_recurrence_sequence_chunkwise_b300/build.py`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, u, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_float
            dp = ctypes.POINTER(ctypes.c_double)
            L.retention_parallel.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, dp, u, vp]
            L.retention_chunkwise.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, dp, vp, vp, vp]
            L.retention_chunkwise_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                                       i, i, i, dp, vp, vp, vp, vp]
            L.retention_chunkwise_backward_ws.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i,
                                                          i, i, i, i, dp, vp, vp, vp, vp,
                                                          ctypes.c_size_t, vp]
            L.retention_chunkwise_backward_ws.restype = ctypes.c_int
            L.retention_chunkwise_backward_workspace_bytes.argtypes = [i, i, i, i, i, i]
            L.retention_chunkwise_backward_workspace_bytes.restype = ctypes.c_size_t
            L.retention_xpos_rotate.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, dp,
                                                ctypes.c_longlong, vp]
            L.rglru_scan.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
            L.retention_recurrent_step.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, dp, vp]
            L.msr_epilogue.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, f, vp, vp, vp]
            L.retention_parallel_gated.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, dp,
                                                   u, f, vp, vp, vp]
            L.retention_chunkwise_host.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, dp,
                                                   vp, vp, i, vp, ctypes.c_size_t, vp, vp, vp]
            L.retention_chunkwise_host_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
            L.retention_chunkwise_host_workspace_bytes.restype = ctypes.c_size_t
            L.retention_chunkwise_host_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i,
                                                           dp, vp, vp, i, vp, vp, vp]
            L.retention_chunkwise_host_static_scratch_bytes.argtypes = []
            L.retention_chunkwise_host_static_scratch_bytes.restype = ctypes.c_size_t
            L.retention_status_string.argtypes = [i]
            L.retention_status_string.restype = ctypes.c_char_p
            L.retention_check_device_error.argtypes = [vp]
            L.retention_msr_layer.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i,
                                              dp, dp, ctypes.c_longlong, u, f, i, vp,
                                              ctypes.c_size_t, vp]
            L.retention_msr_layer.restype = ctypes.c_int
            L.retention_msr_layer_workspace_bytes.argtypes = [i, i, i, i, i, i]
            L.retention_msr_layer_workspace_bytes.restype = ctypes.c_size_t
            L.retention_gemm.argtypes = [vp, vp, vp, i, i, i, i, vp]
            L.retention_gemm.restype = ctypes.c_int
            L.retention_project_heads.argtypes = [vp, vp, vp, i, i, i, i, i, dp, ctypes.c_longlong,
                                                  vp]
            L.retention_project_heads.restype = ctypes.c_int
            L.retention_chunkwise_wait_selftest.argtypes = [vp, vp, vp, vp, vp]
            L.retention_chunkwise_wait_selftest.restype = ctypes.c_int
            L.retention_chunkwise_format_reruns.argtypes = [vp]
            L.retention_chunkwise_format_reruns.restype = ctypes.c_int
            L.retention_parallel_format_reruns.argtypes = [vp]
            L.retention_parallel_format_reruns.restype = ctypes.c_int
            L.retention_kernel_launches.argtypes = []
            L.retention_kernel_launches.restype = ctypes.c_ulonglong
            L.retention_last_kernel.argtypes = []
            L.retention_last_kernel.restype = ctypes.c_int
            L.retention_last_cuda_error.argtypes = []
            L.retention_last_cuda_error.restype = ctypes.c_int
            L.retention_cuda_error_string.argtypes = [ctypes.c_int]
            L.retention_cuda_error_string.restype = ctypes.c_char_p
            for name in ("retention_parallel", "retention_chunkwise", "retention_recurrent_step",
                         "msr_epilogue", "retention_check_device_error",
                         "retention_parallel_gated", "retention_chunkwise_host",
                         "retention_chunkwise_host_noalloc"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().retention_status_string(status).decode()


def _check(func: str, rc: int):
    if rc != RET_OK:
        text = status_string(rc)
        if rc == RET_ERR_CUDA:
            ce = int(lib().retention_last_cuda_error())
            text += "; " + lib().retention_cuda_error_string(ce).decode()
        raise RetentionError(func, rc, text)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return RET_F32
    if t == torch.bfloat16:
        return RET_BF16
    raise TypeError(f"unsupported dtype {t}; use torch.float32 or torch.bfloat16")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _gamma(gamma, H: int):
    g = [float(x) for x in gamma]
    if len(g) != H:
        raise ValueError(f"gamma has {len(g)} entries, expected H={H}")
    return (ctypes.c_double * max(H, 1))(*g)


def retention_parallel(q, k, v, gamma, flags: int = 0, out=None, out_dtype=torch.float32,
                       stream=None):
    """Parallel form (eq.5) with optional normalisation flags.  q,k:[b,H,N,dk] v:[b,H,N,dv]."""
    b, H, N, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((b, H, N, dv), dtype=out_dtype, device=q.device)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    rc = lib().retention_parallel(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _dtype_code(q.dtype),
                                  _dtype_code(out.dtype), b, H, N, dk, dv, _gamma(gamma, H),
                                  flags, _stream(stream))
    _check("retention_parallel", rc)
    return out


def retention_chunkwise(q, k, v, gamma, chunk: int, state_in=None, state_out=None, out=None,
                        out_dtype=torch.float32, stream=None):
    """Chunkwise recurrent form (eq.7).  state_in/state_out: fp32 [b,H,dk,dv] or None."""
    b, H, N, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((b, H, N, dv), dtype=out_dtype, device=q.device)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    for s in (state_in, state_out):
        if s is not None and s.dtype != torch.float32:
            raise TypeError("states are fp32")
    rc = lib().retention_chunkwise(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _dtype_code(q.dtype),
                                   _dtype_code(out.dtype), b, H, N, dk, dv, chunk,
                                   _gamma(gamma, H), _ptr(state_in), _ptr(state_out),
                                   _stream(stream))
    _check("retention_chunkwise", rc)
    return out


def backward_workspace_bytes(out_dtype, b: int, H: int, N: int, dk: int, dv: int) -> int:
    """Workspace bytes of retention_chunkwise_backward_ws (0 where the tensor-core passes
    do not apply)."""
    return int(lib().retention_chunkwise_backward_workspace_bytes(_dtype_code(out_dtype), b, H,
                                                                  N, dk, dv))


def retention_chunkwise_backward(q, k, v, dout, gamma, chunk: int, state_in=None,
                                 dstate_out=None, dstate_in=None, grads=None,
                                 out_dtype=torch.float32, stream=None, workspace=None,
                                 cuda_cores: bool = False):
    """Gradient of retention_chunkwise for L = sum(dout * o) + <dstate_out, final state>.

    Returns (grad_q, grad_k, grad_v, dstate_in); dstate_in is None unless a tensor is
    passed (fp32 [b,H,dk,dv]).  grads: optional preallocated (grad_q, grad_k, grad_v).
    Runs retention_chunkwise_backward_ws (tensor-core passes where they apply; the
    workspace is made here unless given); cuda_cores=True calls the CUDA-core
    retention_chunkwise_backward instead."""
    b, H, N, dk = q.shape
    dv = v.shape[-1]
    if k.dtype != q.dtype or v.dtype != q.dtype or dout.dtype != q.dtype:
        raise TypeError("q, k, v and dout must share one dtype")
    for s in (state_in, dstate_out, dstate_in):
        if s is not None and s.dtype != torch.float32:
            raise TypeError("states are fp32")
    if grads is None:
        grads = (torch.empty((b, H, N, dk), dtype=out_dtype, device=q.device),
                 torch.empty((b, H, N, dk), dtype=out_dtype, device=q.device),
                 torch.empty((b, H, N, dv), dtype=out_dtype, device=q.device))
    gq, gk, gv = grads
    if gk.dtype != gq.dtype or gv.dtype != gq.dtype:
        raise TypeError("the three gradients must share one dtype")
    if cuda_cores:
        rc = lib().retention_chunkwise_backward(
            _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(gq), _ptr(gk), _ptr(gv),
            _dtype_code(q.dtype), _dtype_code(gq.dtype), b, H, N, dk, dv, chunk,
            _gamma(gamma, H), _ptr(state_in), _ptr(dstate_out), _ptr(dstate_in), _stream(stream))
        _check("retention_chunkwise_backward", rc)
        return gq, gk, gv, dstate_in
    # the tensor-core passes need a workspace for the shapes they take (bf16, dk 256,
    # dv and N multiples of 256); other shapes ignore it
    owned = workspace is None and (q.dtype == torch.bfloat16 and dk == 256 and dv % 256 == 0
                                   and N % 256 == 0)
    if owned:
        nbytes = backward_workspace_bytes(gq.dtype, b, H, N, dk, dv)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    wptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else None
    wbytes = ctypes.c_size_t(workspace.numel() if workspace is not None else 0)
    rc = lib().retention_chunkwise_backward_ws(
        _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(gq), _ptr(gk), _ptr(gv),
        _dtype_code(q.dtype), _dtype_code(gq.dtype), b, H, N, dk, dv, chunk, _gamma(gamma, H),
        _ptr(state_in), _ptr(dstate_out), _ptr(dstate_in), wptr, wbytes, _stream(stream))
    if owned:
        workspace.record_stream(stream or torch.cuda.current_stream(q.device))
    _check("retention_chunkwise_backward_ws", rc)
    return gq, gk, gv, dstate_in


def retention_xpos_rotate(q, k, theta, pos0: int = 0, q_out=None, k_out=None, out_dtype=None,
                          stream=None):
    """xPos rotation of q (and k, if given) [b,H,N,dk] at positions pos0 + n; theta: dk/2
    angles.  Returns (q_out, k_out); pass q_out=q (k_out=k) to rotate in place."""
    b, H, N, dk = q.shape
    if k is not None and (k.shape != q.shape or k.dtype != q.dtype):
        raise TypeError("q and k must share shape and dtype")
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if q_out is None:
        q_out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if k is not None and k_out is None:
        k_out = torch.empty(k.shape, dtype=q_out.dtype, device=k.device)
    th = [float(t) for t in theta]
    if len(th) != dk // 2:
        raise ValueError(f"theta has {len(th)} entries, expected dk/2={dk // 2}")
    tarr = (ctypes.c_double * max(len(th), 1))(*th)
    rc = lib().retention_xpos_rotate(_ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out),
                                     _dtype_code(q.dtype), _dtype_code(q_out.dtype), b, H, N,
                                     dk, tarr, int(pos0), _stream(stream))
    _check("retention_xpos_rotate", rc)
    return q_out, k_out


def rglru_scan(x, gate_a, gate_x, lambda_, h0=None, c: float = 8.0, out=None,
               out_dtype=torch.float32, h_last=None, stream=None):
    """RG-LRU scan (Griffin page).  x, gate_a, gate_x: [b,T,D]; lambda_: fp32 [D];
    h0, h_last: fp32 [b,D] or None.  Returns y [b,T,D]."""
    b, T, D = x.shape
    if gate_a.dtype != x.dtype or gate_x.dtype != x.dtype:
        raise TypeError("x, gate_a and gate_x must share one dtype")
    for s in (lambda_, h0, h_last):
        if s is not None and s.dtype != torch.float32:
            raise TypeError("lambda, h0 and h_last are fp32")
    if out is None:
        out = torch.empty((b, T, D), dtype=out_dtype, device=x.device)
    rc = lib().rglru_scan(_ptr(x), _ptr(gate_a), _ptr(gate_x), _ptr(lambda_), _ptr(h0),
                          _ptr(out), _ptr(h_last), _dtype_code(x.dtype), _dtype_code(out.dtype),
                          b, T, D, ctypes.c_float(c), _stream(stream))
    _check("rglru_scan", rc)
    return out


_copy_streams = {}


def _host_ptr(t):
    if t.is_cuda:
        raise ValueError("host tensors expected (pinned CPU memory)")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def chunkwise_host_workspace_bytes(in_dtype, out_dtype, b: int, H: int, dk: int, dv: int,
                                   seg_len: int) -> int:
    return int(lib().retention_chunkwise_host_workspace_bytes(
        _dtype_code(in_dtype), _dtype_code(out_dtype), b, H, dk, dv, seg_len))


def retention_chunkwise_host(q, k, v, gamma, chunk: int, out, seg_len: int, state_in=None,
                             state_out=None, workspace=None, stream=None, copy_streams=None):
    """Chunkwise form over host tensors (pinned CPU q,k:[b,H,N,dk] v,out:[b,H,N,dv]),
    streamed through the device in segments of seg_len tokens.  Device workspace and the
    two copy streams are made here unless given; all work is ordered on `stream`."""
    b, H, N, dk = q.shape
    dv = v.shape[-1]
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    dev = torch.device("cuda", torch.cuda.current_device())
    owned = workspace is None
    if owned:
        nbytes = chunkwise_host_workspace_bytes(q.dtype, out.dtype, b, H, dk, dv, seg_len)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    if copy_streams is None:
        if dev.index not in _copy_streams:
            _copy_streams[dev.index] = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
        copy_streams = _copy_streams[dev.index]
    rc = lib().retention_chunkwise_host(
        _host_ptr(q), _host_ptr(k), _host_ptr(v), _host_ptr(out), _dtype_code(q.dtype),
        _dtype_code(out.dtype), b, H, N, dk, dv, chunk, _gamma(gamma, H), _ptr(state_in),
        _ptr(state_out), seg_len, ctypes.c_void_p(workspace.data_ptr()),
        ctypes.c_size_t(workspace.numel()), _stream(stream),
        ctypes.c_void_p(copy_streams[0].cuda_stream), ctypes.c_void_p(copy_streams[1].cuda_stream))
    if owned:
        # The workspace was allocated on the current stream, but the queued copies and
        # kernels use it on `stream` and the copy streams: keep the caching allocator from
        # handing the block out again before that work is done.
        for s in (stream or torch.cuda.current_stream(dev), *copy_streams):
            workspace.record_stream(s)
    _check("retention_chunkwise_host", rc)
    return out


def chunkwise_host_static_scratch_bytes() -> int:
    return int(lib().retention_chunkwise_host_static_scratch_bytes())


def retention_chunkwise_host_noalloc(q, k, v, gamma, chunk: int, out, seg_len: int,
                                     state_in=None, state_out=None, stream=None,
                                     copy_streams=None):
    """retention_chunkwise_host on the library's static device scratch (no workspace);
    calls on one device must not overlap in time."""
    b, H, N, dk = q.shape
    dv = v.shape[-1]
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    dev = torch.device("cuda", torch.cuda.current_device())
    if copy_streams is None:
        if dev.index not in _copy_streams:
            _copy_streams[dev.index] = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
        copy_streams = _copy_streams[dev.index]
    rc = lib().retention_chunkwise_host_noalloc(
        _host_ptr(q), _host_ptr(k), _host_ptr(v), _host_ptr(out), _dtype_code(q.dtype),
        _dtype_code(out.dtype), b, H, N, dk, dv, chunk, _gamma(gamma, H), _ptr(state_in),
        _ptr(state_out), seg_len, _stream(stream), ctypes.c_void_p(copy_streams[0].cuda_stream),
        ctypes.c_void_p(copy_streams[1].cuda_stream))
    _check("retention_chunkwise_host_noalloc", rc)
    return out


def retention_recurrent_step(q, k, v, state, gamma, out=None, out_dtype=torch.float32,
                             stream=None):
    """One decode step (eq.6), state updated in place.  q,k:[b,H,dk] v:[b,H,dv]."""
    b, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((b, H, dv), dtype=out_dtype, device=q.device)
    if state.dtype != torch.float32:
        raise TypeError("the state is fp32")
    rc = lib().retention_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(state), _ptr(out),
                                        _dtype_code(q.dtype), _dtype_code(out.dtype), b, H, dk,
                                        dv, _gamma(gamma, H), _stream(stream))
    _check("retention_recurrent_step", rc)
    return out


def msr_epilogue(y, g, eps: float = 1e-5, weight=None, bias=None, out=None,
                 out_dtype=torch.float32, stream=None):
    """GroupNorm per (token, head) + swish(G) gate.  y:[b,H,N,dv] g:[b,N,H*dv]."""
    b, H, N, dv = y.shape
    if out is None:
        out = torch.empty((b, N, H * dv), dtype=out_dtype, device=y.device)
    rc = lib().msr_epilogue(_ptr(y), _ptr(g), _ptr(out), _dtype_code(y.dtype),
                            _dtype_code(g.dtype), _dtype_code(out.dtype), b, H, N, dv,
                            float(eps), _ptr(weight), _ptr(bias), _stream(stream))
    _check("msr_epilogue", rc)
    return out


def retention_parallel_gated(q, k, v, g, gamma, flags: int = 0, eps: float = 1e-5, weight=None,
                             bias=None, out=None, out_dtype=torch.float32, stream=None):
    """Parallel form + GroupNorm/swish-gate epilogue in one kernel.  q,k:[b,H,N,dk]
    v:[b,H,N,dv] (bf16), g:[b,N,H*dv]; returns out [b,N,H*dv]."""
    b, H, N, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((b, N, H * dv), dtype=out_dtype, device=q.device)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    rc = lib().retention_parallel_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(out),
                                        _dtype_code(q.dtype), _dtype_code(g.dtype),
                                        _dtype_code(out.dtype), b, H, N, dk, dv, _gamma(gamma, H),
                                        flags, float(eps), _ptr(weight), _ptr(bias),
                                        _stream(stream))
    _check("retention_parallel_gated", rc)
    return out


def kernel_launches() -> int:
    """Kernels the library has launched in this process (host-side counter)."""
    return int(lib().retention_kernel_launches())


def last_kernel() -> str:
    """Name of the kernel this host thread launched last (see RET_KERNEL_* codes)."""
    return KERNEL_NAMES.get(int(lib().retention_last_kernel()), "unknown")


def _doubles(vals):
    if vals is None:
        return None
    v = [float(x) for x in vals]
    return (ctypes.c_double * max(len(v), 1))(*v)


def retention_gemm(a, w, out=None, out_dtype=torch.float32, stream=None):
    """C = A W (tensor cores): a [M, K] bf16, w [K, Nc] bf16 -> [M, Nc]."""
    M, K = a.shape
    Nc = w.shape[1]
    if a.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise TypeError("a and w are bf16")
    if out is None:
        out = torch.empty((M, Nc), dtype=out_dtype, device=a.device)
    rc = lib().retention_gemm(_ptr(a), _ptr(w), _ptr(out), _dtype_code(out.dtype), M, Nc, K,
                              _stream(stream))
    _check("retention_gemm", rc)
    return out


def retention_project_heads(x, w, H: int, d: int, theta=None, pos0: int = 0, out=None,
                            stream=None):
    """Head-major projection with the xPos rotation fused: x [b, N, d_in] bf16, w [d_in, H*d]
    bf16 -> [b, H, N, d] bf16."""
    b, N, d_in = x.shape
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise TypeError("x and w are bf16")
    if theta is not None and len(theta) != d // 2:
        raise ValueError("theta needs d/2 angles")
    if out is None:
        out = torch.empty((b, H, N, d), dtype=torch.bfloat16, device=x.device)
    rc = lib().retention_project_heads(_ptr(x), _ptr(w), _ptr(out), b, N, d_in, H, d,
                                       _doubles(theta), int(pos0), _stream(stream))
    _check("retention_project_heads", rc)
    return out


def msr_layer_workspace_bytes(b: int, N: int, H: int, dk: int, dv: int, chunk: int = 0) -> int:
    return int(lib().retention_msr_layer_workspace_bytes(b, N, H, dk, dv, chunk))


def retention_msr_layer(x, wq, wk, wv, wg, wo, gamma, theta=None, pos0: int = 0, flags: int = 0,
                        eps: float = 1e-5, chunk: int = 0, out=None, out_dtype=torch.float32,
                        workspace=None, stream=None):
    """Gated multi-scale retention layer: x [b, N, D] bf16; wq, wk [D, H*dk]; wv, wg [D, H*dv];
    wo [H*dv, Dout] (bf16).  Returns [b, N, Dout]."""
    b, N, D = x.shape
    H = len(gamma)
    dk, dv, Dout = wq.shape[1] // H, wv.shape[1] // H, wo.shape[1]
    for t in (x, wq, wk, wv, wg, wo):
        if t.dtype != torch.bfloat16:
            raise TypeError("x and the weights are bf16")
    if out is None:
        out = torch.empty((b, N, Dout), dtype=out_dtype, device=x.device)
    owned = workspace is None
    if owned:
        nbytes = msr_layer_workspace_bytes(b, N, H, dk, dv, chunk)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    rc = lib().retention_msr_layer(_ptr(x), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wg), _ptr(wo),
                                   _ptr(out), _dtype_code(out.dtype), b, N, D, H, dk, dv, Dout,
                                   _gamma(gamma, H), _doubles(theta), int(pos0), flags,
                                   float(eps), chunk, ctypes.c_void_p(workspace.data_ptr()),
                                   ctypes.c_size_t(workspace.numel()), _stream(stream))
    if owned:
        workspace.record_stream(stream or torch.cuda.current_stream(x.device))
    _check("retention_msr_layer", rc)
    return out


def chunkwise_wait_selftest(q, k, v, o, stream=None) -> int:
    """Launch the bounded-wait self-test (q, k: bf16 [256,256], v: bf16 [256,128], o: fp32
    [256,128] on the device); returns the launch status, the expiry shows up in
    check_device_error()."""
    return int(lib().retention_chunkwise_wait_selftest(_ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                       _stream(stream)))


def chunkwise_format_reruns(stream=None) -> int:
    """Synchronise and return (and reset) how many units of the pair-of-SMs chunkwise kernel
    re-ran in the bf16 hi/lo format because an fp16 operand left fp16's range."""
    n = int(lib().retention_chunkwise_format_reruns(_stream(stream)))
    if n < 0:
        raise RetentionError("retention_chunkwise_format_reruns", RET_ERR_CUDA, "sync failed")
    return n


def parallel_format_reruns(stream=None) -> int:
    """Synchronise and return (and reset) how many clusters of the pair-of-SMs parallel kernel
    re-ran in the bf16 hi/lo format (fp16 range left, or V too small for fp16)."""
    n = int(lib().retention_parallel_format_reruns(_stream(stream)))
    if n < 0:
        raise RetentionError("retention_parallel_format_reruns", RET_ERR_CUDA, "sync failed")
    return n


def check_device_error(stream=None):
    """Synchronise and raise if a kernel gave up on a bounded wait."""
    _check("retention_check_device_error", lib().retention_check_device_error(_stream(stream)))
