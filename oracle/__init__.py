"""fp64 CPU oracle of the RetNet retention core -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or calls it, and it imports nothing from
the product.  Both sides share only the seeded input generators.

The arithmetic lives in ``retention_oracle.c`` (plain C, fp64); this module
compiles it with gcc on first use and wraps it with ctypes.  ctypes releases
the GIL during each call, so :func:`map_units` can spread independent
(batch, head) units over host threads.

Parity pins: every function here is pinned by tests in
``tests/test_oracle_pins.py`` (closed forms, special cases that reduce to
library routines, the three-form equivalence the RetNet pages state, and
GroupNorm's scale invariance).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "retention_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

NORM_SCALE = 1
NORM_DECAY = 2
NORM_ROWSUM = 4

_default = None
_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile an oracle C source into a shared library (gcc -O2, strict IEEE)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def _f64(a) -> np.ndarray:
    """Exact conversion to a C-contiguous float64 array (bf16/fp32 widen exactly)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        import torch
        a = a.detach().to("cpu").to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name}: oracle rejected its arguments")


class Oracle:
    """ctypes wrapper around one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(ctypes.c_double)
        I = ctypes.c_int
        lib.oracle_parallel.argtypes = [P, P, P, P, I, I, I, I, I, P, ctypes.c_uint]
        lib.oracle_recurrent.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P]
        lib.oracle_recurrent_step.argtypes = [P, P, P, P, P, I, I, I, I, P]
        lib.oracle_chunkwise.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P, P]
        lib.oracle_brute.argtypes = [P, P, P, P, I, I, I, I, I, P]
        lib.oracle_msr_epilogue.argtypes = [P, P, P, I, I, I, I, ctypes.c_double, P, P]
        lib.oracle_chunkwise_backward.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, P]
        lib.oracle_rglru.argtypes = [P, P, P, P, P, P, P, I, I, I, ctypes.c_double]
        lib.oracle_xpos_rotate.argtypes = [P, P, I, I, I, I, P, ctypes.c_longlong]
        for f in ("oracle_parallel", "oracle_recurrent", "oracle_recurrent_step",
                  "oracle_chunkwise", "oracle_brute", "oracle_msr_epilogue",
                  "oracle_chunkwise_backward", "oracle_rglru", "oracle_xpos_rotate"):
            getattr(lib, f).restype = ctypes.c_int
        self.lib = lib

    def parallel(self, q, k, v, gamma, flags: int = 0) -> np.ndarray:
        """eq.(5) with optional normalisations; q,k:[b,H,N,dk] v:[b,H,N,dv]."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gamma)
        b, H, N, dk = q.shape
        dv = v.shape[-1]
        o = np.zeros((b, H, N, dv))
        _check(self.lib.oracle_parallel(_p(q), _p(k), _p(v), _p(o), b, H, N, dk, dv, _p(g),
                                        flags), "parallel")
        return o

    def recurrent(self, q, k, v, gamma, state_in=None, return_state: bool = False):
        """eq.(6) over the whole sequence; optional incoming state [b,H,dk,dv]."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gamma)
        b, H, N, dk = q.shape
        dv = v.shape[-1]
        o = np.zeros((b, H, N, dv))
        si = _f64(state_in)
        so = np.zeros((b, H, dk, dv)) if return_state else None
        _check(self.lib.oracle_recurrent(_p(q), _p(k), _p(v), _p(o), b, H, N, dk, dv, _p(g),
                                         _p(si), _p(so)), "recurrent")
        return (o, so) if return_state else o

    def recurrent_step(self, q, k, v, state, gamma):
        """One decode step; q,k:[b,H,dk] v:[b,H,dv]; returns (o [b,H,dv], new state)."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gamma)
        s = _f64(state).copy()
        b, H, dk = q.shape
        dv = v.shape[-1]
        o = np.zeros((b, H, dv))
        _check(self.lib.oracle_recurrent_step(_p(q), _p(k), _p(v), _p(s), _p(o), b, H, dk, dv,
                                              _p(g)), "recurrent_step")
        return o, s

    def chunkwise(self, q, k, v, gamma, chunk: int, state_in=None, return_state: bool = False):
        """eq.(7) with chunk length ``chunk``; optional incoming state."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gamma)
        b, H, N, dk = q.shape
        dv = v.shape[-1]
        o = np.zeros((b, H, N, dv))
        si = _f64(state_in)
        so = np.zeros((b, H, dk, dv)) if return_state else None
        _check(self.lib.oracle_chunkwise(_p(q), _p(k), _p(v), _p(o), b, H, N, dk, dv, chunk,
                                         _p(g), _p(si), _p(so)), "chunkwise")
        return (o, so) if return_state else o

    def brute(self, q, k, v, gamma) -> np.ndarray:
        """Per-entry sum definition of the unnormalised parallel form."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gamma)
        b, H, N, dk = q.shape
        dv = v.shape[-1]
        o = np.zeros((b, H, N, dv))
        _check(self.lib.oracle_brute(_p(q), _p(k), _p(v), _p(o), b, H, N, dk, dv, _p(g)),
               "brute")
        return o

    def chunkwise_backward(self, q, k, v, dout, gamma, state_in=None, dstate_out=None):
        """Gradient of L = sum(dout * o) + <dstate_out, final state> for the chunkwise
        form (any chunk length gives the same function).  Returns (dq, dk, dv, dstate_in)."""
        q, k, v, do, g = _f64(q), _f64(k), _f64(v), _f64(dout), _f64(gamma)
        b, H, N, dk = q.shape
        dv = v.shape[-1]
        si, ds = _f64(state_in), _f64(dstate_out)
        gq, gk, gv = np.zeros((b, H, N, dk)), np.zeros((b, H, N, dk)), np.zeros((b, H, N, dv))
        gs = np.zeros((b, H, dk, dv))
        _check(self.lib.oracle_chunkwise_backward(_p(q), _p(k), _p(v), _p(do), _p(si), _p(ds),
                                                  _p(gq), _p(gk), _p(gv), _p(gs), b, H, N, dk,
                                                  dv, _p(g)), "chunkwise_backward")
        return gq, gk, gv, gs

    def rglru(self, x, gate_a, gate_x, lambda_, h0=None, c: float = 8.0,
              return_state: bool = False):
        """RG-LRU scan (Griffin page); x, gate_a, gate_x: [b,T,D], lambda_: [D], h0: [b,D]."""
        x, ga, gx, lam = _f64(x), _f64(gate_a), _f64(gate_x), _f64(lambda_)
        b, T, D = x.shape
        h0 = _f64(h0)
        y = np.zeros((b, T, D))
        hl = np.zeros((b, D))
        _check(self.lib.oracle_rglru(_p(x), _p(ga), _p(gx), _p(lam), _p(h0), _p(y), _p(hl),
                                     b, T, D, float(c)), "rglru")
        return (y, hl) if return_state else y

    def xpos_rotate(self, x, theta, pos0: int = 0) -> np.ndarray:
        """xPos rotation of [b,H,N,d] rows at positions pos0 + n; theta: [d/2]."""
        x, th = _f64(x), _f64(theta)
        b, H, N, d = x.shape
        out = np.zeros_like(x)
        _check(self.lib.oracle_xpos_rotate(_p(x), _p(out), b, H, N, d, _p(th), int(pos0)),
               "xpos_rotate")
        return out

    def msr_epilogue(self, y, g, eps: float, weight=None, bias=None) -> np.ndarray:
        """GroupNorm per (token, head) then swish(G) gate; y:[b,H,N,dv] g:[b,N,H*dv]."""
        y, g = _f64(y), _f64(g)
        w, bb = _f64(weight), _f64(bias)
        b, H, N, dv = y.shape
        out = np.zeros((b, N, H * dv))
        _check(self.lib.oracle_msr_epilogue(_p(y), _p(g), _p(out), b, H, N, dv, float(eps),
                                            _p(w), _p(bb)), "msr_epilogue")
        return out


def msr_layer(x, wq, wk, wv, wg, wo, gamma, theta=None, flags: int = 0, eps: float = 1e-5,
              pos0: int = 0, chunk: int | None = None):
    """Gated multi-scale retention layer, [RN2] "門控多尺度 Retention" (its formula was
    lost; the prose and the calls it names survive), composed from numpy matmuls and
    the oracle functions above:
        Q = xPos(X W_Q), K = xPos(X W_K), V = X W_V     per head (head h: columns
                                                       h*dk.. of W_Q, W_K; h*dv.. of W_V)
        Y = retention(Q, K, V, gamma_h)                parallel form with `flags`, or the
                                                       chunkwise form when `chunk` is set
        out = (swish(X W_G) (.) GroupNorm_h(Y)) W_O
    x: [b, N, D]; wq, wk: [D, H*dk]; wv, wg: [D, H*dv]; wo: [H*dv, D']; gamma: [H];
    theta: [dk/2] xPos angles (None: no rotation).  Returns [b, N, D']."""
    x = _f64(x)
    wq, wk, wv, wg, wo = (_f64(w) for w in (wq, wk, wv, wg, wo))
    b, N, _ = x.shape
    H = len(gamma)
    dk, dv = wq.shape[1] // H, wv.shape[1] // H

    def heads(t, d):
        return np.ascontiguousarray(t.reshape(b, N, H, d).transpose(0, 2, 1, 3))

    q, k, v = heads(x @ wq, dk), heads(x @ wk, dk), heads(x @ wv, dv)
    if theta is not None:
        q, k = xpos_rotate(q, theta, pos0), xpos_rotate(k, theta, pos0)
    y = chunkwise(q, k, v, gamma, chunk) if chunk else parallel(q, k, v, gamma, flags)
    return msr_epilogue(y, x @ wg, eps) @ wo


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def parallel(*a, **kw):
    return default().parallel(*a, **kw)


def recurrent(*a, **kw):
    return default().recurrent(*a, **kw)


def recurrent_step(*a, **kw):
    return default().recurrent_step(*a, **kw)


def chunkwise(*a, **kw):
    return default().chunkwise(*a, **kw)


def brute(*a, **kw):
    return default().brute(*a, **kw)


def msr_epilogue(*a, **kw):
    return default().msr_epilogue(*a, **kw)


def chunkwise_backward(*a, **kw):
    return default().chunkwise_backward(*a, **kw)


def rglru(*a, **kw):
    return default().rglru(*a, **kw)


def xpos_rotate(*a, **kw):
    return default().xpos_rotate(*a, **kw)


def map_units(fn, units, threads: int | None = None):
    """Run ``fn(unit)`` for each unit on a thread pool (the C calls drop the GIL)."""
    threads = threads or os.cpu_count() or 1
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, units))
