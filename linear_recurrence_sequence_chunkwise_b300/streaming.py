"""Chunkwise retention over a sequence held in host memory, streamed in segments.

The chunkwise form carries an exact state across any split of the sequence at a chunk
boundary ("Transformer取代者登場！微軟、清華剛推出RetNet：成本低、速度快、性能強（2）",
"Retention" 3), eq.(7): the state R after one segment is the incoming state of the
next).  This helper uses that to
overlap the three parts of an end-to-end call on three CUDA streams: host-to-device
copies of segment s+1, the library's `retention_chunkwise` on segment s (state carried
in an fp32 device buffer through `state_in`/`state_out`), and the device-to-host copy of
segment s-1's output.  It only issues copies and library calls; all arithmetic runs in
the library's kernels.

Host tensors must be pinned and laid out as the library expects ([b][H][N][d]); the
copies move one (batch, head) slice of a segment at a time, which is contiguous in
that layout.
"""
from __future__ import annotations

import torch

from . import binding

_streams: dict = {}


def _side_streams(dev: torch.device):
    """Three streams per device (H2D, compute, D2H), made once and reused."""
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    if key not in _streams:
        _streams[key] = tuple(torch.cuda.Stream(dev) for _ in range(3))
    return _streams[key]


def chunkwise_from_host(hq, hk, hv, gamma, chunk: int, ho, seg_len: int, state=None,
                        device="cuda"):
    """Compute retention_chunkwise(hq, hk, hv) into the pinned host tensor ``ho``.

    hq, hk: [b,H,N,dk], hv: [b,H,N,dv] pinned host tensors (one dtype); ho: [b,H,N,dv]
    pinned host tensor (fp32 or bf16).  ``seg_len`` must be a multiple of ``chunk`` and
    divide N.  ``state`` (optional, fp32 [b,H,dk,dv] on the device) is the incoming
    state and receives the final one.  Returns after all work is enqueued; the caller
    synchronises (``torch.cuda.synchronize()``) before reading ``ho``.
    """
    b, H, N, dk = hq.shape
    dv = hv.shape[-1]
    if seg_len % chunk or N % seg_len:
        raise ValueError("seg_len must be a multiple of chunk and divide N")
    nseg = N // seg_len
    dev = torch.device(device)
    cur = torch.cuda.current_stream(dev)
    h2d, comp, d2h = _side_streams(dev)
    for s in (h2d, comp, d2h):
        s.wait_stream(cur)
    nbuf = min(2, nseg)
    qd = [torch.empty((b, H, seg_len, dk), dtype=hq.dtype, device=dev) for _ in range(nbuf)]
    kd = [torch.empty((b, H, seg_len, dk), dtype=hk.dtype, device=dev) for _ in range(nbuf)]
    vd = [torch.empty((b, H, seg_len, dv), dtype=hv.dtype, device=dev) for _ in range(nbuf)]
    od = [torch.empty((b, H, seg_len, dv), dtype=ho.dtype, device=dev) for _ in range(nbuf)]
    st = state if state is not None else torch.empty((b, H, dk, dv), dtype=torch.float32,
                                                     device=dev)
    comp_done = [None] * nbuf
    d2h_done = [None] * nbuf
    for sgi in range(nseg):
        j = sgi % nbuf
        s0, s1 = sgi * seg_len, (sgi + 1) * seg_len
        with torch.cuda.stream(h2d):
            if comp_done[j] is not None:
                h2d.wait_event(comp_done[j])          # inputs j read by segment sgi-2
            for bi in range(b):
                for h in range(H):
                    qd[j][bi, h].copy_(hq[bi, h, s0:s1], non_blocking=True)
                    kd[j][bi, h].copy_(hk[bi, h, s0:s1], non_blocking=True)
                    vd[j][bi, h].copy_(hv[bi, h, s0:s1], non_blocking=True)
            h2d_done = torch.cuda.Event()
            h2d_done.record(h2d)
        with torch.cuda.stream(comp):
            comp.wait_event(h2d_done)
            if d2h_done[j] is not None:
                comp.wait_event(d2h_done[j])          # output j copied out by segment sgi-2
            first = sgi == 0 and state is None
            binding.retention_chunkwise(qd[j], kd[j], vd[j], gamma, chunk,
                                        state_in=None if first else st, state_out=st,
                                        out=od[j], stream=comp)
            comp_done[j] = torch.cuda.Event()
            comp_done[j].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(comp_done[j])
            for bi in range(b):
                for h in range(H):
                    ho[bi, h, s0:s1].copy_(od[j][bi, h], non_blocking=True)
            d2h_done[j] = torch.cuda.Event()
            d2h_done[j].record(d2h)
    # The segment buffers were allocated on the caller's stream; once that stream
    # waits for the three side streams, their memory can return to its pool.
    for s in (h2d, comp, d2h):
        cur.wait_stream(s)
    return ho
