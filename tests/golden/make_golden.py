"""Writes tests/golden/tiny_oracle.txt: sampled oracle outputs on the tiny workload.

Calls only the oracle and the seeded input generator.  The stored values guard
the oracle and the generator's stream against silent change; they are not
independent pins (those live in tests/test_oracle_pins.py).
Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from linear_recurrence_sequence_chunkwise_b300 import inputs  # noqa: E402


def cases():
    w = inputs.TINY
    q, k, v = inputs.qkv(w)
    g = inputs.randn((w.b, w.N, w.H * w.dv), w.seed + 4, 1.0, "f32")
    yield "parallel_f0", oracle.parallel(q, k, v, w.gamma, 0)
    yield "parallel_f7", oracle.parallel(q, k, v, w.gamma, 7)
    yield "chunkwise_B16", oracle.chunkwise(q, k, v, w.gamma, 16)
    yield "epilogue_f7", oracle.msr_epilogue(oracle.parallel(q, k, v, w.gamma, 7), g, 1e-5)
    # gradient of the chunkwise form with both states, upstream gradient N(0,1)
    do = inputs.randn((w.b, w.H, w.N, w.dv), w.seed + 10, 1.0, "f32")
    s0 = inputs.randn((w.b, w.H, w.dk, w.dv), w.seed + 11, 0.1, "f32")
    ds = inputs.randn((w.b, w.H, w.dk, w.dv), w.seed + 12, 0.1, "f32")
    gq, gk, gv, gs = oracle.chunkwise_backward(q, k, v, do, w.gamma, state_in=s0, dstate_out=ds)
    yield "backward_dq", gq
    yield "backward_dk", gk
    yield "backward_dv", gv
    yield "backward_ds0", gs
    # xPos rotation of q at positions 100.., theta_j = 10000^(-2j/dk)
    yield "xpos_q", oracle.xpos_rotate(q, [10000.0 ** (-j / 8) for j in range(8)], 100)
    # RG-LRU scan on [1, 64, 16] (x, gate pre-activations N(0,1), Lambda of the page's init)
    x, ga, gx = (inputs.randn((1, 64, 16), w.seed + 20 + i, 1.0, "f32") for i in range(3))
    yield "rglru", oracle.rglru(x, ga, gx, inputs.rglru_lambda(16, w.seed + 23),
                                inputs.randn((1, 16), w.seed + 24, 1.0, "f32"))


def sample_idx(n, count=48, seed=7):
    return np.random.Generator(np.random.PCG64(seed)).choice(n, size=count, replace=False)


def main():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.txt")
    with open(path, "w") as f:
        f.write("# name flat_index value  (tiny workload b1 H2 dk16 dv16 N64, fp32 N(0,1) inputs)\n")
        for name, arr in cases():
            flat = arr.reshape(-1)
            for i in sorted(sample_idx(flat.size)):
                f.write(f"{name} {i} {float(flat[i])!r}\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
