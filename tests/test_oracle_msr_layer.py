"""Pins of the oracle's gated multi-scale retention layer (projections around the core).

[RN2] "Transformer取代者登場！微軟、清華剛推出RetNet：成本低、速度快、性能強（2）",
"門控多尺度 Retention" (per-head W_Q, W_K, W_V, a decay per head, swish gate, GroupNorm
per head, W_G and W_O; the formula itself was lost) and "Retention Score 歸一化"
(GroupNorm's scale invariance is why the three score normalisations do not change the
result).  Pins:
  * the three score normalisations leave the layer output unchanged when eps = 0 (the
    page's own claim), and so does any positive scale of W_V;
  * identity projections (D = H*dk = H*dv) reduce the layer to the core calls on the
    head-split input: catches a transposed head split or a wrong head block;
  * permuting the heads (head blocks of W_Q, W_K, W_V, W_G, the rows of W_O and gamma
    together) leaves the output unchanged;
  * shifting every xPos position leaves the output unchanged (relative positions only);
  * the chunkwise form gives the parallel form's result;
  * zeroing any one of W_Q, W_K, W_V, W_G silences the layer exactly.
"""
import numpy as np

import oracle


def rand(shape, seed, scale=1.0):
    return scale * np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def layer_inputs(b=2, N=40, D=24, H=3, dk=4, dv=6, Dout=10, seed=0):
    x = rand((b, N, D), seed)
    s = 1.0 / np.sqrt(D)
    w = dict(wq=rand((D, H * dk), seed + 1, s), wk=rand((D, H * dk), seed + 2, s),
             wv=rand((D, H * dv), seed + 3, s), wg=rand((D, H * dv), seed + 4, s),
             wo=rand((H * dv, Dout), seed + 5, s))
    gamma = [0.9, 0.97, 0.6][:H]
    theta = list(10000.0 ** (-np.arange(dk // 2) / (dk // 2)))
    return x, w, gamma, theta


def rel(a, b):
    return float(np.max(np.abs(a - b)) / np.sqrt(np.mean(b * b)))


def test_normalisations_and_value_scale_do_not_change_the_output():
    x, w, g, th = layer_inputs()
    base = oracle.msr_layer(x, **w, gamma=g, theta=th, flags=0, eps=0.0)
    assert rel(oracle.msr_layer(x, **w, gamma=g, theta=th, flags=7, eps=0.0), base) < 1e-10
    w2 = dict(w, wv=3.7 * w["wv"])
    assert rel(oracle.msr_layer(x, **w2, gamma=g, theta=th, eps=0.0), base) < 1e-10


def test_identity_projections_reduce_to_the_core():
    b, N, H, d = 1, 32, 3, 4
    D = H * d
    x = rand((b, N, D), 10)
    eye = np.eye(D)
    wg = rand((D, D), 11)
    wo = rand((D, 5), 12)
    g = [0.9, 0.8, 0.7]
    got = oracle.msr_layer(x, eye, eye, eye, wg, wo, g, theta=None, flags=7, eps=1e-5)
    xh = np.ascontiguousarray(x.reshape(b, N, H, d).transpose(0, 2, 1, 3))
    want = oracle.msr_epilogue(oracle.parallel(xh, xh, xh, g, 7), x @ wg, 1e-5) @ wo
    assert rel(got, want) < 1e-13


def test_head_permutation_equivariance():
    H, dk, dv = 3, 4, 6
    x, w, g, th = layer_inputs(H=H, dk=dk, dv=dv)
    perm = [2, 0, 1]

    def cols(m, d):
        return np.concatenate([m[:, p * d:(p + 1) * d] for p in perm], axis=1)

    wp = dict(wq=cols(w["wq"], dk), wk=cols(w["wk"], dk), wv=cols(w["wv"], dv),
              wg=cols(w["wg"], dv),
              wo=np.concatenate([w["wo"][p * dv:(p + 1) * dv] for p in perm], axis=0))
    gp = [g[p] for p in perm]
    a = oracle.msr_layer(x, **w, gamma=g, theta=th, flags=7)
    bb = oracle.msr_layer(x, **wp, gamma=gp, theta=th, flags=7)
    assert rel(bb, a) < 1e-12


def test_position_shift_and_chunkwise_form():
    x, w, g, th = layer_inputs(N=48)
    a = oracle.msr_layer(x, **w, gamma=g, theta=th, pos0=0)
    assert rel(oracle.msr_layer(x, **w, gamma=g, theta=th, pos0=5000), a) < 1e-9
    assert rel(oracle.msr_layer(x, **w, gamma=g, theta=th, chunk=16), a) < 1e-10


def test_each_zero_projection_silences_the_layer():
    """W_Q = 0 or W_K = 0 makes every score 0, W_V = 0 every value 0 (GroupNorm of a zero
    row is 0 with eps > 0), W_G = 0 closes the gate (swish(0) = 0): the output is 0 in
    each case, and nonzero for the unmodified weights."""
    x, w, g, th = layer_inputs()
    assert np.max(np.abs(oracle.msr_layer(x, **w, gamma=g, theta=th))) > 0.1
    for name in ("wq", "wk", "wv", "wg"):
        wz = dict(w, **{name: np.zeros_like(w[name])})
        assert np.max(np.abs(oracle.msr_layer(x, **wz, gamma=g, theta=th))) == 0.0, name
