"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test cites the page passage it relies on.  Sources:
  [RN2] "Transformer取代者登場！微軟、清華剛推出RetNet：成本低、速度快、性能強（2）"
  [RVW] "[論文レビュー] Retentive Network: A Successor to Transformer for Large Language Models"

Pins used (a plausible slip anywhere in the oracle fails at least one):
  * closed forms of the geometric decay sums (all-ones inputs, unit vectors);
  * special cases that reduce to library routines: gamma=1 is causal linear
    attention (numpy cumsum of outer products), gamma=0 is the diagonal term,
    N=1 is (q.k) v, GroupNorm + swish equal torch's group_norm and silu;
  * the pages' own invariant: parallel, recurrent and chunkwise forms (and the
    per-entry brute-force sum) agree ([RN2] "Retention" 1)-3), [RVW] ABSTRACT);
  * GroupNorm scale invariance, which is why the score normalisations do not
    change the gated output ([RN2] "Retention Score 歸一化");
  * state hand-off: chunkwise prefix + recurrent steps = the whole sequence.
dk != dv and distinct per-head decays everywhere, so transposed operands and
head mix-ups cannot cancel.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_sequence_chunkwise_b300 import inputs


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(float(np.sqrt(np.mean(b * b))), 1e-300)
    return float(np.max(np.abs(a - b))) / scale


def rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


G3 = [0.9, 0.5, 0.97]


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("form", ["parallel", "recurrent", "chunkwise", "brute"])
def test_all_ones_geometric_closed_form(form):
    """q=k=1, v=1: o_n = dk * sum_{m<=n} gamma^(n-m) = dk (1-gamma^(n+1))/(1-gamma).

    [RN2] "Retention" 1): scores q_n.k_m weighted by the decay gamma^(n-m), causal.
    """
    b, H, N, dk, dv = 1, 3, 24, 5, 3
    q = np.ones((b, H, N, dk)); k = np.ones((b, H, N, dk)); v = np.ones((b, H, N, dv))
    fn = {"parallel": lambda: oracle.parallel(q, k, v, G3),
          "recurrent": lambda: oracle.recurrent(q, k, v, G3),
          "chunkwise": lambda: oracle.chunkwise(q, k, v, G3, 8),
          "brute": lambda: oracle.brute(q, k, v, G3)}[form]
    o = fn()
    for h, g in enumerate(G3):
        n = np.arange(N)
        want = dk * (1 - g ** (n + 1)) / (1 - g)
        for c in range(dv):
            np.testing.assert_allclose(o[0, h, :, c], want, rtol=1e-13)


def test_gamma_one_is_causal_linear_attention():
    """gamma=1: o_n = q_n (sum_{m<=n} k_m^T v_m), a prefix sum (numpy cumsum)."""
    b, H, N, dk, dv = 2, 1, 17, 4, 6
    q, k, v = rand((b, H, N, dk), 1), rand((b, H, N, dk), 2), rand((b, H, N, dv), 3)
    outer = np.einsum("bhna,bhnc->bhnac", k, v)
    pref = np.cumsum(outer, axis=2)
    want = np.einsum("bhna,bhnac->bhnc", q, pref)
    for o in (oracle.parallel(q, k, v, [1.0]), oracle.recurrent(q, k, v, [1.0]),
              oracle.chunkwise(q, k, v, [1.0], 1), oracle.brute(q, k, v, [1.0])):
        assert rel(o, want) < 1e-12


def test_gamma_zero_is_diagonal():
    """gamma=0: only m=n survives (0^0=1): o_n = (q_n.k_n) v_n."""
    b, H, N, dk, dv = 1, 2, 13, 3, 5
    q, k, v = rand((b, H, N, dk), 4), rand((b, H, N, dk), 5), rand((b, H, N, dv), 6)
    want = np.einsum("bhna,bhna->bhn", q, k)[..., None] * v
    for o in (oracle.parallel(q, k, v, [0.0, 0.0]), oracle.recurrent(q, k, v, [0.0, 0.0]),
              oracle.chunkwise(q, k, v, [0.0, 0.0], 13), oracle.brute(q, k, v, [0.0, 0.0])):
        assert rel(o, want) < 1e-13


def test_single_token():
    """N=1: o = (q.k) v for every form, whatever gamma."""
    q, k, v = rand((2, 3, 1, 4), 7), rand((2, 3, 1, 4), 8), rand((2, 3, 1, 2), 9)
    want = np.einsum("bhna,bhna->bhn", q, k)[..., None] * v
    for o in (oracle.parallel(q, k, v, G3), oracle.recurrent(q, k, v, G3),
              oracle.chunkwise(q, k, v, G3, 1), oracle.brute(q, k, v, G3)):
        assert rel(o, want) < 1e-14


def test_two_tokens_by_hand():
    """N=2, dk=dv=1: o_0 = q0 k0 v0, o_1 = q1 (gamma k0 v0 + k1 v1)."""
    q = np.array([2.0, -3.0]).reshape(1, 1, 2, 1)
    k = np.array([0.5, 4.0]).reshape(1, 1, 2, 1)
    v = np.array([-1.0, 0.25]).reshape(1, 1, 2, 1)
    g = 0.75
    want = np.array([2.0 * 0.5 * -1.0, -3.0 * (g * 0.5 * -1.0 + 4.0 * 0.25)])
    for o in (oracle.parallel(q, k, v, [g]), oracle.recurrent(q, k, v, [g]),
              oracle.chunkwise(q, k, v, [g], 2), oracle.chunkwise(q, k, v, [g], 1),
              oracle.brute(q, k, v, [g])):
        np.testing.assert_allclose(o.reshape(-1), want, rtol=1e-15)


# --------------------------------------------------------------------------
# the pages' invariant: three equivalent forms
# --------------------------------------------------------------------------

def test_tiny_workload_three_forms_agree():
    """The tiny workload (b1 H2 d16 N64 chunk 16, fp32 N(0,1) inputs): parallel,
    recurrent, chunkwise and brute force agree to 1e-5 (they agree far tighter
    in fp64).  [RN2] "Retention" 2): "Q, K, V, gamma are the same as eq.5";
    3): chunkwise mixes the two; [RVW] ABSTRACT: three computation paradigms."""
    w = inputs.TINY
    q, k, v = inputs.qkv(w)
    P = oracle.parallel(q, k, v, w.gamma)
    Rr = oracle.recurrent(q, k, v, w.gamma)
    C = oracle.chunkwise(q, k, v, w.gamma, w.chunk)
    Bf = oracle.brute(q, k, v, w.gamma)
    for other in (Rr, C, Bf):
        assert rel(other, P) < 1e-5
        assert rel(other, P) < 1e-12


@pytest.mark.parametrize("chunk", [1, 2, 4, 8, 16, 32, 64])
def test_chunkwise_any_chunk_equals_recurrent(chunk):
    """Every chunk length gives the recurrent result (chunk=1 is eq.6 itself,
    chunk=N is eq.5 inside one chunk).  dk=7, dv=5 so a transposed state fails."""
    b, H, N, dk, dv = 2, 3, 64, 7, 5
    q, k, v = rand((b, H, N, dk), 11), rand((b, H, N, dk), 12), rand((b, H, N, dv), 13)
    want = oracle.recurrent(q, k, v, G3)
    got = oracle.chunkwise(q, k, v, G3, chunk)
    assert rel(got, want) < 1e-12


def test_chunkwise_rejects_ragged_chunk():
    q = np.zeros((1, 1, 10, 2)); v = np.zeros((1, 1, 10, 2))
    with pytest.raises(ValueError):
        oracle.chunkwise(q, q, v, [0.5], 4)


def test_heads_use_their_own_gamma():
    """Multi-scale heads ([RN2] "門控多尺度 Retention"): head h only sees gamma_h."""
    b, H, N, dk, dv = 1, 3, 20, 3, 4
    q, k, v = rand((b, H, N, dk), 21), rand((b, H, N, dk), 22), rand((b, H, N, dv), 23)
    full = oracle.chunkwise(q, k, v, G3, 5)
    for h in range(H):
        one = oracle.recurrent(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], [G3[h]])
        assert rel(full[:, h:h + 1], one) < 1e-12


# --------------------------------------------------------------------------
# score normalisations ([RN2] "Retention Score 歸一化")
# --------------------------------------------------------------------------

def unit_inputs(N, dk, dv, sign=1.0, a=1.0):
    q = np.zeros((1, 3, N, dk)); k = np.zeros((1, 3, N, dk))
    q[..., 0] = a; k[..., 0] = sign * a
    v = np.ones((1, 3, N, dv))
    return q, k, v


def s_closed(g, n):
    return (1 - g ** (n + 1)) / (1 - g)


def test_norm_scale_closed_form():
    """SCALE divides q.k by sqrt(dk): q=k=a e_0, v=1 -> o_n = a^2/sqrt(dk) s_n."""
    N, dk, dv, a = 30, 9, 2, 1.7
    q, k, v = unit_inputs(N, dk, dv, a=a)
    o = oracle.parallel(q, k, v, G3, oracle.NORM_SCALE)
    n = np.arange(N)
    for h, g in enumerate(G3):
        np.testing.assert_allclose(o[0, h, :, 0], a * a / 3.0 * s_closed(g, n), rtol=1e-13)


def test_norm_decay_closed_form():
    """DECAY divides row n of D by sqrt of its sum s_n=(1-g^(n+1))/(1-g):
    q.k=1, v=1 -> o_n = s_n / sqrt(s_n) = sqrt(s_n)."""
    N, dk, dv = 40, 4, 3
    q, k, v = unit_inputs(N, dk, dv)
    o = oracle.parallel(q, k, v, G3, oracle.NORM_DECAY)
    n = np.arange(N)
    for h, g in enumerate(G3):
        np.testing.assert_allclose(o[0, h, :, 1], np.sqrt(s_closed(g, n)), rtol=1e-13)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_norm_rowsum_uses_abs_of_signed_sum(sign):
    """ROWSUM divides row n by max(|sum_m R_nm|, 1).  With q.k = sign*a^2, v=1:
    row sum = sign*a^2*s_n -> o_n = sign*a^2 s_n / max(a^2 s_n, 1).  a^2=0.1 puts
    early rows below the clamp and later ones above it (s_n reaches 10 at g=0.97)."""
    N, dk, dv = 60, 3, 2
    a = math.sqrt(0.1)
    q, k, v = unit_inputs(N, dk, dv, sign=sign, a=a)
    o = oracle.parallel(q, k, v, G3, oracle.NORM_ROWSUM)
    n = np.arange(N)
    for h, g in enumerate(G3):
        rs = 0.1 * s_closed(g, n)
        want = sign * rs / np.maximum(rs, 1.0)
        np.testing.assert_allclose(o[0, h, :, 0], want, rtol=1e-13)
    # both branches of the clamp are exercised for gamma=0.97
    rs97 = 0.1 * s_closed(0.97, n)
    assert (rs97 < 1).any() and (rs97 > 1).any()


def test_all_norms_closed_form():
    """All three flags, q.k = +-a^2, v=1: row weights a^2 g^(n-m)/sqrt(dk)/sqrt(s_n)
    sum to c_n = a^2 sqrt(s_n)/sqrt(dk); output c_n/max(c_n,1) with the sign."""
    N, dk, dv, a = 50, 4, 2, 3.0
    for sign in (1.0, -1.0):
        q, k, v = unit_inputs(N, dk, dv, sign=sign, a=a)
        o = oracle.parallel(q, k, v, G3, 7)
        n = np.arange(N)
        for h, g in enumerate(G3):
            c = a * a * np.sqrt(s_closed(g, n)) / 2.0
            np.testing.assert_allclose(o[0, h, :, 1], sign * c / np.maximum(c, 1.0), rtol=1e-13)


# --------------------------------------------------------------------------
# epilogue: GroupNorm per head + swish gate ([RN2] "門控多尺度 Retention")
# --------------------------------------------------------------------------

def torch_epilogue(y, g, eps, weight=None, bias=None):
    """Library special case: torch.nn.functional.group_norm with H groups over the
    token-major [.., H*dv] channels, then silu(G) (silu is swish with beta=1)."""
    y = torch.from_numpy(y)
    b, H, N, dv = y.shape
    x = y.permute(0, 2, 1, 3).reshape(b * N, H * dv)
    w = None if weight is None else torch.from_numpy(weight)
    bb = None if bias is None else torch.from_numpy(bias)
    yn = torch.nn.functional.group_norm(x, H, w, bb, eps).reshape(b, N, H * dv)
    return (torch.nn.functional.silu(torch.from_numpy(g)) * yn).numpy()


@pytest.mark.parametrize("affine", [False, True])
def test_epilogue_matches_torch_group_norm_and_silu(affine):
    b, H, N, dv = 2, 3, 5, 8
    y = rand((b, H, N, dv), 31) * 3 + 1.5
    g = rand((b, N, H * dv), 32) * 2
    w = rand((H * dv,), 33) if affine else None
    bb = rand((H * dv,), 34) if affine else None
    got = oracle.msr_epilogue(y, g, 1e-5, w, bb)
    want = torch_epilogue(y, g, 1e-5, w, bb)
    assert rel(got, want) < 1e-12


@pytest.mark.parametrize("alpha", [1e-3, 7.0, 1e3])
def test_groupnorm_scale_invariance(alpha):
    """GroupNorm(alpha * head) = GroupNorm(head) (exact when eps = 0)."""
    b, H, N, dv = 1, 4, 6, 16
    y = rand((b, H, N, dv), 41)
    g = rand((b, N, H * dv), 42)
    a = oracle.msr_epilogue(y, g, 0.0)
    c = oracle.msr_epilogue(alpha * y, g, 0.0)
    assert rel(c, a) < 1e-12


def test_groupnorm_statistics():
    """With the gate factored out: each (token, head) group has mean 0 and
    variance sigma^2/(sigma^2+eps) (biased variance)."""
    b, H, N, dv, eps = 1, 2, 3, 32, 0.5
    y = rand((b, H, N, dv), 51) * 0.6
    g = np.full((b, N, H * dv), 2.0)
    out = oracle.msr_epilogue(y, g, eps)
    sw = 2.0 / (1.0 + math.exp(-2.0))
    yn = (out / sw).reshape(b, N, H, dv)
    for n in range(N):
        for h in range(H):
            grp = y[0, h, n]
            s2 = grp.var()
            assert abs(yn[0, n, h].mean()) < 1e-12
            assert abs(yn[0, n, h].var() - s2 / (s2 + eps)) < 1e-12


def test_normalisations_do_not_change_gated_output():
    """[RN2] "Retention Score 歸一化": the three factors are per-row positive
    scalings, so after GroupNorm the output is unchanged (exact at eps = 0)."""
    b, H, N, dk, dv = 1, 3, 40, 6, 10
    q, k, v = rand((b, H, N, dk), 61), rand((b, H, N, dk), 62), rand((b, H, N, dv), 63)
    g = rand((b, N, H * dv), 64)
    base = oracle.parallel(q, k, v, G3, 0)
    for flags in (1, 2, 4, 3, 5, 6, 7):
        normed = oracle.parallel(q, k, v, G3, flags)
        assert rel(oracle.msr_epilogue(normed, g, 0.0), oracle.msr_epilogue(base, g, 0.0)) < 1e-9
    # with eps > 0 the match is approximate only through eps
    normed = oracle.parallel(q, k, v, G3, 7)
    assert rel(oracle.msr_epilogue(normed, g, 1e-5), oracle.msr_epilogue(base, g, 1e-5)) < 5e-2


# --------------------------------------------------------------------------
# state hand-off and decode ([RN2] "訓練/推理": eq.6 for decoding)
# --------------------------------------------------------------------------

def test_chunkwise_prefix_then_decode_steps_equals_whole():
    b, H, N, extra, dk, dv, B = 1, 3, 32, 5, 4, 6, 8
    q, k, v = rand((b, H, N + extra, dk), 71), rand((b, H, N + extra, dk), 72), \
        rand((b, H, N + extra, dv), 73)
    whole = oracle.recurrent(q, k, v, G3)
    pre, state = oracle.chunkwise(q[:, :, :N], k[:, :, :N], v[:, :, :N], G3, B, return_state=True)
    assert rel(pre, whole[:, :, :N]) < 1e-12
    for t in range(N, N + extra):
        o, state = oracle.recurrent_step(q[:, :, t], k[:, :, t], v[:, :, t], state, G3)
        assert rel(o, whole[:, :, t]) < 1e-12


def test_chunkwise_state_in_continues_sequence():
    b, H, N, dk, dv, B = 2, 3, 48, 5, 3, 8
    q, k, v = rand((b, H, N, dk), 81), rand((b, H, N, dk), 82), rand((b, H, N, dv), 83)
    whole, s_end = oracle.chunkwise(q, k, v, G3, B, return_state=True)
    h1, s_mid = oracle.chunkwise(q[:, :, :16], k[:, :, :16], v[:, :, :16], G3, B, return_state=True)
    h2, s_end2 = oracle.chunkwise(q[:, :, 16:], k[:, :, 16:], v[:, :, 16:], G3, 16,
                                  state_in=s_mid, return_state=True)
    assert rel(np.concatenate([h1, h2], axis=2), whole) < 1e-12
    assert rel(s_end2, s_end) < 1e-12


def test_decode_from_nonzero_state_matches_closed_form():
    """One step from S0: S1 = gamma S0 + k^T v, o = q S1 (the updated state)."""
    b, H, dk, dv = 2, 3, 4, 5
    S0 = rand((b, H, dk, dv), 91)
    q, k, v = rand((b, H, dk), 92), rand((b, H, dk), 93), rand((b, H, dv), 94)
    o, S1 = oracle.recurrent_step(q, k, v, S0, G3)
    g = np.array(G3)[None, :, None, None]
    want_S = g * S0 + np.einsum("bha,bhc->bhac", k, v)
    assert rel(S1, want_S) < 1e-14
    assert rel(o, np.einsum("bha,bhac->bhc", q, want_S)) < 1e-14
