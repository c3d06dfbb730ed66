"""Pins of the oracle's chunkwise gradient against facts that do not come from it.

The RetNet pages ([RN2] "Transformer取代者登場！微軟、清華剛推出RetNet：成本低、速度快、
性能強（2）", "訓練/推理": training runs the parallel and chunkwise forms) print no
backward pass, so the gradient is pinned by calculus:
  * the scalar L = sum(dout * o) + <dstate_out, S_final> is linear in each of q, k, v
    and the incoming state separately, so a central difference with ANY step equals the
    directional derivative up to rounding.  The forward oracle (pinned by its own tests
    in test_oracle_pins.py) supplies L, coordinate by coordinate on a tiny case and
    along random directions on a larger one;
  * gamma = 0 leaves only the diagonal term o_n = (q_n . k_n) v_n, whose gradient is
    written out by hand;
  * all-ones inputs with gamma = 1 give counting closed forms;
  * Euler's identity for functions homogeneous of degree one: sum(dout * o) equals
    <dq, q>, and (with no incoming state) <dv, v>.
dk != dv and distinct per-head decays throughout, so a transposed operand or a head
mix-up cannot cancel.
"""
import numpy as np
import pytest

import oracle


def rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def loss(q, k, v, do, gamma, chunk, s0=None, ds=None):
    """L from the forward oracle: sum(dout * o) + <dstate_out, final state>."""
    o, sf = oracle.chunkwise(q, k, v, gamma, chunk, state_in=s0, return_state=True)
    val = float(np.sum(do * o))
    if ds is not None:
        val += float(np.sum(ds * sf))
    return val


def case(seed, b, H, N, dk, dv, with_states=True):
    q = rand((b, H, N, dk), seed)
    k = rand((b, H, N, dk), seed + 1)
    v = rand((b, H, N, dv), seed + 2)
    do = rand((b, H, N, dv), seed + 3)
    s0 = rand((b, H, dk, dv), seed + 4) if with_states else None
    ds = rand((b, H, dk, dv), seed + 5) if with_states else None
    return q, k, v, do, s0, ds


@pytest.mark.parametrize("with_states", [False, True])
def test_every_coordinate_by_central_difference(with_states):
    """Each gradient entry equals (L(x + e_i) - L(x - e_i)) / 2, exact for a linear L."""
    b, H, N, dk, dv, chunk = 1, 2, 8, 4, 3, 4
    gamma = [0.9, 0.6]
    q, k, v, do, s0, ds = case(11, b, H, N, dk, dv, with_states)
    gq, gk, gv, gs = oracle.chunkwise_backward(q, k, v, do, gamma, state_in=s0, dstate_out=ds)
    args = {"q": q, "k": k, "v": v}
    if with_states:
        args["s0"] = s0
    grads = {"q": gq, "k": gk, "v": gv, "s0": gs}
    for name, x in args.items():
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            plus, minus = dict(args), dict(args)
            xp, xm = x.copy(), x.copy()
            xp[idx] += 1.0
            xm[idx] -= 1.0
            plus[name], minus[name] = xp, xm
            lp = loss(plus["q"], plus["k"], plus["v"], do, gamma, chunk, plus.get("s0"), ds)
            lm = loss(minus["q"], minus["k"], minus["v"], do, gamma, chunk, minus.get("s0"), ds)
            fd[idx] = (lp - lm) / 2.0
        scale = max(1.0, float(np.max(np.abs(fd))))
        assert np.max(np.abs(fd - grads[name])) < 1e-11 * scale, name


def test_random_directions_larger_case():
    """Directional derivatives along random directions, chunk 16, N 64, dk 16, dv 24."""
    b, H, N, dk, dv, chunk = 2, 3, 64, 16, 24, 16
    gamma = [0.97, 0.8, 0.999]
    q, k, v, do, s0, ds = case(21, b, H, N, dk, dv)
    gq, gk, gv, gs = oracle.chunkwise_backward(q, k, v, do, gamma, state_in=s0, dstate_out=ds)
    for t in range(3):
        eq, ek, ev, es = (rand(x.shape, 100 + 10 * t + i) for i, x in enumerate((q, k, v, s0)))
        for name, dx in (("q", eq), ("k", ek), ("v", ev), ("s0", es)):
            a = dict(q=q, k=k, v=v, s0=s0)
            m = dict(a)
            a[name] = a[name] + dx
            m[name] = m[name] - dx
            fd = (loss(a["q"], a["k"], a["v"], do, gamma, chunk, a["s0"], ds)
                  - loss(m["q"], m["k"], m["v"], do, gamma, chunk, m["s0"], ds)) / 2.0
            an = float(np.sum({"q": gq, "k": gk, "v": gv, "s0": gs}[name] * dx))
            assert abs(fd - an) <= 1e-10 * max(1.0, abs(an)), (name, fd, an)


def test_gamma_zero_is_the_diagonal_term():
    """gamma = 0: o_n = (q_n.k_n) v_n, so dq_n = (do_n.v_n) k_n, dk_n = (do_n.v_n) q_n,
    dv_n = (q_n.k_n) do_n, and the state (multiplied by gamma^(n+1)) gets no gradient
    except gamma^N dstate_out = 0."""
    b, H, N, dk, dv = 1, 2, 12, 5, 7
    q, k, v, do, s0, ds = case(31, b, H, N, dk, dv)
    gq, gk, gv, gs = oracle.chunkwise_backward(q, k, v, do, [0.0, 0.0], state_in=s0,
                                                dstate_out=None)
    dov = np.einsum("bhnc,bhnc->bhn", do, v)[..., None]
    qk = np.einsum("bhna,bhna->bhn", q, k)[..., None]
    np.testing.assert_allclose(gq, dov * k, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(gk, dov * q, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(gv, qk * do, rtol=1e-13, atol=1e-13)
    assert np.all(gs == 0.0)


def test_all_ones_gamma_one_closed_forms():
    """gamma = 1, q = k = v = dout = 1, no states: each of the n+1 tokens m <= n adds
    (do_n.v_m) k_m, so dq_n = dv (n+1) in every entry; each of the N-m tokens n >= m
    adds (do_n.v_m) q_n and (q_n.k_m) do_n, so dk_m = dv (N-m) and dv_m = dk (N-m); the
    gradient of the (zero) incoming state is sum_n q_n^T do_n = N in every entry."""
    b, H, N, dk, dv = 1, 1, 10, 3, 5
    one = lambda *s: np.ones(s)
    gq, gk, gv, gs = oracle.chunkwise_backward(one(b, H, N, dk), one(b, H, N, dk),
                                                one(b, H, N, dv), one(b, H, N, dv), [1.0])
    n = np.arange(N, dtype=np.float64)
    np.testing.assert_array_equal(gq[0, 0], np.repeat((dv * (n + 1))[:, None], dk, 1))
    np.testing.assert_array_equal(gk[0, 0], np.repeat((dv * (N - n))[:, None], dk, 1))
    np.testing.assert_array_equal(gv[0, 0], np.repeat((dk * (N - n))[:, None], dv, 1))
    np.testing.assert_array_equal(gs[0, 0], np.full((dk, dv), float(N)))


def test_euler_identity_degree_one():
    """o is homogeneous of degree one in q, so sum(dout * o) = <dq, q>; with no incoming
    state o is also homogeneous of degree one in v, so sum(dout * o) = <dv, v>, and
    likewise in k."""
    b, H, N, dk, dv, chunk = 1, 3, 48, 8, 12, 16
    gamma = [0.95, 0.7, 1.0]
    q, k, v, do, _, _ = case(41, b, H, N, dk, dv, with_states=False)
    o = oracle.chunkwise(q, k, v, gamma, chunk)
    L = float(np.sum(do * o))
    gq, gk, gv, _ = oracle.chunkwise_backward(q, k, v, do, gamma)
    for g, x in ((gq, q), (gk, k), (gv, v)):
        assert abs(float(np.sum(g * x)) - L) <= 1e-11 * max(1.0, abs(L))

