"""Pins of the oracle's xPos rotation against facts that do not come from it.

[RN2] "Transformer取代者登場！微軟、清華剛推出RetNet：成本低、速度快、性能強（2）",
"Retention", eqs.(2)-(3) (formulas lost; the prose survives): Q_n e^{i n theta} and
K_m e^{i m theta}, "xPos, a relative position embedding", scores taken with the
conjugate transpose.  Pins:
  * numpy complex arithmetic: each coordinate pair as a complex number times
    numpy.exp(1j * p * theta) (a library routine, not the oracle's cos/sin formulas);
  * theta = 0 is the identity; the norm of every pair is preserved;
  * relative position: the retention score q'_n . k'_m after rotating both depends on
    n - m only, so shifting every position by s (pos0) leaves every score unchanged,
    and the rotated score equals Re(sum_j z_q conj(z_k) e^{i (n-m) theta_j});
  * phases add: rotating by theta1 then theta2 equals rotating by theta1 + theta2.
"""
import numpy as np

import oracle


def rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def thetas(d, seed=0):
    return 10000.0 ** (-np.arange(d // 2) / (d // 2)) * (1 + 0.1 * rand((d // 2,), seed))


def as_complex(x):
    return x[..., 0::2] + 1j * x[..., 1::2]


def test_matches_complex_multiplication():
    b, H, N, d, pos0 = 2, 3, 40, 16, 1234
    x = rand((b, H, N, d), 1)
    th = thetas(d, 2)
    out = oracle.xpos_rotate(x, th, pos0)
    p = pos0 + np.arange(N)
    want = as_complex(x) * np.exp(1j * p[:, None] * th[None, :])
    np.testing.assert_allclose(out[..., 0::2], want.real, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out[..., 1::2], want.imag, rtol=1e-12, atol=1e-12)


def test_zero_theta_is_identity_and_norms_are_kept():
    x = rand((1, 2, 30, 8), 3)
    np.testing.assert_array_equal(oracle.xpos_rotate(x, np.zeros(4), 77), x)
    out = oracle.xpos_rotate(x, thetas(8, 4), 5)
    np.testing.assert_allclose(np.abs(as_complex(out)), np.abs(as_complex(x)), rtol=1e-13)


def test_scores_depend_on_relative_position_only():
    b, H, N, d = 1, 2, 24, 12
    q, k = rand((b, H, N, d), 5), rand((b, H, N, d), 6)
    th = thetas(d, 7)
    s0 = np.einsum("bhnd,bhmd->bhnm", oracle.xpos_rotate(q, th, 0), oracle.xpos_rotate(k, th, 0))
    s1 = np.einsum("bhnd,bhmd->bhnm", oracle.xpos_rotate(q, th, 1000),
                   oracle.xpos_rotate(k, th, 1000))
    np.testing.assert_allclose(s1, s0, rtol=1e-9, atol=1e-9)
    n = np.arange(N)
    phase = np.exp(1j * (n[:, None, None] - n[None, :, None]) * th[None, None, :])
    want = np.einsum("bhnj,bhmj,nmj->bhnm", as_complex(q), np.conj(as_complex(k)), phase).real
    np.testing.assert_allclose(s0, want, rtol=1e-10, atol=1e-10)


def test_phases_add():
    x = rand((1, 1, 16, 6), 8)
    t1, t2 = thetas(6, 9), thetas(6, 10)
    two = oracle.xpos_rotate(oracle.xpos_rotate(x, t1, 3), t2, 3)
    np.testing.assert_allclose(two, oracle.xpos_rotate(x, t1 + t2, 3), rtol=1e-10, atol=1e-10)
