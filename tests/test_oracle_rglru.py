"""Pins of the oracle's RG-LRU scan against facts that do not come from it.

Source: the Griffin page ("Griffin ：將門控線性循環與局部注意力混合以實現高效的語言模型"),
section "實門線性循環單元 (RG-LRU)": r_t = sigmoid(W_a x_t + b_a), i_t = sigmoid(W_x x_t +
b_x), a_t = a^(c r_t) with a = sigmoid(Lambda) and c = 8, h_t = a_t h_{t-1} +
sqrt(1 - a_t^2) (i_t x_t).  Pins:
  * a constant recurrence gate makes a_t a constant alpha per channel, and the scan a
    first-order IIR filter: scipy.signal.lfilter([sqrt(1-alpha^2)], [1, -alpha]) of
    i_t x_t with initial condition alpha h0 (a library routine);
  * r = 0 gives a_t = 1 and a zero input weight: h stays at h0;
  * a = 0 (Lambda -> -inf) gives a_t = 0: h_t = i_t x_t exactly;
  * the unrolled sum h_t = (prod_{s<=t} a_s) h0 + sum_{u<=t} (prod_{u<s<=t} a_s)
    sqrt(1 - a_u^2) i_u x_u, evaluated with numpy cumulative products;
  * the final state equals the last output.
"""
import numpy as np
import pytest
import scipy.signal

import oracle


def rand(shape, seed, scale=1.0):
    return scale * np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def sig(z):
    return 1.0 / (1.0 + np.exp(-z))


def test_constant_gate_is_a_first_order_filter():
    b, T, D, c = 2, 300, 5, 8.0
    x = rand((b, T, D), 1)
    gx = rand((b, T, D), 2)
    ga_const = rand((b, 1, D), 3)
    ga = np.repeat(ga_const, T, axis=1)
    lam = rand((D,), 4, 2.0)
    h0 = rand((b, D), 5)
    y, hl = oracle.rglru(x, ga, gx, lam, h0, c, return_state=True)
    for bi in range(b):
        for d in range(D):
            alpha = sig(lam[d]) ** (c * sig(ga_const[bi, 0, d]))
            u = sig(gx[bi, :, d]) * x[bi, :, d]
            want, _ = scipy.signal.lfilter([np.sqrt(1 - alpha ** 2)], [1.0, -alpha], u,
                                           zi=[alpha * h0[bi, d]])
            np.testing.assert_allclose(y[bi, :, d], want, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(hl, y[:, -1, :])


def test_closed_recurrence_gate_keeps_the_state():
    b, T, D = 1, 50, 4
    x = rand((b, T, D), 11)
    gx = rand((b, T, D), 12)
    ga = np.full((b, T, D), -1e4)          # r = sigmoid(-1e4) = 0 in fp64
    lam = rand((D,), 13)
    h0 = rand((b, D), 14)
    y = oracle.rglru(x, ga, gx, lam, h0)
    np.testing.assert_array_equal(y, np.repeat(h0[:, None, :], T, axis=1))


def test_zero_decay_passes_the_gated_input():
    b, T, D = 2, 40, 3
    x = rand((b, T, D), 21)
    gx = rand((b, T, D), 22)
    ga = rand((b, T, D), 23)
    lam = np.full((D,), -1e4)              # a = sigmoid(-1e4) = 0, a_t = 0^(c r_t) = 0
    y = oracle.rglru(x, ga, gx, lam, rand((b, D), 24))
    np.testing.assert_allclose(y, sig(gx) * x, rtol=1e-15, atol=0)


@pytest.mark.parametrize("c", [8.0, 1.0, 3.5])
def test_unrolled_sum(c):
    b, T, D = 2, 24, 6
    x = rand((b, T, D), 31)
    gx = rand((b, T, D), 32)
    ga = rand((b, T, D), 33)
    lam = rand((D,), 34, 3.0)
    h0 = rand((b, D), 35)
    y = oracle.rglru(x, ga, gx, lam, h0, c)
    at = sig(lam)[None, None, :] ** (c * sig(ga))
    w = np.sqrt(1 - at ** 2) * sig(gx) * x
    want = np.zeros_like(y)
    for t in range(T):
        prod_all = np.prod(at[:, :t + 1], axis=1)
        acc = prod_all * h0
        for u in range(t + 1):
            acc = acc + np.prod(at[:, u + 1:t + 1], axis=1) * w[:, u]
        want[:, t] = acc
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


def test_empty_sequence_returns_the_initial_state():
    h0 = rand((2, 4), 41)
    y, hl = oracle.rglru(np.zeros((2, 0, 4)), np.zeros((2, 0, 4)), np.zeros((2, 0, 4)),
                         np.zeros(4), h0, return_state=True)
    assert y.shape == (2, 0, 4)
    np.testing.assert_array_equal(hl, h0)
