"""The pins are sharp: a mutated copy of the oracle fails them.

Each case copies ``oracle/retention_oracle.c`` to a temporary directory, plants
one plausible slip by text substitution (the committed oracle is untouched),
compiles it and checks that a pin that does not depend on the oracle (a closed
form or a library routine) now rejects it.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "retention_oracle.c")


def mutant(tmp_path, old, new, name):
    text = open(SRC).read()
    assert text.count(old) >= 1, old
    p = tmp_path / f"{name}.c"
    p.write_text(text.replace(old, new, 1))
    return oracle.Oracle(oracle.build(force=True, src=str(p), out=str(tmp_path / f"{name}.so")))


def rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def rel(a, b):
    return float(np.max(np.abs(a - b)) / np.sqrt(np.mean(b * b)))


G = [0.9, 0.5, 0.97]


def gamma_one_truth(q, k, v):
    outer = np.einsum("bhna,bhnc->bhnac", k, v)
    return np.einsum("bhna,bhnac->bhnc", q, np.cumsum(outer, axis=2))


def ones_truth(N, dk, g):
    n = np.arange(N)
    return dk * (1 - g ** (n + 1)) / (1 - g)


CHUNK_MUTATIONS = [
    ("xi_exponent", "xi[j] = gpow(g, j + 1)", "xi[j] = gpow(g, j)"),
    ("zeta_exponent", "zeta[j] = gpow(g, B - 1 - j)", "zeta[j] = gpow(g, B - j)"),
    ("state_not_decayed", "Rn[e] = gB * R[e]", "Rn[e] = R[e]"),
    ("inner_decay_sign", "gpow(g, j - r);", "gpow(g, r - j);"),
]


@pytest.mark.parametrize("name,old,new", CHUNK_MUTATIONS)
def test_chunkwise_mutants_fail_closed_form(tmp_path, name, old, new):
    m = mutant(tmp_path, old, new, name)
    b, H, N, dk, dv = 1, 3, 32, 4, 3
    q = np.ones((b, H, N, dk)); v = np.ones((b, H, N, dv))
    o = m.chunkwise(q, q, v, G, 8)
    worst = max(np.max(np.abs(o[0, h, :, 0] - ones_truth(N, dk, g))) for h, g in enumerate(G))
    assert worst > 1e-6, name


def test_recurrent_mutant_reading_old_state_fails(tmp_path):
    """Reading o_n from S_{n-1} instead of the updated S_n."""
    text_old = "S[(size_t)a * dv + c] = g * S[(size_t)a * dv + c] + kn[a] * vn[c];"
    m = mutant(tmp_path, text_old, "S[(size_t)a * dv + c] = S[(size_t)a * dv + c];",
               "old_state")
    q, k, v = rand((1, 1, 9, 3), 1), rand((1, 1, 9, 3), 2), rand((1, 1, 9, 2), 3)
    assert rel(m.recurrent(q, k, v, [1.0]), gamma_one_truth(q, k, v)) > 1e-3


def test_parallel_transposed_scores_fail(tmp_path):
    """Using k_n.q_m (a transposed score matrix) breaks the gamma=1 prefix sum."""
    m = mutant(tmp_path, "dot(Q + (size_t)n * dk, K + (size_t)m * dk, dk)",
               "dot(Q + (size_t)m * dk, K + (size_t)n * dk, dk)", "transposed")
    q, k, v = rand((1, 1, 9, 3), 4), rand((1, 1, 9, 3), 5), rand((1, 1, 9, 2), 6)
    assert rel(m.parallel(q, k, v, [1.0]), gamma_one_truth(q, k, v)) > 1e-3


def test_rowsum_without_abs_fails(tmp_path):
    m = mutant(tmp_path, "fabs(rs) > 1.0 ? fabs(rs) : 1.0", "rs > 1.0 ? rs : 1.0", "noabs")
    N = 40
    q = np.zeros((1, 1, N, 2)); k = np.zeros((1, 1, N, 2)); v = np.ones((1, 1, N, 1))
    q[..., 0] = 1.0; k[..., 0] = -1.0
    o = m.parallel(q, k, v, [0.9], 4)
    assert np.max(np.abs(o[0, 0, :, 0] + 1.0)) > 0.5   # truth is -1 everywhere


def test_decay_norm_wrong_power_fails(tmp_path):
    m = mutant(tmp_path, "d /= sqrt(drow);", "d /= drow;", "decaynorm")
    N = 20
    q = np.zeros((1, 1, N, 2)); q[..., 0] = 1.0; v = np.ones((1, 1, N, 1))
    o = m.parallel(q, q, v, [0.9], 2)
    n = np.arange(N)
    assert np.max(np.abs(o[0, 0, :, 0] - np.sqrt((1 - 0.9 ** (n + 1)) / 0.1))) > 1e-3


@pytest.mark.parametrize("name,old,new", [
    ("unbiased_var", "var /= dv;", "var /= (dv - 1);"),
    ("swish_sign", "gv / (1.0 + exp(-gv))", "gv / (1.0 + exp(gv))"),
    ("eps_outside", "1.0 / sqrt(var + eps)", "1.0 / (sqrt(var) + eps)"),
])
def test_epilogue_mutants_fail_torch(tmp_path, name, old, new):
    m = mutant(tmp_path, old, new, name)
    b, H, N, dv = 1, 2, 3, 8
    y = rand((b, H, N, dv), 7) * 0.05
    g = rand((b, N, H * dv), 8)
    x = torch.from_numpy(y).permute(0, 2, 1, 3).reshape(b * N, H * dv)
    yn = torch.nn.functional.group_norm(x, H, None, None, 0.1).reshape(b, N, H * dv)
    want = (torch.nn.functional.silu(torch.from_numpy(g)) * yn).numpy()
    assert rel(m.msr_epilogue(y, g, 0.1), want) > 1e-3
    assert rel(oracle.msr_epilogue(y, g, 0.1), want) < 1e-12
