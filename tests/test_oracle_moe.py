"""Pins of the MoE oracle (CPU only).

Checked against per-token explicit loops, special routings that reduce the
block to the dense MLP, token-permutation equivariance, linearity in the
gates, and the within-expert t-way split for t in {1, 2, 4, 8}. Planted
mistakes (gate and up exchanged, gates ignored, tokens sent to the wrong
expert) must fail the brute-force pin.
"""
import importlib
import math

import numpy as np
import pytest

import oracle

moe = importlib.import_module("oracle.moe")


def _loops(x, ids, gates, wg, wu, wd):
    T, H = x.shape
    y = np.zeros((T, H))
    for i in range(T):
        for j in range(ids.shape[1]):
            e = ids[i, j]
            I = wg[e].shape[0]
            h = []
            for c in range(I):
                g = sum(x[i, a] * wg[e][c, a] for a in range(H))
                u = sum(x[i, a] * wu[e][c, a] for a in range(H))
                h.append(g / (1.0 + math.exp(-g)) * u)
            for o in range(H):
                y[i, o] += gates[i, j] * sum(h[c] * wd[e][o, c] for c in range(I))
    return y


def _case(T=6, H=8, I=8, E=4, k=2, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    gates = rng.uniform(0.1, 1.0, (T, k))
    wg = [rng.standard_normal((I, H)) * 0.5 for _ in range(E)]
    wu = [rng.standard_normal((I, H)) * 0.5 for _ in range(E)]
    wd = [rng.standard_normal((H, I)) * 0.5 for _ in range(E)]
    return x, ids, gates, wg, wu, wd


def test_matches_loops():
    c = _case()
    np.testing.assert_allclose(oracle.moe_block(*c), _loops(*c), rtol=1e-11, atol=1e-11)


def test_one_expert_gate_one_is_the_dense_mlp():
    x, ids, gates, wg, wu, wd = _case(k=1)
    ids[:] = 2
    gates[:] = 1.0
    np.testing.assert_allclose(oracle.moe_block(x, ids, gates, wg, wu, wd),
                               oracle.mlp_block(x, wg[2], wu[2], wd[2]), rtol=1e-13, atol=1e-13)


def test_identical_experts_with_gates_summing_to_one_are_the_dense_mlp():
    x, ids, gates, wg, wu, wd = _case(k=3, E=5)
    gates = gates / gates.sum(axis=1, keepdims=True)
    same = lambda w: [w[0]] * len(w)
    np.testing.assert_allclose(oracle.moe_block(x, ids, gates, same(wg), same(wu), same(wd)),
                               oracle.mlp_block(x, wg[0], wu[0], wd[0]), rtol=1e-12, atol=1e-12)


def test_token_permutation_permutes_the_output():
    x, ids, gates, wg, wu, wd = _case(T=9, seed=3)
    perm = np.random.default_rng(4).permutation(9)
    y = oracle.moe_block(x, ids, gates, wg, wu, wd)
    np.testing.assert_allclose(oracle.moe_block(x[perm], ids[perm], gates[perm], wg, wu, wd), y[perm],
                               rtol=1e-13, atol=1e-13)


def test_linear_in_the_gates():
    x, ids, gates, wg, wu, wd = _case(seed=5)
    y = oracle.moe_block(x, ids, gates, wg, wu, wd)
    np.testing.assert_allclose(oracle.moe_block(x, ids, 2.5 * gates, wg, wu, wd), 2.5 * y, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_within_expert_split_is_invariant(t):
    x, ids, gates, wg, wu, wd = _case(T=10, H=16, I=32, E=3, seed=6)
    np.testing.assert_allclose(oracle.moe_block_tp(x, ids, gates, wg, wu, wd, t),
                               oracle.moe_block(x, ids, gates, wg, wu, wd), rtol=1e-12, atol=1e-12)


def test_rejects_bad_routing():
    x, ids, gates, wg, wu, wd = _case()
    with pytest.raises(ValueError):
        oracle.moe_block(x, ids + 10, gates, wg, wu, wd)
    with pytest.raises(ValueError):
        oracle.moe_block(x, ids[:, :1], gates, wg, wu, wd)


def _pin_passes() -> bool:
    try:
        test_matches_loops()
    except AssertionError:
        return False
    return True


def test_pin_passes_unmodified():
    assert _pin_passes()


_mlp = moe.mlp_block


@pytest.mark.parametrize("name,bad", [
    ("mlp_block", lambda x, wg, wu, wd: _mlp(x, wu, wg, wd)),                       # gate and up exchanged
    ("_check_routing", lambda e, g, E, T: (np.asarray(e), np.ones(np.shape(g)))),   # gates ignored
    ("_check_routing", lambda e, g, E, T: ((np.asarray(e) + 1) % E, np.asarray(g))),  # wrong expert
])
def test_planted_mistake_is_caught(monkeypatch, name, bad):
    monkeypatch.setattr(moe, name, bad)
    assert not _pin_passes()
