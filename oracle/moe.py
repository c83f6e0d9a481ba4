"""Mixture-of-experts block with within-expert tensor parallelism (test infrastructure only).

[MLX] "Tensor Parallelism", MoE Expert Parallelism, Within-Expert Parallel:
every expert's FFN is split over the ranks with the same column-parallel
gate/up and row-parallel down pattern as a dense FFN. The pages give no router
arithmetic, so the routing is an input: for every token the ids of the k
experts it goes to and their gate weights. The block's output for a token is
the gate-weighted sum of those experts' FFN outputs (the combine that ends
every top-k MoE layer).

  y[i] = sum_j gate[i, j] * FFN_{e[i, j]}(x[i]),  FFN_e(x) = (silu(x Wg_e) * (x Wu_e)) Wd_e

``moe_block`` is that definition; ``moe_block_tp`` computes each expert
through its t-way split (``mlp_block_tp``) to pin the within-expert layout.
Pinned in ``tests/test_oracle_moe.py``.
"""
from __future__ import annotations

import numpy as np

from .attention import _as_f64
from .tp_block import mlp_block, mlp_block_tp


def _check_routing(expert_ids, gates, n_experts: int, T: int):
    e = np.asarray(expert_ids, np.int64)
    g = _as_f64(gates)
    if e.ndim != 2 or e.shape[0] != T or g.shape != e.shape:
        raise ValueError("expert_ids and gates must both be [T, k]")
    if e.size and (e.min() < 0 or e.max() >= n_experts):
        raise ValueError("expert id out of range")
    return e, g


def moe_block(x, expert_ids, gates, w_gate, w_up, w_down) -> np.ndarray:
    """Top-k MoE combine over per-expert gated MLPs.

    x [T, H]; expert_ids, gates [T, k]; w_gate, w_up: E tensors [I, H]; w_down: E
    tensors [H, I] (stored [out, in]). A token may list an expert once per slot.
    """
    X = _as_f64(x)
    E = len(w_gate)
    e, g = _check_routing(expert_ids, gates, E, X.shape[0])
    y = np.zeros_like(X)
    for ex in range(E):
        rows, slots = np.nonzero(e == ex)
        if rows.size == 0:
            continue
        out = mlp_block(X[rows], _as_f64(w_gate[ex]), _as_f64(w_up[ex]), _as_f64(w_down[ex]))
        np.add.at(y, rows, g[rows, slots][:, None] * out)
    return y


def moe_block_tp(x, expert_ids, gates, w_gate, w_up, w_down, t: int) -> np.ndarray:
    """The same block with every expert computed through its t-way column/row split."""
    X = _as_f64(x)
    E = len(w_gate)
    e, g = _check_routing(expert_ids, gates, E, X.shape[0])
    y = np.zeros_like(X)
    for ex in range(E):
        rows, slots = np.nonzero(e == ex)
        if rows.size == 0:
            continue
        out, _ = mlp_block_tp(X[rows], _as_f64(w_gate[ex]), _as_f64(w_up[ex]), _as_f64(w_down[ex]), t)
        np.add.at(y, rows, g[rows, slots][:, None] * out)
    return y
