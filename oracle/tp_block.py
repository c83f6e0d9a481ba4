"""Float64 restatement of the tensor-parallel linear block (test infrastructure only).

Conventions. A weight is stored as ``nn.Linear`` keeps it, [out, in]. The
pages write the linear layer as Y = XW + b with X [b, k], W [k, n], b [n]
([VSC] "一个矩阵乘法如何被切开"), so their W is the transpose of the stored
array: Y = X @ W_stored.T. No configuration carries a bias.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------- helpers

def bf16_to_f64(x) -> np.ndarray:
    """bf16 values -> float64, exactly.

    Accepts a torch bf16 tensor or an array of raw uint16 bf16 bit patterns.
    A bf16 value is the top half of an IEEE float32, so widening the bits and
    viewing them as float32 is exact, and so is float32 -> float64.
    """
    if not isinstance(x, np.ndarray):            # torch tensor: widening bf16 -> float64 is exact
        import torch
        return x.detach().cpu().to(torch.float64).numpy()
    bits = np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def divide(n: int, t: int) -> int:
    """n / t, refusing a remainder.

    [VSC] "ColumnParallelLinear：沿输出维切权重": the per-partition size is
    output_size // tp_size and must divide exactly.
    """
    if t <= 0 or n % t != 0:
        raise ValueError(f"{n} is not divisible by {t}")
    return n // t


# --------------------------------------------------------------------------- linear layers

def linear(X: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Y = XW for X [b, k] and a stored weight W [n, k] (the pages' W is W.T).

    [VSC] "一个矩阵乘法如何被切开": the dense layer's product, bias-free.
    """
    return np.asarray(X, np.float64) @ np.asarray(W, np.float64).T


def column_parallel(X: np.ndarray, W: np.ndarray, t: int) -> list[np.ndarray]:
    """Per-shard outputs of a column-parallel layer: Y_r = X W_r.

    [VSC] "Column（列）切法" and "ColumnParallelLinear": the weight is split
    along the output dimension into t equal blocks; shard r holds output
    features [r*n/t, (r+1)*n/t) (``narrow(output_dim, r*shard, shard)``) and
    multiplies them by the full, replicated input. [VCR] §12 states the same
    split as A = [A0, ..., A(tp-1)], Yi = X Ai. Concatenating the Y_r along
    the last dimension gives Y; no reduction is needed.
    """
    n = W.shape[0]
    s = divide(n, t)
    return [linear(X, W[r * s:(r + 1) * s]) for r in range(t)]


def row_parallel(X: np.ndarray, W: np.ndarray, t: int) -> list[np.ndarray]:
    """Per-shard partial sums of a row-parallel layer: P_r = X_r W_r.

    [VSC] "Row（行）切法" and "RowParallelLinear": the weight is split along
    its input dimension and the input along its last dimension into t equal
    blocks; shard r computes X_r W_r over input features [r*k/t, (r+1)*k/t).
    [VCR] §12: Y = sum_i Yi, which the all-reduce forms. The caller sums.
    """
    k = W.shape[1]
    s = divide(k, t)
    return [linear(X[:, r * s:(r + 1) * s], W[:, r * s:(r + 1) * s]) for r in range(t)]


def reduce_scatter(partials, t: int) -> list[np.ndarray]:
    """Sequence-parallel end of a row-parallel layer: the t partial sums are added and
    the sum is split by token, rank r keeping rows [r*T/t, (r+1)*T/t).

    [MLX] "Tensor Parallelism", collectives: a reduce-scatter replaces the
    all-reduce when the next layer needs only a shard of the output; [UC]
    "residual_stream" and [VCR] section 4 (PP + SP): with sequence parallelism
    the residual is split across the TP ranks by token, after padding the token
    count. Rows are padded with zeros up to a multiple of t (the padded count is
    t * ceil(T/t)); slice r of the result is what rank r holds.
    """
    y = np.zeros_like(np.asarray(partials[0], np.float64))
    for p in partials:
        y = y + np.asarray(p, np.float64)
    T = y.shape[0]
    per = -(-T // t)
    pad = np.zeros((per * t - T,) + y.shape[1:])
    y = np.concatenate([y, pad], axis=0)
    return [y[r * per:(r + 1) * per] for r in range(t)]


# --------------------------------------------------------------------------- elementwise

def silu(z: np.ndarray) -> np.ndarray:
    """SiLU: z * sigmoid(z), sigmoid(z) = 1 / (1 + exp(-z)).

    The pages name only "the activation on the local shard" of the gated MLP
    ([VCR] §14); the gated Llama MLP's activation is SiLU. Evaluated without
    overflow for large |z|.
    """
    z = np.asarray(z, np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    e = np.exp(z[~pos])
    out[~pos] = z[~pos] * e / (1.0 + e)
    return out


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Gated activation h = silu(gate) * up, gate first, up second.

    [VSC] "MergedColumnParallelLinear": gate_up_proj concatenates gate and up
    along the output dimension (output_sizes=[I, I]); the activation combines
    the two halves on each shard ([VCR] §14 "activation: 在局部分片上完成").
    """
    return silu(g) * np.asarray(u, np.float64)


def rms_norm(r: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """x = r / sqrt(mean_j r_j^2 + eps) * gamma over the hidden dimension.

    [UC] "final_norm" builds ``RMSNorm(hidden_size, eps)``; the pages print no
    formula, so this is the textbook RMSNorm: no centring, no bias, gamma
    applied after normalising.
    """
    r = np.asarray(r, np.float64)
    ms = np.mean(r * r, axis=-1, keepdims=True)
    return r / np.sqrt(ms + eps) * np.asarray(gamma, np.float64)


def add_rms_norm(a: np.ndarray, residual: np.ndarray, gamma: np.ndarray, eps: float):
    """Fused residual add + RMSNorm: r = a + residual, x = RMSNorm(r); returns (x, r).

    [UC] "residual_stream": ``post_attention_layernorm(hidden_states, residual)``
    returns the normalised hidden states and the updated residual; the norms
    and residual adds are unsharded elementwise ops over the full hidden dim.
    """
    r = np.asarray(a, np.float64) + np.asarray(residual, np.float64)
    return rms_norm(r, gamma, eps), r


# --------------------------------------------------------------------------- MLP block

def mlp_block(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """Unsharded gated MLP: y = (silu(x Wg) * (x Wu)) Wd.

    [VCR] §14 and [VSC] "一个典型 block 的列行交替拼装": gate_up_proj, the
    activation, down_proj. This is the plain definition every sharded layout
    must reproduce.
    """
    h = silu_mul(linear(x, w_gate), linear(x, w_up))
    return linear(h, w_down)


def mlp_block_tp(x, w_gate, w_up, w_down, t: int):
    """The same MLP computed through its t-way tensor-parallel layout.

    MergedColumnParallelLinear: shard r holds [gate rows of r ; up rows of r]
    and computes its gate and up outputs; the activation runs on the local
    shard; RowParallelLinear: shard r multiplies its h_r by the matching input
    columns of Wd; the t partial sums are added (the all-reduce). Returns
    (y, [h_r]).
    [VCR] §14; [VSC] "MergedColumnParallelLinear", "RowParallelLinear".
    """
    I = w_gate.shape[0]
    s = divide(I, t)
    h_shards = []
    for r in range(t):
        w_gu_r = np.concatenate([w_gate[r * s:(r + 1) * s], w_up[r * s:(r + 1) * s]], axis=0)
        gu = linear(x, w_gu_r)                       # [T, 2s]: gate half then up half
        h_shards.append(silu_mul(gu[:, :s], gu[:, s:]))
    partials = [linear(h_shards[r], w_down[:, r * s:(r + 1) * s]) for r in range(t)]
    y = np.zeros_like(partials[0])
    for p in partials:                               # ascending shard order
        y = y + p
    return y, h_shards


def mlp_layer(x_in, w_gate, w_up, w_down, residual=None, gamma=None, eps: float = 1e-5,
              norm: bool = False, rows=None) -> dict:
    """The MLP half of a decoder layer as the capture hooks see it.

    With ``norm``: r = x_in + residual, x = RMSNorm(r) ([UC] "residual_stream",
    post_attention_layernorm); otherwise x = x_in and r = residual (may be
    None). Then mlp_out = MLP(x) ([UC] "mlp_out", the reduced down_proj
    output) and residual_stream = mlp_out + r ([UC] "residual_stream": the
    adapter captures hidden_states + residual, the stream after the layer).

    ``rows`` restricts the computation to those token rows (rows are
    independent through the whole block).
    """
    sl = slice(None) if rows is None else np.asarray(rows)
    x_in = np.asarray(x_in, np.float64)[sl]
    r = None if residual is None else np.asarray(residual, np.float64)[sl]
    if norm:
        x, r = add_rms_norm(x_in, r, gamma, eps)
    else:
        x = x_in
    y = mlp_block(x, w_gate, w_up, w_down)
    out = {"mlp_out": y, "residual_out": r}
    out["residual_stream"] = None if r is None else y + r
    return out


# --------------------------------------------------------------------------- attention projections

def gqa_partition(nq: int, nkv: int, t: int):
    """Heads per shard under GQA: (q heads per shard, kv heads per shard, kv replicas).

    [VSC] "MergedColumnParallelLinear / QkvParallelLinear": q heads are split
    evenly (divide(nq, t)); if t >= nkv every shard holds one kv head and each
    kv head is replicated on t / nkv shards, else each shard holds nkv / t kv
    heads and there is one replica.
    """
    q = divide(nq, t)
    if t >= nkv:
        return q, 1, divide(t, nkv)
    return q, divide(nkv, t), 1


def qkv_shard_rows(nq: int, nkv: int, hd: int, t: int):
    """Which rows of [Wq; Wk; Wv] each QKV shard holds, in its output order.

    Shard r's output is [its q heads | its k heads | its v heads], each head
    hd consecutive rows of the stored weight. q heads of shard r are
    r*nq/t .. (r+1)*nq/t - 1. kv heads: r*kv_per .. when kv heads are split;
    when they are replicated (t >= nkv), shard r holds kv head r // replicas
    ([VSC] QkvParallelLinear, num_kv_head_replicas). Returns a list of
    (tensor, row) index arrays, tensor 0 = q, 1 = k, 2 = v.
    """
    q_per, kv_per, rep = gqa_partition(nq, nkv, t)
    shards = []
    for r in range(t):
        q_heads = range(r * q_per, (r + 1) * q_per)
        if rep > 1:
            kv_heads = [r // rep]
        else:
            kv_heads = range(r * kv_per, (r + 1) * kv_per)
        idx = []
        for tensor, heads in ((0, q_heads), (1, kv_heads), (2, kv_heads)):
            for hh in heads:
                for d in range(hd):
                    idx.append((tensor, hh * hd + d))
        shards.append(np.array(idx, dtype=np.int64))
    return shards


def qkv_parallel(x, w_q, w_k, w_v, nq: int, nkv: int, hd: int, t: int) -> np.ndarray:
    """Column-parallel QKV split by head: out[r] = x [Wq_r; Wk_r; Wv_r].

    [VCR] §13: each shard computes the q/k/v heads it owns; not gathered
    (gather_output=False, [VSC] ColumnParallelLinear). Returns [t, T, w_s].
    """
    ws = (w_q, w_k, w_v)
    outs = []
    for rows in qkv_shard_rows(nq, nkv, hd, t):
        W_r = np.stack([np.asarray(ws[a][b], np.float64) for a, b in rows])
        outs.append(linear(x, W_r))
    return np.stack(outs)


def o_proj_parallel(attn_shards, w_o, t: int) -> np.ndarray:
    """Row-parallel o_proj: attn_out = sum_r A_r Wo_r with A_r the local heads of shard r.

    [VCR] §13 (O projection: every shard produces a partial [N, hidden], the
    all-reduce sums them); [UC] "attn_out" (o_proj has already reduced).
    ``attn_shards`` is [t, T, nq*hd/t]. Partials are added in ascending r.
    """
    A = np.concatenate([np.asarray(a, np.float64) for a in attn_shards], axis=1)
    parts = row_parallel(A, w_o, t)
    y = np.zeros_like(parts[0])
    for p in parts:
        y = y + p
    return y
