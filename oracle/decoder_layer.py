"""One whole decoder layer as a chain of the oracle's steps (test infrastructure only).

[VCR] sections 13 and 14 give the order of one tensor-parallel decoder layer:
the column-parallel QKV projection split by head, attention on each rank's own
heads, the row-parallel o_proj with its reduction, then the MLP (column-parallel
gate_up, the activation on the local shard, row-parallel down with its
reduction). [UC] "What the adapter hooks" and "residual_stream": the layer's
fused input_layernorm adds the incoming hidden states to the residual before it
normalises; attn_out and mlp_out are the reduced outputs of self_attn and mlp;
residual_stream is the stream after the layer.

The chain, in float64, with nothing rounded in between (the GPU rounds every
intermediate tensor to bf16; the parity tolerance covers it):

  r1 = hidden + residual             (residual None: r1 = hidden, the first layer)
  x1 = RMSNorm(r1) * gamma_attn      (input_layernorm)
  qkv = qkv_parallel(x1)             (shard-major, not gathered)
  A = attention_core(qkv)            (causal, GQA, sequences packed by offsets)
  attn_out = o_proj_parallel(A)      (sum over the shards)
  r2 = attn_out + r1; x2 = RMSNorm(r2) * gamma_mlp   (post_attention_layernorm)
  mlp_out = (silu(x2 Wg) * (x2 Wu)) Wd
  residual_stream = mlp_out + r2

Pinned in ``tests/test_oracle_layer.py`` against explicit loops on a tiny
layer, special weights that switch one half off, t invariance and planted
mistakes.
"""
from __future__ import annotations

import numpy as np

from .attention import _as_f64, attention_core, attention_rows
from .tp_block import add_rms_norm, mlp_block, o_proj_parallel, qkv_parallel, rms_norm


def decoder_layer(hidden, residual, gamma_attn, w_q, w_k, w_v, w_o, gamma_mlp, w_gate, w_up, w_down,
                  nq: int, nkv: int, hd: int, t: int, cu_seqlens, eps: float = 1e-5, rows=None) -> dict:
    """The tensors of one decoder layer: residual_attn (r1), attn_out, residual_mlp (r2),
    mlp_out, residual_stream, plus the shard-major intermediates qkv and attn (A).

    Inputs are torch bf16 tensors, raw bf16 bits (uint16) or float arrays.
    hidden, residual [T, H]; gamma_attn, gamma_mlp [H]; w_q [nq*hd, H], w_k, w_v [nkv*hd, H],
    w_o [H, nq*hd], w_gate, w_up [I, H], w_down [H, I] (stored [out, in]); cu_seqlens
    [n_seqs + 1] token offsets of the packed sequences.

    ``rows``: compute the outputs of those token rows only. A row's attention reads
    the keys and values of its own sequence up to itself, so r1, x1 and qkv are
    computed for exactly those tokens (rows are independent through the norm and
    the projections); everything after the attention is per row. ``qkv`` is then
    still [t, T, w_s], zero at the tokens no row needs, and every other tensor has
    len(rows) rows.
    """
    f = _as_f64
    cu = np.asarray(cu_seqlens, np.int64)
    hid = f(hidden)
    res = None if residual is None else f(residual)
    T = hid.shape[0]
    if rows is None:
        tok = np.arange(T)
    else:
        rows = np.asarray(rows, np.int64)
        need = np.zeros(T, dtype=bool)
        for row in rows:
            need[cu[np.searchsorted(cu, row, side="right") - 1]:row + 1] = True
        tok = np.nonzero(need)[0]
    if res is None:
        r1 = hid[tok]
        x1 = rms_norm(r1, f(gamma_attn), eps)
    else:
        x1, r1 = add_rms_norm(hid[tok], res[tok], f(gamma_attn), eps)
    qkv_tok = qkv_parallel(x1, f(w_q), f(w_k), f(w_v), nq, nkv, hd, t)
    if rows is None:
        qkv = qkv_tok
        attn = attention_core(qkv, nq, nkv, hd, t, cu)
    else:
        qkv = np.zeros((t, T, qkv_tok.shape[2]))
        qkv[:, tok] = qkv_tok
        attn = attention_rows(qkv, nq, nkv, hd, t, cu, rows)
        r1 = r1[np.searchsorted(tok, rows)]
    attn_out = o_proj_parallel(attn, f(w_o), t)
    x2, r2 = add_rms_norm(attn_out, r1, f(gamma_mlp), eps)
    mlp_out = mlp_block(x2, f(w_gate), f(w_up), f(w_down))
    return {"residual_attn": r1, "qkv": qkv, "attn": attn, "attn_out": attn_out,
            "residual_mlp": r2, "mlp_out": mlp_out, "residual_stream": mlp_out + r2}
