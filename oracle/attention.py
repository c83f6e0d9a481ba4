"""Float64 causal GQA attention over each shard's local heads (test infrastructure only).

The attention core sits between the column-parallel QKV projection and the
row-parallel o_proj. [VCR] section 13 ("Attention 中的 TP 通信") describes it
as each rank running attention on the q/k/v heads it holds; [VSC]
"QkvParallelLinear" fixes which kv heads a shard holds under GQA. The pages
print no attention formula, so this module takes the textbook one, in the
pages' layout:

* scaled dot-product attention: P = softmax(q k^T / sqrt(hd)) over keys,
  out = P v;
* causal within a sequence: query i sees the keys j <= i of its own
  sequence; sequences are packed along the token axis and delimited by
  ``cu_seqlens`` (offsets, first 0, last T);
* q head h reads kv head h // (nq / nkv) (a group of nq / nkv q heads
  shares one kv head);
* q and k are used as the projection produced them: the pages define no
  positional rotation.

Input: the QKV projection's output, [t, T, w_s] with shard r holding
[its q heads | its k heads | its v heads], hd columns per head. Output:
[t, T, q_per * hd], shard r holding its q heads in order, which is the
layout the row-parallel o_proj reads.

Each step is a small function of its own (the kv head of a q head, the
causal mask, the row softmax) so that a test can replace one of them with a
planted mistake and see the pins catch it.
"""
from __future__ import annotations

import numpy as np

from .tp_block import bf16_to_f64, divide, gqa_partition


def _as_f64(x) -> np.ndarray:
    """A torch bf16 tensor, raw bf16 bits (uint16) or a float array -> float64."""
    if isinstance(x, np.ndarray):
        return bf16_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64, copy=False)
    return bf16_to_f64(x)


def kv_head_of(h: int, nq: int, nkv: int) -> int:
    """Global kv head read by global q head h: h // (nq / nkv)."""
    return h // divide(nq, nkv)


def first_kv_head(r: int, nq: int, nkv: int, t: int) -> int:
    """Global index of the first kv head shard r holds ([VSC] QkvParallelLinear:
    split heads r*kv_per.., or the replicated head r // replicas)."""
    _, kv_per, rep = gqa_partition(nq, nkv, t)
    return r // rep if rep > 1 else r * kv_per


def causal_mask(n: int) -> np.ndarray:
    """[n, n] boolean, True where query i may see key j (j <= i)."""
    return np.tril(np.ones((n, n), dtype=bool))


def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row-wise softmax; -inf entries get weight 0 (every row has a finite entry)."""
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=1, keepdims=True)


def attention_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Causal attention of one head over one sequence: q, k, v [n, hd] -> [n, hd]."""
    s = (q @ k.T) * scale
    s = np.where(causal_mask(q.shape[0]), s, -np.inf)
    return softmax_rows(s) @ v


def attention_core(qkv, nq: int, nkv: int, hd: int, t: int, cu_seqlens, scale: float | None = None) -> np.ndarray:
    """Attention over the local heads of every shard: [t, T, w_s] -> [t, T, q_per * hd] (float64)."""
    a = _as_f64(qkv)
    q_per, kv_per, _ = gqa_partition(nq, nkv, t)
    T = a.shape[1]
    if a.shape != (t, T, (q_per + 2 * kv_per) * hd):
        raise ValueError(f"qkv shape {a.shape} does not match the head layout")
    cu = [int(c) for c in cu_seqlens]
    if cu[0] != 0 or cu[-1] != T or any(cu[i] > cu[i + 1] for i in range(len(cu) - 1)):
        raise ValueError("cu_seqlens must rise from 0 to T")
    sc = 1.0 / np.sqrt(hd) if scale is None else float(scale)
    out = np.zeros((t, T, q_per * hd))
    for r in range(t):
        k0 = q_per * hd
        v0 = (q_per + kv_per) * hd
        base = first_kv_head(r, nq, nkv, t)
        for i in range(q_per):
            g = kv_head_of(r * q_per + i, nq, nkv) - base
            q = a[r, :, i * hd:(i + 1) * hd]
            k = a[r, :, k0 + g * hd:k0 + (g + 1) * hd]
            v = a[r, :, v0 + g * hd:v0 + (g + 1) * hd]
            for s in range(len(cu) - 1):
                lo, hi = cu[s], cu[s + 1]
                if hi > lo:
                    out[r, lo:hi, i * hd:(i + 1) * hd] = attention_head(q[lo:hi], k[lo:hi], v[lo:hi], sc)
    return out


def attention_rows(qkv, nq: int, nkv: int, hd: int, t: int, cu_seqlens, rows, scale: float | None = None) -> np.ndarray:
    """attention_core restricted to the given token rows (any order): [t, len(rows), q_per * hd].

    Row i needs only the keys of its own sequence up to i, so sampled rows of
    a long sequence cost O(i) each instead of the whole square.
    """
    a = _as_f64(qkv)
    q_per, kv_per, _ = gqa_partition(nq, nkv, t)
    cu = np.asarray([int(c) for c in cu_seqlens])
    sc = 1.0 / np.sqrt(hd) if scale is None else float(scale)
    out = np.zeros((t, len(rows), q_per * hd))
    for n, row in enumerate(rows):
        s = int(np.searchsorted(cu, row, side="right")) - 1
        lo = int(cu[s])
        for r in range(t):
            k0, v0 = q_per * hd, (q_per + kv_per) * hd
            base = first_kv_head(r, nq, nkv, t)
            for i in range(q_per):
                g = kv_head_of(r * q_per + i, nq, nkv) - base
                q = a[r, row, i * hd:(i + 1) * hd]
                k = a[r, lo:row + 1, k0 + g * hd:k0 + (g + 1) * hd]
                v = a[r, lo:row + 1, v0 + g * hd:v0 + (g + 1) * hd]
                p = softmax_rows(((k @ q) * sc)[None, :])[0]
                out[r, n, i * hd:(i + 1) * hd] = p @ v
    return out
