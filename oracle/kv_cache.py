"""Paged KV cache: the cache write and attention over cached keys (test infrastructure only).

"vLLM Code Reading (Section 5)", §13: each rank's attention kernel writes the KV
cache of the heads it holds; the model runner's _get_slot_mappings turns the
block table into the slot every new token's keys and values go to. The pages
give no layout, so these are the plain readings:

* The cache of shard r holds its kv heads: cache_k[r], cache_v[r] are
  [num_blocks][block_size][kv_per][hd]; slot s is block s // block_size,
  offset s % block_size. A negative slot writes nothing (a padding token).
* Request b's token at position p lives in slot
  block_tables[b][p // block_size] * block_size + p % block_size.
* The new tokens of request b are rows [qsl[b], qsl[b+1]) of qkv and occupy the
  last positions of its seq_lens[b] tokens; a new token at position p attends
  to the request's positions 0..p (causal), read from the cache, which must
  already hold the new tokens' own keys and values (write first, then attend).

``paged_attention`` computes exactly what ``attention_core`` computes for the
same rows of the contiguous sequence, which is how it is pinned
(``tests/test_oracle_kv_cache.py``).
"""
from __future__ import annotations

import numpy as np

from .attention import _as_f64, first_kv_head, kv_head_of, softmax_rows
from .tp_block import gqa_partition


def kv_cache_write(qkv, slot_mapping, cache_k, cache_v, nq: int, nkv: int, hd: int, t: int, block_size: int):
    """Copy every token's k and v heads of every shard into its slot (in place, float64 caches)."""
    a = _as_f64(qkv)
    q_per, kv_per, _ = gqa_partition(nq, nkv, t)
    k0, v0 = q_per * hd, (q_per + kv_per) * hd
    for i, s in enumerate(np.asarray(slot_mapping, np.int64)):
        if s < 0:
            continue
        blk, off = divmod(int(s), block_size)
        for r in range(t):
            cache_k[r, blk, off] = a[r, i, k0:k0 + kv_per * hd].reshape(kv_per, hd)
            cache_v[r, blk, off] = a[r, i, v0:v0 + kv_per * hd].reshape(kv_per, hd)


def slot_of(block_tables, b: int, pos: int, block_size: int) -> int:
    """Cache slot of request b's token at position pos."""
    return int(block_tables[b][pos // block_size]) * block_size + pos % block_size


def paged_attention(qkv, query_start_loc, seq_lens, block_tables, cache_k, cache_v, nq: int, nkv: int, hd: int,
                    t: int, block_size: int, scale: float | None = None) -> np.ndarray:
    """Attention of the new tokens over their requests' cached keys: [t, T, q_per * hd] (float64)."""
    a = _as_f64(qkv)
    ck, cv = _as_f64(cache_k), _as_f64(cache_v)
    q_per, kv_per, _ = gqa_partition(nq, nkv, t)
    T = a.shape[1]
    qsl = [int(c) for c in query_start_loc]
    sc = 1.0 / np.sqrt(hd) if scale is None else float(scale)
    out = np.zeros((t, T, q_per * hd))
    for b in range(len(qsl) - 1):
        n_new = qsl[b + 1] - qsl[b]
        L = int(seq_lens[b])
        if n_new > L:
            raise ValueError("a request has more new tokens than tokens")
        for i in range(qsl[b], qsl[b + 1]):
            p = L - n_new + (i - qsl[b])
            slots = [slot_of(block_tables, b, j, block_size) for j in range(p + 1)]
            blk = np.array([s // block_size for s in slots])
            off = np.array([s % block_size for s in slots])
            for r in range(t):
                base = first_kv_head(r, nq, nkv, t)
                for h in range(q_per):
                    g = kv_head_of(r * q_per + h, nq, nkv) - base
                    q = a[r, i, h * hd:(h + 1) * hd]
                    k = ck[r, blk, off, g]                   # [p + 1, hd]
                    v = cv[r, blk, off, g]
                    w = softmax_rows(((k @ q) * sc)[None, :])[0]
                    out[r, i, h * hd:(h + 1) * hd] = w @ v
    return out
