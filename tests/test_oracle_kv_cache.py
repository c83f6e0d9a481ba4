"""Pins of the paged KV-cache oracle (CPU only).

The cache is filled through slot mappings taken from random, scattered block
tables; attention over the cache must then equal the contiguous attention core
(a separate code path) on the same rows. Also: the write lands every token's
k and v in its slot and nowhere else, padding slots write nothing, and planted
mistakes (a wrong slot formula, a position one off, a wrong kv head) fail.
"""
import importlib

import numpy as np
import pytest

import oracle
from oracle.tp_block import gqa_partition

kvc = importlib.import_module("oracle.kv_cache")
att = importlib.import_module("oracle.attention")


def _setup(nq, nkv, hd, t, lens, new, bs, seed):
    """Full sequences of the given lengths; the last `new[b]` tokens of request b are new."""
    rng = np.random.default_rng(seed)
    q_per, kv_per, _ = gqa_partition(nq, nkv, t)
    ws = (q_per + 2 * kv_per) * hd
    full = [rng.standard_normal((t, L, ws)) for L in lens]
    n_blocks = sum(-(-L // bs) for L in lens) + 3
    perm = rng.permutation(n_blocks)                      # scattered blocks
    tables, used = [], 0
    for L in lens:
        nb = -(-L // bs)
        tables.append(list(perm[used:used + nb]) + [0] * 4)
        used += nb
    cache_k = np.zeros((t, n_blocks, bs, kv_per, hd))
    cache_v = np.zeros_like(cache_k)
    # write every token of every request through its slot mapping
    for b, L in enumerate(lens):
        slots = [int(tables[b][p // bs]) * bs + p % bs for p in range(L)]   # independent of slot_of
        oracle.kv_cache_write(full[b], slots, cache_k, cache_v, nq, nkv, hd, t, bs)
    qkv_new = np.concatenate([f[:, L - n:] for f, L, n in zip(full, lens, new)], axis=1)
    qsl = np.concatenate([[0], np.cumsum(new)])
    return full, tables, cache_k, cache_v, qkv_new, qsl


CASES = [  # nq, nkv, hd, t, lens, new, block_size
    (4, 2, 4, 2, [5, 9, 1], [1, 1, 1], 4),        # decode: one new token each
    (8, 2, 3, 4, [7, 12], [3, 12], 2),            # t > nkv; a chunk and a whole prefill
    (6, 3, 2, 1, [16], [5], 16),                  # one block
]


@pytest.mark.parametrize("nq,nkv,hd,t,lens,new,bs", CASES)
def test_paged_equals_contiguous_attention(nq, nkv, hd, t, lens, new, bs):
    full, tables, ck, cv, qkv_new, qsl = _setup(nq, nkv, hd, t, lens, new, bs, seed=len(lens) + t)
    got = oracle.paged_attention(qkv_new, qsl, lens, tables, ck, cv, nq, nkv, hd, t, bs)
    cat = np.concatenate(full, axis=1)
    cu = np.concatenate([[0], np.cumsum(lens)])
    rows = [int(cu[b] + L - n + j) for b, (L, n) in enumerate(zip(lens, new)) for j in range(n)]
    want = oracle.attention_rows(cat, nq, nkv, hd, t, cu, rows)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_write_lands_in_its_slot_only():
    nq, nkv, hd, t, bs = 4, 2, 3, 2, 4
    q_per, kv_per, _ = gqa_partition(nq, nkv, t)
    rng = np.random.default_rng(7)
    qkv = rng.standard_normal((t, 6, (q_per + 2 * kv_per) * hd))
    slots = [13, -1, 0, 7, -1, 22]
    ck = np.full((t, 6, bs, kv_per, hd), 5.0)
    cv = np.full_like(ck, 5.0)
    oracle.kv_cache_write(qkv, slots, ck, cv, nq, nkv, hd, t, bs)
    touched = np.zeros((6, bs), dtype=bool)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        touched[s // bs, s % bs] = True
        for r in range(t):
            for g in range(kv_per):
                np.testing.assert_array_equal(ck[r, s // bs, s % bs, g], qkv[r, i, (q_per + g) * hd:(q_per + g + 1) * hd])
                np.testing.assert_array_equal(cv[r, s // bs, s % bs, g],
                                              qkv[r, i, (q_per + kv_per + g) * hd:(q_per + kv_per + g + 1) * hd])
    assert np.all(ck[:, ~touched] == 5.0) and np.all(cv[:, ~touched] == 5.0)


def _pin_passes() -> bool:
    try:
        for c in CASES[:2]:
            test_paged_equals_contiguous_attention(*c)
    except (AssertionError, IndexError, ValueError):
        return False
    return True


def test_pin_passes_unmodified():
    assert _pin_passes()


_slot = kvc.slot_of


@pytest.mark.parametrize("name,bad", [
    ("slot_of", lambda tb, b, pos, bs: int(tb[b][pos % bs]) * bs + pos // bs),      # block and offset exchanged
    ("slot_of", lambda tb, b, pos, bs: _slot(tb, b, max(pos - 1, 0), bs)),         # one position early
    ("kv_head_of", lambda h, nq, nkv: h % nkv),                                     # wrong kv head
])
def test_planted_mistake_is_caught(monkeypatch, name, bad):
    # the cache is filled by the test's own slot formula; the mistake is on the reading side
    monkeypatch.setattr(kvc, name, bad)
    assert not _pin_passes()
