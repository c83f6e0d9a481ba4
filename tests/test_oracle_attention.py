"""Pins of the attention-core oracle (CPU only).

The oracle is checked against things it does not compute the same way:
explicit-loop brute force on tiny inputs, closed forms (a zero query
averages the visible values; a one-token sequence returns its own value;
one dominant key selects its value), invariants (sequence packing, a shift
of every key by one vector) and a GQA layout check in which every kv head
carries a distinct constant value. Planted mistakes (wrong kv head, a mask
that lets a query see one key ahead, a softmax without its normaliser, an
unscaled score) must each fail at least one pin.
"""
import math

import numpy as np
import pytest

import oracle
import oracle.attention as att
from oracle.tp_block import gqa_partition


def _layout(nq, nkv, hd, t):
    q_per, kv_per, rep = gqa_partition(nq, nkv, t)
    return q_per, kv_per, rep, (q_per + 2 * kv_per) * hd


def _brute(qkv, nq, nkv, hd, t, cu, scale=None):
    """Per-element loops: for every query, weights exp(score) over the visible keys."""
    q_per, kv_per, rep, ws = _layout(nq, nkv, hd, t)
    group = nq // nkv
    sc = 1.0 / math.sqrt(hd) if scale is None else scale
    T = qkv.shape[1]
    out = np.zeros((t, T, q_per * hd))
    for r in range(t):
        held = [r // rep] if rep > 1 else list(range(r * kv_per, (r + 1) * kv_per))
        for i in range(q_per):
            h = r * q_per + i
            # the kv head whose block of `group` consecutive q heads contains h
            G = next(g for g in range(nkv) if g * group <= h < (g + 1) * group)
            loc = held.index(G)
            for s in range(len(cu) - 1):
                for row in range(cu[s], cu[s + 1]):
                    w = []
                    for j in range(cu[s], row + 1):
                        dot = sum(qkv[r, row, i * hd + d] * qkv[r, j, q_per * hd + loc * hd + d] for d in range(hd))
                        w.append(dot * sc)
                    mx = max(w)
                    e = [math.exp(x - mx) for x in w]
                    tot = sum(e)
                    for d in range(hd):
                        acc = 0.0
                        for jj, j in enumerate(range(cu[s], row + 1)):
                            acc += e[jj] * qkv[r, j, (q_per + kv_per) * hd + loc * hd + d]
                        out[r, row, i * hd + d] = acc / tot
    return out


CASES = [  # nq, nkv, hd, t, cu_seqlens
    (4, 2, 4, 2, [0, 3, 5]),        # two sequences, kv heads split
    (4, 2, 3, 4, [0, 2, 2, 6]),     # t > nkv: kv head replicated; an empty sequence
    (6, 3, 2, 1, [0, 4]),           # t = 1, three groups of two q heads
    (8, 8, 2, 2, [0, 1, 3, 4]),     # MHA (group of one), a one-token sequence
]


@pytest.mark.parametrize("nq,nkv,hd,t,cu", CASES)
def test_matches_brute_force(nq, nkv, hd, t, cu):
    rng = np.random.default_rng(nq * 100 + t)
    ws = _layout(nq, nkv, hd, t)[3]
    qkv = rng.standard_normal((t, cu[-1], ws))
    got = oracle.attention_core(qkv, nq, nkv, hd, t, cu)
    np.testing.assert_allclose(got, _brute(qkv, nq, nkv, hd, t, cu), rtol=1e-12, atol=1e-12)
    rows = list(range(cu[-1]))[::-1]
    np.testing.assert_allclose(oracle.attention_rows(qkv, nq, nkv, hd, t, cu, rows), got[:, rows], rtol=1e-12, atol=1e-12)


def test_zero_query_averages_visible_values():
    nq, nkv, hd, t, cu = 4, 2, 8, 2, [0, 5, 9]
    q_per, kv_per, _, ws = _layout(nq, nkv, hd, t)
    rng = np.random.default_rng(1)
    qkv = rng.standard_normal((t, 9, ws))
    qkv[:, :, :q_per * hd] = 0.0
    got = oracle.attention_core(qkv, nq, nkv, hd, t, cu)
    for r in range(t):
        for i in range(q_per):
            g = i // (nq // nkv)
            v = qkv[r, :, (q_per + kv_per) * hd + g * hd:(q_per + kv_per) * hd + (g + 1) * hd]
            for s in range(len(cu) - 1):
                lo, hi = cu[s], cu[s + 1]
                cum = np.cumsum(v[lo:hi], axis=0) / np.arange(1, hi - lo + 1)[:, None]
                np.testing.assert_allclose(got[r, lo:hi, i * hd:(i + 1) * hd], cum, rtol=1e-13, atol=1e-13)


def test_one_token_sequences_return_their_value():
    nq, nkv, hd, t = 8, 2, 4, 4
    q_per, kv_per, _, ws = _layout(nq, nkv, hd, t)
    qkv = np.random.default_rng(2).standard_normal((t, 6, ws))
    got = oracle.attention_core(qkv, nq, nkv, hd, t, list(range(7)))
    v = qkv[:, :, (q_per + kv_per) * hd:]          # one kv head per shard here (t = 4 > nkv)
    for i in range(q_per):
        np.testing.assert_allclose(got[:, :, i * hd:(i + 1) * hd], v, rtol=0, atol=1e-15)


def test_dominant_key_selects_its_value():
    nq, nkv, hd, t, n = 2, 1, 8, 1, 8
    q_per, kv_per, _, ws = _layout(nq, nkv, hd, t)
    rng = np.random.default_rng(3)
    qkv = np.zeros((t, n, ws))
    target = [0, 0, 1, 2, 2, 4, 3, 6]              # query i picks a key j <= i
    for j in range(n):
        qkv[0, j, q_per * hd + j] = 1.0             # key j = e_j
    for i in range(n):
        qkv[0, i, target[i]] = 200.0                # head 0 query: 200 e_target
        qkv[0, i, hd + (i % hd)] = 200.0            # head 1 query: its own key (i <= i)
    qkv[0, :, (q_per + kv_per) * hd:] = rng.standard_normal((n, hd))
    got = oracle.attention_core(qkv, nq, nkv, hd, t, [0, n])
    v = qkv[0, :, (q_per + kv_per) * hd:]
    np.testing.assert_allclose(got[0, :, :hd], v[target], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[0, :, hd:], v, rtol=0, atol=1e-12)


def test_packing_sequences_does_not_mix_them():
    nq, nkv, hd, t = 4, 2, 4, 2
    ws = _layout(nq, nkv, hd, t)[3]
    rng = np.random.default_rng(4)
    a, b = rng.standard_normal((t, 5, ws)), rng.standard_normal((t, 3, ws))
    packed = oracle.attention_core(np.concatenate([a, b], axis=1), nq, nkv, hd, t, [0, 5, 8])
    np.testing.assert_allclose(packed[:, :5], oracle.attention_core(a, nq, nkv, hd, t, [0, 5]), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(packed[:, 5:], oracle.attention_core(b, nq, nkv, hd, t, [0, 3]), rtol=1e-13, atol=1e-13)


def test_shifting_every_key_by_one_vector_changes_nothing():
    nq, nkv, hd, t, cu = 4, 2, 6, 2, [0, 7]
    q_per, kv_per, _, ws = _layout(nq, nkv, hd, t)
    rng = np.random.default_rng(5)
    qkv = rng.standard_normal((t, 7, ws))
    shifted = qkv.copy()
    shifted[:, :, q_per * hd:(q_per + kv_per) * hd] += np.tile(rng.standard_normal(hd), kv_per)
    np.testing.assert_allclose(oracle.attention_core(shifted, nq, nkv, hd, t, cu),
                               oracle.attention_core(qkv, nq, nkv, hd, t, cu), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("nq,nkv,t", [(32, 8, 4), (8, 2, 4), (8, 2, 8), (6, 3, 3)])
def test_each_q_head_reads_its_group_kv_head(nq, nkv, t):
    # every kv head carries a constant value row (its global index + 1), so any
    # weights give that constant; q head h must return kv_head(h) + 1
    hd = 2
    q_per, kv_per, rep, ws = _layout(nq, nkv, hd, t)
    rng = np.random.default_rng(6)
    qkv = rng.standard_normal((t, 5, ws))
    for r in range(t):
        held = [r // rep] if rep > 1 else list(range(r * kv_per, (r + 1) * kv_per))
        for loc, G in enumerate(held):
            qkv[r, :, (q_per + kv_per) * hd + loc * hd:(q_per + kv_per) * hd + (loc + 1) * hd] = G + 1.0
    got = oracle.attention_core(qkv, nq, nkv, hd, t, [0, 5])
    for r in range(t):
        for i in range(q_per):
            h = r * q_per + i
            want = h * nkv // nq + 1.0                # contiguous groups of nq / nkv q heads
            np.testing.assert_allclose(got[r, :, i * hd:(i + 1) * hd], want, rtol=0, atol=1e-13)


def test_rejects_bad_offsets():
    qkv = np.zeros((1, 4, 12))
    with pytest.raises(ValueError):
        oracle.attention_core(qkv, 2, 1, 3, 1, [0, 3])       # does not end at T
    with pytest.raises(ValueError):
        oracle.attention_core(qkv, 2, 1, 3, 1, [0, 3, 2, 4])  # falls


# ------------------------------------------------------------------ planted mistakes

def _pins_pass() -> bool:
    try:
        test_matches_brute_force(*CASES[0])
        test_matches_brute_force(*CASES[1])
        test_zero_query_averages_visible_values()
        test_dominant_key_selects_its_value()
        for c in [(32, 8, 4), (8, 2, 8)]:
            test_each_q_head_reads_its_group_kv_head(*c)
    except (AssertionError, ValueError, IndexError):   # a wrong value, or a head layout that breaks
        return False
    return True


def test_pins_pass_unmodified():
    assert _pins_pass()


@pytest.mark.parametrize("name,bad", [
    ("kv_head_of", lambda h, nq, nkv: h % nkv),
    ("causal_mask", lambda n: np.tril(np.ones((n, n), dtype=bool), k=1)),
    ("softmax_rows", lambda s: np.exp(s - np.max(s, axis=1, keepdims=True))),
])
def test_planted_mistake_is_caught(monkeypatch, name, bad):
    monkeypatch.setattr(att, name, bad)
    assert not _pins_pass()


def test_unscaled_scores_are_caught():
    nq, nkv, hd, t, cu = CASES[0]
    ws = _layout(nq, nkv, hd, t)[3]
    qkv = np.random.default_rng(400 + t).standard_normal((t, cu[-1], ws))
    bad = oracle.attention_core(qkv, nq, nkv, hd, t, cu, scale=1.0)
    assert np.abs(bad - _brute(qkv, nq, nkv, hd, t, cu)).max() > 1e-3
