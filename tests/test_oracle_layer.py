"""Pins of the decoder-layer oracle (CPU only).

The chain is checked against a tiny layer written out as explicit loops over
the UNSHARDED weights (so the head split, the o_proj reduction and the order
of the adds and norms are all checked at once), against special weights that
switch one half of the layer off, for t invariance (kv heads split and
replicated) and for the first-layer form with no incoming residual. Planted
mistakes in the chain's steps must fail the brute-force pin.
"""
import importlib
import math

import numpy as np
import pytest

import oracle
dl = importlib.import_module("oracle.decoder_layer")   # the module (the package exports its function)

EPS = 1e-5


def _norm_loops(r, g):
    T, H = r.shape
    x = np.zeros_like(r)
    for i in range(T):
        ms = sum(r[i, j] * r[i, j] for j in range(H)) / H
        for j in range(H):
            x[i, j] = r[i, j] / math.sqrt(ms + EPS) * g[j]
    return x


def _matmul_loops(X, W):            # X [T, k], W [n, k] -> X W^T
    T, k = X.shape
    n = W.shape[0]
    Y = np.zeros((T, n))
    for i in range(T):
        for o in range(n):
            Y[i, o] = sum(X[i, c] * W[o, c] for c in range(k))
    return Y


def _layer_loops(p, nq, nkv, hd, cu, residual=True):
    """The whole layer with per-element loops and unsharded weights."""
    hid = p["hidden"]
    r1 = hid + p["residual"] if residual else hid.copy()
    x1 = _norm_loops(r1, p["ga"])
    q = _matmul_loops(x1, p["wq"])
    k = _matmul_loops(x1, p["wk"])
    v = _matmul_loops(x1, p["wv"])
    T = hid.shape[0]
    group = nq // nkv
    A = np.zeros((T, nq * hd))
    for h in range(nq):
        g = next(g for g in range(nkv) if g * group <= h < (g + 1) * group)
        for s in range(len(cu) - 1):
            for i in range(cu[s], cu[s + 1]):
                sc = [sum(q[i, h * hd + d] * k[j, g * hd + d] for d in range(hd)) / math.sqrt(hd)
                      for j in range(cu[s], i + 1)]
                m = max(sc)
                e = [math.exp(z - m) for z in sc]
                tot = sum(e)
                for d in range(hd):
                    A[i, h * hd + d] = sum(e[jj] * v[j, g * hd + d] for jj, j in enumerate(range(cu[s], i + 1))) / tot
    attn_out = _matmul_loops(A, p["wo"])
    r2 = attn_out + r1
    x2 = _norm_loops(r2, p["gm"])
    gt = _matmul_loops(x2, p["wg"])
    up = _matmul_loops(x2, p["wu"])
    hmid = np.zeros_like(gt)
    for i in range(T):
        for c in range(gt.shape[1]):
            hmid[i, c] = gt[i, c] / (1.0 + math.exp(-gt[i, c])) * up[i, c]
    mlp_out = _matmul_loops(hmid, p["wd"])
    return {"residual_attn": r1, "attn_full": A, "attn_out": attn_out, "residual_mlp": r2,
            "mlp_out": mlp_out, "residual_stream": mlp_out + r2}


def _params(H, I, nq, nkv, hd, T, seed):
    rng = np.random.default_rng(seed)
    n = rng.standard_normal
    return {"hidden": n((T, H)), "residual": n((T, H)), "ga": rng.uniform(0.5, 1.5, H),
            "wq": n((nq * hd, H)) * 0.5, "wk": n((nkv * hd, H)) * 0.5, "wv": n((nkv * hd, H)),
            "wo": n((H, nq * hd)) * 0.5, "gm": rng.uniform(0.5, 1.5, H),
            "wg": n((I, H)) * 0.5, "wu": n((I, H)) * 0.5, "wd": n((H, I)) * 0.5}


def _oracle(p, nq, nkv, hd, t, cu, residual=True):
    return oracle.decoder_layer(p["hidden"], p["residual"] if residual else None, p["ga"], p["wq"], p["wk"],
                                p["wv"], p["wo"], p["gm"], p["wg"], p["wu"], p["wd"], nq, nkv, hd, t, cu, EPS)


NQ, NKV, HD, H, I = 4, 2, 2, 8, 8
CU = [0, 3, 5]
KEYS = ("residual_attn", "attn_out", "residual_mlp", "mlp_out", "residual_stream")


@pytest.mark.parametrize("t", [1, 2, 4])      # t = 4 > nkv: each kv head held by two shards
def test_layer_matches_loops(t):
    p = _params(H, I, NQ, NKV, HD, CU[-1], 7)
    want = _layer_loops(p, NQ, NKV, HD, CU)
    got = _oracle(p, NQ, NKV, HD, t, CU)
    for k in KEYS:
        np.testing.assert_allclose(got[k], want[k], rtol=1e-11, atol=1e-11, err_msg=k)
    np.testing.assert_allclose(np.concatenate(list(got["attn"]), axis=1), want["attn_full"], rtol=1e-11, atol=1e-11)


def test_first_layer_without_residual():
    p = _params(H, I, NQ, NKV, HD, CU[-1], 8)
    want = _layer_loops(p, NQ, NKV, HD, CU, residual=False)
    got = _oracle(p, NQ, NKV, HD, 2, CU, residual=False)
    for k in KEYS:
        np.testing.assert_allclose(got[k], want[k], rtol=1e-11, atol=1e-11, err_msg=k)
    zero = dict(p, residual=np.zeros_like(p["residual"]))
    z = _oracle(zero, NQ, NKV, HD, 2, CU)
    for k in KEYS:
        np.testing.assert_array_equal(z[k], got[k])


def test_zero_o_proj_leaves_the_mlp_on_the_residual():
    p = _params(H, I, NQ, NKV, HD, CU[-1], 9)
    p["wo"][:] = 0.0
    got = _oracle(p, NQ, NKV, HD, 2, CU)
    r1 = p["hidden"] + p["residual"]
    np.testing.assert_array_equal(got["attn_out"], 0.0)
    np.testing.assert_array_equal(got["residual_mlp"], r1)
    mlp = oracle.mlp_layer(np.zeros_like(r1), p["wg"], p["wu"], p["wd"], residual=r1, gamma=p["gm"], eps=EPS, norm=True)
    np.testing.assert_allclose(got["residual_stream"], mlp["residual_stream"], rtol=1e-13, atol=1e-13)


def test_zero_gate_leaves_the_stream_after_attention():
    p = _params(H, I, NQ, NKV, HD, CU[-1], 10)
    p["wg"][:] = 0.0
    got = _oracle(p, NQ, NKV, HD, 2, CU)
    np.testing.assert_array_equal(got["mlp_out"], 0.0)
    np.testing.assert_array_equal(got["residual_stream"], got["residual_mlp"])


def test_layer_output_is_independent_of_t_at_a_larger_size():
    nq, nkv, hd, H_, I_ = 8, 4, 8, 32, 64
    cu = [0, 20, 21, 40]
    p = _params(H_, I_, nq, nkv, hd, cu[-1], 11)
    base = _oracle(p, nq, nkv, hd, 1, cu)
    for t in (2, 4, 8):
        got = _oracle(p, nq, nkv, hd, t, cu)
        for k in KEYS:
            np.testing.assert_allclose(got[k], base[k], rtol=1e-10, atol=1e-10, err_msg=f"{k} t={t}")


# ------------------------------------------------------------------ planted mistakes

def _pin_passes() -> bool:
    try:
        for t in (2, 4):
            test_layer_matches_loops(t)
    except AssertionError:
        return False
    return True


def test_pin_passes_unmodified():
    assert _pin_passes()


_orig = {k: getattr(dl, k) for k in ("add_rms_norm", "attention_core", "mlp_block", "o_proj_parallel")}


@pytest.mark.parametrize("name,bad", [
    # the residual handed on is the un-added input, not r = a + residual
    ("add_rms_norm", lambda a, res, g, eps: (_orig["add_rms_norm"](a, res, g, eps)[0], a)),
    # every sequence's queries see the whole batch (offsets dropped)
    ("attention_core", lambda qkv, nq, nkv, hd, t, cu: _orig["attention_core"](qkv, nq, nkv, hd, t, [0, cu[-1]])),
    # gate and up exchanged
    ("mlp_block", lambda x, wg, wu, wd: _orig["mlp_block"](x, wu, wg, wd)),
    # the shard partials are not all summed
    ("o_proj_parallel", lambda A, wo, t: _orig["o_proj_parallel"](A, wo, t) * (1.0 if t == 1 else 0.5)),
])
def test_planted_mistake_is_caught(monkeypatch, name, bad):
    monkeypatch.setattr(dl, name, bad)
    assert not _pin_passes()


def test_rows_subset_matches_the_full_layer():
    nq, nkv, hd, H_, I_ = 8, 4, 8, 32, 64
    cu = [0, 20, 21, 40]
    p = _params(H_, I_, nq, nkv, hd, cu[-1], 12)
    full = _oracle(p, nq, nkv, hd, 2, cu)
    rows = [39, 0, 20, 21, 5]
    sub = oracle.decoder_layer(p["hidden"], p["residual"], p["ga"], p["wq"], p["wk"], p["wv"], p["wo"], p["gm"],
                               p["wg"], p["wu"], p["wd"], nq, nkv, hd, 2, cu, EPS, rows=rows)
    for k in KEYS:
        np.testing.assert_allclose(sub[k], full[k][rows], rtol=1e-12, atol=1e-12, err_msg=k)
