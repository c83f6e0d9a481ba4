"""Pins of the float64 oracle against facts that do not come from the oracle itself.

Each test checks one function against brute force, a closed form, an
algebraic identity the pages state, a library routine, or head counts the
pages print (``tests/golden/``). ``test_planted_mistakes_are_caught`` plants
plausible mistakes in copies of the oracle's functions and checks that the
pins notice them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def rand(*shape):
    return rng.standard_normal(shape)


# --------------------------------------------------------------------------- bf16 conversion

def test_bf16_to_f64_known_bits():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F7F, 0x0001], dtype=np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 0.0, -0.0, (2 - 2 ** -7) * 2.0 ** 127, 2.0 ** -133]
    got = oracle.bf16_to_f64(bits)
    assert list(got) == want
    # the torch-tensor path (a library widening) gives the same values, subnormals included
    tb = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    assert list(oracle.bf16_to_f64(tb)) == want
    t = torch.randn(1000).to(torch.bfloat16)
    t_bits = t.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_to_f64(t), oracle.bf16_to_f64(t_bits))


# --------------------------------------------------------------------------- linear and the split algebra

@pytest.mark.parametrize("b,k,n", [(1, 1, 1), (3, 5, 4), (4, 16, 32)])
def test_linear_brute_force(b, k, n):
    X, W = rand(b, k), rand(n, k)
    Y = np.zeros((b, n))
    for i in range(b):
        for j in range(n):
            s = 0.0
            for kk in range(k):
                s += X[i, kk] * W[j, kk]
            Y[i, j] = s
    np.testing.assert_allclose(oracle.linear(X, W), Y, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_column_shards_concatenate_to_unsharded(t):
    # "Yi = X Ai ... each rank holds n/t columns of Y": concat of shards == Y
    X, W = rand(7, 24), rand(32, 24)
    ys = oracle.column_parallel(X, W, t)
    assert all(y.shape == (7, 32 // t) for y in ys)
    np.testing.assert_allclose(np.concatenate(ys, axis=1), X @ W.T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_row_partials_sum_to_unsharded(t):
    # "Yi = Xi Ai, Y = sum_i Yi"
    X, W = rand(5, 32), rand(12, 32)
    parts = oracle.row_parallel(X, W, t)
    assert len(parts) == t and all(p.shape == (5, 12) for p in parts)
    np.testing.assert_allclose(sum(parts), X @ W.T, rtol=1e-12, atol=1e-12)
    if t > 1:   # a single shard is not the whole answer
        assert not np.allclose(parts[0], X @ W.T)


@pytest.mark.parametrize("T,t", [(8, 4), (10, 4), (3, 8), (5, 1)])
def test_reduce_scatter_slices_the_reduced_rows(T, t):
    # each rank keeps its own token rows of the sum; together (padding removed) they
    # are the all-reduce result, written here as explicit loops over tokens and shards
    X, W = rand(T, 16), rand(6, 16)
    parts = oracle.row_parallel(X, W, 2)
    sl = oracle.reduce_scatter(parts, t)
    per = -(-T // t)
    assert len(sl) == t and all(s.shape == (per, 6) for s in sl)
    for r in range(t):
        for i in range(per):
            tok = r * per + i
            want = [0.0] * 6 if tok >= T else [sum(X[tok, c] * W[o, c] for c in range(16)) for o in range(6)]
            np.testing.assert_allclose(sl[r][i], want, rtol=1e-12, atol=1e-12)


def test_divide_rejects_remainder():
    assert oracle.divide(1408, 2) == 704
    with pytest.raises(ValueError):
        oracle.divide(1408, 3)
    with pytest.raises(ValueError):
        oracle.column_parallel(rand(2, 4), rand(6, 4), 4)


# --------------------------------------------------------------------------- SiLU

def test_silu_closed_forms():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    ln3 = math.log(3.0)                       # sigmoid(ln 3) = 3/4
    np.testing.assert_allclose(oracle.silu(np.array([ln3, -ln3])), [0.75 * ln3, -0.25 * ln3], rtol=1e-15)
    big = oracle.silu(np.array([40.0, -40.0, 800.0, -800.0]))
    assert big[0] == pytest.approx(40.0, rel=1e-15) and big[2] == 800.0
    assert abs(big[1]) < 1e-15 and big[3] == 0.0 and np.all(np.isfinite(big))
    # derivative at 0 is sigmoid(0) = 1/2
    h = 1e-6
    d = (oracle.silu(np.array([h]))[0] - oracle.silu(np.array([-h]))[0]) / (2 * h)
    assert d == pytest.approx(0.5, rel=1e-9)


def test_silu_identities():
    z = rand(1000) * 6
    s = oracle.silu(z)
    np.testing.assert_allclose(s - oracle.silu(-z), z, rtol=1e-13, atol=1e-13)     # z*(sig(z)+sig(-z)) = z
    np.testing.assert_allclose(s, 0.5 * z * (1 + np.tanh(0.5 * z)), rtol=1e-13, atol=1e-15)


def test_silu_mul_gate_first():
    ln3 = math.log(3.0)
    g, u = np.array([0.0, ln3]), np.array([5.0, 2.0])
    np.testing.assert_allclose(oracle.silu_mul(g, u), [0.0, 1.5 * ln3], rtol=1e-15)
    np.testing.assert_allclose(oracle.silu_mul(u, g), [0.0, 2 * 0.5 * 2 * (1 + math.tanh(1.0)) / 2 * ln3], rtol=1e-13)


# --------------------------------------------------------------------------- RMSNorm

def test_rms_norm_constant_row():
    H, c, eps = 64, 0.37, 1e-5
    gamma = rng.uniform(0.9, 1.1, H)
    got = oracle.rms_norm(np.full((1, H), c), gamma, eps)
    np.testing.assert_allclose(got[0], gamma * c / math.sqrt(c * c + eps), rtol=1e-14)


def test_rms_norm_one_hot_row():
    H, v, j, eps = 128, 2.5, 17, 1e-5
    gamma = rng.uniform(0.9, 1.1, H)
    r = np.zeros((1, H))
    r[0, j] = v
    got = oracle.rms_norm(r, gamma, eps)[0]
    want = np.zeros(H)
    want[j] = gamma[j] * math.sqrt(H) * v / math.sqrt(v * v + H * eps)
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=0)


def test_rms_norm_matches_torch_library():
    r, gamma = rand(9, 96), rng.uniform(0.9, 1.1, 96)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(r), (96,), torch.from_numpy(gamma), eps=1e-5)
    np.testing.assert_allclose(oracle.rms_norm(r, gamma, 1e-5), ref.numpy(), rtol=1e-13, atol=1e-14)


def test_add_rms_norm_returns_sum_and_norm():
    a, r0, gamma = rand(4, 32), rand(4, 32), rng.uniform(0.9, 1.1, 32)
    x, r = oracle.add_rms_norm(a, r0, gamma, 1e-5)
    assert np.array_equal(r, a + r0)
    np.testing.assert_allclose(x, oracle.rms_norm(a + r0, gamma, 1e-5), rtol=0, atol=0)
    # scale invariance of the normalisation (eps -> 0)
    np.testing.assert_allclose(oracle.rms_norm(7.0 * r, gamma, 0.0), oracle.rms_norm(r, gamma, 0.0), rtol=1e-13)


# --------------------------------------------------------------------------- MLP block

@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_mlp_block_invariant_across_t(t):
    T, H, I = 6, 16, 32
    x, wg, wu, wd = rand(T, H), rand(I, H) * 0.3, rand(I, H) * 0.3, rand(H, I) * 0.3
    y_ref = oracle.mlp_block(x, wg, wu, wd)
    y, hs = oracle.mlp_block_tp(x, wg, wu, wd, t)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    assert len(hs) == t and all(h.shape == (T, I // t) for h in hs)


def test_mlp_block_brute_force_tiny():
    T, H, I = 2, 3, 4
    x, wg, wu, wd = rand(T, H), rand(I, H), rand(I, H), rand(H, I)
    y = np.zeros((T, H))
    for i in range(T):
        h = []
        for j in range(I):
            g = sum(x[i, k] * wg[j, k] for k in range(H))
            u = sum(x[i, k] * wu[j, k] for k in range(H))
            h.append(0.5 * g * (1 + math.tanh(0.5 * g)) * u)
        for n in range(H):
            y[i, n] = sum(h[j] * wd[n, j] for j in range(I))
    np.testing.assert_allclose(oracle.mlp_block(x, wg, wu, wd), y, rtol=1e-12, atol=1e-12)


def test_mlp_selection_weights():
    # gate row i picks x_{jg[i]}, up row i picks x_{ju[i]}, down row n picks h_{jd[n]}:
    # y[:, n] = silu(x[:, jg[jd[n]]]) * x[:, ju[jd[n]]]
    T, H, I = 5, 8, 6
    x = rand(T, H)
    jg, ju, jd = rng.integers(0, H, I), rng.integers(0, H, I), rng.integers(0, I, H)
    wg, wu, wd = np.zeros((I, H)), np.zeros((I, H)), np.zeros((H, I))
    wg[np.arange(I), jg] = 1.0
    wu[np.arange(I), ju] = 1.0
    wd[np.arange(H), jd] = 1.0
    y = oracle.mlp_block(x, wg, wu, wd)
    g = x[:, jg[jd]]
    want = 0.5 * g * (1 + np.tanh(0.5 * g)) * x[:, ju[jd]]
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-15)


def test_mlp_layer_zero_gate_gives_residual_stream_equal_residual():
    T, H, I = 4, 16, 8
    a, r0, gamma = rand(T, H), rand(T, H), rng.uniform(0.9, 1.1, H)
    out = oracle.mlp_layer(a, np.zeros((I, H)), rand(I, H), rand(H, I), residual=r0, gamma=gamma,
                           norm=True)
    assert np.all(out["mlp_out"] == 0.0)
    assert np.array_equal(out["residual_out"], a + r0)
    assert np.array_equal(out["residual_stream"], a + r0)


def test_mlp_layer_rows_subset_matches_full():
    T, H, I = 9, 16, 8
    a, r0, gamma = rand(T, H), rand(T, H), rng.uniform(0.9, 1.1, H)
    wg, wu, wd = rand(I, H), rand(I, H), rand(H, I)
    full = oracle.mlp_layer(a, wg, wu, wd, residual=r0, gamma=gamma, norm=True)
    rows = [0, 4, 8]
    sub = oracle.mlp_layer(a, wg, wu, wd, residual=r0, gamma=gamma, norm=True, rows=rows)
    for k in ("mlp_out", "residual_out", "residual_stream"):
        np.testing.assert_allclose(sub[k], full[k][rows], rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------- attention projections

def test_gqa_partition_golden():
    with open(os.path.join(GOLDEN, "gqa_head_partition.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert oracle.gqa_partition(c["nq"], c["nkv"], c["t"]) == (
            c["q_per_shard"], c["kv_per_shard"], c["kv_replicas"]), c["cite"]


@pytest.mark.parametrize("nq,nkv,t", [(4, 2, 1), (4, 2, 2), (8, 2, 4), (8, 4, 4), (8, 2, 8)])
def test_qkv_shard_rows_cover_heads(nq, nkv, t):
    hd = 3
    shards = oracle.qkv_shard_rows(nq, nkv, hd, t)
    q_per, kv_per, rep = oracle.gqa_partition(nq, nkv, t)
    allrows = np.concatenate(shards)
    counts = {}
    for a, b in allrows:
        counts[(int(a), int(b))] = counts.get((int(a), int(b)), 0) + 1
    for row in range(nq * hd):
        assert counts[(0, row)] == 1
    for tensor in (1, 2):
        for row in range(nkv * hd):
            assert counts[(tensor, row)] == rep
    for r, s in enumerate(shards):
        assert len(s) == (q_per + 2 * kv_per) * hd
        # q heads of shard r are r*q_per .. in order, each head's hd rows contiguous
        assert list(s[:q_per * hd, 1]) == list(range(r * q_per * hd, (r + 1) * q_per * hd))


@pytest.mark.parametrize("t", [1, 2, 4])
def test_qkv_parallel_is_head_permutation_of_unsharded(t):
    nq, nkv, hd, T, H = 8, 4, 2, 3, 10
    x, wq, wk, wv = rand(T, H), rand(nq * hd, H), rand(nkv * hd, H), rand(nkv * hd, H)
    out = oracle.qkv_parallel(x, wq, wk, wv, nq, nkv, hd, t)
    full = x @ np.concatenate([wq, wk, wv]).T                   # [T, (nq+2nkv)*hd]
    q_per, kv_per = nq // t, nkv // t
    for r in range(t):
        q = full[:, r * q_per * hd:(r + 1) * q_per * hd]
        k0 = nq * hd + r * kv_per * hd
        v0 = (nq + nkv) * hd + r * kv_per * hd
        want = np.concatenate([q, full[:, k0:k0 + kv_per * hd], full[:, v0:v0 + kv_per * hd]], axis=1)
        np.testing.assert_allclose(out[r], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_o_proj_parallel_equals_unsharded(t):
    T, nq, hd, H = 4, 8, 2, 12
    A, wo = rand(T, nq * hd), rand(H, nq * hd)
    shards = np.stack(np.split(A, t, axis=1))
    np.testing.assert_allclose(oracle.o_proj_parallel(shards, wo, t), A @ wo.T, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- capture

def test_capture_hand_example():
    row_req = np.array([0, 0, 0, 1, 2, 2], np.int32)
    row_pos = np.array([0, 1, 2, 57, 0, 1], np.int32)
    A = np.arange(12, dtype=np.float64).reshape(6, 2)
    B = -A
    sel = oracle.pack_key([2, 0, 1, 0, 9], [1, 2, 57, 2, 0])       # (0,2) twice, (9,0) matches nothing
    hdr, rows = oracle.capture_rows(row_req, row_pos, sel, [A, B], [2, 0], layer=7)
    assert hdr.tolist() == [[0, 2, 2, 7, 2], [1, 57, 2, 7, 3], [2, 1, 2, 7, 5],
                            [0, 2, 0, 7, 2], [1, 57, 0, 7, 3], [2, 1, 0, 7, 5]]
    assert rows.tolist() == [[4, 5], [6, 7], [10, 11], [-4, -5], [-6, -7], [-10, -11]]


def test_capture_empty_selection():
    hdr, rows = oracle.capture_rows(np.zeros(3, np.int32), np.arange(3, dtype=np.int32),
                                    oracle.pack_key([5], [5]), [np.ones((3, 4))], [2], 0)
    assert hdr.shape == (0, 5) and rows.shape == (0, 4)


def test_capture_ragged_workload_selects_drawn_rows():
    w = workloads.WORKLOADS["qwen25_7b_ragged_mlp"]
    b = workloads.ragged_batch(w)
    assert int(b["lens"].sum()) == w.T and len(b["lens"]) == w.requests
    keys = oracle.pack_key(b["row_req"], b["row_pos"])
    assert len(np.unique(keys)) == w.T                     # (request, position) is unique per row
    X = np.arange(w.T, dtype=np.float64)[:, None]
    hdr, rows = oracle.capture_rows(b["row_req"], b["row_pos"], b["sel_keys"], [X, X + 0.5], [2, 0], 3)
    n = len(b["sel_rows"])
    assert hdr.shape == (2 * n, 5)
    assert list(hdr[:n, 4]) == list(b["sel_rows"]) and list(hdr[n:, 4]) == list(b["sel_rows"])
    assert list(rows[:n, 0]) == list(b["sel_rows"].astype(float))


# --------------------------------------------------------------------------- planted mistakes

def _pins_pass(mlp_block, rms_norm, linear):
    """A few of the pins above, run against (possibly mutated) oracle functions."""
    ok = True
    T, H, I = 5, 8, 6
    x = rand(T, H)
    jg, ju, jd = rng.integers(0, H, I), rng.integers(0, H, I), rng.integers(0, I, H)
    wg, wu, wd = np.zeros((I, H)), np.zeros((I, H)), np.zeros((H, I))
    wg[np.arange(I), jg] = 1.0
    wu[np.arange(I), ju] = 1.0
    wd[np.arange(H), jd] = 1.0
    g = x[:, jg[jd]]
    ok &= np.allclose(mlp_block(x, wg, wu, wd), 0.5 * g * (1 + np.tanh(0.5 * g)) * x[:, ju[jd]])
    Hn, v, j, eps = 128, 2.5, 17, 1e-5
    gamma = np.ones(Hn)
    r = np.zeros((1, Hn))
    r[0, j] = v
    ok &= np.isclose(rms_norm(r, gamma, eps)[0, j], math.sqrt(Hn) * v / math.sqrt(v * v + Hn * eps))
    X, W = rand(3, 5), rand(4, 5)
    Y = np.array([[sum(X[i, k] * W[n, k] for k in range(5)) for n in range(4)] for i in range(3)])
    try:
        ok &= np.allclose(linear(X, W), Y)
    except ValueError:
        ok = False
    return bool(ok)


def test_planted_mistakes_are_caught():
    o = oracle
    assert _pins_pass(o.mlp_block, o.rms_norm, o.linear)
    mutants = {
        "gate and up swapped": (lambda x, g, u, d: o.linear(o.silu_mul(o.linear(x, u), o.linear(x, g)), d),
                                o.rms_norm, o.linear),
        "activation dropped": (lambda x, g, u, d: o.linear(o.linear(x, g) * o.linear(x, u), d),
                               o.rms_norm, o.linear),
        "eps outside sqrt": (o.mlp_block,
                             lambda r, gm, e: r / (np.sqrt(np.mean(r * r, -1, keepdims=True)) + e) * gm,
                             o.linear),
        "sum instead of mean": (o.mlp_block,
                                lambda r, gm, e: r / np.sqrt(np.sum(r * r, -1, keepdims=True) + e) * gm,
                                o.linear),
        "transposed weight": (o.mlp_block, o.rms_norm, lambda X, W: X @ W),
    }
    for name, fns in mutants.items():
        assert not _pins_pass(*fns), name
