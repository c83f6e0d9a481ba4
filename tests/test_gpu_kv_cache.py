"""Paged KV cache on the GPU (tp_kv_cache_write, tp_paged_attention) against the oracle.

The cache write is a copy: bit-exact. Attention over the cache: normwise
max|gpu - ref| / max|ref| <= 2e-2 per shard (bf16 q, k, v; fp32 scores,
softmax and split merge; bf16 output). The reference is the oracle's paged
attention over the GPU's own cache contents, and for the decode case also the
contiguous attention core on the same rows (the cache must hold exactly the
sequence). Cases: decode (one new token per request) and chunks of new tokens,
a request of one token, scattered blocks of 1 to 64 tokens (24 included), t = 1,
2, 4 and 8 with kv heads split and replicated, the
Llama-3-8B-shaped decode batch at full size, the gathered layout, block ids
and slots out of range. The attention call that writes the new tokens' k and v
itself must leave the same cache bits and return the same output bits as the
separate write followed by attention.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tensor_linear_layers_gb300 as tl

pytestmark = pytest.mark.gpu
TOL = 2e-2
f64 = oracle.bf16_to_f64


@pytest.fixture(scope="module", autouse=True)
def built():
    from tensor_linear_layers_gb300 import _build
    _build.build()
    tl.lib()
    torch.cuda.set_device(0)


def make_attn(H, nq, nkv, t, flags=0):
    w = workloads.Workload("case", "attn", T=1, H=H, nq=nq, nkv=nkv, hd=128, t=t, w_std=0.02, seed=0)
    d = workloads.attn_inputs(w, T=1)
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, t, H, n_q_heads=nq, n_kv_heads=nkv, head_dim=128, flags=flags)
    return tl.TPLinear(cfg, [d[k].cuda() for k in ("w_q", "w_k", "w_v", "w_o")])


def width(nq, nkv, t):
    kv_per = 1 if t >= nkv else nkv // t
    return (nq // t + 2 * kv_per) * 128


def build_case(blk, nq, nkv, t, lens, new, bs, seed, write_new=True):
    """Cache filled with every request's tokens (or only the context before the new ones)
    through the GPU write; returns what the tests need."""
    rng = np.random.default_rng(seed)
    n_blocks = sum(-(-L // bs) for L in lens) + 5
    perm = rng.permutation(n_blocks)
    max_blocks = max(-(-L // bs) for L in lens) + 1
    tables = np.zeros((len(lens), max_blocks), dtype=np.int32)
    used = 0
    for b, L in enumerate(lens):
        nb = -(-L // bs)
        tables[b, :nb] = perm[used:used + nb]
        used += nb
    full = workloads.draw((t, int(sum(lens)), width(nq, nkv, t)), seed, 0)       # every token of every request
    cu = np.concatenate([[0], np.cumsum(lens)])
    slots = np.concatenate([[tables[b, p // bs] * bs + p % bs for p in range(L)] for b, L in enumerate(lens)])
    ck = torch.zeros(blk.kv_cache_shape(n_blocks, bs), dtype=torch.bfloat16, device="cuda")
    cv = torch.zeros_like(ck)
    rows = np.concatenate([np.arange(cu[b] + L - n, cu[b] + L) for b, (L, n) in enumerate(zip(lens, new))])
    wslots = slots.copy()
    if not write_new:
        wslots[rows] = -1
    ws = blk.kv_cache_write(full.cuda(), torch.from_numpy(wslots.astype(np.int32)).cuda(), ck, cv)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    qkv_new = full[:, rows].contiguous()
    qsl = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    return dict(full=full, cu=cu, rows=rows, qkv_new=qkv_new, qsl=qsl, tables=tables, ck=ck, cv=cv, slots=slots)


def run_paged(blk, c, lens, new, bs):
    out, ws = blk.paged_attention(c["qkv_new"].cuda(), torch.from_numpy(c["qsl"]).cuda(),
                                  torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                  torch.from_numpy(c["tables"]).cuda(), c["ck"], c["cv"], max(new), max(lens))
    torch.cuda.synchronize()
    return out, int(ws[:4].view(torch.int32).item())


def rel_err_shards(got, ref):
    g = got.double().cpu().numpy().reshape(ref.shape)
    return max(float(np.max(np.abs(g[r] - ref[r])) / max(np.max(np.abs(ref[r])), 1e-30)) for r in range(ref.shape[0]))


def test_cache_write_is_exact():
    nq, nkv, t, bs = 8, 2, 2, 16
    blk = make_attn(256, nq, nkv, t)
    lens = [37, 5, 100]
    c = build_case(blk, nq, nkv, t, lens, [1, 1, 1], bs, seed=1)
    q_per, kv_per = nq // t, nkv // t
    n_blocks = c["ck"].shape[1]
    want_k = np.zeros((t, n_blocks, bs, kv_per, 128))
    want_v = np.zeros_like(want_k)
    oracle.kv_cache_write(c["full"], c["slots"], want_k, want_v, nq, nkv, 128, t, bs)
    np.testing.assert_array_equal(f64(c["ck"].cpu()), want_k)
    np.testing.assert_array_equal(f64(c["cv"].cpu()), want_v)


@pytest.mark.parametrize("nq,nkv,t,lens,new,bs", [
    (8, 2, 2, [1, 37, 300, 129], [1, 1, 1, 1], 16),     # decode, one token requests, several splits
    (8, 2, 4, [200, 64], [1, 1], 8),                    # t > nkv: kv head replicated
    (4, 4, 2, [90, 17, 400], [5, 17, 3], 16),           # chunks of new tokens (one whole prefill)
    (16, 2, 1, [1000], [2], 32),                        # groups of 8 q heads, more queries than one pass
    (32, 8, 8, [300, 5], [1, 1], 24),                   # t = 8, one kv head per shard, blocks of 24
    (8, 4, 8, [129, 40], [3, 1], 1),                    # t = 8 > nkv: replicated kv heads, blocks of one token
    (4, 4, 1, [700], [1], 64),                          # t = 1, multi-head (one q head per kv head)
])
def test_paged_attention_matches_oracle(nq, nkv, t, lens, new, bs):
    blk = make_attn(256, nq, nkv, t)
    c = build_case(blk, nq, nkv, t, lens, new, bs, seed=len(lens) + t)
    out, st = run_paged(blk, c, lens, new, bs)
    assert st == 0
    ref = oracle.paged_attention(c["qkv_new"], c["qsl"], lens, c["tables"], c["ck"].cpu(), c["cv"].cpu(),
                                 nq, nkv, 128, t, bs)
    assert rel_err_shards(out, ref) <= TOL
    # the same rows of the contiguous sequences through the attention core's oracle
    ref2 = oracle.attention_rows(c["full"], nq, nkv, 128, t, c["cu"], c["rows"])
    assert rel_err_shards(out, ref2) <= TOL


def test_llama3_8b_decode_batch_full_size():
    w = workloads.WORKLOADS["llama3_8b_paged_decode"]
    blk = make_attn(w.H, w.nq, w.nkv, w.t)
    lens = list(w.seq_lens())
    c = build_case(blk, w.nq, w.nkv, w.t, lens, [1] * len(lens), 16, seed=3)
    out, st = run_paged(blk, c, lens, [1] * len(lens), 16)
    assert st == 0
    pick = [0, 5, 17, len(lens) - 1]
    qsl_sub = np.arange(len(pick) + 1, dtype=np.int32)
    ref = oracle.paged_attention(c["qkv_new"][:, pick], qsl_sub, [lens[b] for b in pick], c["tables"][pick],
                                 c["ck"].cpu(), c["cv"].cpu(), w.nq, w.nkv, 128, w.t, 16)
    assert rel_err_shards(out[:, pick], ref) <= TOL


def test_gathered_layout_same_bits():
    nq, nkv, t, lens, new, bs = 8, 2, 2, [70, 130], [2, 1], 16
    a = make_attn(256, nq, nkv, t)
    g = make_attn(256, nq, nkv, t, flags=tl.TP_FLAG_GATHERED)
    c = build_case(a, nq, nkv, t, lens, new, bs, seed=9)
    out_a, _ = run_paged(a, c, lens, new, bs)
    cg = dict(c, qkv_new=c["qkv_new"].permute(1, 0, 2).reshape(sum(new), -1).contiguous())
    out_g, st = run_paged(g, cg, lens, new, bs)
    assert st == 0
    assert torch.equal(out_g, out_a.permute(1, 0, 2).reshape(sum(new), -1))


def test_block_id_out_of_range_reports_shape_error():
    nq, nkv, t, lens, new, bs = 8, 2, 2, [40], [1], 16
    blk = make_attn(256, nq, nkv, t)
    c = build_case(blk, nq, nkv, t, lens, new, bs, seed=4)
    c["tables"][0, 1] = 10_000
    _, st = run_paged(blk, c, lens, new, bs)
    assert st == tl.TP_ERR_SHAPE
    bad = torch.tensor([c["ck"].shape[1] * bs], dtype=torch.int32, device="cuda")       # one past the cache
    ws = blk.kv_cache_write(c["qkv_new"][:, :1].contiguous().cuda(), bad, c["ck"], c["cv"])
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == tl.TP_ERR_SHAPE


@pytest.mark.parametrize("nq,nkv,t,lens,new,bs", [
    (8, 2, 2, [1, 37, 300, 129], [1, 1, 1, 1], 16),     # decode
    (4, 4, 2, [90, 17, 400], [5, 17, 3], 16),           # chunks, one whole prefill
    (8, 2, 2, [270, 50], [30, 2], 16),                  # new tokens on both sides of a split boundary
    (8, 2, 4, [200, 64], [1, 1], 8),                    # t > nkv: each shard writes its replica
])
def test_write_inside_attention_same_bits(nq, nkv, t, lens, new, bs):
    blk = make_attn(256, nq, nkv, t)
    c = build_case(blk, nq, nkv, t, lens, new, bs, seed=20 + len(lens), write_new=False)
    new_slots = c["slots"][c["rows"]].astype(np.int32)
    new_slots[0] = -1                                   # a padding token writes nothing on either path
    new_slots = torch.from_numpy(new_slots).cuda()
    ck2, cv2 = c["ck"].clone(), c["cv"].clone()
    out_f, ws = blk.paged_attention(c["qkv_new"].cuda(), torch.from_numpy(c["qsl"]).cuda(),
                                    torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                    torch.from_numpy(c["tables"]).cuda(), ck2, cv2, max(new), max(lens),
                                    slot_mapping=new_slots)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    wk = blk.kv_cache_write(c["qkv_new"].cuda(), new_slots, c["ck"], c["cv"])
    out_s, st = run_paged(blk, c, lens, new, bs)
    assert st == 0 and int(wk[:4].view(torch.int32).item()) == 0
    assert torch.equal(ck2, c["ck"]) and torch.equal(cv2, c["cv"])
    assert torch.equal(out_f, out_s)


def test_write_inside_attention_slot_out_of_range():
    nq, nkv, t, lens, new, bs = 8, 2, 2, [40, 9], [1, 1], 16
    blk = make_attn(256, nq, nkv, t)
    c = build_case(blk, nq, nkv, t, lens, new, bs, seed=5, write_new=False)
    bad = torch.tensor([c["ck"].shape[1] * bs, int(c["slots"][c["rows"][1]])], dtype=torch.int32, device="cuda")
    _, ws = blk.paged_attention(c["qkv_new"].cuda(), torch.from_numpy(c["qsl"]).cuda(),
                                torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                torch.from_numpy(c["tables"]).cuda(), c["ck"], c["cv"], 1, max(lens),
                                slot_mapping=bad)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == tl.TP_ERR_SHAPE


def test_workspace_of_long_chunks_stays_bounded():
    # a 4096-token chunk of new tokens over 8192 cached ones: fewer splits, not gigabytes of partials
    blk = make_attn(256, 8, 2, 2)
    assert blk.paged_attention_workspace_size(1, 4096, 8192) <= 256 * 2**20 + 4096
    assert blk.paged_attention_workspace_size(32, 1, 4096) < 2**20 * 16      # decode: small
