"""Parity of the attention core (tp_attention_forward, through the C ABI) with the oracle.

Tolerance as for the projections: normwise max|gpu - ref| / max|ref| <= 2e-2
per shard output (bf16 q, k, v; fp32 scores and softmax; P rounded to bf16
for the P V product; bf16 output). The cases cover several 128-query tiles,
ragged tails, one-token and exact-tile sequences, kv heads split and
replicated (t > nkv), plain multi-head (group of one), the Llama-3-8B-shaped
4096-token sequence at full size (sampled rows), the ragged Qwen-shaped batch
in full, determinism, an output only 16-byte aligned, bad offsets and the QKV ->
attention -> o_proj chain.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tensor_linear_layers_gb300 as tl
from tile_rows import tile_rows

pytestmark = pytest.mark.gpu
TOL = 2e-2
f64 = oracle.bf16_to_f64


@pytest.fixture(scope="module", autouse=True)
def built():
    from tensor_linear_layers_gb300 import _build
    _build.build()
    tl.lib()
    torch.cuda.set_device(0)


def status_of(ws: torch.Tensor) -> int:
    torch.cuda.synchronize()
    return int(ws[:4].view(torch.int32).item())


def rel_err_shards(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.double().cpu().numpy().reshape(ref.shape)
    return max(float(np.max(np.abs(g[r] - ref[r])) / max(np.max(np.abs(ref[r])), 1e-30)) for r in range(ref.shape[0]))


def make_attn(H, nq, nkv, t, hd=128, seed=0):
    w = workloads.Workload("case", "attn", T=1, H=H, nq=nq, nkv=nkv, hd=hd, t=t, w_std=0.02, seed=seed)
    d = workloads.attn_inputs(w, T=1)
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, t, H, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd)
    return tl.TPLinear(cfg, [d[k].cuda() for k in ("w_q", "w_k", "w_v", "w_o")]), d


def qkv_width(nq, nkv, t, hd=128):
    kv_per = 1 if t >= nkv else nkv // t
    return (nq // t + 2 * kv_per) * hd


def run(blk, qkv, lens):
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    out = blk.attention_forward(qkv.cuda(), cu, int(max(lens)))
    return out, cu


@pytest.mark.parametrize("nq,nkv,t,lens", [
    (8, 2, 2, [128, 1, 171]),          # exact tile, one-token sequence, two tiles with a tail
    (8, 2, 4, [257]),                  # t > nkv: kv head replicated; three tiles
    (4, 4, 2, [50, 300, 7]),           # one kv head per q head
    (16, 2, 1, [384]),                 # t = 1, groups of 8
])
def test_attention_matches_oracle(nq, nkv, t, lens):
    blk, _ = make_attn(256, nq, nkv, t)
    T = int(sum(lens))
    qkv = workloads.draw((t, T, qkv_width(nq, nkv, t)), 11, 0)
    out, cu = run(blk, qkv, lens)
    ref = oracle.attention_core(qkv, nq, nkv, 128, t, cu.cpu().numpy())
    err = rel_err_shards(out, ref)
    assert err <= TOL, err
    assert status_of(blk.workspace(T)) == 0


def test_llama3_8b_full_size_every_query_tile():
    w = workloads.WORKLOADS["llama3_8b_attn_core_prefill"]
    blk, _ = make_attn(w.H, w.nq, w.nkv, w.t)
    d = workloads.attn_core_inputs(w)
    out, cu = run(blk, d["qkv"], np.diff(d["cu_seqlens"]))
    # the first and last query of every 128-query tile and two between (every work unit's tile)
    rows = [int(r) for r in tile_rows(4096, 4)]
    ref = oracle.attention_rows(d["qkv"], w.nq, w.nkv, w.hd, w.t, d["cu_seqlens"], rows)
    got = out[:, rows]
    err = rel_err_shards(got, ref)
    assert err <= TOL, err
    assert status_of(blk.workspace(d["T"])) == 0


def test_qwen_ragged_batch_in_full():
    w = workloads.WORKLOADS["qwen25_7b_ragged_attn_core"]
    blk, _ = make_attn(w.H, w.nq, w.nkv, w.t)
    d = workloads.attn_core_inputs(w)
    out, cu = run(blk, d["qkv"], np.diff(d["cu_seqlens"]))
    ref = oracle.attention_core(d["qkv"], w.nq, w.nkv, w.hd, w.t, d["cu_seqlens"])
    err = rel_err_shards(out, ref)
    assert err <= TOL, err
    assert status_of(blk.workspace(d["T"])) == 0


def test_run_twice_same_bits():
    blk, _ = make_attn(256, 8, 2, 2)
    lens = [300, 45, 200]
    qkv = workloads.draw((2, 545, qkv_width(8, 2, 2)), 12, 0)
    a, _ = run(blk, qkv, lens)
    b, _ = run(blk, qkv, lens)
    assert torch.equal(a, b)


def test_output_only_16_byte_aligned_same_bits():
    # rows go out with 32-byte stores when the output is 32-byte aligned and with
    # 16-byte stores otherwise; both must write the same values
    blk, _ = make_attn(256, 8, 2, 2)
    lens = [300, 45, 200]
    qkv = workloads.draw((2, 545, qkv_width(8, 2, 2)), 12, 0)
    a, cu = run(blk, qkv, lens)
    big = torch.full((a.numel() + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = big[8:].view(a.shape)
    assert out.data_ptr() % 32 == 16
    blk.attention_forward(qkv.cuda(), cu, int(max(lens)), out=out)
    assert torch.equal(a, out)
    assert status_of(blk.workspace(545)) == 0


def test_bad_offsets_report_shape_error():
    blk, _ = make_attn(256, 8, 2, 2)
    qkv = workloads.draw((2, 64, qkv_width(8, 2, 2)), 13, 0).cuda()
    ws = blk.workspace(64)
    ws.zero_()
    cu = torch.tensor([0, 40, 30, 64], dtype=torch.int32, device="cuda")     # falls
    blk.attention_forward(qkv, cu, 40, ws=ws)
    assert status_of(ws) == tl.TP_ERR_SHAPE
    long = workloads.draw((2, 300, qkv_width(8, 2, 2)), 13, 1).cuda()
    ws = blk.workspace(300)
    ws.zero_()
    blk.attention_forward(long, torch.tensor([0, 300], dtype=torch.int32, device="cuda"), 100, ws=ws)
    assert status_of(ws) == tl.TP_ERR_SHAPE                                   # 300 > 100 rounded up to 128
    ws.zero_()
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    out = blk.attention_forward(qkv, cu, 64, ws=ws)                            # the context still works
    ref = oracle.attention_core(qkv.cpu(), 8, 2, 128, 2, [0, 64])
    assert rel_err_shards(out, ref) <= TOL
    assert status_of(ws) == 0


def test_empty_step_enqueues_nothing():
    blk, _ = make_attn(256, 8, 2, 2)
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert tl.lib().tp_attention_forward(blk.handle, 0, None, cu.data_ptr(), 0, 0, None, None, 0, None) == 0


def test_projection_attention_projection_chain():
    H, nq, nkv, t, lens = 512, 8, 2, 2, [150, 90]
    T = sum(lens)
    w = workloads.Workload("case", "attn", T=T, H=H, nq=nq, nkv=nkv, hd=128, t=t, w_std=0.02, seed=3)
    d = workloads.attn_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, t, H, n_q_heads=nq, n_kv_heads=nkv, head_dim=128)
    blk = tl.TPLinear(cfg, [d[k].cuda() for k in ("w_q", "w_k", "w_v", "w_o")])
    qkv, _ = blk.attn_proj_forward(d["x"].cuda(), None)
    attn, cu = run(blk, qkv, lens)
    _, o = blk.attn_proj_forward(None, attn)
    ref_qkv = oracle.qkv_parallel(f64(d["x"]), f64(d["w_q"]), f64(d["w_k"]), f64(d["w_v"]), nq, nkv, 128, t)
    ref_attn = oracle.attention_core(ref_qkv, nq, nkv, 128, t, [0, lens[0], T])
    ref_o = oracle.o_proj_parallel(ref_attn, f64(d["w_o"]), t)
    assert rel_err_shards(attn, ref_attn) <= TOL
    g = o.double().cpu().numpy()
    assert float(np.max(np.abs(g - ref_o)) / np.max(np.abs(ref_o))) <= TOL
    assert status_of(blk.workspace(T)) == 0


@pytest.mark.parametrize("how", ["one_row", "whole_tile"])
def test_running_max_jump_rescales_o(how):
    # the running max grows by more than the lazy threshold at a later key tile: for a
    # single query row (one lane of a warp) or for every row (a whole scaled key tile)
    nq, nkv, t, lens = 8, 2, 2, [500]
    blk, _ = make_attn(256, nq, nkv, t)
    q_per, kv_per = nq // t, nkv // t
    qkv = workloads.draw((t, 500, qkv_width(nq, nkv, t)), 14, 0).float()
    kc = slice(q_per * 128, (q_per + kv_per) * 128)             # every k head of a shard
    if how == "one_row":
        # key 300 = 8 x query 350 (head 0's kv head): only row 350 sees a score jump
        qkv[:, 300, q_per * 128:q_per * 128 + 128] = 8.0 * qkv[:, 350, 0:128]
    else:
        qkv[:, 256:384, kc] *= 6.0                               # key tile 2 of every sequence row
    qkv = qkv.to(torch.bfloat16)
    out, cu = run(blk, qkv, lens)
    ref = oracle.attention_core(qkv, nq, nkv, 128, t, cu.cpu().numpy())
    assert rel_err_shards(out, ref) <= TOL
    assert status_of(blk.workspace(500)) == 0
