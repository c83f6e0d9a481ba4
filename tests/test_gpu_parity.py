"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Tolerance: normwise max relative error max|gpu - ref| / max|ref| <= 2e-2 per
output tensor (bf16 inputs, fp32 accumulation, bf16 outputs). Integer work
(capture indices, headers, copied rows) is compared bit for bit.
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


def rel_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.double().cpu().numpy().reshape(ref.shape)
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


@pytest.fixture(scope="module", autouse=True)
def built():
    from tensor_linear_layers_gb300 import _build
    _build.build()
    tl.lib()
    torch.cuda.set_device(0)


def status_of(ws: torch.Tensor) -> int:
    torch.cuda.synchronize()
    return int(ws[:4].view(torch.int32).item())


def make_mlp(H, I, t, norm=False, seed=0, w_std=0.02):
    w = workloads.Workload("case", "mlp", T=1, H=H, I=I, t=t, w_std=w_std, norm=norm, seed=seed)
    d = workloads.mlp_inputs(w, T=1)
    cfg = tl.make_config(tl.TP_BLOCK_MLP, t, H, I, rms_eps=1e-5, flags=tl.TP_FLAG_HAS_NORM if norm else 0)
    dev = torch.device("cuda")
    blk = tl.TPLinear(cfg, [d["w_gate"].to(dev), d["w_up"].to(dev), d["w_down"].to(dev)],
                      gamma=None if not norm else d["gamma"].to(dev))
    return blk, d


def mlp_ref(d, x, residual=None, norm=False, rows=None):
    return oracle.mlp_layer(f64(x), f64(d["w_gate"]), f64(d["w_up"]), f64(d["w_down"]),
                            residual=None if residual is None else f64(residual),
                            gamma=None if not norm else f64(d["gamma"]), eps=1e-5, norm=norm, rows=rows)


# ------------------------------------------------------------------ plain GEMM through t = 1

@pytest.mark.parametrize("T", [16, 64, 128, 200])
def test_attention_projections_t1_are_plain_gemms(T):
    H, nq, hd = 512, 4, 128
    w = workloads.Workload("case", "attn", T=T, H=H, nq=nq, nkv=nq, hd=hd, t=1, w_std=0.02)
    d = workloads.attn_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, 1, H, n_q_heads=nq, n_kv_heads=nq, head_dim=hd)
    dev = torch.device("cuda")
    blk = tl.TPLinear(cfg, [d[k].to(dev) for k in ("w_q", "w_k", "w_v", "w_o")])
    qkv, o = blk.attn_proj_forward(d["x"].to(dev), d["attn"].to(dev))
    ref_qkv = oracle.qkv_parallel(f64(d["x"]), f64(d["w_q"]), f64(d["w_k"]), f64(d["w_v"]), nq, nq, hd, 1)
    ref_o = oracle.o_proj_parallel(f64(d["attn"]), f64(d["w_o"]), 1)
    assert rel_err(qkv, ref_qkv) <= TOL
    assert rel_err(o, ref_o) <= TOL
    assert status_of(blk.workspace(T)) == 0


# ------------------------------------------------------------------ MLP, small shapes, every tile path

@pytest.mark.parametrize("T", [1, 7, 16, 33, 100, 129, 300])
def test_tiny_mlp_matches_oracle(T):
    blk, d = make_mlp(512, 1408, 2)                 # I/t = 704: not a multiple of 128
    x = workloads.draw((T, 512), 0, 0)
    out = blk.mlp_forward(x.cuda())
    ref = mlp_ref(d, x)
    assert rel_err(out["mlp_out"], ref["mlp_out"]) <= TOL
    assert status_of(blk.workspace(T)) == 0


@pytest.mark.parametrize("T", [5, 200])
def test_mlp_with_norm_and_residual_stream(T):
    H, I, t = 1024, 2048, 4
    blk, d = make_mlp(H, I, t, norm=True)
    a, r0 = workloads.draw((T, H), 3, 0), workloads.draw((T, H), 3, 1)
    out = blk.mlp_forward(a.cuda(), residual=r0.cuda())
    ref = mlp_ref(d, a, residual=r0, norm=True)
    for k in ("mlp_out", "residual_out", "residual_stream"):
        assert rel_err(out[k], ref[k]) <= TOL, k
    assert status_of(blk.workspace(T)) == 0


# ------------------------------------------------------------------ prefill tails on CTA pairs

@pytest.mark.parametrize("T", [256, 300, 1000, 1300, 1421])
def test_prefill_tails_on_cta_pairs_every_row(T):
    # 8 token tiles, the last one partial (104 rows); 11 tiles, so the odd CTA of the
    # last pair has no tile; 12 tiles, the last one 13 rows. Both GEMMs run on CTA
    # pairs at this shape; every row of every output is compared. With 16 weight tiles
    # per GEMM a launch's last wave is split along K when it is at most half full: T =
    # 256 gives 16 pair units in 4 parts each, T = 300 32 units in 2 parts, T = 1300 and
    # 1421 a 20-unit tail in 3 parts (the last part of a unit adds the parts in order).
    H, I, t = 4096, 2048, 4
    blk, d = make_mlp(H, I, t, norm=True)
    assert [p["engine"] for p in blk.plan(T)] == [1, 1]
    a, r0 = workloads.draw((T, H), 13, 0), workloads.draw((T, H), 13, 1)
    out = blk.mlp_forward(a.cuda(), residual=r0.cuda())
    ref = mlp_ref(d, a, residual=r0, norm=True)
    for k in ("mlp_out", "residual_out", "residual_stream"):
        assert rel_err(out[k], ref[k]) <= TOL, k
    assert status_of(blk.workspace(T)) == 0


@pytest.mark.parametrize("H,T", [(128, 256), (128, 300), (192, 256)])
def test_prefill_split_tail_never_exceeds_k_blocks(H, T):
    # gate_up's K is H: 2 or 3 k-blocks of 64. Its 4 pair units (2I = 1024 weight rows)
    # fill a small part of one wave, so the wave is split along K, into at most as many
    # parts as there are k-blocks: a part with an empty K range would hand its stale
    # accumulator to the reduction. Every row of the output is compared.
    blk, d = make_mlp(H, 512, 1)
    assert blk.plan(T)[0]["engine"] == 1
    a = workloads.draw((T, H), 17, 0)
    out = blk.mlp_forward(a.cuda())
    ref = mlp_ref(d, a)
    assert rel_err(out["mlp_out"], ref["mlp_out"]) <= TOL
    assert status_of(blk.workspace(T)) == 0


@pytest.mark.parametrize("T", [1300, 1421])
def test_attention_projections_tails_on_cta_pairs_every_row(T):
    # QKV and o_proj in one CTA-pair launch, odd and even tile counts with partial tiles
    H, nq, nkv, hd, t = 2048, 16, 4, 128, 2
    w = workloads.Workload("case", "attn", T=T, H=H, nq=nq, nkv=nkv, hd=hd, t=t, w_std=0.02)
    d = workloads.attn_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, t, H, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd)
    blk = tl.TPLinear(cfg, [d[k].cuda() for k in ("w_q", "w_k", "w_v", "w_o")])
    assert blk.plan(T)[0]["engine"] == 1
    qkv, o = blk.attn_proj_forward(d["x"].cuda(), d["attn"].cuda())
    ref_qkv = oracle.qkv_parallel(f64(d["x"]), f64(d["w_q"]), f64(d["w_k"]), f64(d["w_v"]), nq, nkv, hd, t)
    ref_o = oracle.o_proj_parallel(f64(d["attn"]), f64(d["w_o"]), t)
    assert rel_err(qkv, ref_qkv) <= TOL
    assert rel_err(o, ref_o) <= TOL
    assert status_of(blk.workspace(T)) == 0


@pytest.mark.parametrize("t", [1, 2, 4])
@pytest.mark.parametrize("T", [16, 160])
def test_attention_gqa_split_by_head(t, T):
    H, nq, nkv, hd = 256, 8, 2, 64               # t = 4 > nkv: kv heads replicated
    w = workloads.Workload("case", "attn", T=T, H=H, nq=nq, nkv=nkv, hd=hd, t=t, w_std=0.05)
    d = workloads.attn_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, t, H, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd)
    blk = tl.TPLinear(cfg, [d[k].cuda() for k in ("w_q", "w_k", "w_v", "w_o")])
    qkv, o = blk.attn_proj_forward(d["x"].cuda(), d["attn"].cuda())
    ref_qkv = oracle.qkv_parallel(f64(d["x"]), f64(d["w_q"]), f64(d["w_k"]), f64(d["w_v"]), nq, nkv, hd, t)
    ref_o = oracle.o_proj_parallel(f64(d["attn"]), f64(d["w_o"]), t)
    assert tuple(qkv.shape) == ref_qkv.shape
    assert rel_err(qkv, ref_qkv) <= TOL
    assert rel_err(o, ref_o) <= TOL


# ------------------------------------------------------------------ invariants

@pytest.mark.parametrize("T", [32, 256])
def test_results_bit_identical_across_t(T):
    # the t shards are a layout: with I/t a multiple of 128 the kernels run the
    # same tiles and the same K order, so every t gives the same bits
    x = workloads.draw((T, 512), 9, 0).cuda()
    outs = []
    for t in (1, 2, 4, 8):
        blk, d = make_mlp(512, 1024, t)
        outs.append(blk.mlp_forward(x)["mlp_out"].clone())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    ref = mlp_ref(d, x.cpu())
    assert rel_err(outs[0], ref["mlp_out"]) <= TOL


@pytest.mark.parametrize("T", [32, 300])
def test_run_twice_same_bits(T):
    blk, d = make_mlp(1024, 4096, 8, norm=True)
    a, r0 = workloads.draw((T, 1024), 5, 0).cuda(), workloads.draw((T, 1024), 5, 1).cuda()
    o1 = {k: v.clone() for k, v in blk.mlp_forward(a, residual=r0).items()}
    o2 = blk.mlp_forward(a, residual=r0)
    for k in o1:
        assert torch.equal(o1[k], o2[k]), k


def test_zero_tokens_is_a_no_op():
    blk, _ = make_mlp(512, 1408, 2)
    x = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    out = blk.mlp_forward(x)
    assert out["mlp_out"].shape == (0, 512)


def test_stage_entry_points_match_oracle():
    H, I, t, T = 1024, 2048, 4, 48
    blk, d = make_mlp(H, I, t, norm=True)
    a, r0 = workloads.draw((T, H), 7, 0), workloads.draw((T, H), 7, 1)
    x, r = tl.add_rms_norm(a.cuda(), r0.cuda(), d["gamma"].cuda(), 1e-5)
    ref_x, ref_r = oracle.add_rms_norm(f64(a), f64(r0), f64(d["gamma"]), 1e-5)
    assert rel_err(r, ref_r) <= TOL and rel_err(x, ref_x) <= TOL
    h = blk.gate_up(x)
    _, ref_h = oracle.mlp_block_tp(f64(x.cpu()), f64(d["w_gate"]), f64(d["w_up"]), f64(d["w_down"]), t)
    assert rel_err(h, np.stack(ref_h)) <= TOL
    y, s = blk.down(h, residual=r)
    ref_y = oracle.linear(f64(h.cpu()).reshape(t, T, -1).transpose(1, 0, 2).reshape(T, -1), f64(d["w_down"]))
    assert rel_err(y, ref_y) <= TOL
    assert rel_err(s, ref_y + f64(r.cpu())) <= TOL


# ------------------------------------------------------------------ capture

def test_capture_small_exact():
    T, H = 40, 64
    g = torch.Generator().manual_seed(0)
    row_req = torch.randint(0, 5, (T,), generator=g, dtype=torch.int32)
    row_pos = torch.arange(T, dtype=torch.int32)
    A = workloads.draw((T, H), 1, 0)
    B = workloads.draw((T, H), 1, 1)
    sel = oracle.pack_key([int(row_req[3]), int(row_req[3]), int(row_req[17]), 99, int(row_req[39])],
                          [3, 3, 17, 0, 39])
    hdr, rows, n_out, ws = tl.capture_rows(row_req.cuda(), row_pos.cuda(), torch.from_numpy(sel).cuda(),
                                           [A.cuda(), B.cuda()], [2, 0], 11, capacity=16)
    rh, rr = oracle.capture_rows(row_req.numpy(), row_pos.numpy(), sel, [A.float().numpy(), B.float().numpy()],
                                 [2, 0], 11)
    n = int(n_out.item())
    assert n == len(rh) == 6
    assert np.array_equal(hdr[:n, :5].cpu().numpy(), rh)
    assert torch.equal(rows[:n].cpu().float(), torch.from_numpy(rr).float())
    assert status_of(ws) == 0


def test_capture_overflow_reports_capacity():
    T, H = 64, 64
    row_req = torch.zeros(T, dtype=torch.int32)
    row_pos = torch.arange(T, dtype=torch.int32)
    A = workloads.draw((T, H), 2, 0)
    sel = oracle.pack_key([0] * 10, list(range(10)))
    hdr, rows, n_out, ws = tl.capture_rows(row_req.cuda(), row_pos.cuda(), torch.from_numpy(sel).cuda(),
                                           [A.cuda()], [2], 0, capacity=4)
    assert int(n_out.item()) == 10
    assert status_of(ws) == tl.TP_ERR_CAPACITY
    assert hdr[:4, 4].cpu().tolist() == [0, 1, 2, 3]


@pytest.mark.parametrize("T", [300, 20000])
def test_capture_all_ones_key_on_both_paths(T):
    # A row of request -1 at position -1 has the all-ones key, which is also the table's
    # empty-slot marker. T = 300 runs the single-launch capture (each CTA matches every
    # row); T = 20000 is past its 64 rows per thread and runs the two-kernel one.
    H = 64
    row_req = torch.arange(T, dtype=torch.int32) % 97
    row_pos = torch.arange(T, dtype=torch.int32) // 97
    row_req[5] = -1
    row_pos[5] = -1
    A = workloads.draw((T, H), 5, 0)
    rng = np.random.default_rng(4)
    rows_sel = rng.choice(T, 150, replace=False)
    sel = np.concatenate([oracle.pack_key(row_req.numpy()[rows_sel], row_pos.numpy()[rows_sel]),
                          oracle.pack_key([-1], [-1])])
    hdr, rows, n_out, ws = tl.capture_rows(row_req.cuda(), row_pos.cuda(), torch.from_numpy(sel).cuda(),
                                           [A.cuda()], [1], 3, capacity=T)
    rh, rr = oracle.capture_rows(row_req.numpy(), row_pos.numpy(), sel, [A.float().numpy()], [1], 3)
    n = int(n_out.item())
    assert n == len(rh) and 5 in rh[:, 4].tolist()
    assert np.array_equal(hdr[:n, :5].cpu().numpy(), rh)
    assert torch.equal(rows[:n].cpu().float(), torch.from_numpy(rr).float())
    assert status_of(ws) == 0


def test_capture_large_selector_set_uses_global_table():
    T, H = 5000, 64
    row_req = torch.arange(T, dtype=torch.int32) // 100
    row_pos = torch.arange(T, dtype=torch.int32) % 100
    A = workloads.draw((T, H), 4, 0)
    rng = np.random.default_rng(3)
    rows_sel = rng.choice(T, 3000, replace=False)
    sel = np.concatenate([oracle.pack_key(row_req.numpy()[rows_sel], row_pos.numpy()[rows_sel]),
                          oracle.pack_key(np.arange(9000, 14000), np.zeros(5000))])   # 5000 misses
    hdr, rows, n_out, ws = tl.capture_rows(row_req.cuda(), row_pos.cuda(), torch.from_numpy(sel).cuda(),
                                           [A.cuda()], [0], 2, capacity=T)
    n = int(n_out.item())
    assert n == 3000
    assert hdr[:n, 4].cpu().numpy().tolist() == sorted(rows_sel.tolist())
    assert torch.equal(rows[:n].cpu(), A[torch.from_numpy(np.sort(rows_sel))])


# ------------------------------------------------------------------ the five workloads at full size

# rows compared per 128-token tile at full size: every tile (so both tiles of every
# CTA pair) and, on the Llama-3-70B-shaped batch, 4 x 64 = 256 rows
ROWS_PER_TILE = {"llama3_70b_mlp_prefill": 4, "qwen25_7b_ragged_mlp": 8, "llama3_8b_attn_proj_prefill": 4}


@pytest.mark.parametrize("name", ["tiny_mlp", "llama3_8b_mlp_decode", "llama3_70b_mlp_prefill",
                                  "qwen25_7b_ragged_mlp"])
def test_mlp_workload_full_size_every_tile(name):
    w = workloads.WORKLOADS[name]
    d = workloads.mlp_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_MLP, w.t, w.H, w.I, rms_eps=w.eps,
                         flags=tl.TP_FLAG_HAS_NORM if w.norm else 0)
    blk = tl.TPLinear(cfg, [d["w_gate"].cuda(), d["w_up"].cuda(), d["w_down"].cuda()],
                      gamma=None if not w.norm else d["gamma"].cuda())
    out = blk.mlp_forward(d["x"].cuda(), residual=None if d["residual"] is None else d["residual"].cuda())
    assert status_of(blk.workspace(w.T)) == 0
    rows = tile_rows(w.T, ROWS_PER_TILE[name]) if w.T > 128 else None
    if name == "llama3_70b_mlp_prefill":
        assert rows.size >= 256
    ref = mlp_ref(d, d["x"], residual=d["residual"], norm=w.norm, rows=rows)
    sel = slice(None) if rows is None else torch.from_numpy(rows)
    for k in ("mlp_out", "residual_out", "residual_stream"):
        if ref.get(k) is not None:
            assert rel_err(out[k].cpu()[sel], ref[k]) <= TOL, k
    if name == "qwen25_7b_ragged_mlp":
        b = workloads.ragged_batch(w)
        types = [workloads.TENSOR_TYPES["mlp_out"], workloads.TENSOR_TYPES["residual_stream"]]
        hdr, rec, n_out, ws = tl.capture_rows(
            torch.from_numpy(b["row_req"]).cuda(), torch.from_numpy(b["row_pos"]).cuda(),
            torch.from_numpy(b["sel_keys"]).cuda(), [out["mlp_out"], out["residual_stream"]], types,
            layer=0, capacity=2 * len(b["sel_keys"]))
        n = int(n_out.item())
        ms, rs = out["mlp_out"].cpu(), out["residual_stream"].cpu()
        rh, rr = oracle.capture_rows(b["row_req"], b["row_pos"], b["sel_keys"],
                                     [ms.view(torch.int16).numpy(), rs.view(torch.int16).numpy()], types, 0)
        assert n == len(rh) == 2 * 205
        assert np.array_equal(hdr[:n, :5].cpu().numpy(), rh)
        assert np.array_equal(rec[:n].cpu().view(torch.int16).numpy(), rr)
        assert status_of(ws) == 0


def test_attention_workload_full_size_every_tile():
    w = workloads.WORKLOADS["llama3_8b_attn_proj_prefill"]
    d = workloads.attn_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, w.t, w.H, n_q_heads=w.nq, n_kv_heads=w.nkv, head_dim=w.hd)
    blk = tl.TPLinear(cfg, [d[k].cuda() for k in ("w_q", "w_k", "w_v", "w_o")])
    qkv, o = blk.attn_proj_forward(d["x"].cuda(), d["attn"].cuda())
    assert status_of(blk.workspace(w.T)) == 0
    rows = tile_rows(w.T, ROWS_PER_TILE[w.name])
    x = f64(d["x"])[rows]
    ref_qkv = oracle.qkv_parallel(x, f64(d["w_q"]), f64(d["w_k"]), f64(d["w_v"]), w.nq, w.nkv, w.hd, w.t)
    ref_o = oracle.o_proj_parallel(f64(d["attn"])[:, rows], f64(d["w_o"]), w.t)
    assert rel_err(qkv.cpu()[:, torch.from_numpy(rows)], ref_qkv) <= TOL
    assert rel_err(o.cpu()[torch.from_numpy(rows)], ref_o) <= TOL


@pytest.mark.parametrize("T", [1, 16, 32, 100, 128])
def test_fused_decode_block_matches_stage_calls(T):
    # T <= 128 runs as one fused kernel; the stage entry points run the same
    # steps as separate kernels: same residual bits, outputs within tolerance
    H, I, t = 1024, 4096, 4
    blk, d = make_mlp(H, I, t, norm=True)
    a, r0 = workloads.draw((T, H), 11, 0).cuda(), workloads.draw((T, H), 11, 1).cuda()
    for _ in range(3):      # repeated launches reuse the phase counters
        fused = blk.mlp_forward(a, residual=r0)
    x, r = tl.add_rms_norm(a, r0, d["gamma"].cuda(), 1e-5)
    h = blk.gate_up(x)
    y, s = blk.down(h, residual=r)
    assert torch.equal(fused["residual_out"], r)
    ref = mlp_ref(d, a.cpu(), residual=r0.cpu(), norm=True)
    assert rel_err(fused["mlp_out"], ref["mlp_out"]) <= TOL
    assert rel_err(fused["residual_stream"], ref["residual_stream"]) <= TOL
    assert rel_err(fused["mlp_out"], y.double().cpu().numpy()) <= 1e-2
    assert status_of(blk.workspace(T)) == 0


@pytest.mark.parametrize("T", [1, 24])
def test_fused_decode_more_gate_up_tiles_than_sms(T):
    # I / t = 5120 gives 40 gate_up tiles per shard, 320 in all: more than the SMs, so
    # the CTAs after the single norm CTA own two or three gate_up tiles each
    H, I, t = 1024, 40960, 8
    blk, d = make_mlp(H, I, t, norm=True, seed=3)
    assert blk.plan(T)[0]["engine"] == 2
    a, r0 = workloads.draw((T, H), 17, 0), workloads.draw((T, H), 17, 1)
    out = blk.mlp_forward(a.cuda(), residual=r0.cuda())
    ref = mlp_ref(d, a, residual=r0, norm=True)
    for k in ("mlp_out", "residual_out", "residual_stream"):
        assert rel_err(out[k], ref[k]) <= TOL, k
    assert status_of(blk.workspace(T)) == 0


def test_workspace_bound_covers_every_token_count():
    # one workspace sized for max_tokens must serve every T <= max_tokens
    blk, d = make_mlp(512, 1408, 2, norm=True)
    ws = blk.workspace(300)
    for T in list(range(1, 140)) + [200, 255, 256, 257, 299, 300]:
        a = torch.zeros(T, 512, dtype=torch.bfloat16, device="cuda")
        blk.mlp_forward(a, residual=a.clone(), ws=ws)
    assert status_of(ws) == 0
