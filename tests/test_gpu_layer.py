"""Parity of one whole decoder layer (tp_decoder_layer_forward, through the C ABI)
with the oracle's chain, and attn_out capture behind it.

Tolerance as for the single steps: normwise max|gpu - ref| / max|ref| <= 2e-2
for each output tensor (bf16 inputs; every intermediate the GPU hands from one
kernel to the next is rounded to bf16, the oracle rounds nothing). Cases cover
the prefill path (T > 128: CTA-pair GEMMs, attention over several query
tiles), the decode-sized path (T <= 128: swapped GEMMs and the fused MLP
kernel), the first-layer form without an incoming residual, the ragged
Qwen-shaped batch at full size with attn_out / mlp_out / residual_stream
capture, and the Llama-3-8B-shaped 4096-token layer at full size on sampled
rows.
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
KEYS = ("residual_attn", "attn_out", "residual_mlp", "mlp_out", "residual_stream")


@pytest.fixture(scope="module", autouse=True)
def built():
    from tensor_linear_layers_gb300 import _build
    _build.build()
    tl.lib()
    torch.cuda.set_device(0)


def make_layer(w, d, max_tokens):
    dev = "cuda"
    ca = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, w.t, w.H, n_q_heads=w.nq, n_kv_heads=w.nkv, head_dim=w.hd,
                        rms_eps=w.eps, flags=tl.TP_FLAG_HAS_NORM)
    cm = tl.make_config(tl.TP_BLOCK_MLP, w.t, w.H, w.I, rms_eps=w.eps, flags=tl.TP_FLAG_HAS_NORM)
    attn = tl.TPLinear(ca, [d[k].to(dev) for k in ("w_q", "w_k", "w_v", "w_o")], gamma=d["gamma_attn"].to(dev))
    mlp = tl.TPLinear(cm, [d[k].to(dev) for k in ("w_gate", "w_up", "w_down")], gamma=d["gamma_mlp"].to(dev))
    return attn, mlp, tl.TPLayer(attn, mlp, max_tokens)


def ref_layer(w, d, cu, residual=True, rows=None):
    return oracle.decoder_layer(d["hidden"], d["residual"] if residual else None, d["gamma_attn"], d["w_q"],
                                d["w_k"], d["w_v"], d["w_o"], d["gamma_mlp"], d["w_gate"], d["w_up"],
                                d["w_down"], w.nq, w.nkv, w.hd, w.t, cu, w.eps, rows=rows)


def rel_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.double().cpu().numpy()
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def status_of(ws: torch.Tensor) -> int:
    torch.cuda.synchronize()
    return int(ws[:4].view(torch.int32).item())


def run(layer, d, lens, residual=True):
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    out = layer.forward(d["hidden"].cuda(), d["residual"].cuda() if residual else None, cu, int(max(lens)))
    return out, cu.cpu().numpy()


def case(H, I, nq, nkv, t, T, seed):
    return workloads.Workload("case", "layer", T=T, H=H, I=I, nq=nq, nkv=nkv, hd=128, t=t, w_std=0.02,
                              norm=True, seed=seed)


@pytest.mark.parametrize("H,I,nq,nkv,t,lens", [
    (512, 1024, 8, 2, 2, [150, 90, 1]),       # prefill path, a one-token sequence
    (512, 1536, 8, 2, 4, [300]),              # t > nkv (kv heads replicated), three query tiles
    (256, 1024, 4, 4, 2, [40, 1, 30]),        # decode-sized step: swapped GEMMs, fused MLP kernel
    (1024, 2048, 16, 4, 4, [128, 128]),       # exact tiles
])
def test_layer_matches_oracle(H, I, nq, nkv, t, lens):
    T = int(sum(lens))
    w = case(H, I, nq, nkv, t, T, seed=len(lens) + t)
    d = workloads.layer_inputs(w)
    attn, mlp, layer = make_layer(w, d, T)
    out, cu = run(layer, d, lens)
    ref = ref_layer(w, d, cu)
    for k in KEYS:
        err = rel_err(out[k], ref[k])
        assert err <= TOL, (k, err)
    assert status_of(layer.workspace()) == 0


def test_first_layer_without_residual():
    lens = [200, 57]
    w = case(512, 1024, 8, 2, 2, sum(lens), seed=5)
    d = workloads.layer_inputs(w)
    attn, mlp, layer = make_layer(w, d, 512)            # T below max_tokens
    out, cu = run(layer, d, lens, residual=False)
    ref = ref_layer(w, d, cu, residual=False)
    for k in KEYS:
        assert rel_err(out[k], ref[k]) <= TOL, k
    assert torch.equal(out["residual_attn"], d["hidden"].cuda())     # r1 = hidden exactly
    assert status_of(layer.workspace()) == 0


def test_layer_equals_its_steps_bit_for_bit():
    # the layer call runs the same kernels as the separate calls, in the same order
    lens = [180, 20]
    T = sum(lens)
    w = case(512, 1024, 8, 2, 2, T, seed=6)
    d = workloads.layer_inputs(w)
    attn, mlp, layer = make_layer(w, d, T)
    out, cu = run(layer, d, lens)
    x1, r1 = tl.add_rms_norm(d["hidden"].cuda(), d["residual"].cuda(), d["gamma_attn"].cuda(), w.eps)
    qkv, _ = attn.attn_proj_forward(x1, None)
    A = attn.attention_forward(qkv, torch.from_numpy(cu).cuda(), max(lens))
    _, attn_out = attn.attn_proj_forward(None, A)
    m = mlp.mlp_forward(attn_out, r1)
    torch.cuda.synchronize()
    assert torch.equal(out["residual_attn"], r1)
    assert torch.equal(out["attn_out"], attn_out)
    assert torch.equal(out["residual_mlp"], m["residual_out"])
    assert torch.equal(out["mlp_out"], m["mlp_out"])
    assert torch.equal(out["residual_stream"], m["residual_stream"])


def test_bad_offsets_reach_the_layer_status_word():
    w = case(256, 1024, 4, 4, 2, 64, seed=7)
    d = workloads.layer_inputs(w)
    attn, mlp, layer = make_layer(w, d, 64)
    ws = layer.workspace()
    cu = torch.tensor([0, 40, 30, 64], dtype=torch.int32, device="cuda")     # falls
    layer.forward(d["hidden"].cuda(), d["residual"].cuda(), cu, 40)
    assert status_of(ws) == tl.TP_ERR_SHAPE
    with pytest.raises(tl.TPError) as e:                                      # T above max_tokens
        layer.forward(torch.zeros(65, 256, dtype=torch.bfloat16, device="cuda"), None,
                      torch.tensor([0, 65], dtype=torch.int32, device="cuda"), 65)
    assert e.value.code == tl.TP_ERR_SHAPE


def test_qwen_ragged_layer_full_size_with_capture():
    w = workloads.WORKLOADS["qwen25_7b_ragged_layer"]
    d = workloads.layer_inputs(w)
    rb = workloads.ragged_batch(w)
    attn, mlp, layer = make_layer(w, d, w.T)
    out, cu = run(layer, d, rb["lens"])
    # two rows of every 128-token tile, plus rows the capture selects
    rows = np.unique(np.concatenate([rb["sel_rows"][:24], tile_rows(w.T, 2)]))
    ref = ref_layer(w, d, cu, rows=rows)
    for k in KEYS:
        assert rel_err(out[k][rows], ref[k]) <= TOL, k
    assert status_of(layer.workspace()) == 0
    # capture behind the layer, in hook-firing order: attn_out, mlp_out, residual_stream
    names = ("attn_out", "mlp_out", "residual_stream")
    types = [workloads.TENSOR_TYPES[n] for n in names]
    rq = torch.from_numpy(rb["row_req"]).cuda()
    rp = torch.from_numpy(rb["row_pos"]).cuda()
    keys = torch.from_numpy(rb["sel_keys"]).cuda()
    cap = 3 * len(rb["sel_rows"])
    hdr, got_rows, n_out, cws = tl.capture_rows(rq, rp, keys, [out[n] for n in names], types, 0, cap)
    torch.cuda.synchronize()
    assert int(n_out.item()) == cap
    want_h, want_r = oracle.capture_rows(rb["row_req"], rb["row_pos"], rb["sel_keys"],
                                         [workloads.bf16_bits(out[n].cpu()) for n in names], types, 0)
    np.testing.assert_array_equal(hdr[:cap, :5].cpu().numpy(), want_h)
    np.testing.assert_array_equal(workloads.bf16_bits(got_rows[:cap].cpu()), want_r)
    assert int(cws[:4].view(torch.int32).item()) == 0


def test_llama3_8b_layer_full_size_every_tile():
    # the first and last row of every 128-token tile and one between: the rows at the
    # end of the sequence make the oracle project all 4096 tokens' q, k and v
    w = workloads.WORKLOADS["llama3_8b_layer_prefill"]
    d = workloads.layer_inputs(w)
    attn, mlp, layer = make_layer(w, d, w.T)
    out, cu = run(layer, d, [w.T])
    rows = [int(r) for r in tile_rows(w.T, 3, seed=1)]
    ref = ref_layer(w, d, cu, rows=rows)
    for k in KEYS:
        assert rel_err(out[k][rows], ref[k]) <= TOL, k
    assert status_of(layer.workspace()) == 0
