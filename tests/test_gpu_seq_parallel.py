"""Sequence-parallel end of the row-parallel layers (reduce-scatter by token).

With sequence parallelism the all-reduce after a row-parallel layer becomes a
reduce-scatter: rank r keeps the reduced rows [r*T/t, (r+1)*T/t), the token
count padded to a multiple of t ("Tensor Parallelism", collectives;
"Tensor & pipeline parallelism", residual_stream). On one GPU the reduction
is on chip and the scatter is a view: the [T][H] output, in a buffer of
t * ceil(T/t) zeroed rows, read as [t][ceil(T/t)][H]. These tests check that
view against the oracle's reduce_scatter for down and o_proj, with and
without padding.
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


def check_slices(buf: torch.Tensor, ref_slices, t: int):
    per = ref_slices[0].shape[0]
    got = buf.view(t, per, -1).double().cpu().numpy()
    top = max(np.max(np.abs(s)) for s in ref_slices)
    for r in range(t):
        assert float(np.max(np.abs(got[r] - ref_slices[r]))) / top <= TOL, r


@pytest.mark.parametrize("T,t", [(256, 4), (300, 8), (37, 4)])
def test_down_reduce_scatter(T, t):
    H, I = 512, 1024
    w = workloads.Workload("case", "mlp", T=T, H=H, I=I, t=t, w_std=0.02, seed=T + t)
    d = workloads.mlp_inputs(w)
    blk = tl.TPLinear(tl.make_config(tl.TP_BLOCK_MLP, t, H, I), [d[k].cuda() for k in ("w_gate", "w_up", "w_down")])
    h = workloads.draw((t, T, I // t), 40 + T, 0).cuda()
    per = -(-T // t)
    buf = torch.zeros(per * t, H, dtype=torch.bfloat16, device="cuda")
    blk.down(h, out=buf[:T])
    torch.cuda.synchronize()
    hf = np.concatenate(list(f64(h.cpu())), axis=1)
    ref = oracle.reduce_scatter(oracle.row_parallel(hf, f64(d["w_down"]), t), t)
    check_slices(buf, ref, t)


def test_o_proj_reduce_scatter():
    T, H, nq, nkv, t = 200, 512, 8, 2, 4
    w = workloads.Workload("case", "attn", T=T, H=H, nq=nq, nkv=nkv, hd=128, t=t, w_std=0.02, seed=4)
    d = workloads.attn_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, t, H, n_q_heads=nq, n_kv_heads=nkv, head_dim=128)
    blk = tl.TPLinear(cfg, [d[k].cuda() for k in ("w_q", "w_k", "w_v", "w_o")])
    per = -(-T // t)
    buf = torch.zeros(per * t, H, dtype=torch.bfloat16, device="cuda")
    blk.attn_proj_forward(None, d["attn"].cuda(), o_out=buf[:T])
    torch.cuda.synchronize()
    A = np.concatenate(list(f64(d["attn"])), axis=1)
    ref = oracle.reduce_scatter(oracle.row_parallel(A, f64(d["w_o"]), t), t)
    check_slices(buf, ref, t)
