"""Parity of the MoE block (tp_moe_forward, through the C ABI) with the oracle.

Tolerance as for the dense block: normwise max|gpu - ref| / max|ref| <= 2e-2
(bf16 in, fp32 accumulate; each expert's h and output are rounded to bf16, the
gate-weighted sum is taken in fp32 and rounded once). Cases: several experts
per 128-row tile boundary, an expert that receives no token, top_k equal to
the expert count, t = 1 .. 4 within-expert splits, the Mixtral-shaped block at
full size (decode in full, prefill on sampled tokens), ids out of range, and
determinism.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tensor_linear_layers_gb300 as tl
from tile_rows import moe_tile_tokens

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from tensor_linear_layers_gb300 import _build
    _build.build()
    tl.lib()
    torch.cuda.set_device(0)


def make(w, d):
    cfg = tl.make_config(tl.TP_BLOCK_MOE, w.t, w.H, w.I, n_experts=w.experts)
    ws = []
    for e in range(w.experts):
        ws += [d["w_gate"][e].cuda(), d["w_up"][e].cuda(), d["w_down"][e].cuda()]
    return tl.TPLinear(cfg, ws)


def run(blk, d, rows=None):
    x, ids, g = d["x"], d["expert_ids"], d["gates"]
    return blk.moe_forward(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(g).cuda())


def rel_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.double().cpu().numpy()
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def status_of(blk, N) -> int:
    torch.cuda.synchronize()
    return int(blk.workspace(N)[:4].view(torch.int32).item())


def case(T, H, I, E, k, t, seed=0):
    return workloads.Workload("case", "moe", T=T, H=H, I=I, t=t, w_std=0.02, experts=E, top_k=k, seed=seed)


@pytest.mark.parametrize("T,H,I,E,k,t", [
    (37, 256, 512, 4, 2, 2),       # few rows per expert, all in one tile each
    (300, 512, 1024, 8, 2, 4),     # experts spanning several tiles
    (5, 256, 512, 3, 3, 1),        # top_k = every expert, t = 1
    (200, 256, 768, 6, 1, 2),      # top-1: skewed load, some experts nearly empty
])
def test_moe_matches_oracle(T, H, I, E, k, t):
    w = case(T, H, I, E, k, t, seed=T)
    d = workloads.moe_inputs(w)
    blk = make(w, d)
    y = run(blk, d)
    ref = oracle.moe_block(d["x"], d["expert_ids"], d["gates"], d["w_gate"], d["w_up"], d["w_down"])
    assert rel_err(y, ref) <= TOL
    assert status_of(blk, T * k) == 0


def test_expert_without_tokens():
    w = case(64, 256, 512, 4, 1, 2, seed=1)
    d = workloads.moe_inputs(w)
    d["expert_ids"][:] = np.where(d["expert_ids"] == 2, 3, d["expert_ids"])   # expert 2 gets nothing
    blk = make(w, d)
    y = run(blk, d)
    ref = oracle.moe_block(d["x"], d["expert_ids"], d["gates"], d["w_gate"], d["w_up"], d["w_down"])
    assert rel_err(y, ref) <= TOL


def test_mixtral_decode_full():
    w = workloads.WORKLOADS["mixtral_8x7b_moe_decode"]
    d = workloads.moe_inputs(w)
    blk = make(w, d)
    y = run(blk, d)
    ref = oracle.moe_block(d["x"], d["expert_ids"], d["gates"], d["w_gate"], d["w_up"], d["w_down"])
    assert rel_err(y, ref) <= TOL
    assert status_of(blk, w.T * w.top_k) == 0


def test_mixtral_prefill_every_expert_tile():
    w = workloads.WORKLOADS["mixtral_8x7b_moe_prefill"]
    d = workloads.moe_inputs(w)
    blk = make(w, d)
    y = run(blk, d)
    # tokens routed into every 128-row tile of every expert (both tiles of each CTA
    # pair, each expert's last partial tile)
    rows = moe_tile_tokens(d["expert_ids"], per_tile=2)
    ref = oracle.moe_block(d["x"][rows], d["expert_ids"][rows], d["gates"][rows], d["w_gate"], d["w_up"],
                           d["w_down"])
    assert rel_err(y[rows], ref) <= TOL
    assert status_of(blk, w.T * w.top_k) == 0


def test_run_twice_same_bits():
    w = case(300, 512, 1024, 8, 2, 4, seed=3)
    d = workloads.moe_inputs(w)
    blk = make(w, d)
    assert torch.equal(run(blk, d), run(blk, d))


def test_ids_out_of_range_report_shape_error():
    w = case(16, 256, 512, 4, 2, 2, seed=4)
    d = workloads.moe_inputs(w)
    blk = make(w, d)
    bad = dict(d, expert_ids=d["expert_ids"].copy())
    bad["expert_ids"][3, 1] = 4
    y = run(blk, bad)
    assert status_of(blk, 32) == tl.TP_ERR_SHAPE
    assert torch.count_nonzero(y).item() == 0
    blk.workspace(32).zero_()
    y = run(blk, d)                                           # the handle still works
    ref = oracle.moe_block(d["x"], d["expert_ids"], d["gates"], d["w_gate"], d["w_up"], d["w_down"])
    assert rel_err(y, ref) <= TOL
    assert status_of(blk, 32) == 0
