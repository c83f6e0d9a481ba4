"""Failure detection without a GPU fault: every on-chip wait is bounded. A short
wait limit makes the fused decode block's waits run out on purpose; the kernel
must report TP_ERR_TIMEOUT in the status word and leave the CUDA context usable
(the same handle then computes the right answer after the workspace is zeroed).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tensor_linear_layers_gb300 as tl

pytestmark = pytest.mark.gpu
f64 = oracle.bf16_to_f64


def test_wait_limit_runs_out_and_context_survives():
    from tensor_linear_layers_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    H, I, t, T = 1024, 4096, 4, 32
    w = workloads.Workload("case", "mlp", T=T, H=H, I=I, t=t, w_std=0.02, norm=True, seed=4)
    d = workloads.mlp_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_MLP, t, H, I, rms_eps=1e-5, flags=tl.TP_FLAG_HAS_NORM)
    blk = tl.TPLinear(cfg, [d["w_gate"].cuda(), d["w_up"].cuda(), d["w_down"].cuda()], gamma=d["gamma"].cuda())
    a, r0 = d["x"].cuda(), d["residual"].cuda()
    ws = torch.zeros(blk.workspace_size(T), dtype=torch.uint8, device="cuda")
    tl.set_wait_timeout(2_000)            # 2 us: the wait for the first accumulator runs out
    try:
        blk.mlp_forward(a, residual=r0, ws=ws)
        torch.cuda.synchronize()          # returns: nothing hung, nothing faulted
        status = int(ws[:4].view(torch.int32).item())
    finally:
        tl.set_wait_timeout(2_000_000_000)
    assert status == tl.TP_ERR_TIMEOUT
    ws.zero_()
    out = blk.mlp_forward(a, residual=r0, ws=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    ref = oracle.mlp_layer(f64(d["x"]), f64(d["w_gate"]), f64(d["w_up"]), f64(d["w_down"]),
                           residual=f64(d["residual"]), gamma=f64(d["gamma"]), eps=1e-5, norm=True)
    g = out["mlp_out"].double().cpu().numpy()
    assert np.max(np.abs(g - ref["mlp_out"])) / np.max(np.abs(ref["mlp_out"])) <= 2e-2


def test_wait_limit_rejects_nonpositive():
    with pytest.raises(tl.TPError) as e:
        tl.set_wait_timeout(0)
    assert e.value.code == tl.TP_ERR_ARG
