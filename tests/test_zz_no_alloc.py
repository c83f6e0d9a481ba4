"""tp_mlp_forward_no_alloc: the fused decode-shaped MLP block for callers that
cannot allocate device memory (plug-ins that only get memory their host
planned, runtimes whose own allocator owns the device, loops that forbid
allocation after start-up). Its scratch is a fixed array inside the library,
so the test calls it through the C ABI and compares it with tp_mlp_forward,
which runs the same kernel on a caller-provided workspace, on two calls in a
row. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import workloads
import tensor_linear_layers_gb300 as tl

pytestmark = pytest.mark.gpu
TOL = 2e-2


def rel_err(got, ref):
    g, r = got.double().cpu().numpy(), ref.double().cpu().numpy()
    return float(np.max(np.abs(g - r)) / max(np.max(np.abs(r)), 1e-30))


@pytest.fixture(scope="module")
def block():
    from tensor_linear_layers_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    w = workloads.WORKLOADS["llama3_8b_mlp_decode"]
    d = workloads.mlp_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_MLP, w.t, w.H, w.I, rms_eps=w.eps, flags=tl.TP_FLAG_HAS_NORM)
    blk = tl.TPLinear(cfg, [d["w_gate"].cuda(), d["w_up"].cuda(), d["w_down"].cuda()], gamma=d["gamma"].cuda())
    return w, d, blk


def test_no_alloc_matches_workspace_path_twice(block):
    w, d, blk = block
    ref = blk.mlp_forward(d["x"].cuda(), residual=d["residual"].cuda())
    torch.cuda.synchronize()
    assert int(blk.workspace(w.T)[:4].view(torch.int32).item()) == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        # a second input in the second call: the shared scratch must not leak the first call's state
        x = d["x"].cuda() if call == 0 else workloads.draw((w.T, w.H), 77, 0).cuda()
        r = d["residual"].cuda() if call == 0 else workloads.draw((w.T, w.H), 77, 1).cuda()
        if call == 1:
            ref = blk.mlp_forward(x, residual=r)
        out = blk.mlp_forward_no_alloc(x, residual=r, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        for k in ("mlp_out", "residual_out", "residual_stream"):
            assert rel_err(out[k], ref[k]) <= TOL, (call, k)


def test_no_alloc_rejects_what_does_not_fit(block):
    w, d, blk = block
    x = torch.zeros(129, w.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tl.TPError) as e:
        blk.mlp_forward_no_alloc(x, residual=x.clone())
    assert e.value.code == tl.TP_ERR_UNSUPPORTED
