"""tp_mlp_forward_no_alloc: the fused decode-shaped MLP block for callers that
cannot allocate device memory (plug-ins that only get memory their host
planned, runtimes whose own allocator owns the device, loops that forbid
allocation after start-up). Its scratch is a fixed array inside the library.
The tests call it through the C ABI and compare it with the float64 oracle
(normwise max relative error <= 2e-2) and, bit for bit, with tp_mlp_forward,
which runs the same kernel with the same plans on a caller-provided workspace:
two calls in a row, then calls that alternate between two handles (the array
then holds the other handle's counters and is cleared first). This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tensor_linear_layers_gb300 as tl

pytestmark = pytest.mark.gpu
TOL = 2e-2
KEYS = ("mlp_out", "residual_out", "residual_stream")
f64 = oracle.bf16_to_f64


def rel_err(got, ref):
    g = got.double().cpu().numpy()
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def make(w):
    d = workloads.mlp_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_MLP, w.t, w.H, w.I, rms_eps=w.eps, flags=tl.TP_FLAG_HAS_NORM)
    blk = tl.TPLinear(cfg, [d["w_gate"].cuda(), d["w_up"].cuda(), d["w_down"].cuda()], gamma=d["gamma"].cuda())
    return d, blk


def oracle_out(d, x, r):
    return oracle.mlp_layer(f64(x), f64(d["w_gate"]), f64(d["w_up"]), f64(d["w_down"]), residual=f64(r),
                            gamma=f64(d["gamma"]), eps=1e-5, norm=True)


@pytest.fixture(scope="module")
def block():
    from tensor_linear_layers_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    w = workloads.WORKLOADS["llama3_8b_mlp_decode"]
    d, blk = make(w)
    return w, d, blk


def test_no_alloc_matches_oracle_and_workspace_path_twice(block):
    w, d, blk = block
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        # another input in the second call: the shared scratch must not leak the first call's state
        x = d["x"] if call == 0 else workloads.draw((w.T, w.H), 77, 0)
        r = d["residual"] if call == 0 else workloads.draw((w.T, w.H), 77, 1)
        out = blk.mlp_forward_no_alloc(x.cuda(), residual=r.cuda(), status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        ref = oracle_out(d, x, r)
        for k in KEYS:
            assert rel_err(out[k], ref[k]) <= TOL, (call, k)
        # same kernel, same plans, fixed summation order: the same bits as with a workspace
        ws_out = blk.mlp_forward(x.cuda(), residual=r.cuda())
        torch.cuda.synchronize()
        for k in KEYS:
            assert torch.equal(out[k], ws_out[k]), (call, k)


def test_no_alloc_alternating_handles(block):
    w, d, blk = block
    w2 = workloads.Workload("small", "mlp", T=16, H=1024, I=4096, t=4, w_std=0.02, norm=True, seed=5)
    d2, blk2 = make(w2)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for which in (0, 1, 0, 1):
        dd, b, ww = (d, blk, w) if which == 0 else (d2, blk2, w2)
        out = b.mlp_forward_no_alloc(dd["x"].cuda(), residual=dd["residual"].cuda(), status=status)
        ref = b.mlp_forward(dd["x"].cuda(), residual=dd["residual"].cuda())
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for k in KEYS:
            assert torch.equal(out[k], ref[k]), (which, k)


def test_no_alloc_rejects_what_does_not_fit(block):
    w, d, blk = block
    x = torch.zeros(129, w.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tl.TPError) as e:
        blk.mlp_forward_no_alloc(x, residual=x.clone())
    assert e.value.code == tl.TP_ERR_UNSUPPORTED
    # T <= 128 but h alone (128 x 131072 bf16 = 32 MiB) is over the fixed 16 MiB
    H, I = 512, 131072
    z = [torch.zeros(I, H, dtype=torch.bfloat16, device="cuda"), torch.zeros(I, H, dtype=torch.bfloat16, device="cuda"),
         torch.zeros(H, I, dtype=torch.bfloat16, device="cuda")]
    cfg = tl.make_config(tl.TP_BLOCK_MLP, 1, H, I, flags=tl.TP_FLAG_HAS_NORM)
    big = tl.TPLinear(cfg, z, gamma=torch.ones(H, dtype=torch.bfloat16, device="cuda"))
    x = torch.zeros(128, H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tl.TPError) as e:
        big.mlp_forward_no_alloc(x, residual=x.clone())
    assert e.value.code == tl.TP_ERR_UNSUPPORTED
    assert "bytes of scratch" in str(e.value) and str(16 << 20) in str(e.value)


def test_no_alloc_status_argument_is_checked(block):
    w, d, blk = block
    x = d["x"].cuda()
    for bad in (torch.zeros(1, dtype=torch.float32, device="cuda"), torch.zeros(1, dtype=torch.int32),
                torch.zeros(0, dtype=torch.int32, device="cuda")):
        with pytest.raises(ValueError):
            blk.mlp_forward_no_alloc(x, residual=d["residual"].cuda(), status=bad)
