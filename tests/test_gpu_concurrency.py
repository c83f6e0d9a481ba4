"""The fused decode block next to other work on the same GPU.

The block is one launch of one CTA per SM whose CTAs hand work to one another
(norm rows to gate_up, h tiles to down, down partials between splits). It must
not rely on all its CTAs being resident at once: another kernel on another
stream may hold SMs for longer than the on-chip wait limit. Here a helper kernel
holds 100 of the SMs for 400 ms while the block runs on the rest, with the wait
limit cut to 50 ms; the block must finish within that time with status 0 and
match the float64 oracle (normwise max relative error <= 2e-2).
"""
import ctypes
import os
import subprocess
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
import tensor_linear_layers_gb300 as tl

pytestmark = pytest.mark.gpu
TOL = 2e-2
HERE = os.path.dirname(os.path.abspath(__file__))
OCCUPY_NS = 400_000_000
OCCUPY_BLOCKS = 100


@pytest.fixture(scope="module")
def occupier(tmp_path_factory):
    from tensor_linear_layers_gb300 import _build
    _build.build()
    tl.lib()
    torch.cuda.set_device(0)
    so = str(tmp_path_factory.mktemp("occupy") / "occupy_sms.so")
    subprocess.run([_build.nvcc(), *_build.ARCH, "-O2", "-shared", "-Xcompiler", "-fPIC",
                    os.path.join(HERE, "occupy_sms.cu"), "-o", so], check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    lib.occupy_sms.argtypes = [ctypes.c_int, ctypes.c_ulonglong, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.occupy_sms.restype = ctypes.c_int
    return lib


def rel_err(got, ref):
    g = got.double().cpu().numpy()
    return float(np.max(np.abs(g - ref)) / np.max(np.abs(ref)))


@pytest.mark.parametrize("H,I,t,T", [
    (4096, 14336, 8, 32),     # the Llama-3-8B decode shape: gate_up without split-K
    (1024, 4096, 4, 32),      # few gate_up tiles: gate_up with split-K
])
def test_fused_decode_beside_a_kernel_holding_most_sms(occupier, H, I, t, T):
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    assert nsm > OCCUPY_BLOCKS
    w = workloads.Workload("case", "mlp", T=T, H=H, I=I, t=t, w_std=0.02, norm=True, seed=21)
    d = workloads.mlp_inputs(w)
    cfg = tl.make_config(tl.TP_BLOCK_MLP, t, H, I, rms_eps=1e-5, flags=tl.TP_FLAG_HAS_NORM)
    blk = tl.TPLinear(cfg, [d["w_gate"].cuda(), d["w_up"].cuda(), d["w_down"].cuda()], gamma=d["gamma"].cuda())
    assert blk.plan(T)[0]["engine"] == 2
    a, r0 = d["x"].cuda(), d["residual"].cuda()
    ws = blk.workspace(T)
    for _ in range(3):                                 # ordinary launches first: the counters move on
        blk.mlp_forward(a, residual=r0, ws=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0

    started = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    tl.set_wait_timeout(50_000_000)
    try:
        rc = occupier.occupy_sms(OCCUPY_BLOCKS, OCCUPY_NS, 120 * 1024, ctypes.c_void_p(started.data_ptr()),
                                 ctypes.c_void_p(side.cuda_stream))
        assert rc == 0
        time.sleep(0.05)                               # the helper's blocks are running by now
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        out = blk.mlp_forward(a, residual=r0, ws=ws)
        e1.record()
        e1.synchronize()
        busy = not side.query()                        # the helper still holds its SMs
        ms = e0.elapsed_time(e1)
    finally:
        torch.cuda.synchronize()
        tl.set_wait_timeout(2_000_000_000)
    assert int(started.item()) == OCCUPY_BLOCKS
    assert busy, "the block finished only after the helper kernel"
    assert ms < OCCUPY_NS / 1e6
    assert int(ws[:4].view(torch.int32).item()) == 0
    ref = oracle.mlp_layer(oracle.bf16_to_f64(d["x"]), oracle.bf16_to_f64(d["w_gate"]), oracle.bf16_to_f64(d["w_up"]),
                           oracle.bf16_to_f64(d["w_down"]), residual=oracle.bf16_to_f64(d["residual"]),
                           gamma=oracle.bf16_to_f64(d["gamma"]), eps=1e-5, norm=True)
    for k in ("mlp_out", "residual_out", "residual_stream"):
        assert rel_err(out[k], ref[k]) <= TOL, k
    # and the launches after it are ordinary again
    out2 = blk.mlp_forward(a, residual=r0, ws=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    assert torch.equal(out2["mlp_out"], out["mlp_out"])
