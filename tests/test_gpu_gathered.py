"""The gathered activation layout (TP_FLAG_GATHERED: gather_output=True on the
column-parallel side, input_is_parallel=False on the row-parallel side).

"vLLM 源码完全拆解（十一）" ColumnParallelLinear: with gather_output the shards'
outputs are concatenated along the feature dimension, which by the column-split
identity is the unsharded output; RowParallelLinear with input_is_parallel=False
takes that full input and uses its own columns. Only addresses differ from the
shard-major layout, so every result must be bit-identical to it (checked for
each call, prefill- and decode-sized), and the gathered column output must match
the oracle's unsharded definition.
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


def shard_to_gathered(x: torch.Tensor) -> torch.Tensor:
    """[t][T][w] -> [T][t * w]."""
    t, T, w = x.shape
    return x.permute(1, 0, 2).reshape(T, t * w)


def rel_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.double().cpu().numpy()
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def mlp_pair(T, H=512, I=1536, t=4, norm=False):
    w = workloads.Workload("case", "mlp", T=T, H=H, I=I, t=t, w_std=0.02, norm=norm, seed=T)
    d = workloads.mlp_inputs(w)
    flags = tl.TP_FLAG_HAS_NORM if norm else 0
    ws = [d[k].cuda() for k in ("w_gate", "w_up", "w_down")]
    g = None if d["gamma"] is None else d["gamma"].cuda()
    a = tl.TPLinear(tl.make_config(tl.TP_BLOCK_MLP, t, H, I, flags=flags), ws, gamma=g)
    b = tl.TPLinear(tl.make_config(tl.TP_BLOCK_MLP, t, H, I, flags=flags | tl.TP_FLAG_GATHERED), ws, gamma=g)
    return w, d, a, b


@pytest.mark.parametrize("T", [300, 40])
def test_gate_up_and_down_gathered(T):
    w, d, shard, gath = mlp_pair(T)
    x = d["x"].cuda()
    h_s = shard.gate_up(x)
    h_g = gath.gate_up(x)
    torch.cuda.synchronize()
    assert h_g.shape == (T, w.I)
    assert torch.equal(h_g, shard_to_gathered(h_s))
    # the gathered h is the unsharded silu(x Wg) * (x Wu)
    X = f64(d["x"])
    ref = oracle.silu_mul(oracle.linear(X, f64(d["w_gate"])), oracle.linear(X, f64(d["w_up"])))
    assert rel_err(h_g, ref) <= TOL
    y_s, _ = shard.down(h_s)
    y_g, _ = gath.down(h_g)
    torch.cuda.synchronize()
    assert torch.equal(y_s, y_g)


@pytest.mark.parametrize("T", [300, 40])
def test_mlp_forward_gathered_equals_shard_major(T):
    w, d, shard, gath = mlp_pair(T, norm=True)
    x, r = d["x"].cuda(), d["residual"].cuda()
    a = shard.mlp_forward(x, r)
    b = gath.mlp_forward(x, r)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def attn_pair(H=512, nq=8, nkv=2, t=4, flags=0):
    w = workloads.Workload("case", "attn", T=1, H=H, nq=nq, nkv=nkv, hd=128, t=t, w_std=0.02, seed=3)
    d = workloads.attn_inputs(w, T=1)
    ws = [d[k].cuda() for k in ("w_q", "w_k", "w_v", "w_o")]
    mk = lambda f: tl.TPLinear(tl.make_config(tl.TP_BLOCK_ATTN_PROJ, t, H, n_q_heads=nq, n_kv_heads=nkv,
                                              head_dim=128, flags=f), ws)
    return w, d, mk(flags), mk(flags | tl.TP_FLAG_GATHERED)


@pytest.mark.parametrize("T", [300, 40])
def test_attention_projections_gathered(T):
    w, d, shard, gath = attn_pair()
    x = workloads.draw((T, w.H), 20 + T, 0).cuda()
    A = workloads.draw((w.t, T, w.nq * 128 // w.t), 20 + T, 1).cuda()
    q_s, o_s = shard.attn_proj_forward(x, A)
    q_g, o_g = gath.attn_proj_forward(x, shard_to_gathered(A).contiguous())
    torch.cuda.synchronize()
    assert torch.equal(q_g, shard_to_gathered(q_s))
    assert torch.equal(o_g, o_s)
    ref = oracle.qkv_parallel(f64(x.cpu()), f64(d["w_q"]), f64(d["w_k"]), f64(d["w_v"]), w.nq, w.nkv, 128, w.t)
    assert rel_err(q_g, np.concatenate(list(ref), axis=1)) <= TOL


def test_attention_core_gathered():
    w, d, shard, gath = attn_pair(nq=8, nkv=2, t=2)
    lens = [200, 1, 99]
    T = sum(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    qkv = workloads.draw((w.t, T, (w.nq // w.t + 2 * (w.nkv // w.t)) * 128), 31, 0).cuda()
    a_s = shard.attention_forward(qkv, cu, max(lens))
    a_g = gath.attention_forward(shard_to_gathered(qkv).contiguous(), cu, max(lens))
    torch.cuda.synchronize()
    assert a_g.shape == (T, w.nq * 128)
    assert torch.equal(a_g, shard_to_gathered(a_s))


def test_decoder_layer_gathered_equals_shard_major():
    H, I, nq, nkv, t, lens = 512, 1024, 8, 2, 2, [150, 40]
    T = sum(lens)
    w = workloads.Workload("case", "layer", T=T, H=H, I=I, nq=nq, nkv=nkv, hd=128, t=t, w_std=0.02,
                           norm=True, seed=9)
    d = workloads.layer_inputs(w)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    outs = []
    for extra in (0, tl.TP_FLAG_GATHERED):
        ca = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, t, H, n_q_heads=nq, n_kv_heads=nkv, head_dim=128,
                            flags=tl.TP_FLAG_HAS_NORM | extra)
        cm = tl.make_config(tl.TP_BLOCK_MLP, t, H, I, flags=tl.TP_FLAG_HAS_NORM | extra)
        attn = tl.TPLinear(ca, [d[k].cuda() for k in ("w_q", "w_k", "w_v", "w_o")], gamma=d["gamma_attn"].cuda())
        mlp = tl.TPLinear(cm, [d[k].cuda() for k in ("w_gate", "w_up", "w_down")], gamma=d["gamma_mlp"].cuda())
        layer = tl.TPLayer(attn, mlp, T)
        outs.append((layer.forward(d["hidden"].cuda(), d["residual"].cuda(), cu, max(lens)), attn, mlp, layer))
    torch.cuda.synchronize()
    for k in outs[0][0]:
        assert torch.equal(outs[0][0][k], outs[1][0][k]), k
