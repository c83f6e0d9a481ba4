"""Seeded synthetic inputs for the tensor-parallel decoder linear block.

This module only draws random numbers and lays them out in the shapes of the
Llama/Qwen-shaped workloads. It holds none of the block's arithmetic: no
matmul, no activation, no normalisation, no sharding. Both the float64 oracle
(``oracle/``) and the CUDA path (``tensor_linear_layers_gb300``) take their
inputs from here, and nothing else is shared between them.

Recipe (all draws are float32 from ``torch`` CPU generators, rounded to bf16
by round-to-nearest-even with ``Tensor.to(torch.bfloat16)``):

* Every tensor is drawn in chunks of ``CHUNK`` elements. Chunk ``c`` of the
  tensor with index ``i`` in the draw order uses a fresh generator seeded with
  ``seed * 1_000_003 + i * 65_537 + c``, so a tensor is reproducible from
  ``(seed, i)`` alone and the chunks can be drawn on several threads.
* Draw order: activations, residual, weights (gate, up, down -- or q, k, v,
  o), gamma. Weights ~ N(0, w_std), activations ~ N(0, 1),
  gamma ~ U(0.9, 1.1).
* Weights use the ``nn.Linear`` layout [out_features, in_features].

The ragged continuous batch (Qwen2.5-7B-shaped workload) follows the reading
given in the design notes: request lengths ~ Geometric(1/mean_len) from
``numpy.random.default_rng(seed)``, the longest request absorbs the difference
to the token total, a 1-token request is a decode step whose token position is
its context length, and 10 % of the rows are selected for capture.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

CHUNK = 1 << 22

# tensor_type codes of the capture records (hook targets of the capture page)
TENSOR_TYPES = {"residual_stream": 0, "attn_out": 1, "mlp_out": 2, "final_norm": 3}


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "mlp", "attn", "attn_core", "layer", "moe" or "paged" (KV-cache decode attention)
    T: int                    # tokens in the step
    H: int                    # hidden size
    t: int                    # logical tensor-parallel shards
    w_std: float
    I: int = 0                # intermediate size (mlp)
    nq: int = 0               # q heads (attn)
    nkv: int = 0              # kv heads (attn)
    hd: int = 0               # head dim (attn)
    norm: bool = False        # fused residual-add + RMSNorm in front of the MLP
    eps: float = 1e-5
    requests: int = 0         # ragged batch: number of requests (0 = not ragged)
    mean_len: int = 0
    capture_frac: float = 0.0
    experts: int = 0          # moe: experts (each an MLP of intermediate size I)
    top_k: int = 0            # moe: experts per token
    seed: int = 0
    desc: str = field(default="", compare=False)

    def seq_lens(self) -> np.ndarray:
        """Lengths of the packed sequences (attention core): one sequence, or the ragged batch.
        Paged decode: each request's tokens (cached context + its new one), U[256, 4096]."""
        if self.kind == "paged":
            return np.random.default_rng(self.seed + 11).integers(256, 4097, self.T).astype(np.int64)
        return ragged_batch(self)["lens"] if self.requests else np.array([self.T], dtype=np.int64)

    def kv_cache_bytes(self) -> int:
        """Keys and values the paged decode step reads: every request's tokens, all kv heads."""
        return int(self.seq_lens().sum()) * 2 * self.nkv * self.hd * 2

    def attn_core_flops(self) -> float:
        """q k^T and p v over the causal (query, key) pairs of every sequence and q head."""
        L = self.seq_lens().astype(np.float64)
        return 4.0 * self.hd * self.nq * float(np.sum(L * (L + 1) / 2))

    def mlp_flops(self) -> float:
        return 2.0 * self.T * self.H * (2 * self.I) + 2.0 * self.T * self.I * self.H

    def proj_flops(self) -> float:
        qkv_n = (self.nq + 2 * self.nkv) * self.hd
        return 2.0 * self.T * self.H * qkv_n + 2.0 * self.T * self.nq * self.hd * self.H

    def flops(self) -> float:
        if self.kind == "paged":              # q.k and p.v of each request's new token over its tokens
            return 4.0 * self.hd * self.nq * float(self.seq_lens().sum())
        if self.kind == "moe":                # every routed (token, expert) entry through one expert MLP
            return self.top_k * self.mlp_flops()
        if self.kind == "attn_core":
            return self.attn_core_flops()
        if self.kind == "mlp":
            return self.mlp_flops()
        if self.kind == "layer":
            return self.proj_flops() + self.attn_core_flops() + self.mlp_flops()
        return self.proj_flops()

    def weight_bytes(self) -> int:
        proj = 2 * (self.H * (self.nq + 2 * self.nkv) * self.hd + self.nq * self.hd * self.H)
        if self.kind == "attn_core":
            return 0
        if self.kind == "paged":              # the KV cache streamed per step stands in for weights
            return self.kv_cache_bytes()
        if self.kind == "moe":
            return self.experts * 2 * 3 * self.H * self.I
        if self.kind == "mlp":
            return 2 * 3 * self.H * self.I
        if self.kind == "layer":
            return proj + 2 * 3 * self.H * self.I
        return proj

    def activation_bytes(self) -> int:
        """Bytes of activations read or written once by the whole block."""
        T, H = self.T, self.H
        if self.kind == "attn_core":       # qkv in, attention output out
            return 2 * T * (self.nq + 2 * self.nkv) * self.hd + 2 * T * self.nq * self.hd
        if self.kind == "layer":             # hidden, residual in; r1, attn_out, r2, mlp_out, stream out
            return 2 * T * H * 7
        if self.kind == "moe":               # x in, y out
            return 2 * T * H * 2
        if self.kind == "paged":             # each request's new qkv row in, attention row out
            return 2 * T * ((self.nq + 2 * self.nkv) * self.hd + self.nq * self.hd)
        if self.kind == "mlp":
            b = 2 * T * H * 2                # x (or a) in, mlp_out
            if self.norm:
                b += 2 * T * H * 3           # residual in, residual out, residual_stream
            return b
        qkv_n = (self.nq + 2 * self.nkv) * self.hd
        return 2 * T * H + 2 * T * qkv_n + 2 * T * self.nq * self.hd + 2 * T * H


WORKLOADS = {
    "tiny_mlp": Workload(
        "tiny_mlp", "mlp", T=16, H=512, I=1408, t=2, w_std=0.02,
        desc="Tiny Llama-style MLP block, 16 tokens, t=2"),
    "llama3_8b_mlp_decode": Workload(
        "llama3_8b_mlp_decode", "mlp", T=32, H=4096, I=14336, t=8, w_std=0.02, norm=True,
        desc="Llama-3-8B-shaped MLP decode, 32 tokens, t=8, residual add + RMSNorm"),
    "llama3_8b_attn_proj_prefill": Workload(
        "llama3_8b_attn_proj_prefill", "attn", T=4096, H=4096, nq=32, nkv=8, hd=128, t=4,
        w_std=0.02, desc="Llama-3-8B-shaped QKV + o_proj prefill, 4096 tokens, t=4"),
    "llama3_8b_attn_core_prefill": Workload(
        "llama3_8b_attn_core_prefill", "attn_core", T=4096, H=4096, nq=32, nkv=8, hd=128, t=4,
        w_std=0.0, desc="Llama-3-8B-shaped causal GQA attention core, one 4096-token sequence, t=4"),
    "qwen25_7b_ragged_attn_core": Workload(
        "qwen25_7b_ragged_attn_core", "attn_core", T=2048, H=3584, nq=28, nkv=4, hd=128, t=4,
        w_std=0.0, requests=64, mean_len=32,
        desc="Ragged continuous batch, Qwen2.5-7B-shaped attention core, 2048 tokens / 64 requests, t=4"),
    "llama3_8b_layer_prefill": Workload(
        "llama3_8b_layer_prefill", "layer", T=4096, H=4096, I=14336, nq=32, nkv=8, hd=128, t=4,
        w_std=0.02, norm=True,
        desc="Llama-3-8B-shaped decoder layer prefill (norm, QKV, attention, o_proj, add + norm, MLP), "
             "one 4096-token sequence, t=4"),
    "qwen25_7b_ragged_layer": Workload(
        "qwen25_7b_ragged_layer", "layer", T=2048, H=3584, I=18944, nq=28, nkv=4, hd=128, t=4,
        w_std=0.02, norm=True, requests=64, mean_len=32, capture_frac=0.1,
        desc="Ragged continuous batch, Qwen2.5-7B-shaped decoder layer with attn_out / mlp_out / "
             "residual_stream capture, 2048 tokens / 64 requests, t=4"),
    "llama3_8b_paged_decode": Workload(
        "llama3_8b_paged_decode", "paged", T=32, H=4096, nq=32, nkv=8, hd=128, t=4, w_std=0.0,
        desc="Llama-3-8B-shaped decode attention over a paged KV cache, 32 requests of 256-4096 tokens "
             "(block size 16), one new token each, t=4"),
    "mixtral_8x7b_moe_prefill": Workload(
        "mixtral_8x7b_moe_prefill", "moe", T=4096, H=4096, I=14336, t=4, w_std=0.02, experts=8, top_k=2,
        desc="Mixtral-8x7B-shaped MoE block prefill, 4096 tokens, top-2 of 8 experts, each expert split t=4"),
    "mixtral_8x7b_moe_decode": Workload(
        "mixtral_8x7b_moe_decode", "moe", T=32, H=4096, I=14336, t=4, w_std=0.02, experts=8, top_k=2,
        desc="Mixtral-8x7B-shaped MoE block decode, 32 tokens, top-2 of 8 experts, each expert split t=4"),
    "llama3_70b_mlp_prefill": Workload(
        "llama3_70b_mlp_prefill", "mlp", T=8192, H=8192, I=28672, t=8, w_std=0.015,
        desc="Llama-3-70B-shaped MLP prefill, 8192 tokens, t=8"),
    "qwen25_7b_ragged_mlp": Workload(
        "qwen25_7b_ragged_mlp", "mlp", T=2048, H=3584, I=18944, t=4, w_std=0.02, norm=True,
        requests=64, mean_len=32, capture_frac=0.1,
        desc="Ragged continuous batch, Qwen2.5-7B-shaped MLP, 2048 tokens / 64 requests, t=4"),
}


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _chunk_seed(seed: int, index: int, chunk: int) -> int:
    return (seed * 1_000_003 + index * 65_537 + chunk) & 0x7FFF_FFFF_FFFF_FFFF


def draw(shape, seed: int, index: int, kind: str = "normal", a: float = 0.0, b: float = 1.0,
         dtype=torch.bfloat16) -> torch.Tensor:
    """Draw one seeded tensor of ``shape`` on the CPU.

    kind="normal": N(a, b) (mean a, std b); kind="uniform": U(a, b).
    """
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=dtype)
    nchunks = max(1, math.ceil(n / CHUNK))

    def one(c: int) -> None:
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        if hi <= lo:
            return
        g = torch.Generator().manual_seed(_chunk_seed(seed, index, c))
        if kind == "normal":
            v = torch.randn(hi - lo, generator=g) * b + a
        elif kind == "uniform":
            v = torch.rand(hi - lo, generator=g) * (b - a) + a
        else:
            raise ValueError(kind)
        out[lo:hi] = v.to(dtype)

    if nchunks == 1:
        one(0)
    else:
        with ThreadPoolExecutor(min(_threads(), nchunks)) as ex:
            list(ex.map(one, range(nchunks)))
    return out.reshape(shape)


def mlp_inputs(w: Workload, T: int | None = None) -> dict:
    """Inputs of an MLP block: activations, residual, gate/up/down weights, gamma."""
    T = w.T if T is None else T
    H, I, s = w.H, w.I, w.seed
    d = {"x": draw((T, H), s, 0)}                       # a (attn_out) when norm, else x
    d["residual"] = draw((T, H), s, 1) if w.norm else None
    d["w_gate"] = draw((I, H), s, 2, b=w.w_std)
    d["w_up"] = draw((I, H), s, 3, b=w.w_std)
    d["w_down"] = draw((H, I), s, 4, b=w.w_std)
    d["gamma"] = draw((H,), s, 5, kind="uniform", a=0.9, b=1.1) if w.norm else None
    return d


def attn_inputs(w: Workload, T: int | None = None) -> dict:
    """Inputs of the attention projections: x, attention output A (shard-major), q/k/v/o weights."""
    T = w.T if T is None else T
    H, s, hd = w.H, w.seed, w.hd
    d = {"x": draw((T, H), s, 0)}
    # the attention core is not on the path: o_proj takes a synthetic N(0,1) A,
    # laid out as the t local shards [t][T][nq*hd/t] (heads of shard r contiguous)
    d["attn"] = draw((w.t, T, w.nq * hd // w.t), s, 1)
    d["w_q"] = draw((w.nq * hd, H), s, 2, b=w.w_std)
    d["w_k"] = draw((w.nkv * hd, H), s, 3, b=w.w_std)
    d["w_v"] = draw((w.nkv * hd, H), s, 4, b=w.w_std)
    d["w_o"] = draw((H, w.nq * hd), s, 5, b=w.w_std)
    return d


def attn_core_inputs(w: Workload, lens=None) -> dict:
    """Inputs of the attention core: qkv [t][T][w_s] ~ N(0, 1) in the QKV projection's
    layout (shard r: its q heads, k heads, v heads) and the sequence offsets."""
    lens = w.seq_lens() if lens is None else np.asarray(lens, dtype=np.int64)
    T = int(lens.sum())
    if w.t >= w.nkv:
        kv_per = 1
    else:
        kv_per = w.nkv // w.t
    ws = (w.nq // w.t + 2 * kv_per) * w.hd
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return {"qkv": draw((w.t, T, ws), w.seed, 6), "cu_seqlens": cu, "T": T}


def layer_inputs(w: Workload, T: int | None = None) -> dict:
    """Inputs of one decoder layer: hidden states and residual entering it, the
    attention weights (q, k, v, o), the input norm's gamma, the MLP weights
    (gate, up, down) and the post-attention norm's gamma."""
    T = w.T if T is None else T
    H, I, s, hd = w.H, w.I, w.seed, w.hd
    return {
        "hidden": draw((T, H), s, 0), "residual": draw((T, H), s, 1),
        "w_q": draw((w.nq * hd, H), s, 2, b=w.w_std), "w_k": draw((w.nkv * hd, H), s, 3, b=w.w_std),
        "w_v": draw((w.nkv * hd, H), s, 4, b=w.w_std), "w_o": draw((H, w.nq * hd), s, 5, b=w.w_std),
        "gamma_attn": draw((H,), s, 6, kind="uniform", a=0.9, b=1.1),
        "w_gate": draw((I, H), s, 7, b=w.w_std), "w_up": draw((I, H), s, 8, b=w.w_std),
        "w_down": draw((H, I), s, 9, b=w.w_std),
        "gamma_mlp": draw((H,), s, 10, kind="uniform", a=0.9, b=1.1),
    }


def moe_inputs(w: Workload, T: int | None = None) -> dict:
    """Inputs of an MoE block: x ~ N(0, 1), per-expert gate/up/down weights, and the
    routing. Routing recipe: numpy default_rng(seed + 7); expert popularity
    p_e proportional to (e + 1)^-0.5 (a skewed load); each token takes top_k
    distinct experts drawn with those probabilities; its gates are U(0.1, 1)
    draws scaled to sum to one (the shape of a softmax over the chosen logits)."""
    T = w.T if T is None else T
    H, I, s = w.H, w.I, w.seed
    d = {"x": draw((T, H), s, 0)}
    d["w_gate"] = [draw((I, H), s, 2 + 3 * e, b=w.w_std) for e in range(w.experts)]
    d["w_up"] = [draw((I, H), s, 3 + 3 * e, b=w.w_std) for e in range(w.experts)]
    d["w_down"] = [draw((H, I), s, 4 + 3 * e, b=w.w_std) for e in range(w.experts)]
    d.update(moe_routing(w, T))
    return d


def moe_routing(w: Workload, T: int) -> dict:
    rng = np.random.default_rng(w.seed + 7)
    pop = 1.0 / np.sqrt(np.arange(1, w.experts + 1))
    pop = pop / pop.sum()
    ids = np.stack([rng.choice(w.experts, w.top_k, replace=False, p=pop) for _ in range(T)]).astype(np.int32)
    u = rng.uniform(0.1, 1.0, (T, w.top_k))
    gates = (u / u.sum(axis=1, keepdims=True)).astype(np.float32)
    return {"expert_ids": ids.reshape(T, w.top_k), "gates": gates}


def ragged_batch(w: Workload) -> dict:
    """Row -> (request_id, token_pos) map of a ragged continuous batch and capture selectors."""
    rng = np.random.default_rng(w.seed)
    lens = rng.geometric(1.0 / w.mean_len, w.requests).astype(np.int64)
    k = int(np.argmax(lens))
    lens[k] += w.T - int(lens.sum())
    if lens[k] < 1:
        raise ValueError("ragged batch: token total too small for the drawn lengths")
    ctx = rng.integers(16, 4096, size=w.requests)       # context length of decode requests
    row_req = np.repeat(np.arange(w.requests, dtype=np.int32), lens)
    row_pos = np.empty(w.T, dtype=np.int32)
    o = 0
    for j, L in enumerate(lens):
        if L == 1:
            row_pos[o] = ctx[j]                         # 1-token decode row
        else:
            row_pos[o:o + L] = np.arange(L)             # prefill rows 0..L-1
        o += L
    n_sel = int(round(w.capture_frac * w.T))
    rows = rng.choice(w.T, n_sel, replace=False)
    sel = (row_req[rows].astype(np.int64) << 32) | row_pos[rows].astype(np.int64)
    return {"lens": lens, "row_req": row_req, "row_pos": row_pos, "sel_keys": sel,
            "sel_rows": np.sort(rows)}


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 tensor (no arithmetic)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
