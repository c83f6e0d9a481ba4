"""Benchmark of the tensor-parallel MLP block on GB300 (one JSON line on rank 0).

Default workload: Llama-3-8B-shaped MLP decode (32 tokens, hidden 4096,
intermediate 14336, t = 8 logical shards, residual add + RMSNorm). A step is
one pass of the whole block: add + RMSNorm, column-parallel gate_up GEMM with
SiLU*mul, row-parallel down GEMM with the on-chip shard reduction and the
residual-stream epilogue. The metric for decode is weight GB/s (weight bytes
streamed per second); prefill workloads report TFLOP/s.

L2: every step uses one of 4 rotating copies of the weights (4 x 352 MB for
the decode workload), so no step finds its weights in the 129 MB L2.

--impl reference runs the float64 CPU oracle on the host cores instead (the
reference arm of this build: there is no other implementation of the
pages' method to run), each step a bounded sample of the same workload.

Multi-GPU: replicas only. Each rank runs its own copy of the block on its own
token batch (weak scaling); there is no collective on the data path.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import socket
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
import workloads  # noqa: E402

METRIC = "TP-layout MLP block TFLOP/s (prefill) & weight GB/s (decode) vs GB300 roofline"
DEFAULT_WORKLOAD = "llama3_8b_mlp_decode"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--rotate", type=int, default=None,
                    help="input sets rotated across steps (default: 4, or 1 when the weights are over 1 GB)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="default workload only, without the other workloads under detail.configs")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------- ncu traffic
def kernel_sources_hash() -> str:
    import hashlib
    csrc = os.path.join(ROOT, "tensor_linear_layers_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        # every source: the host file chooses the plans (rasterisation, splits) that
        # decide a kernel's DRAM traffic
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(key: str):
    """DRAM bytes per launch from the committed ncu capture of this kernel and
    workload, or None when there is none or the kernel sources changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("csrc_sha256_16") != kernel_sources_hash():
        return None
    k = d.get("kernels", {}).get(key)
    return None if k is None else float(k["traffic_bytes"])


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # nvidia-smi's start-up queries the driver heavily: let it deliver its first
            # sample before the timed region begins
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0:
                time.sleep(0.01)
            time.sleep(0.02)
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        # a short timed region may fall between two samples: take the next one too
        n0, t0 = len(self.lines), time.time()
        while len(self.lines) == n0 and time.time() - t0 < 0.5:
            time.sleep(0.005)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, parts[2:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def hold_stream(stream, n_steps: int):
    """Keep `stream` busy (a bounded spin kernel, about 25 us per step to enqueue, at
    most 50 ms) while the host enqueues the timed steps, so that the device-timed
    region measures the steps back to back and not the host's enqueue lag. Nothing
    of the step runs in it; the end-to-end figure is timed without it."""
    cycles = int(min(50e-3, 1e-3 + 25e-6 * n_steps) * 2.0e9)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(cycles)


# ---------------------------------------------------------------------------- work model
def work_model(w: workloads.Workload):
    decode = (w.kind in ("mlp", "moe") and w.T <= 128) or w.kind == "paged"
    flops = w.flops()
    wbytes = w.weight_bytes()
    abytes = w.activation_bytes()
    return decode, flops, wbytes, abytes


def dominant_kernel_bytes(w: workloads.Workload) -> float:
    """Algorithmic bytes of one gate_up launch: weights read once, x read, h written."""
    return 2.0 * (2 * w.I * w.H + w.T * w.H + w.T * w.I)


def dominant_kernel_flops(w: workloads.Workload) -> float:
    if w.kind == "attn_core":
        return w.flops()
    if w.kind in ("mlp", "layer"):
        return 2.0 * w.T * w.H * 2 * w.I
    return 2.0 * w.T * w.H * (w.nq + 2 * w.nkv) * w.hd


# ---------------------------------------------------------------------------- CPU oracle timing
class OracleSample:
    """A bounded sample of the workload run through the float64 oracle on the host cores.

    MLP: the first ``rows`` tokens and ``feat`` of the I intermediate features
    (the block's output is a sum over intermediate features, so the slice is a
    proportional part of the work and of the weight bytes). Attention: the first
    ``rows`` tokens through both projections.
    """

    def __init__(self, w: workloads.Workload, feat: int, rows: int = 32, seed: int = 0):
        import oracle
        self.oracle = oracle
        self.w = w
        f = oracle.bf16_to_f64
        rng = np.random.default_rng(seed)
        self.rows = min(w.T, rows)
        small = workloads.Workload(**{**w.__dict__, "T": self.rows})
        if w.kind == "attn_core":
            # sampled query rows of the packed sequences; a row i of its sequence costs
            # 4 hd (i + 1) flops per q head
            self.feat = 0
            d = workloads.attn_core_inputs(w)
            self.qkv = d["qkv"]
            self.cu = d["cu_seqlens"]
            self.rows = min(d["T"], rows)
            self.row_ids = np.linspace(0, d["T"] - 1, self.rows).astype(np.int64)
            starts = self.cu[np.searchsorted(self.cu, self.row_ids, side="right") - 1]
            self.flops = 4.0 * w.hd * w.nq * float(np.sum(self.row_ids - starts + 1))
            self.wbytes = 0.0
            return
        if w.kind == "paged":
            # the first `rows` requests' new tokens over their cached keys
            self.feat = 0
            self.rows = min(w.T, rows)
            self.lens = [int(x) for x in w.seq_lens()[:self.rows]]
            q_per, kv_per = w.nq // w.t, (1 if w.t >= w.nkv else w.nkv // w.t)
            width = (q_per + 2 * kv_per) * w.hd
            self.full = workloads.draw((w.t, int(sum(self.lens)), width), seed + 5, 0)
            self.wbytes = float(sum(self.lens) * 2 * w.nkv * w.hd * 2)
            self.flops = 4.0 * w.hd * w.nq * float(sum(self.lens))
            return
        if w.kind == "moe":
            # the first `rows` tokens, every routed entry through its expert
            self.feat = 0
            d = workloads.moe_inputs(w, T=self.rows)
            self.args = d
            self.flops = w.top_k * small.mlp_flops()
            hit = np.unique(d["expert_ids"])
            self.wbytes = float(len(hit) * 2 * 3 * w.H * w.I)
            return
        if w.kind == "layer":
            # the first `rows` tokens: under causal attention they depend on no later
            # token, so the sample is an exact prefix of the whole step's work
            self.feat = 0
            d = workloads.layer_inputs(w, T=self.rows)
            cu_full = np.concatenate([[0], np.cumsum(w.seq_lens())])
            self.cu = np.array([c for c in cu_full if c < self.rows] + [self.rows], np.int64)
            self.args = d
            L = np.diff(self.cu).astype(np.float64)
            self.flops = (small.proj_flops() + small.mlp_flops()
                          + 4.0 * w.hd * w.nq * float(np.sum(L * (L + 1) / 2)))
            self.wbytes = float(w.weight_bytes())
            return
        if w.kind == "mlp":
            self.feat = max(8, min(w.I, feat))
            d = workloads.mlp_inputs(small, T=self.rows)
            cols = np.sort(rng.choice(w.I, self.feat, replace=False))
            tc = torch.from_numpy(cols)
            self.args = (f(d["x"]), f(d["w_gate"][tc]), f(d["w_up"][tc]), f(d["w_down"][:, tc]))
            self.kw = dict(residual=None if d["residual"] is None else f(d["residual"]),
                           gamma=None if d["gamma"] is None else f(d["gamma"]), eps=w.eps, norm=w.norm)
            self.wbytes = 3.0 * w.H * self.feat * 2
            self.flops = 2.0 * self.rows * w.H * 2 * self.feat + 2.0 * self.rows * self.feat * w.H
        else:
            self.feat = 0
            d = workloads.attn_inputs(small, T=self.rows)
            self.args = tuple(f(d[k]) for k in ("x", "w_q", "w_k", "w_v", "w_o", "attn"))
            self.wbytes = float(w.weight_bytes())
            self.flops = w.flops() * self.rows / w.T

    def run(self):
        w, o = self.w, self.oracle
        if w.kind == "attn_core":
            o.attention_rows(self.qkv, w.nq, w.nkv, w.hd, w.t, self.cu, self.row_ids)
            return
        if w.kind == "paged":
            # fill a cache through slots and attend: the oracle's write and read paths
            q_per, kv_per = w.nq // w.t, (1 if w.t >= w.nkv else w.nkv // w.t)
            bs = 16
            nb = sum(-(-L // bs) for L in self.lens)
            ck = np.zeros((w.t, nb, bs, kv_per, w.hd))
            cv = np.zeros_like(ck)
            tables = np.zeros((len(self.lens), max(-(-L // bs) for L in self.lens)), dtype=np.int64)
            used = 0
            for b, L in enumerate(self.lens):
                n = -(-L // bs)
                tables[b, :n] = np.arange(used, used + n)
                used += n
            slots = np.concatenate([[tables[b, p // bs] * bs + p % bs for p in range(L)]
                                    for b, L in enumerate(self.lens)])
            o.kv_cache_write(self.full, slots, ck, cv, w.nq, w.nkv, w.hd, w.t, bs)
            ends = np.cumsum(self.lens) - 1
            o.paged_attention(self.full[:, ends], np.arange(len(self.lens) + 1), self.lens, tables, ck, cv,
                              w.nq, w.nkv, w.hd, w.t, bs)
            return
        if w.kind == "moe":
            d = self.args
            o.moe_block(d["x"], d["expert_ids"], d["gates"], d["w_gate"], d["w_up"], d["w_down"])
            return
        if w.kind == "layer":
            d = self.args
            o.decoder_layer(d["hidden"], d["residual"], d["gamma_attn"], d["w_q"], d["w_k"], d["w_v"], d["w_o"],
                            d["gamma_mlp"], d["w_gate"], d["w_up"], d["w_down"], w.nq, w.nkv, w.hd, w.t,
                            self.cu, w.eps)
            return
        if w.kind == "mlp":
            o.mlp_layer(*self.args, **self.kw)
        else:
            x, wq, wk, wv, wo, A = self.args
            o.qkv_parallel(x, wq, wk, wv, w.nq, w.nkv, w.hd, w.t)
            o.o_proj_parallel(A, wo, w.t)

    def describe(self, n, el):
        w = self.w
        if w.kind == "attn_core":
            what = f"{self.rows} of {w.T} query rows (evenly spaced) through the causal attention of all {w.nq} q heads"
        elif w.kind == "paged":
            what = (f"the first {self.rows} of {w.T} requests ({sum(self.lens)} cached tokens): cache write "
                    f"of every token and decode attention of each request's last token")
        elif w.kind == "moe":
            what = (f"the first {self.rows} of {w.T} tokens, top-{w.top_k} of {w.experts} experts "
                    f"(intermediate {w.I}, hidden {w.H})")
        elif w.kind == "layer":
            what = (f"the first {self.rows} of {w.T} tokens ({len(self.cu) - 1} sequence(s)) through the whole "
                    f"layer: norm, QKV, causal attention, o_proj, add + norm, MLP")
        elif w.kind == "mlp":
            what = f"{self.rows} of {w.T} tokens x {self.feat} of {w.I} intermediate features (hidden {w.H})"
        else:
            what = f"{self.rows} of {w.T} tokens through QKV and o_proj"
        return f"float64 NumPy oracle, {what}, {n} repetitions in {el:.2f} s"

    def value(self, per_s, decode):
        return (self.wbytes / per_s / 1e9, "GB/s") if decode else (self.flops / per_s / 1e12, "TFLOP/s")


def time_reps(sample: OracleSample, n: int) -> float:
    t0 = time.perf_counter()
    for _ in range(n):
        sample.run()
    return time.perf_counter() - t0


def cpu_baseline(w: workloads.Workload, budget_s: float = 12.0):
    """The oracle on a bounded sample of the workload, timed on this host's cores."""
    decode = work_model(w)[0]
    s = OracleSample(w, feat=2048)
    s.run()
    per1 = time_reps(s, 1)
    n = max(1, int(budget_s / max(per1, 1e-6)))
    el = time_reps(s, n)
    v, unit = s.value(el / n, decode)
    return {"value": v, "unit": unit, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": s.describe(n, el)}


def config_obj(w: workloads.Workload, n: int, rotate: int, decode: bool):
    c = {"workload": w.name, "desc": w.desc, "tokens": w.T, "hidden": w.H, "t": w.t}
    if w.kind == "mlp":
        c["intermediate"] = w.I
        c["fused_add_rmsnorm"] = w.norm
    else:
        c.update({"n_q_heads": w.nq, "n_kv_heads": w.nkv, "head_dim": w.hd})
    if w.kind == "layer":
        c["intermediate"] = w.I
        c["sequences"] = int(len(w.seq_lens()))
        c["causal"] = True
    if w.kind == "paged":
        lens = w.seq_lens()
        c.update({"requests": w.T, "cached_tokens": int(lens.sum()), "seq_len_range": [int(lens.min()), int(lens.max())],
                  "block_size": 16, "new_tokens_per_request": 1})
    if w.kind == "moe":
        for k in ("n_q_heads", "n_kv_heads", "head_dim"):
            c.pop(k, None)
        c.update({"intermediate": w.I, "experts": w.experts, "top_k": w.top_k})
    if w.kind == "attn_core":
        c["sequences"] = int(len(w.seq_lens()))
        c["causal"] = True
        qkv_b = 2 * w.T * (w.nq + 2 * (w.nkv if w.t < w.nkv else w.t)) * w.hd
        c["l2"] = f"{rotate} rotating qkv inputs ({rotate * qkv_b / 1e9:.2f} GB) > 129 MB L2"
    elif w.kind == "paged":
        c["l2"] = f"KV cache read per step {w.kv_cache_bytes() / 1e9:.2f} GB > 129 MB L2; {rotate} rotating caches"
    elif w.kind == "moe":
        c["l2"] = f"expert weights {w.weight_bytes() / 1e9:.2f} GB > 129 MB L2; {rotate} rotating inputs"
    elif w.kind == "layer":
        c["l2"] = (f"weights {w.weight_bytes() / 1e9:.2f} GB and the step's intermediates "
                   f"(h alone {2 * w.T * w.I / 1e9:.2f} GB) > 129 MB L2; {rotate} rotating inputs")
    elif rotate == 1:
        c["l2"] = (f"weights {w.weight_bytes() / 1e9:.2f} GB and activations {w.activation_bytes() / 1e9:.2f} GB "
                   f"per step > 129 MB L2 (no rotation needed)")
    else:
        c["l2"] = f"{rotate} rotating weight copies ({rotate * w.weight_bytes() / 1e9:.2f} GB) > 129 MB L2"
    c["parallelism"] = f"replicas x{n}" if n > 1 else "single GPU (t shards on one GPU)"
    return c


# ---------------------------------------------------------------------------- reference arm
def run_reference(args, ws, rank):
    if rank != 0:
        return
    w = workloads.WORKLOADS[args.workload]
    decode = work_model(w)[0]
    K = args.steps if args.steps is not None else 20
    W = args.warmup if args.warmup is not None else 3
    # size one step so that warm-up + K steps take about two minutes in total
    target = max(0.002, min(2.0, 120.0 / max(1, K + W)))
    s = OracleSample(w, feat=2048)
    s.run()
    per = time_reps(s, 1)
    if w.kind == "mlp":
        feat = int(min(w.I, max(8, 2048 * target / max(per, 1e-6))) // 8 * 8)
        s = OracleSample(w, feat=max(8, feat))
    time_reps(s, W)
    el = time_reps(s, K)
    value, unit = s.value(el / K, decode)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
        "steps": K, "warmup": W, "ms_per_step": el / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_obj(w, args.gpus, rotation(w, args.rotate), decode),
        "cpu_baseline": {"value": value, "unit": unit, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                         "sample": s.describe(K, el)},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- our arm
# Workloads measured besides the headline one in a default run, each reported
# under detail.configs with its own roofline, end-to-end and CPU-oracle numbers.
OTHER_CONFIGS = ("tiny_mlp", "llama3_8b_attn_proj_prefill", "llama3_70b_mlp_prefill", "qwen25_7b_ragged_mlp")


def rotation(w: workloads.Workload, requested) -> int:
    """Input sets rotated across steps so that no step finds its inputs in L2: at
    least 4, and enough sets to hold twice the 129 MB L2 (at most 64). A workload
    whose weights alone are over 1 GB (8x the L2) needs none."""
    if requested is not None:
        return max(1, requested)
    per_set = w.weight_bytes() + w.activation_bytes()
    if w.weight_bytes() >= (1 << 30):
        return 1
    return int(min(64, max(4, -(-2 * 129 * 2**20 // max(per_set, 1)))))


def run_ours(args, ws, rank, local):
    import tensor_linear_layers_gb300 as tl
    from tensor_linear_layers_gb300 import _build
    if rank == 0 or ws == 1:
        _build.build()
    barrier(ws)
    tl.lib()
    torch.cuda.set_device(torch.device("cuda", local))
    w = workloads.WORKLOADS[args.workload]
    line = measure(args, w, ws, rank, local, cpu_budget_s=12.0)
    if args.workload == DEFAULT_WORKLOAD and not args.headline_only:
        recs = {}
        for name in OTHER_CONFIGS:
            gc.collect()
            torch.cuda.empty_cache()
            # and the pinned host blocks the caching host allocator keeps: reused by the next
            # workload's transfer buffers they left its end-to-end copies at a fraction of
            # their speed (ragged Qwen block 1050-1430 instead of 558 us per step)
            getattr(torch._C, "_host_emptyCache", lambda: None)()
            r = measure(args, workloads.WORKLOADS[name], ws, rank, local, cpu_budget_s=6.0)
            for k in ("metric", "n_gpus", "higher_is_better", "scaling", "vs_baseline", "dtype", "data"):
                r.pop(k, None)
            recs[name] = r
        line["detail"]["configs"] = recs
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure(args, w: workloads.Workload, ws, rank, local, cpu_budget_s: float):
    """Times one workload (whole steps, the dominant kernel, end to end) and returns its JSON record."""
    import tensor_linear_layers_gb300 as tl
    dev = torch.device("cuda", local)
    decode, flops, wbytes, abytes = work_model(w)
    R = rotation(w, args.rotate)
    if decode:
        K = args.steps if args.steps is not None else 10000
        W = args.warmup if args.warmup is not None else 100
    else:
        K = args.steps if args.steps is not None else 50
        W = args.warmup if args.warmup is not None else 5
    W = max(W, 3)

    # ---- inputs: same weights on every rank, rank-specific activations (replicas)
    if w.kind == "mlp":
        d = workloads.mlp_inputs(w)
        cfg = tl.make_config(tl.TP_BLOCK_MLP, w.t, w.H, w.I, rms_eps=w.eps,
                             flags=tl.TP_FLAG_HAS_NORM if w.norm else 0)
        wl = [d["w_gate"].to(dev), d["w_up"].to(dev), d["w_down"].to(dev)]
        gamma = None if d["gamma"] is None else d["gamma"].to(dev)
        blocks = []
        for r in range(R):
            blocks.append(tl.TPLinear(cfg, wl, gamma=gamma))
        del wl
        xs = [workloads.draw((w.T, w.H), 1000 + rank * R + r, 0).to(dev) for r in range(R)]
        rs = [workloads.draw((w.T, w.H), 1000 + rank * R + r, 1).to(dev) for r in range(R)] if w.norm else [None] * R
        outs = [{"mlp_out": torch.empty_like(xs[0]), "residual_out": torch.empty_like(xs[0]) if w.norm else None,
                 "residual_stream": torch.empty_like(xs[0]) if w.norm else None} for _ in range(R)]
        for o in outs:
            for k in [k for k, v in o.items() if v is None]:
                del o[k]
        wss = [b.workspace(w.T) for b in blocks]
        # T <= 128: the whole block is one fused kernel; larger T: norm + two GEMMs
        launches_per_step = 1 if w.T <= 128 else (1 if w.norm else 0) + 2
        cap = None
        if w.capture_frac > 0:
            # the ragged batch's step ends with the capture of mlp_out and residual_stream
            # rows for the selected (request, position) keys
            b = workloads.ragged_batch(w)
            n_rec = 2 * len(b["sel_keys"])
            cap = {"rq": torch.from_numpy(b["row_req"]).to(dev), "rp": torch.from_numpy(b["row_pos"]).to(dev),
                   "keys": torch.from_numpy(b["sel_keys"]).to(dev), "n": n_rec,
                   "types": [workloads.TENSOR_TYPES["mlp_out"], workloads.TENSOR_TYPES["residual_stream"]],
                   "ws": torch.zeros(tl.capture_workspace_size(w.T, len(b["sel_keys"])), dtype=torch.uint8,
                                     device=dev),
                   "out": [(torch.empty(n_rec, 6, dtype=torch.int32, device=dev),
                            torch.empty(n_rec, w.H, dtype=torch.bfloat16, device=dev),
                            torch.zeros(1, dtype=torch.int64, device=dev)) for _ in range(R)]}
            # one launch while the selector table and the match list fit in shared memory
            # (the library's choice), else a match and a copy launch
            lg = 6
            while (1 << lg) < 2 * len(b["sel_keys"]):
                lg += 1
            launches_per_step += 1 if (lg <= 13 and w.T <= 16384 and (8 << lg) + 4 * w.T <= 160 * 1024) else 2

        def capture(j, o):
            tl.capture_rows(cap["rq"], cap["rp"], cap["keys"], [o["mlp_out"], o["residual_stream"]], cap["types"],
                            0, cap["n"], ws=cap["ws"], out=cap["out"][j])

        def step(i):
            j = i % R
            blocks[j].mlp_forward(xs[j], residual=rs[j], out=outs[j], ws=wss[j])
            if cap is not None:
                capture(j, outs[j])

        def dominant(i):
            j = i % R
            blocks[j].gate_up(xs[j], h_out=hbufs[j], ws=wss[j])
        hbufs = [torch.empty(w.t, w.T, w.I // w.t, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    elif w.kind == "paged":
        dw = workloads.attn_inputs(w, T=1)
        cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, w.t, w.H, n_q_heads=w.nq, n_kv_heads=w.nkv, head_dim=w.hd)
        blocks = [tl.TPLinear(cfg, [dw[k].to(dev) for k in ("w_q", "w_k", "w_v", "w_o")])]
        lens = [int(x) for x in w.seq_lens()]
        bs = 16
        q_per, kv_per = w.nq // w.t, (1 if w.t >= w.nkv else w.nkv // w.t)
        width = (q_per + 2 * kv_per) * w.hd
        nb_req = [-(-L // bs) for L in lens]
        n_blocks = sum(nb_req)
        tables = np.zeros((len(lens), max(nb_req)), dtype=np.int32)
        perm = np.random.default_rng(rank).permutation(n_blocks)   # scattered blocks
        used = 0
        for b, n in enumerate(nb_req):
            tables[b, :n] = perm[used:used + n]
            used += n
        tables_d = torch.from_numpy(tables).to(dev)
        caches = []
        for r_ in range(R):
            ck = torch.empty(blocks[0].kv_cache_shape(n_blocks, bs), dtype=torch.bfloat16, device=dev)
            cv = torch.empty_like(ck)
            for b, L in enumerate(lens):     # the cached context, one request at a time
                full = workloads.draw((w.t, L, width), 1000 + rank * R + r_, b).to(dev)
                slots = torch.from_numpy(np.array([tables[b, p // bs] * bs + p % bs for p in range(L)],
                                                  dtype=np.int32)).to(dev)
                blocks[0].kv_cache_write(full, slots, ck, cv)
            caches.append((ck, cv))
        new_slots = torch.from_numpy(np.array([tables[b, (L - 1) // bs] * bs + (L - 1) % bs
                                               for b, L in enumerate(lens)], dtype=np.int32)).to(dev)
        qkvs = [workloads.draw((w.t, len(lens), width), 2000 + rank * R + r_, 0).to(dev) for r_ in range(R)]
        qsl = torch.arange(len(lens) + 1, dtype=torch.int32, device=dev)
        lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
        aos = [torch.empty(w.t, len(lens), q_per * w.hd, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        pws = torch.zeros(blocks[0].paged_attention_workspace_size(len(lens), 1, max(lens)), dtype=torch.uint8,
                          device=dev)
        wss = [pws]
        launches_per_step = 2           # split attention (it writes the new tokens' k and v first), split merge

        def step(i):
            j = i % R
            ck, cv = caches[j]
            blocks[0].paged_attention(qkvs[j], qsl, lens_d, tables_d, ck, cv, 1, max(lens), out=aos[j], ws=pws,
                                      slot_mapping=new_slots)
        dominant = step
    elif w.kind == "moe":
        d = workloads.moe_inputs(w)
        cfg = tl.make_config(tl.TP_BLOCK_MOE, w.t, w.H, w.I, n_experts=w.experts)
        wl = []
        for e in range(w.experts):
            wl += [d["w_gate"][e].to(dev), d["w_up"][e].to(dev), d["w_down"][e].to(dev)]
        blocks = [tl.TPLinear(cfg, wl)]
        del wl
        ids = torch.from_numpy(d["expert_ids"]).to(dev)
        gts = torch.from_numpy(d["gates"]).to(dev)
        xs = [workloads.draw((w.T, w.H), 1000 + rank * R + r, 0).to(dev) for r in range(R)]
        outs = [torch.empty_like(xs[0]) for _ in range(R)]
        wss = [blocks[0].workspace(w.T * w.top_k)]
        launches_per_step = 5           # routing sort, row gather, grouped gate_up, grouped down, combine

        def step(i):
            j = i % R
            blocks[0].moe_forward(xs[j], ids, gts, out=outs[j], ws=wss[0])
        dominant = step
    elif w.kind == "layer":
        d = workloads.layer_inputs(w, T=1)
        ca = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, w.t, w.H, n_q_heads=w.nq, n_kv_heads=w.nkv, head_dim=w.hd,
                            rms_eps=w.eps, flags=tl.TP_FLAG_HAS_NORM)
        cm = tl.make_config(tl.TP_BLOCK_MLP, w.t, w.H, w.I, rms_eps=w.eps, flags=tl.TP_FLAG_HAS_NORM)
        attn_b = tl.TPLinear(ca, [d[k].to(dev) for k in ("w_q", "w_k", "w_v", "w_o")],
                             gamma=d["gamma_attn"].to(dev))
        mlp_b = tl.TPLinear(cm, [d[k].to(dev) for k in ("w_gate", "w_up", "w_down")],
                            gamma=d["gamma_mlp"].to(dev))
        del d
        layer = tl.TPLayer(attn_b, mlp_b, w.T)
        blocks = [attn_b, mlp_b]
        lens = w.seq_lens()
        cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(dev)
        max_len = int(np.max(lens))
        xs = [workloads.draw((w.T, w.H), 1000 + rank * R + r, 0).to(dev) for r in range(R)]
        rs = [workloads.draw((w.T, w.H), 1000 + rank * R + r, 1).to(dev) for r in range(R)]
        outs = [{k: torch.empty_like(xs[0]) for k in ("residual_attn", "attn_out", "residual_mlp", "mlp_out",
                                                     "residual_stream")} for _ in range(R)]
        wss = [layer.workspace()]
        # norm, QKV, attention (2), o_proj, then the MLP: norm + gate_up + down, or one fused kernel
        launches_per_step = 5 + (1 if w.T <= 128 else 3)
        hbufs = [torch.empty(w.t, w.T, w.I // w.t, dtype=torch.bfloat16, device=dev)]
        gws = mlp_b.workspace(w.T)

        def step(i):
            j = i % R
            layer.forward(xs[j], rs[j], cu, max_len, out=outs[j], ws=wss[0])

        def dominant(i):
            j = i % R
            mlp_b.gate_up(xs[j], h_out=hbufs[0], ws=gws)
    elif w.kind == "attn_core":
        dw = workloads.attn_inputs(w, T=1)
        cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, w.t, w.H, n_q_heads=w.nq, n_kv_heads=w.nkv, head_dim=w.hd)
        blocks = [tl.TPLinear(cfg, [dw[k].to(dev) for k in ("w_q", "w_k", "w_v", "w_o")])]
        dc = workloads.attn_core_inputs(w)
        cu = torch.from_numpy(dc["cu_seqlens"]).to(dev)
        max_len = int(np.max(np.diff(dc["cu_seqlens"])))
        qkvs = [workloads.draw(tuple(dc["qkv"].shape), 1000 + rank * R + r, 6).to(dev) for r in range(R)]
        aos = [torch.empty(w.t, w.T, w.nq // w.t * w.hd, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        wss = [blocks[0].workspace(w.T)]
        launches_per_step = 2          # work-table preparation + the attention kernel

        def step(i):
            j = i % R
            blocks[0].attention_forward(qkvs[j], cu, max_len, out=aos[j], ws=wss[0])
        dominant = step
    else:
        d = workloads.attn_inputs(w)
        cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, w.t, w.H, n_q_heads=w.nq, n_kv_heads=w.nkv, head_dim=w.hd)
        wl = [d[k].to(dev) for k in ("w_q", "w_k", "w_v", "w_o")]
        blocks = [tl.TPLinear(cfg, wl) for _ in range(R)]
        del wl
        xs = [workloads.draw((w.T, w.H), 1000 + rank * R + r, 0).to(dev) for r in range(R)]
        As = [workloads.draw((w.t, w.T, w.nq * w.hd // w.t), 1000 + rank * R + r, 1).to(dev) for r in range(R)]
        wss = [b.workspace(w.T) for b in blocks]
        q_per = w.nq // w.t
        kv_per = 1 if w.t >= w.nkv else w.nkv // w.t
        qkvs = [torch.empty(w.t, w.T, (q_per + 2 * kv_per) * w.hd, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        oos = [torch.empty(w.T, w.H, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        # T > 128: QKV and o_proj share one launch; T <= 128: two launches
        launches_per_step = 1 if w.T > 128 else 2

        def step(i):
            j = i % R
            blocks[j].attn_proj_forward(xs[j], As[j], qkv_out=qkvs[j], o_out=oos[j], ws=wss[j])

        def dominant(i):
            j = i % R
            blocks[j].attn_proj_forward(xs[j], None, qkv_out=qkvs[j], ws=wss[j])
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    # ---- warm-up
    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    for wsb in wss + ([cap["ws"]] if w.kind == "mlp" and cap is not None else []):
        st = int(wsb[:4].view(torch.int32).item())
        if st != 0:
            raise RuntimeError(f"device status {st} after warm-up")

    # ---- timed region: K whole steps, device-timed with events on the launching stream
    sampler = ClockSampler(local)
    sampler.start()
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream, K)
    e0.record(stream)
    for i in range(K):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / K
    ms = max_over_ranks(ms, ws)
    sec = ms / 1e3

    # ---- dominant kernel: in decode the step is a single fused kernel, so its
    # average launch duration is the timed region's per-step time; otherwise the
    # column-parallel GEMM alone, same stream, events around K2 launches
    if launches_per_step == 1 or w.kind in ("attn_core", "moe", "paged"):
        dom_s = sec                    # attention core, MoE, paged decode: every launch of a step (conservative)
    else:
        K2 = min(K, 2000 if decode else 20)
        for i in range(3):
            dominant(i)
        torch.cuda.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_stream(stream, K2)
        d0.record(stream)
        for i in range(K2):
            dominant(i)
        d1.record(stream)
        torch.cuda.synchronize()
        dom_s = d0.elapsed_time(d1) / K2 / 1e3

    # ---- end to end through the public API from pinned host buffers. Every step copies its
    # inputs in and its results out; the copies run on two copy streams, ordered by events,
    # so that step i's compute overlaps step i+1's input copy and step i-1's result copy.
    # E >= 3 sets of activation buffers rotate (a set is refilled only after the compute and
    # the read-back of its previous step); the weights and workspaces rotate with R as in
    # the timed region (steps run one after another on the compute stream, so set e uses
    # weight copy e % R).
    K3 = min(K, 500 if decode else 10)
    E = max(R, 3)

    def extend(lst, make):
        return list(lst) + [make() for _ in range(len(lst), E)]
    if w.kind == "mlp":
        # x and residual in one device buffer, the outputs in another: one copy each way
        names = list(outs[0].keys())
        n_in = 2 if rs[0] is not None else 1
        din = [torch.empty((n_in, w.T, w.H), dtype=torch.bfloat16, device=dev) for _ in range(E)]
        dout = [torch.empty((len(names), w.T, w.H), dtype=torch.bfloat16, device=dev) for _ in range(E)]
        hin = [torch.stack([xs[j % R]] + ([rs[j % R]] if n_in == 2 else [])).cpu().pin_memory() for j in range(E)]
        hout = [torch.empty(dout[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(E)]
        eouts = [{k: dout[j][i] for i, k in enumerate(names)} for j in range(E)]
        in_pairs = lambda j: [(hin[j], din[j])]
        if cap is None:
            out_pairs = lambda j: [(dout[j], hout[j])]
        else:
            # the captured records (headers and rows) come back with the block's outputs
            ecap = extend(cap["out"], lambda: tuple(torch.empty_like(t) for t in cap["out"][0]))
            hcap = [(torch.empty(cap["out"][0][0].shape, dtype=torch.int32, pin_memory=True),
                     torch.empty(cap["out"][0][1].shape, dtype=torch.bfloat16, pin_memory=True)) for _ in range(E)]
            out_pairs = lambda j: [(dout[j], hout[j]), (ecap[j][0], hcap[j][0]), (ecap[j][1], hcap[j][1])]

        def e2e_compute(j):
            blocks[j % R].mlp_forward(din[j][0], residual=din[j][1] if n_in == 2 else None, out=eouts[j],
                                      ws=wss[j % R])
            if cap is not None:
                tl.capture_rows(cap["rq"], cap["rp"], cap["keys"], [eouts[j]["mlp_out"], eouts[j]["residual_stream"]],
                                cap["types"], 0, cap["n"], ws=cap["ws"], out=ecap[j])
    elif w.kind == "paged":
        eq = extend(qkvs, lambda: torch.empty_like(qkvs[0]))
        eo = extend(aos, lambda: torch.empty_like(aos[0]))
        hq = [qkvs[j % R].cpu().pin_memory() for j in range(E)]
        ho = [torch.empty(aos[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(E)]
        in_pairs = lambda j: [(hq[j], eq[j])]
        out_pairs = lambda j: [(eo[j], ho[j])]

        def e2e_compute(j):
            ck, cv = caches[j % R]
            blocks[0].paged_attention(eq[j], qsl, lens_d, tables_d, ck, cv, 1, max(lens), out=eo[j], ws=pws,
                                      slot_mapping=new_slots)
    elif w.kind == "moe":
        ex = extend(xs, lambda: torch.empty_like(xs[0]))
        eo = extend(outs, lambda: torch.empty_like(outs[0]))
        hx = [xs[j % R].cpu().pin_memory() for j in range(E)]
        hid = ids.cpu().pin_memory()
        hg = gts.cpu().pin_memory()
        ho = [torch.empty(xs[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(E)]
        eids = [ids.clone() for _ in range(E)]
        egts = [gts.clone() for _ in range(E)]
        in_pairs = lambda j: [(hx[j], ex[j]), (hid, eids[j]), (hg, egts[j])]
        out_pairs = lambda j: [(eo[j], ho[j])]

        def e2e_compute(j):
            blocks[0].moe_forward(ex[j], eids[j], egts[j], out=eo[j], ws=wss[0])
    elif w.kind == "layer":
        ex = extend(xs, lambda: torch.empty_like(xs[0]))
        er = extend(rs, lambda: torch.empty_like(rs[0]))
        eo = extend(outs, lambda: {k: torch.empty_like(v) for k, v in outs[0].items()})
        hx = [xs[j % R].cpu().pin_memory() for j in range(E)]
        hr = [rs[j % R].cpu().pin_memory() for j in range(E)]
        # the layer's result as the next layer takes it: (hidden = mlp_out, residual = r2)
        hm = [torch.empty(xs[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(E)]
        hres = [torch.empty(xs[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(E)]
        in_pairs = lambda j: [(hx[j], ex[j]), (hr[j], er[j])]
        out_pairs = lambda j: [(eo[j]["mlp_out"], hm[j]), (eo[j]["residual_mlp"], hres[j])]

        def e2e_compute(j):
            layer.forward(ex[j], er[j], cu, max_len, out=eo[j], ws=wss[0])
    elif w.kind == "attn_core":
        eq = extend(qkvs, lambda: torch.empty_like(qkvs[0]))
        eo = extend(aos, lambda: torch.empty_like(aos[0]))
        hq = [qkvs[j % R].cpu().pin_memory() for j in range(E)]
        ho = [torch.empty(aos[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(E)]
        in_pairs = lambda j: [(hq[j], eq[j])]
        out_pairs = lambda j: [(eo[j], ho[j])]

        def e2e_compute(j):
            blocks[0].attention_forward(eq[j], cu, max_len, out=eo[j], ws=wss[0])
    else:
        ex = extend(xs, lambda: torch.empty_like(xs[0]))
        eA = extend(As, lambda: torch.empty_like(As[0]))
        eq = extend(qkvs, lambda: torch.empty_like(qkvs[0]))
        eo = extend(oos, lambda: torch.empty_like(oos[0]))
        hx = [xs[j % R].cpu().pin_memory() for j in range(E)]
        hA = [As[j % R].cpu().pin_memory() for j in range(E)]
        hq = [torch.empty(qkvs[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(E)]
        hoo = [torch.empty(oos[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(E)]
        in_pairs = lambda j: [(hx[j], ex[j]), (hA[j], eA[j])]
        out_pairs = lambda j: [(eq[j], hq[j]), (eo[j], hoo[j])]

        def e2e_compute(j):
            blocks[j % R].attn_proj_forward(ex[j], eA[j], qkv_out=eq[j], o_out=eo[j], ws=wss[j % R])
    h2d = sum(hsrc.numel() * hsrc.element_size() for hsrc, _ in in_pairs(0))
    d2h = sum(hdst.numel() * hdst.element_size() for _, hdst in out_pairs(0))
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(E)]
    ev_comp = [torch.cuda.Event() for _ in range(E)]
    ev_out = [torch.cuda.Event() for _ in range(E)]

    def e2e_run(n, start_ev=None):
        if start_ev is not None:
            s_in.wait_event(start_ev)           # no copy of the timed steps starts before the timer
        for i in range(n):
            j = i % E
            s_in.wait_event(ev_comp[j])         # the set's inputs were consumed by step i - E
            with torch.cuda.stream(s_in):
                for hsrc, ddst in in_pairs(j):
                    ddst.copy_(hsrc, non_blocking=True)
            ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_out[j])        # the set's results were read back after step i - E
            e2e_compute(j)
            ev_comp[j].record(stream)
            s_out.wait_event(ev_comp[j])
            with torch.cuda.stream(s_out):
                for dsrc, hdst in out_pairs(j):
                    hdst.copy_(dsrc, non_blocking=True)
            ev_out[j].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    e2e_run(3)
    torch.cuda.synchronize()
    barrier(ws)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    e2e_run(K3, start_ev=f0)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(f0.elapsed_time(f1) / K3, ws) / 1e3

    for wsb in wss + ([cap["ws"]] if w.kind == "mlp" and cap is not None else []):
        st = int(wsb[:4].view(torch.int32).item())
        if st != 0:
            raise RuntimeError(f"device status {st} after the timed region")

    pk = peaks()
    if decode:
        unit = "GB/s"
        value = ws * wbytes / sec / 1e9
        e2e_value = ws * wbytes / e2e_s / 1e9
        fused = launches_per_step == 1 or w.kind in ("moe", "paged")
        dom_alg = float(wbytes + abytes) if fused else dominant_kernel_bytes(w)
        achieved = dom_alg / dom_s / 1e9
        if w.kind == "paged":
            key, kname = "paged@", "paged decode step: split attention with the new tokens' cache write (paged_attn_kernel), split merge"
        elif w.kind == "moe":
            key, kname = "moe@", "the MoE step: routing, gather, grouped expert GEMMs (tc_gemm_kernel), combine"
        elif fused:
            key, kname = "mlp_decode@", "fused decode MLP block (mlp_decode_kernel)"
        else:
            key, kname = "gate_up@", "gate_up column-parallel GEMM (tc_gemm_kernel<swap, GATE_UP>)"
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"],
                "traffic": ncu_traffic(key + w.name),
                "kernel": kname,
                "algorithmic_bytes_per_launch": dom_alg, "avg_launch_us": dom_s * 1e6,
                "peak_source": pk["source"] + " hbm_gbs (copy, burst)"}
    else:
        unit = "TFLOP/s"
        value = ws * flops / sec / 1e12
        e2e_value = ws * flops / e2e_s / 1e12
        whole = launches_per_step == 1 or w.kind in ("attn_core", "moe")
        dom_alg = flops if whole else dominant_kernel_flops(w)
        achieved = dom_alg / dom_s / 1e12
        if w.kind == "attn_core":
            key, kname = "attn_core@", "causal GQA attention (attn_fwd_kernel, with its work-table preparation)"
        elif w.kind == "layer":
            key, kname = "gate_up@", "the layer's gate_up column-parallel GEMM (tc_gemm_pair_kernel<GATE_UP>)"
        elif w.kind == "moe":
            key, kname = "moe@", "the MoE step: routing, gather, grouped expert GEMMs (tc_gemm_kernel), combine"
        elif whole:
            key, kname = "attn_proj@", "QKV + o_proj in one launch (tc_gemm_pair_kernel<COL, ROW>)"
        else:
            key, kname = "gate_up@", "gate_up column-parallel GEMM (tc_gemm_pair_kernel<GATE_UP>)"
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_tflops"],
                "traffic": ncu_traffic(key + w.name),
                "kernel": kname,
                "algorithmic_flops_per_launch": dom_alg, "avg_launch_us": dom_s * 1e6,
                "peak_source": pk["source"] + " bf16_tflops (cuBLAS burst)"}

    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": config_obj(w, ws, R, decode),
        "roofline": roof, "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": K * launches_per_step,
        "detail": {
            "block_tflops": ws * flops / sec / 1e12,
            "block_gbs_weights_plus_activations": ws * (wbytes + abytes) / sec / 1e9,
            "tokens_per_s": ws * w.T / sec,
            "frac_hbm_measured_weights": (wbytes / sec / 1e9) / pk["hbm_gbs"],
            "frac_hbm_nominal_8tbs_weights": (wbytes / sec / 1e9) / 8000.0,
            "frac_bf16_measured": (flops / sec / 1e12) / pk["bf16_tflops"],
            "plans": blocks[0].plan(w.T),
        },
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, cpu_budget_s)
    return line


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def self_launch(args) -> int:
    """--gpus N > 1 outside torchrun: start N local ranks of this script with
    torch.distributed.run (rendezvous on 127.0.0.1) and return their exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.abspath(__file__)]
    return subprocess.call(cmd + sys.argv[1:])


def main():
    args = parse()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(self_launch(args))
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
