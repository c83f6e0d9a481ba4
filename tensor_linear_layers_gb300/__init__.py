"""Thin ctypes binding of libtplinear.so (include/tp_linear.h).

Argument marshalling only: torch tensors become device pointers and the
current CUDA stream becomes the stream argument; torch allocates the outputs,
packed weights and workspaces. Every step of the block runs in the library's
CUDA kernels. There is no fallback: if the library is missing or cannot load,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtplinear.so")

TP_OK = 0
TP_ERR_ARG, TP_ERR_SHAPE, TP_ERR_UNSUPPORTED, TP_ERR_CUDA, TP_ERR_CAPACITY, TP_ERR_TIMEOUT = (
    -1, -2, -3, -4, -5, -6)
TP_BLOCK_MLP, TP_BLOCK_ATTN_PROJ, TP_BLOCK_MOE = 0, 1, 2
TP_FLAG_HAS_NORM = 1
TP_FLAG_GATHERED = 2

ABI_SYMBOLS = (
    "tp_packed_weight_bytes", "tp_linear_create", "tp_linear_destroy", "tp_workspace_size",
    "tp_mlp_forward", "tp_add_rms_norm", "tp_gate_up_forward", "tp_down_forward",
    "tp_attn_proj_forward", "tp_capture_workspace_size", "tp_capture_rows", "tp_last_error",
    "tp_describe_plan", "tp_mlp_forward_no_alloc", "tp_set_wait_timeout", "tp_attention_forward",
    "tp_layer_create", "tp_layer_destroy", "tp_layer_workspace_size", "tp_decoder_layer_forward",
    "tp_moe_forward", "tp_kv_cache_write", "tp_paged_attention_workspace_size", "tp_paged_attention",
)


class TPError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"tp_linear error {code}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("t", ctypes.c_int32), ("hidden", ctypes.c_int64),
                ("intermediate", ctypes.c_int64), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("flags", ctypes.c_int32), ("n_experts", ctypes.c_int32)]


class LayerIO(ctypes.Structure):
    _fields_ = [("hidden_in", ctypes.c_void_p), ("residual_in", ctypes.c_void_p),
                ("cu_seqlens", ctypes.c_void_p), ("n_seqs", ctypes.c_int32), ("max_seqlen", ctypes.c_int32),
                ("residual_attn", ctypes.c_void_p), ("attn_out", ctypes.c_void_p),
                ("residual_mlp", ctypes.c_void_p), ("mlp_out", ctypes.c_void_p),
                ("residual_stream", ctypes.c_void_p)]


class GemmPlan(ctypes.Structure):
    _fields_ = [("swap_ab", ctypes.c_int32), ("block_n", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("units", ctypes.c_int32), ("grid", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("engine", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load the in-tree library once (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    PI64 = ctypes.POINTER(ctypes.c_int64)
    sig = {
        "tp_packed_weight_bytes": [ctypes.POINTER(Config), PI64, PI64],
        "tp_linear_create": [ctypes.POINTER(Config), ctypes.POINTER(P), I32, P, P, P, P,
                             ctypes.POINTER(P)],
        "tp_linear_destroy": [P],
        "tp_workspace_size": [P, I64, PI64],
        "tp_mlp_forward": [P, I64, P, P, P, P, P, P, I64, P],
        "tp_add_rms_norm": [I64, I64, P, P, P, F, P, P, P],
        "tp_gate_up_forward": [P, I64, P, P, P, I64, P],
        "tp_down_forward": [P, I64, P, P, P, P, P, I64, P],
        "tp_attn_proj_forward": [P, I64, P, P, P, P, P, I64, P],
        "tp_capture_workspace_size": [I64, I64, PI64],
        "tp_capture_rows": [I64, I64, P, P, P, I64, I32, ctypes.POINTER(P), ctypes.POINTER(I32),
                            I32, P, P, I64, P, P, I64, P],
        "tp_describe_plan": [P, I64, ctypes.POINTER(GemmPlan), I32],
        "tp_mlp_forward_no_alloc": [P, I64, P, P, P, P, P, P, P],
        "tp_set_wait_timeout": [I64],
        "tp_attention_forward": [P, I64, P, P, I32, I32, P, P, I64, P],
        "tp_layer_create": [P, P, I64, ctypes.POINTER(P)],
        "tp_layer_destroy": [P],
        "tp_layer_workspace_size": [P, PI64],
        "tp_decoder_layer_forward": [P, I64, ctypes.POINTER(LayerIO), P, I64, P],
        "tp_moe_forward": [P, I64, I32, P, P, P, P, P, I64, P],
        "tp_kv_cache_write": [P, I64, P, P, P, P, I64, I32, P, I64, P],
        "tp_paged_attention_workspace_size": [P, I32, I32, I32, PI64],
        "tp_paged_attention": [P, I64, P, P, P, I32, I32, I32, P, I32, P, P, P, I64, I32, P, P, I64, P],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.tp_last_error.argtypes = []
    L.tp_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(rc: int) -> int:
    if rc < 0:
        raise TPError(rc, lib().tp_last_error().decode(errors="replace"))
    return rc


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _bf16(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor")
    return t


def make_config(kind: int, t: int, hidden: int, intermediate: int = 0, n_q_heads: int = 0,
                n_kv_heads: int = 0, head_dim: int = 0, rms_eps: float = 1e-5, flags: int = 0,
                n_experts: int = 0) -> Config:
    return Config(kind, t, hidden, intermediate, n_q_heads, n_kv_heads, head_dim, rms_eps, flags, n_experts)


def packed_weight_bytes(cfg: Config):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().tp_packed_weight_bytes(ctypes.byref(cfg), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def set_wait_timeout(ns: int) -> None:
    """Wall-clock limit (ns) of every on-chip wait in kernels launched afterwards (default 2 s)."""
    _check(lib().tp_set_wait_timeout(int(ns)))


def capture_workspace_size(T: int, n_sel: int) -> int:
    b = ctypes.c_int64()
    _check(lib().tp_capture_workspace_size(T, n_sel, ctypes.byref(b)))
    return b.value


class TPLinear:
    """One tensor-parallel block (MLP or attention projections) on the current GPU.

    ``weights``: MLP (w_gate [I,H], w_up [I,H], w_down [H,I]); attention
    (w_q, w_k, w_v, w_o), all bf16 CUDA tensors in nn.Linear layout. The
    packed shard buffers are allocated here and owned by this object.
    """

    def __init__(self, cfg: Config, weights: Sequence[torch.Tensor], gamma: Optional[torch.Tensor] = None,
                 stream=None):
        L = lib()
        self.cfg = cfg
        col, row = packed_weight_bytes(cfg)
        dev = weights[0].device
        self.w_col = torch.empty(col // 2, dtype=torch.bfloat16, device=dev)
        self.w_row = torch.empty(row // 2, dtype=torch.bfloat16, device=dev)
        self.gamma = None if gamma is None else _bf16(gamma, "gamma")
        ws = [_bf16(w, "weight") for w in weights]
        arr = (ctypes.c_void_p * len(ws))(*[w.data_ptr() for w in ws])
        h = ctypes.c_void_p()
        _check(L.tp_linear_create(ctypes.byref(cfg), arr, len(ws), _ptr(self.w_col), _ptr(self.w_row),
                                  _ptr(self.gamma), _stream(stream), ctypes.byref(h)))
        self.handle = h
        self._ws = None
        self._ws_sizes = {}

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            lib().tp_linear_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ workspace
    def workspace_size(self, max_tokens: int) -> int:
        got = self._ws_sizes.get(max_tokens)
        if got is None:
            b = ctypes.c_int64()
            _check(lib().tp_workspace_size(self.handle, max_tokens, ctypes.byref(b)))
            got = self._ws_sizes[max_tokens] = b.value
        return got

    def workspace(self, max_tokens: int) -> torch.Tensor:
        """A zero-filled workspace for calls of up to max_tokens tokens (cached, grows on demand)."""
        need = self.workspace_size(max_tokens)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(need, dtype=torch.uint8, device=self.w_col.device)
        return self._ws

    def plan(self, T: int):
        arr = (GemmPlan * 2)()
        n = _check(lib().tp_describe_plan(self.handle, T, arr, 2))
        return [{k: getattr(arr[i], k) for k, _ in GemmPlan._fields_} for i in range(n)]

    # ------------------------------------------------------------------ MLP
    def mlp_forward(self, x: torch.Tensor, residual: Optional[torch.Tensor] = None,
                    residual_stream: bool = True, out: Optional[dict] = None, ws: Optional[torch.Tensor] = None,
                    stream=None) -> dict:
        T, H = x.shape
        norm = bool(self.cfg.flags & TP_FLAG_HAS_NORM)
        o = out if out is not None else {}
        if "mlp_out" not in o:
            o["mlp_out"] = torch.empty_like(x)
        if norm and "residual_out" not in o:
            o["residual_out"] = torch.empty_like(x)
        if residual_stream and residual is not None and "residual_stream" not in o:
            o["residual_stream"] = torch.empty_like(x)
        ws = self.workspace(T) if ws is None else ws
        _check(lib().tp_mlp_forward(self.handle, T, _ptr(_bf16(x, "x")), _ptr(residual), _ptr(o.get("residual_out")),
                                    _ptr(o["mlp_out"]), _ptr(o.get("residual_stream")), _ptr(ws), ws.numel(),
                                    _stream(stream)))
        return o

    def mlp_forward_no_alloc(self, x: torch.Tensor, residual: Optional[torch.Tensor] = None,
                             residual_stream: bool = True, out: Optional[dict] = None,
                             status: Optional[torch.Tensor] = None, stream=None) -> dict:
        """tp_mlp_forward_no_alloc: the decode-shaped block with the library's fixed scratch."""
        T, H = x.shape
        norm = bool(self.cfg.flags & TP_FLAG_HAS_NORM)
        o = out if out is not None else {}
        if "mlp_out" not in o:
            o["mlp_out"] = torch.empty_like(x)
        if norm and "residual_out" not in o:
            o["residual_out"] = torch.empty_like(x)
        if residual_stream and residual is not None and "residual_stream" not in o:
            o["residual_stream"] = torch.empty_like(x)
        if status is not None and (status.dtype != torch.int32 or not status.is_cuda or status.numel() < 1
                                   or status.device != self.w_col.device):
            raise ValueError("status must be an int32 CUDA tensor of at least one element on the block's device")
        _check(lib().tp_mlp_forward_no_alloc(self.handle, T, _ptr(_bf16(x, "x")), _ptr(residual),
                                             _ptr(o.get("residual_out")), _ptr(o["mlp_out"]),
                                             _ptr(o.get("residual_stream")), _ptr(status), _stream(stream)))
        return o

    @property
    def gathered(self) -> bool:
        return bool(self.cfg.flags & TP_FLAG_GATHERED)

    def gate_up(self, x: torch.Tensor, h_out: Optional[torch.Tensor] = None, ws=None, stream=None) -> torch.Tensor:
        """h [t][T][I/t] (shard-major), or [T][I] with TP_FLAG_GATHERED."""
        T = x.shape[0]
        t, Is = self.cfg.t, self.cfg.intermediate // self.cfg.t
        if h_out is None:
            shape = (T, t * Is) if self.gathered else (t, T, Is)
            h_out = torch.empty(shape, dtype=torch.bfloat16, device=x.device)
        ws = self.workspace(T) if ws is None else ws
        _check(lib().tp_gate_up_forward(self.handle, T, _ptr(_bf16(x, "x")), _ptr(h_out), _ptr(ws), ws.numel(),
                                        _stream(stream)))
        return h_out

    def down(self, h_in: torch.Tensor, residual: Optional[torch.Tensor] = None, out=None, stream_out=None,
             ws=None, stream=None):
        T = h_in.shape[0] if self.gathered else h_in.shape[1]
        H = self.cfg.hidden
        out = torch.empty(T, H, dtype=torch.bfloat16, device=h_in.device) if out is None else out
        if residual is not None and stream_out is None:
            stream_out = torch.empty_like(out)
        ws = self.workspace(T) if ws is None else ws
        _check(lib().tp_down_forward(self.handle, T, _ptr(_bf16(h_in, "h_in")), _ptr(residual), _ptr(out),
                                     _ptr(stream_out), _ptr(ws), ws.numel(), _stream(stream)))
        return out, stream_out

    # ------------------------------------------------------------------ paged KV cache
    def kv_cache_shape(self, num_blocks: int, block_size: int):
        """Shape of one of the two caches: [t][num_blocks][block_size][kv heads per shard][head_dim]."""
        c = self.cfg
        kv_per = 1 if c.t >= c.n_kv_heads else c.n_kv_heads // c.t
        return (c.t, num_blocks, block_size, kv_per, c.head_dim)

    def kv_cache_write(self, qkv: torch.Tensor, slot_mapping: torch.Tensor, cache_k: torch.Tensor,
                       cache_v: torch.Tensor, ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """Copy every token's k and v heads into its slot (slot_mapping int32 [T], -1 = skip).
        Returns the 16-byte workspace whose first word is the status."""
        T = qkv.shape[0] if self.gathered else qkv.shape[1]
        _, nb, bs, _, _ = cache_k.shape
        ws = torch.zeros(16, dtype=torch.uint8, device=qkv.device) if ws is None else ws
        _check(lib().tp_kv_cache_write(self.handle, T, _ptr(_bf16(qkv, "qkv")), _ptr(slot_mapping),
                                       _ptr(_bf16(cache_k, "cache_k")), _ptr(_bf16(cache_v, "cache_v")), nb, bs,
                                       _ptr(ws), ws.numel(), _stream(stream)))
        return ws

    def paged_attention_workspace_size(self, n_reqs: int, max_query_len: int, max_seq_len: int) -> int:
        b = ctypes.c_int64()
        _check(lib().tp_paged_attention_workspace_size(self.handle, n_reqs, max_query_len, max_seq_len,
                                                       ctypes.byref(b)))
        return b.value

    def paged_attention(self, qkv: torch.Tensor, query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                        block_tables: torch.Tensor, cache_k: torch.Tensor, cache_v: torch.Tensor,
                        max_query_len: int, max_seq_len: int, out=None, ws=None, stream=None, slot_mapping=None):
        """Attention of the new tokens (rows of qkv) over their requests' cached keys; with
        slot_mapping (int32 [T]) the call also writes the new tokens' k and v to their slots.
        Returns (attn in the attention core's output layout, workspace)."""
        c = self.cfg
        T = qkv.shape[0] if self.gathered else qkv.shape[1]
        n_reqs = query_start_loc.numel() - 1
        _, nb, bs, _, _ = cache_k.shape
        if out is None:
            shape = (T, c.n_q_heads * c.head_dim) if self.gathered else (c.t, T, c.n_q_heads // c.t * c.head_dim)
            out = torch.empty(shape, dtype=torch.bfloat16, device=qkv.device)
        if ws is None:
            ws = torch.zeros(self.paged_attention_workspace_size(n_reqs, max_query_len, max_seq_len),
                             dtype=torch.uint8, device=qkv.device)
        for name, a in (("query_start_loc", query_start_loc), ("seq_lens", seq_lens), ("block_tables", block_tables),
                        ("slot_mapping", slot_mapping)):
            if a is None and name == "slot_mapping":
                continue
            if a.dtype != torch.int32 or not a.is_cuda or not a.is_contiguous():
                raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
        _check(lib().tp_paged_attention(self.handle, T, _ptr(_bf16(qkv, "qkv")), _ptr(query_start_loc),
                                        _ptr(seq_lens), n_reqs, int(max_query_len), int(max_seq_len),
                                        _ptr(block_tables), block_tables.shape[1],
                                        _ptr(slot_mapping), _ptr(_bf16(cache_k, "cache_k")),
                                        _ptr(_bf16(cache_v, "cache_v")), nb, bs, _ptr(out), _ptr(ws), ws.numel(),
                                        _stream(stream)))
        return out, ws

    # ------------------------------------------------------------------ mixture of experts
    def moe_forward(self, x: torch.Tensor, expert_ids: torch.Tensor, gates: torch.Tensor, out=None, ws=None,
                    stream=None) -> torch.Tensor:
        """y [T, H] = sum_j gates[:, j] * expert_{ids[:, j]}(x); ids int32 [T, k], gates fp32 [T, k]."""
        T, k = expert_ids.shape
        if expert_ids.dtype != torch.int32 or gates.dtype != torch.float32 or not expert_ids.is_cuda:
            raise TypeError("expert_ids must be int32 and gates float32 CUDA tensors")
        out = torch.empty_like(x) if out is None else out
        ws = self.workspace(T * k) if ws is None else ws
        _check(lib().tp_moe_forward(self.handle, T, k, _ptr(_bf16(x, "x")), _ptr(expert_ids.contiguous()),
                                    _ptr(gates.contiguous()), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
        return out

    # ------------------------------------------------------------------ attention projections
    def attn_proj_forward(self, x: Optional[torch.Tensor], attn_in: Optional[torch.Tensor],
                          qkv_out=None, o_out=None, ws=None, stream=None):
        c = self.cfg
        T = x.shape[0] if x is not None else (attn_in.shape[0] if self.gathered else attn_in.shape[1])
        q_per = c.n_q_heads // c.t
        kv_per = 1 if c.t >= c.n_kv_heads else c.n_kv_heads // c.t
        w_s = (q_per + 2 * kv_per) * c.head_dim
        dev = self.w_col.device
        if x is not None and qkv_out is None:
            shape = (T, c.t * w_s) if self.gathered else (c.t, T, w_s)
            qkv_out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        if attn_in is not None and o_out is None:
            o_out = torch.empty(T, c.hidden, dtype=torch.bfloat16, device=dev)
        ws = self.workspace(T) if ws is None else ws
        _check(lib().tp_attn_proj_forward(self.handle, T, _ptr(x), _ptr(qkv_out if x is not None else None),
                                          _ptr(attn_in), _ptr(o_out if attn_in is not None else None),
                                          _ptr(ws), ws.numel(), _stream(stream)))
        return qkv_out, o_out

    # ------------------------------------------------------------------ attention core
    def attention_forward(self, qkv: torch.Tensor, cu_seqlens: torch.Tensor, max_seqlen: int,
                          out=None, ws=None, stream=None) -> torch.Tensor:
        """Causal GQA attention of every shard's local heads: qkv [t][T][w_s] (the
        projection's output) -> attn [t][T][nq*hd/t] (o_proj's input). cu_seqlens:
        int32 device tensor [n_seqs + 1] of sequence offsets."""
        c = self.cfg
        T = qkv.shape[0] if self.gathered else qkv.shape[1]
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise TypeError("cu_seqlens must be an int32 CUDA tensor")
        if out is None:
            shape = (T, c.n_q_heads * c.head_dim) if self.gathered else (c.t, T, c.n_q_heads // c.t * c.head_dim)
            out = torch.empty(shape, dtype=torch.bfloat16, device=qkv.device)
        ws = self.workspace(T) if ws is None else ws
        _check(lib().tp_attention_forward(self.handle, T, _ptr(_bf16(qkv, "qkv")), _ptr(cu_seqlens),
                                          cu_seqlens.numel() - 1, int(max_seqlen), _ptr(out), _ptr(ws),
                                          ws.numel(), _stream(stream)))
        return out


class TPLayer:
    """One decoder layer (tp_decoder_layer_forward) over an attention handle and an
    MLP handle, both created with TP_FLAG_HAS_NORM (the input and post-attention
    norms). The handles must outlive this object."""

    def __init__(self, attn: TPLinear, mlp: TPLinear, max_tokens: int):
        self.attn, self.mlp, self.max_tokens = attn, mlp, max_tokens
        h = ctypes.c_void_p()
        _check(lib().tp_layer_create(attn.handle, mlp.handle, max_tokens, ctypes.byref(h)))
        self.handle = h
        b = ctypes.c_int64()
        _check(lib().tp_layer_workspace_size(h, ctypes.byref(b)))
        self.workspace_bytes = b.value
        self._ws = None

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            lib().tp_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace(self) -> torch.Tensor:
        if self._ws is None:
            self._ws = torch.zeros(self.workspace_bytes, dtype=torch.uint8, device=self.attn.w_col.device)
        return self._ws

    def forward(self, hidden: torch.Tensor, residual: Optional[torch.Tensor], cu_seqlens: torch.Tensor,
                max_seqlen: int, out: Optional[dict] = None, residual_stream: bool = True, ws=None,
                stream=None) -> dict:
        """Returns {residual_attn, attn_out, residual_mlp, mlp_out[, residual_stream]}, each [T, H]."""
        T = hidden.shape[0]
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise TypeError("cu_seqlens must be an int32 CUDA tensor")
        o = out if out is not None else {}
        for k in ("residual_attn", "attn_out", "residual_mlp", "mlp_out") + (
                ("residual_stream",) if residual_stream else ()):
            if k not in o:
                o[k] = torch.empty_like(hidden)
        io = LayerIO(_bf16(hidden, "hidden").data_ptr(),
                     None if residual is None else _bf16(residual, "residual").data_ptr(),
                     cu_seqlens.data_ptr(), cu_seqlens.numel() - 1, int(max_seqlen),
                     o["residual_attn"].data_ptr(), o["attn_out"].data_ptr(), o["residual_mlp"].data_ptr(),
                     o["mlp_out"].data_ptr(), o["residual_stream"].data_ptr() if "residual_stream" in o else None)
        ws = self.workspace() if ws is None else ws
        _check(lib().tp_decoder_layer_forward(self.handle, T, ctypes.byref(io), _ptr(ws), ws.numel(),
                                              _stream(stream)))
        return o


def add_rms_norm(a: torch.Tensor, residual: Optional[torch.Tensor], gamma: torch.Tensor, eps: float,
                 residual_out=None, x_out=None, stream=None):
    T, H = a.shape
    residual_out = torch.empty_like(a) if residual_out is None else residual_out
    x_out = torch.empty_like(a) if x_out is None else x_out
    _check(lib().tp_add_rms_norm(T, H, _ptr(_bf16(a, "a")), None if residual is None else _ptr(_bf16(residual, "residual")),
                                 _ptr(_bf16(gamma, "gamma")), eps, _ptr(residual_out), _ptr(x_out),
                                 _stream(stream)))
    return x_out, residual_out


def capture_rows(row_req: torch.Tensor, row_pos: torch.Tensor, sel_keys: torch.Tensor,
                 tensors: Sequence[torch.Tensor], tensor_types: Sequence[int], layer: int, capacity: int,
                 ws: Optional[torch.Tensor] = None, stream=None, out=None):
    """Returns (headers int32 [capacity, 6], rows [capacity, H], n_out int64 device scalar, ws).

    out: optional (headers, rows, n_out) tensors to write instead of new ones."""
    T, H = tensors[0].shape
    dev = tensors[0].device
    if out is not None:
        hdr, rows, n_out = out
        if (hdr.dtype != torch.int32 or hdr.shape[0] < max(capacity, 1) or hdr.shape[1] != 6
                or rows.dtype != torch.bfloat16 or rows.shape[0] < max(capacity, 1) or rows.shape[1] != H
                or n_out.dtype != torch.int64 or n_out.numel() < 1):
            raise ValueError("capture out tensors: int32 [capacity, 6], bf16 [capacity, H], int64 [1]")
    else:
        hdr = torch.empty(max(capacity, 1), 6, dtype=torch.int32, device=dev)
        rows = torch.empty(max(capacity, 1), H, dtype=torch.bfloat16, device=dev)
        n_out = torch.zeros(1, dtype=torch.int64, device=dev)
    need = capture_workspace_size(T, sel_keys.numel())
    ws = torch.zeros(need, dtype=torch.uint8, device=dev) if ws is None else ws
    arr = (ctypes.c_void_p * len(tensors))(*[_bf16(t, "tensor").data_ptr() for t in tensors])
    types = (ctypes.c_int32 * len(tensors))(*tensor_types)
    _check(lib().tp_capture_rows(T, H, _ptr(row_req), _ptr(row_pos), _ptr(sel_keys), sel_keys.numel(),
                                 len(tensors), arr, types, layer, _ptr(hdr), _ptr(rows), capacity,
                                 _ptr(n_out), _ptr(ws), ws.numel(), _stream(stream)))
    return hdr, rows, n_out, ws
