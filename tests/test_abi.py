"""The C ABI without a GPU: the library loads, exports what the header declares,
and rejects bad arguments on the host (the pages' divide() rule, the power-of-2
shard count, null and misaligned pointers) before touching the device.
"""
import ctypes
import os
import re

import pytest

import tensor_linear_layers_gb300 as tl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tp_linear.h")


@pytest.fixture(scope="module")
def L():
    from tensor_linear_layers_gb300 import _build
    _build.build()
    return tl.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tp_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_binding_symbols():
    assert set(declared_functions()) == set(tl.ABI_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_symbols_have_c_linkage():
    out = os.popen(f"nm -D --defined-only {tl.LIB_PATH}").read()
    exported = set(re.findall(r"\bT (tp_[a-z_0-9]+)\b", out))
    assert set(declared_functions()) <= exported


def cfg_mlp(t=2, H=512, I=1408, flags=0):
    return tl.make_config(tl.TP_BLOCK_MLP, t, H, I, flags=flags)


BLOCK = 256 * 64 * 2     # packed weight block: 256 rows x 64 K elements, bf16


def cdiv(a, b):
    return -(-a // b)


def test_packed_bytes_mlp(L):
    # gate_up: t shards x ceil(I/t / 128) blocks of [128 gate | 128 up] rows x ceil(H/64) k-blocks
    col, row = tl.packed_weight_bytes(cfg_mlp())
    assert col == 2 * cdiv(704, 128) * cdiv(512, 64) * BLOCK
    # down: ceil(H/256) row tiles x t shards x ceil(I/t / 64) k-blocks
    assert row == cdiv(512, 256) * 2 * cdiv(704, 64) * BLOCK
    assert col >= 2 * 1408 * 512 * 2 and row >= 512 * 1408 * 2


def test_packed_bytes_attention_gqa(L):
    # 32 q heads, 8 kv heads, hd 128, t=4: shard = 8 q + 2 k + 2 v heads = 1536 rows
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, 4, 4096, n_q_heads=32, n_kv_heads=8, head_dim=128)
    col, row = tl.packed_weight_bytes(cfg)
    assert col == cdiv(4 * 1536, 256) * 64 * BLOCK == 4 * 12 * 128 * 4096 * 2
    assert row == 4096 * 4096 * 2
    # t=8 with 4 kv heads: kv heads replicated, one per shard
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, 8, 4096, n_q_heads=32, n_kv_heads=4, head_dim=128)
    col, _ = tl.packed_weight_bytes(cfg)
    assert col == 8 * (4 + 2) * 128 * 4096 * 2


@pytest.mark.parametrize("cfg,code", [
    (cfg_mlp(t=4, I=1410), tl.TP_ERR_SHAPE),              # divide(): I % t != 0
    (cfg_mlp(t=3, I=1410), tl.TP_ERR_UNSUPPORTED),        # t not a power of 2
    (cfg_mlp(t=16, I=4096), tl.TP_ERR_UNSUPPORTED),
    (cfg_mlp(t=0), tl.TP_ERR_SHAPE),
    (cfg_mlp(H=500), tl.TP_ERR_UNSUPPORTED),
    (cfg_mlp(t=8, I=1416), tl.TP_ERR_UNSUPPORTED),        # I/t = 177, not a multiple of 8
    (cfg_mlp(flags=4), tl.TP_ERR_ARG),
    (tl.make_config(tl.TP_BLOCK_ATTN_PROJ, 4, 4096, n_q_heads=30, n_kv_heads=6, head_dim=128),
     tl.TP_ERR_SHAPE),
    (tl.make_config(tl.TP_BLOCK_ATTN_PROJ, 4, 4096, n_q_heads=24, n_kv_heads=3, head_dim=128),
     tl.TP_ERR_SHAPE),
    (tl.make_config(7, 4, 4096), tl.TP_ERR_ARG),
])
def test_bad_configs_rejected(L, cfg, code):
    with pytest.raises(tl.TPError) as e:
        tl.packed_weight_bytes(cfg)
    assert e.value.code == code


def test_create_rejects_null_and_misaligned_pointers(L):
    cfg = cfg_mlp()
    h = ctypes.c_void_p()
    arr = (ctypes.c_void_p * 3)(0x1000, 0x2000, 0x3000)
    rc = L.tp_linear_create(ctypes.byref(cfg), arr, 2, ctypes.c_void_p(0x4000), ctypes.c_void_p(0x5000),
                            None, None, ctypes.byref(h))
    assert rc == tl.TP_ERR_ARG and b"expected 3" in L.tp_last_error()
    arr_bad = (ctypes.c_void_p * 3)(0x1000, 0x2008, 0x3000)
    rc = L.tp_linear_create(ctypes.byref(cfg), arr_bad, 3, ctypes.c_void_p(0x4000), ctypes.c_void_p(0x5000),
                            None, None, ctypes.byref(h))
    assert rc == tl.TP_ERR_ARG and b"aligned" in L.tp_last_error()
    rc = L.tp_linear_create(ctypes.byref(cfg), arr, 3, None, ctypes.c_void_p(0x5000), None, None,
                            ctypes.byref(h))
    assert rc == tl.TP_ERR_ARG
    cfg_n = cfg_mlp(flags=tl.TP_FLAG_HAS_NORM)
    rc = L.tp_linear_create(ctypes.byref(cfg_n), arr, 3, ctypes.c_void_p(0x4000), ctypes.c_void_p(0x5000),
                            None, None, ctypes.byref(h))
    assert rc == tl.TP_ERR_ARG and b"gamma" in L.tp_last_error()
    assert not h.value


def test_null_handle_and_negative_tokens(L):
    assert L.tp_mlp_forward(None, 4, None, None, None, None, None, None, 0, None) == tl.TP_ERR_ARG
    assert L.tp_add_rms_norm(-1, 512, None, None, None, 1e-5, None, None, None) == tl.TP_ERR_SHAPE
    assert L.tp_add_rms_norm(4, 500, None, None, None, 1e-5, None, None, None) == tl.TP_ERR_UNSUPPORTED


def test_zero_tokens_enqueue_nothing(L):
    # T == 0 is a step with no forward pass: valid pointers, nothing launched, TP_OK
    p = ctypes.c_void_p(0x10000)
    assert L.tp_add_rms_norm(0, 512, p, p, p, 1e-5, p, p, None) == tl.TP_OK


def test_capture_argument_checks(L):
    b = ctypes.c_int64()
    assert L.tp_capture_workspace_size(2048, 205, ctypes.byref(b)) == tl.TP_OK and b.value > 0
    assert L.tp_capture_workspace_size(-1, 1, ctypes.byref(b)) == tl.TP_ERR_SHAPE
    p = ctypes.c_void_p(0x10000)
    arr = (ctypes.c_void_p * 1)(0x10000)
    types = (ctypes.c_int32 * 1)(2)
    rc = L.tp_capture_rows(16, 512, p, p, p, 4, 9, arr, types, 0, p, p, 8, p, p, 1 << 20, None)
    assert rc == tl.TP_ERR_UNSUPPORTED     # more than 8 tensors
    rc = L.tp_capture_rows(16, 512, None, p, p, 4, 1, arr, types, 0, p, p, 8, p, p, 1 << 20, None)
    assert rc == tl.TP_ERR_ARG
    rc = L.tp_capture_rows(16, 512, p, p, p, 4, 1, arr, types, 0, p, p, 8, p, p, 16, None)
    assert rc == tl.TP_ERR_ARG and b"too small" in L.tp_last_error()


def test_wait_limit_must_be_positive(L):
    assert L.tp_set_wait_timeout(0) == tl.TP_ERR_ARG
    assert L.tp_set_wait_timeout(-5) == tl.TP_ERR_ARG
    assert L.tp_set_wait_timeout(2_000_000_000) == tl.TP_OK


def test_layer_calls_reject_null_arguments(L):
    h = ctypes.c_void_p()
    assert L.tp_layer_create(None, None, 128, ctypes.byref(h)) == tl.TP_ERR_ARG and not h.value
    assert L.tp_layer_create(None, None, 128, None) == tl.TP_ERR_ARG
    b = ctypes.c_int64()
    assert L.tp_layer_workspace_size(None, ctypes.byref(b)) == tl.TP_ERR_ARG
    io = tl.LayerIO()
    assert L.tp_decoder_layer_forward(None, 16, ctypes.byref(io), None, 0, None) == tl.TP_ERR_ARG
    assert L.tp_layer_destroy(None) == tl.TP_OK


def test_attention_handle_accepts_the_input_norm_flag(L):
    # the attention handle may carry the layer's input RMSNorm; unknown flags stay errors
    cfg = tl.make_config(tl.TP_BLOCK_ATTN_PROJ, 4, 4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                         flags=tl.TP_FLAG_HAS_NORM)
    assert tl.packed_weight_bytes(cfg)[1] == 4096 * 4096 * 2
    cfg.flags = tl.TP_FLAG_HAS_NORM | tl.TP_FLAG_GATHERED    # gathered layout: accepted
    assert tl.packed_weight_bytes(cfg)[1] == 4096 * 4096 * 2
    cfg.flags = 4
    with pytest.raises(tl.TPError) as e:
        tl.packed_weight_bytes(cfg)
    assert e.value.code == tl.TP_ERR_ARG
    cfg.flags, cfg.rms_eps = tl.TP_FLAG_HAS_NORM, -1.0
    with pytest.raises(tl.TPError) as e:
        tl.packed_weight_bytes(cfg)
    assert e.value.code == tl.TP_ERR_ARG


def test_norm_without_residual_passes_host_checks(L):
    # a first layer has no incoming residual: residual_in may be NULL (T = 0: nothing launched)
    p = ctypes.c_void_p(0x10000)
    assert L.tp_add_rms_norm(0, 512, p, None, p, 1e-5, p, p, None) == tl.TP_OK


def test_moe_config_and_packing(L):
    # each expert is packed in the dense MLP layout, experts one after another
    dense = tl.packed_weight_bytes(cfg_mlp(t=4, H=512, I=1024))
    moe = tl.packed_weight_bytes(tl.make_config(tl.TP_BLOCK_MOE, 4, 512, 1024, n_experts=8))
    assert moe == (8 * dense[0], 8 * dense[1])
    for cfg, code in [
        (tl.make_config(tl.TP_BLOCK_MOE, 4, 512, 1024, n_experts=0), tl.TP_ERR_UNSUPPORTED),
        (tl.make_config(tl.TP_BLOCK_MOE, 4, 512, 1024, n_experts=257), tl.TP_ERR_UNSUPPORTED),
        (tl.make_config(tl.TP_BLOCK_MOE, 4, 512, 1026, n_experts=8), tl.TP_ERR_SHAPE),
        (tl.make_config(tl.TP_BLOCK_MOE, 4, 512, 1024, n_experts=8, flags=tl.TP_FLAG_HAS_NORM), tl.TP_ERR_ARG),
        (tl.make_config(tl.TP_BLOCK_MLP, 4, 512, 1024, n_experts=2), tl.TP_ERR_ARG),
    ]:
        with pytest.raises(tl.TPError) as e:
            tl.packed_weight_bytes(cfg)
        assert e.value.code == code


def test_moe_forward_rejects_null_handle(L):
    assert L.tp_moe_forward(None, 4, 2, None, None, None, None, None, 0, None) == tl.TP_ERR_ARG


def test_kv_cache_calls_reject_null_handle(L):
    p = ctypes.c_void_p(0x10000)
    b = ctypes.c_int64()
    assert L.tp_kv_cache_write(None, 4, p, p, p, p, 16, 16, p, 16, None) == tl.TP_ERR_ARG
    assert L.tp_paged_attention_workspace_size(None, 4, 1, 256, ctypes.byref(b)) == tl.TP_ERR_ARG
    assert L.tp_paged_attention(None, 4, p, p, p, 4, 1, 256, p, 16, None, p, p, 16, 16, p, p, 1 << 20,
                                None) == tl.TP_ERR_ARG
