"""Float64 CPU oracle of the tensor-parallel decoder linear block.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (``--impl reference`` and the ``cpu_baseline`` object) may call it. It
shares no code with the CUDA library; the only common dependency is the
seeded input generator in ``workloads/``, which holds no block arithmetic.

Sources, cited by page title and section throughout:

* [UC]  "Tensor & pipeline parallelism" (Undercurrent internals, vLLM
        parallelism page): what the capture hooks see and how records are
        keyed and ordered.
* [VCR] "vLLM Code Reading (Section 5): GPUWorker.execute_model 与 PP/TP 通信",
        sections 11-14: column/row split identities, attention and MLP TP
        data flow.
* [VSC] "vLLM 源码完全拆解（十一）：模型并行与 Worker 层", sections on the
        linear-layer split, ColumnParallelLinear, MergedColumnParallelLinear /
        QkvParallelLinear, RowParallelLinear and the column-row block.
* [MLX] mlxcel manual "Tensor Parallelism": Weight Sharding Strategies,
        GQA-Aware Attention Sharding.

``attention.py`` holds the attention core between the QKV projection and
o_proj (causal, GQA, sequences packed by offsets); the pages describe it
only as attention over each rank's own heads, so it is the textbook
scaled dot-product attention in their head layout. ``decoder_layer.py``
chains the steps into one decoder layer (input norm, QKV, attention, o_proj,
add + norm, MLP) in the order the pages give. ``moe.py`` is the top-k
mixture-of-experts block whose experts are split by the same column/row
pattern (within-expert tensor parallelism); its routing is an input.
``kv_cache.py`` is the paged KV cache: the write of each new token's keys and
values to its slot, and attention of new tokens over their requests' cached
keys through the block tables.

Every function computes in float64 from bf16 inputs converted exactly. Where
the block has a plain definition (the unsharded Y = XW, SiLU, RMSNorm, row
selection) the oracle is that definition; the sharded variants
(``column_parallel``, ``row_parallel``, ``mlp_block_tp``, ``qkv_parallel``,
``o_proj_parallel``) restate the pages' split algebra and exist to pin the
invariants the pages fix.

Parity status: every function here is pinned by tests in
``tests/test_oracle.py`` (brute force, closed forms, library routines,
page-printed head counts in ``tests/golden/``). None is "parity unpinned".
"""
from .tp_block import (  # noqa: F401
    bf16_to_f64, linear, column_parallel, row_parallel, silu, silu_mul, rms_norm,
    add_rms_norm, mlp_block, mlp_block_tp, mlp_layer, gqa_partition, qkv_shard_rows,
    qkv_parallel, o_proj_parallel, divide, reduce_scatter,
)
from .capture import capture_rows, pack_key  # noqa: F401
from .attention import attention_core, attention_rows, kv_head_of  # noqa: F401
from .decoder_layer import decoder_layer  # noqa: F401
from .moe import moe_block, moe_block_tp  # noqa: F401
from .kv_cache import kv_cache_write, paged_attention, slot_of  # noqa: F401
