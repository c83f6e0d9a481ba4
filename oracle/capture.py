"""Activation-capture reference (test infrastructure only).

[UC] "What the adapter hooks": forward hooks on the decoder layer
(residual_stream), self_attn (attn_out), mlp (mlp_out) and the final norm
(final_norm) fire after the module's forward() returns, i.e. after the
row-parallel reduction. Rows of the step's batch are mapped to
(request_id, token_pos) and the rows whose key was registered are recorded.
[UC] "Duplicate records across TP ranks": a record is keyed by
(request_id, extraction point, layer, token_pos, ...), so a key selected twice
still yields one record per row and tensor. [UC] "Merging records from several
stages": within one worker the capture order is kept; hooks fire in forward
order, one tensor after another, and a hook walks its batch rows in order.
"""
from __future__ import annotations

import numpy as np


def pack_key(req, pos):
    """Selector key of (request_id, token_pos): request in the high 32 bits, position in the low."""
    return (np.asarray(req, np.int64) << 32) | (np.asarray(pos, np.int64) & 0xFFFFFFFF)


def capture_rows(row_req, row_pos, sel_keys, tensors, tensor_types, layer: int):
    """Records for every (tensor, row) whose (request_id, token_pos) is selected.

    Order: tensors in the order given (hook-firing order), rows ascending
    within a tensor. Returns (headers int32 [n, 5] = request_id, token_pos,
    tensor_type, layer, row; rows [n, H] copied unchanged).
    """
    wanted = set(int(k) for k in np.asarray(sel_keys, np.int64).ravel())
    hdrs, rows = [], []
    T = len(row_req)
    for tensor, ttype in zip(tensors, tensor_types):
        for i in range(T):
            if int(pack_key(row_req[i], row_pos[i])) in wanted:
                hdrs.append((int(row_req[i]), int(row_pos[i]), int(ttype), int(layer), i))
                rows.append(np.asarray(tensor[i]))
    H = np.asarray(tensors[0]).shape[1] if len(tensors) else 0
    h = np.array(hdrs, dtype=np.int32).reshape(-1, 5)
    if rows:
        out = np.stack(rows)
    else:
        out = np.zeros((0, H), dtype=np.asarray(tensors[0]).dtype if len(tensors) else np.float64)
    return h, out
