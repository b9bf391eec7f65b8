"""One step of the hot path, composed from the three C-ABI calls (marshalling only).

A decode step ("DeepSeek V4.1", attention/query-latent, Attention.forward with start_pos > 0):
  1. the new token's KV row is rounded through fp8 in place and stored to ring slot
     start_pos % window ("Module attn", act_quant_inplace and the ring-cache paragraph);
  2. the window columns of the index rows are written: the whole ring, oldest first
     ("DeepSeek V4.1", attention/attend, get_window_topk_idxs);
  3. sparse_attn over kv = [ring | compressed rows] with idx = [window cols | compressed cols].

A prefill step at start_pos 0 rounds the whole chunk in place (it is also the window part of kv
for this step), keeps its last `window` rows in the ring, writes one causal window row per query
and runs sparse_attn over kv = [chunk | compressed rows].

The caller lays kv out as [window rows | compressed rows] per sequence and idx as
[window cols | compressed cols], so no concatenation copy is made.
"""
from __future__ import annotations

import torch

from . import dsattn


def decode_step(q: torch.Tensor, kv: torch.Tensor, new_kv: torch.Tensor, sink: torch.Tensor, idx: torch.Tensor,
                start_pos: int, window: int, scale: float, o: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q [b][1][h][d]; kv [b][window + C][d] (ring first); new_kv [b][1][d] raw row of this token
    (rounded in place); idx [b][1][window + K] with the compressed columns already filled."""
    b = q.shape[0]
    dsattn.kv_quant_ring_write(new_kv, kv[:, :window], start_pos, window, stream=stream)
    dsattn.window_topk_idxs(idx, b, 1, start_pos, window, stream=stream)
    return dsattn.sparse_attn(q, kv, sink, idx, scale, o=o, workspace=workspace, stream=stream)


def prefill_step(q: torch.Tensor, kv: torch.Tensor, ring: torch.Tensor, sink: torch.Tensor, idx: torch.Tensor,
                 window: int, scale: float, o: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                 stream=None, pairs: bool = False) -> torch.Tensor:
    """q [b][s][h][d]; kv [b][s + C][d] (the raw chunk first, rounded in place); ring [b][window][d];
    idx [b][s][min(s, window) + K] with the compressed columns already filled.  pairs: neighbouring
    queries share one gather (ds_sparse_attn_prefill; its own workspace size)."""
    b, s = q.shape[0], q.shape[1]
    dsattn.kv_quant_ring_write(kv[:, :s], ring, 0, window, stream=stream)
    dsattn.window_topk_idxs(idx, b, s, 0, window, stream=stream)
    if pairs:
        return dsattn.sparse_attn_prefill(q, kv, sink, idx, scale, o=o, workspace=workspace, stream=stream)
    return dsattn.sparse_attn(q, kv, sink, idx, scale, o=o, workspace=workspace, stream=stream)
