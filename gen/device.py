"""Placing generated inputs in device memory (data movement only).

* ``upload_weights``: host weights (gen.ModelWeights) -> torch CUDA tensors in
  the dict layout ``graph_replay_gb300.Decoder`` binds by role.
* ``place_kv``: a block of logical K or V rows [n, n_kv_heads, head_dim] of one
  sequence -> the decoder's KV store, contiguous [rows, n_kv_heads, cap, hd] or
  paged [num_pages, n_kv_heads, page, hd] through the page table.
"""
from __future__ import annotations

import numpy as np
import torch

from .workloads import LAYER_ROLES


def to_tensor(a: np.ndarray, device) -> torch.Tensor:
    """uint16 arrays hold bf16 bit patterns; float32 arrays stay float32."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def upload_weights(mw, device="cuda:0") -> dict:
    w = {"embed": to_tensor(mw.embed, device), "final_norm": to_tensor(mw.final_norm, device),
         "lm_head": to_tensor(mw.lm_head, device), "layers": []}
    for lw in mw.layers:
        w["layers"].append({r: to_tensor(lw[r], device) for r in LAYER_ROLES})
    return w


def place_kv(store: torch.Tensor, block: np.ndarray, row: int, start: int = 0, slot_map=None, page_size: int = 0):
    """Write logical positions [start, start + n) of sequence `row` into the store."""
    n = block.shape[0]
    if n == 0:
        return
    t = to_tensor(np.ascontiguousarray(block), store.device)      # [n, Hkv, hd]
    if slot_map is None:
        store[row, :, start:start + n, :] = t.permute(1, 0, 2)
        return
    P = page_size
    j = start
    while j < start + n:
        pg = int(slot_map[row][j // P])
        off = j % P
        take = min(P - off, start + n - j)
        store[pg, :, off:off + take, :] = t[j - start:j - start + take].permute(1, 0, 2)
        j += take


def read_kv(store: torch.Tensor, row: int, npos: int, slot_map=None, page_size: int = 0) -> np.ndarray:
    """Logical positions [0, npos) of sequence `row` as [npos, Hkv, hd] (uint16 bf16 bits or float32)."""
    if slot_map is None:
        t = store[row, :, :npos, :].permute(1, 0, 2).contiguous()
    else:
        P = page_size
        parts = []
        for pg_i in range((npos + P - 1) // P):
            pg = int(slot_map[row][pg_i])
            take = min(P, npos - pg_i * P)
            parts.append(store[pg, :, :take, :].permute(1, 0, 2))
        t = torch.cat(parts, 0).contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()
