"""Python face of the captured decode step: torch owns device memory (weights,
workspace) and streams; libgraphdec.so does every step of the computation.

    dec = Decoder(config, weights, cap=8192, rows=1)
    res = dec.step(tokens, pos)          # slot write, one graph launch, readback
    res.ids, res.logits, res.nonfinite
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import _binding as B

_ROLE = {"attn_norm": B.DEC_W_ATTN_NORM, "wq": B.DEC_W_Q, "wk": B.DEC_W_K, "wv": B.DEC_W_V, "wo": B.DEC_W_O,
         "ffn_norm": B.DEC_W_FFN_NORM, "wg": B.DEC_W_GATE, "wu": B.DEC_W_UP, "wd": B.DEC_W_DOWN}
_DT = {torch.float32: B.DEC_DTYPE_F32, torch.bfloat16: B.DEC_DTYPE_BF16}
_DTN = {"f32": B.DEC_DTYPE_F32, "bf16": B.DEC_DTYPE_BF16}


@dataclass
class StepResult:
    logits: Optional[np.ndarray]   # [rows, vocab] float32, if asked for
    ids: np.ndarray                # [rows] int32 greedy token ids
    nonfinite: np.ndarray          # [rows] uint8


class _DevArray:
    """A raw device allocation seen through __cuda_array_interface__ (no copy)."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"data": (ptr, False), "shape": tuple(shape), "typestr": typestr,
                                         "strides": None, "version": 2}


def make_config(n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_hidden, vocab, weight_dtype="bf16",
                kv_dtype="bf16", rms_eps=1e-5, rope_theta=1e4, device=0, wait_timeout_ms=0) -> B.dec_config:
    return B.dec_config(n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_hidden, vocab,
                        _DTN.get(weight_dtype, weight_dtype), _DTN.get(kv_dtype, kv_dtype), device,
                        float(rms_eps), float(rope_theta), int(wait_timeout_ms))


def make_sampler(temperature: float = 0.0, top_k: int = 1, top_p: float = 1.0, min_p: float = 0.0, seed: int = 0,
                 n_logprobs: int = 0) -> B.dec_sampler:
    s = B.dec_sampler()
    s.temperature, s.top_k, s.top_p, s.min_p = float(temperature), int(top_k), float(top_p), float(min_p)
    s.seed, s.n_logprobs = int(seed) & 0xFFFFFFFFFFFFFFFF, int(n_logprobs)
    return s


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


class Decoder:
    """One handle: weights bound by role, one capture (cap, rows, kv layout)."""

    def __init__(self, cfg: B.dec_config, weights: dict, cap: int, rows: int = 1, kv_layout: str = "contiguous",
                 page_size: int = 16, num_pages: int = 0, stream: Optional[torch.cuda.Stream] = None,
                 lib_workspace: bool = False, strategy: str = "graph", sampler: Optional[dict] = None,
                 kv_sweep: str = "cap"):
        self.cfg = cfg
        self.rows, self.cap = rows, cap
        self.layout = B.DEC_KV_PAGED if kv_layout == "paged" else B.DEC_KV_CONTIGUOUS
        self.page_size = page_size if self.layout == B.DEC_KV_PAGED else 0
        self.num_pages = num_pages if self.layout == B.DEC_KV_PAGED else 0
        self.h = B.dec_init(cfg)
        self._weights = weights   # borrowed device memory must outlive the handle
        try:
            B.dec_load_weights(self.h, self._bindings(weights))
            B.dec_set_strategy(self.h, B.DEC_STRATEGY_PERSISTENT if strategy == "persistent" else B.DEC_STRATEGY_GRAPH)
            # "cap": the constant-shape sweep of [0, cap); "pos": stop at the tile holding pos (same results)
            B.dec_set_kv_sweep(self.h, B.DEC_SWEEP_POS if kv_sweep == "pos" else B.DEC_SWEEP_CAP)
            if sampler is not None:   # records the sampling kernel after the head
                B.check(self.h, B.dec_set_sampler(self.h, make_sampler(**sampler)))
            self.ws = None
            ws_ptr, ws_bytes = None, 0
            if not lib_workspace:
                ws_bytes = B.dec_workspace_size(cfg, cap, rows, self.layout, self.page_size, self.num_pages)
                self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=f"cuda:{cfg.device}")
                ws_ptr = self.ws.data_ptr()
            sptr = stream.cuda_stream if stream is not None else None
            B.dec_capture(self.h, cap, rows, self.layout, self.page_size, self.num_pages, ws_ptr, ws_bytes, sptr)
        except Exception:
            B.dec_destroy(self.h)
            self.h = None
            raise
        self.vocab = cfg.vocab
        self.device = torch.device(f"cuda:{cfg.device}")
        self._hstream = torch.cuda.ExternalStream(B.dec_stream(self.h), device=self.device)
        self._ev = torch.cuda.Event()
        self._logits = np.empty((rows, cfg.vocab), dtype=np.float32)
        self._ids = np.empty(rows, dtype=np.int32)
        self._nf = np.empty(rows, dtype=np.uint8)

    def _bindings(self, w: dict):
        out = []

        def add(role, layer, t: torch.Tensor):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("weights must be contiguous CUDA tensors")
            rows = t.shape[0]
            cols = t.shape[1] if t.dim() == 2 else 1
            out.append(B.dec_weight(role, layer, _DT[t.dtype], 0, rows, cols, t.data_ptr()))

        add(B.DEC_W_EMBED, -1, w["embed"])
        add(B.DEC_W_FINAL_NORM, -1, w["final_norm"])
        add(B.DEC_W_LM_HEAD, -1, w["lm_head"])
        for l, lw in enumerate(w["layers"]):
            for name, role in _ROLE.items():
                add(role, l, lw[name])
        return out

    def _after_torch(self) -> None:
        """Order the handle's stream after work torch queued on its current stream
        (e.g. KV pre-fill or input tensors written through torch)."""
        self._ev.record(torch.cuda.current_stream(self.device))
        self._hstream.wait_event(self._ev)

    # ---- stepping ----
    def step(self, tokens, pos, write_map=None, logits: bool = True) -> StepResult:
        tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(self.rows)
        ps = np.ascontiguousarray(pos, dtype=np.int32).reshape(self.rows)
        wm = None if write_map is None else np.ascontiguousarray(write_map, dtype=np.int32).reshape(self.rows)
        self._after_torch()
        rc = B.dec_step(self.h, _ptr(tok), _ptr(ps), _ptr(wm), _ptr(self._logits) if logits else None,
                        _ptr(self._ids), _ptr(self._nf))
        B.check(self.h, rc)
        return StepResult(self._logits.copy() if logits else None, self._ids.copy(), self._nf.copy())

    def chain(self, tokens, pos, n_steps: int):
        """n_steps chained greedy steps from (tokens, pos): the device feeds each
        step's ids to the next; returns (ids [n_steps, rows], nonfinite [n_steps, rows])."""
        tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(self.rows)
        ps = np.ascontiguousarray(pos, dtype=np.int32).reshape(self.rows)
        ids = np.empty((n_steps, self.rows), dtype=np.int32)
        nf = np.empty((n_steps, self.rows), dtype=np.uint8)
        self._after_torch()
        B.check(self.h, B.dec_chain(self.h, int(n_steps), _ptr(tok), _ptr(ps), _ptr(ids), _ptr(nf)))
        return ids, nf

    def prefill(self, pages, tokens, pos0: int = 0):
        """Multi-token prefill of one sequence through the paged step (rows tokens
        per chunk): returns (logits [vocab] after the last token, greedy id)."""
        pg = np.ascontiguousarray(pages, dtype=np.int32).reshape(-1)
        tk = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        logits = np.empty(self.vocab, dtype=np.float32)
        idv = np.zeros(1, dtype=np.int32)
        self._after_torch()
        B.check(self.h, B.dec_prefill(self.h, _ptr(pg), _ptr(tk), int(tk.size), int(pos0), _ptr(logits), _ptr(idv)))
        return logits, int(idv[0])

    def prefill_block(self, tokens, pos0: int = 0, row: int = 0, pages=None):
        """Block prefill of one sequence (tensor-core projections, causal attention
        over the block): row's contiguous K/V, or the sequence on `pages` (paged).
        Returns (logits [vocab] after the last token, greedy id)."""
        tk = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        pg = None if pages is None else np.ascontiguousarray(pages, dtype=np.int32).reshape(-1)
        logits = np.empty(self.vocab, dtype=np.float32)
        idv = np.zeros(1, dtype=np.int32)
        self._after_torch()
        B.check(self.h, B.dec_prefill_block(self.h, int(row), _ptr(pg), _ptr(tk), int(tk.size), int(pos0),
                                            _ptr(logits), _ptr(idv)))
        return logits, int(idv[0])

    def set_sampler(self, **params) -> None:
        """New sampler parameters for the coming steps (the decoder must have been
        built with a sampler); see make_sampler for the fields."""
        B.check(self.h, B.dec_set_sampler(self.h, make_sampler(**params)))

    def logprobs(self, n: int):
        """Top-n logprobs of the last step: (ids [rows, n], logprobs [rows, n])."""
        ids = np.empty((self.rows, n), dtype=np.int32)
        vals = np.empty((self.rows, n), dtype=np.float32)
        B.check(self.h, B.dec_logprobs(self.h, int(n), _ptr(ids), _ptr(vals)))
        return ids, vals

    def launch(self, dev_slots: Optional[torch.Tensor]) -> None:
        """Asynchronous step from a device slot record [3*rows] int32 (tokens, pos, write map)."""
        self._after_torch()
        B.check(self.h, B.dec_launch(self.h, None if dev_slots is None else dev_slots.data_ptr()))

    def wait(self, logits: bool = False) -> StepResult:
        rc = B.dec_wait(self.h, _ptr(self._logits) if logits else None, _ptr(self._ids), _ptr(self._nf))
        B.check(self.h, rc)
        return StepResult(self._logits.copy() if logits else None, self._ids.copy(), self._nf.copy())

    def attention(self, layer: int, qkv: torch.Tensor, pos: torch.Tensor, out: torch.Tensor) -> None:
        """One layer's attention on device tensors: qkv [rows, (Hq+2Hkv)*hd] fp32,
        pos [rows] int32, out [rows, Hq*hd] fp32 (written)."""
        for t, dt in ((qkv, torch.float32), (pos, torch.int32), (out, torch.float32)):
            if not t.is_cuda or not t.is_contiguous() or t.dtype != dt:
                raise ValueError("attention: contiguous CUDA tensors of the documented dtypes")
        self._after_torch()
        B.check(self.h, B.dec_attention(self.h, layer, qkv.data_ptr(), pos.data_ptr(), out.data_ptr()))

    def set_slot_map(self, slot_map: np.ndarray) -> None:
        m = np.ascontiguousarray(slot_map, dtype=np.int32)
        B.check(self.h, B.dec_set_slot_map(self.h, _ptr(m)))

    def set_eager(self, eager: bool) -> None:
        B.dec_set_eager(self.h, eager)

    def reset_state(self) -> None:
        self._after_torch()
        B.check(self.h, B.dec_reset_state(self.h))

    # ---- views of device state ----
    def kv(self, layer: int, which: int) -> torch.Tensor:
        """Zero-copy view of one layer's K (0) or V (1) store:
        contiguous [rows, n_kv_heads, cap, head_dim], paged [num_pages, n_kv_heads, page_size, head_dim]."""
        ptr, nbytes = B.dec_kv_ptr(self.h, layer, which)
        c = self.cfg
        if self.layout == B.DEC_KV_PAGED:
            shape = (self.num_pages, c.n_kv_heads, self.page_size, c.head_dim)
        else:
            shape = (self.rows, c.n_kv_heads, self.cap, c.head_dim)
        if c.kv_dtype == B.DEC_DTYPE_BF16:
            t = torch.as_tensor(_DevArray(ptr, shape, "<i2"), device=f"cuda:{c.device}")
            return t.view(torch.bfloat16)
        return torch.as_tensor(_DevArray(ptr, shape, "<f4"), device=f"cuda:{c.device}")

    def logits_device(self) -> torch.Tensor:
        ptr = B.dec_logits_ptr(self.h)
        return torch.as_tensor(_DevArray(ptr, (self.rows, self.vocab), "<f4"), device=f"cuda:{self.cfg.device}")

    def stream(self) -> torch.cuda.ExternalStream:
        return self._hstream

    def stats(self) -> dict:
        st = B.dec_stats_get(self.h)
        return {f: getattr(st, f) for f, _ in B.dec_stats._fields_}

    def close(self) -> None:
        if self.h:
            B.dec_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
