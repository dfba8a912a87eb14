"""The five synthetic decode workloads and how their inputs are drawn.

Shapes follow the pages' subject, a Llama-style pre-norm decoder
(``x += mixer(norm(x)); x += ffn(norm(x))``, "Models, Registry and the Driver",
standard_stack): an embedding, per layer RMSNorm + QKV + RoPE + attention +
output projection and RMSNorm + SwiGLU MLP, then a final norm and an LM head.

Recipe (all from the counter-based generator, one stream per tensor):
  * matrices and embeddings: N(0, 0.02), stored in the weight dtype;
  * norm gains: exactly 1.0 (``gain_sigma == 0``) or 1 + N(0, gain_sigma);
  * prompt tokens: uniform in [0, vocab);
  * pre-filled KV: N(0, 1) per (layer, K|V, row), in logical order
    [position, kv_head, head_dim], rounded to the KV dtype;
  * paged KV: the page table is a seeded permutation of the pool, row r owning
    pages perm[r * cap/page : (r + 1) * cap/page];
  * per-row positions: fixed lists, or uniform in [0, cap) from a seed.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

from . import normal, ints, permutation


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_hidden: int
    vocab: int
    wdtype: str            # "f32" | "bf16"
    kvdtype: str           # "f32" | "bf16"
    cap: int
    rows: int
    layout: str = "contiguous"   # "contiguous" | "paged"
    page_size: int = 16
    num_pages: int = 0
    rms_eps: float = 1e-5
    rope_theta: float = 1e4
    gain_sigma: float = 0.0
    prompt_len: int = 0
    decode_steps: int = 0
    positions: tuple = ()
    seed: int = 1234

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def weight_bytes(self) -> int:
        """Bytes of every matrix once plus `rows` embedding rows and the gains."""
        es = 2 if self.wdtype == "bf16" else 4
        d, F, V, L = self.d_model, self.ffn_hidden, self.vocab, self.n_layers
        per_layer = (self.q_dim + 2 * self.kv_dim) * d + d * self.q_dim + 3 * F * d + 2 * d
        return es * (L * per_layer + V * d + d + self.rows * d)

    def kv_swept_bytes(self) -> int:
        """Cap-swept K and V bytes per step: rows * layers * 2 * cap * kv_dim."""
        es = 2 if self.kvdtype == "bf16" else 4
        return es * self.rows * self.n_layers * 2 * self.cap * self.kv_dim

    def step_bytes(self) -> int:
        return self.weight_bytes() + self.kv_swept_bytes()


WORKLOADS = {
    # configuration 1: tiny fp32 MHA decoder
    "tiny": Workload("tiny", n_layers=2, d_model=64, n_heads=4, n_kv_heads=4, head_dim=16,
                     ffn_hidden=128, vocab=256, wdtype="f32", kvdtype="f32", cap=64, rows=1,
                     rms_eps=1e-5, rope_theta=1e4, prompt_len=16, decode_steps=32),
    # configuration 2: 1B-class GQA decoder, bf16 weights, fp32 accumulate
    "1b": Workload("1b", n_layers=16, d_model=2048, n_heads=32, n_kv_heads=8, head_dim=64,
                   ffn_hidden=8192, vocab=32000, wdtype="bf16", kvdtype="bf16", cap=4096, rows=1,
                   rope_theta=5e5, prompt_len=128, decode_steps=256),
    # configuration 3: 8B-shape GQA decoder, batch 1, KV pre-filled up to pos
    "8b": Workload("8b", n_layers=32, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128,
                   ffn_hidden=14336, vocab=128256, wdtype="bf16", kvdtype="bf16", cap=8192, rows=1,
                   rope_theta=5e5, positions=(1, 1024, 4096, 8191)),
    # configuration 4: 8B-shape, 8 rows, paged KV (16-token pages, pool of 4096)
    "8b_paged": Workload("8b_paged", n_layers=32, d_model=4096, n_heads=32, n_kv_heads=8,
                         head_dim=128, ffn_hidden=14336, vocab=128256, wdtype="bf16",
                         kvdtype="bf16", cap=8192, rows=8, layout="paged", page_size=16,
                         num_pages=4096, rope_theta=5e5),
    # configuration 5: 1B-class decoder, long capacity, 4 rows
    "1b_long": Workload("1b_long", n_layers=16, d_model=2048, n_heads=32, n_kv_heads=8,
                        head_dim=64, ffn_hidden=8192, vocab=32000, wdtype="bf16", kvdtype="bf16",
                        cap=32768, rows=4, rope_theta=5e5, positions=(100, 8000, 20000, 32767)),
}
# configuration 1 with non-trivial norm gains (pins the gain multiply)
WORKLOADS["tiny_gain"] = WORKLOADS["tiny"].replace(name="tiny_gain", gain_sigma=0.1)


# stream ids: (kind << 40) | (layer << 16) | (row << 4) | sub
_K_WEIGHT, _K_TOKEN, _K_KV, _K_PAGE, _K_POS = 1, 2, 3, 4, 5
LAYER_ROLES = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")
GLOBAL_ROLES = ("embed", "final_norm", "lm_head")


def STREAM(kind: int, layer: int = 0, row: int = 0, sub: int = 0) -> int:
    return (kind << 40) | ((layer & 0xFFFFFF) << 16) | ((row & 0xFFF) << 4) | (sub & 0xF)


@dataclass
class ModelWeights:
    """Host copies of every weight, in nn.Linear layout [out, in] (C order)."""
    wl: Workload
    embed: np.ndarray
    final_norm: np.ndarray
    lm_head: np.ndarray
    layers: List[dict] = field(default_factory=list)


def _weight_shape(wl: Workload, role: str):
    d, F = wl.d_model, wl.ffn_hidden
    return {
        "attn_norm": (d,), "ffn_norm": (d,), "final_norm": (d,),
        "wq": (wl.q_dim, d), "wk": (wl.kv_dim, d), "wv": (wl.kv_dim, d),
        "wo": (d, wl.q_dim), "wg": (F, d), "wu": (F, d), "wd": (d, F),
        "embed": (wl.vocab, d), "lm_head": (wl.vocab, d),
    }[role]


def _draw(wl: Workload, role: str, layer: int):
    shape = _weight_shape(wl, role)
    if role.endswith("norm"):
        sub = {"attn_norm": 1, "ffn_norm": 6, "final_norm": 14}[role]
        if wl.gain_sigma == 0.0:
            one = np.float32(1.0)
            if wl.wdtype == "bf16":
                return np.full(shape, 0x3F80, dtype=np.uint16)
            return np.full(shape, one, dtype=np.float32)
        return normal(wl.seed, STREAM(_K_WEIGHT, layer, 0, sub), shape, sigma=wl.gain_sigma,
                      mean=1.0, dtype=wl.wdtype)
    sub = {"wq": 2, "wk": 3, "wv": 4, "wo": 5, "wg": 7, "wu": 8, "wd": 9,
           "embed": 12, "lm_head": 13}[role]
    return normal(wl.seed, STREAM(_K_WEIGHT, layer, 0, sub), shape, sigma=0.02, dtype=wl.wdtype)


def make_weights(wl: Workload) -> ModelWeights:
    mw = ModelWeights(wl=wl, embed=_draw(wl, "embed", 0xFFFF),
                      final_norm=_draw(wl, "final_norm", 0xFFFF),
                      lm_head=_draw(wl, "lm_head", 0xFFFF))
    for l in range(wl.n_layers):
        mw.layers.append({r: _draw(wl, r, l) for r in LAYER_ROLES})
    return mw


def prompt_tokens(wl: Workload, row: int = 0, n: Optional[int] = None) -> np.ndarray:
    n = wl.prompt_len if n is None else n
    return ints(wl.seed, STREAM(_K_TOKEN, 0, row), 0, wl.vocab, n)


def kv_prefill(wl: Workload, layer: int, which: int, row: int, npos: int,
               start: int = 0) -> np.ndarray:
    """N(0,1) K (which=0) or V (which=1) for logical positions [start, start+npos):
    array [npos, n_kv_heads, head_dim] in the KV dtype."""
    per = wl.kv_dim
    return normal(wl.seed, STREAM(_K_KV, layer, row, which), (npos, wl.n_kv_heads, wl.head_dim),
                  sigma=1.0, dtype=wl.kvdtype, offset=start * per)


def slot_map(wl: Workload) -> np.ndarray:
    """Page table [rows, cap/page_size]: a seeded permutation of the pool."""
    ppr = wl.cap // wl.page_size
    perm = permutation(wl.seed, STREAM(_K_PAGE), wl.num_pages)
    return perm[: wl.rows * ppr].reshape(wl.rows, ppr).copy()


def row_positions(wl: Workload) -> np.ndarray:
    """One decode position per row: the fixed list, else uniform in [0, cap)."""
    if wl.positions and len(wl.positions) == wl.rows:
        return np.asarray(wl.positions, dtype=np.int32)
    return ints(wl.seed, STREAM(_K_POS), 0, wl.cap, wl.rows)
