"""Shared helpers of the GPU parity tests: build a decoder for a workload,
compare its outputs with the oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np

import gen
import oracle

# tolerances: bf16 weights with fp32 accumulation, and the fp32 tiny model
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
F32_REL = 1e-4
GREEDY_MARGIN = 0.05


def make_decoder(wl, mw=None, device="cuda:0", **kw):
    import torch  # noqa: F401
    from gen.device import upload_weights
    from graph_replay_gb300 import Decoder, make_config

    if mw is None:
        mw = gen.make_weights(wl)
    cfg = make_config(wl.n_layers, wl.d_model, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.ffn_hidden, wl.vocab,
                      wl.wdtype, wl.kvdtype, wl.rms_eps, wl.rope_theta, device=int(str(device).split(":")[-1]),
                      wait_timeout_ms=kw.pop("wait_timeout_ms", 0))
    w = upload_weights(mw, device)
    dec = Decoder(cfg, w, cap=wl.cap, rows=wl.rows, kv_layout=wl.layout, page_size=wl.page_size,
                  num_pages=wl.num_pages, **kw)
    return dec, mw


def errors(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = gpu - ref
    max_abs = float(np.abs(d).max())
    rel_l2 = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300))
    rel_max = float(max_abs / max(np.abs(ref).max(), 1e-300))
    return max_abs, rel_l2, rel_max


def assert_close(gpu, ref, wl, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    # NaN or Inf where the oracle is finite fails at any tolerance
    bad = np.isfinite(ref) & ~np.isfinite(gpu)
    assert not bad.any(), f"{what}: non-finite GPU values where the oracle is finite"
    max_abs, rel_l2, rel_max = errors(gpu, ref)
    if wl.wdtype == "f32":
        assert rel_max <= F32_REL and rel_l2 <= F32_REL, f"{what}: rel max {rel_max:.3e}, rel L2 {rel_l2:.3e}"
    else:
        assert max_abs <= BF16_MAX_ABS and rel_l2 <= BF16_REL_L2, \
            f"{what}: max abs {max_abs:.3e}, rel L2 {rel_l2:.3e}"
    return max_abs, rel_l2


def assert_close_state(gpu, ref, wl, what=""):
    """Carried K/V state.  Stored values are rounded to the KV dtype, and the GPU
    rounds an fp32 value where the oracle rounds the exact one, so a value near a
    rounding midpoint may land one storage ulp away: each element may differ by
    max(logit max-abs bound, one bf16 ulp = 2^-7 |ref| at most); relative L2 as
    for logits.  fp32 stores keep the fp32 bound."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bad = np.isfinite(ref) & ~np.isfinite(gpu)
    assert not bad.any(), f"{what}: non-finite GPU values where the oracle is finite"
    if wl.kvdtype == "f32" and wl.wdtype == "f32":
        return assert_close(gpu, ref, wl, what)
    d = np.abs(gpu - ref)
    bound = np.maximum(BF16_MAX_ABS, np.abs(ref) * 2.0 ** -7)
    worst = float((d / bound).max())
    _, rel_l2, _ = errors(gpu, ref)
    assert worst <= 1.0 and rel_l2 <= BF16_REL_L2, f"{what}: worst |d|/bound {worst:.3f}, rel L2 {rel_l2:.3e}"
    return worst, rel_l2


def assert_greedy(gpu_id, ref_logits, what=""):
    """Bit-exact id wherever the oracle's top-2 margin exceeds 0.05; otherwise the
    GPU id must be one of the oracle's near-top candidates."""
    ref_id = oracle.argmax(ref_logits)
    margin = oracle.top2_margin(ref_logits)
    if margin > GREEDY_MARGIN:
        assert int(gpu_id) == ref_id, f"{what}: id {gpu_id} != oracle {ref_id} (margin {margin:.3f})"
        return True
    top = float(np.max(ref_logits))
    assert ref_logits[int(gpu_id)] >= top - GREEDY_MARGIN, f"{what}: id {gpu_id} is not a near-top candidate"
    return False


def kv_as_float(a: np.ndarray) -> np.ndarray:
    return gen.bf16_bits_to_f32(a) if a.dtype == np.uint16 else a
