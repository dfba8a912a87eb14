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


# ---- shared GPU cases (called by the parity tests of each step strategy) ----

def run_sequence(wl, n_prompt, n_decode, mw=None, check_kv=True, **kw):
    """Prompt stepped token by token, then greedy decode fed with the oracle's pick."""
    from gen.device import read_kv
    dec, mw = make_decoder(wl, mw, **kw)
    orc = oracle.Oracle(mw, cap=wl.cap)
    toks = list(gen.prompt_tokens(wl, n=n_prompt))
    strict = 0
    pos = 0
    for i in range(n_prompt + n_decode):
        t = toks[i]
        res = dec.step([t], [pos])
        ref = orc.step(0, t, pos)
        assert_close(res.logits[0], ref, wl, f"{wl.name} step {i} pos {pos}")
        assert res.nonfinite[0] == 0
        assert int(res.ids[0]) == int(np.argmax(res.logits[0]))   # device argmax = argmax of its logits
        strict += assert_greedy(res.ids[0], ref, f"{wl.name} step {i}")
        if i + 1 >= n_prompt:
            toks.append(oracle.argmax(ref))
        pos += 1
    if check_kv:
        n = pos
        for l in range(wl.n_layers):
            for which, store in ((0, orc.K[0][l]), (1, orc.V[0][l])):
                got = kv_as_float(read_kv(dec.kv(l, which), 0, n))
                assert_close_state(got, kv_as_float(store[:n]), wl, f"{wl.name} KV layer {l} which {which}")
    st = dec.stats()
    dec.close()
    return strict, st


def prefill_both(dec, orc, wl, row, npos, slot_map=None):
    from gen.device import place_kv
    for l in range(wl.n_layers):
        for which in (0, 1):
            blk = gen.kv_prefill(wl, l, which, row, npos)
            place_kv(dec.kv(l, which), blk, row, 0, slot_map, wl.page_size)
            store = orc.K[0][l] if which == 0 else orc.V[0][l]
            store[:npos] = blk


def prefilled_positions_case(wl, **kw):
    """One step at each of wl.positions over KV pre-filled N(0,1) below pos: logits,
    greedy id and the K write at pos against the oracle, the prefill untouched."""
    dec, mw = make_decoder(wl, **kw)
    orc = oracle.Oracle(mw, cap=wl.cap)
    tok = int(gen.prompt_tokens(wl, n=1)[0])
    for pos in wl.positions:
        dec.reset_state()
        for l in range(wl.n_layers):
            orc.K[0][l][:] = 0
            orc.V[0][l][:] = 0
        prefill_both(dec, orc, wl, 0, pos)
        res = dec.step([tok], [pos])
        ref = orc.step(0, tok, pos)
        assert_close(res.logits[0], ref, wl, f"{wl.name} pos {pos}")
        assert_greedy(res.ids[0], ref, f"{wl.name} pos {pos}")
        from gen.device import read_kv
        for l in (0, wl.n_layers // 2, wl.n_layers - 1):
            got = kv_as_float(read_kv(dec.kv(l, 0), 0, pos + 1))
            assert_close_state(got[pos], kv_as_float(orc.K[0][l][pos]), wl, f"{wl.name} K write layer {l}")
            assert np.array_equal(got[:pos], kv_as_float(orc.K[0][l][:pos]))   # prefill untouched
    dec.close()


def paged_case(base: str, rows: int, n_steps: int, n_layers=None, **kw):
    """Paged KV through a seeded random page table, rows at independent positions,
    compared with the oracle row by row; the KV write lands only at WriteMap."""
    import torch
    wl = gen.WORKLOADS[base]
    shape = dict(name=f"{base}_paged{rows}", rows=rows, layout="paged", page_size=16,
                 num_pages=rows * wl.cap // 16 + 7)
    if n_layers:
        shape["n_layers"] = n_layers
    wl = wl.replace(**shape)
    dec, mw = make_decoder(wl, **kw)
    sm = gen.permutation(wl.seed, 99, wl.num_pages)[: rows * (wl.cap // 16)].reshape(rows, wl.cap // 16)
    dec.set_slot_map(sm)
    orcs = [oracle.Oracle(mw, cap=wl.cap) for _ in range(rows)]
    start = [int(x) for x in gen.ints(wl.seed, 98, 0, wl.cap - n_steps, rows)]
    toks = [gen.prompt_tokens(wl, row=r, n=n_steps) for r in range(rows)]
    for i in range(n_steps):
        pos = [start[r] + i for r in range(rows)]
        before = [dec.kv(l, 0).clone() for l in range(wl.n_layers)]
        res = dec.step([toks[r][i] for r in range(rows)], pos)
        wmap = [int(sm[r][p // 16]) * 16 + p % 16 for r, p in enumerate(pos)]
        for l in range(wl.n_layers):
            diff = (dec.kv(l, 0) != before[l]).any(dim=3).any(dim=1)   # [pages, page]
            got = sorted((int(a) * 16 + int(b)) for a, b in torch.nonzero(diff).tolist())
            assert got == sorted(wmap), (l, got, wmap)
        for r in range(rows):
            # the oracle sees only positions the step wrote: zeros before start (same as the GPU pool)
            ref = orcs[r].step(0, int(toks[r][i]), pos[r])
            assert_close(res.logits[r], ref, wl, f"{wl.name} row {r} step {i}")
            assert_greedy(res.ids[r], ref)
    dec.close()
