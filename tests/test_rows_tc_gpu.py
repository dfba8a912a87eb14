"""Multi-row decode (2..8 rows, bf16 weights): the projections run on the
tensor-core GEMV.  Parity against the oracle row by row, capture versus eager
bit-exact, and the paged 8-row 8B-shape configuration at full size.

"Execution", sections "A constant-shape decode graph" (rows at independent
positions in one graph), "Slot buffers" (SlotMap / WriteMap) and
"Verification" (tier 1 bit-exact, tier 2 tolerance); "Models, Registry and the
Driver", section "The Model" (StepShape: rows x one new token).
"""
from __future__ import annotations

import os

import numpy as np
import pytest

import gen
import oracle
from tests._harness import (assert_close, assert_greedy, kv_as_float, make_decoder, paged_case,
                            assert_close_state)

pytestmark = pytest.mark.gpu


def test_paged_1b_rows8():
    # 8 rows at independent positions through a random page table (the paged configuration's
    # row count on the 1B shape, 4 layers)
    paged_case("1b", 8, 4, n_layers=4)


def test_rows3_prompt_matches_oracle():
    # an odd row count: the activation rows past R are zero inside the tensor-core tiles
    wl = gen.WORKLOADS["1b"].replace(name="1b_r3", n_layers=3, cap=512, rows=3)
    dec, mw = make_decoder(wl)
    orcs = [oracle.Oracle(mw, cap=wl.cap) for _ in range(3)]
    toks = [gen.prompt_tokens(wl, row=r, n=12) for r in range(3)]
    start = [0, 5, 200]
    for i in range(12):
        pos = [start[r] + i for r in range(3)]
        res = dec.step([int(toks[r][i]) for r in range(3)], pos)
        for r in range(3):
            ref = orcs[r].step(0, int(toks[r][i]), pos[r])
            assert_close(res.logits[r], ref, wl, f"row {r} step {i}")
            assert_greedy(res.ids[r], ref, f"row {r} step {i}")
            assert int(res.ids[r]) == int(np.argmax(res.logits[r]))
    from gen.device import read_kv
    for r in range(3):
        for l in range(wl.n_layers):
            got = kv_as_float(read_kv(dec.kv(l, 0), r, start[r] + 12))[start[r]:]
            assert_close_state(got, kv_as_float(orcs[r].K[0][l][start[r]:start[r] + 12]), wl, f"K row {r} layer {l}")
    dec.close()


def test_rows_capture_equals_eager_bit_exact():
    # tier 1: the recorded graph and eager launches of the same kernels agree bit for bit
    import torch
    wl = gen.WORKLOADS["1b"].replace(name="1b_r4", n_layers=2, cap=256, rows=4)
    dec, mw = make_decoder(wl)
    toks = [gen.prompt_tokens(wl, row=r, n=20) for r in range(4)]

    def run():
        out = []
        for i in range(20):
            out.append(dec.step([int(toks[r][i]) for r in range(4)], [i, i + 3, i + 50, 2 * i]).logits.copy())
        kv = [dec.kv(l, w).clone() for l in range(wl.n_layers) for w in (0, 1)]
        return out, kv

    g_logits, g_kv = run()
    dec.reset_state()
    dec.set_eager(True)
    e_logits, e_kv = run()
    dec.reset_state()
    dec.set_eager(False)
    a_logits, _ = run()
    dec.close()
    for a, b, c in zip(g_logits, e_logits, a_logits):
        assert np.array_equal(a, b)
        assert np.array_equal(a, c)
    for a, b in zip(g_kv, e_kv):
        assert torch.equal(a, b)


def test_tensor_core_and_cuda_core_gemv_agree():
    # the same 4-row steps through the tensor-core GEMV and through the CUDA-core GEMV
    wl = gen.WORKLOADS["1b"].replace(name="1b_r4b", n_layers=2, cap=256, rows=4)
    mw = gen.make_weights(wl)
    toks = [gen.prompt_tokens(wl, row=r, n=6) for r in range(4)]

    def run():
        dec, _ = make_decoder(wl, mw)
        out = [dec.step([int(toks[r][i]) for r in range(4)], [i] * 4).logits.copy() for i in range(6)]
        dec.close()
        return out

    tc = run()
    old = os.environ.get("GRAPHDEC_GEMV")
    os.environ["GRAPHDEC_GEMV"] = "simd"
    try:
        simd = run()
    finally:
        if old is None:
            del os.environ["GRAPHDEC_GEMV"]
        else:
            os.environ["GRAPHDEC_GEMV"] = old
    for a, b in zip(tc, simd):
        assert not np.array_equal(a, b)   # two different kernels ran
        assert_close(a, b, wl, "tensor-core vs CUDA-core GEMV")


@pytest.mark.parametrize("mode", ["box", "rowcopy"])
def test_each_tensor_core_gemv_matches_the_oracle(mode):
    # every projection through one of the two tensor-core GEMVs (TMA boxes with
    # split K, or one bulk copy per weight row), 3 rows, against the oracle
    wl = gen.WORKLOADS["1b"].replace(name=f"1b_{mode}", n_layers=2, cap=256, rows=3)
    old = os.environ.get("GRAPHDEC_GEMV")
    os.environ["GRAPHDEC_GEMV"] = mode
    try:
        dec, mw = make_decoder(wl)
    finally:
        if old is None:
            del os.environ["GRAPHDEC_GEMV"]
        else:
            os.environ["GRAPHDEC_GEMV"] = old
    orcs = [oracle.Oracle(mw, cap=wl.cap) for _ in range(3)]
    toks = [gen.prompt_tokens(wl, row=r, n=8) for r in range(3)]
    for i in range(8):
        pos = [i, i + 40, i + 100]
        res = dec.step([int(toks[r][i]) for r in range(3)], pos)
        for r in range(3):
            ref = orcs[r].step(0, int(toks[r][i]), pos[r])
            assert_close(res.logits[r], ref, wl, f"{mode} row {r} step {i}")
            assert_greedy(res.ids[r], ref, f"{mode} row {r} step {i}")
    dec.close()


@pytest.mark.slow
def test_8b_paged_rows8_prefilled():
    # the paged configuration at full size: 8 rows, 16-token pages in a pool of 4096, SlotMap a
    # seeded permutation, each row at its own position with K/V pre-filled N(0,1) below it
    wl = gen.WORKLOADS["8b_paged"]
    dec, mw = make_decoder(wl)
    sm = gen.slot_map(wl)
    dec.set_slot_map(sm)
    positions = [int(p) for p in gen.row_positions(wl)]
    toks = [int(t) for t in gen.prompt_tokens(wl, n=wl.rows)]
    from gen.device import place_kv, read_kv
    for r in range(wl.rows):
        for l in range(wl.n_layers):
            for which in (0, 1):
                place_kv(dec.kv(l, which), gen.kv_prefill(wl, l, which, r, positions[r]), r, 0, sm, wl.page_size)
    res = dec.step(toks, positions)
    orc = oracle.Oracle(mw, cap=wl.cap)
    for r in range(wl.rows):
        p = positions[r]
        for l in range(wl.n_layers):
            orc.K[0][l][:] = 0
            orc.V[0][l][:] = 0
            orc.K[0][l][:p] = gen.kv_prefill(wl, l, 0, r, p)
            orc.V[0][l][:p] = gen.kv_prefill(wl, l, 1, r, p)
        ref = orc.step(0, toks[r], p)
        assert_close(res.logits[r], ref, wl, f"8b_paged row {r} pos {p}")
        assert_greedy(res.ids[r], ref, f"8b_paged row {r}")
        for l in (0, wl.n_layers - 1):
            got = kv_as_float(read_kv(dec.kv(l, 1), r, p + 1, sm, wl.page_size))
            assert_close_state(got[p], kv_as_float(orc.V[0][l][p]), wl, f"V write row {r} layer {l}")
    dec.close()
