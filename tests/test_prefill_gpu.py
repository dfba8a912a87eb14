"""Multi-token prefill of one sequence (dec_prefill) through the paged step:
rows of a chunk are consecutive positions of the sequence and share its pages
("Models, Registry and the Driver", section "The Model": a step shape is rows x
new tokens; positions are absolute, so a prefill continues from a position).

Pinned against the oracle's direct full causal pass, and bit-exact against the
same tokens stepped one at a time (per token the arithmetic is that of a
decode step), whatever the chunking.
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle
from graph_replay_gb300 import _binding as B
from tests._harness import assert_close, assert_close_state, assert_greedy, kv_as_float, make_decoder

pytestmark = pytest.mark.gpu

ROWS = 8
CAP = 256
PAGE = 16


def _wl(n_layers=3):
    ppr = CAP // PAGE
    return gen.WORKLOADS["1b"].replace(name="1b_pf", n_layers=n_layers, cap=CAP, rows=ROWS, layout="paged",
                                       page_size=PAGE, num_pages=ROWS * ppr + 9)


def _tables(wl):
    ppr = CAP // PAGE
    perm = gen.permutation(wl.seed, 31, wl.num_pages)
    return perm[: ROWS * ppr].reshape(ROWS, ppr).copy()


def _seq_kv(dec, wl, pages, n):
    """K and V of positions [0, n) of the sequence on `pages`, per layer (storage bits)."""
    from gen.device import read_kv
    sm = pages.reshape(1, -1)
    return [[read_kv(dec.kv(l, w), 0, n, sm, PAGE) for w in (0, 1)] for l in range(wl.n_layers)]


def test_prefill_matches_full_causal_oracle():
    wl = _wl()
    dec, mw = make_decoder(wl)
    tables = _tables(wl)
    dec.set_slot_map(tables)
    toks = gen.prompt_tokens(wl, n=37)
    logits, pick = dec.prefill(tables[2], toks, 0)
    orc = oracle.Oracle(mw, cap=CAP, alloc_kv=False)
    ref_logits, K, V = orc.full_causal(toks)
    assert_close(logits, ref_logits[-1], wl, "prefill logits after the last token")
    assert_greedy(pick, ref_logits[-1], "prefill greedy pick")
    got = _seq_kv(dec, wl, tables[2], len(toks))
    for l in range(wl.n_layers):
        assert_close_state(kv_as_float(got[l][0]), kv_as_float(K[l]), wl, f"prefill K layer {l}")
        assert_close_state(kv_as_float(got[l][1]), kv_as_float(V[l]), wl, f"prefill V layer {l}")
    dec.close()


def test_prefill_chunking_and_decode_are_bit_identical():
    import torch
    wl = _wl(n_layers=2)
    dec, _ = make_decoder(wl)
    tables = _tables(wl)
    dec.set_slot_map(tables)
    toks = gen.prompt_tokens(wl, n=37)
    seq = 5

    def pool():
        return [dec.kv(l, w).clone() for l in range(wl.n_layers) for w in (0, 1)]

    la, ia = dec.prefill(tables[seq], toks, 0)                   # 5 chunks, the last one short
    kv_a = _seq_kv(dec, wl, tables[seq], len(toks))
    pool_a = pool()
    dec.reset_state()
    dec.prefill(tables[seq], toks[:20], 0)
    lb, ib = dec.prefill(tables[seq], toks[20:], 20)            # continues from a position
    kv_b = _seq_kv(dec, wl, tables[seq], len(toks))
    assert np.array_equal(la, lb) and ia == ib
    for x, y in zip(kv_a, kv_b):
        assert np.array_equal(x[0], y[0]) and np.array_equal(x[1], y[1])
    # the same tokens one decode step at a time on row `seq` (its own page table row)
    dec.reset_state()
    for p, t in enumerate(toks):
        tk = [0] * ROWS
        ps = [0] * ROWS
        tk[seq], ps[seq] = int(t), p
        res = dec.step(tk, ps)
    kv_c = _seq_kv(dec, wl, tables[seq], len(toks))
    assert np.array_equal(res.logits[seq], la) and int(res.ids[seq]) == ia
    for x, y in zip(kv_a, kv_c):
        assert np.array_equal(x[0], y[0]) and np.array_equal(x[1], y[1])
    # the prefill touched only the sequence's slots of positions [0, 37)
    dec.reset_state()
    before = pool()
    dec.prefill(tables[seq], toks, 0)
    after = pool()
    want = sorted(int(tables[seq][p // PAGE]) * PAGE + p % PAGE for p in range(len(toks)))
    for b_, a_ in zip(before, after):
        diff = (a_ != b_).any(dim=3).any(dim=1)   # [pages, page]
        got = sorted(int(pg) * PAGE + int(o) for pg, o in torch.nonzero(diff).tolist())
        assert set(got) <= set(want)
    assert any(not torch.equal(x, y) for x, y in zip(before, after))
    assert all(torch.equal(x, y) for x, y in zip(pool_a, after))   # same bytes as the first prefill
    dec.close()


def test_prefill_then_decode_matches_oracle():
    wl = _wl()
    dec, mw = make_decoder(wl)
    tables = _tables(wl)
    dec.set_slot_map(tables)
    toks = gen.prompt_tokens(wl, n=21)
    _, pick = dec.prefill(tables[0], toks, 0)
    orc = oracle.Oracle(mw, cap=CAP)
    for p, t in enumerate(toks):
        ref = orc.step(0, int(t), p)
    cur, pos = oracle.argmax(ref), len(toks)
    for i in range(6):
        tk = [0] * ROWS
        ps = [0] * ROWS
        tk[0], ps[0] = cur, pos
        res = dec.step(tk, ps)
        ref = orc.step(0, cur, pos)
        assert_close(res.logits[0], ref, wl, f"decode after prefill, step {i}")
        cur, pos = oracle.argmax(ref), pos + 1
    dec.close()


def test_prefill_refusals():
    wl = _wl(n_layers=1)
    dec, _ = make_decoder(wl)
    tables = _tables(wl)
    dec.set_slot_map(tables)
    with pytest.raises(B.DecError) as e:
        dec.prefill(tables[0], [1] * 10, CAP - 5)
    assert e.value.status == B.DEC_E_RANGE
    bad = tables[0].copy()
    bad[3] = wl.num_pages
    with pytest.raises(B.DecError) as e:
        dec.prefill(bad, [1, 2, 3], 0)
    assert e.value.status == B.DEC_E_RANGE
    dec.close()
    wc = gen.WORKLOADS["1b"].replace(name="1b_pfc", n_layers=1, cap=CAP, rows=2)
    dec, _ = make_decoder(wc)
    with pytest.raises(B.DecError) as e:
        dec.prefill(np.zeros(CAP // PAGE, np.int32), [1, 2], 0)
    assert e.value.status == B.DEC_E_UNSUPPORTED
    dec.close()
