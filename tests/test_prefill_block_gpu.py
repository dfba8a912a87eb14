"""Block prefill of one sequence (dec_prefill_block): the prompt's projections
on the tensor cores in blocks of 128 tokens, causal attention over the block,
every layer's K/V written into the sequence's store ("Models, Registry and the
Driver", section "The Model": a step shape is rows x new tokens; positions are
absolute, so a prefill is a step continuing from a position).

Pinned against the oracle's direct full causal pass (logits after the last
token, greedy pick, and the carried K/V of every layer and position) under the
parity tolerances of "Execution", section "Verification"."""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle
from graph_replay_gb300 import _binding as B
from tests._harness import assert_close, assert_close_state, assert_greedy, kv_as_float, make_decoder

pytestmark = pytest.mark.gpu


def _kv_rows(dec, wl, n, row=0, pages=None):
    """K and V of positions [0, n) of one sequence, per layer (storage bits)."""
    from gen.device import read_kv
    sm = None if pages is None else np.asarray(pages).reshape(1, -1)
    return [[read_kv(dec.kv(l, w), 0 if sm is not None else row, n, sm, wl.page_size) for w in (0, 1)]
            for l in range(wl.n_layers)]


def _check(dec, wl, mw, toks, logits, pick, row=0, pages=None, what="prefill"):
    orc = oracle.Oracle(mw, cap=wl.cap, alloc_kv=False)
    ref_logits, K, V = orc.full_causal(toks)
    assert_close(logits, ref_logits[-1], wl, f"{what}: logits after the last token")
    assert_greedy(pick, ref_logits[-1], f"{what}: greedy pick")
    got = _kv_rows(dec, wl, len(toks), row, pages)
    for l in range(wl.n_layers):
        assert_close_state(kv_as_float(got[l][0]), kv_as_float(K[l]), wl, f"{what}: K layer {l}")
        assert_close_state(kv_as_float(got[l][1]), kv_as_float(V[l]), wl, f"{what}: V layer {l}")


def test_prefill_block_1b_prompt_contiguous():
    # the 1B-class configuration's prompt length (128 tokens), one block
    wl = gen.WORKLOADS["1b"].replace(name="1b_pfb", n_layers=4, cap=512)
    dec, mw = make_decoder(wl)
    toks = gen.prompt_tokens(wl, n=wl.prompt_len)
    logits, pick = dec.prefill_block(toks, 0)
    _check(dec, wl, mw, toks, logits, pick)
    dec.close()


def test_prefill_block_paged_two_blocks_and_a_row():
    # 200 tokens: a full block and a short one, into a random page table; the
    # contiguous capture of the same model fills row 1 of two rows
    wl = gen.WORKLOADS["1b"].replace(name="1b_pfbp", n_layers=3, cap=256, rows=2, layout="paged", page_size=16,
                                     num_pages=40)
    dec, mw = make_decoder(wl)
    perm = gen.permutation(wl.seed, 33, wl.num_pages)
    pages = perm[: wl.cap // wl.page_size].copy()
    toks = gen.prompt_tokens(wl, n=200)
    logits, pick = dec.prefill_block(toks, 0, pages=pages)
    _check(dec, wl, mw, toks, logits, pick, pages=pages, what="paged prefill")
    dec.close()
    wc = wl.replace(name="1b_pfbc", layout="contiguous", num_pages=0)
    dec, _ = make_decoder(wc, mw)
    logits, pick = dec.prefill_block(toks, 0, row=1)
    _check(dec, wc, mw, toks, logits, pick, row=1, what="contiguous row 1")
    dec.close()


def test_prefill_block_8b_shape_paged():
    # head_dim 128 over a random page table: the attention's per-page TMA boxes
    wl = gen.WORKLOADS["8b"].replace(name="8b_pfbp", n_layers=1, cap=512, vocab=2048, positions=(), layout="paged",
                                     page_size=16, num_pages=48)
    dec, mw = make_decoder(wl)
    perm = gen.permutation(wl.seed, 35, wl.num_pages)
    pages = perm[: wl.cap // wl.page_size].copy()
    toks = gen.prompt_tokens(wl, n=300)
    logits, pick = dec.prefill_block(toks, 0, pages=pages)
    _check(dec, wl, mw, toks, logits, pick, pages=pages, what="8B-shape paged prefill")
    dec.close()


def test_prefill_block_1024_tokens():
    wl = gen.WORKLOADS["1b"].replace(name="1b_pfb1k", n_layers=2, cap=1024, vocab=2048)
    dec, mw = make_decoder(wl)
    toks = gen.prompt_tokens(wl, n=1024)
    logits, pick = dec.prefill_block(toks, 0)
    _check(dec, wl, mw, toks, logits, pick, what="1024-token prefill")
    dec.close()


def test_prefill_block_continues_from_a_position_then_decodes():
    wl = gen.WORKLOADS["1b"].replace(name="1b_pfbc2", n_layers=3, cap=512)
    dec, mw = make_decoder(wl)
    toks = gen.prompt_tokens(wl, n=160)
    dec.prefill_block(toks[:100], 0)
    logits, pick = dec.prefill_block(toks[100:], 100)
    _check(dec, wl, mw, toks, logits, pick, what="prefill continued at 100")
    # the decode graph reads what the prefill wrote
    orc = oracle.Oracle(mw, cap=wl.cap)
    for p, t in enumerate(toks):
        ref = orc.step(0, int(t), p)
    cur, pos = oracle.argmax(ref), len(toks)
    for i in range(5):
        res = dec.step([cur], [pos])
        ref = orc.step(0, cur, pos)
        assert_close(res.logits[0], ref, wl, f"decode after the block prefill, step {i}")
        cur, pos = oracle.argmax(ref), pos + 1
    dec.close()


def test_prefill_block_8b_shape():
    # head_dim 128 and the 8B-shape projections, one layer
    wl = gen.WORKLOADS["8b"].replace(name="8b_pfb", n_layers=1, cap=256, vocab=4096, positions=())
    dec, mw = make_decoder(wl)
    toks = gen.prompt_tokens(wl, n=150)
    logits, pick = dec.prefill_block(toks, 0)
    _check(dec, wl, mw, toks, logits, pick, what="8B-shape prefill")
    dec.close()


def test_prefill_block_8b_shape_1024_tokens():
    # a full pass of 8 token blocks at the 8B shape: the O and down projections
    # run unsplit and add into the residual rows in their own epilogue
    wl = gen.WORKLOADS["8b"].replace(name="8b_pfb1k", n_layers=1, cap=1024, vocab=4096, positions=())
    dec, mw = make_decoder(wl)
    toks = gen.prompt_tokens(wl, n=1024)
    logits, pick = dec.prefill_block(toks, 0)
    _check(dec, wl, mw, toks, logits, pick, what="8B-shape 1024-token prefill")
    dec.close()


def test_prefill_block_two_passes():
    # 1300 tokens: a pass of 1024 and one of 276 that attends to the first pass's K/V
    wl = gen.WORKLOADS["1b"].replace(name="1b_pfb2p", n_layers=2, cap=1536, vocab=2048)
    dec, mw = make_decoder(wl)
    toks = gen.prompt_tokens(wl, n=1300)
    logits, pick = dec.prefill_block(toks, 0)
    _check(dec, wl, mw, toks, logits, pick, what="two-pass prefill")
    dec.close()


@pytest.mark.parametrize("base, n_layers, n", [("1b", 2, 200), ("8b", 1, 150)])
def test_prefill_block_gqa_group_of_two(base, n_layers, n):
    # two query heads per kv head: the attention kernel's 32-token query blocks
    wl = gen.WORKLOADS[base].replace(name=f"{base}_pfbg2", n_kv_heads=gen.WORKLOADS[base].n_heads // 2,
                                     n_layers=n_layers, cap=512, vocab=2048, positions=())
    dec, mw = make_decoder(wl)
    toks = gen.prompt_tokens(wl, n=n)
    logits, pick = dec.prefill_block(toks, 0)
    _check(dec, wl, mw, toks, logits, pick, what=f"{base} group-2 prefill")
    dec.close()


def test_prefill_block_refusals():
    wl = gen.WORKLOADS["1b"].replace(name="1b_pfbr", n_layers=1, cap=256)
    dec, _ = make_decoder(wl)
    for args, code in (((np.ones(10, np.int32), 250), B.DEC_E_RANGE), ((np.array([wl.vocab], np.int32), 0), B.DEC_E_RANGE)):
        with pytest.raises(B.DecError) as e:
            dec.prefill_block(*args)
        assert e.value.status == code
    with pytest.raises(B.DecError) as e:
        dec.prefill_block([1, 2], 0, row=1)
    assert e.value.status == B.DEC_E_RANGE
    assert dec.stats()["state"] == 0
    dec.close()
    dec, _ = make_decoder(gen.WORKLOADS["tiny"])
    with pytest.raises(B.DecError) as e:
        dec.prefill_block([1, 2], 0)
    assert e.value.status == B.DEC_E_UNSUPPORTED
    dec.close()
