"""Chained greedy steps (dec_chain): the device feeds each step's pick to the
next step's Token slot and the host waits once ("Models, Registry and the
Driver", section "The Driver": RowWork::Chain).

Pinned two ways: bit-identical to the same steps fed back by the host through
dec_step (same kernels, same inputs: ids and the whole K/V state), and against
the oracle's own greedy feed-back wherever its top-2 margin decides the pick.
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle
from graph_replay_gb300 import _binding as B
from tests._harness import GREEDY_MARGIN, make_decoder

pytestmark = pytest.mark.gpu


def _prompt(dec, wl, toks, start):
    n = toks.shape[1]
    for i in range(n):
        res = dec.step(toks[:, i], [start[r] + i for r in range(wl.rows)])
    return res.ids.copy(), [start[r] + n for r in range(wl.rows)]


def _chain_vs_host(wl, n_prompt, n_chain, start, slot_map=None, **kw):
    import torch
    dec, _ = make_decoder(wl, **kw)
    if slot_map is not None:
        dec.set_slot_map(slot_map)
    toks = np.stack([gen.prompt_tokens(wl, row=r, n=n_prompt) for r in range(wl.rows)])

    def kv():
        return [dec.kv(l, w).clone() for l in range(wl.n_layers) for w in (0, 1)]

    first, pos = _prompt(dec, wl, toks, start)
    ids_c, nf_c = dec.chain(first, pos, n_chain)
    kv_c = kv()
    dec.reset_state()
    first_h, pos_h = _prompt(dec, wl, toks, start)
    assert np.array_equal(first, first_h)
    ids_h = []
    cur = first_h
    for i in range(n_chain):
        res = dec.step(cur, [pos_h[r] + i for r in range(wl.rows)], logits=False)
        ids_h.append(res.ids.copy())
        cur = res.ids
    kv_h = kv()
    st = dec.stats()
    dec.close()
    assert np.array_equal(ids_c, np.stack(ids_h))
    assert not nf_c.any()
    for a, b in zip(kv_c, kv_h):
        assert torch.equal(a, b)
    return ids_c, st


def test_chain_equals_host_fed_steps_rows1():
    wl = gen.WORKLOADS["1b"].replace(name="1b_c1", n_layers=2, cap=256)
    _chain_vs_host(wl, 8, 40, [0])


def test_chain_equals_host_fed_steps_persistent():
    wl = gen.WORKLOADS["1b"].replace(name="1b_c1p", n_layers=2, cap=256)
    _chain_vs_host(wl, 8, 40, [0], strategy="persistent")


def test_chain_equals_host_fed_steps_rows4():
    wl = gen.WORKLOADS["1b"].replace(name="1b_c4", n_layers=2, cap=256, rows=4)
    _chain_vs_host(wl, 5, 24, [0, 17, 100, 3])


def test_chain_equals_host_fed_steps_persistent_rows4():
    wl = gen.WORKLOADS["1b"].replace(name="1b_c4p", n_layers=2, cap=256, rows=4)
    _, st = _chain_vs_host(wl, 5, 24, [0, 17, 100, 3], strategy="persistent")
    assert st["strategy"] == 1


def test_chain_equals_host_fed_steps_paged_rows3():
    wl = gen.WORKLOADS["1b"].replace(name="1b_cp3", n_layers=2, cap=256, rows=3, layout="paged",
                                     page_size=16, num_pages=3 * 16 + 5)
    sm = gen.permutation(wl.seed, 7, wl.num_pages)[: 3 * 16].reshape(3, 16)
    _chain_vs_host(wl, 4, 30, [0, 30, 200], slot_map=sm)


def test_chain_tiny_fp32_against_oracle_greedy():
    # the oracle feeds back its own argmax; the chain must pick the same ids
    # while every oracle margin exceeds the greedy tolerance
    wl = gen.WORKLOADS["tiny"]
    dec, mw = make_decoder(wl)
    orc = oracle.Oracle(mw, cap=wl.cap)
    toks = gen.prompt_tokens(wl, n=wl.prompt_len)
    for p, t in enumerate(toks):
        ref = orc.step(0, int(t), p)
        res = dec.step([int(t)], [p], logits=False)
    first = oracle.argmax(ref)
    assert int(res.ids[0]) == first
    n = wl.decode_steps
    ids, _ = dec.chain([first], [len(toks)], n)
    dec.close()
    cur = first
    for i in range(n):
        ref = orc.step(0, cur, len(toks) + i)
        if oracle.top2_margin(ref) <= GREEDY_MARGIN:
            break
        cur = oracle.argmax(ref)
        assert int(ids[i, 0]) == cur, f"chained step {i}"


def test_chain_refuses_out_of_range():
    wl = gen.WORKLOADS["1b"].replace(name="1b_cr", n_layers=1, cap=64)
    dec, _ = make_decoder(wl)
    with pytest.raises(B.DecError) as e:
        dec.chain([1], [60], 5)          # 60 + 5 > cap
    assert e.value.status == B.DEC_E_RANGE
    with pytest.raises(B.DecError) as e:
        dec.chain([1], [0], 0)
    assert e.value.status == B.DEC_E_RANGE
    ids, _ = dec.chain([1], [59], 5)     # ends exactly at cap - 1
    assert ids.shape == (5, 1)
    dec.close()
