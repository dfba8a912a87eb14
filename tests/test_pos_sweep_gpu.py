"""The pos-bounded K/V sweep (DEC_SWEEP_POS) against the constant-shape sweep.

The method's attention always sweeps [0, cap) and hides the positions after
pos with a mask ("Execution", "A constant-shape decode graph").  With
DEC_SWEEP_POS each split stops loading K/V after the tile that holds pos.  The
tiles it leaves out hold no visible key, and the kernel does no arithmetic on
a block without one, so logits, ids, flags and the carried K/V state must be
bit-identical to the full sweep.  Every position after pos holds NaN / Inf /
1e30 garbage here, so a stray read of a skipped tile would show."""
import numpy as np
import pytest

import gen
from _harness import make_decoder

pytestmark = pytest.mark.gpu


def _garbage_like(t):
    import torch
    g = torch.tensor([float("nan"), float("inf"), -float("inf"), 1e30], dtype=torch.bfloat16, device=t.device)
    return g.repeat(t.numel() // 4 + 1)[: t.numel()].view(t.shape)


def _same_state(a, b, wl):
    import torch
    for l in range(wl.n_layers):
        for w in (0, 1):
            assert torch.equal(a.kv(l, w).view(torch.int16), b.kv(l, w).view(torch.int16)), (l, w)


def _same_step(rc, rp, what):
    assert np.array_equal(rc.logits, rp.logits), what
    assert np.array_equal(rc.ids, rp.ids), what
    assert np.array_equal(rc.nonfinite, rp.nonfinite), what
    assert not rc.nonfinite.any(), f"{what}: garbage after pos reached the logits"


def _contiguous_pair(wl, positions):
    """Two decoders on one set of weights, K/V pre-filled up to each row's
    position and garbage after it."""
    from gen.device import place_kv
    dec_c, mw = make_decoder(wl)
    dec_p, _ = make_decoder(wl, mw=mw, kv_sweep="pos")
    for dec in (dec_c, dec_p):
        for l in range(wl.n_layers):
            for w in (0, 1):
                store = dec.kv(l, w)
                store.copy_(_garbage_like(store))
                for r, p in enumerate(positions):
                    place_kv(store, gen.kv_prefill(wl, l, w, r, p), r)
    return dec_c, dec_p


def test_pos_sweep_bit_identical_one_row():
    wl = gen.WORKLOADS["1b"].replace(name="1b_sweep_r1", n_layers=2, vocab=1024, cap=4096)
    P = 3000
    dec_c, dec_p = _contiguous_pair(wl, [P])
    toks = gen.prompt_tokens(wl, n=8)
    # first position, stage and split edges, the last pre-filled position
    for i, p in enumerate([0, 127, 128, 129, 1100, 2047, 2999, P]):
        _same_step(dec_c.step([toks[i]], [p]), dec_p.step([toks[i]], [p]), f"pos {p}")
    _same_state(dec_c, dec_p, wl)
    st_c, st_p = dec_c.stats(), dec_p.stats()
    assert st_c["kernels_per_step"] == st_p["kernels_per_step"]   # same graph, fewer bytes
    dec_c.close()
    dec_p.close()


def test_pos_sweep_bit_identical_four_rows():
    # several rows: every row's K/V is written before attention (the pre-written path)
    wl = gen.WORKLOADS["1b"].replace(name="1b_sweep_r4", n_layers=2, vocab=1024, cap=2048, rows=4)
    positions = [3, 700, 1500, 2046]
    dec_c, dec_p = _contiguous_pair(wl, positions)
    toks = [gen.prompt_tokens(wl, row=r, n=2) for r in range(4)]
    for i in range(2):
        pos = [p + i for p in positions]
        step = [int(toks[r][i]) for r in range(4)]
        _same_step(dec_c.step(step, pos), dec_p.step(step, pos), f"step {i}")
    _same_state(dec_c, dec_p, wl)
    dec_c.close()
    dec_p.close()


def test_pos_sweep_bit_identical_paged_rows2():
    import torch
    from gen.device import place_kv
    base = gen.WORKLOADS["1b"]
    wl = base.replace(name="1b_sweep_paged", n_layers=2, vocab=1024, cap=1024, rows=2, layout="paged",
                      page_size=16, num_pages=2 * 1024 // 16 + 7)
    sm = gen.permutation(wl.seed, 97, wl.num_pages)[: 2 * (wl.cap // 16)].reshape(2, wl.cap // 16)
    positions = [17, 900]
    dec_c, mw = make_decoder(wl)
    dec_p, _ = make_decoder(wl, mw=mw, kv_sweep="pos")
    for dec in (dec_c, dec_p):
        dec.set_slot_map(sm)
        for l in range(wl.n_layers):
            for w in (0, 1):
                pool = dec.kv(l, w)
                pool.copy_(_garbage_like(pool))   # unmapped pages and positions after pos
                for r, p in enumerate(positions):
                    place_kv(pool, gen.kv_prefill(wl, l, w, r, p), r, 0, sm, wl.page_size)
    toks = [gen.prompt_tokens(wl, row=r, n=3) for r in range(2)]
    for i in range(3):
        pos = [p + i for p in positions]
        step = [int(toks[r][i]) for r in range(2)]
        _same_step(dec_c.step(step, pos), dec_p.step(step, pos), f"paged step {i}")
    _same_state(dec_c, dec_p, wl)
    dec_c.close()
    dec_p.close()
    del torch


def test_pos_sweep_refusals():
    from graph_replay_gb300 import _binding as B
    wl = gen.WORKLOADS["1b"].replace(name="1b_sweep_refuse", n_layers=2, vocab=1024, cap=256)
    with pytest.raises(RuntimeError, match="GRAPH"):
        make_decoder(wl, strategy="persistent", kv_sweep="pos")
    with pytest.raises(RuntimeError, match="tensor-core attention"):
        make_decoder(gen.WORKLOADS["tiny"], kv_sweep="pos")
    dec, _ = make_decoder(wl)
    assert B.lib().dec_set_kv_sweep(dec.h, B.DEC_SWEEP_POS) == B.DEC_E_STATE   # after capture
    dec.close()
