"""GPU parity of the persistent whole-step kernel (DEC_STRATEGY_PERSISTENT)
against the fp64 oracle, under the same tolerances as the graph strategy
("Execution", section "Verification", tiers 1-2), plus its own invariants:
one kernel per step, replay equal to eager bit for bit, masked positions
never reaching the result, the KV write landing only at pos."""
import numpy as np
import pytest

import gen
import oracle
from _harness import (assert_close, assert_greedy, make_decoder, paged_case, prefilled_positions_case,
                      run_sequence)

pytestmark = pytest.mark.gpu

PERSIST = dict(strategy="persistent")


def test_persistent_1b_prompt_then_greedy():
    wl = gen.WORKLOADS["1b"]
    strict, st = run_sequence(wl, wl.prompt_len, 128, **PERSIST)
    assert strict > 0
    assert st["strategy"] == 1
    assert st["kernels_per_step"] == 1 and st["graph_nodes"] == 1


def test_persistent_replay_equals_eager_bit_exact():
    import torch
    wl = gen.WORKLOADS["1b"].replace(name="1b_l2", n_layers=2, cap=256)
    dec, mw = make_decoder(wl, **PERSIST)
    toks = gen.prompt_tokens(wl, n=40)

    def run():
        out = [dec.step([t], [p]).logits[0].copy() for p, t in enumerate(toks)]
        kv = [dec.kv(l, w).clone() for l in range(wl.n_layers) for w in (0, 1)]
        return out, kv

    graph_logits, graph_kv = run()
    dec.reset_state()
    dec.set_eager(True)
    eager_logits, eager_kv = run()
    dec.reset_state()
    dec.set_eager(False)
    again_logits, again_kv = run()
    dec.close()
    for a, b, c in zip(graph_logits, eager_logits, again_logits):
        assert np.array_equal(a, b)
        assert np.array_equal(a, c)
    for a, b, c in zip(graph_kv, eager_kv, again_kv):
        assert torch.equal(a, b) and torch.equal(a, c)


def test_persistent_close_to_graph_strategy():
    # the two strategies differ only in fp32 summation order
    wl = gen.WORKLOADS["1b"].replace(name="1b_l4", n_layers=4, cap=512)
    mw = gen.make_weights(wl)
    toks = gen.prompt_tokens(wl, n=24)
    outs = {}
    for strat in ("graph", "persistent"):
        dec, _ = make_decoder(wl, mw, strategy=strat)
        outs[strat] = [dec.step([t], [p]).logits[0].copy() for p, t in enumerate(toks)]
        dec.close()
    for i, (a, b) in enumerate(zip(outs["graph"], outs["persistent"])):
        assert_close(b, a, wl, f"persistent vs graph step {i}")


def test_persistent_garbage_after_pos_is_bit_identical():
    import torch
    wl = gen.WORKLOADS["1b"].replace(name="1b_l3", n_layers=3, cap=1024)
    dec, mw = make_decoder(wl, **PERSIST)
    toks = gen.prompt_tokens(wl, n=300)
    for p, t in enumerate(toks[:-1]):
        dec.step([t], [p])
    P = len(toks) - 1
    saved = [dec.kv(l, w).clone() for l in range(wl.n_layers) for w in (0, 1)]
    clean = dec.step([toks[-1]], [P])
    garbage = torch.tensor([float("nan"), float("inf"), -float("inf"), 1e30], dtype=torch.bfloat16,
                           device="cuda:0")
    for k, (l, w) in enumerate((l, w) for l in range(wl.n_layers) for w in (0, 1)):
        store = dec.kv(l, w)
        store.copy_(saved[k])
        tail = store[:, :, P + 1:, :]
        tail.copy_(garbage.repeat(tail.numel() // 4 + 1)[: tail.numel()].view(tail.shape))
    dirty = dec.step([toks[-1]], [P])
    dec.close()
    assert np.array_equal(clean.logits, dirty.logits)
    assert np.array_equal(clean.ids, dirty.ids)


def test_persistent_kv_write_touches_only_pos():
    import torch
    wl = gen.WORKLOADS["1b"].replace(name="1b_l2b", n_layers=2, cap=512)
    dec, mw = make_decoder(wl, **PERSIST)
    for p, t in enumerate(gen.prompt_tokens(wl, n=10)):
        dec.step([t], [p])
    before = [dec.kv(l, w).clone() for l in range(2) for w in (0, 1)]
    dec.step([5], [200])
    for k, (l, w) in enumerate((l, w) for l in range(2) for w in (0, 1)):
        changed = (dec.kv(l, w) != before[k]).any(dim=3).any(dim=1)[0]
        idx = torch.nonzero(changed).flatten().tolist()
        assert idx == [200], (l, w, idx)
    dec.close()


def test_persistent_paged_1b_row1():
    paged_case("1b", 1, 6, n_layers=4, **PERSIST)


def _rows_case(rows, n_steps, n_layers=4, cap=1024, eager_check=True):
    """Rows at independent positions with K/V pre-filled N(0,1) below each row's
    start, stepped together through the persistent kernel and compared with one
    oracle per row; replaying the same steps eagerly gives the same bits."""
    import torch
    from gen.device import place_kv
    wl = gen.WORKLOADS["1b"].replace(name=f"1b_prows{rows}", rows=rows, n_layers=n_layers, cap=cap)
    dec, mw = make_decoder(wl, **PERSIST)
    st = dec.stats()
    assert st["strategy"] == 1 and st["kernels_per_step"] == 1
    start = [int(x) for x in gen.ints(wl.seed, 97, 0, cap - n_steps, rows)]
    toks = [gen.prompt_tokens(wl, row=r, n=n_steps) for r in range(rows)]
    orcs = []
    for r in range(rows):
        orc = oracle.Oracle(mw, cap=cap)
        for l in range(n_layers):
            for which in (0, 1):
                kv = gen.kv_prefill(wl, l, which, r, start[r])
                place_kv(dec.kv(l, which), kv, r)
                (orc.K if which == 0 else orc.V)[0][l][: start[r]] = kv
        orcs.append(orc)
    before = [dec.kv(l, w).clone() for l in range(n_layers) for w in (0, 1)]

    def run():
        out = []
        for i in range(n_steps):
            res = dec.step([int(toks[r][i]) for r in range(rows)], [start[r] + i for r in range(rows)])
            out.append((res.logits.copy(), res.ids.copy(), res.nonfinite.copy()))
        return out

    got = run()
    for i, (logits, ids, nf) in enumerate(got):
        for r in range(rows):
            ref = orcs[r].step(0, int(toks[r][i]), start[r] + i)
            assert_close(logits[r], ref, wl, f"rows {rows} row {r} step {i}")
            assert_greedy(ids[r], ref, f"rows {rows} row {r} step {i}")
            assert nf[r] == 0
    if eager_check:
        kv_graph = [dec.kv(l, w).clone() for l in range(n_layers) for w in (0, 1)]
        for t, b in zip([dec.kv(l, w) for l in range(n_layers) for w in (0, 1)], before):
            t.copy_(b)
        dec.set_eager(True)
        again = run()
        dec.set_eager(False)
        for (a, ia, _), (b, ib, _) in zip(got, again):
            assert np.array_equal(a, b) and np.array_equal(ia, ib)
        for a, l_w in zip(kv_graph, [(l, w) for l in range(n_layers) for w in (0, 1)]):
            assert torch.equal(a, dec.kv(*l_w))
    dec.close()


@pytest.mark.parametrize("rows", [2, 4])
def test_persistent_1b_rows_at_independent_positions(rows):
    _rows_case(rows, n_steps=6)


def test_persistent_unsupported_shape_is_refused():
    # fp32 weights have no persistent kernel: the capture reports it, nothing launches
    from graph_replay_gb300._binding import DEC_E_UNSUPPORTED, DecError
    with pytest.raises(DecError) as ei:
        make_decoder(gen.WORKLOADS["tiny"], **PERSIST)
    assert ei.value.status == DEC_E_UNSUPPORTED


@pytest.mark.parametrize("base, rows, layout", [("1b", 2, "paged"), ("1b", 3, "contiguous"), ("8b", 2, "contiguous")])
def test_persistent_multi_row_shapes_without_a_kernel_are_refused(base, rows, layout):
    # several rows run on the whole-step kernel for the 1B-class shape with
    # contiguous K/V at 2 or 4 rows only; anything else is refused at capture
    from graph_replay_gb300._binding import DEC_E_UNSUPPORTED, DecError
    shape = dict(name=f"{base}_pref{rows}{layout[0]}", rows=rows, n_layers=1, cap=256, vocab=1024, layout=layout)
    if layout == "paged":
        shape.update(page_size=16, num_pages=rows * 16 + 3)
    wl = gen.WORKLOADS[base].replace(**shape)
    with pytest.raises(DecError) as ei:
        make_decoder(wl, **PERSIST)
    assert ei.value.status == DEC_E_UNSUPPORTED


@pytest.mark.slow
def test_persistent_8b_decode_at_prefilled_positions():
    prefilled_positions_case(gen.WORKLOADS["8b"], **PERSIST)
