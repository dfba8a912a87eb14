"""GPU parity of the persistent whole-step kernel (DEC_STRATEGY_PERSISTENT)
against the fp64 oracle, under the same tolerances as the graph strategy
("Execution", section "Verification", tiers 1-2), plus its own invariants:
one kernel per step, replay equal to eager bit for bit, masked positions
never reaching the result, the KV write landing only at pos."""
import numpy as np
import pytest

import gen
import oracle
from _harness import assert_close, make_decoder, paged_case, prefilled_positions_case, run_sequence

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


def test_persistent_unsupported_shape_is_refused():
    # fp32 weights have no persistent kernel: the capture reports it, nothing launches
    from graph_replay_gb300._binding import DEC_E_UNSUPPORTED, DecError
    with pytest.raises(DecError) as ei:
        make_decoder(gen.WORKLOADS["tiny"], **PERSIST)
    assert ei.value.status == DEC_E_UNSUPPORTED


@pytest.mark.slow
def test_persistent_8b_decode_at_prefilled_positions():
    prefilled_positions_case(gen.WORKLOADS["8b"], **PERSIST)
