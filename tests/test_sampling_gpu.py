"""The sampling suffix on the device (temperature / top-k / top-p / min-p,
counter-based uniform, top-n logprobs) against the oracle's sampler run on the
same logits ("Models, Registry and the Driver", section "The Driver":
Head::Sample).

The pick is a floating-point decision: the GPU sums fp32 weights in a fixed
order, the oracle fp64.  A pick must equal the oracle's unless the oracle's
cumulative weight at a cut or at the uniform lies within 1e-5 (relative) of
the boundary between the two picks; then the GPU pick must be the neighbour.
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle
from graph_replay_gb300 import _binding as B
from tests._harness import make_decoder

pytestmark = pytest.mark.gpu

SAMPLER = dict(temperature=0.8, top_k=40, top_p=0.9, min_p=0.02, seed=1234, n_logprobs=4)


def _check_pick(gpu_id, logits, row, pos, s):
    u = oracle.uniform(s["seed"], row, pos)
    tok, order, S, last = oracle.sample(logits, s["temperature"], s["top_k"], s["top_p"], s["min_p"], u)
    if int(gpu_id) == tok:
        return True
    # only at a boundary: the uniform, the top-p cut or the min-p cut within 1e-5 of it
    tot = S[last]
    j = list(order).index(tok)
    assert int(gpu_id) in [int(x) for x in order[max(0, j - 1): j + 2]], (gpu_id, tok)
    near_u = min(abs(u * tot - S[j]), abs(u * tot - (S[j - 1] if j else 0.0))) <= 1e-5 * tot
    near_p = abs(S[last] - s["top_p"] * S[-1]) <= 1e-5 * S[-1] or \
        (last > 0 and abs(S[last - 1] - s["top_p"] * S[-1]) <= 1e-5 * S[-1])
    q = np.exp((np.asarray(logits, np.float64)[order] - np.max(logits)) / s["temperature"])
    near_m = bool(np.any(np.abs(q - s["min_p"]) <= 1e-5))
    assert near_u or near_p or near_m, (gpu_id, tok, u)
    return False


def _run(wl, steps, sampler, **kw):
    dec, mw = make_decoder(wl, sampler=sampler, **kw)
    toks = np.stack([gen.prompt_tokens(wl, row=r, n=steps) for r in range(wl.rows)])
    exact = 0
    for i in range(steps):
        pos = [i + 3 * r for r in range(wl.rows)]
        res = dec.step(toks[:, i], pos)
        for r in range(wl.rows):
            exact += _check_pick(res.ids[r], res.logits[r], r, pos[r], sampler)
        ids, lp = dec.logprobs(sampler["n_logprobs"])
        for r in range(wl.rows):
            want_ids, want_lp = oracle.top_logprobs(res.logits[r], sampler["n_logprobs"])
            assert list(ids[r]) == [int(x) for x in want_ids]
            assert np.allclose(lp[r], want_lp, atol=1e-4)
    dec.close()
    return exact


@pytest.mark.parametrize("name, rows, strategy", [("1b", 2, "graph"), ("1b", 1, "persistent"), ("tiny", 1, "graph")])
def test_sampled_ids_match_the_oracle_sampler(name, rows, strategy):
    wl = gen.WORKLOADS[name].replace(name=f"{name}_s", n_layers=2, cap=128, rows=rows)
    exact = _run(wl, 24, SAMPLER, strategy=strategy)
    assert exact >= 24 * rows - 1


def test_temperature_zero_is_greedy_and_parameters_change_in_place():
    wl = gen.WORKLOADS["1b"].replace(name="1b_s0", n_layers=2, cap=128, rows=2)
    mw = gen.make_weights(wl)
    plain, _ = make_decoder(wl, mw)
    dec, _ = make_decoder(wl, mw, sampler=dict(temperature=0.0, n_logprobs=2))
    toks = np.stack([gen.prompt_tokens(wl, row=r, n=10) for r in range(2)])
    for i in range(10):
        a = plain.step(toks[:, i], [i, i])
        b = dec.step(toks[:, i], [i, i])
        assert np.array_equal(a.logits, b.logits)
        assert np.array_equal(a.ids, b.ids)
    s = dict(temperature=1.0, top_k=50, top_p=0.95, min_p=0.0, seed=7, n_logprobs=2)
    dec.set_sampler(**s)
    for i in range(10, 20):
        res = dec.step(toks[:, i - 10], [i, i])
        for r in range(2):
            _check_pick(res.ids[r], res.logits[r], r, i, s)
    dec.set_sampler(temperature=0.0, n_logprobs=2)
    res = dec.step(toks[:, 0], [20, 20])
    assert list(res.ids) == [int(np.argmax(res.logits[r])) for r in range(2)]
    plain.close()
    dec.close()


def test_chain_feeds_the_sampled_ids():
    wl = gen.WORKLOADS["1b"].replace(name="1b_sc", n_layers=2, cap=128, rows=2)
    dec, _ = make_decoder(wl, sampler=SAMPLER)
    first = [5, 9]
    ids_c, _ = dec.chain(first, [0, 0], 16)
    dec.reset_state()
    cur = np.array(first)
    for i in range(16):
        res = dec.step(cur, [i, i], logits=False)
        assert np.array_equal(res.ids, ids_c[i])
        cur = res.ids
    dec.close()


def test_sampler_refusals():
    wl = gen.WORKLOADS["1b"].replace(name="1b_sr", n_layers=1, cap=64)
    dec, _ = make_decoder(wl)
    with pytest.raises(B.DecError) as e:
        dec.set_sampler(temperature=1.0, top_k=10)          # nothing recorded at capture
    assert e.value.status == B.DEC_E_STATE
    dec.close()
    with pytest.raises(B.DecError) as e:
        make_decoder(wl, sampler=dict(temperature=1.0, top_k=5000))
    assert e.value.status == B.DEC_E_INVALID
    dec, _ = make_decoder(wl, sampler=dict(temperature=0.0, n_logprobs=2))
    with pytest.raises(B.DecError) as e:
        dec.logprobs(3)
    assert e.value.status == B.DEC_E_INVALID
    dec.close()
