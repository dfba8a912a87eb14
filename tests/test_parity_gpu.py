"""GPU parity: the captured decode step against the fp64 oracle, through the C ABI.

Tolerances ("Execution", section "Verification", tiers 1-2): integer and
movement work bit-exact (KV write addresses, paged maps, capture versus eager,
greedy ids where the oracle's top-2 margin exceeds 0.05); logits and the
carried KV state within max-abs 2e-2 and relative L2 5e-3 for bf16 weights
with fp32 accumulation, and within 1e-4 relative for the fp32 tiny model.
"""
import numpy as np
import pytest

import gen
import oracle
from _harness import (assert_close, assert_close_state, assert_greedy, kv_as_float, make_decoder, paged_case,
                      prefilled_positions_case, run_sequence)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "tiny_gain"])
def test_tiny_prompt_then_greedy(name):
    wl = gen.WORKLOADS[name]
    strict, st = run_sequence(wl, wl.prompt_len, wl.decode_steps)
    assert st["replays"] == wl.prompt_len + wl.decode_steps
    assert st["graph_nodes"] == st["kernels_per_step"]


@pytest.mark.parametrize("kv_heads", [1, 2])
def test_tiny_gqa_groups(kv_heads):
    wl = gen.WORKLOADS["tiny"].replace(name=f"tiny_kv{kv_heads}", n_kv_heads=kv_heads)
    run_sequence(wl, 16, 8)


def test_tiny_bf16_weights_and_kv():
    wl = gen.WORKLOADS["tiny"].replace(name="tiny_bf16", wdtype="bf16", kvdtype="bf16")
    run_sequence(wl, 16, 16)


def test_1b_prompt_then_greedy():
    # configuration 2: 128 prompt tokens stepped in, then 256 greedy decode steps
    wl = gen.WORKLOADS["1b"]
    strict, st = run_sequence(wl, wl.prompt_len, wl.decode_steps)
    assert strict > 0


def test_capture_equals_eager_bit_exact():
    # "Execution", section "Verification", tier 1: capture versus eager on one device is bit-exact
    wl = gen.WORKLOADS["1b"].replace(name="1b_l2", n_layers=2, cap=256)
    dec, mw = make_decoder(wl)
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
    again_logits, _ = run()
    st = dec.stats()
    dec.close()
    for a, b, c in zip(graph_logits, eager_logits, again_logits):
        assert np.array_equal(a, b)
        assert np.array_equal(a, c)
    import torch
    for a, b in zip(graph_kv, eager_kv):
        assert torch.equal(a, b)
    assert st["eager_steps"] == len(toks)


def test_garbage_after_pos_is_bit_identical():
    # masked positions never reach the result ("Execution", section "A constant-shape decode graph")
    import torch
    wl = gen.WORKLOADS["1b"].replace(name="1b_l3", n_layers=3, cap=1024)
    dec, mw = make_decoder(wl)
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


def test_kv_write_touches_only_pos():
    import torch
    wl = gen.WORKLOADS["1b"].replace(name="1b_l2b", n_layers=2, cap=512)
    dec, mw = make_decoder(wl)
    for p, t in enumerate(gen.prompt_tokens(wl, n=10)):
        dec.step([t], [p])
    before = [dec.kv(l, w).clone() for l in range(2) for w in (0, 1)]
    dec.step([5], [200])   # a later position, gap in between
    for k, (l, w) in enumerate((l, w) for l in range(2) for w in (0, 1)):
        changed = (dec.kv(l, w) != before[k]).any(dim=3).any(dim=1)[0]   # [cap]
        idx = torch.nonzero(changed).flatten().tolist()
        assert idx == [200], (l, w, idx)
    dec.close()


@pytest.mark.slow
def test_8b_decode_at_prefilled_positions():
    # configuration 3 at full size: one step at pos in {1, 1024, 4096, 8191} over KV pre-filled N(0,1)
    prefilled_positions_case(gen.WORKLOADS["8b"])


@pytest.mark.slow
@pytest.mark.parametrize("strategy", ["graph", "persistent"])
def test_1b_long_cap_rows4(strategy):
    # configuration 5: cap 32768, 4 rows at pos {100, 8000, 20000, 32767}
    wl = gen.WORKLOADS["1b_long"]
    dec, mw = make_decoder(wl, strategy=strategy)
    positions = gen.row_positions(wl)
    toks = gen.prompt_tokens(wl, n=wl.rows)
    from gen.device import place_kv
    for r in range(wl.rows):
        for l in range(wl.n_layers):
            for which in (0, 1):
                place_kv(dec.kv(l, which), gen.kv_prefill(wl, l, which, r, int(positions[r])), r)
    res = dec.step(toks, positions)
    for r in range(wl.rows):
        orc = oracle.Oracle(mw, cap=wl.cap)
        for l in range(wl.n_layers):
            orc.K[0][l][: positions[r]] = gen.kv_prefill(wl, l, 0, r, int(positions[r]))
            orc.V[0][l][: positions[r]] = gen.kv_prefill(wl, l, 1, r, int(positions[r]))
        ref = orc.step(0, int(toks[r]), int(positions[r]))
        assert_close(res.logits[r], ref, wl, f"1b_long row {r}")
        assert_greedy(res.ids[r], ref, f"1b_long row {r}")
        del orc
    dec.close()


def test_paged_tiny_rows2():
    paged_case("tiny", 2, 12)


def test_paged_1b_rows4():
    paged_case("1b", 4, 6, n_layers=4)


@pytest.mark.parametrize("name, rows", [("1b", 2), ("8b", 1)])
def test_attention_op_against_oracle(name, rows):
    """dec_attention alone: RoPE, K/V write at pos, masked full-capacity sweep,
    against the oracle's rotation, storage rounding and causal attention."""
    import torch
    base = gen.WORKLOADS[name]
    wl = base.replace(name=f"{name}_attn", n_layers=2, vocab=1024, cap=2048, rows=rows)
    dec, mw = make_decoder(wl)
    from gen.device import place_kv, read_kv
    positions = [1500, 777][:rows]
    for r in range(rows):
        for which in (0, 1):
            place_kv(dec.kv(1, which), gen.kv_prefill(wl, 1, which, r, positions[r]), r)
    qkv_h = gen.normal(wl.seed, 77, (rows, wl.q_dim + 2 * wl.kv_dim), sigma=1.0, dtype="f32")
    qkv = torch.from_numpy(qkv_h).cuda()
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda:0")
    out = torch.empty(rows, wl.q_dim, dtype=torch.float32, device="cuda:0")
    dec.attention(1, qkv, pos, out)
    got = out.cpu().numpy()
    hd, G = wl.head_dim, wl.n_heads // wl.n_kv_heads
    for r in range(rows):
        p = positions[r]
        K = gen.kv_prefill(wl, 1, 0, r, p + 1).copy()
        V = gen.kv_prefill(wl, 1, 1, r, p + 1).copy()
        q = qkv_h[r, : wl.q_dim].astype(np.float64).reshape(wl.n_heads, hd)
        k = qkv_h[r, wl.q_dim: wl.q_dim + wl.kv_dim].astype(np.float64).reshape(wl.n_kv_heads, hd)
        v = qkv_h[r, wl.q_dim + wl.kv_dim:].astype(np.float64).reshape(wl.n_kv_heads, hd)
        for gi in range(wl.n_kv_heads):
            kr = oracle.rope(k[gi], p, wl.rope_theta)
            K[p, gi] = [oracle.bf16_round(z) for z in kr]
            V[p, gi] = [oracle.bf16_round(z) for z in v[gi]]
        # the store now holds the oracle's rounding of the new k, v at p (one storage ulp allowed)
        got_k = kv_as_float(read_kv(dec.kv(1, 0), r, p + 1))
        assert_close_state(got_k[p], kv_as_float(K[p]), wl, "attention op K write")
        ref = np.concatenate([oracle.attend(oracle.rope(q[i], p, wl.rope_theta), K[:, i // G], V[:, i // G])
                              for i in range(wl.n_heads)])
        assert_close(got[r], ref, wl, f"attention op row {r}")
    dec.close()
