"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks one oracle function against a closed form, an invariant, a
special case that reduces to a library routine, or a hand-derived value, so
that a plausible slip (a dropped term, a wrong sign or index, a transposed
operand) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import expit, softmax as sp_softmax

import gen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------- bf16 storage rounding ----------------

def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            yield line.split(None, 2)


@pytest.mark.parametrize("row", list(_golden_rows("bf16_rounding.txt")), ids=lambda r: r[0])
def test_bf16_rounding_golden(row):
    src, bits, _why = row
    v = float(src) if src in ("inf", "-inf") else float.fromhex(src)
    assert oracle.bf16_round(v) == int(bits, 16)


def test_bf16_rounding_matches_torch_on_binary32_values():
    # For values already representable in binary32, one rounding to bf16 is
    # what torch's float32 -> bfloat16 conversion does (a library routine).
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.standard_normal(4000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 4000),
                           rng.standard_normal(1000).astype(np.float32)]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_value_widening_is_exact():
    for bits in (0x3F80, 0xC020, 0x4049, 0x0001, 0x7F7F):
        f = np.array([bits], dtype=np.uint16)
        assert oracle.bf16_value(bits) == float(gen.bf16_bits_to_f32(f)[0])


# ---------------- RMSNorm ----------------

def test_rmsnorm_hand_values():
    # x = (3, 4): mean(x^2) = 12.5; with eps = 0 and unit gain the output is x / sqrt(12.5)
    out = oracle.rmsnorm([3.0, 4.0], np.ones(2), 0.0)
    assert np.allclose(out, [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=0, atol=1e-15)
    # eps sits inside the root: x = (1, 1, 1, 1), eps = 1 -> 1 / sqrt(2)
    out = oracle.rmsnorm(np.ones(4), np.ones(4), 1.0)
    assert np.allclose(out, 1 / math.sqrt(2.0), rtol=0, atol=1e-15)


def test_rmsnorm_unit_rms_and_gain():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(257)
    out = oracle.rmsnorm(x, np.ones(257), 0.0)
    assert abs(math.sqrt(np.mean(out ** 2)) - 1.0) < 1e-13
    # scale invariance with eps -> 0
    out2 = oracle.rmsnorm(1e3 * x, np.ones(257), 0.0)
    assert np.allclose(out, out2, rtol=1e-13, atol=0)
    # the gain multiplies element-wise (not 1 + g)
    g = rng.uniform(0.5, 2.0, 257)
    assert np.allclose(oracle.rmsnorm(x, g, 0.0), out * g, rtol=1e-14, atol=0)
    # bf16 and fp32 gains are read exactly
    gb = gen.normal(3, 4, (257,), sigma=0.1, mean=1.0, dtype="bf16")
    assert np.allclose(oracle.rmsnorm(x, gb, 0.0), out * gen.bf16_bits_to_f32(gb), rtol=1e-14, atol=0)


# ---------------- matrix-vector ----------------

@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_matvec_against_numpy(dt):
    W = gen.normal(11, 12, (37, 53), sigma=0.5, dtype=dt)
    h = np.random.default_rng(2).standard_normal(53)
    Wf = gen.bf16_bits_to_f32(W) if dt == "bf16" else W
    ref = Wf.astype(np.float64) @ h      # numpy, a library routine; non-square catches a transpose
    assert np.allclose(oracle.matvec(W, h), ref, rtol=1e-13, atol=1e-13)


# ---------------- RoPE ----------------

def test_rope_hd2_is_a_rotation_by_pos_radians():
    # head_dim 2: one pair, frequency theta^0 = 1, so the angle is pos radians
    for pos in (0, 1, 5, 1000):
        out = oracle.rope([1.0, 0.0], pos, 10000.0)
        assert np.allclose(out, [math.cos(pos), math.sin(pos)], atol=1e-15)
        out = oracle.rope([0.0, 1.0], pos, 10000.0)
        assert np.allclose(out, [-math.sin(pos), math.cos(pos)], atol=1e-15)


def test_rope_frequency_and_half_split_pairing():
    # hd = 8, theta = 1e4: w_i = 1e4^(-2i/8) = 10^(-i); component i pairs with i + 4
    hd, theta, pos = 8, 1e4, 3
    for i in range(4):
        v = np.zeros(hd)
        v[i] = 1.0
        out = oracle.rope(v, pos, theta)
        ang = pos * 10.0 ** (-i)
        exp = np.zeros(hd)
        exp[i] = math.cos(ang)
        exp[i + 4] = math.sin(ang)
        assert np.allclose(out, exp, atol=1e-14), i


def test_rope_invariants():
    rng = np.random.default_rng(3)
    hd = 128
    q = rng.standard_normal(hd)
    k = rng.standard_normal(hd)
    # pos 0 is the identity
    assert np.array_equal(oracle.rope(q, 0, 5e5), q)
    # per-pair norms are preserved
    out = oracle.rope(q, 777, 5e5)
    n0 = np.hypot(q[:64], q[64:])
    n1 = np.hypot(out[:64], out[64:])
    assert np.allclose(n0, n1, rtol=1e-12, atol=0)
    # q(p) . k(p') depends only on p - p'
    a = oracle.rope(q, 40, 1e4) @ oracle.rope(k, 15, 1e4)
    b = oracle.rope(q, 1040, 1e4) @ oracle.rope(k, 1015, 1e4)
    assert abs(a - b) < 1e-10


# ---------------- softmax, SiLU, argmax ----------------

def test_softmax_against_scipy_and_shift():
    rng = np.random.default_rng(4)
    s = rng.standard_normal(50) * 5
    assert np.allclose(oracle.softmax(s), sp_softmax(s), rtol=1e-14, atol=0)
    assert np.allclose(oracle.softmax(s + 1000.0), sp_softmax(s), rtol=1e-12, atol=0)
    two = oracle.softmax([math.log(3.0), 0.0])
    assert np.allclose(two, [0.75, 0.25], atol=1e-16)


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    for z in (-7.5, -1.0, 0.3, 2.0, 30.0):
        assert abs(oracle.silu(z) - z * expit(z)) < 1e-15 * max(1.0, abs(z))
        # silu(-z) = silu(z) - z
        assert abs(oracle.silu(-z) - (oracle.silu(z) - z)) < 1e-14 * max(1.0, abs(z))


def test_argmax_lowest_index_on_ties():
    assert oracle.argmax([1.0, 3.0, 2.0, 3.0]) == 1
    assert oracle.argmax([-5.0, -5.0]) == 0
    rng = np.random.default_rng(5)
    v = rng.integers(0, 20, 1000).astype(np.float64)
    assert oracle.argmax(v) == int(np.argmax(v))   # numpy also returns the first maximum


# ---------------- one attention head ----------------

def test_attend_single_position_returns_v0():
    rng = np.random.default_rng(6)
    q = rng.standard_normal(16)
    K = rng.standard_normal((1, 16))
    V = rng.standard_normal((1, 16))
    assert np.array_equal(oracle.attend(q, K, V), V[0])


def test_attend_scale_is_inverse_sqrt_hd():
    # scores q.k / sqrt(hd) = (ln 3, 0) -> weights (3/4, 1/4)
    hd = 16
    q = np.zeros(hd)
    q[0] = math.sqrt(hd) * math.log(3.0)
    K = np.zeros((2, hd))
    K[0, 0] = 1.0
    V = np.zeros((2, hd))
    V[0, :] = 4.0
    V[1, :] = 8.0
    assert np.allclose(oracle.attend(q, K, V), 0.75 * 4.0 + 0.25 * 8.0, atol=1e-14)


def test_attend_equal_keys_give_mean_and_library_softmax():
    rng = np.random.default_rng(8)
    q = rng.standard_normal(8)
    K = np.tile(rng.standard_normal(8), (5, 1))
    V = rng.standard_normal((5, 8))
    assert np.allclose(oracle.attend(q, K, V), V.mean(axis=0), atol=1e-15)
    K = rng.standard_normal((7, 8))
    w = sp_softmax(K @ q / math.sqrt(8))
    assert np.allclose(oracle.attend(q, K, V := rng.standard_normal((7, 8))), w @ V, atol=1e-14)
    # bf16 K/V are read exactly
    Kb = gen.normal(1, 9, (7, 8), dtype="bf16")
    Vb = gen.normal(1, 10, (7, 8), dtype="bf16")
    Kf, Vf = gen.bf16_bits_to_f32(Kb).astype(np.float64), gen.bf16_bits_to_f32(Vb).astype(np.float64)
    assert np.allclose(oracle.attend(q, Kb, Vb), sp_softmax(Kf @ q / math.sqrt(8)) @ Vf, atol=1e-14)


# ---------------- whole steps ----------------

def _tiny(**kw):
    wl = gen.WORKLOADS["tiny"].replace(**kw)
    return wl, gen.make_weights(wl)


@pytest.mark.parametrize("name", ["tiny", "tiny_gain"])
def test_stepping_equals_full_causal_pass(name):
    wl = gen.WORKLOADS[name]
    mw = gen.make_weights(wl)
    o = oracle.Oracle(mw, cap=wl.cap)
    toks = gen.prompt_tokens(wl)
    stepped = np.array([o.step(0, t, p) for p, t in enumerate(toks)])
    full, Ks, Vs = o.full_causal(toks)
    assert np.abs(stepped - full).max() <= 1e-12
    for l in range(wl.n_layers):
        assert np.array_equal(Ks[l], o.K[0][l][: len(toks)])
        assert np.array_equal(Vs[l], o.V[0][l][: len(toks)])


def test_garbage_after_pos_leaves_logits_bit_identical():
    wl, mw = _tiny()
    toks = gen.prompt_tokens(wl)
    a = oracle.Oracle(mw, cap=wl.cap)
    b = oracle.Oracle(mw, cap=wl.cap)
    garbage = np.array([np.nan, np.inf, -np.inf, 1e30], dtype=np.float32)
    for p, t in enumerate(toks):
        la = a.step(0, t, p)
        for l in range(wl.n_layers):     # poison every position after p
            tail = b.K[0][l][p + 1:]
            tail[...] = np.resize(garbage, tail.shape)
            b.V[0][l][p + 1:][...] = np.resize(garbage[::-1], tail.shape)
        lb = b.step(0, t, p)
        assert np.array_equal(la, lb)


def test_gqa_equals_mha_with_duplicated_kv_heads():
    # A GQA model (4 q heads, 2 kv heads) must equal the MHA model whose K/V
    # projections repeat each kv head for its group of G = 2 q heads.
    wl = gen.WORKLOADS["tiny"].replace(n_kv_heads=2, name="tiny_gqa")
    mw = gen.make_weights(wl)
    hd, G = wl.head_dim, wl.n_heads // wl.n_kv_heads
    wl2 = wl.replace(n_kv_heads=wl.n_heads)
    mw2 = gen.ModelWeights(wl=wl2, embed=mw.embed, final_norm=mw.final_norm, lm_head=mw.lm_head)
    for lw in mw.layers:
        d2 = dict(lw)
        for r in ("wk", "wv"):
            heads = lw[r].reshape(wl.n_kv_heads, hd, wl.d_model)
            d2[r] = np.ascontiguousarray(np.repeat(heads, G, axis=0).reshape(wl.n_heads * hd, wl.d_model))
        mw2.layers.append(d2)
    a = oracle.Oracle(mw, cap=wl.cap)
    b = oracle.Oracle(mw2, cap=wl.cap)
    for p, t in enumerate(gen.prompt_tokens(wl)[:8]):
        assert np.abs(a.step(0, t, p) - b.step(0, t, p)).max() <= 1e-13


def test_zero_mixer_and_ffn_reduce_to_embedding_head():
    # Wo = 0 and Wd = 0 leave x = E[token]; logits = W_head (rmsnorm(E[token]) * g)
    wl, mw = _tiny(gain_sigma=0.1)
    for lw in mw.layers:
        lw["wo"] = np.zeros_like(lw["wo"])
        lw["wd"] = np.zeros_like(lw["wd"])
    o = oracle.Oracle(mw, cap=wl.cap)
    tok = 77
    x = mw.embed[tok].astype(np.float64)
    g = mw.final_norm.astype(np.float64)
    h = x / math.sqrt(np.mean(x * x) + wl.rms_eps) * g
    ref = mw.lm_head.astype(np.float64) @ h
    assert np.allclose(o.step(0, tok, 5), ref, rtol=1e-12, atol=1e-14)


def test_swiglu_block_special_case():
    # one layer with a zero mixer: x1 = x + Wd (silu(Wg h) * (Wu h)), h = rmsnorm(x) g
    # (the textbook SwiGLU feed-forward, evaluated with numpy / scipy routines)
    wl, mw = _tiny(n_layers=1, gain_sigma=0.1)
    mw.layers[0]["wo"] = np.zeros_like(mw.layers[0]["wo"])
    o = oracle.Oracle(mw, cap=wl.cap)
    tok = 201
    f64 = lambda a: a.astype(np.float64)
    lw = mw.layers[0]
    x = f64(mw.embed[tok])
    h = x / math.sqrt(np.mean(x * x) + wl.rms_eps) * f64(lw["ffn_norm"])
    gt, up = f64(lw["wg"]) @ h, f64(lw["wu"]) @ h
    x1 = x + f64(lw["wd"]) @ (gt * expit(gt) * up)
    hf = x1 / math.sqrt(np.mean(x1 * x1) + wl.rms_eps) * f64(mw.final_norm)
    assert np.allclose(o.step(0, tok, 0), f64(mw.lm_head) @ hf, rtol=1e-12, atol=1e-14)


def test_step_refuses_out_of_range():
    wl, mw = _tiny()
    o = oracle.Oracle(mw, cap=wl.cap)
    with pytest.raises(ValueError):
        o.step(0, wl.vocab, 0)
    with pytest.raises(ValueError):
        o.step(0, 0, wl.cap)


def test_kv_write_stores_rounded_projection_at_pos_only():
    # bf16 weights and KV: at pos 0 RoPE is the identity, so the stored k and v
    # are the bf16 rounding of Wk h and Wv h with h = rmsnorm(E[token]) g
    # (numpy matmul); every other position of the store is left untouched.
    wl, mw = _tiny(n_layers=1, wdtype="bf16", kvdtype="bf16", gain_sigma=0.1)
    o = oracle.Oracle(mw, cap=wl.cap)
    before_k = o.K[0][0].copy()
    tok = 9
    o.step(0, tok, 0)
    f = lambda a: gen.bf16_bits_to_f32(a).astype(np.float64)
    lw = mw.layers[0]
    x = f(mw.embed[tok])
    h = x / math.sqrt(np.mean(x * x) + wl.rms_eps) * f(lw["attn_norm"])
    k = f(lw["wk"]) @ h
    v = f(lw["wv"]) @ h
    exp_k = np.array([oracle.bf16_round(z) for z in k], dtype=np.uint16)
    exp_v = np.array([oracle.bf16_round(z) for z in v], dtype=np.uint16)
    assert np.array_equal(o.K[0][0][0].ravel(), exp_k)
    assert np.array_equal(o.V[0][0][0].ravel(), exp_v)
    assert np.array_equal(o.K[0][0][1:], before_k[1:])
    # a later step writes only its own position
    k1 = o.K[0][0].copy()
    o.step(0, 3, 7)
    changed = np.nonzero((o.K[0][0] != k1).any(axis=(1, 2)))[0]
    assert list(changed) == [7]


# ---- sampling suffix ----

def test_splitmix64_published_outputs():
    # the first three outputs of splitmix64 started at 0, as published with the generator
    assert [oracle.splitmix64_at(0, i) for i in range(3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                                               0x06C45D188009454F]


def test_uniform_is_in_unit_interval_and_varies():
    us = [oracle.uniform(99, r, p) for r in range(3) for p in range(200)]
    assert all(0.0 <= u < 1.0 for u in us)
    assert len(set(us)) == len(us)
    assert abs(np.mean(us) - 0.5) < 0.05


def test_sample_limits_reduce_to_greedy():
    rng = np.random.default_rng(3)
    l = rng.normal(size=50)
    g = int(np.argmax(l))
    for u in (0.0, 0.37, 0.999):
        assert oracle.sample(l, 0.0, 10, 1.0, 0.0, u)[0] == g        # temperature 0
        assert oracle.sample(l, 1.3, 1, 1.0, 0.0, u)[0] == g         # top_k = 1
        assert oracle.sample(l, 1.3, 50, 1e-9, 0.0, u)[0] == g       # tiny top_p
        assert oracle.sample(l, 1.3, 50, 1.0, 0.999, u)[0] == g      # min_p near 1


def test_sample_top_p_and_min_p_cuts():
    # probabilities 0.5, 0.3, 0.2 at temperature 1: cumulative 0.5, 0.8, 1.0
    l = np.log([0.5, 0.3, 0.2])
    for top_p, last in ((0.49, 0), (0.51, 1), (0.79, 1), (0.81, 2), (1.0, 2)):
        assert oracle.sample(l, 1.0, 3, top_p, 0.0, 0.0)[3] == last
    # relative probabilities 1, 0.6, 0.4
    assert oracle.sample(l, 1.0, 3, 1.0, 0.5, 0.0)[3] == 1
    assert oracle.sample(l, 1.0, 3, 1.0, 0.61, 0.0)[3] == 0
    assert oracle.sample(l, 1.0, 3, 0.81, 0.39, 0.0)[3] == 2
    assert oracle.sample(l, 1.0, 3, 0.81, 0.41, 0.0)[3] == 1


def test_sample_frequencies_equal_the_kept_softmax():
    # u on a fine grid: each kept token is picked for exactly its share of the grid
    from scipy.special import softmax
    rng = np.random.default_rng(11)
    l = rng.normal(size=12) * 2
    T, k, top_p, min_p, M = 0.7, 8, 0.9, 0.05, 20000
    picks = np.array([oracle.sample(l, T, k, top_p, min_p, (i + 0.5) / M)[0] for i in range(M)])
    order = list(np.argsort(-l, kind="stable"))[:k]
    p = softmax(l[order] / T)
    keep = 0
    while np.sum(p[: keep + 1]) < top_p - 1e-12:
        keep += 1
    keep = min(keep, int(np.sum(p / p[0] >= min_p)) - 1)
    want = p[: keep + 1] / np.sum(p[: keep + 1])
    for j, tok in enumerate(order):
        freq = np.mean(picks == tok)
        assert abs(freq - (want[j] if j <= keep else 0.0)) <= 1.0 / M + 1e-12, (j, freq)


def test_sample_ties_go_to_the_lower_index():
    l = np.array([1.0, 3.0, 2.0, 3.0, 3.0])
    tok, order, _, _ = oracle.sample(l, 1.0, 2, 1.0, 0.0, 0.99)
    assert list(order) == [1, 3]
    assert tok == 3
    ids, _ = oracle.top_logprobs(l, 4)
    assert list(ids) == [1, 3, 4, 2]


def test_top_logprobs_closed_form():
    from scipy.special import logsumexp
    ids, lp = oracle.top_logprobs([0.0, np.log(3.0)], 2)
    assert list(ids) == [1, 0]
    assert np.allclose(lp, [np.log(0.75), np.log(0.25)], atol=1e-15)
    rng = np.random.default_rng(5)
    l = rng.normal(size=1000) * 3
    ids, lp = oracle.top_logprobs(l, 5)
    assert np.allclose(lp, l[ids] - logsumexp(l), atol=1e-12)
