"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one piece of the oracle against a closed form, an invariant
of the definition, a library routine (torch fp64 ops, torch's bf16 rounding),
or brute force on a model small enough to work out by hand.  They are chosen
so that a plausible slip (a dropped term, a wrong sign or index, the other
RoPE pairing, the wrong GQA head map, an off-by-one in the causal window)
fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

RNG = np.random.default_rng(1234)


def bf16_bits(a) -> np.ndarray:
    """float values -> bf16 bit patterns via torch's own float32 -> bf16 rounding."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_vals(bits) -> np.ndarray:
    return synth.bf16_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


# --------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch():
    x = np.concatenate([RNG.standard_normal(20000) * 10.0 ** RNG.integers(-6, 6, 20000),
                        [0.0, -0.0, 1.0, -2.5, 1e30, -1e-30]])
    ours = np.array([oracle.round_bf16(v) for v in x], dtype=np.uint16)
    assert np.array_equal(ours, bf16_bits(x))


def test_round_bf16_ties_to_even():
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 0x3F80          # halfway, even below
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82      # halfway, even above
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC040) == -3.0


# --------------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("c", [1.0, 1.5, -0.75])
def test_rmsnorm_rms_equals_gain(c):
    x = RNG.standard_normal(256) * 3.0
    g = bf16_bits(np.full(256, c))
    eps = 1e-5
    y = oracle.rmsnorm(x, g, eps)
    ms = np.mean(x * x)
    assert math.isclose(np.sqrt(np.mean(y * y)), abs(c) * math.sqrt(ms / (ms + eps)), rel_tol=1e-12)
    y0 = oracle.rmsnorm(x, g, 0.0)
    assert math.isclose(np.sqrt(np.mean(y0 * y0)), abs(c), rel_tol=1e-12)


def test_rmsnorm_scale_invariant_and_gain_elementwise():
    x = RNG.standard_normal(512)
    ones = bf16_bits(np.ones(512))
    g = bf16_bits(RNG.normal(1.0, 0.1, 512))
    a = oracle.rmsnorm(x, ones, 0.0)
    b = oracle.rmsnorm(7.25 * x, ones, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-13)
    np.testing.assert_allclose(oracle.rmsnorm(x, g, 0.0), a * bf16_vals(g), rtol=1e-13)
    # no mean subtraction: a constant vector normalises to +-1, not to 0
    np.testing.assert_allclose(oracle.rmsnorm(np.full(8, 3.0), ones[:8], 0.0), np.ones(8), rtol=1e-15)


# ------------------------------------------------------------------------ RoPE

def test_rope_position_zero_is_identity():
    v = RNG.standard_normal(64)
    assert np.array_equal(oracle.rope(v, 0, 10000.0), v)


def test_rope_closed_form_head_dim_4():
    # hd = 4: pairs (0, 2) and (1, 3), frequencies theta^0 = 1 and theta^(-1/2)
    v = np.array([1.0, 2.0, 3.0, 4.0])
    pos, theta = 3, 10000.0
    a0, a1 = pos * 1.0, pos / 100.0
    want = [1 * math.cos(a0) - 3 * math.sin(a0), 2 * math.cos(a1) - 4 * math.sin(a1),
            3 * math.cos(a0) + 1 * math.sin(a0), 4 * math.cos(a1) + 2 * math.sin(a1)]
    np.testing.assert_allclose(oracle.rope(v, pos, theta), want, rtol=0, atol=1e-14)


@pytest.mark.parametrize("hd,theta", [(64, 10000.0), (128, 500000.0)])
def test_rope_preserves_pair_norms(hd, theta):
    v = RNG.standard_normal(hd)
    r = oracle.rope(v, 1234, theta)
    h = hd // 2
    np.testing.assert_allclose(v[:h] ** 2 + v[h:] ** 2, r[:h] ** 2 + r[h:] ** 2, rtol=1e-12)


def test_rope_relative_position_and_composition():
    hd, theta = 64, 500000.0
    q, k = RNG.standard_normal(hd), RNG.standard_normal(hd)
    for m, n in [(5, 2), (100, 37), (4000, 3999), (31000, 7)]:
        lhs = oracle.rope(q, m, theta) @ oracle.rope(k, n, theta)
        rhs = oracle.rope(q, m - n, theta) @ k
        assert math.isclose(lhs, rhs, rel_tol=1e-9, abs_tol=1e-9)
    v = RNG.standard_normal(hd)
    np.testing.assert_allclose(oracle.rope(oracle.rope(v, 17, theta), 230, theta), oracle.rope(v, 247, theta),
                               rtol=1e-9, atol=1e-12)


# --------------------------------------------------------------------- softmax

def test_softmax_properties():
    s = RNG.standard_normal(100) * 4
    p = oracle.softmax(s)
    assert math.isclose(p.sum(), 1.0, rel_tol=1e-14)
    np.testing.assert_allclose(oracle.softmax(s + 123.5), p, rtol=1e-12)
    big = oracle.softmax(np.array([1e4, 1e4 - 1.0, -1e4]))
    assert np.all(np.isfinite(big))
    np.testing.assert_allclose(big[:2], [1 / (1 + math.exp(-1)), 1 / (1 + math.exp(1))], rtol=1e-14)
    assert big[2] == 0.0
    a, b = 0.3, -1.7
    np.testing.assert_allclose(oracle.softmax([a, b]), [1 / (1 + math.exp(b - a)), 1 / (1 + math.exp(a - b))],
                               rtol=1e-15)


# ------------------------------------------------------------------- attention

def test_attention_single_position_returns_v():
    hd = 64
    q = RNG.standard_normal(hd)
    k = bf16_bits(RNG.standard_normal((1, hd)))
    v = bf16_bits(RNG.standard_normal((1, hd)))
    assert np.array_equal(oracle.attention_head(q, k, v), bf16_vals(v[0]))


def test_attention_two_positions_closed_form():
    hd = 4
    q = np.array([1.0, 0.5, -1.0, 2.0])
    k = bf16_bits([[1, 0, 0, 1], [0, 2, 1, 0]])
    v = bf16_bits([[1, 2, 3, 4], [-4, 0, 8, 1]])
    s0 = (1 + 2) / 2.0
    s1 = (1.0 - 1.0) / 2.0
    w0 = 1 / (1 + math.exp(s1 - s0))
    want = w0 * np.array([1, 2, 3, 4]) + (1 - w0) * np.array([-4, 0, 8, 1])
    np.testing.assert_allclose(oracle.attention_head(q, k, v), want, rtol=1e-14)


def test_attention_equal_keys_average_values():
    hd, ctx = 8, 9
    q = RNG.standard_normal(hd)
    k = np.tile(bf16_bits(RNG.standard_normal(hd)), (ctx, 1))
    v = bf16_bits(RNG.standard_normal((ctx, hd)))
    np.testing.assert_allclose(oracle.attention_head(q, k, v), bf16_vals(v).mean(axis=0), rtol=1e-13, atol=1e-15)


def test_silu_and_argmax():
    for x in (-3.0, -0.5, 0.0, 1.25, 8.0):
        assert math.isclose(oracle.silu(x), x / (1 + math.exp(-x)), rel_tol=1e-15, abs_tol=1e-300)
    assert oracle.argmax_f32([1.0, 3.0, 3.0, -2.0]) == (1, False)
    assert oracle.argmax_f32([1.0, float("nan"), 0.5]) == (0, True)
    # ties decided in float: these two differ only below float resolution
    assert oracle.argmax_f32([1.0, 1.0 + 1e-12]) == (0, False)


# ---------------------------------------------------------- whole decode step

def tiny_shape(**kw):
    d = dict(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn=96, vocab=50,
             rms_eps=1e-5, rope_theta=10000.0, tie_embeddings=False)
    d.update(kw)
    return synth.ModelShape(**d)


def as_t(bits):
    return torch.from_numpy(bf16_vals(bits))


def torch_causal_forward(m, tokens, mats=None):
    """Full causal forward over the whole sequence with torch fp64 library ops
    (F.rms_norm, F.scaled_dot_product_attention with is_causal and enable_gqa,
    F.silu, matmul).  K and V are rounded to bf16 (via float32, torch's
    rounding) after RoPE, as a bf16 cache holds them.  mats: fp64 tensors to
    use for the matrices instead of the model's bf16 ones (per kind a list
    per layer, and "lm_head")."""
    s = m["shape"]
    if mats is not None:
        def W(kind, l=None):
            return mats[kind] if l is None else mats[kind][l]
    else:
        def W(kind, l=None):
            if l is not None:
                return as_t(m[kind][l])
            return as_t(m["embed"] if m["lm_head"] is None else m["lm_head"])
    T, hd = len(tokens), s.head_dim
    x = as_t(m["embed"])[torch.as_tensor(tokens, dtype=torch.long)]
    pos = torch.arange(T, dtype=torch.float64)
    inv = torch.tensor([s.rope_theta ** (-(2.0 * i) / hd) for i in range(hd // 2)], dtype=torch.float64)
    ang = pos[:, None] * inv[None, :]
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rope(t):  # t [heads, T, hd]
        a, b = t[..., : hd // 2], t[..., hd // 2:]
        return torch.cat([a * cos - b * sin, b * cos + a * sin], dim=-1)

    def rb(t):
        return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)

    for l in range(s.n_layers):
        xn = F.rms_norm(x, (s.hidden,), as_t(m["attn_norm"][l]), eps=s.rms_eps)
        q = (xn @ W("wq", l).T).view(T, s.n_q_heads, hd).transpose(0, 1)
        k = (xn @ W("wk", l).T).view(T, s.n_kv_heads, hd).transpose(0, 1)
        v = (xn @ W("wv", l).T).view(T, s.n_kv_heads, hd).transpose(0, 1)
        q, k, v = rope(q), rb(rope(k)), rb(v)
        o = F.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True, enable_gqa=True)[0]
        x = x + o.transpose(0, 1).reshape(T, -1) @ W("wo", l).T
        xn = F.rms_norm(x, (s.hidden,), as_t(m["ffn_norm"][l]), eps=s.rms_eps)
        u = F.silu(xn @ W("w_gate", l).T) * (xn @ W("w_up", l).T)
        x = x + u @ W("w_down", l).T
    h = F.rms_norm(x, (s.hidden,), as_t(m["final_norm"]), eps=s.rms_eps)
    return (h @ W("lm_head").T).numpy(), h.numpy()


@pytest.mark.parametrize("kw", [dict(), dict(tie_embeddings=True), dict(n_kv_heads=4), dict(n_kv_heads=1)])
def test_decode_matches_torch_causal_forward(kw):
    s = tiny_shape(**kw)
    m = synth.make_model(s, seed=7, std=0.2, gains="normal")
    tokens = synth.uniform_tokens(12, s.vocab, 7, 99)
    want_logits, want_h = torch_causal_forward(m, tokens)
    o = oracle.OracleDecoder(m, max_seq=16)
    for p, t in enumerate(tokens):
        lg, h = o.step(int(t), p)
        np.testing.assert_allclose(lg, want_logits[p], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(h, want_h[p], rtol=1e-9, atol=1e-11)
    # slots above the last position are untouched
    assert not o.kcache[:, :, len(tokens):, :].any()


def test_gqa_equals_mha_with_repeated_kv():
    """q head h must read kv head h // (q_heads / kv_heads): a GQA model equals
    the MHA model whose K/V projections repeat each kv head for its q heads."""
    s = tiny_shape(n_q_heads=4, n_kv_heads=2)
    m = synth.make_model(s, seed=11, std=0.2)
    s2 = tiny_shape(n_q_heads=4, n_kv_heads=4)
    m2 = dict(m, shape=s2)
    hd = s.head_dim
    rep = lambda w: np.concatenate([w[(h // 2) * hd:(h // 2 + 1) * hd] for h in range(4)], axis=0)
    m2["wk"] = [rep(w) for w in m["wk"]]
    m2["wv"] = [rep(w) for w in m["wv"]]
    a, b = oracle.OracleDecoder(m, 8), oracle.OracleDecoder(m2, 8)
    for p, t in enumerate([3, 9, 27, 4, 4]):
        la, _ = a.step(t, p)
        lb, _ = b.step(t, p)
        np.testing.assert_allclose(la, lb, rtol=1e-12, atol=1e-14)


def _hand_model(E, W_lm=None, wq=None, wk=None, wv=None, wo=None, wg=None, wu=None, wd=None):
    """H=2, 1 layer, 1 q head / 1 kv head, head_dim 2, ffn 2; all gains 1."""
    V = len(E)
    s = synth.ModelShape(1, 2, 1, 1, 2, 2, V, 1e-5, 10000.0, W_lm is None)
    z = np.zeros((2, 2))
    f = lambda w: bf16_bits(z if w is None else w)
    ones = bf16_bits(np.ones(2))
    return {"shape": s, "embed": bf16_bits(E), "lm_head": None if W_lm is None else bf16_bits(W_lm),
            "final_norm": ones, "attn_norm": [ones], "ffn_norm": [ones], "wq": [f(wq)], "wk": [f(wk)],
            "wv": [f(wv)], "wo": [f(wo)], "w_gate": [f(wg)], "w_up": [f(wu)], "w_down": [f(wd)]}


def _rms(x, eps=1e-5):
    x = np.asarray(x, dtype=np.float64)
    return x / math.sqrt(float(np.mean(x * x)) + eps)


def test_brute_force_zeroed_blocks():
    E = [[3.0, 4.0], [1.0, -1.0], [0.5, 2.0], [-2.0, 0.25]]
    W_lm = [[1.0, 0.0], [0.0, 1.0], [1.0, 1.0], [-1.0, 0.5]]
    o = oracle.OracleDecoder(_hand_model(E, W_lm=W_lm), 4)
    for p, t in enumerate([0, 1, 2]):
        lg, h = o.step(t, p)
        np.testing.assert_allclose(h, _rms(E[t]), rtol=1e-15)
        np.testing.assert_allclose(lg, np.array(W_lm) @ _rms(E[t]), rtol=1e-15)


def test_brute_force_tied_zeroed_blocks_argmax():
    E = np.array([[3.0, 4.0], [1.0, -1.0], [0.5, 2.0], [-2.0, 0.25], [4.0, 4.0]])
    o = oracle.OracleDecoder(_hand_model(E), 4)
    for t in range(len(E)):
        lg, _ = o.step(t, 0)
        want = E @ _rms(E[t])
        np.testing.assert_allclose(lg, want, rtol=1e-15)
        assert oracle.argmax_f32(lg)[0] == int(np.argmax(want))


def test_brute_force_attention_adds_normed_value():
    """W_q = W_k = 0 (all scores 0: uniform attention), W_v = W_o = I, FFN off."""
    E = [[1.0, 1.0], [3.0, 4.0], [0.0, 1.0]]
    W_lm = [[1.0, 0.0], [0.0, 1.0], [1.0, -1.0]]
    I = np.eye(2)
    o = oracle.OracleDecoder(_hand_model(E, W_lm=W_lm, wv=I, wo=I), 4)
    # pos 0: the only value is bf16(RMSNorm(E[0])) = bf16(0.999995..) = 1.0
    v0 = bf16_vals(bf16_bits(_rms(E[0])))
    assert np.array_equal(v0, [1.0, 1.0])
    lg, h = o.step(0, 0)
    np.testing.assert_allclose(h, _rms(np.array(E[0]) + v0), rtol=1e-15)
    # pos 1: the uniform average of both cached values is added
    v1 = bf16_vals(bf16_bits(_rms(E[1])))
    lg, h = o.step(1, 1)
    np.testing.assert_allclose(h, _rms(np.array(E[1]) + (v0 + v1) / 2), rtol=1e-14)
    np.testing.assert_allclose(lg, np.array(W_lm) @ h, rtol=1e-14)


def test_brute_force_swiglu_branch():
    E = [[3.0, 4.0], [1.0, -2.0]]
    W_lm = [[1.0, 0.0], [0.0, 1.0]]
    wg, wu, wd = np.eye(2), np.array([[2.0, 0.0], [0.0, -1.0]]), np.array([[1.0, 1.0], [0.0, 1.0]])
    o = oracle.OracleDecoder(_hand_model(E, W_lm=W_lm, wg=wg, wu=wu, wd=wd), 4)
    silu = lambda a: a / (1 + math.exp(-a))
    for p, t in enumerate([0, 1]):
        x = np.array(E[t])
        xn = _rms(x)
        u = np.array([silu(xn[0]) * 2 * xn[0], silu(xn[1]) * -xn[1]])
        x2 = x + wd @ u
        lg, h = o.step(t, p)
        np.testing.assert_allclose(h, _rms(x2), rtol=1e-14)
        np.testing.assert_allclose(lg, _rms(x2), rtol=1e-14)


def test_kv_append_is_bf16_of_rotated_k():
    s = tiny_shape()
    m = synth.make_model(s, seed=5, std=0.3)
    o = oracle.OracleDecoder(m, 8)
    tokens = [7, 1, 30]
    for p, t in enumerate(tokens):
        o.step(t, p)
    # recompute layer 0's K/V at position 2 from its definition with torch ops
    x = as_t(m["embed"])[tokens[2]]
    xn = F.rms_norm(x, (s.hidden,), as_t(m["attn_norm"][0]), eps=s.rms_eps).numpy()
    k = as_t(m["wk"][0]).numpy() @ xn
    v = as_t(m["wv"][0]).numpy() @ xn
    for g in range(s.n_kv_heads):
        kr = oracle.rope(k[g * 16:(g + 1) * 16], 2, s.rope_theta)
        assert np.array_equal(o.kcache[0, g, 2], bf16_bits(kr))
        assert np.array_equal(o.vcache[0, g, 2], bf16_bits(v[g * 16:(g + 1) * 16]))


# ---------------------------------------------------------------- sampling
#
# The sampler draws from softmax(logits / T) by the Gumbel-max rule with
# SplitMix64 noise (cloud.baidu.com/article/9434380, section 5, steps 1 and 5;
# the rule and the generator are the reading taken where the page names only
# the temperature).  Pinned: the generator's output indexing against the
# generator stepped one output at a time and its widely reproduced first
# output for seed 0; the uniformity of U; the sampled frequencies against the
# softmax probabilities at two temperatures (a wrong sign of G, a missing log
# or a wrong temperature scale fails it); the greedy limits.

_GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1


def _stepped_splitmix64(seed, n):
    """The generator as published: add gamma to the state, output the mixed state."""
    out, st = [], seed
    for _ in range(n):
        st = (st + _GAMMA) & _M64
        z = st
        z ^= z >> 30
        z = (z * 0xBF58476D1CE4E5B9) & _M64
        z ^= z >> 27
        z = (z * 0x94D049BB133111EB) & _M64
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_output_indexing():
    for seed in (0, 1, 0xDEADBEEF, _M64):
        assert [oracle.splitmix64_output(seed, i) for i in range(24)] == _stepped_splitmix64(seed, 24)
    assert oracle.splitmix64_output(0, 0) == 0xE220A8397B1DCDAF   # the first output for seed 0
    # counter i = pos * 2^32 + v
    z = oracle.splitmix64_output(5, (3 << 32) | 7)
    assert oracle.uniform_f32(5, 3, 7) == ((z >> 41) + 0.5) / 2.0 ** 23   # exact in fp32
    # the extremes of U stay inside (0, 1) in fp32
    assert np.float32((0 + 0.5) / 2.0 ** 23) > 0 and np.float32(((1 << 23) - 1 + 0.5) / 2.0 ** 23) < 1


def test_uniform_noise_is_uniform_and_open():
    u = np.array([oracle.uniform_f32(123, p, v) for p in range(4) for v in range(5000)])
    assert 0.0 < u.min() and u.max() < 1.0
    counts, _ = np.histogram(u, bins=20, range=(0.0, 1.0))
    expect = len(u) / 20
    chi2 = float(np.sum((counts - expect) ** 2 / expect))
    assert chi2 < 43.8, chi2   # 19 degrees of freedom, p = 0.001


@pytest.mark.parametrize("temperature", [1.0, 0.5])
def test_gumbel_max_draws_follow_softmax(temperature):
    logits = np.array([0.5, -1.0, 2.0, 0.0, 1.2, -0.3])
    inv = float(np.float32(1.0 / temperature))
    n = 30000
    counts = np.zeros(len(logits))
    for k in range(n):
        tok, nf = oracle.sample_f32(logits, inv, 99, k)
        assert not nf
        counts[tok] += 1
    z = logits * inv
    prob = np.exp(z - z.max())
    prob /= prob.sum()
    chi2 = float(np.sum((counts - n * prob) ** 2 / (n * prob)))
    assert chi2 < 20.5, (chi2, counts / n, prob)   # 5 degrees of freedom, p = 0.001


def test_sampling_limits_and_special_values():
    rng = np.random.default_rng(4)
    logits = rng.normal(size=50)
    greedy = int(np.argmax(logits))
    for pos in range(20):
        assert oracle.sample_f32(logits, 0.0, 7, pos)[0] == greedy          # temperature <= 0: greedy
        assert oracle.sample_f32(logits, 1e6, 7, pos)[0] == greedy          # temperature -> 0
    dominant = logits.copy()
    dominant[17] += 60.0                                                    # P(any other) < 50 e^-60
    assert all(oracle.sample_f32(dominant, 1.0, 11, pos)[0] == 17 for pos in range(50))
    bad = logits.copy()
    bad[greedy] = np.nan
    tok, nf = oracle.sample_f32(bad, 1.0, 3, 0)
    assert nf and tok != greedy
    assert oracle.sample_f32(np.full(4, np.inf), 1.0, 3, 0) == (-1, True)   # no finite logit


# ---------------------------------------------------------------- top-p (nucleus) sampling

def _draw_counts(logits, inv, top_p, n, seed=77):
    counts = np.zeros(len(logits))
    for k in range(n):
        tok, nf = oracle.sample_topp_f32(logits, inv, top_p, seed, k)
        assert not nf
        counts[tok] += 1
    return counts


@pytest.mark.parametrize("temperature,top_p,expect", [
    # q = [0.5, 0.3, 0.15, 0.05]: mass strictly above each token 0, 0.5, 0.8, 0.95
    (1.0, 0.7, [0.5 / 0.8, 0.3 / 0.8, 0.0, 0.0]),
    (1.0, 0.81, [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95, 0.0]),
    # T = 0.5 squares the probabilities: q' = [0.25, 0.09, 0.0225, 0.0025] / 0.365, mass above
    # token 2 = 0.34 / 0.365 = 0.9315 >= 0.9 (untempered it would be 0.8 < 0.9 and token 2 kept)
    (0.5, 0.9, [0.25 / 0.34, 0.09 / 0.34, 0.0, 0.0]),
])
def test_topp_draws_follow_the_truncated_renormalised_softmax(temperature, top_p, expect):
    """Closed-form nucleus: logits ln q with q known, so the kept set and the
    renormalised distribution are worked out by hand (comments); 30 000 draws
    must match it (chi-square) and never leave the kept set."""
    logits = np.log(np.array([0.5, 0.3, 0.15, 0.05]))
    inv = float(np.float32(1.0 / temperature))
    n = 30000
    counts = _draw_counts(logits, inv, top_p, n)
    expect = np.array(expect)
    assert np.all(counts[expect == 0] == 0), counts
    kept = expect > 0
    chi2 = float(np.sum((counts[kept] - n * expect[kept]) ** 2 / (n * expect[kept])))
    assert chi2 < 13.8, (chi2, counts / n, expect)   # at most 2 degrees of freedom, p = 0.001


def test_topp_ties_and_limits():
    # two tokens tie for the top: each has no mass strictly above it, so both are kept
    logits = np.array([1.0, 1.0, 0.0, -5.0])
    counts = _draw_counts(logits, 1.0, 0.1, 20000)
    assert counts[2] == 0 and counts[3] == 0
    assert abs(counts[0] / 20000 - 0.5) < 0.02
    # top_p >= 1 keeps every token: the same draws as plain sampling
    rng = np.random.default_rng(6)
    lg = rng.normal(size=40)
    for pos in range(100):
        assert oracle.sample_topp_f32(lg, 0.8, 1.0, 5, pos)[0] == oracle.sample_f32(lg, 0.8, 5, pos)[0]
    # a tiny nucleus holds only the most probable token
    top = int(np.argmax(lg))
    assert all(oracle.sample_topp_f32(lg, 1.0, 1e-9, 5, pos)[0] == top for pos in range(50))
    # temperature <= 0 stays greedy whatever top_p is
    assert oracle.sample_topp_f32(lg, 0.0, 0.5, 5, 3)[0] == top
    # non-finite logits are skipped and flagged
    bad = lg.copy()
    bad[top] = np.nan
    tok, nf = oracle.sample_topp_f32(bad, 1.0, 0.9, 5, 0)
    assert nf and tok != top



# ---------------------------------------------------------------- weight-only INT8

def test_q8_quantizer_exact_cases_and_bound():
    """Rows that are integer multiples of a power-of-two step quantize exactly
    (the scale is max|w| / 127 and every code is the multiple); any row obeys
    |w - q s| <= s / 2 (plus the float rounding of w / s) with |q| <= 127 and
    the largest |w| at code +-127; a
    zero row gets scale 0 and codes 0; per-column scaling is the same on W^T."""
    k = np.array([[-127, -3, 0, 5, 127, 64], [1, -1, 2, -2, 0, 0], [0, 0, 0, 0, 0, 0]], dtype=np.float64)
    steps = np.array([2.0 ** -10, 2.0 ** -4, 1.0])
    w = (k * steps[:, None]).astype(np.float32)
    bits = (w.view(np.uint32) >> 16).astype(np.uint16)           # exact in bf16
    q, sc = oracle.quantize_q8(bits)
    assert np.array_equal(q[0], k[0].astype(np.int8))             # max|w| = 127 steps: scale = step
    assert sc[0] == np.float32(2.0 ** -10) and sc[2] == 0.0 and not q[2].any()
    assert np.array_equal(q[1], np.round(k[1] * 127 / 2).astype(np.int8))   # row 1: max 2 -> scale 2/127
    rng = np.random.default_rng(3)
    wr = synth.normal_bf16((17, 40), 9, 1, 0.0, 0.05)
    q, sc = oracle.quantize_q8(wr)
    vals = bf16_vals(wr)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    # the quotient w / s is rounded in float before the code is: |w/s - q| <= 1/2 + 128 * 2^-24
    bound = sc[:, None].astype(np.float64) * (0.5 + 128 * 2.0 ** -24)
    assert np.all(np.abs(vals - q * sc[:, None].astype(np.float64)) <= bound)
    assert np.all(np.abs(q[np.arange(17), np.argmax(np.abs(vals), axis=1)]) == 127)
    qc, scc = oracle.quantize_q8(wr, col_scaled=True)
    qt, sct = oracle.quantize_q8(np.ascontiguousarray(wr.T))
    assert np.array_equal(qc, qt.T) and np.array_equal(scc, sct)


def test_q8_gemv_equals_dequantized_matmul():
    rng = np.random.default_rng(5)
    wr = synth.normal_bf16((23, 31), 4, 2, 0.0, 0.1)
    x = rng.normal(size=31)
    for col in (False, True):
        q, sc = oracle.quantize_q8(wr, col_scaled=col)
        deq = q.astype(np.float64) * (sc[None, :] if col else sc[:, None]).astype(np.float64)
        np.testing.assert_allclose(oracle.gemv_q8(q, sc, x, col_scaled=col), deq @ x, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("kw", [dict(), dict(tie_embeddings=True)])
def test_q8_decode_matches_torch_causal_forward_on_dequantized_weights(kw):
    """The oracle's int8 decode step equals the torch fp64 causal forward run
    on the dequantized matrices (codes times their row scales, or column scales
    for w_down), at every position."""
    s = tiny_shape(**kw)
    m = synth.make_model(s, seed=8, std=0.2, gains="normal")
    q8 = oracle.quantize_model_q8(m)

    def deq(kind, pair):
        q, sc = pair
        return torch.from_numpy(q.astype(np.float64) * (sc[None, :] if kind == "w_down" else sc[:, None]))

    mats = {kind: [deq(kind, p) for p in q8[kind]] for kind in oracle.Q8_KINDS}
    mats["lm_head"] = deq("lm_head", q8["lm_head"])
    tokens = synth.uniform_tokens(10, s.vocab, 8, 98)
    want_logits, want_h = torch_causal_forward(m, tokens, mats)
    o = oracle.OracleDecoder(m, max_seq=16, q8=q8)
    for p, t in enumerate(tokens):
        lg, h = o.step(int(t), p)
        np.testing.assert_allclose(lg, want_logits[p], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(h, want_h[p], rtol=1e-9, atol=1e-11)


# ---------------------------------------------------------------- weight-only INT4

def test_q4_quantizer_exact_cases_and_bound():
    """The INT4 quantizer (symmetric absmax, 7 levels a side): rows that are
    integer multiples of a power-of-two step with max 7 steps come back exactly;
    a row of max 7 steps with half-step values puts them at exact ties, which go
    to the even code (2.5 -> 2, 3.5 -> 4, -0.5 -> 0, -1.5 -> -2); any row obeys |w - q s| <= s/2
    (plus the float rounding of w / s) with |q| <= 7 and the largest |w| at +-7;
    a zero row gets scale 0 and codes 0; per-column scaling is the same on W^T."""
    k = np.array([[-7, -3, 0, 5, 7, 1], [7, 2.5, 3.5, -0.5, -1.5, 0], [0, 0, 0, 0, 0, 0]], dtype=np.float64)
    steps = np.array([2.0 ** -6, 2.0 ** -4, 1.0])
    w = (k * steps[:, None]).astype(np.float32)
    bits = (w.view(np.uint32) >> 16).astype(np.uint16)           # exact in bf16
    q, sc = oracle.quantize_q4(bits)
    assert np.array_equal(q[0], k[0].astype(np.int8))             # max|w| = 7 steps: scale = step
    assert sc[0] == np.float32(2.0 ** -6) and sc[2] == 0.0 and not q[2].any()
    assert sc[1] == np.float32(2.0 ** -4)
    assert np.array_equal(q[1], np.array([7, 2, 4, 0, -2, 0], dtype=np.int8))    # ties to even
    wr = synth.normal_bf16((19, 48), 9, 3, 0.0, 0.05)
    q, sc = oracle.quantize_q4(wr)
    vals = bf16_vals(wr)
    assert np.all(np.abs(q.astype(np.int32)) <= 7) and len(np.unique(q)) == 15
    bound = sc[:, None].astype(np.float64) * (0.5 + 8 * 2.0 ** -24)
    assert np.all(np.abs(vals - q * sc[:, None].astype(np.float64)) <= bound)
    assert np.all(np.abs(q[np.arange(19), np.argmax(np.abs(vals), axis=1)]) == 7)
    qc, scc = oracle.quantize_q4(wr, col_scaled=True)
    qt, sct = oracle.quantize_q4(np.ascontiguousarray(wr.T))
    assert np.array_equal(qc, qt.T) and np.array_equal(scc, sct)


def test_q4_codes_are_q8_codes_of_a_coarser_grid():
    """Brute force over every bf16 value in [-1, 1] against a row maximum of 1:
    the INT4 code of w is the nearest integer (ties to even) to w * 7, the
    closed form of absmax with 7 levels, computed here in float like the
    quantizer's own division."""
    u = np.arange(0x0000, 0x3F81, dtype=np.uint32)          # +0 .. 1.0 in bf16
    mags = (u << 16).view(np.float32)
    vals = np.concatenate([mags, -mags])
    bits = ((vals.view(np.uint32) >> 16).astype(np.uint16))
    row = np.concatenate([bits, np.array([0x3F80], dtype=np.uint16)])[None, :]   # max|w| = 1 exactly
    q, sc = oracle.quantize_q4(row)
    s = np.float32(1.0) / np.float32(7.0)
    assert sc[0] == s
    want = np.rint(np.concatenate([vals, [1.0]]).astype(np.float32) / s).clip(-7, 7)
    assert np.array_equal(q[0].astype(np.float32), want)


@pytest.mark.parametrize("kw", [dict(), dict(tie_embeddings=True)])
def test_q4_decode_matches_torch_causal_forward_on_dequantized_weights(kw):
    """The oracle's int4 decode step equals the torch fp64 causal forward run
    on the dequantized matrices (codes times their row scales, or column scales
    for w_down), at every position."""
    s = tiny_shape(**kw)
    m = synth.make_model(s, seed=18, std=0.2, gains="normal")
    q4 = oracle.quantize_model_q4(m)
    assert all(np.abs(q).max() <= 7 for kind in oracle.Q8_KINDS for q, _ in q4[kind])

    def deq(kind, pair):
        q, sc = pair
        return torch.from_numpy(q.astype(np.float64) * (sc[None, :] if kind == "w_down" else sc[:, None]))

    mats = {kind: [deq(kind, p) for p in q4[kind]] for kind in oracle.Q8_KINDS}
    mats["lm_head"] = deq("lm_head", q4["lm_head"])
    tokens = synth.uniform_tokens(10, s.vocab, 9, 98)
    want_logits, want_h = torch_causal_forward(m, tokens, mats)
    o = oracle.OracleDecoder(m, max_seq=16, q8=q4)
    for p, t in enumerate(tokens):
        lg, h = o.step(int(t), p)
        np.testing.assert_allclose(lg, want_logits[p], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(h, want_h[p], rtol=1e-9, atol=1e-11)
