"""GPU decode megakernel vs the CPU oracle, through the C ABI.

Small shapes run every step of their workload teacher-forced; they span several
tiles per CTA, ragged last tiles (FFN slice, vocab, O rows), multi-block KV
chunks, odd CTAs-per-group counts and both GQA ratios.  The five benchmark
workloads run at full size and full length in the launch configuration the
benchmark uses, every step teacher-forced against the oracle, with the 99%
greedy-agreement bar enforced.
"""
import numpy as np
import pytest

import oracle
import synth
from decode_megakernel_05_gb300 import Decoder, mk
from tests.parity import Report, run_teacher_forced

pytestmark = pytest.mark.gpu


def make(shape, seed, max_seq, gains="ones", std=0.02, tuning=None, perop=False):
    m = synth.make_model(shape, seed, std=std, gains=gains)
    return m, Decoder(m, max_seq, tuning=tuning, perop=perop), oracle.OracleDecoder(m, max_seq)


def test_tiny_workload_teacher_forced():
    w = synth.WORKLOADS["tiny"]
    m, dec, orc = make(w.shape, w.seed_weights, w.max_seq())
    prompt = synth.make_prompt(w)
    rep = run_teacher_forced(dec, orc, prompt, 0, w.prompt_len + w.decode - 1)
    print("workload tiny", rep.summary())
    rep.check(workload=True)
    # K/V appended by the fused kernel equal the oracle's bf16 cache (up to a rounding flip)
    for l in range(w.shape.n_layers):
        k, v = dec.get_kv(l, 0, rep.steps)
        for got, ref in ((k, orc.kcache[l, :, :rep.steps]), (v, orc.vcache[l, :, :rep.steps])):
            g32, r32 = synth.bf16_to_f32(got), synth.bf16_to_f32(ref)
            assert np.mean(got == ref) > 0.97
            assert np.max(np.abs(g32 - r32)) <= 2 ** -7 * np.max(np.abs(r32))
    dec.close()


@pytest.mark.parametrize("tied,gains", [(True, "normal"), (False, "normal")])
def test_tiny_variants(tied, gains):
    s = synth.ModelShape(2, 256, 4, 2, 64, 688, 1024, 1e-5, 10000.0, tied)
    m, dec, orc = make(s, 17, 128, gains=gains, std=0.05)
    toks = synth.uniform_tokens(20, s.vocab, 17, 5)
    rep = run_teacher_forced(dec, orc, toks, 0, 40)
    print(rep.summary())
    rep.check()
    dec.close()


MID = synth.ModelShape(2, 512, 8, 2, 64, 1000, 5003, 1e-5, 10000.0, False)


@pytest.mark.parametrize("grid,prefill", [(0, 0), (14, 0), (2, 700), (6, 300)])
def test_mid_shape_ragged(grid, prefill):
    """H=512, G=4, F=1000 (ragged FFN slices), V=5003 (ragged LM rows); grid 2
    and 6 put one and three CTAs in each KV group, so a CTA walks several KV
    blocks (online softmax across blocks)."""
    tun = mk.tuning(grid_ctas=grid) if grid else None
    m, dec, orc = make(MID, 23, 1024, gains="normal", std=0.04, tuning=tun)
    if prefill:
        ks, vs = synth.make_kv(MID, prefill, 29)
        dec.set_kv(ks, vs, prefill)
        orc.set_kv(ks, vs, prefill)
    toks = synth.uniform_tokens(8, MID.vocab, 23, 7)
    rep = run_teacher_forced(dec, orc, toks, prefill, 24)
    print(rep.summary())
    rep.check()
    dec.close()


@pytest.mark.parametrize("grid,prefill,build", [(0, 5001, 2), (6, 3000, 2), (6, 3000, 1), (0, 0, 2), (14, 37, 2),
                                               (14, 37, 1)])
def test_long_context_build(grid, prefill, build):
    """H=512, G=4 has a build whose attention runs on the tensor cores (build 2)
    beside the lane-parallel one (build 1); both read the K/V rows
    chunk-permuted in the cache.  A 5001-position prefill on the full grid
    (ragged per-CTA chunks) and 3000 positions on 3 CTAs per KV group (each CTA
    walks about a thousand positions, many KV blocks); decoding from position 0
    (blocks of the current row alone, 16-position chunks mostly past the end)
    and a 37-position prefill on 7 CTAs per group (a few positions per CTA).
    The K/V rows the kernel appends read back (through the permuted layout) as
    the oracle's."""
    tun = mk.tuning(grid_ctas=grid) if grid else None
    m, dec, orc = make(MID, 47, 8192, gains="normal", std=0.04, tuning=tun)
    assert dec.info.attn_tc == 1
    dec.set_debug(mk.MK_DBG_ATTN_BUILD, build)
    if prefill:
        ks, vs = synth.make_kv(MID, prefill, 53)
        dec.set_kv(ks, vs, prefill)
        orc.set_kv(ks, vs, prefill)
    steps = 8 if prefill > 1000 else 20
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, MID.vocab, 47, 3), prefill, steps)
    print(rep.summary())
    rep.check()
    for l in range(MID.n_layers):
        k, v = dec.get_kv(l, prefill, rep.steps)
        for got, ref in ((k, orc.kcache[l, :, prefill:prefill + rep.steps]),
                         (v, orc.vcache[l, :, prefill:prefill + rep.steps])):
            g32, r32 = synth.bf16_to_f32(got), synth.bf16_to_f32(ref)
            assert np.mean(got == ref) > 0.97
            assert np.max(np.abs(g32 - r32)) <= 2 ** -7 * np.max(np.abs(r32))
    dec.close()


def test_attention_build_switch_by_context():
    """By default a step runs the tensor-core attention build once the context
    gives every CTA attn_tc_min_ctx / CTAs-per-group positions: with 3 per CTA on
    7 CTAs per group the switch comes at context 21, inside one teacher-forced
    run from position 0, and parity holds on both sides of it."""
    m, dec, orc = make(MID, 71, 8192, gains="normal", std=0.04, tuning=mk.tuning(grid_ctas=14))
    dec.set_debug(mk.MK_DBG_ATTN_CTAS, 7)   # all 7 CTAs of a group attend at every context
    dec.set_debug(mk.MK_DBG_ATTN_TC_MIN, 3)
    info = mk.mk_get_info(dec.ctx)
    assert info.attn_tc == 1 and info.attn_tc_min_ctx == 21
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, MID.vocab, 71, 3), 0, 40)
    print(rep.summary())
    rep.check()
    dec.close()


@pytest.mark.parametrize("grid,prefill,ctas,build", [(0, 300, 1, 2), (0, 300, 2, 2), (0, 300, 5, 2), (0, 300, 76, 2),
                                                     (14, 900, 3, 2), (14, 900, 3, 1), (0, 40, 1, 1), (14, 0, 4, 2)])
def test_attention_split_forced(grid, prefill, ctas, build):
    """The length-adaptive split: the first `ctas` CTAs of each KV group run
    the attention (the others go from the QKV to the combine), forced at 1 ..
    all 76 CTAs per group of the full grid and at 3 of 7, with the tensor-core
    build (2) and the lane-parallel one (1); decoding from position 0 with
    more attention CTAs than positions gives CTAs with empty shares."""
    tun = mk.tuning(grid_ctas=grid) if grid else None
    m, dec, orc = make(MID, 79, 2048, gains="normal", std=0.04, tuning=tun)
    dec.set_debug(mk.MK_DBG_ATTN_BUILD, build)
    dec.set_debug(mk.MK_DBG_ATTN_CTAS, ctas)
    if prefill:
        ks, vs = synth.make_kv(MID, prefill, 83)
        dec.set_kv(ks, vs, prefill)
        orc.set_kv(ks, vs, prefill)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, MID.vocab, 79, 3), prefill, 10)
    print(grid, prefill, ctas, build, rep.summary())
    rep.check()
    dec.close()


def test_attention_split_grows_with_context():
    """By default a step at context ctx runs its attention on
    ceil(ctx / attn_pos_per_cta) CTAs per KV group: with 7 positions per CTA
    the count grows from 1 to 6 inside one run from position 0, and from 1 to
    3 on the hd=128 shape (both on the tensor-core build)."""
    m, dec, orc = make(MID, 89, 256, gains="normal", std=0.04, tuning=mk.tuning(grid_ctas=14))
    assert dec.info.attn_pos_per_cta > 0
    dec.set_debug(mk.MK_DBG_ATTN_POS_PER_CTA, 7)
    assert mk.mk_get_info(dec.ctx).attn_pos_per_cta == 7
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, MID.vocab, 89, 3), 0, 40)
    print(rep.summary())
    rep.check()
    dec.close()
    s = synth.ModelShape(2, 1024, 8, 2, 128, 1536, 4099, 1e-5, 500000.0, False)
    m, dec, orc = make(s, 97, 256, gains="normal", std=0.03, tuning=mk.tuning(grid_ctas=6))
    dec.set_debug(mk.MK_DBG_ATTN_POS_PER_CTA, 6)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, s.vocab, 97, 3), 0, 16)
    print(rep.summary())
    rep.check()
    dec.close()


def test_decode_up_to_the_last_cache_slot():
    """max_seq = 40: forty teacher-forced steps from position 0 end at the last
    cache slot (pos = max_seq - 1) on the tensor-core build; position max_seq
    is refused."""
    m, dec, orc = make(MID, 73, 40, gains="normal", std=0.04)
    assert dec.info.attn_tc == 1
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, MID.vocab, 73, 3), 0, 40)
    print(rep.summary())
    rep.check()
    assert mk.load().mk_decode_step(dec.ctx, 1, 40, None, dec.stream) == mk.MK_ERR_INVALID_ARG
    assert dec.status() == mk.MK_OK
    dec.close()


def test_kv_rows_round_trip_long_context():
    """set_kv / get_kv hide the long-context build's chunk-permuted rows: a
    window at an odd offset reads back bit for bit."""
    m = synth.make_model(MID, 5, std=0.04)
    dec = Decoder(m, 8192)
    assert dec.info.attn_tc == 1
    ks, vs = synth.make_kv(MID, 301, 7)
    dec.set_kv(ks, vs, 301)
    for l in range(MID.n_layers):
        k, v = dec.get_kv(l, 13, 251)
        assert np.array_equal(k, ks[l][:, 13:264]) and np.array_equal(v, vs[l][:, 13:264])
    dec.close()


@pytest.mark.parametrize("grid,build", [(0, 1), (0, 2), (6, 1), (6, 2)])
def test_head_dim_128_shape(grid, build):
    """hd=128, G=4 (the 8B head layout, chunk-permuted cache rows), both
    attention builds (1: lane-parallel, 2: tensor cores, four warps per
    16-position chunk with 32 dims of O each): 200 pre-filled positions spread
    over the full grid and over 3 CTAs per KV group (two 128-row blocks per
    CTA)."""
    s = synth.ModelShape(2, 1024, 8, 2, 128, 1536, 4099, 1e-5, 500000.0, False)
    tun = mk.tuning(grid_ctas=grid) if grid else None
    m, dec, orc = make(s, 31, 512, gains="normal", std=0.03, tuning=tun)
    assert dec.info.attn_tc == 1
    dec.set_debug(mk.MK_DBG_ATTN_BUILD, build)
    ks, vs = synth.make_kv(s, 200, 37)
    dec.set_kv(ks, vs, 200)
    orc.set_kv(ks, vs, 200)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, s.vocab, 31, 3), 200, 12)
    print(rep.summary())
    rep.check()
    dec.close()


def test_greedy_generate_matches_oracle_tokens():
    """mk_generate_greedy (device-side token feedback, host prompt in / tokens out)
    reproduces the oracle's own greedy continuation of the tiny workload."""
    w = synth.WORKLOADS["tiny"]
    m, dec, orc = make(w.shape, w.seed_weights, w.max_seq())
    prompt = synth.make_prompt(w)
    rc, out = dec.generate_greedy(prompt, 0, w.decode)
    assert rc == 0
    tok, want = None, []
    for p in range(w.prompt_len + w.decode - 1):
        t_in = int(prompt[p]) if p < w.prompt_len else tok
        lg, _ = orc.step(t_in, p)
        tok, _ = oracle.argmax_f32(lg)
        if p >= w.prompt_len - 1:
            want.append(tok)
    assert list(out) == want
    dec.close()


def test_perop_baseline_matches_oracle():
    w = synth.WORKLOADS["tiny"]
    m, dec, orc = make(w.shape, w.seed_weights, w.max_seq(), perop=True)
    prompt = synth.make_prompt(w)
    rep = run_teacher_forced(dec, orc, prompt, 0, 20, perop=True)
    print(rep.summary())
    rep.check()
    n = dec.step_perop(1, 20)
    assert n == 9 * w.shape.n_layers + 5
    dec.close()


def test_perop_baseline_long_context_layout():
    """The per-operator path appends to and reads the cache in the long-context
    build's chunk-permuted layout, after a prefill through set_kv."""
    m, dec, orc = make(MID, 61, 8192, gains="normal", std=0.04, perop=True)
    assert dec.info.attn_tc == 1
    ks, vs = synth.make_kv(MID, 45, 67)
    dec.set_kv(ks, vs, 45)
    orc.set_kv(ks, vs, 45)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, MID.vocab, 61, 3), 45, 12, perop=True)
    print(rep.summary())
    rep.check()
    dec.close()


# ------------------------------------------------------------ full-size workloads

def _full(name):
    """The whole workload, teacher-forced at every step: the 1B prompt run
    (512 tokens from an empty cache, positions 0..511) and its 256 decode
    steps (positions 512..767); or, on a pre-filled cache of P positions, the
    seeded first token at P and the decode steps after it (128 at 2048 and at
    4096 on the 8B shape, 64 at 32768)."""
    w = synth.WORKLOADS[name]
    m, dec, orc = make(w.shape, w.seed_weights, w.max_seq())
    del m
    if w.prefill:
        ks, vs = synth.make_kv(w.shape, w.prefill, w.seed_kv)
        dec.set_kv(ks, vs, w.prefill)
        orc.set_kv(ks, vs, w.prefill)
        del ks, vs
        toks, start, n_steps = [synth.make_first_token(w)], w.prefill, w.decode
    else:
        toks, start, n_steps = synth.make_prompt(w), 0, w.prompt_len + w.decode
    rep = run_teacher_forced(dec, orc, toks, start, n_steps)
    print("workload", name, rep.summary(), "grid", dec.info.grid_ctas, "stages", dec.info.ring_stages)
    rep.check(workload=True)
    dec.close()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["1b", "1b-2k", "1b-32k", "8b-4k"])
def test_full_size_workloads_full_length(name):
    _full(name)


WIDE = synth.ModelShape(2, 2048, 32, 8, 64, 2304, 4099, 1e-5, 500000.0, False)


@pytest.mark.parametrize("shape,seed", [(WIDE, 41), (MID, 43)], ids=["H2048", "H512"])
def test_hidden_width_gemv(shape, seed):
    """The hidden-width GEMVs (QKV, gate/up: column blocks with activations in
    registers, transposed butterfly, groups taking turns on tiles) on the
    1B-like width H=2048 and on H=512, with ragged FFN slices and LM rows."""
    m, dec, orc = make(shape, seed, 256, gains="normal", std=0.03)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(6, shape.vocab, seed, 3), 0, 10)
    print(shape.hidden, rep.summary())
    rep.check()
    dec.close()


# ------------------------------------------------------------ sampling and stop

def _oracle_keys(lg_ref, inv, seed, pos):
    """The oracle's sampling keys fmaf(logit, 1/T, G) for every token (for near-tie checks)."""
    g = np.array([oracle.gumbel_f32(seed, pos, v) for v in range(len(lg_ref))], dtype=np.float32)
    return lg_ref.astype(np.float32) * np.float32(inv) + g


@pytest.mark.parametrize("temperature", [0.7, 1.3])
def test_sampling_matches_oracle(temperature):
    """Teacher-forced sampled steps on the H=512 shape (V = 5003): the fused
    Gumbel-max choice equals the oracle's from its own logits, except where
    the oracle's top two keys are within the logit error (a near tie)."""
    m, dec, orc = make(MID, 61, 256, gains="normal", std=0.04)
    inv = float(np.float32(1.0 / temperature))
    seed = 0x5EED0000 + int(temperature * 10)
    tok, agree, steps = 5, 0, 24
    for pos in range(steps):
        lg_ref, _ = orc.step(tok, pos)
        dec.step_sample(tok, pos, temperature, seed, logits=True)
        lg = dec.logits.cpu().numpy().astype(np.float64)
        got = dec.get_argmax()
        want, nf = oracle.sample_f32(lg_ref, inv, seed, pos)
        assert not nf
        dl = float(np.max(np.abs(lg - lg_ref)))
        assert dl <= 5e-2
        if got == want:
            agree += 1
        else:
            keys = np.sort(_oracle_keys(lg_ref, inv, seed, pos))
            assert keys[-1] - keys[-2] <= 2 * dl * inv + 1e-5, (pos, got, want)
        tok = want
    assert agree >= steps - 1, agree
    assert dec.status() == 0
    dec.close()


def test_generate_with_sampling_and_stop_token():
    """mk_generate: the sampled sequence equals the oracle's (each fed its own
    previous token); with a stop token it ends right after the first one
    (-1 after it, later launches do nothing), and the next call runs again."""
    s = synth.ModelShape(2, 256, 4, 2, 64, 688, 1024, 1e-5, 10000.0, False)
    m, dec, orc = make(s, 71, 128, gains="normal", std=0.05)
    prompt = synth.uniform_tokens(6, s.vocab, 71, 9)
    n_new, temperature, seed = 16, 0.9, 1234
    inv = float(np.float32(1.0 / temperature))

    def oracle_generate():
        out, tok = [], 0
        for k in range(len(prompt) + n_new - 1):
            tok = int(prompt[k]) if k < len(prompt) else out[-1]
            lg_ref, _ = orc.step(tok, k)
            if k >= len(prompt) - 1:
                out.append(oracle.sample_f32(lg_ref, inv, seed, k)[0])
        return out

    want = oracle_generate()
    rc, got, n = dec.generate(prompt, 0, n_new, temperature, seed)
    assert rc == 0 and n == n_new
    assert list(got) == want
    # stop at the first generated token that has not appeared before it (index >= 2)
    j = next(i for i in range(2, n_new) if want[i] not in want[:i])
    rc, got, n = dec.generate(prompt, 0, n_new, temperature, seed, eos_id=want[j])
    assert rc == 0 and n == j + 1
    assert list(got[:j + 1]) == want[:j + 1] and all(t == -1 for t in got[j + 1:])
    # a full run again: the stop flag is reset by every call
    rc, got, n = dec.generate(prompt, 0, n_new, temperature, seed)
    assert rc == 0 and n == n_new and list(got) == want
    dec.close()


def _nucleus_bounds(lg_ref, inv, top_p, dl):
    """Loose and strict nucleus of the oracle's logits: the GPU decides membership
    from logits within dl of the oracle's (x within dl/T) with fp32 sums, so near
    the boundary either decision is valid.  Returns (loose set, strict set)."""
    x = lg_ref.astype(np.float32) * np.float32(inv)
    e = np.exp(x.astype(np.float64) - float(x.max()))
    z = e.sum()
    order = np.argsort(-x, kind="stable")
    xs, es = x[order], e[order]
    above = np.zeros(len(x))
    acc, k = 0.0, 0
    while k < len(xs):
        j = k
        while j < len(xs) and xs[j] == xs[k]:
            j += 1
        above[order[k:j]] = acc
        acc += es[k:j].sum()
        k = j
    slack = top_p * (np.exp(2.0 * dl * inv) - 1.0) + 1e-4
    return set(np.nonzero(above < (top_p + slack) * z)[0]), set(np.nonzero(above < (top_p - slack) * z)[0])


@pytest.mark.parametrize("temperature,top_p", [(1.0, 0.9), (0.2, 0.5)])
def test_topp_sampling_matches_oracle(temperature, top_p):
    """Top-p inside the launch (H=512 shape, V = 5003): the fused choice equals
    the oracle's nucleus sample from its own logits, except where the nucleus
    boundary or the top two keys sit within the logit error (both choices
    valid); the chosen token is always inside the loosened nucleus and no key
    of the tightened nucleus beats it."""
    m, dec, orc = make(MID, 67, 256, gains="normal", std=0.04)
    dec.set_top_p(top_p)
    inv = float(np.float32(1.0 / temperature))
    seed = 0x70B0 + int(100 * top_p)
    tok, agree, steps = 11, 0, 24
    for pos in range(steps):
        dec.step_sample(tok, pos, temperature, seed, logits=True)
        lg_ref, _ = orc.step(tok, pos)
        lg = dec.logits.cpu().numpy().astype(np.float64)
        got = dec.get_argmax()
        want, nf = oracle.sample_topp_f32(lg_ref, inv, top_p, seed, pos)
        assert not nf
        dl = float(np.max(np.abs(lg - lg_ref)))
        assert dl <= 5e-2
        if got == want:
            agree += 1
        else:
            loose, strict = _nucleus_bounds(lg_ref, inv, top_p, dl)
            keys = _oracle_keys(lg_ref, inv, seed, pos)
            assert got in loose, (pos, got, want)
            assert keys[got] >= max(keys[v] for v in strict) - (2 * dl * inv + 1e-5), (pos, got, want)
        tok = want
    assert agree >= steps - 2, agree
    assert dec.status() == 0
    dec.close()


def test_topp_tiny_nucleus_then_back_to_plain_sampling():
    """A nucleus of 1e-6 of the mass holds only the most probable token, so the
    sampled token is the argmax of the step's own logits; setting top_p back to
    1 then samples as without it (the oracle's plain Gumbel-max choice, near
    ties allowed); out-of-range values are refused."""
    m, dec, orc = make(MID, 71, 64, gains="normal", std=0.04)
    inv = float(np.float32(1.0 / 0.8))
    dec.set_top_p(1e-6)
    for pos in range(6):
        lg = dec.step_sample(5 + pos, pos, 0.8, 4242, logits=True).cpu().numpy()
        orc.step(5 + pos, pos)
        assert dec.get_argmax() == int(np.argmax(lg))
    dec.set_top_p(1.0)
    for pos in range(6, 12):
        lg = dec.step_sample(5 + pos, pos, 0.8, 4242, logits=True).cpu().numpy().astype(np.float64)
        lg_ref, _ = orc.step(5 + pos, pos)
        got, (want, _) = dec.get_argmax(), oracle.sample_f32(lg_ref, inv, 4242, pos)
        if got != want:
            dl = float(np.max(np.abs(lg - lg_ref)))
            keys = np.sort(_oracle_keys(lg_ref, inv, 4242, pos))
            assert keys[-1] - keys[-2] <= 2 * dl * inv + 1e-5, (pos, got, want)
    lib = mk.load()
    for bad in (0.0, -0.5, 1.5, float("nan")):
        assert lib.mk_set_top_p(dec.ctx, bad) == mk.MK_ERR_INVALID_ARG
    assert dec.status() == 0
    dec.close()
