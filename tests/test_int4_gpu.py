"""Weight-only INT4 streams (mk_tuning.weight_int4) against the oracle's int4 model.

The library quantizes every matrix on the device when it loads the weights
(symmetric absmax with 7 levels a side: fp32 scale max|w| / 7 per output row,
per input column for W_down, codes in [-7, 7] rounded half to even from a
float quotient) and packs two codes a byte; the oracle quantizes the same
bf16 matrices on the CPU (oracle.quantize_q4).  Both decide each code in the
same float arithmetic, so

  - the arena, read back and unpacked here from the documented nibble format
    by code of its own, holds exactly the oracle's codes and scales,
  - the decode step meets the bf16 path's tolerances against the oracle's
    fp64 forward on the dequantized matrices (tests/parity.py).

Shapes cover the three int4 builds, as for int8: (head_dim 64, 2 query heads
per KV head, hidden 256), the 1B layout (64, 4, 2048, standard and
long-context attention) and the 8B layout (128, 4, 4096).
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from decode_megakernel_05_gb300 import Decoder, mk
from tests.parity import run_teacher_forced
from tests.test_int8_gpu import SLOT, TINY, WIDE, WIDE_HD128, decode_arena_q8, read_arena

pytestmark = pytest.mark.gpu


def make_q4(shape, seed, max_seq, gains="normal", std=0.03, tuning=None):
    m = synth.make_model(shape, seed, std=std, gains=gains)
    q4 = oracle.quantize_model_q4(m)
    dec = Decoder(m, max_seq, tuning=tuning, int4=True)
    return m, q4, dec, oracle.OracleDecoder(m, max_seq, q8=q4)


@pytest.mark.parametrize("shape,grid,tied", [(TINY, 0, False), (TINY, 2, True), (WIDE, 0, False),
                                             (WIDE, 24, True), (WIDE_HD128, 0, False)],
                         ids=["tiny", "tiny-g2-tied", "wide", "wide-g24-tied", "hd128"])
def test_arena_holds_the_oracle_int4_codes_and_scales(shape, grid, tied):
    shape = dataclasses.replace(shape, tie_embeddings=tied)
    tun = mk.tuning(grid_ctas=grid) if grid else None
    m = synth.make_model(shape, 6, std=0.03, gains="normal")
    q4 = oracle.quantize_model_q4(m)
    dec = Decoder(m, 64, tuning=tun, int4=True)
    info = dec.info
    # int4 streams default to 24 KB tiles in 8 ring slots (the same 192 KB ring)
    assert info.weight_int4 == 1 and info.weight_int8 == 0
    assert info.slot_bytes == 3 * SLOT // 4 and info.ring_stages == 8
    arena = read_arena(dec)
    codes, scales, lm_q, lm_s, cover, end = decode_arena_q8(arena, shape, info.grid_ctas, bits=4,
                                                            slot=info.slot_bytes)
    assert end == info.arena_bytes
    for name in oracle.Q8_KINDS:
        for l in range(shape.n_layers):
            rq, rs = q4[name][l]
            assert np.array_equal(codes[name][l], rq), (name, l)
            assert np.array_equal(scales[name][l].view(np.uint32), rs.view(np.uint32)), (name, l)
    rq, rs = q4["lm_head"]
    assert np.array_equal(lm_q, rq)
    assert np.array_equal(lm_s.view(np.uint32), rs.view(np.uint32))
    # every code byte sits in exactly one place, two codes each
    assert cover.max() == 1
    assert 2 * int(cover.sum()) == sum(q.size for k in oracle.Q8_KINDS for q, _ in q4[k]) + rq.size
    # the stream is the packed codes plus scales and padding: about a quarter of the bf16 arena
    bf = mk.mk_arena_bytes(mk.config_from_shape(shape, 64), tun, info.grid_ctas)
    assert 0.25 * bf < info.arena_bytes < 0.31 * bf
    # and the step's weight bytes: matrices at half a byte a weight, one fp32 scale per row / column
    s = shape
    qd, kvd = s.n_q_heads * s.head_dim, s.n_kv_heads * s.head_dim
    mat = s.n_layers * (qd * s.hidden + 2 * kvd * s.hidden + s.hidden * qd + 3 * s.ffn * s.hidden) + \
        s.vocab * s.hidden
    scl = 4 * (s.n_layers * (qd + 2 * kvd + s.hidden + 3 * s.ffn) + s.vocab)
    assert info.weight_bytes_per_token == mat // 2 + scl + 2 * (s.n_layers * 2 * s.hidden + 2 * s.hidden)
    dec.close()


def test_tiny_workload_int4():
    w = synth.WORKLOADS["tiny"]
    m, q4, dec, orc = make_q4(w.shape, w.seed_weights, w.max_seq(), gains="ones", std=0.02)
    rep = run_teacher_forced(dec, orc, synth.make_prompt(w), 0, w.prompt_len + w.decode - 1)
    print("tiny int4", rep.summary())
    rep.check(workload=True)
    dec.close()


@pytest.mark.parametrize("grid,tied,prefill", [(2, True, 0), (6, False, 90)])
def test_tiny_int4_multi_tile(grid, tied, prefill):
    """Grid 2 (one CTA per KV group): 512 LM rows, 344 FFN columns and the whole
    QKV block per CTA, so every phase walks several int4 tiles with a ragged
    last one; grid 6 after a 90-position prefill."""
    shape = dataclasses.replace(TINY, tie_embeddings=tied)
    tun = mk.tuning(grid_ctas=grid)
    m, q4, dec, orc = make_q4(shape, 21 + grid, 256, tuning=tun)
    if prefill:
        ks, vs = synth.make_kv(shape, prefill, 23)
        dec.set_kv(ks, vs, prefill)
        orc.set_kv(ks, vs, prefill)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(6, shape.vocab, grid, 5), prefill, 24)
    print(grid, tied, rep.summary())
    rep.check()
    dec.close()


@pytest.mark.parametrize("prefill,build,slot_kib", [(0, 0, 0), (3000, 1, 0), (3000, 2, 0), (0, 0, 32)])
def test_wide_int4_both_attention_builds(prefill, build, slot_kib):
    """The 1B layout on the int4 stream: the standard build, and after a
    3000-position prefill both attention builds (lane-parallel, tensor cores);
    also with 32 KB tiles (30 rows of 2048 codes, a warp's share of a tile
    in 8 passes of four rows) instead of the default 24 KB."""
    tun = mk.tuning(ring_stages=6, slot_kib=32) if slot_kib else None
    m, q4, dec, orc = make_q4(WIDE, 33, 4096, tuning=tun)
    assert dec.info.attn_tc == 1
    dec.set_debug(mk.MK_DBG_ATTN_BUILD, build)
    if prefill:
        ks, vs = synth.make_kv(WIDE, prefill, 39)
        dec.set_kv(ks, vs, prefill)
        orc.set_kv(ks, vs, prefill)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, WIDE.vocab, 33, 3), prefill, 12)
    print(prefill, build, rep.summary())
    rep.check()
    dec.close()


@pytest.mark.parametrize("build", [0, 1, 2])
def test_hd128_int4(build):
    """The 8B layer width and head layout on the int4 stream over 300
    pre-filled positions, with each attention build (by context, lane-parallel,
    tensor cores; the long-context build computes QKV in the float form)."""
    m, q4, dec, orc = make_q4(WIDE_HD128, 45, 512)
    assert dec.info.attn_tc == 1
    dec.set_debug(mk.MK_DBG_ATTN_BUILD, build)
    ks, vs = synth.make_kv(WIDE_HD128, 300, 47)
    dec.set_kv(ks, vs, 300)
    orc.set_kv(ks, vs, 300)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, WIDE_HD128.vocab, 45, 3), 300, 10)
    print(rep.summary())
    rep.check()
    dec.close()


def test_int4_generate_matches_oracle_tokens():
    """Greedy generation inside one call on the int4 stream reproduces the
    oracle's int4 greedy tokens."""
    w = synth.WORKLOADS["tiny"]
    m, q4, dec, orc = make_q4(w.shape, w.seed_weights, w.max_seq(), gains="ones", std=0.02)
    prompt = [int(t) for t in synth.make_prompt(w)[:8]]
    rc, toks = dec.generate_greedy(prompt, 0, 16)
    assert rc == mk.MK_OK
    ref = []
    tok = prompt[0]
    for p in range(len(prompt) + 16 - 1):
        if p < len(prompt):
            tok = prompt[p]
        lg, _ = orc.step(tok, p)
        tok, _ = oracle.argmax_f32(lg)
        if p >= len(prompt) - 1:
            ref.append(tok)
    assert list(toks) == ref
    dec.close()


def test_int4_digits_with_activation_outliers():
    """Norm gains of 64 and 32 on a few channels make those entries of the
    norm output ~50x the rest and set the 22-bit digits' scale; the int4
    stream's teacher-forced logits and hidden state stay within the parity
    bounds of the oracle's fp64 int4 forward."""
    m = synth.make_model(WIDE, 49, std=0.03, gains="normal")
    for kind in ("attn_norm", "ffn_norm"):
        for l in range(WIDE.n_layers):
            g = m[kind][l].copy()
            g[5], g[999], g[2046] = 0x4280, 0x4200, 0x4280   # bf16 64, 32, 64
            m[kind][l] = g
    fn = m["final_norm"].copy()
    fn[11] = 0x4280
    m["final_norm"] = fn
    q4 = oracle.quantize_model_q4(m)
    dec = Decoder(m, 256, int4=True)
    orc = oracle.OracleDecoder(m, 256, q8=q4)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, WIDE.vocab, 49, 3), 0, 10)
    print(rep.summary())
    rep.check()
    dec.close()


def test_int4_topp_sampling_matches_oracle():
    """Temperature and top-p on the int4 stream: the fused draw equals the
    oracle's nucleus sample from its int4 logits, up to the boundary cases
    the logit error allows."""
    from tests.test_parity_gpu import _nucleus_bounds, _oracle_keys
    m, q4, dec, orc = make_q4(TINY, 73, 128)
    dec.set_top_p(0.9)
    inv = float(np.float32(1.0 / 0.8))
    seed, tok, agree, steps = 0x5EED4, 9, 0, 24
    for pos in range(steps):
        dec.step_sample(tok, pos, 0.8, seed, logits=True)
        lg_ref, _ = orc.step(tok, pos)
        lg = dec.logits.cpu().numpy().astype(np.float64)
        got = dec.get_argmax()
        want, nf = oracle.sample_topp_f32(lg_ref, inv, 0.9, seed, pos)
        assert not nf
        dl = float(np.max(np.abs(lg - lg_ref)))
        assert dl <= 5e-2
        if got == want:
            agree += 1
        else:
            loose, strict = _nucleus_bounds(lg_ref, inv, 0.9, dl)
            keys = _oracle_keys(lg_ref, inv, seed, pos)
            assert got in loose, (pos, got, want)
            assert keys[got] >= max(keys[v] for v in strict) - (2 * dl * inv + 1e-5), (pos, got, want)
        tok = want
    assert agree >= steps - 2, agree
    assert dec.status() == 0
    dec.close()


def test_int4_refusals():
    """One weight form at a time, and the bf16-only paths stay closed."""
    w = synth.WORKLOADS["tiny"]
    m = synth.make_model(w.shape, 3)
    lib = mk.load()
    cfg = mk.config_from_shape(w.shape, 64)
    both = mk.tuning(weight_int8=1, weight_int4=1)
    out = mk.ctypes.c_void_p()
    assert lib.mk_create(mk.ctypes.byref(cfg), mk.ctypes.byref(both), 0, mk.ctypes.byref(out)) == \
        mk.MK_ERR_INVALID_ARG
    with pytest.raises(mk.MkError):
        Decoder(m, 64, int4=True, perop=True)
    dec = Decoder(m, 64, int4=True)
    toks = np.arange(4, dtype=np.int32)
    assert lib.mk_prefill(dec.ctx, toks.ctypes.data, 4, 0, None, dec.stream) == mk.MK_ERR_UNSUPPORTED
    dec.close()


@pytest.mark.slow
def test_full_size_int4():
    """The 1B workload on the int4 stream in the launch configuration the
    benchmark times: the prompt run from an empty cache (its first 96
    positions), teacher-forced against the oracle's int4 forward."""
    w = synth.WORKLOADS["1b"]
    m, q4, dec, orc = make_q4(w.shape, w.seed_weights, w.max_seq(), gains="ones", std=0.02)
    del m, q4
    rep = run_teacher_forced(dec, orc, synth.make_prompt(w), 0, 96)
    print("workload int4 1b", rep.summary())
    rep.check(workload=True)
    dec.close()
