"""Weight-only INT8 streams (mk_tuning.weight_int8) against the oracle's int8 model.

The library quantizes every matrix on the device when it loads the weights;
the oracle quantizes the same bf16 matrices on the CPU (oracle.quantize_q8:
symmetric absmax, fp32 scale max|w| / 127 per output row, per input column
for W_down, codes rounded half to even from a float quotient).  Both decide
each code in the same float arithmetic, so

  - the arena, read back and decoded here from the documented int8 tile
    format by code of its own, holds exactly the oracle's codes and scales,
  - the decode step then meets the bf16 path's tolerances against the
    oracle's fp64 forward on the dequantized matrices (tests/parity.py).

Shapes cover the three int8 builds: (head_dim 64, 2 query heads per KV head,
hidden 256), the 1B layout (64, 4, 2048, standard and long-context
attention) and the 8B layout (128, 4, 4096).
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from decode_megakernel_05_gb300 import Decoder, mk
from tests.parity import run_teacher_forced

pytestmark = pytest.mark.gpu

SLOT = 32768
TINY = synth.ModelShape(2, 256, 4, 2, 64, 688, 1024, 1e-5, 10000.0, False)
WIDE = synth.ModelShape(2, 2048, 32, 8, 64, 2304, 4099, 1e-5, 500000.0, False)
WIDE_HD128 = synth.ModelShape(2, 4096, 32, 8, 128, 1000, 3001, 1e-5, 500000.0, False)


def split(n, parts, k):
    return (k * n) // parts


def pad16(b):
    return (b + 15) // 16 * 16


def row_bytes(K, bits=8):
    """Stream bytes of K codes: one a byte (int8) or two a byte (int4)."""
    return K if bits == 8 else K // 2


def tile_bytes(R, K, extra, bits=8):
    """R int8 / int4 rows of K, their R scales and `extra` more scales, padded to 16 bytes."""
    return pad16(R * row_bytes(K, bits) + 4 * (R + extra))


def tile_rows(K, gu_extra, bits=8, slot=SLOT):
    """Even rows per tile: as many as fit a slot with their scales (and, for the
    hidden-width tiles, the half-as-many W_down column scales of a GU tile)."""
    r = (slot // row_bytes(K, bits)) & ~1
    while r > 2 and tile_bytes(r, K, r // 2 if gu_extra else 0, bits) > slot:
        r -= 2
    return r


def unpack_q4(b):
    """int4 codes from stream bytes: each 4-byte group holds 8 codes, byte k
    code k in its low nibble and code k + 4 in its high one, each as q + 8."""
    g = b.reshape(-1, 4)
    out = np.empty((g.shape[0], 8), np.int8)
    out[:, :4] = (g & 0x0F).astype(np.int8) - 8
    out[:, 4:] = (g >> 4).astype(np.int8) - 8
    return out.reshape(-1)


def decode_arena_q8(arena, s, grid, bits=8, slot=SLOT):
    """Codes and scales of every matrix read out of an int8 (or, bits = 4,
    int4) arena, the W_down column scales, and a per-byte coverage count of
    the code bytes."""
    H, hd, kvh, F, V, L = s.hidden, s.head_dim, s.n_kv_heads, s.ffn, s.vocab, s.n_layers
    G = s.n_q_heads // kvh
    CPG, hd2, KO = grid // kvh, hd // 2, G * hd
    NP = (G + 2) * hd2
    TRh, TRo = tile_rows(H, True, bits, slot), tile_rows(KO, False, bits, slot)
    JT, JD = TRh // 2, slot // row_bytes(H, bits)
    # QKV tiles hold at most a third of the largest per-CTA QKV share (rounded
    # up to an even count, at least 2), so three consumer groups share the rows
    max_rows = 2 * -(-NP // CPG)
    TRq = min(TRh, max(2, (-(-max_rows // 3) + 1) // 2 * 2))
    qd, kvd = s.n_q_heads * hd, kvh * hd
    shapes = {"wq": (qd, H), "wk": (kvd, H), "wv": (kvd, H), "wo": (H, qd), "w_gate": (F, H), "w_up": (F, H),
              "w_down": (H, F)}
    codes = {k: [np.zeros(sh, np.int8) for _ in range(L)] for k, sh in shapes.items()}
    scales = {k: [np.full(sh[0] if k != "w_down" else sh[1], np.nan, np.float32) for _ in range(L)]
              for k, sh in shapes.items()}
    lm_q, lm_s = np.zeros((V, H), np.int8), np.full(V, np.nan, np.float32)
    cover = np.zeros(arena.size, np.int32)
    off = 0

    def codes_at(o, n):   # the stream stores each code q as the byte q + 128 (int4: packed nibbles)
        nb = row_bytes(n, bits)
        cover[o:o + nb] += 1
        if bits == 4:
            return unpack_q4(arena[o:o + nb])
        return (arena[o:o + n] ^ np.uint8(0x80)).view(np.int8)

    def f32_at(o, n):
        return arena[o:o + 4 * n].view(np.float32)

    def put_scale(arr, idx, val):
        # a row scale stored more than once (W_o rows, once per KV group) must agree
        assert np.isnan(arr[idx]) or arr[idx] == val
        arr[idx] = val

    def row_tiles(rows, K, TR, sink):
        """rows: the stored order; sink(k, codes, scale) for the k-th row."""
        nonlocal off
        for r in range(0, len(rows), TR):
            R = min(TR, len(rows) - r)
            rb = row_bytes(K, bits)
            sc = f32_at(off + R * rb, R)
            for i in range(R):
                sink(r + i, codes_at(off + i * rb, K), sc[i])
            off += tile_bytes(R, K, 0, bits)

    for c in range(grid):
        g, i = c // CPG, c % CPG
        start = off
        p0, p1 = split(NP, CPG, i), split(NP, CPG, i + 1)
        r0, r1 = split(H, CPG, i), split(H, CPG, i + 1)
        j0, j1 = split(F, grid, c), split(F, grid, c + 1)
        v0, v1 = split(V, grid, c), split(V, grid, c + 1)
        for l in range(L):
            qkv = []
            for p in range(p0, p1):
                slot_, d = p // hd2, p % hd2
                for dd in (d, d + hd2):
                    if slot_ < G:
                        qkv.append(("wq", (g * G + slot_) * hd + dd))
                    elif slot_ == G:
                        qkv.append(("wk", g * hd + dd))
                    else:
                        qkv.append(("wv", g * hd + dd))

            def qkv_sink(k, cd, sc):
                name, row = qkv[k]
                codes[name][l][row] = cd
                put_scale(scales[name][l], row, sc)
            row_tiles(qkv, H, TRq, qkv_sink)

            def o_sink(k, cd, sc):
                codes["wo"][l][r0 + k, g * KO:(g + 1) * KO] = cd
                put_scale(scales["wo"][l], r0 + k, sc)
            row_tiles(list(range(r0, r1)), KO, TRo, o_sink)
            hb = row_bytes(H, bits)
            for j in range(j0, j1, JT):
                n = min(JT, j1 - j)
                sc = f32_at(off + 2 * n * hb, 3 * n)
                for jj in range(n):
                    codes["w_gate"][l][j + jj] = codes_at(off + jj * hb, H)
                    codes["w_up"][l][j + jj] = codes_at(off + (n + jj) * hb, H)
                    put_scale(scales["w_gate"][l], j + jj, sc[jj])
                    put_scale(scales["w_up"][l], j + jj, sc[n + jj])
                    put_scale(scales["w_down"][l], j + jj, sc[2 * n + jj])
                off += tile_bytes(2 * n, H, n, bits)
            for j in range(j0, j1, JD):
                for jj in range(j, min(j + JD, j1)):
                    codes["w_down"][l][:, jj] = codes_at(off, H)
                    off += hb

        def lm_sink(k, cd, sc):
            lm_q[v0 + k] = cd
            put_scale(lm_s, v0 + k, sc)
        row_tiles(list(range(v0, v1)), H, TRh, lm_sink)
        used = off - start
        off = start + (used + 255) // 256 * 256
    return codes, scales, lm_q, lm_s, cover, off


def make_q8(shape, seed, max_seq, gains="normal", std=0.03, tuning=None):
    m = synth.make_model(shape, seed, std=std, gains=gains)
    q8 = oracle.quantize_model_q8(m)
    dec = Decoder(m, max_seq, tuning=tuning, int8=True)
    return m, q8, dec, oracle.OracleDecoder(m, max_seq, q8=q8)


def read_arena(dec):
    a = np.empty(dec.info.arena_bytes, np.uint8)
    mk.mk_read_arena(dec.ctx, 0, a.size, a.ctypes.data, dec.stream)
    return a


@pytest.mark.parametrize("shape,grid,tied", [(TINY, 0, False), (TINY, 2, True), (TINY, 6, False),
                                             (WIDE, 0, False), (WIDE, 24, True), (WIDE_HD128, 0, False)],
                         ids=["tiny", "tiny-g2-tied", "tiny-g6", "wide", "wide-g24-tied", "hd128"])
def test_arena_holds_the_oracle_codes_and_scales(shape, grid, tied):
    shape = dataclasses.replace(shape, tie_embeddings=tied)
    tun = mk.tuning(grid_ctas=grid) if grid else None
    m = synth.make_model(shape, 5, std=0.03, gains="normal")
    q8 = oracle.quantize_model_q8(m)
    dec = Decoder(m, 64, tuning=tun, int8=True)
    info = dec.info
    assert info.weight_int8 == 1 and info.slot_bytes == SLOT
    arena = read_arena(dec)
    codes, scales, lm_q, lm_s, cover, end = decode_arena_q8(arena, shape, info.grid_ctas)
    assert end == info.arena_bytes
    for name in oracle.Q8_KINDS:
        for l in range(shape.n_layers):
            rq, rs = q8[name][l]
            assert np.array_equal(codes[name][l], rq), (name, l)
            assert np.array_equal(scales[name][l].view(np.uint32), rs.view(np.uint32)), (name, l)
    rq, rs = q8["lm_head"]
    assert np.array_equal(lm_q, rq)
    assert np.array_equal(lm_s.view(np.uint32), rs.view(np.uint32))
    # every code sits in exactly one place
    assert cover.max() == 1
    assert int(cover.sum()) == sum(q.size for k in oracle.Q8_KINDS for q, _ in q8[k]) + rq.size
    # the stream is the int8 bytes plus scales and padding: about half the bf16 arena
    bf = mk.mk_arena_bytes(mk.config_from_shape(shape, 64), tun, info.grid_ctas)
    assert 0.5 * bf < info.arena_bytes < 0.56 * bf
    dec.close()


def test_tiny_workload_int8():
    w = synth.WORKLOADS["tiny"]
    m, q8, dec, orc = make_q8(w.shape, w.seed_weights, w.max_seq(), gains="ones", std=0.02)
    rep = run_teacher_forced(dec, orc, synth.make_prompt(w), 0, w.prompt_len + w.decode - 1)
    print("tiny int8", rep.summary())
    rep.check(workload=True)
    dec.close()


@pytest.mark.parametrize("grid,tied,prefill", [(2, True, 0), (6, False, 90), (0, False, 0)])
def test_tiny_int8_multi_tile(grid, tied, prefill):
    """Grid 2 (one CTA per KV group): 512 LM rows, 344 FFN columns and the whole
    QKV block per CTA, so every phase walks several int8 tiles with a ragged
    last one, and a GU tile carries 62 W_down column scales."""
    shape = dataclasses.replace(TINY, tie_embeddings=tied)
    tun = mk.tuning(grid_ctas=grid) if grid else None
    m, q8, dec, orc = make_q8(shape, 11 + grid, 256, tuning=tun)
    if prefill:
        ks, vs = synth.make_kv(shape, prefill, 13)
        dec.set_kv(ks, vs, prefill)
        orc.set_kv(ks, vs, prefill)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(6, shape.vocab, grid, 3), prefill, 24)
    print(grid, tied, rep.summary())
    rep.check()
    dec.close()


@pytest.mark.parametrize("prefill,build", [(0, 0), (3000, 1), (3000, 2)])
def test_wide_int8_both_attention_builds(prefill, build):
    """The 1B layout (H=2048, 4 query heads of 64 per KV group): the standard
    int8 build, and after a 3000-position prefill both attention builds
    (lane-parallel, tensor cores) over the same int8 weight stream."""
    m, q8, dec, orc = make_q8(WIDE, 31, 4096)
    assert dec.info.attn_tc == 1
    dec.set_debug(mk.MK_DBG_ATTN_BUILD, build)
    if prefill:
        ks, vs = synth.make_kv(WIDE, prefill, 37)
        dec.set_kv(ks, vs, prefill)
        orc.set_kv(ks, vs, prefill)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, WIDE.vocab, 31, 3), prefill, 12)
    print(prefill, build, rep.summary())
    rep.check()
    dec.close()


def test_int8_digits_with_activation_outliers():
    """The int8 build holds the norm output as 22-bit fixed point with one
    scale per vector, set by its largest entry.  Norm gains of 64 and 32 on a
    few channels make those entries ~50x the rest (which then keep ~16 bits
    relative to themselves); the teacher-forced logits and hidden state stay
    within the parity bounds of the oracle's fp64 int8 forward."""
    m = synth.make_model(WIDE, 47, std=0.03, gains="normal")
    for kind in ("attn_norm", "ffn_norm"):
        for l in range(WIDE.n_layers):
            g = m[kind][l].copy()
            g[7], g[1000], g[2047] = 0x4280, 0x4200, 0x4280   # bf16 64, 32, 64
            m[kind][l] = g
    fn = m["final_norm"].copy()
    fn[3] = 0x4280
    m["final_norm"] = fn
    q8 = oracle.quantize_model_q8(m)
    dec = Decoder(m, 256, int8=True)
    orc = oracle.OracleDecoder(m, 256, q8=q8)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, WIDE.vocab, 47, 3), 0, 10)
    print(rep.summary())
    rep.check()
    dec.close()


def test_hd128_int8():
    """The 8B layer width and head layout on the int8 stream (integer dot
    products over the activation's digits; this width has no tensor-core
    attention build in int8: with the digits it spilled) over 300 pre-filled
    positions."""
    m, q8, dec, orc = make_q8(WIDE_HD128, 41, 512)
    assert dec.info.attn_tc == 0
    ks, vs = synth.make_kv(WIDE_HD128, 300, 43)
    dec.set_kv(ks, vs, 300)
    orc.set_kv(ks, vs, 300)
    rep = run_teacher_forced(dec, orc, synth.uniform_tokens(4, WIDE_HD128.vocab, 41, 3), 300, 10)
    print(rep.summary())
    rep.check()
    dec.close()


def test_int8_generate_matches_oracle_tokens():
    """Greedy generation inside one call on the int8 stream reproduces the
    oracle's int8 greedy tokens (teacher-forced parity above bounds the logits;
    here the tokens feed back)."""
    w = synth.WORKLOADS["tiny"]
    m, q8, dec, orc = make_q8(w.shape, w.seed_weights, w.max_seq(), gains="ones", std=0.02)
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


def test_int8_topp_sampling_matches_oracle():
    """Temperature and top-p on the int8 stream (the LM head's int8 rows feed
    the same in-launch nucleus search): the fused draw equals the oracle's
    nucleus sample from its int8 logits, up to the boundary cases the logit
    error allows."""
    from tests.test_parity_gpu import _nucleus_bounds, _oracle_keys
    m, q8, dec, orc = make_q8(TINY, 71, 128)
    dec.set_top_p(0.9)
    inv = float(np.float32(1.0 / 1.0))
    seed, tok, agree, steps = 0x5EED, 7, 0, 24
    for pos in range(steps):
        dec.step_sample(tok, pos, 1.0, seed, logits=True)
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


def test_int8_refuses_the_bf16_only_paths():
    w = synth.WORKLOADS["tiny"]
    m = synth.make_model(w.shape, 3)
    lib = mk.load()
    with pytest.raises(mk.MkError):
        Decoder(m, 64, int8=True, perop=True)
    dec = Decoder(m, 64, int8=True)
    toks = np.arange(4, dtype=np.int32)
    assert lib.mk_prefill(dec.ctx, toks.ctypes.data, 4, 0, None, dec.stream) == mk.MK_ERR_UNSUPPORTED
    buf = np.empty(16, np.uint8)
    assert lib.mk_read_arena(dec.ctx, dec.info.arena_bytes - 8, 16, buf.ctypes.data, dec.stream) == \
        mk.MK_ERR_INVALID_ARG
    assert lib.mk_read_arena(dec.ctx, -1, 4, buf.ctypes.data, dec.stream) == mk.MK_ERR_INVALID_ARG
    dec.close()
    # no int8 build for this shape (H = 512)
    mid = synth.ModelShape(2, 512, 8, 2, 64, 1000, 5003, 1e-5, 10000.0, False)
    cfg = mk.config_from_shape(mid, 64)
    t = mk.tuning(weight_int8=1)
    out = mk.ctypes.c_void_p()
    assert lib.mk_create(mk.ctypes.byref(cfg), mk.ctypes.byref(t), 0, mk.ctypes.byref(out)) == \
        mk.MK_ERR_UNSUPPORTED


# ------------------------------------------------------------ full-size

@pytest.mark.slow
@pytest.mark.parametrize("name,steps", [("1b", 96), ("1b-32k", 24)])
def test_full_size_int8(name, steps):
    """The 1B workloads on the int8 stream in the launch configuration the
    benchmark times: the prompt run from an empty cache (its first 96
    positions), and 24 steps after a 32768-position prefill (the long-context
    build), teacher-forced against the oracle's int8 forward."""
    w = synth.WORKLOADS[name]
    m, q8, dec, orc = make_q8(w.shape, w.seed_weights, w.max_seq(), gains="ones", std=0.02)
    del m, q8
    if w.prefill:
        ks, vs = synth.make_kv(w.shape, w.prefill, w.seed_kv)
        dec.set_kv(ks, vs, w.prefill)
        orc.set_kv(ks, vs, w.prefill)
        del ks, vs
        toks, start = [synth.make_first_token(w)], w.prefill
    else:
        toks, start = synth.make_prompt(w), 0
    rep = run_teacher_forced(dec, orc, toks, start, steps)
    print("workload int8", name, rep.summary())
    rep.check(workload=True)
    dec.close()
