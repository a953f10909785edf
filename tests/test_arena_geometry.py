"""The weight arena's size from the documented tile format, on the CPU.

mk_arena_bytes (host only) sizes the re-laid-out weight stream for a shape,
a tuning and a grid.  Here the same size is walked out independently from the
tile format include/mk.h and the library's layout notes describe: per CTA and
layer the QKV rows in tiles of TRq rows, the O rows (K = G * head_dim) in tiles
of TRo, the gate/up groups of JT j's, the W_down columns; then the LM rows in
tiles of TRh; each CTA's stream padded to 256 bytes.  bf16 rows are 2 bytes a
weight; int8 / int4 rows 1 byte / half a byte a weight plus one fp32 scale a
row (a gate/up tile also carries its j's W_down column scales), each tile
padded to 16 bytes.  The int8 / int4 QKV tiles hold at most a third of the
largest per-CTA QKV share, and int4 tiles default to 24 KB.
"""
import pytest

import synth
from decode_megakernel_05_gb300 import mk

SHAPES = {
    "tiny": synth.ModelShape(2, 256, 4, 2, 64, 688, 1024, 1e-5, 10000.0, False),
    "1b-layer": synth.ModelShape(2, 2048, 32, 8, 64, 8192, 4099, 1e-5, 500000.0, False),
    "8b-layer": synth.ModelShape(2, 4096, 32, 8, 128, 14336, 3001, 1e-5, 500000.0, False),
}


def split(n, parts, k):
    return (k * n) // parts


def pad(b, a):
    return (b + a - 1) // a * a


def expected_arena(s, grid, bits, slot):
    H, hd, kvh, F, V, L = s.hidden, s.head_dim, s.n_kv_heads, s.ffn, s.vocab, s.n_layers
    G = s.n_q_heads // kvh
    CPG, KO, NP = grid // kvh, G * hd, (G + 2) * (hd // 2)

    def rb(K):                         # stream bytes of a row of K weights
        return {16: 2 * K, 8: K, 4: K // 2}[bits]

    def tile(R, K, extra=0):           # R rows (+ their scales and `extra` more for int rows)
        return pad(R * rb(K) + (4 * (R + extra) if bits != 16 else 0), 16)

    def rows_per_tile(K, gu):
        if bits == 16:
            return (slot // (2 * K)) & ~1
        r = (slot // rb(K)) & ~1
        while r > 2 and tile(r, K, r // 2 if gu else 0) > slot:
            r -= 2
        return r

    TRh, TRo = rows_per_tile(H, True), rows_per_tile(KO, False)
    TRq = TRh
    if bits != 16:
        share = 2 * -(-NP // CPG)                      # the largest per-CTA QKV rows
        TRq = min(TRh, max(2, (-(-share // 3) + 1) // 2 * 2))
    JT, JD = TRh // 2, slot // rb(H)
    assert JD >= 1

    def row_tiles(n, TR, K):
        return sum(tile(min(TR, n - r), K) for r in range(0, n, TR))

    total = 0
    for c in range(grid):
        i = c % CPG
        npairs = split(NP, CPG, i + 1) - split(NP, CPG, i)
        norows = split(H, CPG, i + 1) - split(H, CPG, i)
        nj = split(F, grid, c + 1) - split(F, grid, c)
        nv = split(V, grid, c + 1) - split(V, grid, c)
        layer = row_tiles(2 * npairs, TRq, H) + row_tiles(norows, TRo, KO)
        layer += sum(tile(2 * min(JT, nj - j), H, min(JT, nj - j)) for j in range(0, nj, JT))
        layer += nj * rb(H)                            # W_down columns, JD a tile
        total += pad(L * layer + row_tiles(nv, TRh, H), 256)
    return total


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("bits", [16, 8, 4])
@pytest.mark.parametrize("grid", [8, 48, 152])
def test_arena_bytes_follow_the_tile_format(shape, bits, grid):
    s = SHAPES[shape]
    if grid % s.n_kv_heads:
        pytest.skip("grid must be a multiple of the KV heads")
    cfg = mk.config_from_shape(s, 64)
    q = dict(weight_int8=int(bits == 8), weight_int4=int(bits == 4))
    default_slot = 24 * 1024 if bits == 4 else 32 * 1024
    assert mk.mk_arena_bytes(cfg, mk.tuning(**q), grid) == expected_arena(s, grid, bits, default_slot)
    for kib in (16, 32):
        got = mk.mk_arena_bytes(cfg, mk.tuning(slot_kib=kib, **q), grid)
        assert got == expected_arena(s, grid, bits, kib * 1024), (kib, got)


def test_int4_stream_is_about_a_quarter_of_bf16():
    s = SHAPES["8b-layer"]
    cfg = mk.config_from_shape(s, 64)
    bf = mk.mk_arena_bytes(cfg, None, 152)
    q8 = mk.mk_arena_bytes(cfg, mk.tuning(weight_int8=1), 152)
    q4 = mk.mk_arena_bytes(cfg, mk.tuning(weight_int4=1), 152)
    assert 0.50 * bf < q8 < 0.51 * bf
    assert 0.25 * bf < q4 < 0.26 * bf


def test_one_weight_form_at_a_time():
    cfg = mk.config_from_shape(SHAPES["tiny"], 64)
    assert mk.mk_arena_bytes(cfg, mk.tuning(weight_int8=1, weight_int4=1), 8) == -1
