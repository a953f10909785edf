"""Offline re-layout round trip (CPU): the arena mk_relayout_host builds is
decoded here from the documented stream format (include/mk.h, mk_internal.h)
by independent Python code, and must reproduce every source matrix bit-exactly
and cover the arena without overlap."""
import numpy as np
import pytest

import synth
from decode_megakernel_05_gb300 import mk


def split(n, parts, k):
    return (k * n) // parts


def tile_rows(K, slot):
    return (slot // (2 * K)) & ~1


def decode_arena(arena, s, grid, slot=32768):
    """Returns dict of reconstructed matrices and a coverage count per arena byte."""
    H, hd, G, kvh, F, V, L = s.hidden, s.head_dim, s.n_q_heads // s.n_kv_heads, s.n_kv_heads, s.ffn, s.vocab, s.n_layers
    CPG, hd2, KO = grid // kvh, hd // 2, G * hd
    NP = (G + 2) * hd2
    JT = tile_rows(H, slot) // 2
    u16 = arena.view(np.uint16)
    cover = np.zeros(arena.size // 2, dtype=np.int32)
    out = {k: [np.zeros(shape, np.uint16) for _ in range(L)] for k, shape in
           [("wq", (s.n_q_heads * hd, H)), ("wk", (kvh * hd, H)), ("wv", (kvh * hd, H)), ("wo", (H, s.n_q_heads * hd)),
            ("w_gate", (F, H)), ("w_up", (F, H)), ("w_down", (H, F))]}
    lm = np.zeros((V, H), np.uint16)
    off = 0  # in uint16 elements

    def take(n):
        nonlocal off
        a = u16[off:off + n]
        cover[off:off + n] += 1
        off += n
        return a

    for c in range(grid):
        g, i = c // CPG, c % CPG
        start = off
        p0, p1 = split(NP, CPG, i), split(NP, CPG, i + 1)
        r0, r1 = split(H, CPG, i), split(H, CPG, i + 1)
        j0, j1 = split(F, grid, c), split(F, grid, c + 1)
        v0, v1 = split(V, grid, c), split(V, grid, c + 1)
        for l in range(L):
            for p in range(p0, p1):
                slot_, d = p // hd2, p % hd2
                for dd in (d, d + hd2):
                    row = take(H)
                    if slot_ < G:
                        out["wq"][l][(g * G + slot_) * hd + dd] = row
                    elif slot_ == G:
                        out["wk"][l][g * hd + dd] = row
                    else:
                        out["wv"][l][g * hd + dd] = row
            for r in range(r0, r1):
                out["wo"][l][r, g * KO:(g + 1) * KO] = take(KO)
            for j in range(j0, j1, JT):
                n = min(JT, j1 - j)
                for jj in range(n):
                    out["w_gate"][l][j + jj] = take(H)
                for jj in range(n):
                    out["w_up"][l][j + jj] = take(H)
            for j in range(j0, j1):
                out["w_down"][l][:, j] = take(H)
        for v in range(v0, v1):
            lm[v] = take(H)
        used = (off - start) * 2
        off = start + ((used + 255) // 256 * 256) // 2
    return out, lm, cover, off * 2


@pytest.mark.parametrize("grid,tied,shape_kw", [
    (152, False, {}), (152, True, {}), (14, False, {}), (2, True, {}),
    (152, False, dict(hidden=512, n_q_heads=8, n_kv_heads=2, ffn=1000, vocab=5003)),
    (24, True, dict(hidden=512, n_q_heads=16, n_kv_heads=8, head_dim=128, ffn=72, vocab=333)),
])
def test_relayout_round_trip(grid, tied, shape_kw):
    d = dict(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=688, vocab=1024,
             rms_eps=1e-5, rope_theta=1e4, tie_embeddings=tied)
    d.update(shape_kw)
    s = synth.ModelShape(**d)
    m = synth.make_model(s, seed=3)
    cfg = mk.config_from_shape(s, 64)
    nbytes = mk.mk_arena_bytes(cfg, None, grid)
    assert nbytes > 0
    arena = np.full(nbytes, 0xAB, dtype=np.uint8)
    keep = []

    def hp(a):
        keep.append(np.ascontiguousarray(a))
        return keep[-1].ctypes.data

    ptrs = {"embed": hp(m["embed"]), "final_norm": hp(m["final_norm"]),
            "lm_head": None if m["lm_head"] is None else hp(m["lm_head"])}
    for name in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"):
        ptrs[name] = [hp(a) for a in m[name]]
    w, _t = mk.weights_struct(ptrs, on_device=False)
    mk.mk_relayout_host(cfg, None, grid, w, arena.ctypes.data)
    out, lm, cover, end = decode_arena(arena, s, grid)
    assert end == nbytes
    for name, mats in out.items():
        for l in range(s.n_layers):
            assert np.array_equal(mats[l], m[name][l]), (name, l)
    assert np.array_equal(lm, m["embed"] if tied else m["lm_head"])
    # every element of every matrix sits in exactly one place; the rest is stream padding
    assert cover.max() == 1
    n_weights = sum(a.size for k in out for a in m[k]) + lm.size
    assert int(cover.sum()) == n_weights
