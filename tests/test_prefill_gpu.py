"""Batched prefill (mk_prefill) against the oracle's token-by-token prompt.

The prefill runs the prompt's rows through each layer together (tensor-core
GEMMs, causal attention over the cache).  Its result is defined by the
decode step it replaces: after it, the cache must hold the K/V rows that n
decode steps write (the oracle's bf16 rows, up to a rounding flip), the last
token's logits and final hidden state must match the oracle's within the
decode tolerances, its greedy token must be the argmax of those logits, and
decode steps that follow must keep parity.
"""
import numpy as np
import pytest

import oracle
import synth
from decode_megakernel_05_gb300 import Decoder, mk
from tests.parity import HIDDEN_TOL, LOGIT_TOL, run_teacher_forced

pytestmark = pytest.mark.gpu

MID = synth.ModelShape(2, 512, 8, 2, 64, 1000, 5003, 1e-5, 10000.0, False)
HD128 = synth.ModelShape(2, 1024, 8, 2, 128, 1536, 4099, 1e-5, 500000.0, False)


def _check_kv(dec, orc, shape, p0, n):
    """The cache rows the prefill wrote against the oracle's bf16 rows.
    Layer 0's rows come from the embedding through one GEMM and are bit-equal
    up to rounding flips: a value within the difference between the
    tensor-core and the oracle's sums of a bf16 rounding boundary lands on the
    neighbouring bf16.  So every mismatch of layer 0 must lie within one bf16
    step of the oracle's value plus the fp32 sum's own error, bounded here by
    2^-16 of the row's largest magnitude (it decides values far below the
    row's scale, where it spans several of their steps), and flips stay rare
    (at most 1 %; the sum's error, and with it the flip rate, grows with the
    K = hidden of the product: 0.04 % at 512, 0.4 % at 2048, 0.7 % at 4096).
    Each flip moves an attention output of a later layer by up to one bf16
    step of one V element times its weight, so deeper layers drift further;
    their rows are bounded by the tolerances their inputs carry, checked here
    against the row's largest magnitude."""
    for l in range(shape.n_layers):
        k, v = dec.get_kv(l, p0, n)
        for nm, got, ref in (("K", k, orc.kcache[l, :, p0:p0 + n]), ("V", v, orc.vcache[l, :, p0:p0 + n])):
            g32, r32 = synth.bf16_to_f32(got), synth.bf16_to_f32(ref)
            eq = float(np.mean(got == ref))
            row_max = np.max(np.abs(r32), axis=-1, keepdims=True)
            rel = np.abs(g32.astype(np.float64) - r32) / row_max
            print(f"  layer {l} {nm}: bit-equal {eq:.4f}, mean |d|/rowmax {rel.mean():.2e}, max {rel.max():.2e}")
            if l == 0:
                assert eq > 0.99, eq
                step = np.abs(r32) * 2.0 ** -7 + 1e-30                  # one bf16 step at the value (upper bound)
                slack = np.broadcast_to(row_max, r32.shape) * 2.0 ** -16
                dev = np.abs(g32.astype(np.float64) - r32)
                assert np.all(dev <= step + slack), "layer 0: a mismatch beyond a rounding flip"
            assert rel.mean() <= 2e-3 and rel.max() <= 2 ** -4, (l, nm, rel.mean(), rel.max())


def _prefill_vs_oracle(dec, orc, shape, tokens, start):
    lg_ref = h_ref = None
    for i, tk in enumerate(tokens):
        lg_ref, h_ref = orc.step(int(tk), start + i)
    lg = dec.prefill(tokens, start).cpu().numpy().astype(np.float64)
    h = dec.get_hidden().cpu().numpy().astype(np.float64)
    dl = float(np.max(np.abs(lg - lg_ref)))
    hrel = float(np.max(np.abs(h - h_ref)) / np.max(np.abs(h_ref)))
    print(f"prefill n={len(tokens)} start={start}: max|dlogit|={dl:.3e} hidden_rel={hrel:.3e}")
    assert dl <= LOGIT_TOL and hrel <= HIDDEN_TOL
    assert dec.get_argmax() == int(np.argmax(lg.astype(np.float32)))   # the kernel's own greedy token
    top2 = np.sort(lg_ref.astype(np.float32))[-2:]
    if float(top2[1] - top2[0]) >= 2 * dl:                              # not a near tie: the oracle's too
        assert dec.get_argmax() == oracle.argmax_f32(lg_ref)[0]
    _check_kv(dec, orc, shape, start, len(tokens))
    assert dec.status() == 0


def test_prefill_tiny_prompt_then_decode():
    """The tiny workload's 32-token prompt in one prefill, then its 16 decode
    steps teacher-forced on the cache the prefill wrote."""
    w = synth.WORKLOADS["tiny"]
    m = synth.make_model(w.shape, w.seed_weights)
    dec, orc = Decoder(m, w.max_seq(), perop=True), oracle.OracleDecoder(m, w.max_seq())
    prompt = synth.make_prompt(w)
    _prefill_vs_oracle(dec, orc, w.shape, prompt, 0)
    # decode continues from the prefilled cache, fed the oracle's greedy tokens
    tok = dec.get_argmax()
    rep = run_teacher_forced(dec, orc, [tok], w.prompt_len, w.decode)
    print("decode after prefill", rep.summary())
    rep.check()
    dec.close()


@pytest.mark.parametrize("grid,prefill,n", [(0, 300, 37), (14, 0, 61), (0, 700, 1), (6, 41, 130)])
def test_prefill_mid_shape(grid, prefill, n):
    """H=512, G=4 (the permuted cache layout), F=1000 and V=5003 (ragged GEMM
    edges): prompts after a pre-filled cache (attention over cache + prompt),
    from position 0, a single row, and more rows than one GEMM tile."""
    tun = mk.tuning(grid_ctas=grid) if grid else None
    m = synth.make_model(MID, 101, std=0.04, gains="normal")
    dec = Decoder(m, 1024, tuning=tun, perop=True)
    orc = oracle.OracleDecoder(m, 1024)
    if prefill:
        ks, vs = synth.make_kv(MID, prefill, 103)
        dec.set_kv(ks, vs, prefill)
        orc.set_kv(ks, vs, prefill)
    toks = synth.uniform_tokens(n, MID.vocab, 101, 9)
    _prefill_vs_oracle(dec, orc, MID, toks, prefill)
    rep = run_teacher_forced(dec, orc, [dec.get_argmax()], prefill + n, 4)
    rep.check()
    dec.close()


@pytest.mark.parametrize("gemm", [0, 1], ids=["tcgen05", "mma_sync"])
def test_prefill_gemm_paths(gemm):
    """Both GEMM engines of the prefill (MK_DBG_PREFILL_GEMM: 0 tcgen05 with TMA
    tiles and TMEM accumulators, the default; 1 mma.sync) on the ragged H=512
    shape, 130 rows after 41 pre-filled positions (two 128-row tiles, N and K
    tails), meet the same bars against the oracle."""
    m = synth.make_model(MID, 113, std=0.04, gains="normal")
    dec = Decoder(m, 1024, perop=True)
    dec.set_debug(mk.MK_DBG_PREFILL_GEMM, gemm)
    orc = oracle.OracleDecoder(m, 1024)
    ks, vs = synth.make_kv(MID, 41, 117)
    dec.set_kv(ks, vs, 41)
    orc.set_kv(ks, vs, 41)
    _prefill_vs_oracle(dec, orc, MID, synth.uniform_tokens(130, MID.vocab, 113, 9), 41)
    dec.close()


W8B = synth.ModelShape(2, 4096, 32, 8, 128, 14336, 3001, 1e-5, 500000.0, False)


def test_prefill_8b_width():
    """The 8B layer width (H 4096, 4 heads of 128 per KV group, F 14336): the
    gate/up product takes 256-wide tiles (N = 28672), O-proj and down split K
    across two CTAs with the atomic epilogue, 150 rows (two 128-row tiles)
    after 40 pre-filled positions."""
    m = synth.make_model(W8B, 127, std=0.02, gains="normal")
    dec, orc = Decoder(m, 512, perop=True), oracle.OracleDecoder(m, 512)
    ks, vs = synth.make_kv(W8B, 40, 131)
    dec.set_kv(ks, vs, 40)
    orc.set_kv(ks, vs, 40)
    _prefill_vs_oracle(dec, orc, W8B, synth.uniform_tokens(150, W8B.vocab, 127, 5), 40)
    dec.close()


def test_prefill_head_dim_128():
    """hd=128 (the 8B head layout, chunk-permuted cache rows) with 100 pre-filled positions."""
    m = synth.make_model(HD128, 107, std=0.03, gains="normal")
    dec, orc = Decoder(m, 512, perop=True), oracle.OracleDecoder(m, 512)
    ks, vs = synth.make_kv(HD128, 100, 109)
    dec.set_kv(ks, vs, 100)
    orc.set_kv(ks, vs, 100)
    _prefill_vs_oracle(dec, orc, HD128, synth.uniform_tokens(70, HD128.vocab, 107, 3), 100)
    dec.close()


def test_prefill_argument_errors():
    w = synth.WORKLOADS["tiny"]
    m = synth.make_model(w.shape, w.seed_weights)
    lib = mk.load()
    toks = np.arange(8, dtype=np.int32)
    plain = Decoder(m, 64)   # no row-major weights: refused
    assert lib.mk_prefill(plain.ctx, toks.ctypes.data, 8, 0, None, plain.stream) == mk.MK_ERR_STATE
    plain.close()
    dec = Decoder(m, 64, perop=True)
    assert lib.mk_prefill(dec.ctx, toks.ctypes.data, 0, 0, None, dec.stream) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_prefill(dec.ctx, toks.ctypes.data, 8, 57, None, dec.stream) == mk.MK_ERR_INVALID_ARG
    bad = toks.copy()
    bad[3] = w.shape.vocab
    assert lib.mk_prefill(dec.ctx, bad.ctypes.data, 8, 0, None, dec.stream) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_prefill(dec.ctx, toks.ctypes.data, 8, 56, None, dec.stream) == mk.MK_OK
    assert dec.status() == mk.MK_OK
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_PREFILL_GEMM, 2) == mk.MK_ERR_INVALID_ARG
    dec.close()


@pytest.mark.slow
def test_prefill_1b_prompt_512():
    """The 1B workload's 512-token prompt in one prefill against the oracle's
    512 decode steps: every K/V row of positions 0..511 in all 16 layers and the
    logits of position 511."""
    w = synth.WORKLOADS["1b"]
    m = synth.make_model(w.shape, w.seed_weights)
    dec = Decoder(m, w.max_seq(), perop=True)
    orc = oracle.OracleDecoder(m, w.max_seq())
    del m
    _prefill_vs_oracle(dec, orc, w.shape, synth.make_prompt(w), 0)
    dec.close()
