"""Failure detection without a GPU fault.

A debug knob makes one CTA skip one flag arrival, so every CTA waiting on that
flag runs into its bounded wait (here 20 ms): the launch gives up, latches
MK_ERR_DEVICE_TIMEOUT in the device status word, resets its flags, and the
context stays usable -- the next step (rewound to the same position) matches
the oracle again.  Nothing traps, faults or spins without a limit.
"""
import numpy as np
import pytest

import oracle
import synth
from decode_megakernel_05_gb300 import Decoder, mk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    w = synth.WORKLOADS["tiny"]
    m = synth.make_model(w.shape, w.seed_weights)
    dec = Decoder(m, w.max_seq())
    yield w, m, dec
    dec.close()


@pytest.mark.parametrize("sync_id", [0, 1, 2, 3, 4 + 2])
def test_skipped_arrival_times_out_and_context_recovers(tiny, sync_id):
    w, m, dec = tiny
    orc = oracle.OracleDecoder(m, w.max_seq())
    prompt = synth.make_prompt(w)
    for p in range(3):
        orc.step(int(prompt[p]), p)
        dec.step(int(prompt[p]), p)
    assert dec.status() == mk.MK_OK
    dec.set_debug(mk.MK_DBG_WAIT_LIMIT_NS, 20_000_000)
    # CTA 5 skips its arrival; the attention partials (sync_id 1) come only
    # from the CTAs that run the step's attention, which always include CTA 0
    cta = 0 if sync_id == 1 else 5
    dec.set_debug(mk.MK_DBG_SKIP_ARRIVAL, cta * 65536 + sync_id)
    dec.step(int(prompt[3]), 3)
    assert dec.status() == mk.MK_ERR_DEVICE_TIMEOUT
    dec.set_debug(mk.MK_DBG_SKIP_ARRIVAL, -1)
    dec.set_debug(mk.MK_DBG_WAIT_LIMIT_NS, 1_000_000_000)
    ref, _ = orc.step(int(prompt[3]), 3)
    got = dec.step(int(prompt[3]), 3).cpu().numpy()
    assert dec.status() == mk.MK_OK
    assert np.max(np.abs(got - ref)) <= 5e-2


def test_generate_greedy_reports_timeout(tiny):
    w, m, dec = tiny
    dec.set_debug(mk.MK_DBG_WAIT_LIMIT_NS, 20_000_000)
    dec.set_debug(mk.MK_DBG_SKIP_ARRIVAL, 0 * 65536 + 3)
    rc, _ = dec.generate_greedy([1, 2, 3], 0, 2)
    assert rc == mk.MK_ERR_DEVICE_TIMEOUT
    dec.set_debug(mk.MK_DBG_SKIP_ARRIVAL, -1)
    dec.set_debug(mk.MK_DBG_WAIT_LIMIT_NS, 1_000_000_000)
    rc, _ = dec.generate_greedy([1, 2, 3], 0, 2)
    assert rc == mk.MK_OK


def test_argument_errors_return_codes_without_launch(tiny):
    w, m, dec = tiny
    lib = mk.load()
    assert lib.mk_decode_step(dec.ctx, w.shape.vocab, 0, None, dec.stream) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_decode_step(dec.ctx, -1, 0, None, dec.stream) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_decode_step(dec.ctx, 1, dec.max_seq, None, dec.stream) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_decode_step_greedy(dec.ctx, -5, None, dec.stream) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_set_debug(dec.ctx, 99, 0) == mk.MK_ERR_INVALID_ARG
    # attention-build knobs: this shape (2 query heads per KV group) has no tensor-core build
    assert dec.info.attn_tc == 0 and dec.info.attn_tc_min_ctx == -1
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_ATTN_BUILD, 2) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_ATTN_BUILD, 3) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_ATTN_TC_MIN, -1) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_ATTN_TC_MIN, dec.max_seq + 1) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_ATTN_BUILD, 0) == mk.MK_OK
    # attention-split knobs: 0 .. CTAs per group, positions per CTA >= 1
    cpg = dec.info.ctas_per_group
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_ATTN_CTAS, -1) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_ATTN_CTAS, cpg + 1) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_ATTN_POS_PER_CTA, 0) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_ATTN_CTAS, cpg) == mk.MK_OK
    assert mk.mk_get_info(dec.ctx).attn_pos_per_cta == 0
    assert lib.mk_set_debug(dec.ctx, mk.MK_DBG_ATTN_CTAS, 0) == mk.MK_OK
    assert mk.mk_get_info(dec.ctx).attn_pos_per_cta == dec.info.attn_pos_per_cta > 0
    # a K/V window past the end of the cache
    k = np.zeros((w.shape.n_kv_heads, 2, w.shape.head_dim), dtype=np.uint16)
    v = np.zeros_like(k)
    assert lib.mk_get_kv(dec.ctx, 0, dec.max_seq - 1, 2, k.ctypes.data, v.ctypes.data, dec.stream) == \
        mk.MK_ERR_INVALID_ARG
    assert lib.mk_set_kv(dec.ctx, 0, k.ctypes.data, v.ctypes.data, dec.max_seq + 1, dec.stream) == \
        mk.MK_ERR_INVALID_ARG
    assert dec.status() == mk.MK_OK


def test_decode_before_weights_is_a_state_error():
    w = synth.WORKLOADS["tiny"]
    ctx = mk.mk_create(mk.config_from_shape(w.shape, 64))
    try:
        assert mk.load().mk_decode_step(ctx, 1, 0, None, None) == mk.MK_ERR_STATE
    finally:
        mk.mk_destroy(ctx)


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_nonfinite_logits_report_numeric(int8):
    """An infinite final-norm gain makes the step's logits non-finite: the step
    reports MK_ERR_NUMERIC (the int8 build's integer dot products carry it
    through the activation scale), and once the gain is finite again the next
    context decodes cleanly."""
    w = synth.WORKLOADS["tiny"]
    m = synth.make_model(w.shape, w.seed_weights)
    bad = dict(m)
    bad["final_norm"] = m["final_norm"].copy()
    bad["final_norm"][5] = 0x7F80   # bf16 +inf
    dec = Decoder(bad, w.max_seq(), int8=int8)
    lg = dec.step(3, 0, logits=True)
    assert dec.status() == mk.MK_ERR_NUMERIC
    assert not np.isfinite(lg.cpu().numpy()).all()
    dec.close()
    dec = Decoder(m, w.max_seq(), int8=int8)
    lg = dec.step(3, 0, logits=True)
    assert dec.status() == mk.MK_OK
    assert np.isfinite(lg.cpu().numpy()).all()
    dec.close()
