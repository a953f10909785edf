"""The allocation-free greedy argmax (mk_argmax_f32_noalloc) through the C ABI.

Callers that cannot call cudaMalloc -- engines that reserve all device memory
up front, or code that must not allocate on its hot path -- can pick the greedy
token of logits they already hold with this entry point: its scratch is a fixed
array inside the library.  Here it must return exactly the token the fused
decode step picked (mk_get_argmax) for the same logits, on two calls in a row
(the second call finds the first call's leftovers in the shared scratch).

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest

import synth
from decode_megakernel_05_gb300 import Decoder, mk

pytestmark = pytest.mark.gpu


def test_noalloc_argmax_matches_fused_step_twice():
    import torch

    w = synth.WORKLOADS["tiny"]
    m = synth.make_model(w.shape, w.seed_weights, std=0.05)
    dec = Decoder(m, w.max_seq())
    prompt = synth.make_prompt(w)
    out = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    try:
        for pos in range(2):   # two calls in a row
            logits = dec.step(int(prompt[pos]), pos)
            rc = mk.mk_argmax_f32_noalloc(logits.data_ptr(), w.shape.vocab, out.data_ptr(), dec.stream)
            assert rc == mk.MK_OK
            got = int(out.item())
            assert got == dec.get_argmax()                                  # the existing entry point
            assert got == int(np.argmax(logits.cpu().numpy()))             # first index of the maximum
        assert dec.status() == mk.MK_OK
    finally:
        dec.close()


def test_noalloc_argmax_rejects_sizes_beyond_its_scratch():
    import torch

    x = torch.zeros(8, dtype=torch.float32, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = mk.load()
    assert lib.mk_argmax_f32_noalloc(x.data_ptr(), mk.MK_NOALLOC_ARGMAX_MAX_N + 1, out.data_ptr(),
                                     None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_argmax_f32_noalloc(x.data_ptr(), 0, out.data_ptr(), None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_argmax_f32_noalloc(None, 8, out.data_ptr(), None) == mk.MK_ERR_INVALID_ARG
    # ties go to the lowest index, as in the fused step
    x[3] = 2.5
    x[5] = 2.5
    assert lib.mk_argmax_f32_noalloc(x.data_ptr(), 8, out.data_ptr(), None) == mk.MK_OK
    assert int(out.item()) == 3


def _argmax(x, n, out, stream=None):
    rc = mk.load().mk_argmax_f32_noalloc(x.data_ptr(), n, out.data_ptr(), stream)
    assert rc == mk.MK_OK, mk.mk_strerror(rc)
    return int(out.item())


def test_noalloc_argmax_across_blocks_then_a_smaller_call():
    """n = 128256 (the 1B vocabulary: 31 full blocks of 4096 logits and a
    partial one) needs the reduction across block partials.  The maximum sits
    in the last, partial block; an equal value planted in an earlier block must
    win (lowest index).  A call of n = 5000 follows on the same stream, with
    the larger call's partials still in the shared scratch: it must read only
    its own two."""
    import torch

    n = 128256
    g = torch.Generator().manual_seed(1234)
    x = torch.randn(n, generator=g, dtype=torch.float32).cuda()
    out = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    x[127000] = 9.0                     # last block only: it must win
    assert _argmax(x, n, out) == 127000 == int(np.argmax(x.cpu().numpy()))
    x[70000] = 9.0                      # an equal value in an earlier block: the lower index wins
    assert _argmax(x, n, out) == 70000 == int(np.argmax(x.cpu().numpy()))
    small = x[:5000].clone()
    small[4500] = 7.5                   # in the second block of the smaller call
    assert _argmax(small, 5000, out) == 4500 == int(np.argmax(small.cpu().numpy()))
    assert _argmax(x, n, out) == 70000  # and the large call again after it


def test_noalloc_argmax_nonfinite_and_signed_zero():
    """No finite logit gives -1; NaN and infinities are skipped; -0.0 and +0.0
    are equal, so the lower index wins whichever sign comes first."""
    import torch

    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    nan = torch.full((9000,), float("nan"), dtype=torch.float32, device="cuda")
    assert _argmax(nan, 9000, out) == -1
    nan[8500] = -3.0
    nan[100] = float("inf")
    nan[200] = float("-inf")
    assert _argmax(nan, 9000, out) == 8500
    for vals in ([-0.0, 0.0], [0.0, -0.0]):
        z = torch.tensor(vals, dtype=torch.float32, device="cuda")
        assert _argmax(z, 2, out) == 0 == int(np.argmax(z.cpu().numpy()))
