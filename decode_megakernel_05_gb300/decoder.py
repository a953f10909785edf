"""Convenience wrapper around one decode-megakernel context.

It only marshals: numpy weight arrays are handed to ``mk_load_weights`` as host
pointers (the library copies and re-lays them out on the device), device
buffers are torch tensors, and every step is one call into the C ABI.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import mk

_LAYER_NAMES = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


class Decoder:
    def __init__(self, model: dict, max_seq: int, device: int = 0, tuning: mk.mk_tuning | None = None,
                 perop: bool = False, int8: bool = False, int4: bool = False):
        """int8 / int4: stream weight-only INT8 / INT4 matrices (quantized on the device at load,
        mk_tuning.weight_int8 / weight_int4)."""
        import torch

        if int8 or int4:
            t = mk.mk_tuning()
            if tuning is not None:
                ctypes.memmove(ctypes.byref(t), ctypes.byref(tuning), ctypes.sizeof(t))
            t.weight_int8 = int(bool(int8))
            t.weight_int4 = int(bool(int4))
            tuning = t

        self.torch = torch
        self.shape = s = model["shape"]
        self.max_seq = int(max_seq)
        self.device = device
        self.cfg = mk.config_from_shape(s, self.max_seq)
        self.ctx = mk.mk_create(self.cfg, tuning, device)
        try:
            if perop:
                mk.mk_enable_perop(self.ctx, True)
            keep = []

            def hp(a):
                a = np.ascontiguousarray(a, dtype=np.uint16)
                keep.append(a)
                return a.ctypes.data

            ptrs = {"embed": hp(model["embed"]), "final_norm": hp(model["final_norm"]),
                    "lm_head": None if model["lm_head"] is None else hp(model["lm_head"])}
            for name in _LAYER_NAMES:
                ptrs[name] = [hp(a) for a in model[name]]
            w, _tbl = mk.weights_struct(ptrs, on_device=False)
            mk.mk_load_weights(self.ctx, w, self.stream)
            del keep
            self.info = mk.mk_get_info(self.ctx)
        except Exception:
            mk.mk_destroy(self.ctx)
            self.ctx = None
            raise
        dev = torch.device("cuda", device)
        self.logits = torch.empty(s.vocab, dtype=torch.float32, device=dev)
        self.hidden = torch.empty(s.hidden, dtype=torch.float32, device=dev)
        self.argmax_buf = torch.empty(1, dtype=torch.int32, device=dev)

    @property
    def stream(self) -> int:
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def set_kv(self, ks, vs, n_pos: int):
        """Pre-fill positions [0, n_pos) from host bf16 arrays [kv_heads][n_pos][head_dim] per layer."""
        for l in range(self.shape.n_layers):
            k = np.ascontiguousarray(ks[l], dtype=np.uint16)
            v = np.ascontiguousarray(vs[l], dtype=np.uint16)
            mk.mk_set_kv(self.ctx, l, k.ctypes.data, v.ctypes.data, n_pos, self.stream)

    def get_kv(self, layer: int, pos0: int, n_pos: int):
        s = self.shape
        k = np.empty((s.n_kv_heads, n_pos, s.head_dim), dtype=np.uint16)
        v = np.empty_like(k)
        mk.mk_get_kv(self.ctx, layer, pos0, n_pos, k.ctypes.data, v.ctypes.data, self.stream)
        return k, v

    def step(self, token: int, pos: int, logits=True):
        """One fused decode step; returns the device logits tensor (or None)."""
        ptr = self.logits.data_ptr() if logits else None
        mk.mk_decode_step(self.ctx, int(token), int(pos), ptr, self.stream)
        return self.logits if logits else None

    def step_greedy(self, pos: int, logits=False):
        """One fused step fed with the previous step's argmax (device-resident)."""
        ptr = self.logits.data_ptr() if logits else None
        mk.mk_decode_step_greedy(self.ctx, int(pos), ptr, self.stream)

    def step_sample(self, token: int, pos: int, temperature: float, seed: int, logits=False):
        """One fused step whose next token is sampled at `temperature` (<= 0: greedy);
        token = -1 feeds the previous step's chosen token from device memory."""
        ptr = self.logits.data_ptr() if logits else None
        mk.mk_decode_step_sample(self.ctx, int(token), int(pos), float(temperature), int(seed), ptr, self.stream)
        return self.logits if logits else None

    def set_top_p(self, top_p: float):
        """Nucleus mass of the sampled steps from now on (1 = every token)."""
        mk.mk_set_top_p(self.ctx, float(top_p))

    def prefill(self, tokens, start_pos: int = 0, logits=True):
        """Batched prefill of host tokens at positions start_pos..; returns the device logits of
        the last token (or None).  Needs the decoder built with perop=True (row-major weights)."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        ptr = self.logits.data_ptr() if logits else None
        mk.mk_prefill(self.ctx, t.ctypes.data, t.size, int(start_pos), ptr, self.stream)
        return self.logits if logits else None

    def step_perop(self, token: int, pos: int, logits=True) -> int:
        ptr = self.logits.data_ptr() if logits else None
        return mk.mk_decode_step_perop(self.ctx, int(token), int(pos), ptr, self.stream)

    def get_hidden(self):
        mk.mk_get_hidden(self.ctx, self.hidden.data_ptr(), self.stream)
        return self.hidden

    def get_argmax(self) -> int:
        mk.mk_get_argmax(self.ctx, self.argmax_buf.data_ptr(), self.stream)
        return int(self.argmax_buf.item())

    def generate_greedy(self, prompt, start_pos: int, n_new: int):
        """Host prompt in, host tokens out (one call, n_prompt + n_new - 1 launches)."""
        p = np.ascontiguousarray(prompt, dtype=np.int32)
        out = np.zeros(n_new, dtype=np.int32)
        rc = mk.mk_generate_greedy(self.ctx, p.ctypes.data, p.size, start_pos, n_new, out.ctypes.data, self.stream)
        return rc, out

    def generate(self, prompt, start_pos: int, n_new: int, temperature: float = 0.0, seed: int = 0, eos_id: int = -1):
        """Sampled generation with an optional stop token: (code, tokens with -1 after the stop, count)."""
        p = np.ascontiguousarray(prompt, dtype=np.int32)
        out = np.zeros(n_new, dtype=np.int32)
        n = np.zeros(1, dtype=np.int32)
        rc = mk.mk_generate(self.ctx, p.ctypes.data, p.size, start_pos, n_new, float(temperature), int(seed),
                            int(eos_id), out.ctypes.data, n.ctypes.data, self.stream)
        return rc, out, int(n[0])

    def status(self) -> int:
        return mk.mk_status(self.ctx)

    def set_debug(self, knob: int, value: int):
        mk.mk_set_debug(self.ctx, knob, value)

    def close(self):
        if self.ctx:
            self.torch.cuda.synchronize(self.device)
            mk.mk_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
