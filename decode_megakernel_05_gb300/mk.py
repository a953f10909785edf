"""Thin ctypes binding of the decode megakernel C ABI (include/mk.h).

Every function here marshals arguments and calls the function of the same name
in ``libmk.so``; all computation runs in the library's CUDA kernels.  PyTorch
is used by callers only for device memory and streams: pass ``tensor.data_ptr()``
for device buffers and ``torch.cuda.current_stream().cuda_stream`` for streams.

The library is built in-tree (``decode_megakernel_05_gb300/_build/libmk.so``);
loading raises if it is missing and cannot be built, so no caller can silently
run without it.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MK_OK = 0
MK_ERR_INVALID_ARG = -1
MK_ERR_OOM = -2
MK_ERR_CUDA = -3
MK_ERR_DEVICE_TIMEOUT = -4
MK_ERR_NUMERIC = -5
MK_ERR_STATE = -6
MK_ERR_UNSUPPORTED = -7
MK_DBG_SKIP_ARRIVAL = 1
MK_DBG_WAIT_LIMIT_NS = 2
MK_DBG_TRACE = 3
MK_DBG_TRACE_DETAIL = 5
MK_DBG_INFLIGHT = 6
MK_DBG_INFLIGHT_LAT = 7
MK_DBG_PF_LEAD = 8
MK_DBG_PF_DEPTH = 9
MK_DBG_ATTN_BUILD = 10
MK_DBG_ATTN_TC_MIN = 11
MK_DBG_ATTN_CTAS = 12
MK_DBG_ATTN_POS_PER_CTA = 13
MK_DBG_STREAM_TAIL = 14
MK_DBG_PREFILL_GEMM = 15
MK_NOALLOC_ARGMAX_BLOCKS = 1024
MK_NOALLOC_ARGMAX_MAX_N = MK_NOALLOC_ARGMAX_BLOCKS * 4096

_i32, _i64, _f32, _P = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p


class mk_config(ctypes.Structure):
    _fields_ = [("n_layers", _i32), ("hidden", _i32), ("n_q_heads", _i32), ("n_kv_heads", _i32),
                ("head_dim", _i32), ("ffn", _i32), ("vocab", _i32), ("max_seq", _i32),
                ("rms_eps", _f32), ("rope_theta", _f32), ("tie_embeddings", _i32)]


class mk_tuning(ctypes.Structure):
    _fields_ = [("ring_stages", _i32), ("slot_kib", _i32), ("l2_prefetch_kib", _i32), ("grid_ctas", _i32),
                ("weight_int8", _i32), ("weight_int4", _i32)]


class mk_weights(ctypes.Structure):
    _fields_ = [("embed", _P), ("lm_head", _P), ("final_norm", _P), ("attn_norm", _P), ("wq", _P), ("wk", _P),
                ("wv", _P), ("wo", _P), ("ffn_norm", _P), ("w_gate", _P), ("w_up", _P), ("w_down", _P),
                ("on_device", _i32)]


class mk_info(ctypes.Structure):
    _fields_ = [("grid_ctas", _i32), ("ctas_per_group", _i32), ("block_threads", _i32), ("ring_stages", _i32),
                ("slot_bytes", _i32), ("smem_bytes", _i32), ("sm_count", _i32), ("l2_prefetch_bytes", _i32),
                ("arena_bytes", _i64), ("weight_bytes_per_token", _i64), ("kv_bytes_per_position", _i64),
                ("device_bytes", _i64), ("attn_tc", _i32), ("attn_tc_min_ctx", _i32),
                ("attn_pos_per_cta", _i32), ("weight_int8", _i32), ("weight_int4", _i32)]


# (name, restype, argtypes) of every exported function, in header order.
SIGNATURES = [
    ("mk_create", _i32, [ctypes.POINTER(mk_config), ctypes.POINTER(mk_tuning), ctypes.c_int, ctypes.POINTER(_P)]),
    ("mk_load_weights", _i32, [_P, ctypes.POINTER(mk_weights), _P]),
    ("mk_set_kv", _i32, [_P, _i32, _P, _P, _i32, _P]),
    ("mk_get_kv", _i32, [_P, _i32, _i32, _i32, _P, _P, _P]),
    ("mk_read_arena", _i32, [_P, _i64, _i64, _P, _P]),
    ("mk_decode_step", _i32, [_P, _i32, _i32, _P, _P]),
    ("mk_decode_step_greedy", _i32, [_P, _i32, _P, _P]),
    ("mk_generate_greedy", _i32, [_P, _P, _i32, _i32, _i32, _P, _P]),
    ("mk_decode_step_sample", _i32, [_P, _i32, _i32, ctypes.c_float, ctypes.c_uint64, _P, _P]),
    ("mk_set_top_p", _i32, [_P, ctypes.c_float]),
    ("mk_generate", _i32, [_P, _P, _i32, _i32, _i32, ctypes.c_float, ctypes.c_uint64, _i32, _P, _P, _P]),
    ("mk_get_hidden", _i32, [_P, _P, _P]),
    ("mk_get_argmax", _i32, [_P, _P, _P]),
    ("mk_status", _i32, [_P]),
    ("mk_enable_perop", _i32, [_P, _i32]),
    ("mk_decode_step_perop", _i32, [_P, _i32, _i32, _P, _P, ctypes.POINTER(_i32)]),
    ("mk_prefill", _i32, [_P, _P, _i32, _i32, _P, _P]),
    ("mk_get_info", _i32, [_P, ctypes.POINTER(mk_info)]),
    ("mk_argmax_f32_noalloc", _i32, [_P, _i32, _P, _P]),
    ("mk_set_debug", _i32, [_P, _i32, _i64]),
    ("mk_strerror", ctypes.c_char_p, [ctypes.c_int]),
    ("mk_last_cuda_error", ctypes.c_char_p, []),
    ("mk_destroy", None, [_P]),
    ("mk_arena_bytes", _i64, [ctypes.POINTER(mk_config), ctypes.POINTER(mk_tuning), _i32]),
    ("mk_relayout_host", _i32, [ctypes.POINTER(mk_config), ctypes.POINTER(mk_tuning), _i32,
                                ctypes.POINTER(mk_weights), _P]),
]

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Loads libmk.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing")
            lib = ctypes.CDLL(path)
            for name, res, args in SIGNATURES:
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


class MkError(RuntimeError):
    def __init__(self, code: int, what: str):
        lib = load()
        msg = lib.mk_strerror(code).decode()
        detail = lib.mk_last_cuda_error().decode() if code == MK_ERR_CUDA else ""
        super().__init__(f"{what} failed: {msg} ({code}) {detail}".rstrip())
        self.code = code


def check(code: int, what: str) -> int:
    if code != MK_OK:
        raise MkError(code, what)
    return code


def config_from_shape(shape, max_seq: int) -> mk_config:
    return mk_config(shape.n_layers, shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.ffn,
                     shape.vocab, max_seq, shape.rms_eps, shape.rope_theta, int(shape.tie_embeddings))


def tuning(ring_stages=0, slot_kib=0, l2_prefetch_kib=0, grid_ctas=0, weight_int8=0, weight_int4=0) -> mk_tuning:
    return mk_tuning(ring_stages, slot_kib, l2_prefetch_kib, grid_ctas, int(weight_int8), int(weight_int4))


class _PtrTable:
    """Keeps ctypes pointer arrays alive for an mk_weights struct."""

    def __init__(self):
        self.keep = []

    def arr(self, ptrs):
        a = (_P * len(ptrs))(*ptrs)
        self.keep.append(a)
        return ctypes.cast(a, _P)


def weights_struct(ptrs: dict, on_device: bool):
    """ptrs: name -> int pointer (or list of int pointers for per-layer names)."""
    t = _PtrTable()
    w = mk_weights()
    w.embed = ptrs["embed"]
    w.lm_head = ptrs.get("lm_head")
    w.final_norm = ptrs["final_norm"]
    for name in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"):
        setattr(w, name, t.arr(ptrs[name]))
    w.on_device = int(on_device)
    return w, t


# ------------------------------------------------------------------ same-name wrappers

def mk_create(cfg: mk_config, tun: mk_tuning | None = None, device: int = 0) -> int:
    out = _P()
    check(load().mk_create(ctypes.byref(cfg), ctypes.byref(tun) if tun else None, device, ctypes.byref(out)),
          "mk_create")
    return out.value


def mk_load_weights(ctx: int, w: mk_weights, stream: int = 0) -> None:
    check(load().mk_load_weights(ctx, ctypes.byref(w), stream), "mk_load_weights")


def mk_set_kv(ctx: int, layer: int, k_ptr: int, v_ptr: int, n_pos: int, stream: int = 0) -> None:
    check(load().mk_set_kv(ctx, layer, k_ptr, v_ptr, n_pos, stream), "mk_set_kv")


def mk_get_kv(ctx: int, layer: int, pos0: int, n_pos: int, k_out: int, v_out: int, stream: int = 0) -> None:
    check(load().mk_get_kv(ctx, layer, pos0, n_pos, k_out, v_out, stream), "mk_get_kv")


def mk_read_arena(ctx: int, offset: int, nbytes: int, out_ptr: int, stream: int = 0) -> None:
    check(load().mk_read_arena(ctx, offset, nbytes, out_ptr, stream), "mk_read_arena")


def mk_decode_step(ctx: int, token: int, pos: int, logits_ptr: int | None, stream: int = 0) -> None:
    check(load().mk_decode_step(ctx, token, pos, logits_ptr, stream), "mk_decode_step")


def mk_decode_step_greedy(ctx: int, pos: int, logits_ptr: int | None, stream: int = 0) -> None:
    check(load().mk_decode_step_greedy(ctx, pos, logits_ptr, stream), "mk_decode_step_greedy")


def mk_generate_greedy(ctx: int, prompt_ptr: int, n_prompt: int, start_pos: int, n_new: int, out_ptr: int,
                       stream: int = 0) -> int:
    """Returns the library's code (MK_OK or a latched device status) without raising."""
    return load().mk_generate_greedy(ctx, prompt_ptr, n_prompt, start_pos, n_new, out_ptr, stream)


def mk_decode_step_sample(ctx: int, token: int, pos: int, temperature: float, seed: int, logits_ptr: int | None,
                          stream: int = 0) -> None:
    check(load().mk_decode_step_sample(ctx, token, pos, temperature, seed, logits_ptr, stream), "mk_decode_step_sample")


def mk_set_top_p(ctx: int, top_p: float) -> None:
    check(load().mk_set_top_p(ctx, top_p), "mk_set_top_p")


def mk_generate(ctx: int, prompt_ptr: int, n_prompt: int, start_pos: int, n_new: int, temperature: float, seed: int,
                eos_id: int, out_ptr: int, n_out_ptr: int | None, stream: int = 0) -> int:
    """Returns the library's code (MK_OK or a latched device status) without raising."""
    return load().mk_generate(ctx, prompt_ptr, n_prompt, start_pos, n_new, temperature, seed, eos_id, out_ptr,
                              n_out_ptr, stream)


def mk_get_hidden(ctx: int, out_ptr: int, stream: int = 0) -> None:
    check(load().mk_get_hidden(ctx, out_ptr, stream), "mk_get_hidden")


def mk_get_argmax(ctx: int, out_ptr: int, stream: int = 0) -> None:
    check(load().mk_get_argmax(ctx, out_ptr, stream), "mk_get_argmax")


def mk_status(ctx: int) -> int:
    return load().mk_status(ctx)


def mk_enable_perop(ctx: int, keep_rowmajor: bool = True) -> None:
    check(load().mk_enable_perop(ctx, int(keep_rowmajor)), "mk_enable_perop")


def mk_prefill(ctx: int, tokens_ptr: int, n: int, start_pos: int, logits_ptr: int | None, stream: int = 0) -> None:
    check(load().mk_prefill(ctx, tokens_ptr, n, start_pos, logits_ptr, stream), "mk_prefill")


def mk_decode_step_perop(ctx: int, token: int, pos: int, logits_ptr: int | None, stream: int = 0) -> int:
    n = _i32(0)
    check(load().mk_decode_step_perop(ctx, token, pos, logits_ptr, stream, ctypes.byref(n)), "mk_decode_step_perop")
    return n.value


def mk_get_info(ctx: int) -> mk_info:
    info = mk_info()
    check(load().mk_get_info(ctx, ctypes.byref(info)), "mk_get_info")
    return info


def mk_argmax_f32_noalloc(logits_ptr: int, n: int, out_ptr: int, stream: int = 0) -> int:
    """Greedy token of n device fp32 logits into out_ptr (device int32) with no
    allocation; returns the library's code without raising."""
    return load().mk_argmax_f32_noalloc(logits_ptr, n, out_ptr, stream)


def mk_set_debug(ctx: int, knob: int, value: int) -> None:
    check(load().mk_set_debug(ctx, knob, value), "mk_set_debug")


def mk_strerror(code: int) -> str:
    return load().mk_strerror(code).decode()


def mk_destroy(ctx: int) -> None:
    load().mk_destroy(ctx)


def mk_arena_bytes(cfg: mk_config, tun: mk_tuning | None, grid_ctas: int) -> int:
    return load().mk_arena_bytes(ctypes.byref(cfg), ctypes.byref(tun) if tun else None, grid_ctas)


def mk_relayout_host(cfg: mk_config, tun: mk_tuning | None, grid_ctas: int, w: mk_weights, arena_ptr: int) -> None:
    check(load().mk_relayout_host(ctypes.byref(cfg), ctypes.byref(tun) if tun else None, grid_ctas, ctypes.byref(w),
                                  arena_ptr), "mk_relayout_host")
