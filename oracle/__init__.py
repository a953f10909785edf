"""CPU oracle for the bs=1 Llama-style decode step (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The product path (the
``decode_megakernel_05_gb300`` package and its CUDA library) never calls it.

Everything is computed in double from the same bf16 weights the GPU path
receives; see oracle.c for the definition and the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p


class _OracleModelC(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
        ("vocab", ctypes.c_int32), ("max_seq", ctypes.c_int32),
        ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
        ("embed", _P), ("lm_head", _P), ("final_norm", _P),
        ("attn_norm", _P), ("wq", _P), ("wk", _P), ("wv", _P), ("wo", _P),
        ("ffn_norm", _P), ("w_gate", _P), ("w_up", _P), ("w_down", _P), ("q8", _P),
    ]


class _OracleQ8C(ctypes.Structure):
    _fields_ = [("q", _P * 7), ("s", _P * 7), ("lm_q", _P), ("lm_s", _P)]

# the int8 matrices in the order of oracle_q8 (w_down's scales are per input column)
Q8_KINDS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc -O2, OpenMP, no fast-math)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fno-fast-math", "-fno-semantic-interposition", "-shared", "-fPIC", "-o", tmp, src, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_round_bf16.argtypes = [ctypes.c_double]
            L.oracle_round_bf16.restype = ctypes.c_uint16
            L.oracle_rmsnorm.argtypes = [_P, _P, ctypes.c_int, ctypes.c_double, _P]
            L.oracle_gemv.argtypes = [_P, ctypes.c_int64, ctypes.c_int64, _P, _P]
            L.oracle_rope.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_double]
            L.oracle_softmax.argtypes = [_P, ctypes.c_int, _P]
            L.oracle_attention_head.argtypes = [_P, _P, _P, ctypes.c_int, ctypes.c_int, _P]
            L.oracle_silu.argtypes = [ctypes.c_double]
            L.oracle_silu.restype = ctypes.c_double
            L.oracle_argmax_f32.argtypes = [_P, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
            L.oracle_argmax_f32.restype = ctypes.c_int
            L.oracle_decode_step.argtypes = [ctypes.POINTER(_OracleModelC), _P, _P, ctypes.c_int, ctypes.c_int, _P, _P]
            L.oracle_decode_step.restype = ctypes.c_int
            L.oracle_quantize_q8.argtypes = [_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _P, _P]
            L.oracle_quantize_q8.restype = None
            L.oracle_quantize_q4.argtypes = [_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _P, _P]
            L.oracle_quantize_q4.restype = None
            L.oracle_gemv_q8.argtypes = [_P, _P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _P, _P]
            L.oracle_gemv_q8.restype = None
            L.oracle_splitmix64_output.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            L.oracle_splitmix64_output.restype = ctypes.c_uint64
            L.oracle_uniform_f32.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int]
            L.oracle_uniform_f32.restype = ctypes.c_float
            L.oracle_gumbel_f32.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int]
            L.oracle_gumbel_f32.restype = ctypes.c_float
            L.oracle_sample_f32.argtypes = [_P, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_int,
                                            ctypes.POINTER(ctypes.c_int)]
            L.oracle_sample_f32.restype = ctypes.c_int
            L.oracle_sample_topp_f32.argtypes = [_P, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_uint64,
                                                 ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
            L.oracle_sample_topp_f32.restype = ctypes.c_int
            for f in (L.oracle_rmsnorm, L.oracle_gemv, L.oracle_rope, L.oracle_softmax, L.oracle_attention_head):
                f.restype = None
            _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ---------------------------------------------------------------- single ops

def bf16_to_double(b: int) -> float:
    return lib().oracle_bf16_to_double(int(b))


def round_bf16(v: float) -> int:
    return lib().oracle_round_bf16(float(v))


def rmsnorm(x, g_bf16, eps: float) -> np.ndarray:
    x, px = _c(x, np.float64)
    g, pg = _c(g_bf16, np.uint16)
    y = np.empty_like(x)
    lib().oracle_rmsnorm(px, pg, x.size, eps, y.ctypes.data)
    return y


def gemv(w_bf16, x) -> np.ndarray:
    w, pw = _c(w_bf16, np.uint16)
    x, px = _c(x, np.float64)
    y = np.empty(w.shape[0], dtype=np.float64)
    lib().oracle_gemv(pw, w.shape[0], w.shape[1], px, y.ctypes.data)
    return y


def rope(v, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, dtype=np.float64, copy=True)
    lib().oracle_rope(v.ctypes.data, v.size, int(pos), float(theta))
    return v


def softmax(s) -> np.ndarray:
    s, ps = _c(s, np.float64)
    p = np.empty_like(s)
    lib().oracle_softmax(ps, s.size, p.ctypes.data)
    return p


def attention_head(q, k_bf16, v_bf16) -> np.ndarray:
    q, pq = _c(q, np.float64)
    k, pk = _c(k_bf16, np.uint16)
    v, pv = _c(v_bf16, np.uint16)
    out = np.empty(q.size, dtype=np.float64)
    lib().oracle_attention_head(pq, pk, pv, k.shape[0], q.size, out.ctypes.data)
    return out


def silu(x: float) -> float:
    return lib().oracle_silu(float(x))


def argmax_f32(logits):
    lg, pl = _c(logits, np.float64)
    nf = ctypes.c_int(0)
    idx = lib().oracle_argmax_f32(pl, lg.size, ctypes.byref(nf))
    return idx, bool(nf.value)


def splitmix64_output(seed: int, i: int) -> int:
    return int(lib().oracle_splitmix64_output(ctypes.c_uint64(seed), ctypes.c_uint64(i)))


def uniform_f32(seed: int, pos: int, v: int) -> float:
    return float(lib().oracle_uniform_f32(ctypes.c_uint64(seed), int(pos), int(v)))


def gumbel_f32(seed: int, pos: int, v: int) -> float:
    return float(lib().oracle_gumbel_f32(ctypes.c_uint64(seed), int(pos), int(v)))


def sample_f32(logits, inv_temp: float, seed: int, pos: int):
    """(token, any non-finite logit): Gumbel-max sample of softmax(logits * inv_temp); inv_temp <= 0 is greedy."""
    lg, pl = _c(logits, np.float64)
    nf = ctypes.c_int(0)
    idx = lib().oracle_sample_f32(pl, lg.size, ctypes.c_float(inv_temp), ctypes.c_uint64(seed), int(pos),
                                  ctypes.byref(nf))
    return idx, bool(nf.value)


def sample_topp_f32(logits, inv_temp: float, top_p: float, seed: int, pos: int):
    """(token, any non-finite logit): Gumbel-max sample of softmax(logits * inv_temp) restricted to
    the nucleus {v : mass of the tokens strictly more probable than v < top_p}; top_p >= 1 keeps all."""
    lg, pl = _c(logits, np.float64)
    nf = ctypes.c_int(0)
    idx = lib().oracle_sample_topp_f32(pl, lg.size, ctypes.c_float(inv_temp), ctypes.c_double(top_p),
                                       ctypes.c_uint64(seed), int(pos), ctypes.byref(nf))
    return idx, bool(nf.value)


def quantize_q8(w_bf16, col_scaled: bool = False):
    """(int8 codes [rows][cols], fp32 scales [rows] or [cols]) of a bf16 matrix (oracle_quantize_q8)."""
    w, pw = _c(w_bf16, np.uint16)
    rows, cols = w.shape
    q = np.empty((rows, cols), dtype=np.int8)
    sc = np.empty(cols if col_scaled else rows, dtype=np.float32)
    lib().oracle_quantize_q8(pw, rows, cols, int(col_scaled), q.ctypes.data, sc.ctypes.data)
    return q, sc


def quantize_q4(w_bf16, col_scaled: bool = False):
    """(int4 codes in [-7, 7], one per int8 [rows][cols]; fp32 scales [rows] or [cols]) of a bf16
    matrix (oracle_quantize_q4)."""
    w, pw = _c(w_bf16, np.uint16)
    rows, cols = w.shape
    q = np.empty((rows, cols), dtype=np.int8)
    sc = np.empty(cols if col_scaled else rows, dtype=np.float32)
    lib().oracle_quantize_q4(pw, rows, cols, int(col_scaled), q.ctypes.data, sc.ctypes.data)
    return q, sc


def gemv_q8(q, scale, x, col_scaled: bool = False) -> np.ndarray:
    q, pq = _c(q, np.int8)
    sc, ps = _c(scale, np.float32)
    x, px = _c(x, np.float64)
    y = np.empty(q.shape[0], dtype=np.float64)
    lib().oracle_gemv_q8(pq, ps, int(col_scaled), q.shape[0], q.shape[1], px, y.ctypes.data)
    return y


def quantize_model_q8(model: dict) -> dict:
    """The oracle's own weight-only INT8 form of a model: per layer and matrix
    kind (codes, scales), and the LM head's (the embedding's when tied)."""
    out = {k: [quantize_q8(w, col_scaled=(k == "w_down")) for w in model[k]] for k in Q8_KINDS}
    out["lm_head"] = quantize_q8(model["embed"] if model["lm_head"] is None else model["lm_head"])
    return out


def quantize_model_q4(model: dict) -> dict:
    """The oracle's weight-only INT4 form of a model, laid out like quantize_model_q8's (codes in
    [-7, 7] held one per int8); OracleDecoder(q8=...) computes with it the same way."""
    out = {k: [quantize_q4(w, col_scaled=(k == "w_down")) for w in model[k]] for k in Q8_KINDS}
    out["lm_head"] = quantize_q4(model["embed"] if model["lm_head"] is None else model["lm_head"])
    return out


# ---------------------------------------------------------------- decode step

class OracleDecoder:
    """The oracle's model + its own bf16 K/V cache [L][kv_heads][max_seq][head_dim]."""

    def __init__(self, model: dict, max_seq: int, q8: dict | None = None):
        """q8: the model's int8 (quantize_model_q8) or int4 (quantize_model_q4) form to compute with
        instead of the bf16 matrices."""
        s = model["shape"]
        self.shape, self.max_seq, self._keep = s, int(max_seq), []
        c = _OracleModelC()
        c.n_layers, c.hidden, c.n_q_heads, c.n_kv_heads = s.n_layers, s.hidden, s.n_q_heads, s.n_kv_heads
        c.head_dim, c.ffn, c.vocab, c.max_seq = s.head_dim, s.ffn, s.vocab, self.max_seq
        c.rms_eps, c.rope_theta = float(s.rms_eps), float(s.rope_theta)

        def ptr(a):
            a = np.ascontiguousarray(a, dtype=np.uint16)
            self._keep.append(a)
            return a.ctypes.data

        def ptrs(lst):
            arr = (ctypes.c_void_p * len(lst))(*[ptr(a) for a in lst])
            self._keep.append(arr)
            return ctypes.cast(arr, ctypes.c_void_p).value

        c.embed = ptr(model["embed"])
        c.lm_head = c.embed if model["lm_head"] is None else ptr(model["lm_head"])
        c.final_norm = ptr(model["final_norm"])
        for name in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"):
            setattr(c, name, ptrs(model[name]))
        c.q8 = None
        if q8 is not None:
            qc = _OracleQ8C()

            def keep(a, dt):
                a = np.ascontiguousarray(a, dtype=dt)
                self._keep.append(a)
                return a.ctypes.data

            def plist(lst):
                arr = (ctypes.c_void_p * len(lst))(*lst)
                self._keep.append(arr)
                return ctypes.cast(arr, ctypes.c_void_p).value

            for i, kind in enumerate(Q8_KINDS):
                qc.q[i] = plist([keep(q, np.int8) for q, _ in q8[kind]])
                qc.s[i] = plist([keep(sc, np.float32) for _, sc in q8[kind]])
            qc.lm_q = keep(q8["lm_head"][0], np.int8)
            qc.lm_s = keep(q8["lm_head"][1], np.float32)
            self._keep.append(qc)
            c.q8 = ctypes.cast(ctypes.pointer(qc), ctypes.c_void_p).value
        self._c = c
        shp = (s.n_layers, s.n_kv_heads, self.max_seq, s.head_dim)
        self.kcache = np.zeros(shp, dtype=np.uint16)
        self.vcache = np.zeros(shp, dtype=np.uint16)

    def set_kv(self, ks, vs, n_pos: int):
        """Pre-fill positions 0..n_pos-1 of every layer (bf16 [kv_heads][n_pos][head_dim])."""
        for l in range(self.shape.n_layers):
            self.kcache[l, :, :n_pos, :] = ks[l]
            self.vcache[l, :, :n_pos, :] = vs[l]

    def step(self, token: int, pos: int):
        """Returns (logits float64 [vocab], hidden float64 [hidden])."""
        s = self.shape
        logits = np.empty(s.vocab, dtype=np.float64)
        hidden = np.empty(s.hidden, dtype=np.float64)
        rc = lib().oracle_decode_step(ctypes.byref(self._c), self.kcache.ctypes.data, self.vcache.ctypes.data,
                                      int(token), int(pos), logits.ctypes.data, hidden.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle_decode_step rejected token={token} pos={pos}")
        return logits, hidden
