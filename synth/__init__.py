"""Seeded synthetic inputs for the bs=1 Llama-style decode workloads.

This module only draws inputs (bf16 weights, norm gains, pre-filled K/V,
token ids) and describes the five workloads.  It holds none of the decode
arithmetic; the CPU oracle and the GPU path both consume what it returns.

Every array is a pure function of (seed, stream id, element index) through the
counter-based generator in ``synth.c``: weights and pre-filled K/V are
``bf16(mean + std * N(0, 1))`` draws, token ids are uniform over the vocab.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into synth/_build/libsynth.so (plain gcc, OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, src, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, u64, d = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
            lib.synth_fill_normal_bf16.argtypes = [ctypes.c_void_p, i64, u64, u64, d, d]
            lib.synth_fill_normal_f32.argtypes = [ctypes.c_void_p, i64, u64, u64, d, d]
            lib.synth_fill_uniform_i32.argtypes = [ctypes.c_void_p, i64, u64, u64, ctypes.c_int32, ctypes.c_int32]
            for f in (lib.synth_fill_normal_bf16, lib.synth_fill_normal_f32, lib.synth_fill_uniform_i32):
                f.restype = None
            _lib = lib
    return _lib


def normal_bf16(shape, seed: int, stream: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of mean + std * N(0,1) draws."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_fill_normal_bf16(out.ctypes.data, out.size, seed, stream, mean, std)
    return out


def normal_f32(shape, seed: int, stream: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().synth_fill_normal_f32(out.ctypes.data, out.size, seed, stream, mean, std)
    return out


def uniform_tokens(n: int, vocab: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_fill_uniform_i32(out.ctypes.data, n, seed, stream, 0, vocab)
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (a.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# Model shapes and workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class ModelShape:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float
    rope_theta: float
    tie_embeddings: bool


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int            # seeds are offset by 100 * index
    shape: ModelShape
    prompt_len: int       # tokens decoded one by one from an empty cache (0 if pre-filled)
    prefill: int          # positions of K/V pre-filled with N(0,1) bf16 (0 if prompt-driven)
    decode: int           # decode steps after the prompt / pre-fill

    @property
    def start_pos(self) -> int:
        return self.prompt_len if self.prompt_len else self.prefill

    def max_seq(self, slack: int = 64) -> int:
        n = self.start_pos + self.decode + slack
        return (n + 63) // 64 * 64

    @property
    def seed_weights(self) -> int:
        return 100 * self.index + 0

    @property
    def seed_tokens(self) -> int:
        return 100 * self.index + 1

    @property
    def seed_kv(self) -> int:
        return 100 * self.index + 2


TINY = ModelShape(2, 256, 4, 2, 64, 688, 1024, 1e-5, 10000.0, False)
LLAMA_1B = ModelShape(16, 2048, 32, 8, 64, 8192, 128256, 1e-5, 500000.0, True)
LLAMA_8B = ModelShape(32, 4096, 32, 8, 128, 14336, 128256, 1e-5, 500000.0, False)

WORKLOADS = {
    "tiny": Workload("tiny", 0, TINY, prompt_len=32, prefill=0, decode=16),
    "1b": Workload("1b", 1, LLAMA_1B, prompt_len=512, prefill=0, decode=256),
    "1b-2k": Workload("1b-2k", 2, LLAMA_1B, prompt_len=0, prefill=2048, decode=128),
    "8b-4k": Workload("8b-4k", 3, LLAMA_8B, prompt_len=0, prefill=4096, decode=128),
    "1b-32k": Workload("1b-32k", 4, LLAMA_1B, prompt_len=0, prefill=32768, decode=64),
    # a 4-layer slice of the 8B shape (vocab 32000): the 8B kernels on about 1-2 GB, for full profiler
    # captures (not a benchmark workload)
    "8b-4l-4k": Workload("8b-4l-4k", 5, dataclasses.replace(LLAMA_8B, n_layers=4, vocab=32000), prompt_len=0,
                         prefill=4096, decode=16),
}

# Stream ids of every drawn tensor.
_S_EMBED, _S_LM_HEAD, _S_FINAL_NORM = 1, 2, 3
_LAYER_KINDS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")
_S_PROMPT, _S_FIRST_TOKEN = 20000, 20001


def _layer_stream(layer: int, kind: str) -> int:
    return 100 + 16 * layer + _LAYER_KINDS.index(kind)


def _kv_stream(layer: int, which: int) -> int:
    return 1_000_000 + 2 * layer + which


def layer_matrix_shapes(s: ModelShape):
    qd, kvd = s.n_q_heads * s.head_dim, s.n_kv_heads * s.head_dim
    return {
        "attn_norm": (s.hidden,), "wq": (qd, s.hidden), "wk": (kvd, s.hidden), "wv": (kvd, s.hidden),
        "wo": (s.hidden, qd), "ffn_norm": (s.hidden,), "w_gate": (s.ffn, s.hidden),
        "w_up": (s.ffn, s.hidden), "w_down": (s.hidden, s.ffn),
    }


def make_model(s: ModelShape, seed: int, std: float = 0.02, gains: str = "ones") -> dict:
    """Random-init bf16 weights of shape ``s`` (numpy uint16 bit patterns, [out, in]).

    Matrices and embeddings are N(0, std).  Norm gains are 1.0 (``gains="ones"``)
    or N(1, 0.1) (``gains="normal"``) so that the gain multiply is exercised.
    """
    shapes = layer_matrix_shapes(s)

    def gain(stream):
        if gains == "ones":
            return np.full((s.hidden,), 0x3F80, dtype=np.uint16)
        return normal_bf16((s.hidden,), seed, stream, 1.0, 0.1)

    m = {"shape": s, "embed": normal_bf16((s.vocab, s.hidden), seed, _S_EMBED, 0.0, std)}
    m["lm_head"] = None if s.tie_embeddings else normal_bf16((s.vocab, s.hidden), seed, _S_LM_HEAD, 0.0, std)
    m["final_norm"] = gain(_S_FINAL_NORM)
    for kind in _LAYER_KINDS:
        m[kind] = []
    for l in range(s.n_layers):
        for kind in _LAYER_KINDS:
            st = _layer_stream(l, kind)
            if kind.endswith("norm"):
                m[kind].append(gain(st))
            else:
                m[kind].append(normal_bf16(shapes[kind], seed, st, 0.0, std))
    return m


def make_kv(s: ModelShape, n_pos: int, seed: int):
    """Pre-filled cache: per layer K and V as bf16 [kv_heads, n_pos, head_dim], N(0, 1).

    K is taken to be already rotated (post-RoPE), as a cache written by earlier
    decode steps would hold it.
    """
    ks, vs = [], []
    for l in range(s.n_layers):
        ks.append(normal_bf16((s.n_kv_heads, n_pos, s.head_dim), seed, _kv_stream(l, 0)))
        vs.append(normal_bf16((s.n_kv_heads, n_pos, s.head_dim), seed, _kv_stream(l, 1)))
    return ks, vs


def make_prompt(w: Workload) -> np.ndarray:
    return uniform_tokens(w.prompt_len, w.shape.vocab, w.seed_tokens, _S_PROMPT)


def make_first_token(w: Workload) -> int:
    return int(uniform_tokens(1, w.shape.vocab, w.seed_tokens, _S_FIRST_TOKEN)[0])


def weight_bytes_per_token(s: ModelShape) -> int:
    """bf16 bytes of every weight the decode step reads once, plus one embedding row."""
    per_layer = sum(int(np.prod(v)) for v in layer_matrix_shapes(s).values())
    return 2 * (s.n_layers * per_layer + s.vocab * s.hidden + s.hidden + s.hidden)


def kv_bytes_read(s: ModelShape, ctx: int) -> int:
    """bf16 K and V bytes attended over at context length ``ctx`` (all layers)."""
    return 2 * s.n_layers * s.n_kv_heads * s.head_dim * ctx * 2
