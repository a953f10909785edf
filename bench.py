#!/usr/bin/env python3
"""Benchmark of the bs=1 decode megakernel (one fused kernel launch per token).

Default workload: the Llama-3.2-1B shape (16 layers, hidden 2048, 32 q / 8 kv
heads, head_dim 64, SwiGLU 8192, vocab 128256, tied embeddings, RoPE theta
500000), random-init bf16 weights N(0, 0.02), a 512-token uniform prompt (run
through the batched prefill, timed on its own), then greedy decode steps at
context lengths 513..768; a timed run longer than 256 steps rewinds to position
512 so every step stays inside that window.

One step = one decode token = one kernel launch: RMSNorm + QKV GEMV + RoPE +
K/V append, GQA attention, O-proj + residual, RMSNorm + gate/up + SiLU + down +
residual for all 16 layers, final RMSNorm, LM-head GEMV and the greedy argmax.

Timing: W untimed warm-up steps, then exactly K steps between a barrier +
cuda.synchronize on both sides, CUDA events on the launching stream around
every step (p50/p99), max over ranks.  Every step streams 2.47 GB of weights,
far more than the 129 MB L2, so no L2 flush is needed between steps.

Multi-GPU (torchrun): bs=1 decode does not shard; each rank runs an independent
replica on its own GPU and `value` is the total tokens/s of all replicas.

--impl reference times the CPU oracle (the plain fp64 C reference) on the host
cores, on the same workload, metric and unit.

For the prompt workloads the line also carries "prefill": the 512-token prompt
through the batched prefill (mk_prefill: tcgen05 GEMMs, tensor-core causal
attention), CUDA-event timed
on its own and against the same prompt as 512 fused decode launches; its
roofline is tensor-bound against the measured bf16 peak.  It also carries
"int8" and "int4": the same decode steps on a weight-only INT8 / INT4 context
(the int8 / int4 build of the fused kernel), CUDA-event timed, each with its
own HBM roofline.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "bs=1 decode tokens/s, ms/token p50/p99; achieved HBM TB/s vs GB300 peak"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="1b", help="tiny | 1b | 1b-2k | 8b-4k | 1b-32k (8b-4l-4k: profiling case)")
    ap.add_argument("--perop", action="store_true", help="time the unfused per-operator baseline instead")
    ap.add_argument("--ring-stages", type=int, default=0)
    ap.add_argument("--slot-kib", type=int, default=0)
    ap.add_argument("--l2-prefetch-kib", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-prefill", action="store_true", help="skip the batched-prefill measurement")
    ap.add_argument("--no-int8", action="store_true", help="skip the weight-only INT8 decode measurement")
    ap.add_argument("--no-int4", action="store_true", help="skip the weight-only INT4 decode measurement")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def dist_barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def dist_max(world: int, x: float, device=None) -> float:
    """Maximum of a host float over all ranks (the whole-job time)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", device) if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(world: int, x: float, device=None) -> float:
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", device) if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(world: int, tokens_this_rank: int, seconds_this_rank: float, device=None):
    """Whole-job throughput: all ranks' tokens over the slowest rank's time."""
    t = dist_max(world, seconds_this_rank, device)
    n = dist_sum(world, tokens_this_rank, device)
    return n / t, t


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while it runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.rows, self.proc, self.gpu = [], None, gpu_index
        self.interval = interval_ms
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", f"-i={self.gpu}",
                 f"-lms={self.interval}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._th = threading.Thread(target=self._read, daemon=True)
        self._th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        lo, hi = (self.t0 or 0) - 0.05, (self.t1 or time.time()) + 0.05
        sel = [r for t, r in self.rows if lo <= t <= hi] or [r for _, r in self.rows[-3:]]
        mhz = [float(r[1]) for r in sel if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in sel if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in sel:
            for k, name in enumerate(names):
                if len(r) > 5 + k and r[5 + k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sel)}


# ------------------------------------------------------------------ helpers

def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return 6800.0, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def measured_bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s bf16 (no MEASURED_PEAKS.json)"


def prefill_flops(s, n: int) -> float:
    """Algorithmic FLOPs of a batched prefill of n tokens: 2 per weight of the
    layer matrices per token, the causal attention (q.k and p.v over the
    positions each row attends, all heads), and the LM head for the last row."""
    per_layer = ((s.n_q_heads + 2 * s.n_kv_heads) * s.head_dim * s.hidden + s.hidden * s.n_q_heads * s.head_dim
                 + 3 * s.ffn * s.hidden)
    attn = 4 * s.n_q_heads * s.head_dim * (n * (n + 1) // 2)
    return float(2 * s.n_layers * per_layer * n + s.n_layers * attn + 2 * s.vocab * s.hidden)


def time_prefill(dec, w, torch, reps: int = 5):
    """CUDA-event time of the batched prefill of the workload's prompt (warm,
    then reps timed calls, each rewriting positions 0..n-1), and of the same
    prompt as one fused decode launch per token."""
    import synth

    prompt = synth.make_prompt(w)
    st = torch.cuda.current_stream()
    for _ in range(2):
        dec.prefill(prompt, 0, logits=False)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        dec.prefill(prompt, 0, logits=False)
    e1.record(st)
    torch.cuda.synchronize()
    pf_ms = e0.elapsed_time(e1) / reps
    e0.record(st)
    rc, _ = dec.generate_greedy(prompt, 0, 1)
    e1.record(st)
    torch.cuda.synchronize()
    assert rc == 0, f"prompt run failed: {rc}"
    dl_ms = e0.elapsed_time(e1)
    dec.prefill(prompt, 0, logits=False)   # leaves the prefill's cache and next token for the decode steps
    torch.cuda.synchronize()
    n = len(prompt)
    fl = prefill_flops(w.shape, n)
    peak, src = measured_bf16_peak()
    achieved = fl / (pf_ms * 1e-3) / 1e12
    return {"prompt_tokens": n, "ms": pf_ms, "tokens_per_s": n / (pf_ms * 1e-3),
            "launches": 9 * w.shape.n_layers + 5,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "peak_source": src,
                         "algorithmic_flops": fl,
                         "tensor_work_tflops": 3 * achieved,
                         "note": "tcgen05 GEMMs (TMA tiles, TMEM accumulators) with each fp32 activation as "
                                 "three bf16 parts: about 3x the tensor work of the algorithmic FLOPs "
                                 "(tensor_work_tflops counts it); causal attention on mma.sync"},
            "decode_launch_prompt_ms": dl_ms, "speedup_vs_decode_launches": dl_ms / pf_ms}


def time_int8(a, w, local, torch, positions, peak, peak_src, bits=8):
    """The same decode steps on a weight-only INT8 (bits = 8) or INT4 (bits = 4)
    context (codes and per-row / per-column fp32 scales streamed, dequantized
    in registers): its context built the way the bf16 one was (pre-filled
    cache, or the prompt as decode launches), then W warm-up and K
    CUDA-event-timed greedy steps at the same positions; roofline against the
    quantized stream's algorithmic bytes."""
    import synth
    from decode_megakernel_05_gb300 import Decoder, mk

    s = w.shape
    max_seq = (w.start_pos + w.decode + 64 + 63) // 64 * 64
    m = synth.make_model(s, w.seed_weights)
    dec = Decoder(m, max_seq, device=local, tuning=mk.tuning(a.ring_stages, a.slot_kib, a.l2_prefetch_kib, 0,
                                                             int(bits == 8), int(bits == 4)))
    tag = f"int{bits}"
    del m
    info = dec.info
    st = torch.cuda.current_stream()
    if w.prefill:
        ks, vs = synth.make_kv(s, w.prefill, w.seed_kv)
        dec.set_kv(ks, vs, w.prefill)
        del ks, vs
        dec.step(synth.make_first_token(w), w.prefill, logits=False)
    else:
        rc, _ = dec.generate_greedy(synth.make_prompt(w), 0, 1)
        assert rc == 0, f"{tag} prompt run failed: {rc}"
    for k in range(a.warmup):
        dec.step_greedy(positions[k])
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps + 1)]
    ev[0].record(st)
    for k in range(a.steps):
        dec.step_greedy(positions[a.warmup + k])
        ev[k + 1].record(st)
    torch.cuda.synchronize()
    assert dec.status() == 0, f"{tag} device status {dec.status()}"
    per = sorted(ev[k].elapsed_time(ev[k + 1]) for k in range(a.steps))
    total_s = ev[0].elapsed_time(ev[-1]) / 1e3
    ctxs = [p + 1 for p in positions[a.warmup:]]
    alg = info.weight_bytes_per_token + info.kv_bytes_per_position * float(np.mean(ctxs))
    achieved = alg / (total_s / a.steps) / 1e9
    dec.close()
    return {"value": a.steps / total_s, "unit": UNIT, "ms_per_token_p50": per[len(per) // 2],
            "ms_per_token_p99": per[min(len(per) - 1, int(round(0.99 * (len(per) - 1))))],
            "gpu_launches": a.steps, "dtype": f"{tag} weights, fp32 arithmetic",
            "weights": f"symmetric absmax {tag} (codes in [-{2 ** (bits - 1) - 1}, {2 ** (bits - 1) - 1}]), "
                       "fp32 scale per output row (per input column for w_down), quantized on the device at load",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_src,
                         "traffic": (load_profile_traffic(a.workload + "_" + tag) or {}).get("dram_bytes_per_launch"),
                         "algorithmic_bytes_per_launch": alg,
                         "kernel": f"mk_decode_kernel, {tag} build (1 launch = 1 token)"}}


KERNEL_SOURCES = ("mk_kernel.cuh", "mk_kernel.cu", "mk_internal.h")


def kernel_source_hash() -> str:
    """sha256 over the fused kernel's source files with their comments and
    blank lines removed (the ncu traffic figure is only valid for the kernel
    it was measured on; a comment does not change the kernel)."""
    import hashlib
    import re

    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "decode_megakernel_05_gb300", "csrc", f)) as fh:
            src = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in src.splitlines())
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()


def load_profile_traffic(workload: str):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary
    (profiles/traffic_<workload>.txt, "key: value" lines), if any, and only if
    it was measured on the kernel sources as they are now."""
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    try:
        out = {}
        for line in open(p):
            if ":" in line and not line.lstrip().startswith("#"):
                k, v = line.split(":", 1)
                out[k.strip()] = v.strip()
        if out.get("kernel_source_sha256") != kernel_source_hash():
            return None
        return {"dram_bytes_per_launch": float(out["dram_bytes_per_launch"]), "kernel": out.get("kernel")}
    except Exception:
        return None


def step_positions(w, warmup: int, steps: int):
    """Positions of warm-up and timed steps: start..start+255, then rewinding."""
    start = w.start_pos
    span = w.decode
    return [start + (k % span) for k in range(warmup + steps)]


def cpu_baseline(w, budget_s: float, ctx_pos: int):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    workload: decode steps of the same model at the same context length, from
    a seeded pre-filled cache (same per-step cost as a prompt-built cache)."""
    import oracle
    import synth

    s = w.shape
    m = synth.make_model(s, w.seed_weights)
    orc = oracle.OracleDecoder(m, ctx_pos + 64)
    ks, vs = synth.make_kv(s, ctx_pos, w.seed_kv + 7)
    orc.set_kv(ks, vs, ctx_pos)
    tok = 1
    times = []
    t_all = time.perf_counter()
    while True:
        t = time.perf_counter()
        lg, _ = orc.step(tok, ctx_pos + len(times))
        times.append(time.perf_counter() - t)
        tok, _ = oracle.argmax_f32(lg)
        if len(times) >= 2 and time.perf_counter() - t_all > budget_s:
            break
        if len(times) >= 64:
            break
    sec = sum(times)
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": len(times) / sec, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(times)} oracle decode steps ({w.name} model, fp64 C + OpenMP) at positions "
                      f"{ctx_pos}..{ctx_pos + len(times) - 1} from a seeded pre-filled cache",
            "ms_per_token_p50": 1e3 * statistics.median(times)}


# ------------------------------------------------------------------ our arm

def run_ours(a, world, rank, local):
    import torch

    import synth
    from decode_megakernel_05_gb300 import Decoder, mk

    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    w = synth.WORKLOADS[a.workload]
    s = w.shape
    max_seq = w.start_pos + w.decode + 64
    max_seq = (max_seq + 63) // 64 * 64
    tun = mk.tuning(a.ring_stages, a.slot_kib, a.l2_prefetch_kib, 0)
    m = synth.make_model(s, w.seed_weights)
    # the row-major weight copies serve the per-operator baseline and the batched prefill
    want_prefill = bool(w.prompt_len) and not a.no_prefill and not a.perop
    dec = Decoder(m, max_seq, device=local, tuning=tun, perop=a.perop or want_prefill)
    del m
    info = dec.info
    stream = torch.cuda.current_stream()
    # context: the prompt (batched prefill, timed on its own; or one decode launch
    # per token, untimed), or a pre-filled cache
    prefill = None
    if w.prefill:
        ks, vs = synth.make_kv(s, w.prefill, w.seed_kv)
        dec.set_kv(ks, vs, w.prefill)
        del ks, vs
        first = synth.make_first_token(w)
        dec.step(first, w.prefill, logits=False)
        pos0 = w.prefill + 1
    elif want_prefill:
        prefill = time_prefill(dec, w, torch)
        pos0 = w.prompt_len
    else:
        prompt = synth.make_prompt(w)
        rc, _ = dec.generate_greedy(prompt, 0, 1)
        assert rc == 0, f"prompt run failed: {rc}"
        pos0 = w.prompt_len
    positions = [pos0 + (k % (w.decode - 1)) for k in range(a.warmup + a.steps)]

    def one(pos):
        if a.perop:   # the per-operator baseline is fed a fixed host token
            return dec.step_perop(1, pos, logits=False)
        dec.step_greedy(pos)
        return 1

    launches_per_step = 1
    for k in range(a.warmup):
        launches_per_step = one(positions[k])
    torch.cuda.synchronize()
    assert dec.status() == 0

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps + 1)]
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    dist_barrier(world, local)
    torch.cuda.synchronize()
    clk.mark("t0")
    ev[0].record(stream)
    for k in range(a.steps):
        one(positions[a.warmup + k])
        ev[k + 1].record(stream)
    torch.cuda.synchronize()
    clk.mark("t1")
    dist_barrier(world, local)
    clk.stop()
    st = dec.status()
    assert st == 0, f"device status {st}"
    per = [ev[k].elapsed_time(ev[k + 1]) for k in range(a.steps)]
    total_s = ev[0].elapsed_time(ev[-1]) / 1e3
    value, t_job = aggregate(world, a.steps, total_s, local)
    per_sorted = sorted(per)
    p50 = per_sorted[len(per) // 2]
    p99 = per_sorted[min(len(per) - 1, int(round(0.99 * (len(per) - 1))))]
    ctxs = [p + 1 for p in positions[a.warmup:]]
    kv_per_pos = info.kv_bytes_per_position
    alg_bytes = info.weight_bytes_per_token + kv_per_pos * float(np.mean(ctxs))
    mean_s = total_s / a.steps
    peak, peak_src = measured_peak()
    achieved = alg_bytes / mean_s / 1e9
    traffic = load_profile_traffic(a.workload) if not a.perop else None

    e2e = None
    if not a.no_e2e and not a.perop:
        # Through the public API with host buffers: every step copies its input
        # token from pinned host memory to the device and reads the generated
        # token back (mk_generate_greedy with one prompt token, one new token).
        tok = torch.zeros(1, dtype=torch.int32).pin_memory()
        out = torch.zeros(1, dtype=torch.int32).pin_memory()
        tok[0] = dec.get_argmax()
        from decode_megakernel_05_gb300 import mk as mkb
        n_e2e = a.steps
        dist_barrier(world, local)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for k in range(n_e2e):
            rc = mkb.mk_generate_greedy(dec.ctx, tok.data_ptr(), 1, positions[a.warmup + k], 1, out.data_ptr(),
                                        dec.stream)
            if rc != 0:
                raise RuntimeError(f"mk_generate_greedy: {rc}")
            tok[0] = out[0]
        t_e2e = time.perf_counter() - t0
        dist_barrier(world, local)
        e2e_val, _ = aggregate(world, n_e2e, t_e2e, local)
        e2e = {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 4,
               "api": "mk_generate_greedy(host prompt of 1 token, 1 new token) per step, pinned buffers"}

    int8 = int4 = None
    if not a.no_int8 and not a.perop:
        dec.close()
        int8 = time_int8(a, w, local, torch, positions, peak, peak_src)
    if not a.no_int4 and not a.perop:
        dec.close()
        int4 = time_int8(a, w, local, torch, positions, peak, peak_src, bits=4)

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        dec.close()
        cpu = cpu_baseline(w, a.cpu_seconds, w.start_pos)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": 1e3 * t_job / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {
                "workload": {"1b": "llama-3.2-1b-shape bs=1 greedy decode, prompt 512, context 513-768",
                             "tiny": "tiny llama-style bs=1 decode (L2-resident)",
                             "1b-2k": "llama-3.2-1b-shape bs=1 decode, KV pre-filled 2048",
                             "8b-4k": "llama-3-8b-shape bs=1 decode, KV pre-filled 4096",
                             "1b-32k": "llama-3.2-1b-shape bs=1 decode, KV pre-filled 32768",
                             "8b-4l-4k": "4-layer slice of the llama-3-8b shape (vocab 32000), KV pre-filled "
                                         "4096: profiling case"}[a.workload],
                "weights": "bf16 random-init N(0,0.02), fp32 activations and accumulation, bf16 KV cache",
                "path": "per-operator baseline" if a.perop else "fused megakernel, 1 launch per token",
                "l2": f"inputs larger than L2: {info.weight_bytes_per_token / 1e9:.2f} GB of weights per step",
                "grid_ctas": info.grid_ctas, "block_threads": info.block_threads, "ring_stages": info.ring_stages,
                "slot_bytes": info.slot_bytes, "l2_prefetch_bytes": info.l2_prefetch_bytes,
                "parallelism": "replicas" if world > 1 else "single GPU",
            },
            "ms_per_token_p50": p50, "ms_per_token_p99": p99,
            "achieved_hbm_tbs": achieved / 1e3,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_src,
                         "traffic": (traffic or {}).get("dram_bytes_per_launch"),
                         "algorithmic_bytes_per_launch": alg_bytes,
                         "kernel": "mk_decode_kernel (the fused step; 1 launch = 1 token)"},
            "gpu_launches": launches_per_step * a.steps,
            "launches_per_token": launches_per_step,
            "clocks": clk.summary(),
        }
        if prefill:
            line["prefill"] = prefill
        if int8:
            line["int8"] = int8
        if int4:
            line["int4"] = int4
        if e2e:
            line["e2e"] = e2e
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm (the oracle)

def run_reference(a, world, rank, local):
    if rank != 0:
        return
    import synth

    w = synth.WORKLOADS[a.workload]
    budget = 150.0
    import oracle

    s = w.shape
    m = synth.make_model(s, w.seed_weights)
    ctx_pos = w.start_pos
    orc = oracle.OracleDecoder(m, ctx_pos + a.warmup + a.steps + 64)
    ks, vs = synth.make_kv(s, ctx_pos, w.seed_kv + 7)
    orc.set_kv(ks, vs, ctx_pos)
    del ks, vs
    tok = 1
    pos = ctx_pos
    t_first = None
    for _ in range(max(1, min(a.warmup, 3))):
        t = time.perf_counter()
        lg, _ = orc.step(tok, pos)
        t_first = time.perf_counter() - t
        tok, _ = oracle.argmax_f32(lg)
        pos += 1
    n = a.steps
    if t_first * a.steps > budget:
        n = max(1, int(budget / t_first))
    times = []
    for _ in range(n):
        t = time.perf_counter()
        lg, _ = orc.step(tok, pos)
        times.append(time.perf_counter() - t)
        tok, _ = oracle.argmax_f32(lg)
        pos += 1
    sec = sum(times)
    value = len(times) / sec
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    sample = (f"{len(times)} of {a.steps} requested decode steps of the CPU oracle (fp64 C + OpenMP) on the "
              f"{w.name} model at positions {ctx_pos + min(a.warmup, 3)}.. from a seeded pre-filled cache")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * sec / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "oracle": "plain fp64 CPU reference"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    a = parse()
    world, rank, local = dist_env()
    if a.impl == "reference":
        run_reference(a, world, rank, local)
    else:
        run_ours(a, world, rank, local)


if __name__ == "__main__":
    main()
