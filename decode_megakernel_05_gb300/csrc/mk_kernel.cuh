#pragma once
// mk_kernel.cuh - the persistent bs=1 decode megakernel (one launch per token).
//
// One CTA per SM (grid = n_kv_heads * floor(SMs / n_kv_heads)).  Each CTA has
//   - MK_NCW (12) consumer warps that run the segments of every layer,
//   - a producer warp that streams the CTA's pre-laid-out weight tiles (and its
//     share of the KV cache) into a ring of shared-memory slots with bulk
//     asynchronous copies, guarded by full/empty mbarriers, so tile k+1..k+S
//     load while tile k is consumed (the in-kernel prefetch loop of
//     cloud.baidu.com/article/9434380, section 5, step 3),
//   - a prefetch warp that walks the same tile stream further ahead and asks
//     L2 to fetch it, so HBM keeps streaming while consumers wait on a flag.
// Weights do not depend on activations, so the producer never waits on a
// flag: it runs ahead through segment and layer boundaries, which is what keeps
// the weight stream from stalling at the points where a per-operator framework
// ends one kernel and starts the next (same page, section 4.1).
//
// Segment boundaries are inter-CTA flags (counters in global memory, release
// increments and acquire polls, every wait bounded by %globaltimer):
//   A[l][g]: query/key/value rows of KV group g written (the group's CTAs)
//   B[l][g]: attention partials of group g written       (the group's CTAs)
//   C[l]   : attention block added into the residual      (all CTAs)
//   E[l]   : FFN block added into the residual            (all CTAs)
// Per layer: segment A (RMSNorm + QKV GEMV + RoPE + K/V append) -> A ->
// segment B (split-K GQA attention -> B -> combine + O-proj split by KV group,
// atomically added to the residual) -> C -> segment C (RMSNorm + gate/up GEMV +
// SiLU*up, then the down projection split over the FFN dimension, atomically
// added to the residual) -> E.  After the last layer: RMSNorm, LM-head GEMV,
// greedy argmax (packed 64-bit atomicMax), and the last CTA to finish resets
// the flags for the next launch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mk_internal.h"

// Building with -DMK_NO_TRACE compiles the segment/tile trace out entirely.
#ifdef MK_NO_TRACE
#define MK_TRACE_ON false
#else
#define MK_TRACE_ON true
#endif

namespace mk {
namespace {  // internal linkage: every kernel variant is its own translation unit

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b, uint32_t count = 1) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
// Waits (suspended, up to a hint of 20 us per call) for the phase of the
// given parity to complete; returns false when the hint ran out first.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}
// Bulk copy global -> shared completing on an mbarrier.  The L2 policy marks
// the lines evict-first: every byte streamed here is read once per step, so
// consumed lines should leave L2 before lines prefetched for later tiles.
// Non-blocking: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(smem_u32(b)), "r"(parity)
                 : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Vector fp32 reduction into global memory (no return value).
__device__ __forceinline__ void red_add_v4(float* p, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}
// Tagged words: fp32 value in the low half, the launch tag in the high half.
// A naturally aligned 64-bit access is single-copy atomic, so a reader that
// sees this launch's tag in a word also sees the value written with it.
__device__ __forceinline__ uint64_t ll_pack(float v, uint32_t tag) {
    return ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(v);
}
__device__ __forceinline__ void st_ll(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_ll2(uint64_t* p, uint64_t a, uint64_t b) {
    asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ ulonglong2 ld_ll2(const uint64_t* p) {
    ulonglong2 r;
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(r.x), "=l"(r.y) : "l"(p) : "memory");
    return r;
}
__device__ __forceinline__ bool ll_ok(const ulonglong2 w, uint32_t tag) {
    return ((uint32_t)(w.x >> 32) == tag) & ((uint32_t)(w.y >> 32) == tag);
}

// Barrier over the consumer threads that also ORs a per-thread flag: every
// participant gets the same answer, so an abort decision is uniform.
__device__ __forceinline__ bool bar_or(bool f) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 q, %1, 0; bar.red.or.pred p, 1, %2, q; selp.u32 %0, 1, 0, p; }"
        : "=r"(r)
        : "r"((uint32_t)f), "n"(MK_NCT)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }
// A shared-memory value re-read where it is used (volatile: not kept in a
// register across the code in between).
__device__ __forceinline__ int ldv(const int& x) { return *reinterpret_cast<const volatile int*>(&x); }

// 8 bf16 (one 16-byte chunk, lower address first) -> fp32
__device__ __forceinline__ void unpack8(const uint4 w, float f[8]) {
    f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xFFFF0000u);
    f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xFFFF0000u);
    f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xFFFF0000u);
}
__device__ __forceinline__ float dot8(const uint4 w, const float* x) {
    float f[8];
    unpack8(w, f);
    float a = f[0] * x[0];
#pragma unroll
    for (int e = 1; e < 8; ++e) a = fmaf(f[e], x[e], a);
    return a;
}
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32, one MUFU
// instruction; relative error about 2^-22): the softmax weights only.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// ------------------------------------------------------------------ shared state

// Work split of a warp-row GEMV phase (O-proj, LM head), computed once per
// launch: the tile count, rows per lane group and pass, warps per group, and
// each warp's group and index in it (the divisions stay out of the layer loop).
struct GemvCfg {
    int16_t ntiles, rw, wpg, ngrp;
    int8_t grp[MK_NCW], wg[MK_NCW];
};

struct Misc {                // lives at geo.off_misc (MK_MISC_BYTES)
    int abort;               // CTA-local: consumers gave up (producers stop)
    int token;
    int par;
    int is_last;
    float xscale;            // int8 build: scale of the digits in xv (mk_xdigits)
    unsigned long long copy_bytes;  // bytes issued by the copy producer (paces the L2 prefetcher)
    uint32_t pf_sink;               // the L2 warmer's xor of what it loaded (keeps the loads)
    unsigned long long cwait;       // trace: ns thread 0 spent waiting for ring data
    float alpha[8];          // per head: 1 / (sum of the combine weights)
    float best_val[64];
    int best_idx[64];
    uint32_t tile_bytes[16]; // bytes of the tile in each ring slot (schedule check)
    int slot_tile[16];       // index (in the step's tile stream) of the tile each slot holds
    int streaming;           // consumers are in a streaming segment (sets the producer's in-flight limit)
    uint32_t tag;            // this launch's tag for tagged words (sequence number + 1)
    MkCtaPlan plan;          // this CTA's plan (read from here: keeps registers free in the layer loop)
    // per-CTA constants of the step, read where used (not held in registers
    // across the layer loop): the attention share [ka, ke) + current position
    // (mk_attn_share), whether this CTA runs the attention, the residual rows
    // [dr0, dr1) it adds in the down projection
    int ka, ke, has_cur, att, dr0, dr1;
    GemvCfg ocfg, lmcfg;     // work split of the O-proj and LM-head phases
    float cwt[MK_MAX_CPG_G]; // attention-combine weights [CPG][G]
    float cl[MK_MAX_CPG_G];  // attention partial sums l [CPG][G]
    uint4 stage[32];         // K and V rows of the current position (2 * hd bf16)
    uint4 zrow;              // 16 zero bytes: the rows past a block's end in the tensor-core attention
};
static_assert(sizeof(Misc) <= MK_MISC_BYTES, "misc area");

// Dynamic shared memory of the kernel; Smem names its regions.  Each region's
// address is computed where it is used, from the offset in the kernel
// parameters (a constant-bank operand), instead of 13 pointers held in
// registers for the whole launch.
extern __shared__ __align__(1024) uint8_t mk_dsmem[];
struct Smem {
    const MkGeom* g;   // the kernel parameters' geometry
    __device__ __forceinline__ uint8_t* ring() const { return mk_dsmem; }
    __device__ __forceinline__ uint64_t* full() const { return reinterpret_cast<uint64_t*>(mk_dsmem + g->off_full); }
    __device__ __forceinline__ uint64_t* empty() const { return reinterpret_cast<uint64_t*>(mk_dsmem + g->off_empty); }
    __device__ __forceinline__ float* xv() const { return reinterpret_cast<float*>(mk_dsmem + g->off_xv); }            // [H]
    __device__ __forceinline__ float* ov() const { return reinterpret_cast<float*>(mk_dsmem + g->off_ov); }            // [G*hd]
    // [rows][NKB] column-block partial sums of the QKV / gate-up rows
    __device__ __forceinline__ float* part() const { return reinterpret_cast<float*>(mk_dsmem + g->off_part); }
    __device__ __forceinline__ float* u() const { return reinterpret_cast<float*>(mk_dsmem + g->off_u); }              // [max_nj] SiLU(gate)*up
    // raw residual of this CTA's O rows (group 0 only)
    __device__ __forceinline__ float* xres() const { return reinterpret_cast<float*>(mk_dsmem + g->off_xres); }
    // raw residual of rows split(H, nC, c)
    __device__ __forceinline__ float* xres2() const { return reinterpret_cast<float*>(mk_dsmem + g->off_xres2); }
    // cos[hd/2], sin[hd/2] at this position
    __device__ __forceinline__ float* rope() const { return reinterpret_cast<float*>(mk_dsmem + g->off_rope); }
    __device__ __forceinline__ float* red() const { return reinterpret_cast<float*>(mk_dsmem + g->off_red); }          // [2][MK_NCT]
    // attention (m, l) per position group and head: [2][PPP][G]
    __device__ __forceinline__ float* sc() const { return reinterpret_cast<float*>(mk_dsmem + g->off_sc); }
    __device__ __forceinline__ Misc* misc() const { return reinterpret_cast<Misc*>(mk_dsmem + g->off_misc); }
};

// Segment trace (off unless MkParams::trace is set): thread 0 of the consumers
// stamps %globaltimer at the end of each segment.
#define MK_TRACE(slot_)                                                                  \
    do {                                                                                  \
        if (MK_TRACE_ON && p.trace && threadIdx.x == 0)                                                  \
            p.trace[(size_t)blockIdx.x * MK_TRACE_STRIDE + (slot_)] = gtimer();           \
    } while (0)

// Detail marks (trace with detail only): slot 1600 + 16*layer + (ev_), thread 0's
// time (detail 2: its SM clock instead, and no per-tile records), for the first 24 layers.
#define MK_TRACE_D(l_, ev_)                                                              \
    do {                                                                                  \
        if (MK_TRACE_ON && p.trace && p.trace_detail && threadIdx.x == 0 && (l_) < 24)    \
            p.trace[(size_t)blockIdx.x * MK_TRACE_STRIDE + 1600 + 16 * (l_) + (ev_)] =     \
                p.trace_detail == 2 ? (unsigned long long)clock64() : gtimer();             \
    } while (0)

// Per-phase consumer ring-wait (trace only): slot 1024 + 8*layer + phase.
#define MK_TRACE_CWAIT(slot_)                                                            \
    do {                                                                                  \
        if (MK_TRACE_ON && p.trace && threadIdx.x == 0) {                                                \
            p.trace[(size_t)blockIdx.x * MK_TRACE_STRIDE + 1024 + (slot_)] = s.misc()->cwait; \
            s.misc()->cwait = 0;                                                            \
        }                                                                                 \
    } while (0)

// ------------------------------------------------------------------ waits

__device__ bool wait_counter(const MkParams& p, const uint32_t* ctr, uint32_t target) {
    uint64_t t0 = gtimer();
    uint32_t it = 0;
    while (ld_acquire(ctr) < target) {
        if ((++it & 15u) == 0) {
            if (*(volatile uint32_t*)p.status & MK_ST_ABORT) return false;
            if (gtimer() - t0 > (uint64_t)p.wait_limit_ns) {
                atomicOr(p.status, MK_ST_TIMEOUT | MK_ST_ABORT);
                return false;
            }
        }
    }
    return true;
}

__device__ bool wait_mbar(const MkParams& p, uint64_t* b, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(b, parity)) return true;
    uint64_t t0 = gtimer();
    while (!mbar_try_wait(b, parity)) {
        if (*abort) return false;
        if (gtimer() - t0 > (uint64_t)p.wait_limit_ns) {
            atomicOr(p.status, MK_ST_TIMEOUT | MK_ST_ABORT);
            *abort = 1;
            return false;
        }
    }
    return true;
}

// Between polls of tagged words: false (and the abort bit, and on time-out the
// timeout bit) when the wait must end.  t0 = 0 on the first call.  The abort
// bit (a global load, an L2 round trip) is read on every 8th call only.
__device__ __forceinline__ bool ll_backoff(const MkParams& p, uint64_t& t0) {
    if ((t0 & 7u) == 7u && (*(volatile uint32_t*)p.status & MK_ST_ABORT)) return false;
    const uint64_t now = gtimer() | 1u;   // never 0: t0 == 0 marks the first call
    if (t0 == 0) {
        t0 = now & ~7ull;   // the low 3 bits count calls
    } else {
        if (now - t0 > (uint64_t)p.wait_limit_ns) {
            atomicOr(p.status, MK_ST_TIMEOUT | MK_ST_ABORT);
            return false;
        }
        t0 = (t0 & ~7ull) | ((t0 + 1u) & 7ull);
    }
    __nanosleep(64);
    return true;
}
// Reads 8 tagged words (16-byte aligned) once all carry `tag`.
__device__ __forceinline__ bool ll_read8(const MkParams& p, const uint64_t* src, uint32_t tag, float v[8]) {
    uint64_t t0 = 0;
    for (;;) {
        const ulonglong2 a = ld_ll2(src), b = ld_ll2(src + 2), c = ld_ll2(src + 4), d = ld_ll2(src + 6);
        if (ll_ok(a, tag) & ll_ok(b, tag) & ll_ok(c, tag) & ll_ok(d, tag)) {
            v[0] = __uint_as_float((uint32_t)a.x); v[1] = __uint_as_float((uint32_t)a.y);
            v[2] = __uint_as_float((uint32_t)b.x); v[3] = __uint_as_float((uint32_t)b.y);
            v[4] = __uint_as_float((uint32_t)c.x); v[5] = __uint_as_float((uint32_t)c.y);
            v[6] = __uint_as_float((uint32_t)d.x); v[7] = __uint_as_float((uint32_t)d.y);
            return true;
        }
        if (!ll_backoff(p, t0)) return false;
    }
}

// Arrive on a flag counter (thread 0 of the consumers, after a consumer barrier).
__device__ __forceinline__ void arrive(const MkParams& p, int idx, int sync_id) {
    if (p.dbg_skip_sync == sync_id && p.dbg_skip_cta == (int)blockIdx.x) return;
    // release: cumulative over the CTA's writes ordered before it by the consumer barrier
    red_release_add(p.cnt + idx, 1u);
}

// ------------------------------------------------------------------ tile stream

// The tile walk (mk_walk_tiles) lives in mk_internal.h so the host can check it.
template <class F>
__device__ __forceinline__ void walk_tiles(const MkParams& p, const MkCtaPlan& pl, F&& f) {
    mk_walk_tiles(p.geo, pl, p.arena, p.kc, p.vc, p.pos, p.attn_ctas, f);
}

__device__ void producer_copy(const MkParams& p, const MkCtaPlan& pl, const Smem& s) {
    volatile int* abort = &s.misc()->abort;
    const int ns = p.geo.ns;
    const uint32_t slot_bytes = (uint32_t)p.geo.slot;
    const uint64_t pol = l2_evict_first_policy();
    uint32_t k = 0;
    bool stop = false;
    unsigned long long pwait = 0;
    unsigned long long* tr = (MK_TRACE_ON && p.trace && p.trace_detail == 1) ? p.trace + (size_t)blockIdx.x * MK_TRACE_STRIDE : nullptr;
    const uint32_t lim_s = (uint32_t)(p.inflight < ns ? p.inflight : ns);
    const uint32_t lim_l = (uint32_t)(p.inflight_lat < ns ? p.inflight_lat : ns);
    uint32_t slot = 0, ph = 0;   // k mod ns and floor(k / ns) mod 2, kept incrementally
    walk_tiles(p, pl, [&](const void* src, uint32_t bytes) {
        if (stop) return;
        const uint64_t tw = tr ? gtimer() : 0;
        // at most lim copies in flight: tile k - lim has landed (its slot is
        // not reused before tile k + ns - lim, so the parity is unambiguous).
        // Few bytes in flight while the consumers are latency-bound keep the
        // queues short for their flag polls and activation loads.
        const uint32_t lim = *(volatile int*)&s.misc()->streaming ? lim_s : lim_l;
        if (lim < (uint32_t)ns && k >= lim) {
            const bool wrap = slot < lim;   // tile k - lim sits in the previous round of slots
            const uint32_t s2 = wrap ? slot + ns - lim : slot - lim, ph2 = wrap ? ph ^ 1u : ph;
            if (!wait_mbar(p, &s.full()[s2], ph2, abort)) { stop = true; return; }
        }
        if (!wait_mbar(p, &s.empty()[slot], ph ^ 1u, abort)) { stop = true; return; }
        if (tr) {
            pwait += gtimer() - tw;
            if ((k & 15u) == 0 && (k >> 4) < 64) tr[1536 + (k >> 4)] = pwait;
        }
        s.misc()->tile_bytes[slot] = bytes;
        *(volatile int*)&s.misc()->slot_tile[slot] = (int)k;
        if (tr && k < 512) tr[2560 + k] = gtimer();   // trace: issue time of tile k
        mbar_expect_tx(&s.full()[slot], bytes);
        bulk_g2s(s.ring() + (size_t)slot * slot_bytes, src, bytes, &s.full()[slot], pol);
        ++k;
        if (++slot == (uint32_t)ns) { slot = 0; ph ^= 1u; }
        *(volatile unsigned long long*)&s.misc()->copy_bytes += bytes;
    });
    if (tr) tr[1535] = gtimer();
    // Drain: wait for the copies still in flight before this warp leaves.
    const uint32_t first = k > (uint32_t)ns ? k - ns : 0u;
    for (uint32_t q = first; q < k; ++q) {
        uint64_t t0 = gtimer();
        while (!mbar_try_wait(&s.full()[q % ns], (q / ns) & 1u)) {
            if (gtimer() - t0 > (uint64_t)p.wait_limit_ns) {
                atomicOr(p.status, MK_ST_TIMEOUT | MK_ST_ABORT);
                break;
            }
        }
    }
}

// L2 warmer (the whole prefetch warp): walks the same tile stream as the copy
// producer and brings tiles' 128-byte lines into L2 with one plain 4-byte load
// per line, so the copy later reads L2 instead of HBM.  (Measured: a plain
// load per line leaves the whole line in L2 for a later bulk copy;
// prefetch.global.L2 and non-coherent loads do so only in part.)  It leaves
// the first pf_lead_bytes past the copy cursor alone -- the ring fetches those
// as soon as consumers free slots -- and warms at most l2_pf_bytes beyond
// them.  It works only while the consumers are latency-bound, when HBM is
// otherwise idle, with pf_depth tiles of warming loads in flight.
__device__ void producer_prefetch(const MkParams& p, const MkCtaPlan& pl, const Smem& s) {
    if (p.l2_pf_bytes <= 0) return;
    const int lane = threadIdx.x & 31;
    volatile int* abort = &s.misc()->abort;
    const unsigned long long ahead = (unsigned long long)p.l2_pf_bytes;
    const unsigned long long lead = (unsigned long long)p.pf_lead_bytes;
    const bool two = p.pf_depth > 1;
    unsigned long long issued = 0;
    uint32_t sink = 0, prev = 0, kw = 0;
    bool stop = false;
    unsigned long long* tr = (MK_TRACE_ON && p.trace && p.trace_detail && lane == 0)
                                 ? p.trace + (size_t)blockIdx.x * MK_TRACE_STRIDE : nullptr;
    walk_tiles(p, pl, [&](const void* src, uint32_t bytes) {
        if (stop) return;
        uint64_t t0 = 0;
        const uint32_t kt = kw++;
        for (;;) {
            const unsigned long long cb = *(volatile unsigned long long*)&s.misc()->copy_bytes;
            const bool streaming = *(volatile int*)&s.misc()->streaming;
            if (issued + bytes <= cb + lead) break;   // copied, or the ring fetches it next
            if (!streaming && issued <= cb + lead + ahead) {
                if (tr && kt < 256) tr[1792 + kt] = gtimer();   // trace: when tile kt was warmed
                const char* b = reinterpret_cast<const char*>(src);
                uint32_t acc = 0;
                for (uint32_t off = (uint32_t)lane * 128u; off < bytes; off += 32u * 128u) {
                    uint32_t v;
                    asm volatile("ld.global.b32 %0, [%1];" : "=r"(v) : "l"(b + off) : "memory");
                    acc ^= v;
                }
                // consumed in order with the loads: with depth 1 the next tile's
                // loads wait for these, with depth 2 for the previous tile's
                if (two) {
                    asm volatile("xor.b32 %0, %0, %1;" : "+r"(sink) : "r"(prev));
                    prev = acc;
                } else {
                    asm volatile("xor.b32 %0, %0, %1;" : "+r"(sink) : "r"(acc));
                }
                break;
            }
            if (*abort) { stop = true; return; }
            if (t0 == 0) t0 = gtimer();
            else if (gtimer() - t0 > (uint64_t)p.wait_limit_ns) { stop = true; return; }
            __nanosleep(256);
        }
        issued += bytes;
    });
    asm volatile("xor.b32 %0, %0, %1;" : "+r"(sink) : "r"(prev));
    // a real use of every loaded word: without it the compiler may drop the
    // xors and with them the loads (or the waits for them)
    if (lane == 0) *(volatile uint32_t*)&s.misc()->pf_sink = sink;
}

// ------------------------------------------------------------------ consumer pieces

// Consumer-side cursor over the ring.
struct Ring {
    uint32_t k = 0;
    uint32_t sp = 0;   // slot k mod ns (low 16 bits) and phase floor(k / ns) mod 2 (bit 16), kept incrementally
    // trace only (lane 0 of each warp): ns spent taking tiles, between take
    // and release, and releasing
    unsigned long long t_take = 0, t_comp = 0, t_rel = 0, t_mark = 0;
    __device__ __forceinline__ uint32_t slot() const { return sp & 0xFFFFu; }
    __device__ __forceinline__ uint32_t ph() const { return sp >> 16; }
    // next tile (no division: slot and phase wrap by comparison)
    __device__ __forceinline__ void advance(int ns) {
        ++k;
        sp = ((sp & 0xFFFFu) + 1u == (uint32_t)ns) ? ((sp ^ 0x10000u) & 0x10000u) : sp + 1u;
    }
};

// Ring protocol.  Tile k of the step's stream lives in slot k % ns.  A warp
// that reads tile k first waits until the producer has claimed the slot for
// tile k (slot_tile), then for the slot's full barrier (the parity is then
// unambiguous even if the warp skipped earlier tiles), reads it, and arrives
// on the slot's empty barrier with weight MK_NCW / (number of warps reading
// the tile), so the barrier completes exactly when every reader is done.  Warps
// that do not read a tile only advance their cursor.
__device__ __forceinline__ bool take_tile(const MkParams& p, const Smem& s, Ring& rg, uint32_t expect_bytes,
                                          const uint8_t*& tile) {
    const uint32_t slot = rg.slot(), ph = rg.ph();
    bool ok = true;
    if ((threadIdx.x & 31) == 0) {
        const uint64_t tw = (MK_TRACE_ON && p.trace && p.trace_detail == 1) ? gtimer() : 0;
        ok = !s.misc()->abort;
        if (ok && *(volatile int*)&s.misc()->slot_tile[slot] != (int)rg.k) {
            const uint64_t t0 = gtimer();
            while (*(volatile int*)&s.misc()->slot_tile[slot] != (int)rg.k) {
                if (s.misc()->abort) { ok = false; break; }
                if (gtimer() - t0 > (uint64_t)p.wait_limit_ns) {
                    atomicOr(p.status, MK_ST_TIMEOUT | MK_ST_ABORT);
                    s.misc()->abort = 1;
                    ok = false;
                    break;
                }
                __nanosleep(64);
            }
        }
        ok = ok && wait_mbar(p, &s.full()[slot], ph, &s.misc()->abort);
        if (tw) {
            const uint64_t t1 = gtimer();
            if (threadIdx.x == 0) s.misc()->cwait += t1 - tw;
            rg.t_take += t1 - tw;
            rg.t_mark = t1;
        }
        if (ok && s.misc()->tile_bytes[slot] != expect_bytes) {
            atomicOr(p.status, MK_ST_SCHEDULE | MK_ST_ABORT);
            s.misc()->abort = 1;
            ok = false;
        }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    tile = s.ring() + (size_t)slot * p.geo.slot;
    if (MK_TRACE_ON && p.trace && p.trace_detail == 1 && (threadIdx.x & 31) == 0 && rg.k < 512)   // trace: a reader got tile k
        p.trace[(size_t)blockIdx.x * MK_TRACE_STRIDE + 3072 + rg.k] = gtimer();
    return ok;
}
// Done reading tile k; `weight` = MK_NCW / (warps reading it).  Advances the cursor.
__device__ __forceinline__ void release_tile(const MkParams& p, const Smem& s, Ring& rg, uint32_t weight = 1) {
    const uint64_t t2 = (MK_TRACE_ON && p.trace && p.trace_detail == 1 && (threadIdx.x & 31) == 0) ? gtimer() : 0;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        mbar_arrive(&s.empty()[rg.slot()], weight);
        if (t2 && rg.k < 512) p.trace[(size_t)blockIdx.x * MK_TRACE_STRIDE + 3584 + rg.k] = gtimer();
        if (t2) {
            rg.t_comp += t2 - rg.t_mark;
            rg.t_rel += gtimer() - t2;
        }
    }
    rg.advance(p.geo.ns);
}
// take_tile for a tile that has most likely landed long ago (the attention's
// K/V blocks, fetched during the previous layer): if the whole warp sees the
// slot claimed for tile k and its copy complete, every lane goes on at once --
// no lane-0 chain of loads, no shuffle; otherwise take_tile.  The decision is
// a warp vote, so no lane can return here while lane 0 goes on to take_tile's
// full-warp shuffle.
__device__ __forceinline__ bool take_landed(const MkParams& p, const Smem& s, Ring& rg, uint32_t expect_bytes,
                                            const uint8_t*& tile) {
    const uint32_t slot = rg.slot(), ph = rg.ph();
    bool fast = false;
    if (!(MK_TRACE_ON && p.trace && p.trace_detail == 1)) {
        const int claim = *(volatile int*)&s.misc()->slot_tile[slot];
        const int abt = *(volatile int*)&s.misc()->abort;
        fast = claim == (int)rg.k && !abt && mbar_test_wait(&s.full()[slot], ph) &&
               s.misc()->tile_bytes[slot] == expect_bytes;
    }
    if (__all_sync(0xFFFFFFFFu, fast)) {
        tile = s.ring() + (size_t)slot * p.geo.slot;
        return true;
    }
    return take_tile(p, s, rg, expect_bytes, tile);
}
// Trace only: lane 0 of each warp stores its ring accounting at slots
// 2304 + 16 * warp + 3 * e + {0 take, 1 between, 2 release} and clears it.
__device__ __forceinline__ void trace_ring(const MkParams& p, Ring& rg, int e) {
    if (MK_TRACE_ON && p.trace && p.trace_detail == 1 && (threadIdx.x & 31) == 0) {
        unsigned long long* tr = p.trace + (size_t)blockIdx.x * MK_TRACE_STRIDE + 2304 + 16 * (threadIdx.x >> 5) + 3 * e;
        tr[0] = rg.t_take; tr[1] = rg.t_comp; tr[2] = rg.t_rel;
    }
    rg.t_take = rg.t_comp = rg.t_rel = 0;
}

// ---- warp-row GEMV over one phase's tiles
//
// A tile holds up to TR rows of K bf16 (row-major).  LPR = min(32, K/8) lanes
// share a row, each owning MR = K/(8*LPR) chunks of 8 consecutive columns
// (chunk j of lane ll covers columns (j*LPR + ll)*8 ..).  The activation
// vector sits in shared memory in "split" order (xsplit): the first 4 values
// of every 8-column chunk c at [4c, 4c+4), the last 4 at [K/2 + 4c, ...), so
// a warp's 16-byte reads of one half are consecutive and bank-conflict free.
// A warp works on 4 rows at a time, so every activation chunk read from shared
// memory feeds 4 rows.  When a tile needs fewer than MK_NCW warps the consumer
// warps form groups that take alternate tiles; otherwise every warp works on
// every tile.  A row is reduced inside its LPR lanes and its first lane hands
// the sum to epi().  Every warp waits for every tile and arrives on its empty
// barrier (total weight MK_NCW per tile), but only the tile's group
// reads it.
// Smallest divisor of the consumer warp count that is >= need (warps that
// share a tile; a divisor, so every tile's readers arrive with equal weights).
__device__ __forceinline__ int group_size(int need) {
#pragma unroll
    for (int d = 1; d < MK_NCW; ++d)
        if (MK_NCW % d == 0 && d >= need) return d;
    return MK_NCW;
}

__device__ __forceinline__ int xsplit(int i, int K) { return ((i >> 3) << 2) + (i & 3) + ((i & 4) ? (K >> 1) : 0); }

__device__ __forceinline__ float2 bf2_lo_hi(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ void fma_chunk(const uint4 w, const float4 xl, const float4 xh, float2& a0, float2& a1) {
    a0 = __ffma2_rn(bf2_lo_hi(w.x), make_float2(xl.x, xl.y), a0);
    a1 = __ffma2_rn(bf2_lo_hi(w.y), make_float2(xl.z, xl.w), a1);
    a0 = __ffma2_rn(bf2_lo_hi(w.z), make_float2(xh.x, xh.y), a0);
    a1 = __ffma2_rn(bf2_lo_hi(w.w), make_float2(xh.z, xh.w), a1);
}

// Weight-only INT8 chunks: 8 codes (8 bytes, columns in the same order as a
// bf16 chunk's 8 columns) -> fp32.  The stream stores each code q as the
// byte q + 128, which becomes the low byte of the mantissa of 2^23 (exact);
// 2^23 + 128 comes off: bytes k and k+1 of a give the pair of values.
__device__ __forceinline__ uint2 lds64(const void* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ float2 i8pair(uint32_t a, int k) {
    const float x = __uint_as_float(__byte_perm(a, 0x4B000000u, 0x7540u + k));
    const float y = __uint_as_float(__byte_perm(a, 0x4B000000u, 0x7540u + k + 1));
    return __fadd2_rn(make_float2(x, y), make_float2(-8388736.f, -8388736.f));
}
__device__ __forceinline__ void fma_chunk8(const uint2 w, const float4 xl, const float4 xh, float2& a0, float2& a1) {
    const uint32_t lo = w.x, hi = w.y;
    a0 = __ffma2_rn(i8pair(lo, 0), make_float2(xl.x, xl.y), a0);
    a1 = __ffma2_rn(i8pair(lo, 2), make_float2(xl.z, xl.w), a1);
    a0 = __ffma2_rn(i8pair(hi, 0), make_float2(xh.x, xh.y), a0);
    a1 = __ffma2_rn(i8pair(hi, 2), make_float2(xh.z, xh.w), a1);
}
// Weight-only INT4 chunks: 8 codes in one word, byte k holding code k + 8 in
// its low nibble and code k + 4 + 8 in its high one (columns as a bf16
// chunk's); the nibbles, spread one a byte, take the int8 route above with
// 2^23 + 8 coming off.
__device__ __forceinline__ uint32_t lds32(const void* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint32_t nib_lo(uint32_t w) { return w & 0x0F0F0F0Fu; }          // codes 0..3
__device__ __forceinline__ uint32_t nib_hi(uint32_t w) { return (w >> 4) & 0x0F0F0F0Fu; }   // codes 4..7
__device__ __forceinline__ float2 i4pair(uint32_t a, int k) {
    const float x = __uint_as_float(__byte_perm(a, 0x4B000000u, 0x7540u + k));
    const float y = __uint_as_float(__byte_perm(a, 0x4B000000u, 0x7540u + k + 1));
    return __fadd2_rn(make_float2(x, y), make_float2(-8388616.f, -8388616.f));
}
__device__ __forceinline__ void fma_chunk4(const uint32_t w, const float4 xl, const float4 xh, float2& a0, float2& a1) {
    const uint32_t lo = nib_lo(w), hi = nib_hi(w);
    a0 = __ffma2_rn(i4pair(lo, 0), make_float2(xl.x, xl.y), a0);
    a1 = __ffma2_rn(i4pair(lo, 2), make_float2(xl.z, xl.w), a1);
    a0 = __ffma2_rn(i4pair(hi, 0), make_float2(xh.x, xh.y), a0);
    a1 = __ffma2_rn(i4pair(hi, 2), make_float2(xh.z, xh.w), a1);
}
// Stream bytes of K weights of form WB (2 bf16, 1 int8, 0 int4), and of one
// 8-weight chunk.
template <int WB> __host__ __device__ constexpr int wrow_bytes(int K) { return WB == 0 ? K / 2 : K * WB; }
template <int WB> __host__ __device__ constexpr int wchunk_bytes() { return WB == 0 ? 4 : 8 * WB; }
// A chunk of 8 weights: 16 bytes of bf16 (WB = 2), 8 bytes of int8 (WB = 1)
// or 4 bytes of int4 (WB = 0).
template <int WB> struct WChunk;
template <> struct WChunk<2> {
    using T = uint4;
    static __device__ __forceinline__ T load(const void* p) { return lds128(p); }
    static __device__ __forceinline__ T zero() { return make_uint4(0u, 0u, 0u, 0u); }
    static __device__ __forceinline__ void fma(const T w, const float4 xl, const float4 xh, float2& a0, float2& a1) {
        fma_chunk(w, xl, xh, a0, a1);
    }
};
template <> struct WChunk<1> {
    using T = uint2;
    static __device__ __forceinline__ T load(const void* p) { return lds64(p); }
    static __device__ __forceinline__ T zero() { return make_uint2(0x80808080u, 0x80808080u); }   // codes 0
    static __device__ __forceinline__ void fma(const T w, const float4 xl, const float4 xh, float2& a0, float2& a1) {
        fma_chunk8(w, xl, xh, a0, a1);
    }
};
template <> struct WChunk<0> {
    using T = uint32_t;
    static __device__ __forceinline__ T load(const void* p) { return lds32(p); }
    static __device__ __forceinline__ T zero() { return 0x88888888u; }   // codes 0
    static __device__ __forceinline__ void fma(const T w, const float4 xl, const float4 xh, float2& a0, float2& a1) {
        fma_chunk4(w, xl, xh, a0, a1);
    }
};

// ---- int8 dot products on integers (mk_xdigits)
//
// In the int8 build the hidden-width activation y (the RMSNorm output that
// QKV, gate/up and the LM head read) is held as y = X * sx with X an integer
// of at most 22 bits plus sign, written as three signed bytes,
// X = d2 * 2^16 + d1 * 2^8 + d0.  A row's dot product with the biased codes
// b = q + 128 is then three exact integer sums per lane, sum b * d_k, each
// 4 products per dp4a, less the per-lane constant 128 * sum d_k, combined in
// fp32 and scaled by sx and the row scale.  xv holds, per group of 4
// split-order columns (uint4 entry 4m .. 4m+3), the words of d0, d1 and d2.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {   // sum of unsigned a bytes x signed b bytes
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ float dig_combine(const int (&acc)[3], const int (&bias)[3]) {
    return fmaf((float)(acc[2] - bias[2]), 65536.f, fmaf((float)(acc[1] - bias[1]), 256.f, (float)(acc[0] - bias[0])));
}
// The lane's digit words of chunk ch (4 low-half and 4 high-half columns) and
// their share of the per-lane constant (the code bias, 128 for int8 and 8 for
// int4 (WB = 0), times the sum of the digits).
template <int WB = 1>
__device__ __forceinline__ void dig_load(const uint4* xq, int K, int ch, uint32_t (&d)[6], int (&bias)[3]) {
    constexpr uint32_t BIAS = WB == 0 ? 0x08080808u : 0x80808080u;
    const uint4 a = xq[ch], b = xq[K / 8 + ch];
    d[0] = a.x; d[1] = a.y; d[2] = a.z; d[3] = b.x; d[4] = b.y; d[5] = b.z;
#pragma unroll
    for (int k = 0; k < 3; ++k) bias[k] = dp4a_us(BIAS, d[k + 3], dp4a_us(BIAS, d[k], bias[k]));
}
// 8 biased codes (w.x: the 4 low-half columns, w.y: the 4 high-half ones) into the three sums.
__device__ __forceinline__ void dig_fma(const uint2 w, const uint32_t (&d)[6], int (&acc)[3]) {
#pragma unroll
    for (int k = 0; k < 3; ++k) acc[k] = dp4a_us(w.y, d[k + 3], dp4a_us(w.x, d[k], acc[k]));
}
// The same for an int4 chunk: its low nibbles are the low-half columns' codes, its high ones the others'.
__device__ __forceinline__ void dig_fma(const uint32_t w, const uint32_t (&d)[6], int (&acc)[3]) {
    dig_fma(make_uint2(nib_lo(w), nib_hi(w)), d, acc);
}

// Dot products of up to 4 rows (nv valid, rows r0 + k*step) with the
// split-order vector xs; each lane covers MR chunks of 8 columns (wchunk_bytes<WB>() bytes).
template <int MR, int LPR, int WB = 2>
__device__ __forceinline__ void dot_rows4(const uint8_t* r0, size_t step, int nv, const float* xs, int K, int ll,
                                          float o[4]) {
    float2 a[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r][0] = a[r][1] = make_float2(0.f, 0.f);
    const float4* xlo = reinterpret_cast<const float4*>(xs);
    const float4* xhi = reinterpret_cast<const float4*>(xs + (K >> 1));
#pragma unroll (MR < 8 ? MR : 8)
    for (int j = 0; j < MR; ++j) {
        const int ch = j * LPR + ll;
        const float4 xl = xlo[ch], xh = xhi[ch];
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (r < nv) WChunk<WB>::fma(WChunk<WB>::load(r0 + r * step + (size_t)ch * wchunk_bytes<WB>()), xl, xh, a[r][0], a[r][1]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) o[r] = (a[r][0].x + a[r][0].y) + (a[r][1].x + a[r][1].y);
}
// The same over int8 / int4 rows and the digits of the activation (xq); bias:
// the lane's constant over its MR chunks.  o[r] is in units of the activation scale.
template <int MR, int LPR, int WB = 1>
__device__ __forceinline__ void dot_rows4_dig(const uint8_t* r0, size_t step, int nv, const uint4* xq, int K, int ll,
                                              const int (&bias)[3], float o[4]) {
    int acc[4][3];
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[r][0] = acc[r][1] = acc[r][2] = 0;
#pragma unroll (MR < 8 ? MR : 8)
    for (int j = 0; j < MR; ++j) {
        const int ch = j * LPR + ll;
        const uint4 a = xq[ch], b = xq[K / 8 + ch];
        const uint32_t d[6] = {a.x, a.y, a.z, b.x, b.y, b.z};
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (r < nv) dig_fma(WChunk<WB>::load(r0 + r * step + (size_t)ch * wchunk_bytes<WB>()), d, acc[r]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) o[r] = dig_combine(acc[r], bias);
}

// GEMV over one phase's tiles (rows of K = MR * 8 * LPR columns, LPR lanes per
// row, RPP = 32 / LPR rows side by side in a warp).  A warp handles rw rows
// per lane group and pass (rw in {1, 2, 4}): with many tiles rw = 4 (each
// activation chunk feeds 4 rows: least shared-memory traffic), with few tiles
// rw shrinks so more warps share a tile and the phase ends sooner.
// The work split of a warp-row GEMV phase over nrows rows in tiles of TR rows,
// RPP rows side by side per warp: rows per lane group (rw) the largest of 4, 2,
// 1 that still lets every tile of a short phase run at once (or 4 when the
// phase has many tiles); groups of wpg warps take the tiles in turn.
__device__ void gemv_cfg(GemvCfg& c, int nrows, int TR, int RPP, int rwmax = 4) {
    const int ntiles = (nrows + TR - 1) / TR;
    int rw = rwmax, wpg = group_size((TR + rwmax * RPP - 1) / (rwmax * RPP));
    if (ntiles < MK_NCW / wpg) {
        for (int cand = 1; cand <= rwmax; cand <<= 1) {
            const int wp = group_size((TR + cand * RPP - 1) / (cand * RPP));
            if (MK_NCW / wp >= ntiles) { rw = cand; wpg = wp; break; }
        }
    }
    c.ntiles = (int16_t)ntiles; c.rw = (int16_t)rw; c.wpg = (int16_t)wpg; c.ngrp = (int16_t)(MK_NCW / wpg);
    for (int w = 0; w < MK_NCW; ++w) { c.grp[w] = (int8_t)(w / wpg); c.wg[w] = (int8_t)(w % wpg); }
}

// WB = 1 / 0: int8 / int4 rows, each row's sum times the row's scale from the
// tile's tail before epi() gets it.
// DIG (int8 / int4 rows only): vec holds the activation's digits (mk_xdigits), and
// each row's sum is also scaled by s.misc()->xscale.  HOLDF (bf16 rows of at
// most 4 chunks a lane): a warp with one pass on a tile loads its chunks into
// registers and releases the slot before the arithmetic.
template <int MR, int LPR, int WB, bool DIG = false, bool HOLDF = false, class Epi>
__device__ __forceinline__ bool gemv_phase_t(const MkParams& p, const Smem& s, Ring& ring, const float* vec,
                                             int nrows, int TR, const GemvCfg& cfg, bool ab, Epi&& epi,
                                             int trace_slot = -1, int dl = 0, int dmark = -1) {
    static_assert(!DIG || WB != 2, "digits are the int8 / int4 rows' activation form");
    constexpr int K = MR * 8 * LPR;
    constexpr int RPP = 32 / LPR;
    constexpr int CBY = wchunk_bytes<WB>();
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LPR, ll = lane % LPR;
    const int ntiles = cfg.ntiles, rw = cfg.rw, wpg = cfg.wpg, ngrp = cfg.ngrp;
    const int grp = cfg.grp[w], wg = cfg.wg[w];
    const int rows_per_warp = rw * RPP;
    const size_t rb = (size_t)wrow_bytes<WB>(K);
    int bias[3] = {0, 0, 0};
    float xsc = 1.f;
    if constexpr (DIG) {
        const uint4* xq = reinterpret_cast<const uint4*>(vec);
#pragma unroll (MR < 8 ? MR : 8)
        for (int j = 0; j < MR; ++j) {
            uint32_t d[6];
            dig_load<WB>(xq, K, j * LPR + ll, d, bias);
        }
        xsc = s.misc()->xscale;
    }
    int turn = 0;   // ti mod ngrp
    for (int ti = 0; ti < ntiles && !ab; ++ti) {
        const bool mine = turn == grp;
        if (++turn == ngrp) turn = 0;
        if (!mine) { ring.advance(p.geo.ns); continue; }   // another group's tile
        const int R = min(TR, nrows - ti * TR);
        const uint8_t* tile;
        const bool ok = take_tile(p, s, ring, (uint32_t)mk_row_tile_bytes(R, K, WB, 0), tile);
        if (trace_slot >= 0 && MK_TRACE_ON && p.trace && p.trace_detail == 1 && threadIdx.x == 0 && ti < 256)
            p.trace[(size_t)blockIdx.x * MK_TRACE_STRIDE + trace_slot + ti] = gtimer();
        if (dmark >= 0 && ti == 0) MK_TRACE_D(dl, dmark);   // thread 0 took its first tile
        if constexpr (DIG && MR <= 16) {
            // int8 / int4 rows of up to 2048 columns, one pass per warp on this tile:
            // the warp's codes and row scales go to registers and the slot is
            // released before the arithmetic, so the copy producer refills it
            // while the warp computes (a slot's turn is then the copy's latency
            // plus the loads, not plus the whole pass)
            constexpr int HR = MR <= 8 ? 4 : 2;   // rows held (64 registers of codes)
            if (ok && wpg * rows_per_warp >= R && rw <= HR) {
                const int r0 = wg * rows_per_warp + sub;
                const int nv = r0 < R ? min(rw, (R - r0 + RPP - 1) / RPP) : 0;
                typename WChunk<WB>::T cw[HR][MR];
#pragma unroll
                for (int r = 0; r < HR; ++r)
#pragma unroll
                    for (int j = 0; j < MR; ++j)
                        cw[r][j] = r < nv ? WChunk<WB>::load(tile + (size_t)(r0 + r * RPP) * rb + (size_t)(j * LPR + ll) * CBY)
                                          : WChunk<WB>::zero();
                const float* scl = reinterpret_cast<const float*>(tile + (size_t)R * rb);
                float sr[HR];
#pragma unroll
                for (int k = 0; k < HR; ++k) sr[k] = k < nv ? scl[r0 + k * RPP] * xsc : 0.f;
                release_tile(p, s, ring, (uint32_t)(MK_NCW / wpg));
                int acc[HR][3];
#pragma unroll
                for (int r = 0; r < HR; ++r) acc[r][0] = acc[r][1] = acc[r][2] = 0;
                const uint4* xq = reinterpret_cast<const uint4*>(vec);
#pragma unroll
                for (int j = 0; j < MR; ++j) {
                    const int ch = j * LPR + ll;
                    const uint4 a = xq[ch], b = xq[K / 8 + ch];
                    const uint32_t d[6] = {a.x, a.y, a.z, b.x, b.y, b.z};
#pragma unroll
                    for (int r = 0; r < HR; ++r) dig_fma(cw[r][j], d, acc[r]);
                }
                float v[HR];
#pragma unroll
                for (int k = 0; k < HR; ++k) {
                    v[k] = dig_combine(acc[k], bias);
                    if (k < rw) {
#pragma unroll
                        for (int o = LPR >> 1; o >= 1; o >>= 1) v[k] += __shfl_xor_sync(0xFFFFFFFFu, v[k], o);
                    }
                }
                if (ll == 0) {
#pragma unroll
                    for (int k = 0; k < HR; ++k)
                        if (k < nv) epi(ti * TR + r0 + k * RPP, v[k] * sr[k]);
                }
                continue;
            }
        }
        if constexpr (HOLDF && !DIG && WB == 2 && MR <= 4) {
            // bf16 rows of up to MR * 8 * LPR columns, one pass per warp on this
            // tile: the warp's chunks go to registers and the slot is released
            // before the arithmetic
            if (ok && wpg * rows_per_warp >= R) {
                const int r0 = wg * rows_per_warp + sub;
                const int nv = r0 < R ? min(rw, (R - r0 + RPP - 1) / RPP) : 0;
                uint4 cw[4][MR];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int j = 0; j < MR; ++j)
                        cw[r][j] = r < nv ? lds128(tile + (size_t)(r0 + r * RPP) * rb + (size_t)(j * LPR + ll) * 16)
                                          : make_uint4(0u, 0u, 0u, 0u);
                release_tile(p, s, ring, (uint32_t)(MK_NCW / wpg));
                float2 a[4][2];
#pragma unroll
                for (int r = 0; r < 4; ++r) a[r][0] = a[r][1] = make_float2(0.f, 0.f);
                const float4* xlo = reinterpret_cast<const float4*>(vec);
                const float4* xhi = reinterpret_cast<const float4*>(vec + (K >> 1));
#pragma unroll
                for (int j = 0; j < MR; ++j) {
                    const int ch = j * LPR + ll;
                    const float4 xl = xlo[ch], xh = xhi[ch];
#pragma unroll
                    for (int r = 0; r < 4; ++r) fma_chunk(cw[r][j], xl, xh, a[r][0], a[r][1]);
                }
                float v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[k] = (a[k][0].x + a[k][0].y) + (a[k][1].x + a[k][1].y);
                    if (k < rw) {
#pragma unroll
                        for (int o = LPR >> 1; o >= 1; o >>= 1) v[k] += __shfl_xor_sync(0xFFFFFFFFu, v[k], o);
                    }
                }
                if (ll == 0) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (k < nv) epi(ti * TR + r0 + k * RPP, v[k]);
                }
                continue;
            }
        }
        if (ok) {
            for (int base = wg * rows_per_warp; base < R; base += wpg * rows_per_warp) {
                // this lane group's rows: base + sub + k*RPP, k < rw
                const int r0 = base + sub;
                const int nv = r0 < R ? min(rw, (R - r0 + RPP - 1) / RPP) : 0;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if constexpr (DIG) {
                    if (nv > 0)
                        dot_rows4_dig<MR, LPR, WB>(tile + r0 * rb, rb * RPP, nv, reinterpret_cast<const uint4*>(vec), K,
                                                   ll, bias, v);
                } else {
                    if (nv > 0) dot_rows4<MR, LPR, WB>(tile + r0 * rb, rb * RPP, nv, vec, K, ll, v);
                }
                if (dmark >= 0 && ti == 0 && base == 0) {   // detail trace: the first pass's dot products done
                    float z = v[0] + v[1] + v[2] + v[3];
                    asm volatile("" : "+f"(z));
                    if (z == 12345.f) v[0] += 1.f;
                    MK_TRACE_D(dl, 13);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (k < rw) {
#pragma unroll
                        for (int o = LPR >> 1; o >= 1; o >>= 1) v[k] += __shfl_xor_sync(0xFFFFFFFFu, v[k], o);
                    }
                }
                if (ll == 0) {
                    const float* scl = reinterpret_cast<const float*>(tile + (size_t)R * rb);   // int8 / int4: row scales
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (k < nv) epi(ti * TR + r0 + k * RPP, WB != 2 ? v[k] * (scl[r0 + k * RPP] * xsc) : v[k]);
                }
                if (dmark >= 0 && ti == 0 && base == 0) MK_TRACE_D(dl, 14);   // its sums handed to epi
            }
        }
        release_tile(p, s, ring, (uint32_t)(MK_NCW / wpg));
        if (dmark >= 0 && ti == 0) MK_TRACE_D(dl, 15);   // the first tile released
        if (!ok) ab = true;     // this warp gave up; the barrier below makes it uniform
    }
    if (dmark >= 0) MK_TRACE_D(dl, dmark + 1);   // thread 0 done with its tiles
    return bar_or(ab);
}

// ---- GEMV for rows of K = 256 * MH columns (QKV, gate/up)
//
// The consumer warps form NG groups of WPG = MK_NCW / NG warps; tile ti goes to
// group ti % NG, so NG tiles are worked on at once and each is held for the
// time its group needs.  Inside a group warp (row slot rs, column block cb):
// the column block is CPL = MH / NKB chunks of 8 columns per lane, chunk
// (cb * CPL + j) * 32 + lane, whose activations the lane keeps in registers
// for the whole phase.  Row R of the phase (tiles of TR rows in order) belongs
// to row slot R % NRS; a warp takes its rows of a tile four at a time, reduces
// the four partial dot products over the warp with a transposed butterfly
// (6 shuffles) and stores them in part[R * NKB + cb].  The caller sums the NKB
// partials of a row after the phase barrier.
template <int MH, int NG>
struct WideGemv {
    static constexpr int K = MH * 256;
    static constexpr int WPG = MK_NCW / NG;
    static constexpr int NKB0 = (WPG % 4 == 0) ? 4 : (WPG % 2 == 0) ? 2 : 1;
    static constexpr int NKB = MH < NKB0 ? MH : NKB0;
    static constexpr int CPL = MH / NKB;
    static constexpr int NRS = WPG / NKB;
    static constexpr bool ok = (MK_NCW % NG == 0) && (MH % NKB == 0) && (WPG % NKB == 0) && CPL <= 4;
};
// part[] stride per row: the largest NKB any group count uses for this width
template <int MH>
struct WidePart { static constexpr int NKB = MH < 4 ? MH : 4; };

// WB = 1 / 0 (int8 / int4 rows): the same columns per chunk (8 or 4 bytes
// instead of 16), and each row's partials times the row's scale from the tile's tail; a GU tile's
// W_down column scales (after the row scales) go to tsink[j] for the j's it
// covers (the caller multiplies them into SiLU(gate) * up).  DG: the int rows
// as integer dot products over the activation's digits (xs holds mk_xdigits),
// or, DG = false, dequantized to fp32 against an fp32 xs.
template <int MH, int NG, int WB, bool DG = (WB != 2)>
__device__ __forceinline__ bool gemv_wide(const MkParams& p, const Smem& s, Ring& ring, const float* xs, int nrows,
                                          int TR, bool ab, float* part, float* tsink) {
    using W = WideGemv<MH, NG>;
    using C = WChunk<WB>;
    constexpr int K = W::K, NKB = W::NKB, CPL = W::CPL, NRS = W::NRS, WPG = W::WPG;
    constexpr int PS = WidePart<MH>::NKB;
    static_assert(W::ok && NKB <= PS, "wide GEMV mapping");
    // rows of a tile per warp at most: 16 chunks of 16 bytes per lane (slots of
    // 32 KB at most), 32 chunks of 8 bytes for int8, 64 of 4 bytes for int4
    constexpr int RPW = (16 / CPL) * (WB == 2 ? 1 : WB == 1 ? 2 : 4);
    constexpr int RB = wrow_bytes<WB>(K), CBY = wchunk_bytes<WB>();
    constexpr int NPS = RPW / 4;    // passes of four rows
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = w / WPG, wg = w % WPG;
    const int cb = wg % NKB, rs = wg / NKB;
    // the lane's activations for the whole phase: fp32, or the digits and
    // the lane's constant (int rows with DG, mk_xdigits)
    static_assert(!DG || WB != 2, "digits are the int rows' activation form");
    float4 xl[DG ? 1 : CPL], xh[DG ? 1 : CPL];
    uint32_t xd[DG ? CPL : 1][6];
    int bias[3] = {0, 0, 0};
    float xsc = 1.f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        const int ch = (cb * CPL + j) * 32 + lane;
        if constexpr (!DG) {
            xl[j] = reinterpret_cast<const float4*>(xs)[ch];
            xh[j] = reinterpret_cast<const float4*>(xs + K / 2)[ch];
        } else {
            dig_load<WB>(reinterpret_cast<const uint4*>(xs), K, ch, xd[j], bias);
        }
    }
    if constexpr (DG) xsc = s.misc()->xscale;
    const int ntiles = (nrows + TR - 1) / TR;
    for (int ti = 0; ti < ntiles && !ab; ++ti) {
        if (NG > 1 && (ti % NG) != grp) { ring.advance(p.geo.ns); continue; }   // another group's tile
        const int R0 = ti * TR, R = min(TR, nrows - R0);
        const uint8_t* tile;
        const bool ok = take_tile(p, s, ring, (uint32_t)mk_row_tile_bytes(R, K, WB, tsink ? R / 2 : 0), tile);
        // this warp's rows of the tile: r0, r0 + NRS, ... (nrow of them)
        int r0 = rs - R0 % NRS;
        if (r0 < 0) r0 += NRS;
        const int nrow = (ok && r0 < R) ? (R - r0 + NRS - 1) / NRS : 0;
        // int8 / int4: the R row scales follow the rows (then, in a GU tile,
        // the R / 2 W_down column scales of its j's); each lane that writes a
        // row's partial keeps that row's scale per pass (read before the
        // release), or, for int4 shares of up to 32 rows, lane i keeps row i's
        // and a pass fetches it with a shuffle (one register instead of eight)
        constexpr bool LANE_SCL = WB == 0 && RPW <= 32;
        float scl[LANE_SCL ? 1 : NPS];
        if constexpr (WB != 2) {
            const float* sc = reinterpret_cast<const float*>(tile + (size_t)R * RB);
            if (tsink && ok && wg == 0)
                for (int i = lane; i < R / 2; i += 32) tsink[R0 / 2 + i] = sc[R + i];
            if constexpr (LANE_SCL) {
                scl[0] = lane < nrow ? sc[r0 + lane * NRS] * xsc : 0.f;
            } else {
#pragma unroll
                for (int pb = 0; pb < NPS; ++pb) {
                    const int rr = 4 * pb + (lane >> 3);
                    scl[pb] = rr < nrow ? sc[r0 + rr * NRS] * xsc : 0.f;
                }
            }
        }
        // rows qb .. qb+3 of the share: dot products, transposed butterfly (lane
        // bit 4 picks rows {0,1} / {2,3}, bit 3 one row of the pair; bits 0-2
        // finish the sum) and the column-block partials into `part`
        auto pass = [&](int qb, auto&& chunk) {
            const int nv = min(4, nrow - qb);
            float v[4];
            if constexpr (!DG) {
                float2 a[4][2];
#pragma unroll
                for (int q = 0; q < 4; ++q) a[q][0] = a[q][1] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < CPL; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (qb + q < nrow) C::fma(chunk(qb + q, j), xl[j], xh[j], a[q][0], a[q][1]);
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = (a[q][0].x + a[q][0].y) + (a[q][1].x + a[q][1].y);
            } else {
                int acc[4][3];
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = acc[q][2] = 0;
#pragma unroll
                for (int j = 0; j < CPL; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (qb + q < nrow) dig_fma(chunk(qb + q, j), xd[j], acc[q]);
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = dig_combine(acc[q], bias);   // rows past nrow: not stored
            }
            const bool up = lane & 16, b3 = lane & 8;
            float k0 = up ? v[2] : v[0], k1 = up ? v[3] : v[1];
            k0 += __shfl_xor_sync(0xFFFFFFFFu, up ? v[0] : v[2], 16);
            k1 += __shfl_xor_sync(0xFFFFFFFFu, up ? v[1] : v[3], 16);
            float kk = b3 ? k1 : k0;
            kk += __shfl_xor_sync(0xFFFFFFFFu, b3 ? k0 : k1, 8);
            kk += __shfl_xor_sync(0xFFFFFFFFu, kk, 4);
            kk += __shfl_xor_sync(0xFFFFFFFFu, kk, 2);
            kk += __shfl_xor_sync(0xFFFFFFFFu, kk, 1);
            if constexpr (LANE_SCL) kk *= __shfl_sync(0xFFFFFFFFu, scl[0], qb + (lane >> 3));
            else if constexpr (WB != 2) kk *= scl[qb >> 2];
            const int q = lane >> 3;               // row of the four this lane holds
            if ((lane & 7) == 0 && q < nv) {
                float* pr = part + (R0 + r0 + (qb + q) * NRS) * PS;
                pr[cb] = kk;
                if (NKB < PS && cb == 0) {         // unused column-block slots read as zero
#pragma unroll
                    for (int c2 = NKB; c2 < PS; ++c2) pr[c2] = 0.f;
                }
            }
        };
        auto at = [&](int q, int j) {              // this lane's chunk of row q, chunk j of the share
            return tile + (size_t)(r0 + q * NRS) * RB + ((cb * CPL + j) * 32 + lane) * CBY;
        };
        // (int8 / int4 rows of 256 columns, up to 32 / 64 per warp, are read as
        // used: held whole beside their scales they spilled)
        if constexpr (CPL <= 2 && !(WB != 2 && CPL == 1)) {
            // Load the warp's whole share of the tile, then release the slot at
            // once: the copy producer refills it while this warp computes (the
            // arrival's release semantics order it after these loads).
            typename C::T wv[RPW][CPL];
#pragma unroll
            for (int q = 0; q < RPW; ++q)
#pragma unroll
                for (int j = 0; j < CPL; ++j) wv[q][j] = q < nrow ? C::load(at(q, j)) : C::zero();
            release_tile(p, s, ring, (uint32_t)NG);
#pragma unroll
            for (int qb = 0; qb < RPW; qb += 4)
                if (qb < nrow) pass(qb, [&](int q, int j) { return wv[q][j]; });
        } else {
            // four or more activation chunks per lane: the share would not fit
            // the registers beside them, so it is read as used, released after
#pragma unroll
            for (int qb = 0; qb < RPW; qb += 4)
                if (qb < nrow) pass(qb, [&](int q, int j) { return C::load(at(q, j)); });
            release_tile(p, s, ring, (uint32_t)NG);
        }
        if (!ok) ab = true;     // this warp gave up; the barrier below makes it uniform
    }
    return bar_or(ab);
}
// Three groups of four warps measured fastest of 1, 2, 3 and 6 groups on the
// 1B shape; a compile-time choice keeps one copy of the loop in the layer code.
constexpr int MK_GEMV_GROUPS = MK_WIDE_GROUPS;
template <int MH, int WB, bool DG = (WB != 2)>
__device__ __forceinline__ bool gemv_fifo(const MkParams& p, const Smem& s, Ring& ring, const float* xs, int nrows,
                                          int TR, bool ab, float* part, float* tsink = nullptr) {
    return gemv_wide<MH, MK_GEMV_GROUPS, WB, DG>(p, s, ring, xs, nrows, TR, ab, part, tsink);
}
// Sum of the NKB column-block partials of row R of a FIFO GEMV phase.
template <int MH>
__device__ __forceinline__ float wide_row(const float* part, int R) {
    constexpr int NKB = WidePart<MH>::NKB;
    float a = part[R * NKB];
#pragma unroll
    for (int c = 1; c < NKB; ++c) a += part[R * NKB + c];
    return a;
}

// RMSNorm of x (fp32 global, or the bf16 embedding row when xb != nullptr) into
// s.xv() (split order, for the GEMV), with gain g (fp32).  The raw values of rows
// [keep0, keep0 + nkeep) are also kept in `keep` (the residual this CTA adds
// later).  All loads of a thread (x and gains) are issued together, so the
// norm costs one L2 round trip.  Returns the uniform abort flag.
template <int NPT>   // ceil(H / consumer threads) values per thread
__device__ bool rmsnorm_to_xv(const MkParams& p, const Smem& s, const float* x, const uint16_t* xb, const float* g,
                              bool abort_in, float* keep, int keep0, int nkeep) {
    const int H = p.geo.H, t = threadIdx.x;
    float xr[NPT], gv[NPT];
#pragma unroll
    for (int k = 0; k < NPT; ++k) {
        const int i = t + k * MK_NCT;
        xr[k] = i < H ? (xb ? bf2f(xb[i]) : __ldcg(x + i)) : 0.f;
        gv[k] = i < H ? __ldg(g + i) : 0.f;
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < NPT; ++k) {
        const int i = t + k * MK_NCT;
        if ((unsigned)(i - keep0) < (unsigned)nkeep) keep[i - keep0] = xr[k];
        ss = fmaf(xr[k], xr[k], ss);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((t & 31) == 0) s.red()[t >> 5] = ss;
    bool ab = bar_or(abort_in);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < MK_NCW; ++w) tot += s.red()[w];
    const float inv = rsqrtf(tot / (float)H + p.eps);
#pragma unroll
    for (int k = 0; k < NPT; ++k) {
        const int i = t + k * MK_NCT;
        if (i < H) s.xv()[xsplit(i, H)] = xr[k] * inv * gv[k];   // split order for the GEMV
    }
    return bar_or(ab);
}

// The same norm for the int8 build's integer dot products: s.xv() receives
// y = x * rsqrt(mean x^2 + eps) * g as digits (mk_xdigits), its scale goes to
// s.misc()->xscale, and hid (if given) receives y itself.  A thread takes
// groups of 8 consecutive elements: their x and g load as 16-byte vectors and
// their digits leave as two 16-byte entries (the group's low and high split
// halves).  sx = max |y| / (2^22 - 1), so every X = rint(y / sx) has at most 22
// bits plus sign; a non-finite value makes sx non-finite, and the step's
// logits with it.
template <int NPG>   // ceil(H / 8 / consumer threads) groups per thread
__device__ bool rmsnorm_to_dig(const MkParams& p, const Smem& s, const float* x, const uint16_t* xb, const float* g,
                               bool abort_in, float* keep, int keep0, int nkeep, float* hid = nullptr) {
    const int H = p.geo.H, t = threadIdx.x;
    float xr[NPG][8], gv[NPG][8];
#pragma unroll
    for (int k = 0; k < NPG; ++k) {
        const int e0 = 8 * (t + k * MK_NCT);
        if (e0 < H) {
            if (xb) {
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(xb + e0));
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = bf2_lo_hi(ww[q]);
                    xr[k][2 * q] = f.x; xr[k][2 * q + 1] = f.y;
                }
            } else {
                const float4 a = __ldcg(reinterpret_cast<const float4*>(x + e0));
                const float4 b = __ldcg(reinterpret_cast<const float4*>(x + e0 + 4));
                xr[k][0] = a.x; xr[k][1] = a.y; xr[k][2] = a.z; xr[k][3] = a.w;
                xr[k][4] = b.x; xr[k][5] = b.y; xr[k][6] = b.z; xr[k][7] = b.w;
            }
            const float4 c = __ldg(reinterpret_cast<const float4*>(g + e0));
            const float4 d = __ldg(reinterpret_cast<const float4*>(g + e0 + 4));
            gv[k][0] = c.x; gv[k][1] = c.y; gv[k][2] = c.z; gv[k][3] = c.w;
            gv[k][4] = d.x; gv[k][5] = d.y; gv[k][6] = d.z; gv[k][7] = d.w;
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) xr[k][q] = gv[k][q] = 0.f;
        }
    }
    float ss = 0.f, mx = 0.f;
#pragma unroll
    for (int k = 0; k < NPG; ++k)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = 8 * (t + k * MK_NCT) + q;
            if ((unsigned)(i - keep0) < (unsigned)nkeep) keep[i - keep0] = xr[k][q];
            ss = fmaf(xr[k][q], xr[k][q], ss);
            const float a = fabsf(xr[k][q] * gv[k][q]);
            mx = (a != a) ? INFINITY : fmaxf(mx, a);   // max |x g|; NaN counts as +inf
        }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    }
    if ((t & 31) == 0) { s.red()[t >> 5] = ss; s.red()[MK_NCW + (t >> 5)] = mx; }
    bool ab = bar_or(abort_in);
    float tot = 0.f, m = 0.f;
#pragma unroll
    for (int w = 0; w < MK_NCW; ++w) { tot += s.red()[w]; m = fmaxf(m, s.red()[MK_NCW + w]); }
    const float inv = rsqrtf(tot / (float)H + p.eps);
    const float my = m * inv;
    const float sx = my == 0.f ? 1.f : my * (1.f / 4194303.f);
    const float isx = 1.f / sx;
    uint4* xq = reinterpret_cast<uint4*>(s.xv());
#pragma unroll
    for (int k = 0; k < NPG; ++k) {
        const int a = t + k * MK_NCT, e0 = 8 * a;
        if (e0 < H) {
            uint32_t w[2][3] = {{0u, 0u, 0u}, {0u, 0u, 0u}};   // [low/high half][digit]
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float y = xr[k][q] * inv * gv[k][q];
                if (hid) hid[e0 + q] = y;
                const int xi = __float2int_rn(y * isx);
                const int d0 = (int)(int8_t)(xi & 0xFF);
                const int x1 = (xi - d0) >> 8;
                const int d1 = (int)(int8_t)(x1 & 0xFF);
                const int d2 = (x1 - d1) >> 8;
                const int sh = 8 * (q & 3);
                w[q >> 2][0] |= (uint32_t)(d0 & 0xFF) << sh;
                w[q >> 2][1] |= (uint32_t)(d1 & 0xFF) << sh;
                w[q >> 2][2] |= (uint32_t)(d2 & 0xFF) << sh;
            }
            xq[a] = make_uint4(w[0][0], w[0][1], w[0][2], 0u);             // split positions 4a .. 4a+3
            xq[H / 8 + a] = make_uint4(w[1][0], w[1][1], w[1][2], 0u);     // H/2 + 4a .. H/2 + 4a+3
        }
    }
    if (t == 0) s.misc()->xscale = sx;
    return bar_or(ab);
}

// Grid-wide barrier on counter idx: every CTA's writes before it (made
// visible by the consumer barrier and the release arrival) are seen by every
// CTA after it.  Returns the uniform abort flag.
__device__ __forceinline__ bool grid_sync(const MkParams& p, int idx, bool ab) {
    ab = bar_or(ab);
    if (threadIdx.x == 0 && !ab) red_release_add(p.cnt + idx, 1u);
    bool bad = ab;
    if (threadIdx.x == 0 && !bad) bad = !wait_counter(p, p.cnt + idx, (uint32_t)p.geo.nC);
    return bar_or(bad);
}

// Order-preserving 32-bit key of a float (larger float -> larger key).
__device__ __forceinline__ uint32_t f2key(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Thread 0 waits on a counter; the result is made uniform by the barrier.
__device__ __forceinline__ bool sync_wait(const MkParams& p, int idx, uint32_t target, bool abort_in) {
    bool bad = abort_in;
    if (threadIdx.x == 0 && !bad) bad = !wait_counter(p, p.cnt + idx, target);
    return bar_or(bad);
}

// ------------------------------------------------------------------ attention

// Split-K decode attention for one CTA's share of positions.  Lane layout:
// TPP = G*HD/8 consecutive threads cover one position, thread (h, dc) owning
// head h and dims [8dc, 8dc+8) of that position; NCT/TPP positions are
// processed side by side.  Scores: 8-dim partial dots reduced over the HD/8
// lanes of a head.  Softmax is online (exp2, running max per head, rescaled
// sums).  V: each thread accumulates its head's 8 dims over its positions, and
// the position groups are summed with shared-memory atomics at the end.
// HPL_: heads per lane (the K/V chunks load and unpack once for HPL heads);
// the kernel runs one.
template <int HD, int G, int HPL_ = 1>
struct Attn {
    static constexpr int DC = HD / 8;                // lanes per head and position (8 dims each)
    static constexpr int HPL = HPL_;
    static constexpr int HG = G / HPL;               // head groups per position
    static constexpr int TPP = HG * DC;              // threads per position
    static constexpr int PPP = MK_NCT / TPP;         // positions per pass (position groups)
    static constexpr int PPW = TPP < 32 ? 32 / TPP : 1;   // position groups per warp
    static constexpr int NMG = PPP / PPW;            // groups after merging within warps
    static_assert(MK_NCT % TPP == 0 && (DC & (DC - 1)) == 0 && DC <= 32 && (32 % TPP == 0 || TPP % 32 == 0),
                  "attention lane layout");
    static_assert(NMG * G * HD <= 8 * MK_NCT, "parked attention partials fit the xv scratch");
    static_assert(NMG == MK_NCW || TPP >= 32, "one parked group per warp when positions share warps");

    // Per-thread online softmax over positions [0, n) of a block: thread
    // (pp, hg, dc) takes positions q = pp, pp + PPP, ..., four at a time, for
    // its HPL heads: it scores them (8-dim partial dots in packed fp32x2,
    // reduced over the DC lanes), rescales each head's running (m, l, acc)
    // once to the chunk's maximum and folds each position in with its exp2
    // weight.  q < nr from the ring tiles kt/vt, q == nr from the staged
    // current row (st: K, then V).  No barrier.  The thread's 8 q dims per
    // head (pre-scaled) are read from shared memory at qsa for every round of
    // positions instead of being held in registers across the block loop:
    // with them held, the kernel spilled under its 128-register budget.
    static __device__ __forceinline__ void online(const uint8_t* kt, const uint8_t* vt, int nr, const uint8_t* st,
                                                  int n, int pos0, uint32_t qsa, float (&m)[HPL],
                                                  float (&lsum)[HPL], float2 (&a2)[HPL][4]) {
        constexpr int CH = 4;                          // positions per thread and chunk
        constexpr bool SWZ = mk_attn_tc(HD, G);        // ring rows chunk-permuted by position (pos0 + q)
        const int t = threadIdx.x, pp = t / TPP, dc = t % DC;
        for (int q0 = 0; q0 < n; q0 += CH * PPP) {     // uniform trip count across the warp
            float qr[HPL][8];
#pragma unroll
            for (int j = 0; j < HPL; ++j) {   // volatile: re-read every round, not hoisted into registers
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(qr[j][0]), "=f"(qr[j][1]), "=f"(qr[j][2]), "=f"(qr[j][3]) : "r"(qsa + 4u * j * HD));
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(qr[j][4]), "=f"(qr[j][5]), "=f"(qr[j][6]), "=f"(qr[j][7]) : "r"(qsa + 4u * j * HD + 16u));
            }
            float sc[CH][HPL];
            uint4 vw[CH];
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int q = q0 + c * PPP + pp;
                float2 d[HPL];
#pragma unroll
                for (int j = 0; j < HPL; ++j) d[j] = make_float2(0.f, 0.f);
                vw[c] = make_uint4(0u, 0u, 0u, 0u);
                if (q < n) {
                    const size_t ro = (size_t)q * HD * 2 + ((SWZ ? (dc ^ ((pos0 + q) & 7)) : dc) << 4);
                    const uint4 kw = lds128(q < nr ? kt + ro : st + dc * 16);
                    vw[c] = lds128(q < nr ? vt + ro : st + HD * 2 + dc * 16);
                    const float2 k0 = bf2_lo_hi(kw.x), k1 = bf2_lo_hi(kw.y), k2 = bf2_lo_hi(kw.z), k3 = bf2_lo_hi(kw.w);
#pragma unroll
                    for (int j = 0; j < HPL; ++j) {
                        d[j] = __ffma2_rn(k0, make_float2(qr[j][0], qr[j][1]), d[j]);
                        d[j] = __ffma2_rn(k1, make_float2(qr[j][2], qr[j][3]), d[j]);
                        d[j] = __ffma2_rn(k2, make_float2(qr[j][4], qr[j][5]), d[j]);
                        d[j] = __ffma2_rn(k3, make_float2(qr[j][6], qr[j][7]), d[j]);
                    }
                }
#pragma unroll
                for (int j = 0; j < HPL; ++j) sc[c][j] = d[j].x + d[j].y;
            }
#pragma unroll
            for (int c = 0; c < CH; ++c)
#pragma unroll
                for (int j = 0; j < HPL; ++j)
#pragma unroll
                    for (int o = DC / 2; o >= 1; o >>= 1) sc[c][j] += __shfl_xor_sync(0xFFFFFFFFu, sc[c][j], o);
#pragma unroll
            for (int j = 0; j < HPL; ++j) {
                float cm = m[j];
#pragma unroll
                for (int c = 0; c < CH; ++c)
                    if (q0 + c * PPP + pp < n) cm = fmaxf(cm, sc[c][j]);
                if (cm != -INFINITY) {                 // this thread has a position in the chunk (or before)
                    const float corr = ex2_approx(m[j] - cm);   // m = -inf before the first position: 0
                    const float2 c2 = make_float2(corr, corr);
                    lsum[j] *= corr;
#pragma unroll
                    for (int k = 0; k < 4; ++k) a2[j][k] = __ffma2_rn(a2[j][k], c2, make_float2(0.f, 0.f));
#pragma unroll
                    for (int c = 0; c < CH; ++c) {
                        if (q0 + c * PPP + pp < n) {
                            const float pw = ex2_approx(sc[c][j] - cm);
                            const float2 p2 = make_float2(pw, pw);
                            lsum[j] += pw;
                            a2[j][0] = __ffma2_rn(bf2_lo_hi(vw[c].x), p2, a2[j][0]);
                            a2[j][1] = __ffma2_rn(bf2_lo_hi(vw[c].y), p2, a2[j][1]);
                            a2[j][2] = __ffma2_rn(bf2_lo_hi(vw[c].z), p2, a2[j][2]);
                            a2[j][3] = __ffma2_rn(bf2_lo_hi(vw[c].w), p2, a2[j][3]);
                        }
                    }
                    m[j] = cm;
                }
            }
        }
    }
    // Merges the PPW position groups that share a warp (lanes TPP apart) into
    // the lanes of the first one (same head group and dims), with exp2 weights
    // to the common maximum.
    static __device__ __forceinline__ void merge_warp(float (&m)[HPL], float (&lsum)[HPL], float2 (&a2)[HPL][4]) {
#pragma unroll
        for (int o = TPP; o < 32; o <<= 1) {
#pragma unroll
            for (int j = 0; j < HPL; ++j) {
                const float mo = __shfl_xor_sync(0xFFFFFFFFu, m[j], o);
                const float lo = __shfl_xor_sync(0xFFFFFFFFu, lsum[j], o);
                float2 ao[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    ao[k].x = __shfl_xor_sync(0xFFFFFFFFu, a2[j][k].x, o);
                    ao[k].y = __shfl_xor_sync(0xFFFFFFFFu, a2[j][k].y, o);
                }
                const float M = fmaxf(m[j], mo);
                const float w1 = (m[j] == -INFINITY) ? 0.f : ex2_approx(m[j] - M);
                const float w2 = (mo == -INFINITY) ? 0.f : ex2_approx(mo - M);
                lsum[j] = w1 * lsum[j] + w2 * lo;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    a2[j][k] = make_float2(w1 * a2[j][k].x + w2 * ao[k].x, w1 * a2[j][k].y + w2 * ao[k].y);
                m[j] = M;
            }
        }
    }
    // The merged group's lanes park (m, l) per head in sc and acc in xv:
    // xv[group][G*HD], sc[group*G + h] (m) and sc[NMG*G + group*G + h] (l).
    static __device__ __forceinline__ void park(const Smem& s, const float (&m)[HPL], const float (&lsum)[HPL],
                                                const float2 (&a2)[HPL][4]) {
        const int t = threadIdx.x, pp = t / TPP, hg = (t % TPP) / DC, dc = t % DC;
        if (pp % PPW != 0) return;                     // merged into the warp's first group
        const int grp = pp / PPW;
#pragma unroll
        for (int j = 0; j < HPL; ++j) {
            const int h = hg * HPL + j;
            float4* sp = reinterpret_cast<float4*>(s.xv() + grp * (G * HD) + h * HD + dc * 8);
            sp[0] = make_float4(a2[j][0].x, a2[j][0].y, a2[j][1].x, a2[j][1].y);
            sp[1] = make_float4(a2[j][2].x, a2[j][2].y, a2[j][3].x, a2[j][3].y);
            if (dc == 0) { s.sc()[grp * G + h] = m[j]; s.sc()[NMG * G + grp * G + h] = lsum[j]; }
        }
    }
};

// ---- long-context attention on the tensor cores (HD = 64 or 128, G = 4)
//
// At long contexts a CTA attends to thousands of positions per layer, and the
// per-position arithmetic of the lane-parallel softmax above (partial dots
// reduced by shuffles, bf16 unpacking, one dependent FMA chain per head) takes
// about twice as long as the K/V bytes take to arrive.  The contraction is
// dense, though: per 16 positions, S = [q_hi; q_lo] K^T is a 16x8xHD product
// and O += P V a 16xHDx16 one, so each warp runs them as mma.m16n8k16 (bf16
// in, fp32 accumulate), keeping q, P and O in registers:
//   - scores: A = q of the group's 4 heads split into a bf16 high part (rows
//     0-3) and the bf16 rounding of the remainder (rows 4-7), B = 8 K rows
//     from ldmatrix; row h plus row h+4 is q.k to about 2^-16 relative, and
//     the two halves meet with one shuffle (lanes 16 apart hold them);
//   - the accumulator of two score tiles is, lane for lane, the A fragment of
//     the P.V product (positions along k), so P never leaves registers; P is
//     split the same way (rows 0-3 high part, rows 4-7 remainder);
//   - V^T comes from ldmatrix.trans of the same rows.
// The cache's chunk permutation (mk_kv_index) keeps each 8x8 matrix load free
// of bank conflicts.  Warps take the 16-position chunks of the CTA's range in
// turn (continuing across blocks); each keeps its own online softmax state
// (m, l per head, O rows) and parks it in the same form as the lane-parallel
// version, so the partial that leaves the CTA is computed the same way.  With
// 128-dim heads four warps take each chunk: each computes the scores' partial
// sums over 32 of the 128 dims, the four meet through shared memory and add
// the partials in the same order (so they hold the same scores, m and l), and
// each accumulates 32 dims of O (mk_attn_tc_split).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
// D = A B + C for one m16n8k16 tile whose A rows 8-15 are zero: only the
// accumulator of rows 0-7 (c0, c1 of each lane) is carried.
// volatile: kept in program order with the matrix loads around it, so a
// product's operands are loaded just before it (hoisted loads of later
// operands had made the kernel spill under its 128-register budget).
__device__ __forceinline__ void mma_rows8(float& c0, float& c1, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    float d2, d3;
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %13};"
        : "=f"(c0), "=f"(c1), "=f"(d2), "=f"(d3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(0.f), "f"(0.f));
}
// bf16x2 of (x, y) rounded to nearest even: x in the low half.
__device__ __forceinline__ uint32_t pack_bf2(float x, float y) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(y), "f"(x));
    return r;
}
// (x, y) as bf16 high parts (lo == false) or as the bf16 of what they leave (lo).
__device__ __forceinline__ uint32_t split_bf2(float x, float y, bool lo) {
    const uint32_t h = pack_bf2(x, y);
    if (!lo) return h;
    return pack_bf2(x - __uint_as_float(h << 16), y - __uint_as_float(h & 0xFFFF0000u));
}

// Where the q poll leaves the score products' A fragments for the tensor-core
// attention: fragment word f (= 2 * k step + half, 0 .. 2*HD/16 - 1) of lane L
// at word (f / 4) * 128 + 4 * L + f % 4 of s.red() (free during the attention),
// so a lane reads its words back with 16-byte loads.  Lane L holds row L / 4 of
// [q_hi; q_lo]: head (L / 4) mod 4, the bf16 high parts for L < 16 and the
// bf16 of the remainders for L >= 16, dims 16 ks + 8 half + 2 (L mod 4) (+1).
// Warps that share each 16-position chunk of the tensor-core attention (each
// accumulates HD / split dims of O: with all 128 dims in one warp, or 64, the
// 8B-width build spilled under its 128-register budget) and the groups its
// warps park.
__host__ __device__ constexpr int mk_attn_tc_split(int hd) { return hd == 128 ? 4 : 1; }
__host__ __device__ constexpr int mk_attn_tc_groups(int hd) { return MK_NCW / mk_attn_tc_split(hd); }
// Barrier of the DS warps of chunk stream wi (named barriers 2, 3, 4; the
// consumers' barrier is 1).
__device__ __forceinline__ void stream_sync(int wi) {
    if (wi == 0) asm volatile("bar.sync 2, 128;" ::: "memory");
    else if (wi == 1) asm volatile("bar.sync 3, 128;" ::: "memory");
    else asm volatile("bar.sync 4, 128;" ::: "memory");
}
__device__ __forceinline__ int qfrag_word(int f, int lane) { return (f >> 2) * 128 + 4 * lane + (f & 3); }

// The block loop of the tensor-core attention (q of the group's heads already
// split into A fragments in qf, pre-scaled).  Positions [ka, ke) come from the
// ring in blocks of KB (K tile then V tile, rows chunk-permuted by position);
// the current position (staged, plain row order) follows the last block when
// has_cur.  Returns the abort flag (not yet uniform); the warps' states are
// parked for the caller.  The fragments are read back from shared memory for
// every 16-position chunk rather than held in registers across the loop: held,
// they made the kernel spill under its 128-register budget.
template <int HD, int G>
__device__ __forceinline__ bool attn_tc_blocks(const MkParams& p, const Smem& s, Ring& ring, int l, int ka, int ke,
                                               bool has_cur, bool ab, const uint32_t* qf) {
    static_assert(mk_attn_tc(HD, G), "tensor-core attention: 4 heads of 64 or 128 dims per KV group");
    constexpr int NKS = HD / 16;         // 16-dim k steps of a score tile
    constexpr int DS = mk_attn_tc_split(HD);   // warps sharing a chunk, each carrying HD / DS dims of O
    constexpr int NWP = MK_NCW / DS;     // chunk streams (warp sets) = parked groups
    constexpr int DW = HD / DS;          // dims of O per warp
    constexpr int ND = DW / 8;           // 8-dim tiles of O per warp
    constexpr int NMG = mk_attn_tc_groups(HD);
    static_assert(NMG == NWP && NMG * G * HD + (DS > 1 ? 2 * NWP * DS * 64 : 0) <= 8 * MK_NCT,
                  "parked groups and the score exchange fit the xv scratch");
    static_assert(DS == 1 || (DS * 32 == 128 && NWP == 3), "named barriers of 128 threads, one per stream");
    const MkGeom& g = p.geo;
    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    const int dh = DS == 1 ? 0 : w / NWP, wi = DS == 1 ? w : w % NWP;   // this warp's dims of O, its chunk stream
    const bool lo = lane >= 16;          // this lane's rows hold the remainder parts (4-7)
    const int qd = 2 * (lane & 3);       // first of this lane's two k (or n) indices in a tile
    const uint32_t qfa = smem_u32(qf + qfrag_word(0, lane));
    float o[ND][2];
#pragma unroll
    for (int j = 0; j < ND; ++j) o[j][0] = o[j][1] = 0.f;
    float m = -INFINITY, lsum = 0.f;
    MK_TRACE_D(l, 1);
    const uint32_t zaddr = smem_u32(&s.misc()->zrow);
    const uint32_t staddr = smem_u32(s.misc()->stage);
    const int nring = ke > ka ? ke - ka : 0;
    const int nblk = (nring + g.KB - 1) / g.KB;
    const int nbt = (nblk == 0 && has_cur) ? 1 : nblk;
    if (t == 0 && nblk > 1) *(volatile int*)&s.misc()->streaming = 1;
    int cbase = 0;                       // chunks of the earlier blocks (stream wi takes chunk indices = wi mod NWP)
    uint32_t rnd = 0;                    // 128 dims: chunk rounds of this stream (the score exchange's buffer)
    for (int b = 0; b < nbt && !ab; ++b) {
        const int q0 = ka + b * g.KB;
        const int nr = (b < nblk) ? min(g.KB, ke - q0) : 0;
        const int n = nr + ((has_cur && b == nbt - 1) ? 1 : 0);
        const uint8_t *kt = nullptr, *vt = nullptr;
        bool ok = true;
        if (nr > 0) {
            Ring rv = ring;
            rv.advance(g.ns);            // the V tile follows the K tile in the stream
            ok = take_landed(p, s, ring, (uint32_t)(nr * HD * 2), kt) && take_landed(p, s, rv, (uint32_t)(nr * HD * 2), vt);
        }
        // 128 dims: the warps of a stream meet at a named barrier, which has no
        // time limit, so they all run a block's chunks or none of them
        if constexpr (DS > 1) ok = !bar_or(!ok);
        if (b == 0) MK_TRACE_D(l, 5);
        if (ok) {
            const uint32_t ka_ = kt ? smem_u32(kt) : 0u, va_ = vt ? smem_u32(vt) : 0u;
            // shared-memory address of 16-byte chunk cc of block row i (K or V):
            // ring rows below nr, then the staged current row, then a zero row
            auto row = [&](uint32_t base, uint32_t stoff, int i, int cc) -> uint32_t {
                if (i < nr) return base + (uint32_t)i * (HD * 2) + ((uint32_t)(cc ^ ((q0 + i) & 7)) << 4);
                if (i < n) return staddr + stoff + ((uint32_t)cc << 4);
                return zaddr;
            };
            const int nch = (n + 15) >> 4;
            int ci = wi - cbase % NWP;
            if (ci < 0) ci += NWP;
            for (; ci < nch; ci += NWP) {
                const int c0 = 16 * ci;
                // scores of the chunk's two 8-position tiles
                float sv[2][2];
                if constexpr (HD == 64) {
                    // both 8-position tiles at once: the q fragments serve both, and
                    // their products form two independent chains
                    uint32_t qa[NKS][2];   // A fragments of [q_hi; q_lo] (volatile: re-read per chunk)
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(qa[0][0]), "=r"(qa[0][1]), "=r"(qa[1][0]), "=r"(qa[1][1]) : "r"(qfa));
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(qa[2][0]), "=r"(qa[2][1]), "=r"(qa[3][0]), "=r"(qa[3][1]) : "r"(qfa + 512u));
                    float c[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
                    for (int x = 0; x < NKS / 2; ++x)
#pragma unroll
                        for (int tt = 0; tt < 2; ++tt) {
                            uint32_t kb[4];   // the tile's 8x8 matrices of chunks 4x .. 4x+3: two k steps
                            ldsm_x4(kb, row(ka_, 0u, c0 + 8 * tt + (lane & 7), 4 * x + (lane >> 3)));
                            mma_rows8(c[tt][0], c[tt][1], qa[2 * x][0], qa[2 * x][1], kb[0], kb[1]);
                            mma_rows8(c[tt][0], c[tt][1], qa[2 * x + 1][0], qa[2 * x + 1][1], kb[2], kb[3]);
                        }
#pragma unroll
                    for (int tt = 0; tt < 2; ++tt) {
                        // high part + remainder: lanes 16 apart hold the same head and positions
                        const float c0_ = c[tt][0] + __shfl_xor_sync(0xFFFFFFFFu, c[tt][0], 16);
                        const float c1_ = c[tt][1] + __shfl_xor_sync(0xFFFFFFFFu, c[tt][1], 16);
                        const int pi = c0 + 8 * tt + qd;
                        sv[tt][0] = pi < n ? c0_ : -INFINITY;
                        sv[tt][1] = pi + 1 < n ? c1_ : -INFINITY;
                    }
                } else {
                    // 128 dims: the DS warps of a stream split the scores' k
                    // steps (warp dh takes dims 32 dh .. 32 dh + 31), leave their
                    // partial scores in shared memory (double-buffered by round),
                    // meet at the stream's named barrier and add the DS partials
                    // in the same order, so all of them hold the same scores (and
                    // so the same m, l and P)
                    float c[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
                    uint32_t qa[2][2];
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(qa[0][0]), "=r"(qa[0][1]), "=r"(qa[1][0]), "=r"(qa[1][1])
                                 : "r"(qfa + 512u * dh));
#pragma unroll
                    for (int tt = 0; tt < 2; ++tt) {
                        uint32_t kb[4];   // the tile's 8x8 matrices of chunks 4dh .. 4dh+3
                        ldsm_x4(kb, row(ka_, 0u, c0 + 8 * tt + (lane & 7), 4 * dh + (lane >> 3)));
                        mma_rows8(c[tt][0], c[tt][1], qa[0][0], qa[0][1], kb[0], kb[1]);
                        mma_rows8(c[tt][0], c[tt][1], qa[1][0], qa[1][1], kb[2], kb[3]);
                    }
                    // high part + remainder: lanes 16 apart hold the same head and positions
#pragma unroll
                    for (int tt = 0; tt < 2; ++tt) {
                        c[tt][0] += __shfl_xor_sync(0xFFFFFFFFu, c[tt][0], 16);
                        c[tt][1] += __shfl_xor_sync(0xFFFFFFFFu, c[tt][1], 16);
                    }
                    float4* xb = reinterpret_cast<float4*>(s.xv() + NMG * G * HD) + ((rnd & 1) * NWP + wi) * (DS * 16);
                    ++rnd;
                    if (lane < 16) xb[dh * 16 + lane] = make_float4(c[0][0], c[0][1], c[1][0], c[1][1]);
                    stream_sync(wi);
                    float4 sc4 = xb[lane & 15];
#pragma unroll
                    for (int q = 1; q < DS; ++q) {
                        const float4 v = xb[q * 16 + (lane & 15)];
                        sc4.x += v.x; sc4.y += v.y; sc4.z += v.z; sc4.w += v.w;
                    }
                    const int pi = c0 + qd;
                    sv[0][0] = pi < n ? sc4.x : -INFINITY;
                    sv[0][1] = pi + 1 < n ? sc4.y : -INFINITY;
                    sv[1][0] = pi + 8 < n ? sc4.z : -INFINITY;
                    sv[1][1] = pi + 9 < n ? sc4.w : -INFINITY;
                }
                // online softmax per head (row): the quad of lanes sharing a row agrees on the maximum
                float cm = fmaxf(fmaxf(m, fmaxf(sv[0][0], sv[0][1])), fmaxf(sv[1][0], sv[1][1]));
                cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 1));
                cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 2));
                const float corr = ex2_approx(m - cm);   // 0 before the first position
                const float p00 = ex2_approx(sv[0][0] - cm), p01 = ex2_approx(sv[0][1] - cm);
                const float p10 = ex2_approx(sv[1][0] - cm), p11 = ex2_approx(sv[1][1] - cm);
                lsum = fmaf(lsum, corr, (p00 + p01) + (p10 + p11));
                m = cm;
#pragma unroll
                for (int j = 0; j < ND; ++j) { o[j][0] *= corr; o[j][1] *= corr; }
                const uint32_t pa0 = split_bf2(p00, p01, lo), pa2 = split_bf2(p10, p11, lo);
                // O += P V over this warp's dims: V^T fragments of d tiles
                // ND dh + 2jj, ND dh + 2jj + 1 (rows c0.. and c0+8..)
#pragma unroll
                for (int jj = 0; jj < ND / 2; ++jj) {
                    const int mt = lane >> 3;
                    uint32_t vb[4];
                    ldsm_x4_trans(vb, row(va_, (uint32_t)(HD * 2), c0 + 8 * (mt & 1) + (lane & 7),
                                          ND * dh + 2 * jj + (mt >> 1)));
                    mma_rows8(o[2 * jj][0], o[2 * jj][1], pa0, pa2, vb[0], vb[1]);
                    mma_rows8(o[2 * jj + 1][0], o[2 * jj + 1][1], pa0, pa2, vb[2], vb[3]);
                }
            }
            cbase += nch;
        }
        if (b == 0) MK_TRACE_D(l, 6);
        if (nr > 0) { release_tile(p, s, ring); release_tile(p, s, ring); }
        if (!ok) ab = true;     // made uniform by the caller's barrier
    }
    if (t == 0 && nblk > 1) *(volatile int*)&s.misc()->streaming = 0;
    MK_TRACE_D(l, 2);
    // the warp's state: l summed over the quad, O rows h and h+4 added; park
    // (m, l) per head in sc and O (this warp's dims) in xv[wi] like the
    // lane-parallel version (the DS warps of a stream hold the same m and l)
    lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 1);
    lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 2);
#pragma unroll
    for (int j = 0; j < ND; ++j) {
        o[j][0] += __shfl_xor_sync(0xFFFFFFFFu, o[j][0], 16);
        o[j][1] += __shfl_xor_sync(0xFFFFFFFFu, o[j][1], 16);
    }
    if (!ab && !lo) {
        const int h = lane >> 2;
        float* xp = s.xv() + wi * (G * HD) + h * HD + DW * dh + qd;
#pragma unroll
        for (int j = 0; j < ND; ++j) *reinterpret_cast<float2*>(xp + 8 * j) = make_float2(o[j][0], o[j][1]);
        if ((lane & 3) == 0 && dh == 0) { s.sc()[wi * G + h] = m; s.sc()[NMG * G + wi * G + h] = lsum; }
    }
    return ab;
}

// The attention of one CTA over its positions with HPL heads per lane: this
// thread's q dims (tagged words), the block loop (online softmax), the merge
// of the position groups sharing a warp and the parking of the warps' groups
// in smem for the partial.  Returns the uniform abort flag (one barrier).
template <int HD, int G, int HPL, bool TC>
__device__ __forceinline__ bool attn_run(const MkParams& p, const Smem& s, Ring& ring, int l, int ka, int ke,
                                         bool has_cur, bool ab) {
    bool late = false;
    constexpr float qscale = (HD == 64 ? 0.125f : 0.08838834764831845f) * 1.4426950408889634f;   // log2(e)/sqrt(hd)
    static_assert(HD == 64 || HD == 128, "attention head sizes");
    using A = Attn<HD, G, HPL>;
    const MkGeom& g = p.geo;
    const MkCtaPlan& pl = s.misc()->plan;
    const int t = threadIdx.x;
    const int hg_ = (t % A::TPP) / A::DC, dc_ = t % A::DC;
    // q of the group's G heads (G*HD tagged words): every 16-byte chunk is
    // polled by one thread, consecutive chunks by consecutive lanes, so one
    // warp instruction reads four whole 128-byte lines and the CTA reads each
    // line once (had every thread read the q values it needs, the 12 position
    // groups would read the same words, ~48x the requests on the same L2
    // lines, in all CTAs of the group at once).  The poller scales its two
    // values by log2(e)/sqrt(hd) and leaves them in `ov` (free until the
    // combine) for the lane-parallel build, or, for the tensor-core build,
    // split into bf16 high and low parts in the A-fragment words they belong
    // to (qfrag_word).
    constexpr int NQC = G * HD / 2;
    static_assert(NQC + HD / 4 <= MK_NCT, "q poll and current-row staging side by side");
    float* qs = s.ov();
    uint32_t* qf = reinterpret_cast<uint32_t*>(s.red());
    // The CTA that also takes the current position stages its K and V rows
    // (bf16, from their tagged copies) with the threads after the q pollers,
    // so both polls cost one L2 round trip.
    if (!ab && has_cur && t >= NQC && t < NQC + HD / 4) {
        const int u = t - NQC;
        float kv[8];
        late = !ll_read8(p, p.kvll + (((size_t)l * g.kvh + pl.g) * 2 + (u < HD / 8 ? 0 : 1)) * HD + (u % (HD / 8)) * 8,
                         s.misc()->tag, kv);
        uint4 w;
        w.x = (uint32_t)f2bf(kv[0]) | ((uint32_t)f2bf(kv[1]) << 16);
        w.y = (uint32_t)f2bf(kv[2]) | ((uint32_t)f2bf(kv[3]) << 16);
        w.z = (uint32_t)f2bf(kv[4]) | ((uint32_t)f2bf(kv[5]) << 16);
        w.w = (uint32_t)f2bf(kv[6]) | ((uint32_t)f2bf(kv[7]) << 16);
        s.misc()->stage[u] = w;
    }
    if (!ab) {
        const uint32_t tag = s.misc()->tag;
        const uint64_t* qsrc = p.qll + (size_t)l * g.qh * HD + (size_t)pl.g * G * HD;
        for (int c = t; c < NQC && !late; c += MK_NCT) {
            uint64_t t0 = 0;
            for (;;) {
                const ulonglong2 w = ld_ll2(qsrc + 2 * c);
                if (ll_ok(w, tag)) {
                    const float q0 = __uint_as_float((uint32_t)w.x) * qscale;
                    const float q1 = __uint_as_float((uint32_t)w.y) * qscale;
                    if constexpr (TC) {
                        // dims d, d+1 of head h: fragment word 2 (d / 16) + (d / 8) % 2 of
                        // lane 4h + (d % 8) / 2 (high part) and of lane 16 + 4h + (d % 8) / 2
                        const int h = (2 * c) / HD, d = (2 * c) % HD;
                        const int f = 2 * (d >> 4) + ((d >> 3) & 1), ln = 4 * h + ((d & 7) >> 1);
                        qf[qfrag_word(f, ln)] = split_bf2(q0, q1, false);
                        qf[qfrag_word(f, ln + 16)] = split_bf2(q0, q1, true);
                    } else {
                        *reinterpret_cast<float2*>(qs + 2 * c) = make_float2(q0, q1);
                    }
                    break;
                }
                if (!ll_backoff(p, t0)) { late = true; break; }
            }
        }
    }
    ab = bar_or(ab || late);
    MK_TRACE_D(l, 0);   // q in shared memory
    if constexpr (TC) return attn_tc_blocks<HD, G>(p, s, ring, l, ka, ke, has_cur, ab, qf);
    const uint32_t qsa = smem_u32(qs + (hg_ * HPL) * HD + dc_ * 8);   // this thread's q dims (pre-scaled)
    float m_[HPL], l_[HPL];
    float2 acc[HPL][4];
#pragma unroll
    for (int j = 0; j < HPL; ++j) {
        m_[j] = -INFINITY;
        l_[j] = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[j][k] = make_float2(0.f, 0.f);
    }
    MK_TRACE_D(l, 1);   // every thread has its q
    const int nring = ke > ka ? ke - ka : 0;
    const int nblk = (nring + g.KB - 1) / g.KB;
    const int nbt = (nblk == 0 && has_cur) ? 1 : nblk;
    const uint8_t* st = reinterpret_cast<const uint8_t*>(s.misc()->stage);
    // several K/V blocks (long contexts) stream like weights: lift the
    // producer's latency-phase in-flight limit for the block loop
    if (t == 0 && nblk > 1) *(volatile int*)&s.misc()->streaming = 1;
    for (int b = 0; b < nbt && !ab; ++b) {
        const int q0 = ka + b * g.KB;
        const int nr = (b < nblk) ? min(g.KB, ke - q0) : 0;
        const int n = nr + ((has_cur && b == nbt - 1) ? 1 : 0);
        const uint8_t *kt = st, *vt = st;
        bool ok = true;
        if (nr > 0) {
            Ring rv = ring;
            rv.advance(g.ns);      // the V tile follows the K tile in the stream
            ok = take_tile(p, s, ring, (uint32_t)(nr * HD * 2), kt) && take_tile(p, s, rv, (uint32_t)(nr * HD * 2), vt);
        }
        if (b == 0) MK_TRACE_D(l, 5);   // first block's K and V taken
        if (ok) A::online(kt, vt, nr, st, n, q0, qsa, m_, l_, acc);
        if (b == 0) MK_TRACE_D(l, 6);   // first block's softmax done
        if (nr > 0) { release_tile(p, s, ring); release_tile(p, s, ring); }
        if (!ok) ab = true;     // made uniform by the barrier below
    }
    if (t == 0 && nblk > 1) *(volatile int*)&s.misc()->streaming = 0;
    MK_TRACE_D(l, 2);   // softmax over the blocks done
    // merge the position groups: first those sharing a warp (shuffles), then
    // the warps' groups park (m, l) per head and acc in smem (xv, free between
    // QKV and the FFN norm); after the caller's barrier each output element is
    // rescaled to the group-wide maximum and summed
    A::merge_warp(m_, l_, acc);
    if (!ab) A::park(s, m_, l_, acc);
    return ab;
}

// ------------------------------------------------------------------ sampling

// Gumbel noise for sampling by the Gumbel-max rule: argmax_v (logit_v / T + G_v)
// is distributed as softmax(logit / T).  U_v comes from SplitMix64 (Steele,
// Lea and Flood, "Fast splittable pseudorandom number generators", OOPSLA
// 2014) in its counter form -- output i of the generator seeded with s is
// mix(s + (i + 1) * 0x9E3779B97F4A7C15) -- with i = pos * 2^32 + v; U takes
// the top 23 bits, (bits + 0.5) * 2^-23, exact in fp32 and never 0 or 1;
// G = -ln(-ln U) in fp32.
__device__ __forceinline__ float mk_gumbel(uint64_t seed, int pos, int v) {
    uint64_t z = seed + ((((uint64_t)(uint32_t)pos << 32) | (uint32_t)v) + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    const float u = ((float)(uint32_t)(z >> 41) + 0.5f) * 1.1920928955078125e-07f;   // exact: 24 significant bits
    return -logf(-logf(u));
}

// ------------------------------------------------------------------ the kernel

// HD: head_dim; G: query heads per KV head; MH = H / 256, the 8-column chunks
// each lane owns in a row of H (the GEMV width of QKV, gate/up and LM head);
// LC: long-context build: the attention runs on the tensor cores (16-position
// chunks per warp; shapes with 4 query heads of 64 dims per KV group), which
// pays once every CTA attends to more positions than one chunk per warp; on
// short contexts the lane-parallel attention of the standard build has the
// shorter dependency chain.  The host picks the build per step.
// WB: streamed weight form, 2 (bf16), 1 (weight-only INT8) or 0 (weight-only INT4).
template <int HD, int G, int MH, int LC, int WB>
__global__ void __launch_bounds__(MK_BLOCK, 1) mk_decode_kernel(const __grid_constant__ MkParams p) {
    static_assert(G <= MK_NCW, "one consumer warp per query head of a KV group (softmax, combine weights)");
    static_assert(!LC || mk_attn_tc(HD, G), "the long-context build's attention runs on 4 heads of 64 or 128 dims");
    // generation already stopped (an earlier launch sampled the stop token):
    // every CTA returns before touching any state
    if (p.stop && *(volatile int32_t*)p.stop) return;
    constexpr int KO = G * HD;                         // O-proj row length
    constexpr int LPRO = KO >= 32 * 4 ? KO / 32 : 4;   // short rows: 4 chunks per lane
    constexpr int MO = KO / (8 * LPRO);
    static_assert(LPRO <= 32 && 32 % LPRO == 0 && MO * 8 * LPRO == KO, "O-proj row mapping");
    const MkGeom& g = p.geo;
    Smem s;
    s.g = &p.geo;

    const int t = threadIdx.x;
    const int c = blockIdx.x;

    if (t == 0) {
        for (int i = 0; i < g.ns; ++i) {
            mbar_init(&s.full()[i], 1);
            mbar_init(&s.empty()[i], MK_NCW);
            s.misc()->slot_tile[i] = -1;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s.misc()->abort = 0;
        s.misc()->streaming = 0;
        s.misc()->copy_bytes = 0;
        s.misc()->cwait = 0;
        s.misc()->is_last = 0;
        int tok = p.token_ptr ? *p.token_ptr : p.token;
        if (tok < 0 || tok >= g.V) {
            if (c == 0) atomicOr(p.status, MK_ST_BADTOKEN);
            tok = 0;
        }
        s.misc()->token = tok;
        s.misc()->zrow = make_uint4(0u, 0u, 0u, 0u);
        s.misc()->plan = p.plans[c];
        {
            int ka_, ke_;
            bool hc_;
            mk_attn_share(p.pos, p.attn_ctas, s.misc()->plan.i, &ka_, &ke_, &hc_);
            s.misc()->ka = ka_;
            s.misc()->ke = ke_;
            s.misc()->has_cur = hc_ ? 1 : 0;
            s.misc()->att = s.misc()->plan.i < p.attn_ctas ? 1 : 0;
            s.misc()->dr0 = (int)mk_split(g.H, g.nC, c);
            s.misc()->dr1 = (int)mk_split(g.H, g.nC, c + 1);
        }
        {
            constexpr int KO = G * HD, LPRO = KO >= 32 * 4 ? KO / 32 : 4;
            gemv_cfg(s.misc()->ocfg, s.misc()->plan.norows, g.TRo, 32 / LPRO);
            gemv_cfg(s.misc()->lmcfg, s.misc()->plan.nv, g.TRh, 1, (WB != 2 && MH > 8) ? 2 : 4);
        }
        {
            const uint32_t sq = *(volatile uint32_t*)p.seq;
            s.misc()->par = (int)(sq & 1u);
            s.misc()->tag = sq + 1u;
        }
        for (int h = 0; h < 8; ++h) s.misc()->alpha[h] = 0.f;
    }
    __syncthreads();
    const MkCtaPlan& pl = s.misc()->plan;

    const int warp = t >> 5;
    if (warp == MK_PRODUCER_WARP) {
        if ((t & 31) == 0) producer_copy(p, pl, s);
        return;
    }
    if (warp == MK_PREFETCH_WARP) {
        producer_prefetch(p, pl, s);
        return;
    }

    // ======================= consumers (MK_NCT threads) =======================
    const int H = g.H, L = g.L, hd2 = HD / 2;
    const int par = s.misc()->par, token = s.misc()->token;
    // the launch tag of the tagged words is read from s.misc()->tag where used
    // (the layer loop runs at the register limit)
    const size_t state = (size_t)H;
    float* xa = p.xacc + (size_t)par * 2 * L * state;              // this launch's residual states
    {   // zero the other parity's states for the next launch
        float* xz = p.xacc + (size_t)(par ^ 1) * 2 * L * state;
        const size_t n = 2 * (size_t)L * state;
        const size_t lo = mk_split((int64_t)n, g.nC, c), hi = mk_split((int64_t)n, g.nC, c + 1);
        for (size_t i = lo + t; i < hi; i += MK_NCT) xz[i] = 0.f;
    }
    const uint16_t* emb = p.embed + (size_t)token * H;
    // this CTA's share of the attention (the first A CTAs of each KV group
    // split the positions, the others go from the QKV straight to the combine)
    // and the rows whose residual it adds: s.misc() (ka, ke, has_cur, att, dr0, dr1)
    const int A = p.attn_ctas;
    for (int d = t; d < hd2; d += MK_NCT) {       // RoPE angles of this position
        s.rope()[d] = p.rope_cos[(size_t)p.pos * hd2 + d];
        s.rope()[hd2 + d] = p.rope_sin[(size_t)p.pos * hd2 + d];
    }

    Ring ring;
    bool ab = false;
    // QKV of int rows as integer dot products over the norm output's digits,
    // except in the 8B-width long-context build, where that GEMV beside the
    // tensor-core attention of 128-dim heads spilled 44-48 bytes: there the
    // attention norm writes fp32 and QKV dequantizes its rows to fp32
    constexpr bool QDIG = WB != 2 && !(LC != 0 && MH > 8);

    MK_TRACE(16 * L + 3);
    for (int l = 0; l < L && !ab; ++l) {
        // ---------------- segment A: RMSNorm + QKV GEMV + RoPE + K/V append
        MK_TRACE(16 * l + 0);
        const float* xin = (l == 0) ? nullptr : xa + (size_t)(2 * l - 1) * state;
        if constexpr (QDIG)
            ab = rmsnorm_to_dig<(MH * 32 + MK_NCT - 1) / MK_NCT>(p, s, xin, l == 0 ? emb : nullptr, p.attn_norm + (size_t)l * H,
                                                               ab, s.xres(), pl.orow0, pl.g == 0 ? pl.norows : 0);
        else
            ab = rmsnorm_to_xv<(MH * 256 + MK_NCT - 1) / MK_NCT>(p, s, xin, l == 0 ? emb : nullptr, p.attn_norm + (size_t)l * H, ab, s.xres(), pl.orow0,
                           pl.g == 0 ? pl.norows : 0);
        MK_TRACE(16 * l + 1);
        ab = gemv_fifo<MH, WB, QDIG>(p, s, ring, s.xv(), 2 * pl.npairs, g.TRq, ab, s.part());
        if (t == 0 && p.stream_tail == 2) *(volatile int*)&s.misc()->streaming = 0;
        MK_TRACE(16 * l + 2);
        MK_TRACE_CWAIT(8 * l + 0);
        if (!ab) {
            for (int j = t; j < pl.npairs; j += MK_NCT) {
                const int pair = pl.pair0 + j, slot = pair / hd2, d = pair % hd2;
                float a = wide_row<MH>(s.part(), 2 * j), b = wide_row<MH>(s.part(), 2 * j + 1);
                if (slot <= G) {
                    const float cs = s.rope()[d], sn = s.rope()[hd2 + d];
                    const float a2 = a * cs - b * sn, b2 = b * cs + a * sn;
                    a = a2; b = b2;
                }
                // q and the current K/V go out as tagged words (the debug knob
                // can withhold them, so that the readers' bounded wait runs out)
                const bool pub = !(p.dbg_skip_sync == 4 * l + 0 && p.dbg_skip_cta == c);
                if (slot < G) {
                    uint64_t* q = p.qll + (size_t)l * g.qh * HD + (size_t)(pl.g * G + slot) * HD;
                    if (pub) { st_ll(q + d, ll_pack(a, s.misc()->tag)); st_ll(q + d + hd2, ll_pack(b, s.misc()->tag)); }
                } else {
                    uint16_t* dst = (slot == G ? p.kc : p.vc) + ((size_t)l * g.kvh + pl.g) * g.max_seq * HD;
                    const uint16_t ab16 = f2bf(a), bb16 = f2bf(b);
                    dst[mk_kv_index(p.pos, d, HD, mk_attn_tc(HD, G))] = ab16;
                    dst[mk_kv_index(p.pos, d + hd2, HD, mk_attn_tc(HD, G))] = bb16;
                    uint64_t* kv = p.kvll + (((size_t)l * g.kvh + pl.g) * 2 + (slot - G)) * HD;
                    if (pub) { st_ll(kv + d, ll_pack(bf2f(ab16), s.misc()->tag)); st_ll(kv + d + hd2, ll_pack(bf2f(bb16), s.misc()->tag)); }
                }
            }
        }
        ab = bar_or(ab);
        MK_TRACE(16 * l + 3);
        MK_TRACE(16 * l + 4);

        // ---------------- segment B: split-K attention over this CTA's positions
        MK_TRACE_D(l, 7);        // segment B entered
        {
            // Blocks of up to KB past positions from the ring (the K tile and
            // the V tile of a block are held together); the last attention
            // CTA of the group appends the current position (staged) to its
            // last block, or runs it as a block of its own when it has no past.
            // (att is the same for the whole CTA: the barriers inside stay uniform.)
            if (ldv(s.misc()->att))
                ab = attn_run<HD, G, 1, LC != 0>(p, s, ring, l, ldv(s.misc()->ka), ldv(s.misc()->ke),
                                                 ldv(s.misc()->has_cur) != 0, ab);
        }
        ab = bar_or(ab);
        constexpr int PSTR = G * HD + 2 * G;                   // tagged words per partial
        if (ldv(s.misc()->att) && !ab && !(p.dbg_skip_sync == 4 * l + 1 && p.dbg_skip_cta == c)) {
            constexpr int PPP = LC ? mk_attn_tc_groups(HD) : Attn<HD, G>::NMG;   // parked groups
            uint64_t* dst = p.partll + (((size_t)l * g.kvh + pl.g) * g.CPG + pl.i) * PSTR;
            for (int i = t; i < G * HD; i += MK_NCT) {
                const int h = i / HD;
                float M = -INFINITY;
#pragma unroll
                for (int q = 0; q < PPP; ++q) M = fmaxf(M, s.sc()[q * G + h]);
                float a = 0.f, L = 0.f;
                if (M != -INFINITY) {   // no position at all: an empty partial (m = -inf, l = 0)
#pragma unroll
                    for (int q = 0; q < PPP; ++q) {
                        const float wq = exp2f(s.sc()[q * G + h] - M);
                        a = fmaf(wq, s.xv()[q * (G * HD) + i], a);
                        L = fmaf(wq, s.sc()[PPP * G + q * G + h], L);
                    }
                }
                st_ll(dst + i, ll_pack(a, s.misc()->tag));
                if (i % HD == 0) st_ll2(dst + G * HD + 2 * h, ll_pack(M, s.misc()->tag), ll_pack(L, s.misc()->tag));
            }
        }
        ab = bar_or(ab);
        MK_TRACE(16 * l + 5);
        MK_TRACE_CWAIT(8 * l + 1);
        MK_TRACE(16 * l + 6);

        // combine the group's A partials -> o (the G heads of this KV group):
        // weights exp2(m_j - M) / sum_j exp2(m_j - M) l_j.  A team of CT lanes
        // owns one float4 of o and takes the partials j = lane (mod CT); the
        // team sums with shuffles.  The partials are tagged words polled
        // directly (no flag): the first CB of every thread and the (m, l)
        // words go out in one poll, so a short group costs one L2 round trip
        // once its last member has written.
        if (!ab) {
            constexpr int NO4 = G * HD / 4;                     // float4s of o
            constexpr int CT = (NO4 * 32 <= MK_NCT) ? 32 : (NO4 * 16 <= MK_NCT) ? 16 : (NO4 * 8 <= MK_NCT) ? 8
                             : (NO4 * 4 <= MK_NCT) ? 4 : (NO4 * 2 <= MK_NCT) ? 2 : 1;
            constexpr int CB = MK_COMBINE_LOADS;
            constexpr int NPASS = (NO4 * CT + MK_NCT - 1) / MK_NCT;   // team passes over o
            static_assert(NPASS == 1 || CT == 1, "combine mapping");
            const uint64_t* pg = p.partll + ((size_t)l * g.kvh + pl.g) * g.CPG * PSTR;   // this group's partials
            const int cl_ = t % CT;
            float4 v[CB];
            bool late = false;
            // (o4, batch k0) -> v[]: the tagged words of partials j = cl_ + (k0 + k) * CT,
            // polled until every one carries this launch's tag
            auto load_batch_once = [&](int o4, int k0) {
                bool ok = true;
#pragma unroll
                for (int k = 0; k < CB; ++k) {
                    const int j = cl_ + (k0 + k) * CT;
                    if (o4 < NO4 && j < A) {
                        const uint64_t* w = pg + (size_t)j * PSTR + o4 * 4;
                        const ulonglong2 a = ld_ll2(w), b = ld_ll2(w + 2);
                        ok = ok & ll_ok(a, s.misc()->tag) & ll_ok(b, s.misc()->tag);
                        v[k] = make_float4(__uint_as_float((uint32_t)a.x), __uint_as_float((uint32_t)a.y),
                                           __uint_as_float((uint32_t)b.x), __uint_as_float((uint32_t)b.y));
                    } else {
                        v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                return ok;
            };
            auto load_batch = [&](int o4, int k0) {
                uint64_t t0 = 0;
                for (;;) {
                    if (load_batch_once(o4, k0)) return true;
                    if (!ll_backoff(p, t0)) return false;
                }
            };
            float* cw = s.red();                       // [CPG*G] maxima (red is free here)
            {   // first batch and this thread's (m, l) words in one poll: one round trip
                uint64_t t0 = 0;
                for (;;) {
                    bool ok = load_batch_once(t / CT, 0);
                    for (int i = t; i < A * G; i += MK_NCT) {
                        const ulonglong2 w = ld_ll2(pg + (size_t)(i / G) * PSTR + G * HD + 2 * (i % G));
                        ok = ok & ll_ok(w, s.misc()->tag);
                        cw[i] = __uint_as_float((uint32_t)w.x);
                        s.misc()->cl[i] = __uint_as_float((uint32_t)w.y);
                    }
                    if (ok) break;
                    if (!ll_backoff(p, t0)) { late = true; break; }
                }
            }
            MK_TRACE_D(l, 3);   // thread 0's first partials arrived
            if (bar_or(late)) ab = true;
            MK_TRACE_D(l, 4);   // every thread's first partials arrived
            if (!ab && (t >> 5) < G) {   // warp h: head h, lanes over the partials
                const int hh = t >> 5, ln = t & 31;
                float mx = -INFINITY;
                for (int j = ln; j < A; j += 32) mx = fmaxf(mx, cw[j * G + hh]);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
                float den = 0.f;
                for (int j = ln; j < A; j += 32) {
                    const float mj = cw[j * G + hh];
                    const float wj = (mj == -INFINITY) ? 0.f : exp2f(mj - mx);
                    den = fmaf(wj, s.misc()->cl[j * G + hh], den);
                    s.misc()->cwt[j * G + hh] = wj;
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, o);
                if (ln == 0) s.misc()->alpha[hh] = 1.f / den;
            }
            MK_TRACE_D(l, 10);   // combine weights done (thread 0)
            bar_or(false);
#pragma unroll 1
            for (int ps = 0; ps < NPASS && !ab; ++ps) {
                const int o4 = t / CT + ps * (MK_NCT / CT);
                const int h = (o4 * 4) / HD;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int k0 = 0; k0 * CT < A; k0 += CB) {
                    if (k0 > 0 || ps > 0) {   // further batches (large groups or several passes)
                        if (!load_batch(o4, k0)) late = true;
                    }
#pragma unroll
                    for (int k = 0; k < CB; ++k) {
                        const int j = cl_ + (k0 + k) * CT;
                        if (o4 < NO4 && j < A) {
                            const float wt = s.misc()->cwt[j * G + h];
                            a.x = fmaf(wt, v[k].x, a.x); a.y = fmaf(wt, v[k].y, a.y);
                            a.z = fmaf(wt, v[k].z, a.z); a.w = fmaf(wt, v[k].w, a.w);
                        }
                    }
                }
#pragma unroll
                for (int o = CT >> 1; o >= 1; o >>= 1) {
                    a.x += __shfl_xor_sync(0xFFFFFFFFu, a.x, o); a.y += __shfl_xor_sync(0xFFFFFFFFu, a.y, o);
                    a.z += __shfl_xor_sync(0xFFFFFFFFu, a.z, o); a.w += __shfl_xor_sync(0xFFFFFFFFu, a.w, o);
                }
                if (cl_ == 0 && o4 < NO4) {
                    const float sc = s.misc()->alpha[h];
                    // 4 consecutive values of one head: one half of a split chunk
                    *reinterpret_cast<float4*>(s.ov() + xsplit(o4 * 4, G * HD)) =
                        make_float4(a.x * sc, a.y * sc, a.z * sc, a.w * sc);
                }
            }
            if (late) ab = true;      // made uniform by the barrier below
            MK_TRACE_D(l, 11);   // thread 0's share of o written
        }
        ab = bar_or(ab);
        MK_TRACE(16 * l + 7);

        // O-proj (rows of this CTA, columns of this group) + residual, atomically
        float* xo = xa + (size_t)(2 * l) * state;
        // (the O-proj's slots released before its arithmetic, so the copy producer
        // refills them with gate/up tiles sooner: in the 1B-width long-context
        // build, where it fits the registers; the other builds spilled with it)
        ab = gemv_phase_t<MO, LPRO, WB, false, (KO == 256 && LC != 0 && MH >= 8)>(p, s, ring, s.ov(), pl.norows, g.TRo, s.misc()->ocfg, ab, [&](int r, float v) {
            if (pl.g == 0) v += s.xres()[r];   // group 0 carries the residual of these rows
            atomicAdd(xo + pl.orow0 + r, v);
        }, -1, l, 8);
        MK_TRACE(16 * l + 8);
        MK_TRACE_CWAIT(8 * l + 2);
        if (t == 0 && !ab) arrive(p, mk_cnt_C(g, l), 4 * l + 2);
        MK_TRACE_D(l, 12);   // attention-block arrival issued
        ab = sync_wait(p, mk_cnt_C(g, l), (uint32_t)g.nC, ab);
        MK_TRACE(16 * l + 9);

        // ---------------- segment C: RMSNorm + gate/up + SiLU*up, then down
        if constexpr (WB != 2)
            ab = rmsnorm_to_dig<(MH * 32 + MK_NCT - 1) / MK_NCT>(p, s, xo, nullptr, p.ffn_norm + (size_t)l * H, ab, s.xres2(),
                                                               ldv(s.misc()->dr0), ldv(s.misc()->dr1) - ldv(s.misc()->dr0));
        else
            ab = rmsnorm_to_xv<(MH * 256 + MK_NCT - 1) / MK_NCT>(p, s, xo, nullptr, p.ffn_norm + (size_t)l * H, ab, s.xres2(),
                                                                 ldv(s.misc()->dr0), ldv(s.misc()->dr1) - ldv(s.misc()->dr0));
        MK_TRACE(16 * l + 10);
        if (t == 0) *(volatile int*)&s.misc()->streaming = 1;   // gate/up and down stream
        if (l == 3) trace_ring(p, ring, 4);   // everything before this layer's FFN (discarded)
        {
            // a GU tile holds n gate rows then the n up rows of the same j's
            // (int8: and W_down's column scales of those j's, which the GEMV
            // leaves in u and which multiply into SiLU(gate) * up)
            const int JT = g.JT;
            ab = gemv_fifo<MH, WB>(p, s, ring, s.xv(), 2 * pl.nj, 2 * JT, ab, s.part(), WB != 2 ? s.u() : nullptr);
            for (int j = t; j < pl.nj; j += MK_NCT) {
                const int q = j / JT, jj = j % JT;
                const int n = min(JT, pl.nj - q * JT);
                const float gt = wide_row<MH>(s.part(), q * 2 * JT + jj);
                const float up = wide_row<MH>(s.part(), q * 2 * JT + n + jj);
                s.u()[j] = gt / (1.f + __expf(-gt)) * up * (WB != 2 ? s.u()[j] : 1.f);
            }
        }
        MK_TRACE(16 * l + 11);
        MK_TRACE_CWAIT(8 * l + 3);
        if (l == 3) trace_ring(p, ring, 0);
        // down projection: this CTA's FFN columns j, all H rows (split-K).  A D
        // tile is [j][H] bf16.  The consumer threads form P groups of TP
        // threads that take turns on the tiles (tile b goes to group b % P), and
        // thread tp of a group owns the 8-row chunks tp + m*TP (m < CPT) of the
        // output, so a warp reads 32 consecutive 16-byte chunks of one column.
        // The phases' partial sums are folded through xv (P-1 -> ... -> 0),
        // then phase 0 adds the residual of this CTA's rows and reduces into
        // the residual stream with vector atomics.
        ab = bar_or(ab);                                        // u complete, xv free
        float* xf = xa + (size_t)(2 * l + 1) * state;
        {
            constexpr int NCH = 32 * MH;                        // 8-row chunks of H
            constexpr int TP = NCH < 128 ? NCH : 128;           // threads per j-phase
            constexpr int P = MK_NCT / TP;                      // j-phases
            constexpr int CPT = NCH / TP;                       // chunks per thread
            static_assert(MK_NCT % TP == 0 && NCH % TP == 0 && P >= 2, "down-projection mapping");
            const int jp = t / TP, tp = t % TP;
            float2 da[CPT][4];
#pragma unroll
            for (int m = 0; m < CPT; ++m)
#pragma unroll
                for (int k = 0; k < 4; ++k) da[m][k] = make_float2(0.f, 0.f);
            for (int j0 = 0, b = 0; j0 < pl.nj && !ab; j0 += g.JD, ++b) {
                if (b % P != jp) { ring.advance(p.geo.ns); continue; }   // another group's tile
                const int n = min(g.JD, pl.nj - j0);
                const uint8_t* tile;
                const bool ok = take_tile(p, s, ring, (uint32_t)(n * wrow_bytes<WB>(H)), tile);
                if constexpr (TP == 128 && CPT <= 2 && !LC && WB == 2) {
                    // a thread's share is 16 chunks (slots of 32 KB): loaded
                    // whole, then the slot is released before the arithmetic
                    // (not in the long-context build, whose attention already
                    // holds more registers)
                    constexpr int NJ = 16 / CPT;
                    uint4 wv[NJ][CPT];
#pragma unroll
                    for (int jj = 0; jj < NJ; ++jj)
#pragma unroll
                        for (int m = 0; m < CPT; ++m)
                            wv[jj][m] = (ok && jj < n) ? lds128(tile + (size_t)jj * H * 2 + (size_t)(tp + m * TP) * 16)
                                                       : make_uint4(0u, 0u, 0u, 0u);
                    release_tile(p, s, ring, (uint32_t)P);  // TP / 32 readers, weight P each
#pragma unroll
                    for (int jj = 0; jj < NJ; ++jj) {
                        if (ok && jj < n) {
                            const float uj = s.u()[j0 + jj];
                            const float2 u2 = make_float2(uj, uj);
#pragma unroll
                            for (int m = 0; m < CPT; ++m) {
                                da[m][0] = __ffma2_rn(bf2_lo_hi(wv[jj][m].x), u2, da[m][0]);
                                da[m][1] = __ffma2_rn(bf2_lo_hi(wv[jj][m].y), u2, da[m][1]);
                                da[m][2] = __ffma2_rn(bf2_lo_hi(wv[jj][m].z), u2, da[m][2]);
                                da[m][3] = __ffma2_rn(bf2_lo_hi(wv[jj][m].w), u2, da[m][3]);
                            }
                        }
                    }
                } else {
                    if (ok) {
#pragma unroll (CPT <= 2 ? 2 : 1)
                        for (int jj = 0; jj < n; ++jj) {
                            const float uj = s.u()[j0 + jj];
                            const float2 u2 = make_float2(uj, uj);
                            const uint8_t* col = tile + (size_t)jj * wrow_bytes<WB>(H);
#pragma unroll
                            for (int m = 0; m < CPT; ++m) {
                                if constexpr (WB == 2) {
                                    const uint4 w = lds128(col + (size_t)(tp + m * TP) * 16);
                                    da[m][0] = __ffma2_rn(bf2_lo_hi(w.x), u2, da[m][0]);
                                    da[m][1] = __ffma2_rn(bf2_lo_hi(w.y), u2, da[m][1]);
                                    da[m][2] = __ffma2_rn(bf2_lo_hi(w.z), u2, da[m][2]);
                                    da[m][3] = __ffma2_rn(bf2_lo_hi(w.w), u2, da[m][3]);
                                } else if constexpr (WB == 1) {   // 8 rows of int8 (u already carries W_down's column scale)
                                    const uint2 w = lds64(col + (size_t)(tp + m * TP) * 8);
                                    const uint32_t lo = w.x, hi = w.y;
                                    da[m][0] = __ffma2_rn(i8pair(lo, 0), u2, da[m][0]);
                                    da[m][1] = __ffma2_rn(i8pair(lo, 2), u2, da[m][1]);
                                    da[m][2] = __ffma2_rn(i8pair(hi, 0), u2, da[m][2]);
                                    da[m][3] = __ffma2_rn(i8pair(hi, 2), u2, da[m][3]);
                                } else {   // 8 rows of int4 (low nibbles rows 0-3, high ones rows 4-7)
                                    const uint32_t w = lds32(col + (size_t)(tp + m * TP) * 4);
                                    const uint32_t lo = nib_lo(w), hi = nib_hi(w);
                                    da[m][0] = __ffma2_rn(i4pair(lo, 0), u2, da[m][0]);
                                    da[m][1] = __ffma2_rn(i4pair(lo, 2), u2, da[m][1]);
                                    da[m][2] = __ffma2_rn(i4pair(hi, 0), u2, da[m][2]);
                                    da[m][3] = __ffma2_rn(i4pair(hi, 2), u2, da[m][3]);
                                }
                            }
                        }
                    }
                    release_tile(p, s, ring, (uint32_t)P);  // TP / 32 readers, weight P each
                }
                if (!ok) ab = true;     // this warp gave up; the barrier below makes it uniform
            }
            MK_TRACE(16 * l + 14);
            if (t == 0 && p.stream_tail == 0) *(volatile int*)&s.misc()->streaming = 0;
            if (l == 3) trace_ring(p, ring, 1);
            // fold the phases: phase q adds what phase q+1 left in xv (element
            // e of chunk c at xv[e * NCH + c]: lane-consecutive, conflict free)
#pragma unroll 1
            for (int q = P - 1; q >= 0; --q) {
                if (q < P - 1) ab = bar_or(ab);
                if (jp == q && !ab) {
#pragma unroll
                    for (int m = 0; m < CPT; ++m) {
                        const int cc = tp + m * TP;
                        if (q < P - 1) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                da[m][k].x += s.xv()[(2 * k) * NCH + cc];
                                da[m][k].y += s.xv()[(2 * k + 1) * NCH + cc];
                            }
                        }
                        if (q > 0) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                s.xv()[(2 * k) * NCH + cc] = da[m][k].x;
                                s.xv()[(2 * k + 1) * NCH + cc] = da[m][k].y;
                            }
                        } else {
                            // rows 8cc .. 8cc+7; this CTA carries the residual of rows [dr0, dr1)
                            const int dr0 = ldv(s.misc()->dr0), dr1 = ldv(s.misc()->dr1);
                            float r[8] = {da[m][0].x, da[m][0].y, da[m][1].x, da[m][1].y,
                                          da[m][2].x, da[m][2].y, da[m][3].x, da[m][3].y};
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int rr = 8 * cc + e - dr0;
                                if ((unsigned)rr < (unsigned)(dr1 - dr0)) r[e] += s.xres2()[rr];
                            }
                            red_add_v4(xf + 8 * cc, make_float4(r[0], r[1], r[2], r[3]));
                            red_add_v4(xf + 8 * cc + 4, make_float4(r[4], r[5], r[6], r[7]));
                        }
                    }
                }
            }
            MK_TRACE(16 * l + 15);
        }
        ab = bar_or(ab);
        MK_TRACE(16 * l + 12);
        MK_TRACE_CWAIT(8 * l + 4);
        if (t == 0 && !ab) arrive(p, mk_cnt_E(g, l), 4 * l + 3);
        ab = sync_wait(p, mk_cnt_E(g, l), (uint32_t)g.nC, ab);
        if (t == 0 && p.stream_tail == 1) *(volatile int*)&s.misc()->streaming = 0;
        MK_TRACE(16 * l + 13);
    }

    // ---------------- final RMSNorm + LM head + argmax
    {
        const float* xl = xa + (size_t)(2 * L - 1) * state;
        if constexpr (WB != 2)
            ab = rmsnorm_to_dig<(MH * 32 + MK_NCT - 1) / MK_NCT>(p, s, xl, nullptr, p.final_norm, ab, nullptr, 0, 0,
                                                               c == 0 ? p.hidden : nullptr);
        else
            ab = rmsnorm_to_xv<(MH * 256 + MK_NCT - 1) / MK_NCT>(p, s, xl, nullptr, p.final_norm, ab, nullptr, 0, 0);
        MK_TRACE(16 * L + 0);
        if (t == 0) *(volatile int*)&s.misc()->streaming = 1;   // the LM head streams
        if (WB == 2 && c == 0 && !ab)
            for (int i = t; i < H; i += MK_NCT) p.hidden[i] = s.xv()[xsplit(i, H)];
        float bv = -INFINITY;
        int bi = -1;
        bool nonfinite = false;
        // top-p: the logits go to scratch and the phase only finds max(logit / T)
        const bool topp = p.inv_temp > 0.f && p.top_p < 1.f;
        ab = gemv_phase_t<MH, 32, WB, WB != 2>(p, s, ring, s.xv(), pl.nv, g.TRh, s.misc()->lmcfg, ab, [&](int r, float lg) {
            const int v = pl.v0 + r;
            if (p.logits) p.logits[v] = lg;
            if (isfinite(lg)) {
                if (topp) {
                    p.lgs[v] = lg;
                    bv = fmaxf(bv, lg * p.inv_temp);
                } else {
                    // greedy: the logit; sampling: logit / T plus this token's Gumbel noise
                    // (inline behind a uniform branch: measured the cheapest form for greedy steps)
                    const float key = p.inv_temp > 0.f ? fmaf(lg, p.inv_temp, mk_gumbel(p.seed, p.pos, v)) : lg;
                    if (key > bv || (key == bv && v < bi)) { bv = key; bi = v; }
                }
            } else {
                if (topp) p.lgs[v] = lg;
                nonfinite = true;
            }
        }, 2048);
        MK_TRACE(16 * L + 1);
        MK_TRACE_CWAIT(8 * L + 5);
        if (nonfinite) atomicOr(p.status, MK_ST_NUMERIC);
        if (topp) {
            // Nucleus (cloud.baidu.com/article/9434380, section 5, step 1: top-p
            // beside the temperature): with x = logit / T, keep the tokens whose
            // strictly more probable tokens carry less than p of the mass, then
            // Gumbel-max among them.  The threshold is found by bisection on x:
            // the interval (lo, hi] holds it, with mass(x > lo) >= p Z and
            // mass(x > hi) < p Z; each round splits it at 32 candidates, every
            // CTA adds the exp(x - M) of its logits into the 33 intervals, the
            // sums meet in global memory across a grid-wide barrier, and every
            // CTA keeps the sub-interval where the mass above crosses p Z.  After
            // MK_TP_ITERS rounds the kept tokens are those with x > lo.
            float* hs = s.red();                  // [0, 33) interval masses; [40..42] lo, hi, pZ
            if ((t & 31) == 0) s.misc()->best_val[t >> 5] = bv;
            ab = bar_or(ab);
            if (t == 0 && !ab) {
                float m = -INFINITY;
                for (int i = 0; i < MK_NCW; ++i) m = fmaxf(m, s.misc()->best_val[i]);
                if (m != -INFINITY) atomicMax(&p.tp->mkey, (unsigned long long)f2key(m));
            }
            ab = grid_sync(p, mk_cnt_tp(g, 0), ab);
            const unsigned long long mk_ = __ldcg(&p.tp->mkey);
            const float M = mk_ ? key2f((uint32_t)mk_) : 0.f;
            if (t == 0) { hs[40] = M - 104.f; hs[41] = M; hs[42] = 0.f; }
            for (int it = 0; it < MK_TP_ITERS && !ab; ++it) {
                if (t < MK_TP_BINS) hs[t] = 0.f;
                ab = bar_or(ab);
                const float lo = hs[40], hi = hs[41], w = (hi - lo) * (1.f / 32.f);
                for (int r = t; r < pl.nv; r += MK_NCT) {
                    const float y = __ldcg(p.lgs + pl.v0 + r);
                    const float x = y * p.inv_temp;
                    if (!isfinite(y) || !(x > lo)) continue;
                    // interval b: tau_b < x <= tau_b+1, tau_k = lo + k w (tau_32 = hi); 32: x > hi
                    int b = 32;
                    if (!(x > hi)) {
                        b = min(31, max(0, (int)((x - lo) / w)));
                        while (b > 0 && !(fmaf(w, (float)b, lo) < x)) --b;
                        while (b < 31 && fmaf(w, (float)(b + 1), lo) < x) ++b;
                    }
                    atomicAdd(&hs[b], exp2f((x - M) * 1.4426950408889634f));
                }
                ab = bar_or(ab);
                if (t < MK_TP_BINS && !ab && hs[t] != 0.f) atomicAdd(&p.tp->hist[it][t], hs[t]);
                ab = grid_sync(p, mk_cnt_tp(g, it + 1), ab);
                if (t == 0 && !ab) {
                    // C_k = mass(x > tau_k) = sum of intervals k .. 32
                    float cs[MK_TP_BINS];
                    float cum = 0.f;
                    for (int k = MK_TP_BINS - 1; k >= 0; --k) { cum += __ldcg(&p.tp->hist[it][k]); cs[k] = cum; }
                    float pz = hs[42];
                    if (it == 0) { pz = p.top_p * cs[0]; hs[42] = pz; }
                    int ks = 0;                       // the last candidate with mass above >= p Z
                    for (int k = 31; k > 0; --k) if (cs[k] >= pz) { ks = k; break; }
                    hs[40] = ks == 0 ? lo : fmaf(w, (float)ks, lo);
                    hs[41] = ks == 31 ? hi : fmaf(w, (float)(ks + 1), lo);
                }
                ab = bar_or(ab);
            }
            // Gumbel-max over the kept tokens
            const float lo = hs[40];
            bv = -INFINITY;
            bi = -1;
            for (int r = t; r < pl.nv; r += MK_NCT) {
                const int v = pl.v0 + r;
                const float y = __ldcg(p.lgs + v);
                if (!isfinite(y) || !(y * p.inv_temp > lo)) continue;
                const float key = fmaf(y, p.inv_temp, mk_gumbel(p.seed, p.pos, v));
                if (key > bv || (key == bv && v < bi)) { bv = key; bi = v; }
            }
            // the thread's best into lane 0 of its warp (as the phase above leaves it)
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
                const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
                if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) { bv = ov; bi = oi; }
            }
        }
        if ((t & 31) == 0) { s.misc()->best_val[t >> 5] = bv; s.misc()->best_idx[t >> 5] = bi; }
        ab = bar_or(ab);
        if (t == 0 && !ab) {
            float v = -INFINITY;
            int idx = -1;
            for (int i = 0; i < MK_NCW; ++i) {
                const int ii = s.misc()->best_idx[i];
                const float vv = s.misc()->best_val[i];
                if (ii >= 0 && (idx < 0 || vv > v || (vv == v && ii < idx))) { v = vv; idx = ii; }
            }
            if (idx >= 0) {
                uint32_t u = __float_as_uint(v);
                u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
                const unsigned long long key = ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)idx);
                atomicMax(p.amax, key);
            }
        }
    }

    // ---------------- end of step: the last CTA publishes the token and resets the flags
    MK_TRACE(16 * L + 2);
    if (t == 0 && ab) s.misc()->abort = 1;   // lets the producer warps stop and drain
    if (t == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(p.cnt + mk_cnt_done(g), 1u);
        s.misc()->is_last = (prev == (uint32_t)g.nC - 1) ? 1 : 0;
    }
    bar_or(false);
    if (s.misc()->is_last) {
        __threadfence();
        const int ntot = mk_cnt_done(g);
        for (int i = t; i < ntot; i += MK_NCT) p.cnt[i] = 0u;
        if (t == 0) {
            const unsigned long long key = atomicMax(p.amax, 0ull);
            int tok = 0;
            if (key == 0ull) atomicOr(p.status, MK_ST_NUMERIC);
            else tok = (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
            *p.next_token = tok;
            if (p.tokens_out) p.tokens_out[p.out_idx] = tok;
            if (p.stop && p.tokens_out && tok == p.eos_id) *p.stop = 1;   // generated the stop token
            *p.amax = 0ull;
            if (p.inv_temp > 0.f && p.top_p < 1.f) {
                p.tp->mkey = 0ull;
                for (int k = 0; k < MK_TP_ITERS; ++k)
                    for (int b = 0; b < MK_TP_BINS; ++b) p.tp->hist[k][b] = 0.f;
            }
            p.cnt[ntot] = 0u;
            atomicAdd(p.seq, 1u);
            atomicAnd(p.status, ~MK_ST_ABORT);
            __threadfence();
        }
    }
}

}  // namespace
}  // namespace mk


