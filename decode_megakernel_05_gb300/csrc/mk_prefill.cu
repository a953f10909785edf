// mk_prefill.cu - batched prefill: the prompt's rows go through every layer
// together, as dense products on the tensor cores, instead of one decode
// launch per prompt token (cloud.baidu.com/article/9434380, sections 2 and 8,
// problem 2: prefill and decode are separate phases with different
// bottlenecks; the prompt is a dense, compute-bound contraction where decode
// is a GEMV).
//
// Per layer, over the n prompt rows (positions start .. start + n - 1):
//   RMSNorm -> QKV GEMM -> RoPE, K/V rows written to the cache (bf16, the
//   cache's layout) -> causal attention over the cache [0, position] ->
//   O-proj GEMM + residual -> RMSNorm -> gate/up GEMM -> SiLU(gate) * up ->
//   down GEMM + residual;
// then the final RMSNorm of the last row, the LM head and the greedy argmax,
// which leaves the next token where a following decode step reads it.
//
// The GEMMs run on mma.sync m16n8k16 (bf16 inputs, fp32 accumulation) with
// the weights as stored (bf16) and every fp32 activation split into three
// bf16 parts (its rounding, the rounding of the remainder, the rounding of
// what is left), three products per tile: the parts carry the activation to
// about 2^-26 relative, as exactly as the decode path's fp32 activations.
// (Two parts, 2^-17, were measured first: after 16 layers of attention the
// K/V rows drifted to 80% bit-equal with the token-by-token oracle.)
#include <cuda.h>   // CUtensorMap and its enums; the encoder itself comes through the runtime
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mk_prefill.h"

namespace {

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Element of dim d of position p in one KV head's cache rows (swz: the row's
// 16-byte chunk index XORed with p mod 8, the layout the long-context
// attention reads).
__device__ __forceinline__ int64_t kv_index(int64_t p, int d, int hd, int swz) {
    const int c = d >> 3;
    return p * hd + (((swz ? (c ^ (int)(p & 7)) : c) << 3) | (d & 7));
}

// ---------------------------------------------------------------- GEMM
//
// C[M][N] = A[M][K] . W[N][K]^T (+ R[M][N]), A fp32 row-major, W bf16
// row-major (its rows are the output features), C and R fp32 row-major.
// CTA tile 64 x 128, k-steps of 32, 4 warps each 32 x 64 (2 x 8 mma tiles),
// two shared-memory stages: the weight tile arrives by cp.async (16 bytes, the
// K tail zero-filled), the activation tile is loaded to registers, split into
// its three bf16 parts and stored while the previous stage is multiplied.
// Rows are padded to 40 bf16 (80 bytes) so the 8x8 matrix loads hit eight
// different 16-byte bank groups.
constexpr int GBM = 64, GBN = 128, GBK = 32, GLD = 40;

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// bf16x2 of (x, y), x in the low half, round to nearest even
__device__ __forceinline__ uint32_t pack_bf2(float x, float y) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(y), "f"(x));
    return r;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

struct GemmSmem {
    uint16_t a[3][2][GBM][GLD];   // activation parts (high, middle, low) x stage
    uint16_t b[2][GBN][GLD];
};

template <bool RES>
__global__ void __launch_bounds__(128) gemm_split_kernel(const float* __restrict__ A, const uint16_t* __restrict__ W,
                                                         const float* R, float* C, int M, int N, int K) {
    extern __shared__ __align__(16) uint8_t gemm_smem[];
    GemmSmem& sm = *reinterpret_cast<GemmSmem*>(gemm_smem);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int m0 = blockIdx.y * GBM, n0 = blockIdx.x * GBN;
    const int wm = (warp >> 1) * 32, wn = (warp & 1) * 64;   // the warp's 32 x 64 sub-tile
    const int nk = (K + GBK - 1) / GBK;
    float acc[2][8][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

    float4 areg[4];
    // activation tile kt -> registers (float4 f = t + 128 q: row f / 8, columns 4 (f % 8) ..)
    auto load_a = [&](int kt) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int f = t + 128 * q, r = f >> 3, c = (f & 7) * 4;
            const int gr = m0 + r, gc = kt * GBK + c;
            areg[q] = (gr < M && gc < K) ? *reinterpret_cast<const float4*>(A + (size_t)gr * K + gc)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto store_a = [&](int st) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int f = t + 128 * q, r = f >> 3, c = (f & 7) * 4;
            float e[4] = {areg[q].x, areg[q].y, areg[q].z, areg[q].w};
#pragma unroll
            for (int part = 0; part < 3; ++part) {   // each part the bf16 rounding of what the earlier leave
                const uint32_t p01 = pack_bf2(e[0], e[1]), p23 = pack_bf2(e[2], e[3]);
                *reinterpret_cast<uint2*>(&sm.a[part][st][r][c]) = make_uint2(p01, p23);
                e[0] -= __uint_as_float(p01 << 16);
                e[1] -= __uint_as_float(p01 & 0xFFFF0000u);
                e[2] -= __uint_as_float(p23 << 16);
                e[3] -= __uint_as_float(p23 & 0xFFFF0000u);
            }
        }
    };
    // weight tile kt -> stage st (16-byte pieces idx = t + 128 q: row idx / 4, piece idx % 4)
    auto load_b = [&](int kt, int st) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = t + 128 * q, r = idx >> 2, seg = idx & 3;
            const int gn = n0 + r, gk = kt * GBK + seg * 8;
            const bool in = gn < N && gk < K;
            const uint16_t* src = in ? W + (size_t)gn * K + gk : W;
            cp_async16(smem_u32(&sm.b[st][r][seg * 8]), src, in ? 16u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    load_a(0);
    load_b(0, 0);
    store_a(0);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    for (int kt = 0; kt < nk; ++kt) {
        const int st = kt & 1;
        const bool more = kt + 1 < nk;
        if (more) {
            load_b(kt + 1, st ^ 1);
            load_a(kt + 1);
        }
#pragma unroll
        for (int kk = 0; kk < GBK; kk += 16) {
            uint32_t af[3][2][4];   // the three parts' fragments of the warp's two m-tiles
#pragma unroll
            for (int part = 0; part < 3; ++part)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int r = wm + 16 * i + (lane & 15), c = kk + (lane >> 4) * 8;
                    ldsm_x4(af[part][i], smem_u32(&sm.a[part][st][r][c]));
                }
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                uint32_t bb[4];   // n-tiles j and j+1: b0, b1 of each
                const int r = wn + 8 * j + (lane & 7) + ((lane >> 4) << 3), c = kk + ((lane >> 3) & 1) * 8;
                ldsm_x4(bb, smem_u32(&sm.b[st][r][c]));
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int part = 2; part >= 0; --part) {   // smallest part first
                        mma_bf16(acc[i][j], af[part][i], bb[0], bb[1]);
                        mma_bf16(acc[i][j + 1], af[part][i], bb[2], bb[3]);
                    }
            }
        }
        if (more) {
            store_a(st ^ 1);
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
    }
    // accumulator (i, j): rows wm + 16 i + lane / 4 (+ 8), columns wn + 8 j + 2 (lane % 4) (+ 1)
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = m0 + wm + 16 * i + (lane >> 2) + 8 * h;
                const int c = n0 + wn + 8 * j + 2 * (lane & 3);
                if (r >= M) continue;
                float v0 = acc[i][j][2 * h], v1 = acc[i][j][2 * h + 1];
                float* dst = C + (size_t)r * N + c;
                if ((N & 1) == 0 && c + 1 < N) {   // 8-byte aligned pair
                    if (RES) { const float2 q = *reinterpret_cast<const float2*>(R + (size_t)r * N + c); v0 += q.x; v1 += q.y; }
                    *reinterpret_cast<float2*>(dst) = make_float2(v0, v1);
                } else {
                    if (c < N) dst[0] = v0 + (RES ? R[(size_t)r * N + c] : 0.f);
                    if (c + 1 < N) dst[1] = v1 + (RES ? R[(size_t)r * N + c + 1] : 0.f);
                }
            }
}

// ---------------------------------------------------------------- tcgen05 GEMM
//
// The same product on the fifth-generation tensor cores.  A's three bf16 parts
// come from the kernel that produced A (RMSNorm, attention, SiLU * up write
// them instead of fp32), stored [3][rows][K]; the tensor map sees them as a
// [3][M][K] box grid, so rows past M read as zero.  A CTA owns a 128 x 128 tile
// of C (128 x 256 for wide outputs: half the activation re-reads from L2) and
// walks K in blocks of 64 (one 128-byte row of each operand):
//   - warp 0, one thread: TMA (cp.async.bulk.tensor) copies of the three A
//     part tiles and the W tile of a K block into one of three stages, with
//     the 128-byte swizzle, completing on the stage's full barrier;
//   - warp 1: allocates BN TMEM columns (the fp32 accumulator: lane = row
//     of the tile, column = column); one thread issues, per K block, 12
//     tcgen05.mma (3 parts x 4 steps of K = 16, M = 128, N = BN, bf16 in,
//     fp32 accumulate, smallest part first) and commits them to the stage's
//     empty barrier, and after the last block to the done barrier;
//   - warps 2-5: wait for done, read the accumulator with tcgen05.ld (warp w
//     reads TMEM lanes 32 (w mod 4) ..), add the residual and store C; or,
//     when the residual is C itself, add the product into C with vector
//     atomics, which lets ksplit CTAs (grid z) share one tile's K range (the
//     outputs of 2048 columns would otherwise fill 64 of the 152 SMs).
// Every wait is bounded (%globaltimer, 2 s); a time-out sets the time-out bit
// (0x1) of the status word and the CTA still frees its TMEM.  The K tail and the rows of W
// past N come in as zeros (TMA's out-of-bounds fill).
constexpr int TBM = 128, TBK = 64;
constexpr uint32_t T_PART = TBM * TBK * 2;                  // 16 KB: one part's A tile
constexpr uint64_t T_WAIT_NS = 2000000000ull;
// Tile width, stages and shared memory per width: 128 wide in 3 stages of 64 KB, 256 wide in 2 of 80 KB.
template <int BN> struct TcCfg {
    static constexpr int ST = BN == 256 ? 2 : 3;
    static constexpr uint32_t WT = (uint32_t)BN * TBK * 2;          // the W tile
    static constexpr uint32_t STAGE = 3 * T_PART + WT;
    static constexpr uint32_t SMEM = ST * STAGE + 1024 + 128;       // stages, alignment slack, barriers
    // instruction descriptor: kind::f16, bf16 A and B (both K-major), fp32 D, M = 128, N = BN
    static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                      ((uint32_t)(TBM >> 4) << 24);
};

__device__ __forceinline__ uint64_t gtimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Bounded wait for phase `parity` of an mbarrier; false (and the status bit) on time-out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* status) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = gtimer_ns();
    while (!mbar_try(bar, parity)) {
        if (gtimer_ns() - t0 > T_WAIT_NS) {
            atomicOr(status, 0x1u);
            return false;
        }
    }
    return true;
}
// Shared-memory matrix descriptor of a K-major operand tile with the 128-byte
// swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);   // start address / 16
    d |= (uint64_t)1 << 16;                              // leading-dimension offset (not used with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;                    // stride between 8-row groups / 16
    d |= (uint64_t)1 << 46;                              // descriptor version
    d |= (uint64_t)2 << 61;                              // 128-byte swizzle
    return d;
}
template <int BN>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, const float* R,
                   float* C, int M, int N, int K, int ksplit, uint32_t* status) {
    using Cfg = TcCfg<BN>;
    constexpr int TST = Cfg::ST;
    constexpr int TBN = BN;
    constexpr uint32_t T_STAGE = Cfg::STAGE, T_IDESC = Cfg::IDESC;
    extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
    // the stages need 1024-byte alignment (the swizzle pattern repeats every 8 rows of 128 bytes)
    const uint32_t raw = smem_u32(tc_smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + TST * T_STAGE;           // full[TST], empty[TST], done, then the TMEM address
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (TST + s); };
    const uint32_t done = bars + 8u * (2 * TST);
    const uint32_t taddr_slot = done + 8u;
    uint32_t* taddr_ptr = reinterpret_cast<uint32_t*>(tc_smem_raw + (taddr_slot - raw));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * TBM, n0 = blockIdx.x * TBN;
    // this CTA's K blocks [kb0, kb0 + nkb); ksplit > 1 only with the atomic epilogue (R == C)
    const int nkb_all = (K + TBK - 1) / TBK;
    const int kb0 = (int)(((int64_t)blockIdx.z * nkb_all) / ksplit);
    const int nkb = (int)(((int64_t)(blockIdx.z + 1) * nkb_all) / ksplit) - kb0;
    const bool atomic_add = R == C;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TST; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(taddr_slot),
                     "r"((uint32_t)TBN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(taddr_ptr);

    if (warp == 0 && lane == 0) {
        // producer
        const uint64_t pa = reinterpret_cast<uint64_t>(&tmA), pw = reinterpret_cast<uint64_t>(&tmW);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % TST;
            const uint32_t ph = (uint32_t)(kb / TST) & 1u;
            if (kb >= TST && !mbar_wait(empty(s), ph ^ 1u, status)) break;
            const uint32_t st = base + (uint32_t)s * T_STAGE;
            mbar_expect(full(s), T_STAGE);
            for (int part = 0; part < 3; ++part)
                asm volatile(
                    "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
                    "%4}], [%5];" ::"r"(st + (uint32_t)part * T_PART),
                    "l"(pa), "r"((kb0 + kb) * TBK), "r"(m0), "r"(part), "r"(full(s))
                    : "memory");
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
                "[%4];" ::"r"(st + 3u * T_PART),
                "l"(pw), "r"((kb0 + kb) * TBK), "r"(n0), "r"(full(s))
                : "memory");
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        bool ok = true;
        for (int kb = 0; kb < nkb && ok; ++kb) {
            const int s = kb % TST;
            const uint32_t ph = (uint32_t)(kb / TST) & 1u;
            if (!mbar_wait(full(s), ph, status)) { ok = false; break; }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t st = base + (uint32_t)s * T_STAGE;
            const uint64_t wd = sw128_desc(st + 3u * T_PART);
            for (int part = 2; part >= 0; --part) {
                const uint64_t ad = sw128_desc(st + (uint32_t)part * T_PART);
#pragma unroll
                for (int kk = 0; kk < TBK / 16; ++kk) {
                    // advancing K by 16 bf16 (32 bytes) inside the swizzle row: start address + 2 (16-byte units)
                    const uint32_t acc = (kb > 0 || part < 2 || kk > 0) ? 1u : 0u;
                    asm volatile(
                        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
                        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(tmem),
                        "l"(ad + 2ull * kk), "l"(wd + 2ull * kk), "r"(T_IDESC), "r"(acc)
                        : "memory");
                }
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(empty(s))
                         : "memory");
        }
        if (ok)
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(done)
                         : "memory");
    } else if (warp >= 2) {
        // epilogue: TMEM lanes 32 q .. 32 q + 31 are rows m0 + 32 q + lane
        const bool ok = mbar_wait(done, 0u, status);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int q = warp & 3;
        const int row = m0 + 32 * q + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < TBN && ok; c0 += 32) {
            uint32_t v[32];
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
                "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                  "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                  "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
                  "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                : "r"(ta)
                : "memory");
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (row < M && atomic_add) {
                const int cb = n0 + c0;
                float* dst = C + (size_t)row * N + cb;
                if ((N & 3) == 0 && cb + 32 <= N) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + j), "f"(__uint_as_float(v[j])),
                                     "f"(__uint_as_float(v[j + 1])), "f"(__uint_as_float(v[j + 2])),
                                     "f"(__uint_as_float(v[j + 3]))
                                     : "memory");
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (cb + j < N) atomicAdd(dst + j, __uint_as_float(v[j]));
                }
            } else if (row < M) {
                const int cb = n0 + c0;
                float* dst = C + (size_t)row * N + cb;
                const float* res = R ? R + (size_t)row * N + cb : nullptr;
                if ((N & 3) == 0 && cb + 32 <= N) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        float4 o = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                               __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
                        if (res) {
                            const float4 r4 = *reinterpret_cast<const float4*>(res + j);
                            o.x += r4.x; o.y += r4.y; o.z += r4.z; o.w += r4.w;
                        }
                        *reinterpret_cast<float4*>(dst + j) = o;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (cb + j < N) dst[j] = __uint_as_float(v[j]) + (res ? res[j] : 0.f);
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)TBN)
                     : "memory");
    }
}

// The three bf16 parts of v (its rounding, the rounding of the remainder, and
// of what is left) at P[i], P[i + ps], P[i + 2 ps]; a pair (x, y) at i, i + 1.
__device__ __forceinline__ void store_parts2(uint16_t* P, size_t ps, size_t i, float x, float y) {
#pragma unroll
    for (int part = 0; part < 3; ++part) {
        const uint32_t b = pack_bf2(x, y);
        *reinterpret_cast<uint32_t*>(P + part * ps + i) = b;
        x -= __uint_as_float(b << 16);
        y -= __uint_as_float(b & 0xFFFF0000u);
    }
}

// ---------------------------------------------------------------- row kernels

__global__ void embed_rows_kernel(const uint16_t* E, const int32_t* tok, int n, int V, int H, float* X,
                                  uint32_t* status) {
    const int i = blockIdx.x;
    int tk = tok[i];
    if (tk < 0 || tk >= V) {
        if (threadIdx.x == 0) atomicOr(status, 0x4u);
        tk = 0;
    }
    for (int d = threadIdx.x; d < H; d += blockDim.x) X[(size_t)i * H + d] = bf(E[(size_t)tk * H + d]);
}

// y = x / sqrt(mean(x^2) + eps) * g for row blockIdx.x, to Y (fp32) and/or
// to the parts P (row stride H, part stride ps).
__global__ void rmsnorm_rows_kernel(const float* X, const float* g, int H, float eps, float* Y, uint16_t* P,
                                    size_t ps) {
    __shared__ float red[32];
    const float* x = X + (size_t)blockIdx.x * H;
    float ss = 0.f;
    for (int d = threadIdx.x; d < H; d += blockDim.x) ss = fmaf(x[d], x[d], ss);
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    const float inv = rsqrtf(tot / (float)H + eps);
    if (Y) {
        float* y = Y + (size_t)blockIdx.x * H;
        for (int d = threadIdx.x; d < H; d += blockDim.x) y[d] = x[d] * inv * g[d];
    }
    if (P)
        for (int d = 2 * threadIdx.x; d < H; d += 2 * blockDim.x)
            store_parts2(P, ps, (size_t)blockIdx.x * H + d, x[d] * inv * g[d], x[d + 1] * inv * g[d + 1]);
}

// RoPE on the q and k heads of row blockIdx.y (position start + row), then the
// K and V rows to the cache as bf16; q stays fp32 in place.
__global__ void rope_kv_rows_kernel(float* QKV, int nqkv, const float* cs, const float* sn, int start, int qh,
                                    int kvh, int hd, int max_seq, int layer, uint16_t* kc, uint16_t* vc, int swz) {
    const int half = hd / 2, row = blockIdx.y, pos = start + row;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (qh + 2 * kvh) * half) return;
    const int h = idx / half, d = idx % half;
    float* v = QKV + (size_t)row * nqkv + (size_t)h * hd;
    float a = v[d], b = v[d + half];
    if (h < qh + kvh) {
        const float c = cs[(size_t)pos * half + d], s = sn[(size_t)pos * half + d];
        const float a2 = a * c - b * s, b2 = b * c + a * s;
        a = a2;
        b = b2;
    }
    if (h < qh) {
        v[d] = a;
        v[d + half] = b;
    } else {
        const int g = (h < qh + kvh) ? h - qh : h - qh - kvh;
        uint16_t* dst = ((h < qh + kvh) ? kc : vc) + ((size_t)layer * kvh + g) * max_seq * hd;
        dst[kv_index(pos, d, hd, swz)] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
        dst[kv_index(pos, d + half, hd, swz)] = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    }
}

// Causal attention, one warp per (row, query head): positions [0, start + row]
// of the head's KV group from the cache.  Lanes take the positions of a
// 32-position chunk for the scores (each lane a whole K row); the chunk's
// weights then go lane by lane to every lane, which accumulates its HD / 32
// dims of V.  Online softmax across chunks (max-subtracted).
template <int HD>
__global__ void attn_rows_kernel(const float* QKV, int nqkv, const uint16_t* kc, const uint16_t* vc, int n, int start,
                                 int qh, int kvh, int max_seq, int layer, int swz, float* out) {
    constexpr int DPL = HD / 32;   // dims of V per lane
    __shared__ float qs[4][HD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = blockIdx.x * 4 + warp;
    const int row = gid / qh, h = gid % qh;
    if (row >= n) return;
    const int g = h / (qh / kvh), ctx = start + row + 1;
    const float scale = rsqrtf((float)HD);
    for (int d = lane; d < HD; d += 32) qs[warp][d] = QKV[(size_t)row * nqkv + (size_t)h * HD + d] * scale;
    __syncwarp();
    const uint16_t* K = kc + ((size_t)layer * kvh + g) * max_seq * HD;
    const uint16_t* Vv = vc + ((size_t)layer * kvh + g) * max_seq * HD;
    float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = 0.f;
    for (int j0 = 0; j0 < ctx; j0 += 32) {
        const int j = j0 + lane;
        float s = -INFINITY;
        if (j < ctx) {
            s = 0.f;
            const uint4* kr = reinterpret_cast<const uint4*>(K + (size_t)j * HD);
#pragma unroll 4
            for (int c = 0; c < HD / 8; ++c) {
                const uint4 w = kr[swz ? (c ^ (j & 7)) : c];
                const uint32_t e4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    s = fmaf(qs[warp][8 * c + 2 * q], __uint_as_float(e4[q] << 16), s);
                    s = fmaf(qs[warp][8 * c + 2 * q + 1], __uint_as_float(e4[q] & 0xFFFF0000u), s);
                }
            }
        }
        float cm = s;
#pragma unroll
        for (int of = 16; of >= 1; of >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, of));
        const float mn = fmaxf(m, cm);
        const float corr = (m == -INFINITY) ? 0.f : __expf(m - mn);
        const float pj = (j < ctx) ? __expf(s - mn) : 0.f;
        float ps = pj;
#pragma unroll
        for (int of = 16; of >= 1; of >>= 1) ps += __shfl_xor_sync(0xFFFFFFFFu, ps, of);
        l = l * corr + ps;
        m = mn;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[e] *= corr;
        const int nj = min(32, ctx - j0);
#pragma unroll 8
        for (int jj = 0; jj < nj; ++jj) {
            const float w = __shfl_sync(0xFFFFFFFFu, pj, jj);
            const int p = j0 + jj;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[e] = fmaf(w, bf(Vv[kv_index(p, lane * DPL + e, HD, swz)]), o[e]);
        }
    }
    const float inv = 1.f / l;
    float* dst = out + (size_t)row * qh * HD + (size_t)h * HD + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; ++e) dst[e] = o[e] * inv;
}

// U[row][j] = silu(GU[row][j]) * GU[row][F + j]
// u = SiLU(gate) * up per row, to U (fp32) or to the parts P (part stride ps);
// a thread takes two neighbouring columns (F is even).
__global__ void silu_mul_kernel(const float* GU, int n, int F, float* U, uint16_t* P, size_t ps) {
    const size_t i = 2 * ((size_t)blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= (size_t)n * F) return;
    const size_t row = i / F, j = i % F;
    const float* gu = GU + row * 2 * F;
    const float g0 = gu[j], g1 = gu[j + 1], u0 = gu[F + j], u1 = gu[F + j + 1];
    const float a = g0 / (1.f + __expf(-g0)) * u0, b = g1 / (1.f + __expf(-g1)) * u1;
    if (P) {
        store_parts2(P, ps, i, a, b);
    } else {
        U[i] = a;
        U[i + 1] = b;
    }
}

__device__ __forceinline__ unsigned long long pack_key(float v, int idx) {
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)idx);
}

// Greedy token of the logits: lowest index on ties, non-finite logits skipped
// and flagged (status bit 2); part[] holds one partial key per block.
__global__ void argmax_blocks_kernel(const float* lg, int V, unsigned long long* part, uint32_t* status) {
    __shared__ unsigned long long red[32];
    unsigned long long best = 0ull;
    bool bad = false;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < V; i += gridDim.x * blockDim.x) {
        const float v = lg[i];
        if (isfinite(v)) {
            const unsigned long long k = pack_key(v, i);
            best = k > best ? k : best;
        } else {
            bad = true;
        }
    }
    if (bad) atomicOr(status, 0x2u);
    for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long k = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = k > best ? k : best;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) best = red[w] > best ? red[w] : best;
        part[blockIdx.x] = best;
    }
}

__global__ void argmax_final_kernel(const unsigned long long* part, int n, int32_t* out, uint32_t* status) {
    if (threadIdx.x != 0) return;
    unsigned long long best = 0ull;
    for (int i = 0; i < n; ++i) best = part[i] > best ? part[i] : best;
    if (best == 0ull) {
        atomicOr(status, 0x2u);
        *out = 0;
    } else {
        *out = (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
    }
}

// Causal attention on the tensor cores (flash style, mma.sync m16n8k16): a
// CTA takes 16 query rows (positions start + r0 ..) and the G query heads of
// one KV group.  Its keys are split NS ways: key set s (warps s*G .. s*G+G-1,
// warp s*G + i on head g * G + i) takes the 16-position K/V tiles s, s + NS,
// ..., so each tile is loaded once (un-permuting the cache's chunk order) and
// read by the G warps of its set, the set's next tile in flight while one is
// used (two buffers, cp.async, the set's own named barrier).  Per tile: S =
// q . K^T with q split into its bf16 rounding and the rounding of the
// remainder (q . k to about 2^-17 relative), the causal mask, an online
// softmax in base 2 (q pre-scaled by log2(e) / sqrt(hd)), P split the same
// way, O += P . V (V read transposed by ldmatrix).  The score accumulator of
// two 8-position tiles is, lane for lane, the A fragment of P . V, so P never
// goes through shared memory.  At the end the key sets' (m, l, O) meet in
// shared memory and set 0 writes the rows.  (The last row block of a prompt
// walks all of its keys; with NS = 2 that walk is half as long.)
template <int HD, int NS>
__global__ void __launch_bounds__(256) attn_tc_rows_kernel(const float* QKV, int nqkv, const uint16_t* kc,
                                                            const uint16_t* vc, int n, int start, int qh, int kvh,
                                                            int max_seq, int layer, int swz, float* out, uint16_t* P,
                                                            size_t ps) {
    static_assert(NS == 1 || NS == 2, "one or two key sets (named barriers 1 and 2)");
    constexpr int KL = HD + 8;                 // padded smem rows: 8 ldmatrix row addresses hit 8 bank groups
    extern __shared__ __align__(16) uint16_t at_smem[];
    const int G = qh / kvh;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
    const int ks_ = warp / G, hw = warp % G, nt_ = 32 * G;   // key set, head in the group, threads per set
    uint16_t* ks0 = at_smem + ks_ * (4 * 16 * KL);   // this set's K [2 buffers][16][KL], then V
    uint16_t* vs0 = ks0 + 2 * 16 * KL;
    uint16_t* qs = at_smem + NS * (4 * 16 * KL) + hw * (2 * 16 * KL);   // the head's q parts [2][16][KL]
    const int r0 = blockIdx.x * 16, grp = blockIdx.y, h = grp * G + hw;
    const float qscale = 1.4426950408889634f * rsqrtf((float)HD);
    // q rows r0 .. r0 + 15 of head h -> two bf16 parts in smem (rows past n are zero), by key set 0
    if (ks_ == 0) {
        for (int i = lane; i < 16 * HD / 2; i += 32) {
            const int r = i / (HD / 2), d = (i % (HD / 2)) * 2;
            float x = 0.f, y = 0.f;
            if (r0 + r < n) {
                const float* q = QKV + (size_t)(r0 + r) * nqkv + (size_t)h * HD + d;
                x = q[0] * qscale;
                y = q[1] * qscale;
            }
            const uint32_t hi = pack_bf2(x, y);
            const uint32_t lo = pack_bf2(x - __uint_as_float(hi << 16), y - __uint_as_float(hi & 0xFFFF0000u));
            *reinterpret_cast<uint32_t*>(qs + r * KL + d) = hi;
            *reinterpret_cast<uint32_t*>(qs + 16 * KL + r * KL + d) = lo;
        }
    }
    const uint16_t* K = kc + ((size_t)layer * kvh + grp) * max_seq * HD;
    const uint16_t* Vv = vc + ((size_t)layer * kvh + grp) * max_seq * HD;
    const int kend = min(start + r0 + 16, start + n);   // keys [0, kend): the last row attends start + r0 + 15
    float o[HD / 8][4];
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows g8 and g8 + 8
    const int qp0 = start + r0 + g8, qp1 = qp0 + 8;             // their positions
    const int st_ = threadIdx.x - ks_ * nt_;                    // thread index in the key set
    // K and V rows j0 .. j0 + 15 -> buffer b in plain chunk order (cp.async; rows past kend zero-filled)
    auto load_tile = [&](int j0, int b) {
        for (int i = st_; i < 2 * 16 * (HD / 8); i += nt_) {
            const int which = i / (16 * (HD / 8)), rem = i % (16 * (HD / 8));
            const int r = rem / (HD / 8), c = rem % (HD / 8), p = j0 + r;
            const bool in = p < kend;
            const int pc = (swz && in) ? (c ^ (p & 7)) : c;
            const uint16_t* src = (which ? Vv : K) + (size_t)(in ? p : 0) * HD + 8 * pc;
            cp_async16(smem_u32((which ? vs0 : ks0) + (b * 16 + r) * KL + 8 * c), src, in ? 16u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // the key set's barrier (named barrier 1 + set; the whole CTA uses 0)
    auto set_sync = [&]() {   // constant barrier ids (a register id would reserve all 16)
        if (ks_ == 0) asm volatile("bar.sync 1, %0;" ::"r"(nt_) : "memory");
        else asm volatile("bar.sync 2, %0;" ::"r"(nt_) : "memory");
    };
    if (16 * ks_ < kend) load_tile(16 * ks_, 0);
    __syncthreads();   // q is stored
    for (int j0 = 16 * ks_, b = 0; j0 < kend; j0 += 16 * NS, b ^= 1) {
        const uint16_t* ks = ks0 + b * 16 * KL;
        const uint16_t* vs = vs0 + b * 16 * KL;
        if (j0 + 16 * NS < kend) {
            load_tile(j0 + 16 * NS, b ^ 1);   // its buffer was released by the barrier ending the last round
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        set_sync();   // this tile landed for every thread of the set
        // S = q . K^T: 16 rows x 16 positions (two n-tiles of 8)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < HD; kk += 16) {
            uint32_t kb[4];   // b fragments of positions 0-7 (kb[0], kb[1]) and 8-15 (kb[2], kb[3])
            {
                const int mtx = lane >> 3, key = (mtx >> 1) * 8 + (lane & 7), dim = kk + (mtx & 1) * 8;
                ldsm_x4(kb, smem_u32(ks + key * KL + dim));
            }
#pragma unroll
            for (int part = 1; part >= 0; --part) {
                uint32_t qa[4];
                const int row = lane & 15, dim = kk + (lane >> 4) * 8;
                ldsm_x4(qa, smem_u32(qs + part * 16 * KL + row * KL + dim));
                mma_bf16(sc[0], qa, kb[0], kb[1]);
                mma_bf16(sc[1], qa, kb[2], kb[3]);
            }
        }
        // causal mask; lane holds rows g8 (e 0, 1) and g8 + 8 (e 2, 3), positions j0 + 8 nt + 2 t4 (+1)
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kp = j0 + 8 * nt + 2 * t4 + (e & 1);
                const int qp = (e < 2) ? qp0 : qp1;
                if (kp > qp || kp >= kend) sc[nt][e] = -INFINITY;
                if (e < 2) mx0 = fmaxf(mx0, sc[nt][e]); else mx1 = fmaxf(mx1, sc[nt][e]);
            }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        // a row with no visible position yet (a padding row) keeps m = -inf and weights 0
        const float c0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0), c1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
        float ps0 = 0.f, ps1 = 0.f;
        uint32_t pa[2][4];   // P as the A fragment of P . V: [part][reg]
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float mm = (e < 2) ? mn0 : mn1;
                pv[e] = (sc[nt][e] == -INFINITY) ? 0.f : exp2f(sc[nt][e] - mm);
            }
            ps0 += pv[0] + pv[1];
            ps1 += pv[2] + pv[3];
            // a0a1 = rows g8, positions 2t4 .. (tile 0) / a4a5 (tile 1); a2a3, a6a7 the rows g8 + 8
            const uint32_t h01 = pack_bf2(pv[0], pv[1]), h23 = pack_bf2(pv[2], pv[3]);
            pa[0][2 * nt] = h01;
            pa[0][2 * nt + 1] = h23;
            pa[1][2 * nt] = pack_bf2(pv[0] - __uint_as_float(h01 << 16), pv[1] - __uint_as_float(h01 & 0xFFFF0000u));
            pa[1][2 * nt + 1] = pack_bf2(pv[2] - __uint_as_float(h23 << 16), pv[3] - __uint_as_float(h23 & 0xFFFF0000u));
        }
        ps0 += __shfl_xor_sync(0xFFFFFFFFu, ps0, 1);
        ps0 += __shfl_xor_sync(0xFFFFFFFFu, ps0, 2);
        ps1 += __shfl_xor_sync(0xFFFFFFFFu, ps1, 1);
        ps1 += __shfl_xor_sync(0xFFFFFFFFu, ps1, 2);
        l0 = l0 * c0 + ps0;
        l1 = l1 * c1 + ps1;
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int j = 0; j < HD / 8; ++j) {
            o[j][0] *= c0; o[j][1] *= c0;
            o[j][2] *= c1; o[j][3] *= c1;
        }
        // O += P . V: dims in n-tiles of 8, two per transposed 8x8 quad load
#pragma unroll
        for (int nd = 0; nd < HD; nd += 16) {
            uint32_t vb[4];
            {
                const int mtx = lane >> 3, key = (mtx & 1) * 8 + (lane & 7), dim = nd + (mtx >> 1) * 8;
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                             : "=r"(vb[0]), "=r"(vb[1]), "=r"(vb[2]), "=r"(vb[3])
                             : "r"(smem_u32(vs + key * KL + dim)));
            }
#pragma unroll
            for (int part = 1; part >= 0; --part) {
                mma_bf16(o[nd / 8], pa[part], vb[0], vb[1]);
                mma_bf16(o[nd / 8 + 1], pa[part], vb[2], vb[3]);
            }
        }
        set_sync();   // every warp of the set is done with this buffer before the copy two tiles on refills it
    }
    if constexpr (NS > 1) {
        // key sets 1 .. NS-1 leave (m, l, O) in shared memory (the tile buffers and q are free now), lane by
        // lane; set 0 merges them with exp2 weights to the common maximum
        constexpr int NV = HD / 2 + 4;             // floats per lane
        float* mb = reinterpret_cast<float*>(at_smem);
        __syncthreads();
        if (ks_ > 0) {
            float* d = mb + ((size_t)((ks_ - 1) * G + hw) * NV) * 32 + lane;
#pragma unroll
            for (int j = 0; j < HD / 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) d[(4 * j + e) * 32] = o[j][e];
            d[(HD / 2) * 32] = m0; d[(HD / 2 + 1) * 32] = m1; d[(HD / 2 + 2) * 32] = l0; d[(HD / 2 + 3) * 32] = l1;
        }
        __syncthreads();
        if (ks_ > 0) return;
#pragma unroll 1
        for (int q = 1; q < NS; ++q) {
            const float* d = mb + ((size_t)((q - 1) * G + hw) * NV) * 32 + lane;
            const float mb0 = d[(HD / 2) * 32], mb1 = d[(HD / 2 + 1) * 32];
            const float M0 = fmaxf(m0, mb0), M1 = fmaxf(m1, mb1);
            const float a0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M0), b0 = mb0 == -INFINITY ? 0.f : exp2f(mb0 - M0);
            const float a1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M1), b1 = mb1 == -INFINITY ? 0.f : exp2f(mb1 - M1);
            l0 = a0 * l0 + b0 * d[(HD / 2 + 2) * 32];
            l1 = a1 * l1 + b1 * d[(HD / 2 + 3) * 32];
#pragma unroll
            for (int j = 0; j < HD / 8; ++j) {
                o[j][0] = a0 * o[j][0] + b0 * d[(4 * j + 0) * 32];
                o[j][1] = a0 * o[j][1] + b0 * d[(4 * j + 1) * 32];
                o[j][2] = a1 * o[j][2] + b1 * d[(4 * j + 2) * 32];
                o[j][3] = a1 * o[j][3] + b1 * d[(4 * j + 3) * 32];
            }
            m0 = M0;
            m1 = M1;
        }
    }
    // rows r0 + g8 and r0 + g8 + 8, dims 8 j + 2 t4 (+1): fp32 to out, or the parts to P
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) {
        const int d = 8 * j + 2 * t4;
        const size_t e0 = (size_t)(r0 + g8) * qh * HD + (size_t)h * HD + d, e1 = e0 + (size_t)8 * qh * HD;
        if (r0 + g8 < n) {
            if (P) store_parts2(P, ps, e0, o[j][0] * i0, o[j][1] * i0);
            else *reinterpret_cast<float2*>(out + e0) = make_float2(o[j][0] * i0, o[j][1] * i0);
        }
        if (r0 + g8 + 8 < n) {
            if (P) store_parts2(P, ps, e1, o[j][2] * i1, o[j][3] * i1);
            else *reinterpret_cast<float2*>(out + e1) = make_float2(o[j][2] * i1, o[j][3] * i1);
        }
    }
}

// Key sets of the prefill attention: two where the CTA stays within 256 threads.
inline int attn_tc_sets(int G) { return G <= 4 ? 2 : 1; }
template <int HD>
size_t attn_tc_smem(int G) {
    const size_t tiles = (size_t)(attn_tc_sets(G) * 4 * 16 + G * 2 * 16) * (HD + 8) * 2;
    const size_t merge = (size_t)(attn_tc_sets(G) - 1) * G * (HD / 2 + 4) * 32 * 4;   // fits inside `tiles`
    return tiles > merge ? tiles : merge;
}

template <bool RES>
void gemm(const float* A, const uint16_t* W, const float* R, float* C, int M, int N, int K, cudaStream_t st) {
    const dim3 grid((N + GBN - 1) / GBN, (M + GBM - 1) / GBM);
    gemm_split_kernel<RES><<<grid, 128, sizeof(GemmSmem), st>>>(A, W, R, C, M, N, K);
}

// cuTensorMapEncodeTiled, fetched from the driver through the runtime (no
// link against the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Tensor map of a row-major bf16 matrix [rows][inner] read in boxes of 64 x
// box_rows with the 128-byte swizzle (out-of-bounds elements read as zero).
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)TBK, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return g_encode && g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                                es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the three parts [3][rows][K] of an M-row activation, read in
// boxes of 64 x 128 x 1: rows M .. past the last tile read as zero.
bool make_parts_map(CUtensorMap* m, const uint16_t* parts, uint64_t K, uint64_t M, uint64_t rows) {
    const cuuint64_t dims[3] = {K, M, 3};
    const cuuint64_t strides[2] = {K * 2, rows * K * 2};
    const cuuint32_t box[3] = {(cuuint32_t)TBK, (cuuint32_t)TBM, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return g_encode && g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(parts), dims, strides,
                                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// C = A . W^T (+ R) on the tcgen05 path, A given as its parts [3][rows][K] (1 launch).
// Outputs of 8192 columns or more take 256-wide tiles.
cudaError_t gemm_tc(const uint16_t* parts, int rows, const uint16_t* W, const float* R, float* C, int M, int N, int K,
                    uint32_t* status, cudaStream_t st) {
    const int Mp = (M + TBM - 1) / TBM * TBM;
    const int bn = N >= 8192 ? 256 : 128;
    CUtensorMap ma, mw;
    if (!make_parts_map(&ma, parts, (uint64_t)K, (uint64_t)M, (uint64_t)rows) ||
        !make_map(&mw, W, (uint64_t)K, (uint64_t)N, bn))
        return cudaErrorInvalidValue;
    const int tiles = ((N + bn - 1) / bn) * (Mp / TBM), nkb = (K + TBK - 1) / TBK;
    // a residual product adds into C with atomics, so its K range may be split until the grid covers the SMs
    int ksplit = 1;
    if (R == C)
        while (ksplit < 4 && tiles * ksplit * 2 <= 160 && nkb >= 8 * ksplit * 2) ksplit *= 2;
    const dim3 grid((N + bn - 1) / bn, Mp / TBM, ksplit);
    if (bn == 256)
        gemm_tc_kernel<256><<<grid, 192, TcCfg<256>::SMEM, st>>>(ma, mw, R, C, M, N, K, ksplit, status);
    else
        gemm_tc_kernel<128><<<grid, 192, TcCfg<128>::SMEM, st>>>(ma, mw, R, C, M, N, K, ksplit, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t mk_prefill_prepare() {
    cudaError_t e = cudaFuncSetAttribute(gemm_split_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(GemmSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_split_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(GemmSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)TcCfg<128>::SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)TcCfg<256>::SMEM);
    // up to 8 query heads per KV group (one key set), or 4 with two sets
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_tc_rows_kernel<64, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attn_tc_smem<64>(8));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_tc_rows_kernel<128, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attn_tc_smem<128>(8));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_tc_rows_kernel<64, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attn_tc_smem<64>(4));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_tc_rows_kernel<128, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attn_tc_smem<128>(4));
    if (e == cudaSuccess && !g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn) g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        else if (e == cudaSuccess) e = cudaErrorSymbolNotFound;
    }
    return e;
}

int mk_prefill_launch(const MkPrefillArgs& a, cudaStream_t st, cudaError_t* err) {
    const int H = a.H, hd = a.hd, qh = a.qh, kvh = a.kvh, F = a.F, n = a.n;
    const int nqkv = (qh + 2 * kvh) * hd, qd = qh * hd;
    int launches = 0;
    *err = cudaSuccess;
    // tcgen05 path (a.parts): each GEMM's activation goes from its producer to the parts buffer as
    // [3][parts_rows][K]; otherwise fp32 activations and the mma.sync GEMMs
    const bool tc = a.parts != nullptr;
    uint16_t* P = a.parts;
    const size_t prow = (size_t)a.parts_rows;
    auto note = [&](cudaError_t e) { if (e != cudaSuccess && *err == cudaSuccess) *err = e; };
    auto gemm_any = [&](const float* A, const uint16_t* W, const float* R, float* C, int M, int N, int K) {
        if (tc) note(gemm_tc(P, (int)prow, W, R, C, M, N, K, a.status, st));
        else if (R) gemm<true>(A, W, R, C, M, N, K, st);
        else gemm<false>(A, W, R, C, M, N, K, st);
        ++launches;
    };
    embed_rows_kernel<<<n, 256, 0, st>>>(a.embed, a.tokens, n, a.V, H, a.x, a.status); ++launches;
    for (int l = 0; l < a.L; ++l) {
        rmsnorm_rows_kernel<<<n, 256, 0, st>>>(a.x, a.attn_norm + (size_t)l * H, H, a.eps, tc ? nullptr : a.xn, P,
                                               prow * H); ++launches;
        gemm_any(a.xn, a.wqkv[l], nullptr, a.qkv, n, nqkv, H);
        rope_kv_rows_kernel<<<dim3(((qh + 2 * kvh) * hd / 2 + 127) / 128, n), 128, 0, st>>>(
            a.qkv, nqkv, a.rope_cos, a.rope_sin, a.start, qh, kvh, hd, a.max_seq, l, a.kc, a.vc, a.swz); ++launches;
        const int warps = n * qh, G = qh / kvh;
        const dim3 tgrid((n + 15) / 16, kvh);
        const int nsets = attn_tc_sets(G);
        if (a.attn_tc && hd == 64 && nsets == 2)
            attn_tc_rows_kernel<64, 2><<<tgrid, 32 * G * 2, attn_tc_smem<64>(G), st>>>(
                a.qkv, nqkv, a.kc, a.vc, n, a.start, qh, kvh, a.max_seq, l, a.swz, a.att, P, prow * qd);
        else if (a.attn_tc && hd == 64)
            attn_tc_rows_kernel<64, 1><<<tgrid, 32 * G, attn_tc_smem<64>(G), st>>>(
                a.qkv, nqkv, a.kc, a.vc, n, a.start, qh, kvh, a.max_seq, l, a.swz, a.att, P, prow * qd);
        else if (a.attn_tc && nsets == 2)
            attn_tc_rows_kernel<128, 2><<<tgrid, 32 * G * 2, attn_tc_smem<128>(G), st>>>(
                a.qkv, nqkv, a.kc, a.vc, n, a.start, qh, kvh, a.max_seq, l, a.swz, a.att, P, prow * qd);
        else if (a.attn_tc)
            attn_tc_rows_kernel<128, 1><<<tgrid, 32 * G, attn_tc_smem<128>(G), st>>>(
                a.qkv, nqkv, a.kc, a.vc, n, a.start, qh, kvh, a.max_seq, l, a.swz, a.att, P, prow * qd);
        else if (hd == 64)
            attn_rows_kernel<64><<<(warps + 3) / 4, 128, 0, st>>>(a.qkv, nqkv, a.kc, a.vc, n, a.start, qh, kvh,
                                                                   a.max_seq, l, a.swz, a.att);
        else
            attn_rows_kernel<128><<<(warps + 3) / 4, 128, 0, st>>>(a.qkv, nqkv, a.kc, a.vc, n, a.start, qh, kvh,
                                                                    a.max_seq, l, a.swz, a.att);
        ++launches;
        gemm_any(a.att, a.wo[l], a.x, a.x, n, H, qd);   // residual in place
        rmsnorm_rows_kernel<<<n, 256, 0, st>>>(a.x, a.ffn_norm + (size_t)l * H, H, a.eps, tc ? nullptr : a.xn, P,
                                               prow * H); ++launches;
        gemm_any(a.xn, a.wgu[l], nullptr, a.gu, n, 2 * F, H);
        silu_mul_kernel<<<(int)(((size_t)n * F / 2 + 255) / 256), 256, 0, st>>>(a.gu, n, F, a.u, P, prow * F);
        ++launches;
        gemm_any(a.u, a.wd[l], a.x, a.x, n, H, F);
    }
    // the last row: final norm (kept as the step's hidden state), LM head, argmax
    const float* xlast = a.x + (size_t)(n - 1) * H;
    rmsnorm_rows_kernel<<<1, 256, 0, st>>>(xlast, a.final_norm, H, a.eps, a.hidden, P, prow * H); ++launches;
    gemm_any(a.hidden, a.lm, nullptr, a.logits, 1, a.V, H);
    argmax_blocks_kernel<<<a.amax_blocks, 256, 0, st>>>(a.logits, a.V, a.amax_part, a.status); ++launches;
    argmax_final_kernel<<<1, 32, 0, st>>>(a.amax_part, a.amax_blocks, a.next_token, a.status); ++launches;
    note(cudaGetLastError());
    return launches;
}
