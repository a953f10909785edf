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

// y = x / sqrt(mean(x^2) + eps) * g for row blockIdx.x
__global__ void rmsnorm_rows_kernel(const float* X, const float* g, int H, float eps, float* Y) {
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
    float* y = Y + (size_t)blockIdx.x * H;
    for (int d = threadIdx.x; d < H; d += blockDim.x) y[d] = x[d] * inv * g[d];
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
__global__ void silu_mul_kernel(const float* GU, int n, int F, float* U) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)n * F) return;
    const size_t row = i / F, j = i % F;
    const float gt = GU[row * 2 * F + j], up = GU[row * 2 * F + F + j];
    U[i] = gt / (1.f + __expf(-gt)) * up;
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

template <bool RES>
void gemm(const float* A, const uint16_t* W, const float* R, float* C, int M, int N, int K, cudaStream_t st) {
    const dim3 grid((N + GBN - 1) / GBN, (M + GBM - 1) / GBM);
    gemm_split_kernel<RES><<<grid, 128, sizeof(GemmSmem), st>>>(A, W, R, C, M, N, K);
}

}  // namespace

cudaError_t mk_prefill_prepare() {
    cudaError_t e = cudaFuncSetAttribute(gemm_split_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(GemmSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_split_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(GemmSmem));
    return e;
}

int mk_prefill_launch(const MkPrefillArgs& a, cudaStream_t st, cudaError_t* err) {
    const int H = a.H, hd = a.hd, qh = a.qh, kvh = a.kvh, F = a.F, n = a.n;
    const int nqkv = (qh + 2 * kvh) * hd, qd = qh * hd;
    int launches = 0;
    *err = cudaSuccess;
    embed_rows_kernel<<<n, 256, 0, st>>>(a.embed, a.tokens, n, a.V, H, a.x, a.status); ++launches;
    for (int l = 0; l < a.L; ++l) {
        rmsnorm_rows_kernel<<<n, 256, 0, st>>>(a.x, a.attn_norm + (size_t)l * H, H, a.eps, a.xn); ++launches;
        gemm<false>(a.xn, a.wqkv[l], nullptr, a.qkv, n, nqkv, H, st); ++launches;
        rope_kv_rows_kernel<<<dim3(((qh + 2 * kvh) * hd / 2 + 127) / 128, n), 128, 0, st>>>(
            a.qkv, nqkv, a.rope_cos, a.rope_sin, a.start, qh, kvh, hd, a.max_seq, l, a.kc, a.vc, a.swz); ++launches;
        const int warps = n * qh;
        if (hd == 64)
            attn_rows_kernel<64><<<(warps + 3) / 4, 128, 0, st>>>(a.qkv, nqkv, a.kc, a.vc, n, a.start, qh, kvh,
                                                                   a.max_seq, l, a.swz, a.att);
        else
            attn_rows_kernel<128><<<(warps + 3) / 4, 128, 0, st>>>(a.qkv, nqkv, a.kc, a.vc, n, a.start, qh, kvh,
                                                                    a.max_seq, l, a.swz, a.att);
        ++launches;
        gemm<true>(a.att, a.wo[l], a.x, a.x, n, H, qd, st); ++launches;   // residual in place
        rmsnorm_rows_kernel<<<n, 256, 0, st>>>(a.x, a.ffn_norm + (size_t)l * H, H, a.eps, a.xn); ++launches;
        gemm<false>(a.xn, a.wgu[l], nullptr, a.gu, n, 2 * F, H, st); ++launches;
        silu_mul_kernel<<<(int)(((size_t)n * F + 255) / 256), 256, 0, st>>>(a.gu, n, F, a.u); ++launches;
        gemm<true>(a.u, a.wd[l], a.x, a.x, n, H, F, st); ++launches;
    }
    // the last row: final norm (kept as the step's hidden state), LM head, argmax
    const float* xlast = a.x + (size_t)(n - 1) * H;
    rmsnorm_rows_kernel<<<1, 256, 0, st>>>(xlast, a.final_norm, H, a.eps, a.hidden); ++launches;
    gemm<false>(a.hidden, a.lm, nullptr, a.logits, 1, a.V, H, st); ++launches;
    argmax_blocks_kernel<<<a.amax_blocks, 256, 0, st>>>(a.logits, a.V, a.amax_part, a.status); ++launches;
    argmax_final_kernel<<<1, 32, 0, st>>>(a.amax_part, a.amax_blocks, a.next_token, a.status); ++launches;
    *err = cudaGetLastError();
    return launches;
}
