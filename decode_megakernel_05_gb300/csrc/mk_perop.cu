// mk_perop.cu - the unfused baseline: the same decode step launched as one
// kernel per operator on plain row-major weights.  This is the per-operator
// path the fused kernel replaces (cloud.baidu.com/article/9434380, section 4.1:
// every operator its own launch with its own start, tail and implicit sync),
// kept for the fusion-off ablation and for debugging (same page, sections 5
// step 5 and 7).  Per layer: RMSNorm, QKV GEMV (one concatenated matrix),
// RoPE + K/V append, attention partials, attention combine, O GEMV + residual,
// RMSNorm, gate/up GEMV + SwiGLU, down GEMV + residual; then embedding (first),
// final RMSNorm, LM-head GEMV and a two-stage argmax.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mk_perop.h"

namespace {

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
// Element of dim d of position p in a KV head's cache rows: with swz the
// row's 16-byte chunk index is XORed with p mod 8 (the layout the
// long-context fused kernel reads).
__device__ __forceinline__ int64_t kvi(int64_t p, int d, int hd, int swz) {
    const int c = d >> 3;
    return p * hd + (((swz ? (c ^ (int)(p & 7)) : c) << 3) | (d & 7));
}

__global__ void embed_kernel(const uint16_t* E, const int32_t* tok_ptr, int tok_arg, int V, int H, float* x,
                             uint32_t* status) {
    int tok = tok_ptr ? *tok_ptr : tok_arg;
    if (tok < 0 || tok >= V) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, 0x4u);
        tok = 0;
    }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < H; i += gridDim.x * blockDim.x)
        x[i] = bf(E[(int64_t)tok * H + i]);
}

__global__ void rmsnorm_kernel(const float* x, const float* g, int H, float eps, float* y) {
    __shared__ float red[32];
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    const float inv = rsqrtf(tot / (float)H + eps);
    for (int i = threadIdx.x; i < H; i += blockDim.x) y[i] = x[i] * inv * g[i];
}

// y[r] = W[r] . v (warp per row, 16-byte loads); mode 0: store, 1: y = res + W v
// (in place allowed), 2: SwiGLU: rows r and r + nout of W give gate and up, y[r] =
// silu(gate) * up.
template <int MODE>
__global__ void gemv_kernel(const uint16_t* W, const float* v, int K, int nout, const float* res, float* y) {
    extern __shared__ float vs[];
    for (int i = threadIdx.x; i < K; i += blockDim.x) vs[i] = v[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * (blockDim.x >> 5) + warp;
    if (r >= nout) return;
    float a0 = 0.f, a1 = 0.f;
    const uint4* w0 = reinterpret_cast<const uint4*>(W + (int64_t)r * K);
    const uint4* w1 = reinterpret_cast<const uint4*>(W + (int64_t)(r + nout) * K);
    for (int c = lane; c < K / 8; c += 32) {
        const float* xv = vs + c * 8;
        uint4 q = w0[c];
        uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            a0 = fmaf(__uint_as_float(u[e] << 16), xv[2 * e], a0);
            a0 = fmaf(__uint_as_float(u[e] & 0xFFFF0000u), xv[2 * e + 1], a0);
        }
        if (MODE == 2) {
            q = w1[c];
            uint32_t u2[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                a1 = fmaf(__uint_as_float(u2[e] << 16), xv[2 * e], a1);
                a1 = fmaf(__uint_as_float(u2[e] & 0xFFFF0000u), xv[2 * e + 1], a1);
            }
        }
    }
    for (int o = 16; o >= 1; o >>= 1) {
        a0 += __shfl_xor_sync(0xFFFFFFFFu, a0, o);
        if (MODE == 2) a1 += __shfl_xor_sync(0xFFFFFFFFu, a1, o);
    }
    if (lane == 0) {
        if (MODE == 0) y[r] = a0;
        else if (MODE == 1) y[r] = res[r] + a0;
        else y[r] = a0 / (1.f + __expf(-a0)) * a1;
    }
}

// RoPE on q and k heads of the fused qkv vector, then K/V append (bf16).
__global__ void rope_append_kernel(float* qkv, const float* cs, const float* sn, int pos, int qh, int kvh, int hd,
                                   int max_seq, int layer, uint16_t* kc, uint16_t* vc, int swz) {
    const int half = hd / 2;
    const int nh = qh + 2 * kvh;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= nh * half) return;
    const int h = idx / half, d = idx % half;
    float* v = qkv + (int64_t)h * hd;
    float a = v[d], b = v[d + half];
    if (h < qh + kvh) {
        const float c = cs[(int64_t)pos * half + d], s = sn[(int64_t)pos * half + d];
        const float a2 = a * c - b * s, b2 = b * c + a * s;
        a = a2; b = b2;
    }
    if (h < qh) {
        v[d] = a; v[d + half] = b;
    } else {
        const int g = (h < qh + kvh) ? h - qh : h - qh - kvh;
        uint16_t* dst = ((h < qh + kvh) ? kc : vc) + ((int64_t)layer * kvh + g) * max_seq * hd;
        dst[kvi(pos, d, hd, swz)] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
        dst[kvi(pos, d + half, hd, swz)] = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    }
}

// Attention partials: block (q head, split); positions split into `nsplit`
// chunks of ctx; writes (m, l) and the unnormalised accumulator.
__global__ void attn_partial_kernel(const float* q, const uint16_t* kc, const uint16_t* vc, int ctx, int qh, int kvh,
                                    int hd, int max_seq, int layer, int nsplit, float* pml, float* pacc, int swz) {
    extern __shared__ float sm[];
    float* qs = sm;            // [hd]
    float* sc = sm + hd;       // [chunk]
    const int h = blockIdx.x, sp = blockIdx.y, g = h / (qh / kvh);
    const int a = (int)((int64_t)sp * ctx / nsplit), b = (int)((int64_t)(sp + 1) * ctx / nsplit);
    const float scale = rsqrtf((float)hd);
    for (int d = threadIdx.x; d < hd; d += blockDim.x) qs[d] = q[(int64_t)h * hd + d] * scale;
    __syncthreads();
    const uint16_t* K = kc + ((int64_t)layer * kvh + g) * max_seq * hd;
    const uint16_t* Vv = vc + ((int64_t)layer * kvh + g) * max_seq * hd;
    for (int p = a + threadIdx.x; p < b; p += blockDim.x) {
        // the row's 16-byte chunks in dim order (each one load), dims ascending
        const uint4* kr = reinterpret_cast<const uint4*>(K + (int64_t)p * hd);
        float s = 0.f;
        for (int c = 0; c < hd / 8; ++c) {
            const uint4 w = kr[swz ? (c ^ (p & 7)) : c];
            const uint32_t e[4] = {w.x, w.y, w.z, w.w};
            for (int j = 0; j < 4; ++j) {
                s = fmaf(qs[8 * c + 2 * j], bf((uint16_t)(e[j] & 0xFFFFu)), s);
                s = fmaf(qs[8 * c + 2 * j + 1], bf((uint16_t)(e[j] >> 16)), s);
            }
        }
        sc[p - a] = s;
    }
    __syncthreads();
    __shared__ float mred[32], lred[32];
    float m = -INFINITY;
    for (int p = threadIdx.x; p < b - a; p += blockDim.x) m = fmaxf(m, sc[p]);
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) mred[threadIdx.x >> 5] = m;
    __syncthreads();
    m = -INFINITY;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, mred[w]);
    float l = 0.f;
    for (int p = threadIdx.x; p < b - a; p += blockDim.x) {
        const float e = __expf(sc[p] - m);
        sc[p] = e;
        l += e;
    }
    for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
    if ((threadIdx.x & 31) == 0) lred[threadIdx.x >> 5] = l;
    __syncthreads();
    l = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) l += lred[w];
    const int64_t pb = (int64_t)h * nsplit + sp;
    for (int d = threadIdx.x; d < hd; d += blockDim.x) {
        float acc = 0.f;
        for (int p = a; p < b; ++p) acc = fmaf(sc[p - a], bf(Vv[kvi(p, d, hd, swz)]), acc);
        pacc[pb * hd + d] = acc;
    }
    if (threadIdx.x == 0) { pml[pb * 2] = (b > a) ? m : -INFINITY; pml[pb * 2 + 1] = l; }
}

__global__ void attn_combine_kernel(const float* pml, const float* pacc, int nsplit, int hd, float* out) {
    const int h = blockIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pml[((int64_t)h * nsplit + s) * 2]);
    for (int d = threadIdx.x; d < hd; d += blockDim.x) {
        float num = 0.f, den = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const int64_t pb = (int64_t)h * nsplit + s;
            const float m = pml[pb * 2];
            const float w = (m == -INFINITY) ? 0.f : __expf(m - M);
            den = fmaf(w, pml[pb * 2 + 1], den);
            num = fmaf(w, pacc[pb * hd + d], num);
        }
        out[(int64_t)h * hd + d] = num / den;
    }
}

__device__ __forceinline__ unsigned long long pack_key(float v, int idx) {
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)idx);
}

__global__ void argmax_partial_kernel(const float* lg, int V, unsigned long long* part, uint32_t* status) {
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
    if (best == 0ull) { atomicOr(status, 0x2u); *out = 0; }
    else *out = (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
}

}  // namespace

// Launches every operator of one step; returns the number of kernel launches.
int mk_perop_step(const MkPerOp& P, int token, const int32_t* token_ptr, int pos, float* logits, cudaStream_t st,
                  cudaError_t* err) {
    int n = 0;
    const int H = P.H, hd = P.hd, qh = P.qh, kvh = P.kvh, F = P.F, V = P.V;
    const int nqkv = (qh + 2 * kvh) * hd;
    const int ctx = pos + 1;
    const int nsplit = (ctx + P.attn_chunk - 1) / P.attn_chunk;
    const int rows_per_block = 8;
    auto blocks = [&](int rows) { return (rows + rows_per_block - 1) / rows_per_block; };
    float* lg = logits ? logits : P.logits_tmp;
    *err = cudaSuccess;
    embed_kernel<<<(H + 255) / 256, 256, 0, st>>>(P.embed, token_ptr, token, V, H, P.x, P.status); ++n;
    for (int l = 0; l < P.L; ++l) {
        rmsnorm_kernel<<<1, 1024, 0, st>>>(P.x, P.attn_norm + (int64_t)l * H, H, P.eps, P.xn); ++n;
        gemv_kernel<0><<<blocks(nqkv), 256, H * 4, st>>>(P.wqkv[l], P.xn, H, nqkv, nullptr, P.qkv); ++n;
        rope_append_kernel<<<((qh + 2 * kvh) * hd / 2 + 255) / 256, 256, 0, st>>>(
            P.qkv, P.rope_cos, P.rope_sin, pos, qh, kvh, hd, P.max_seq, l, P.kc, P.vc, P.kv_swz); ++n;
        attn_partial_kernel<<<dim3(qh, nsplit), 128, (hd + P.attn_chunk) * 4, st>>>(
            P.qkv, P.kc, P.vc, ctx, qh, kvh, hd, P.max_seq, l, nsplit, P.pml, P.pacc, P.kv_swz); ++n;
        attn_combine_kernel<<<qh, 128, 0, st>>>(P.pml, P.pacc, nsplit, hd, P.attn); ++n;
        gemv_kernel<1><<<blocks(H), 256, qh * hd * 4, st>>>(P.wo[l], P.attn, qh * hd, H, P.x, P.x); ++n;
        rmsnorm_kernel<<<1, 1024, 0, st>>>(P.x, P.ffn_norm + (int64_t)l * H, H, P.eps, P.xn); ++n;
        gemv_kernel<2><<<blocks(F), 256, H * 4, st>>>(P.wgu[l], P.xn, H, F, nullptr, P.u); ++n;
        gemv_kernel<1><<<blocks(H), 256, F * 4, st>>>(P.wd[l], P.u, F, H, P.x, P.x); ++n;
    }
    rmsnorm_kernel<<<1, 1024, 0, st>>>(P.x, P.final_norm, H, P.eps, P.hidden); ++n;
    gemv_kernel<0><<<blocks(V), 256, H * 4, st>>>(P.lm, P.hidden, H, V, nullptr, lg); ++n;
    argmax_partial_kernel<<<P.amax_blocks, 256, 0, st>>>(lg, V, P.amax_part, P.status); ++n;
    argmax_final_kernel<<<1, 32, 0, st>>>(P.amax_part, P.amax_blocks, P.next_token, P.status); ++n;
    *err = cudaGetLastError();
    return n;
}

cudaError_t mk_perop_prepare(int max_smem_k_bytes) {
    // the down GEMV stages F floats of input in shared memory
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_k_bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_k_bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_k_bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_k_bytes);
    return e;
}
