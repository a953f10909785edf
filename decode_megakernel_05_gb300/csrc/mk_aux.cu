// mk_aux.cu - one-time device kernels used when a context is set up: the weight
// re-layout gathers, the RoPE cos/sin table and the widening of norm gains.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mk_aux.h"

// One block per stored row: copy ncols bf16 (a multiple of 8) from
// src[src_row][col0 ..] to arena + dst_off, 16 bytes per thread step.
__global__ void mk_relayout_rows_kernel(uint8_t* arena, const uint16_t* src, int64_t src_cols, const MkRowCopy* ops,
                                        int n) {
    const int i = blockIdx.x;
    if (i >= n) return;
    const MkRowCopy op = ops[i];
    const uint4* s = reinterpret_cast<const uint4*>(src + op.src_row * src_cols + op.col0);
    uint4* d = reinterpret_cast<uint4*>(arena + op.dst_off);
    for (int k = threadIdx.x; k < op.ncols / 8; k += blockDim.x) d[k] = s[k];
}

// Column gather of W_down [H][F]: arena + dst_off receives columns j0 .. j0+nj-1,
// each as H contiguous bf16.  Block (op, row chunk); thread = one row.
__global__ void mk_relayout_cols_kernel(uint8_t* arena, const uint16_t* src, int H, int F, const MkColCopy* ops,
                                        int n) {
    const int i = blockIdx.x;
    if (i >= n) return;
    const MkColCopy op = ops[i];
    const int r = blockIdx.y * blockDim.x + threadIdx.x;
    if (r >= H) return;
    uint16_t* d = reinterpret_cast<uint16_t*>(arena + op.dst_off);
    const uint16_t* s = src + (int64_t)r * F + op.j0;
    for (int jj = 0; jj < op.nj; ++jj) d[(int64_t)jj * H + r] = s[jj];
}

// cos/sin of pos * theta^(-2i/hd) for pos < max_seq, i < hd/2, evaluated in
// double and stored as float [max_seq][hd/2].
__global__ void mk_rope_table_kernel(float* cs, float* sn, int max_seq, int hd, double theta) {
    const int half = hd / 2;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)max_seq * half) return;
    const int pos = (int)(idx / half), i = (int)(idx % half);
    const double inv = pow(theta, -(2.0 * (double)i) / (double)hd);
    double s, c;
    sincos((double)pos * inv, &s, &c);
    cs[idx] = (float)c;
    sn[idx] = (float)s;
}

__global__ void mk_bf16_to_f32_kernel(const uint16_t* src, float* dst, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = __uint_as_float((uint32_t)src[i] << 16);
}

// One thread per 16-byte chunk of a row; chunk cc of position pos sits at
// chunk cc ^ (pos mod 8) of the cache row when swz.
__global__ void mk_kv_rows_kernel(uint4* plain, uint4* cache_layer, int kvh, int n_pos, int pos0, int max_seq, int nch,
                                  int swz, int to_cache) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)kvh * n_pos * nch) return;
    const int cc = (int)(i % nch);
    const int64_t r = i / nch;
    const int h = (int)(r / n_pos), pos = pos0 + (int)(r % n_pos);
    uint4* c = cache_layer + ((int64_t)h * max_seq + pos) * nch + (swz ? (cc ^ (pos & 7)) : cc);
    if (to_cache) *c = plain[i];
    else plain[i] = *c;
}

// One block per group (a row, or a column when col_scaled): the group's
// largest |w| by a block reduction, then every code.
// qmax: 127 (int8, codes stored as q + 128) or 7 (int4, codes stored as q + 8,
// one a byte until the re-layout packs them).
__global__ void mk_quantize_q8_kernel(const uint16_t* w, int64_t rows, int64_t cols, int col_scaled, int qmax,
                                      int8_t* q, float* scale) {
    __shared__ float red[32];
    const int64_t gi = blockIdx.x;
    const int64_t len = col_scaled ? rows : cols;
    auto at = [&](int64_t k) { return col_scaled ? k * cols + gi : gi * cols + k; };
    float amax = 0.f;
    for (int64_t k = threadIdx.x; k < len; k += blockDim.x)
        amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)w[at(k)] << 16)));
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
    const float qm = (float)qmax;
    const float sg = __fdiv_rn(amax, qm);
    if (threadIdx.x == 0) scale[gi] = sg;
    const int bias = qmax == 7 ? 8 : 128;
    for (int64_t k = threadIdx.x; k < len; k += blockDim.x) {
        float c = 0.f;
        if (sg > 0.f) c = rintf(__fdiv_rn(__uint_as_float((uint32_t)w[at(k)] << 16), sg));
        c = fminf(fmaxf(c, -qm), qm);
        reinterpret_cast<uint8_t*>(q)[at(k)] = (uint8_t)((int)c + bias);   // stored biased
    }
}

// INT4 rows: one block per stored row, ncols biased codes (one a byte, a
// multiple of 8) packed two a byte (group of 8 -> 4 bytes, byte k = weight k
// low, weight k + 4 high), and the row's scale.
__global__ void mk_relayout_rows_q4_kernel(uint8_t* arena, const int8_t* q, int64_t cols, const float* scale,
                                           const MkRowCopyQ* ops, int n) {
    const int i = blockIdx.x;
    if (i >= n) return;
    const MkRowCopyQ op = ops[i];
    const uint8_t* s = reinterpret_cast<const uint8_t*>(q) + op.src_row * cols + op.col0;
    uint8_t* d = arena + op.dst_off;
    for (int b = threadIdx.x; b < op.ncols / 2; b += blockDim.x) {
        const int c0 = 8 * (b >> 2) + (b & 3);
        d[b] = (uint8_t)((s[c0] & 0xF) | ((s[c0 + 4] & 0xF) << 4));
    }
    if (threadIdx.x == 0) *reinterpret_cast<float*>(arena + op.scale_off) = scale[op.src_row];
}

// INT4 W_down [H][F]: columns j0 .. j0+nj-1 as H/2 contiguous bytes each, rows
// packed as above (byte b: rows 8 (b / 4) + b % 4 and 4 more).
__global__ void mk_relayout_cols_q4_kernel(uint8_t* arena, const int8_t* q, int H, int F, const MkColCopy* ops, int n) {
    const int i = blockIdx.x;
    if (i >= n) return;
    const MkColCopy op = ops[i];
    const int b = blockIdx.y * blockDim.x + threadIdx.x;
    if (b >= H / 2) return;
    const int r0 = 8 * (b >> 2) + (b & 3);
    const uint8_t* lo = reinterpret_cast<const uint8_t*>(q) + (int64_t)r0 * F + op.j0;
    const uint8_t* hi = lo + 4LL * F;
    uint8_t* d = arena + op.dst_off + b;
    for (int jj = 0; jj < op.nj; ++jj) d[(int64_t)jj * (H / 2)] = (uint8_t)((lo[jj] & 0xF) | ((hi[jj] & 0xF) << 4));
}

// One block per stored row: ncols int8 (a multiple of 16) and the row's scale.
__global__ void mk_relayout_rows_q8_kernel(uint8_t* arena, const int8_t* q, int64_t cols, const float* scale,
                                           const MkRowCopyQ* ops, int n) {
    const int i = blockIdx.x;
    if (i >= n) return;
    const MkRowCopyQ op = ops[i];
    const uint4* s = reinterpret_cast<const uint4*>(q + op.src_row * cols + op.col0);
    uint4* d = reinterpret_cast<uint4*>(arena + op.dst_off);
    for (int k = threadIdx.x; k < op.ncols / 16; k += blockDim.x) d[k] = s[k];
    if (threadIdx.x == 0) *reinterpret_cast<float*>(arena + op.scale_off) = scale[op.src_row];
}

// Column gather of an int8 W_down [H][F]: columns j0 .. j0+nj-1 as H contiguous bytes each.
__global__ void mk_relayout_cols_q8_kernel(uint8_t* arena, const int8_t* q, int H, int F, const MkColCopy* ops, int n) {
    const int i = blockIdx.x;
    if (i >= n) return;
    const MkColCopy op = ops[i];
    const int r = blockIdx.y * blockDim.x + threadIdx.x;
    if (r >= H) return;
    int8_t* d = reinterpret_cast<int8_t*>(arena + op.dst_off);
    const int8_t* s = q + (int64_t)r * F + op.j0;
    for (int jj = 0; jj < op.nj; ++jj) d[(int64_t)jj * H + r] = s[jj];
}

__global__ void mk_scatter_scales_kernel(uint8_t* arena, const float* scale, const MkScaleCopy* ops, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) *reinterpret_cast<float*>(arena + ops[i].dst_off) = scale[ops[i].idx];
}

cudaError_t mk_launch_quantize(const uint16_t* w, int64_t rows, int64_t cols, int col_scaled, int bits, int8_t* q,
                               float* scale, cudaStream_t st) {
    const int64_t ng = col_scaled ? cols : rows;
    if (ng <= 0) return cudaSuccess;
    if (bits != 8 && bits != 4) return cudaErrorInvalidValue;
    mk_quantize_q8_kernel<<<(unsigned)ng, 256, 0, st>>>(w, rows, cols, col_scaled, bits == 8 ? 127 : 7, q, scale);
    return cudaGetLastError();
}
cudaError_t mk_launch_quantize_q8(const uint16_t* w, int64_t rows, int64_t cols, int col_scaled, int8_t* q,
                                  float* scale, cudaStream_t st) {
    return mk_launch_quantize(w, rows, cols, col_scaled, 8, q, scale, st);
}
cudaError_t mk_launch_relayout_rows_q4(uint8_t* arena, const int8_t* q, int64_t cols, const float* scale,
                                       const MkRowCopyQ* ops, int n, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    mk_relayout_rows_q4_kernel<<<n, 128, 0, st>>>(arena, q, cols, scale, ops, n);
    return cudaGetLastError();
}
cudaError_t mk_launch_relayout_cols_q4(uint8_t* arena, const int8_t* q, int H, int F, const MkColCopy* ops, int n,
                                       cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    dim3 grid((unsigned)n, (unsigned)((H / 2 + 127) / 128));
    mk_relayout_cols_q4_kernel<<<grid, 128, 0, st>>>(arena, q, H, F, ops, n);
    return cudaGetLastError();
}
cudaError_t mk_launch_relayout_rows_q8(uint8_t* arena, const int8_t* q, int64_t cols, const float* scale,
                                       const MkRowCopyQ* ops, int n, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    mk_relayout_rows_q8_kernel<<<n, 128, 0, st>>>(arena, q, cols, scale, ops, n);
    return cudaGetLastError();
}
cudaError_t mk_launch_relayout_cols_q8(uint8_t* arena, const int8_t* q, int H, int F, const MkColCopy* ops, int n,
                                       cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    dim3 grid(n, (H + 255) / 256);
    mk_relayout_cols_q8_kernel<<<grid, 256, 0, st>>>(arena, q, H, F, ops, n);
    return cudaGetLastError();
}
cudaError_t mk_launch_scatter_scales(uint8_t* arena, const float* scale, const MkScaleCopy* ops, int n,
                                     cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    mk_scatter_scales_kernel<<<(n + 255) / 256, 256, 0, st>>>(arena, scale, ops, n);
    return cudaGetLastError();
}

cudaError_t mk_launch_kv_rows(uint16_t* plain, uint16_t* cache_layer, int kvh, int n_pos, int pos0, int max_seq, int hd,
                              int swz, int to_cache, cudaStream_t st) {
    const int nch = hd / 8;
    if (swz && nch < 8) return cudaErrorInvalidValue;
    const int64_t n = (int64_t)kvh * n_pos * nch;
    if (n <= 0) return cudaSuccess;
    mk_kv_rows_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(reinterpret_cast<uint4*>(plain),
                                                                  reinterpret_cast<uint4*>(cache_layer), kvh, n_pos,
                                                                  pos0, max_seq, nch, swz, to_cache);
    return cudaGetLastError();
}

cudaError_t mk_launch_relayout_rows(uint8_t* arena, const uint16_t* src, int64_t src_cols, const MkRowCopy* ops, int n,
                                    cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    mk_relayout_rows_kernel<<<n, 128, 0, st>>>(arena, src, src_cols, ops, n);
    return cudaGetLastError();
}
cudaError_t mk_launch_relayout_cols(uint8_t* arena, const uint16_t* src, int H, int F, const MkColCopy* ops, int n,
                                    cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    dim3 grid(n, (H + 255) / 256);
    mk_relayout_cols_kernel<<<grid, 256, 0, st>>>(arena, src, H, F, ops, n);
    return cudaGetLastError();
}
cudaError_t mk_launch_rope_table(float* cs, float* sn, int max_seq, int hd, double theta, cudaStream_t st) {
    const int64_t n = (int64_t)max_seq * (hd / 2);
    mk_rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(cs, sn, max_seq, hd, theta);
    return cudaGetLastError();
}
cudaError_t mk_launch_bf16_to_f32(const uint16_t* src, float* dst, int64_t n, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    mk_bf16_to_f32_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(src, dst, n);
    return cudaGetLastError();
}
