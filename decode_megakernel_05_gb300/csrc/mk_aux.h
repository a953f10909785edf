// mk_aux.h - set-up kernels and the re-layout copy descriptors (internal).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

struct MkRowCopy {     // arena + dst_off <- src[src_row][col0 .. col0 + ncols)
    int64_t dst_off;
    int64_t src_row;
    int32_t col0, ncols;
};
struct MkColCopy {     // arena + dst_off <- columns j0 .. j0+nj-1 of W_down, each H contiguous
    int64_t dst_off;
    int32_t j0, nj;
};

// Weight-only INT8 re-layout: arena + dst_off <- ncols int8 of q[src_row][col0 ..],
// and the row's scale (fp32) at arena + scale_off.
struct MkRowCopyQ {
    int64_t dst_off;
    int64_t src_row;
    int32_t col0, ncols;
    int64_t scale_off;
};
// arena + dst_off (fp32) <- scale[idx]
struct MkScaleCopy {
    int64_t dst_off;
    int64_t idx;
};

// Symmetric absmax INT8 quantization of a bf16 matrix [rows][cols] per row
// (or per column with col_scaled): scale = max|w| / 127, code = round(w /
// scale) ties to even, both float operations rounded to nearest; a group of
// zeros gets scale 0 and codes 0.  Each code q is written as the byte q + 128.
cudaError_t mk_launch_quantize_q8(const uint16_t* w, int64_t rows, int64_t cols, int col_scaled, int8_t* q,
                                  float* scale, cudaStream_t st);
cudaError_t mk_launch_relayout_rows_q8(uint8_t* arena, const int8_t* q, int64_t cols, const float* scale,
                                       const MkRowCopyQ* ops, int n, cudaStream_t st);
cudaError_t mk_launch_relayout_cols_q8(uint8_t* arena, const int8_t* q, int H, int F, const MkColCopy* ops, int n,
                                       cudaStream_t st);
// The same quantization with bits = 8 (as above) or 4 (scale = max|w| / 7,
// codes in [-7, 7], each written as the byte q + 8).
cudaError_t mk_launch_quantize(const uint16_t* w, int64_t rows, int64_t cols, int col_scaled, int bits, int8_t* q,
                               float* scale, cudaStream_t st);
// INT4 re-layout of such codes: rows (ncols codes -> ncols / 2 bytes) and
// W_down columns (H codes -> H / 2 bytes), packed as the stream keeps them.
cudaError_t mk_launch_relayout_rows_q4(uint8_t* arena, const int8_t* q, int64_t cols, const float* scale,
                                       const MkRowCopyQ* ops, int n, cudaStream_t st);
cudaError_t mk_launch_relayout_cols_q4(uint8_t* arena, const int8_t* q, int H, int F, const MkColCopy* ops, int n,
                                       cudaStream_t st);
cudaError_t mk_launch_scatter_scales(uint8_t* arena, const float* scale, const MkScaleCopy* ops, int n,
                                     cudaStream_t st);

cudaError_t mk_launch_relayout_rows(uint8_t* arena, const uint16_t* src, int64_t src_cols, const MkRowCopy* ops, int n,
                                    cudaStream_t st);
cudaError_t mk_launch_relayout_cols(uint8_t* arena, const uint16_t* src, int H, int F, const MkColCopy* ops, int n,
                                    cudaStream_t st);
cudaError_t mk_launch_rope_table(float* cs, float* sn, int max_seq, int hd, double theta, cudaStream_t st);
cudaError_t mk_launch_bf16_to_f32(const uint16_t* src, float* dst, int64_t n, cudaStream_t st);
// K or V rows of one layer between a plain [kvh][n_pos][hd] bf16 buffer and the
// cache ([kvh][max_seq][hd] from cache_layer), positions pos0 .. pos0+n_pos-1,
// each row's 16-byte chunks permuted as the cache keeps them (swz); to_cache
// selects the direction.  Both buffers are device memory.
cudaError_t mk_launch_kv_rows(uint16_t* plain, uint16_t* cache_layer, int kvh, int n_pos, int pos0, int max_seq, int hd,
                              int swz, int to_cache, cudaStream_t st);
// Records a failed CUDA call as the text mk_last_cuda_error() returns ("what:
// error string (code)") and maps it to MK_ERR_OOM or MK_ERR_CUDA.
int mk_record_cuda_error(cudaError_t e, const char* what);
