// mk_prefill.h - launch description of the batched prefill (internal).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

struct MkPrefillArgs {
    int L, H, qh, kvh, hd, F, V, max_seq;
    float eps;
    int n, start;                  // prompt rows, position of the first
    int swz;                       // cache rows chunk-permuted by position
    const int32_t* tokens;         // [n] device
    // row-major bf16 weights: [qkv rows][H], [H][qh*hd], [2F][H] (gate then up), [H][F] per layer
    const uint16_t* const* wqkv;
    const uint16_t* const* wo;
    const uint16_t* const* wgu;
    const uint16_t* const* wd;
    const uint16_t *embed, *lm;    // [V][H]
    const float *attn_norm, *ffn_norm, *final_norm, *rope_cos, *rope_sin;
    uint16_t *kc, *vc;
    // fp32 workspace: x, xn [n][H], qkv [n][qkv rows], att [n][qh*hd], gu [n][2F], u [n][F]
    float *x, *xn, *qkv, *att, *gu, *u;
    // the three bf16 parts of a GEMM's activations, [3][parts_rows][K] for the GEMM's K (room for
    // max(H, F, qh*hd)); null: fp32 activations and the GEMMs on mma.sync instead of tcgen05
    uint16_t* parts;
    int parts_rows;
    int attn_tc;                   // 1: the causal attention on the tensor cores (query heads per KV group <= 8)
    float* hidden;                 // [H] final-norm output of the last row
    float* logits;                 // [V] logits of the last row
    unsigned long long* amax_part;
    int amax_blocks;
    int32_t* next_token;
    uint32_t* status;
};

// Allows the GEMMs their dynamic shared memory and fetches the tensor-map
// encoder (once per device).
cudaError_t mk_prefill_prepare();
// Enqueues the whole prefill on st; returns the number of kernel launches.
int mk_prefill_launch(const MkPrefillArgs& a, cudaStream_t st, cudaError_t* err);
