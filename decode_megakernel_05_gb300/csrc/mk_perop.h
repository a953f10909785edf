// mk_perop.h - device state of the unfused per-operator baseline (internal).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

struct MkPerOp {
    int L, H, qh, kvh, hd, F, V, max_seq;
    float eps;
    int attn_chunk;          // positions per attention split
    int amax_blocks;
    // row-major weights
    const uint16_t* embed;
    const uint16_t* lm;
    std::vector<uint16_t*> wqkv, wo, wgu, wd;   // [qkv rows][H], [H][qh*hd], [2F][H] (gate then up), [H][F]
    const float *attn_norm, *ffn_norm, *final_norm, *rope_cos, *rope_sin;
    uint16_t *kc, *vc;
    int kv_swz;              // cache rows chunk-permuted by position (the long-context layout)
    // activations / scratch
    float *x, *xn, *qkv, *attn, *u, *hidden, *pml, *pacc, *logits_tmp;
    unsigned long long* amax_part;
    int32_t* next_token;
    uint32_t* status;
};

int mk_perop_step(const MkPerOp& P, int token, const int32_t* token_ptr, int pos, float* logits, cudaStream_t st,
                  cudaError_t* err);
cudaError_t mk_perop_prepare(int max_smem_k_bytes);
