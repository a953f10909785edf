/*
 * mk.h - C ABI of the GB300 batch-size-1 decode megakernel library.
 *
 * The library runs autoregressive decode of a Llama-style decoder one token at
 * a time with a KV cache (the single-request, bs=1 decode problem of
 * cloud.baidu.com/article/9434380, sections 1-3), as ONE persistent CUDA
 * kernel launch per token.  Inside that launch the per-layer segments
 * (cloud.baidu.com/article/9434380, section 5, step 2):
 *   A: RMSNorm + fused Q/K/V GEMV + RoPE + K/V append,
 *   B: GQA attention over the cache (split over CTAs) + output projection
 *      + residual,
 *   C: RMSNorm + gate/up GEMV + SiLU*up + down GEMV + residual,
 * and finally RMSNorm, the LM-head GEMV and the greedy argmax, are separated
 * by inter-CTA flags instead of kernel boundaries, while a producer warp per
 * CTA streams pre-laid-out bf16 weight tiles into a shared-memory ring with
 * bulk asynchronous copies so that weight loading never stops between
 * segments (cloud.baidu.com/article/9434380, sections 4.2 and 5, step 3;
 * developer.baidu.com/article/detail.html?id=8006242, section 4.1).
 *
 * Conventions (all entry points):
 *   - Every function returns MK_OK (0) or a negative MK_ERR_* code.  Argument
 *     errors are detected on the host before anything is launched.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued on it and the call returns without waiting,
 *     unless the function says it synchronizes.
 *   - Device-side errors (a bounded wait that timed out, a non-finite logit,
 *     a token id read from device memory that is out of range) are latched
 *     into a status word on the device; mk_status() reads and clears it, and
 *     mk_generate_greedy() checks it before returning.
 *   - A context is not thread-safe and must be used from one stream at a time.
 *   - All pointers to caller data are borrowed for the duration of the call;
 *     the caller keeps ownership.
 */
#ifndef MK_H
#define MK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_OK 0
#define MK_ERR_INVALID_ARG (-1)    /* bad pointer, size, shape, token or position */
#define MK_ERR_OOM (-2)            /* device or host allocation failed */
#define MK_ERR_CUDA (-3)           /* a CUDA runtime call failed (see mk_last_cuda_error) */
#define MK_ERR_DEVICE_TIMEOUT (-4) /* a device-side wait ran past its limit; the launch gave up */
#define MK_ERR_NUMERIC (-5)        /* a logit was NaN or infinite */
#define MK_ERR_STATE (-6)          /* call out of order (e.g. decode before weights are loaded) */
#define MK_ERR_UNSUPPORTED (-7)    /* shape outside what the kernels are built for */

typedef struct mk_ctx mk_ctx; /* opaque, owned by the library */

/* Model shape.  Weights are bf16, activations fp32. */
typedef struct {
    int32_t n_layers;
    int32_t hidden;        /* H */
    int32_t n_q_heads;     /* qh */
    int32_t n_kv_heads;    /* kvh; qh % kvh == 0 (grouped-query attention) */
    int32_t head_dim;      /* hd: 64 or 128 */
    int32_t ffn;           /* F (SwiGLU inner size) */
    int32_t vocab;         /* V */
    int32_t max_seq;       /* KV-cache capacity in positions */
    float rms_eps;         /* RMSNorm epsilon */
    float rope_theta;      /* RoPE base */
    int32_t tie_embeddings;/* 1: LM head = embedding matrix */
} mk_config;

/* Tuning knobs of the fused kernel (cloud.baidu.com/article/9434380, section 6:
 * tile granularity, pipeline depth and on-chip buffer split are configuration,
 * not constants).  Zero in any field selects the default. */
typedef struct {
    int32_t ring_stages;     /* shared-memory ring slots per CTA (default: as many as fit, <= 6,
                                or <= 8 for weight_int4); 1 = no overlap of loading and compute
                                ("prefetch off") */
    int32_t slot_kib;        /* bytes per ring slot / weight tile, KiB (maximum 32; default 32, or 24
                                for weight_int4) */
    int32_t l2_prefetch_kib; /* how far (KiB of tile stream) each CTA prefetches into L2 ahead of
                                its ring copies (default, zero or negative: off -- on this path the
                                extra L2 traffic cost more than the hidden latency saved) */
    int32_t grid_ctas;       /* CTAs of the persistent grid (default: n_kv_heads * floor(SMs / n_kv_heads));
                                must be a multiple of n_kv_heads and fit one CTA per SM */
    int32_t weight_int8;     /* nonzero: weight-only INT8 (stapisi.com/news/3904786, section 6:
                                quantization fused into the kernels).  mk_load_weights quantizes
                                every matrix on the device -- symmetric absmax, one fp32 scale
                                s = max|w| / 127 per output row (per input column for w_down),
                                codes round(w / s) ties to even in [-127, 127], both divisions
                                rounded to nearest -- and the step streams the codes (each as the
                                byte code + 128) and the scales,
                                dequantizing in registers (activations, accumulation, norms, the
                                embedding row and the KV cache stay as in the bf16 path).
                                Built for (head_dim, q heads per KV head, hidden) = (64, 2, 256),
                                (64, 4, 2048) and (128, 4, 4096); other shapes return
                                MK_ERR_UNSUPPORTED from mk_create, as do mk_enable_perop(.., 1),
                                mk_prefill and mk_relayout_host on an int8 context / tuning */
    int32_t weight_int4;     /* nonzero: weight-only INT4 (the same page and section), the INT8
                                scheme with 7 levels a side: s = max|w| / 7 per output row (per
                                input column for w_down), codes round(w / s) ties to even in
                                [-7, 7], both divisions rounded to nearest; the step streams two
                                codes a byte (each as the nibble code + 8) and the fp32 scales.
                                Built for the same three shapes as INT8, with the same
                                restrictions; setting both weight_int8 and weight_int4 is
                                MK_ERR_INVALID_ARG from mk_create and mk_relayout_host */
} mk_tuning;

/* Weights, row-major [out, in] bf16 (raw 16-bit patterns).  Either all host
 * pointers (on_device = 0) or all device pointers (on_device = 1). */
typedef struct {
    const void* embed;              /* [V][H] */
    const void* lm_head;            /* [V][H]; NULL iff tie_embeddings */
    const void* final_norm;         /* [H] */
    const void* const* attn_norm;   /* n_layers pointers, each [H] */
    const void* const* wq;          /* each [qh*hd][H] */
    const void* const* wk;          /* each [kvh*hd][H] */
    const void* const* wv;          /* each [kvh*hd][H] */
    const void* const* wo;          /* each [H][qh*hd] */
    const void* const* ffn_norm;    /* each [H] */
    const void* const* w_gate;      /* each [F][H] */
    const void* const* w_up;        /* each [F][H] */
    const void* const* w_down;      /* each [H][F] */
    int32_t on_device;
} mk_weights;

/* Read-only facts about a context (for benchmarks and tests). */
typedef struct {
    int32_t grid_ctas, ctas_per_group, block_threads, ring_stages, slot_bytes;
    int32_t smem_bytes, sm_count, l2_prefetch_bytes;
    int64_t arena_bytes;             /* re-laid-out weight stream bytes on the device */
    int64_t weight_bytes_per_token;  /* weight bytes one step reads: matrices (bf16, or int8 / int4 codes
                                        + fp32 scales), gains and 1 embedding row at 2 bytes a value */
    int64_t kv_bytes_per_position;   /* bf16 K+V bytes one attended position costs (all layers) */
    int64_t device_bytes;            /* everything the context allocated on the device */
    int32_t attn_tc;                 /* 1: a build whose attention runs on the tensor cores exists
                                        for this shape (4 query heads of 64 dims per KV group) */
    int32_t attn_tc_min_ctx;         /* context length (pos + 1) from which a step launches that
                                        build; shorter contexts run the lane-parallel attention
                                        (-1 without attn_tc) */
    int32_t attn_pos_per_cta;        /* length-adaptive split: a step at context ctx runs its
                                        attention on ceil(ctx / attn_pos_per_cta) CTAs of each KV
                                        group, at most ctas_per_group (0: the count is forced
                                        with MK_DBG_ATTN_CTAS) */
    int32_t weight_int8;             /* 1: the context streams weight-only INT8 (mk_tuning) */
    int32_t weight_int4;             /* 1: the context streams weight-only INT4 (mk_tuning) */
} mk_info;

/* Create a context on CUDA device `device`: validates the shape, sizes the
 * persistent grid to the SM count, allocates the weight arena, the bf16 KV
 * cache [n_layers][kvh][max_seq][hd] (K and V), fp32 scratch and the RoPE
 * table.  `tuning` may be NULL.  On success *out owns everything. */
int mk_create(const mk_config* cfg, const mk_tuning* tuning, int device, mk_ctx** out);

/* Offline weight re-layout (cloud.baidu.com/article/9434380, section 9: lay
 * weights out in access order ahead of time).  Copies every matrix into the
 * arena as per-CTA streams of contiguous bf16 tiles in the order the kernel
 * consumes them.  Synchronizes `stream` before returning, so the caller may
 * free its buffers afterwards. */
int mk_load_weights(mk_ctx* ctx, const mk_weights* w, void* stream);

/* Pre-fill cache positions [0, n_pos) of one layer.  k, v: bf16 [kvh][n_pos][hd],
 * host or device memory; K must already be rotated (post-RoPE), as decode
 * steps store it.  Synchronizes `stream`.  Where the cache keeps its rows
 * chunk-permuted (mk_info.attn_tc), the rows pass through a temporary device
 * buffer of 4 * kvh * n_pos * hd bytes, allocated and freed by the call
 * (MK_ERR_OOM if it cannot be had); the caller's layout is the same either
 * way. */
int mk_set_kv(mk_ctx* ctx, int32_t layer, const void* k, const void* v, int32_t n_pos, void* stream);

/* Copy cache positions [pos0, pos0 + n_pos) of one layer out to k_out, v_out
 * (bf16 [kvh][n_pos][hd], host or device memory, rows in plain order whatever
 * the cache's layout; a temporary device buffer as for mk_set_kv).
 * Synchronizes `stream`. */
int mk_get_kv(mk_ctx* ctx, int32_t layer, int32_t pos0, int32_t n_pos, void* k_out, void* v_out, void* stream);

/* Copy bytes [offset, offset + bytes) of the device weight arena (the
 * re-laid-out tile streams, mk_info.arena_bytes long) to `out` (host or
 * device memory); synchronizes `stream`.  For layout checks of streams only
 * the device builds (weight-only INT8).  MK_ERR_INVALID_ARG for a range
 * outside the arena, MK_ERR_STATE before mk_load_weights. */
int mk_read_arena(mk_ctx* ctx, int64_t offset, int64_t bytes, void* out, void* stream);

/* One decode step (one kernel launch): feed `token` at position `pos`, write
 * its K/V into cache slot `pos`, attend over slots [0, pos], and write the
 * fp32 logits [V] to `logits_out` (device memory, caller-owned; NULL = do not
 * store logits).  The greedy argmax is always computed and kept on the device
 * (mk_get_argmax).  Requires 0 <= token < V and 0 <= pos < max_seq; slots
 * above `pos` are ignored, so rewinding to an earlier `pos` is allowed.
 * Asynchronous. */
int mk_decode_step(mk_ctx* ctx, int32_t token, int32_t pos, float* logits_out, void* stream);

/* One decode step fed with the previous step's greedy token, which the kernel
 * reads from device memory (no host round trip between tokens).  Otherwise as
 * mk_decode_step.  The token after mk_create is 0.  Asynchronous. */
int mk_decode_step_greedy(mk_ctx* ctx, int32_t pos, float* logits_out, void* stream);

/* Greedy generation (cloud.baidu.com/article/9434380, section 5, step 5:
 * sampling and multi-step state advance run on the fused path).  Feeds the
 * n_prompt prompt tokens (host int32) at positions start_pos.., then n_new - 1
 * more steps, each fed the previous step's argmax, which the kernel reads from
 * device memory: no host round trip between tokens.  Writes the n_new
 * generated tokens to out_tokens (host int32 [n_new]).  Launches
 * n_prompt + n_new - 1 kernels, synchronizes `stream` once (the tokens and the
 * status word are copied back behind the launches) and returns the device
 * status (MK_ERR_DEVICE_TIMEOUT / MK_ERR_NUMERIC), clearing it, if one was
 * latched.  The library holds 4 bytes of pinned host memory per context for
 * that status copy. */
int mk_generate_greedy(mk_ctx* ctx, const int32_t* prompt, int32_t n_prompt, int32_t start_pos,
                       int32_t n_new, int32_t* out_tokens, void* stream);

/* Sampling (cloud.baidu.com/article/9434380, section 5: step 1 fixes the
 * sampling parameters such as the temperature; step 5 re-verifies sampling
 * and the stop condition on the fused path).  The next token is drawn from
 * softmax(logits / temperature) by the Gumbel-max rule, inside the argmax of
 * the same launch: token = argmax_v fmaf(logit_v, 1/temperature, G_v) over
 * the finite logits (lowest index on ties), G_v = -ln(-ln U_v) in fp32, and
 * U_v = ((z >> 41) + 0.5) * 2^-23 with z output i = pos * 2^32 + v of
 * SplitMix64 seeded with `seed` in its counter form, mix(seed + (i + 1) *
 * 0x9E3779B97F4A7C15) (Steele, Lea and Flood, OOPSLA 2014).  temperature <= 0
 * is greedy.  With a top-p below 1 (mk_set_top_p) the Gumbel-max runs over the
 * nucleus only: with x_v = logit_v * (1/temperature), token v is kept iff the
 * tokens with a larger x carry less than top_p of softmax(x)'s mass (tied
 * tokens are kept or dropped together), which samples from softmax(x)
 * restricted to the nucleus and renormalised.  The threshold is found inside
 * the same launch (a bisection on x over grid-wide reductions, 8 of them; the
 * boundary is resolved to 104 / 32^7 in x, and the masses are fp32 sums).
 *
 * One sampled step: as mk_decode_step, fed `token` (0..V-1), or with token =
 * -1 the previous step's chosen token from device memory.  The chosen token
 * is left on the device (mk_get_argmax).  Asynchronous. */
int mk_decode_step_sample(mk_ctx* ctx, int32_t token, int32_t pos, float temperature, uint64_t seed,
                          float* logits_out, void* stream);

/* Nucleus mass of the sampled steps of this context (mk_decode_step_sample,
 * mk_generate with temperature > 0) from now on: 0 < top_p <= 1, 1 (the
 * default) keeps every token.  Anything else returns MK_ERR_INVALID_ARG. */
int mk_set_top_p(mk_ctx* ctx, float top_p);

/* Generation with sampling and a stop token: as mk_generate_greedy, with the
 * tokens chosen as in mk_decode_step_sample.  With eos_id >= 0, generation
 * stops at the first generated token equal to eos_id: every later launch
 * returns at once (no K/V written, no state advanced).  out_tokens (host
 * int32 [n_new]) receives the tokens up to and including it and -1 after;
 * *n_out (may be NULL) their number.  Synchronizes `stream`; returns the
 * device status like mk_generate_greedy. */
int mk_generate(mk_ctx* ctx, const int32_t* prompt, int32_t n_prompt, int32_t start_pos, int32_t n_new,
                float temperature, uint64_t seed, int32_t eos_id, int32_t* out_tokens, int32_t* n_out,
                void* stream);

/* The last step's final-norm hidden state (fp32 [H]) into `out` (device). */
int mk_get_hidden(mk_ctx* ctx, float* out, void* stream);

/* The last step's greedy token (int32) into `out` (device). */
int mk_get_argmax(mk_ctx* ctx, int32_t* out, void* stream);

/* Synchronizes the context's last stream, reads and clears the device status
 * word.  Returns MK_OK, MK_ERR_DEVICE_TIMEOUT, MK_ERR_NUMERIC or
 * MK_ERR_INVALID_ARG (a device-read token id was out of range). */
int mk_status(mk_ctx* ctx);

/* Unfused baseline of the same step: the same arithmetic launched as one
 * kernel per operator (9 per layer + 5: 149 for the 16-layer 1B shape), on plain row-major weights
 * (cloud.baidu.com/article/9434380, section 5, step 5 keeps the per-operator
 * path for comparison and debugging; section 7 asks for the fusion-off
 * ablation).  Needs mk_load_weights to have run with keep_rowmajor = 1 in
 * mk_enable_perop before it.  Asynchronous; returns the number of kernel
 * launches it issued through *n_launches (may be NULL). */
int mk_enable_perop(mk_ctx* ctx, int32_t keep_rowmajor);
int mk_decode_step_perop(mk_ctx* ctx, int32_t token, int32_t pos, float* logits_out, void* stream,
                         int32_t* n_launches);

/* Batched prefill (cloud.baidu.com/article/9434380, sections 2 and 8, problem
 * 2: prefill and decode are separate phases; the prompt is a dense,
 * compute-bound contraction).  Runs the n prompt tokens (host int32, each in
 * 0..V-1) at positions start_pos .. start_pos + n - 1 through every layer
 * together: RMSNorm, tensor-core GEMMs for QKV, O, gate/up and down (bf16
 * weights, each fp32 activation split into two bf16 parts), RoPE, the K/V rows
 * written to the cache, causal attention over positions [0, position].  The
 * cache then holds what n decode steps would have written (up to rounding
 * order), the last row's final-norm hidden state is kept (mk_get_hidden), its
 * logits go to logits_out (device fp32 [V], or NULL), and its greedy token is
 * left on the device for mk_decode_step_greedy / mk_get_argmax.  Needs the
 * row-major weight copies (mk_enable_perop(ctx, 1) before mk_load_weights;
 * MK_ERR_STATE otherwise) and F, H multiples of 8 (MK_ERR_UNSUPPORTED).
 * Requires start_pos + n <= max_seq.  Allocates its fp32 workspace (about
 * n * (4H + 3F + qkv rows + qh*hd) * 4 bytes) on the first call and when a
 * longer prompt arrives, synchronizing the stream then; otherwise
 * asynchronous.  Device-side errors (a non-finite logit) are latched in the
 * status word (mk_status). */
int mk_prefill(mk_ctx* ctx, const int32_t* tokens, int32_t n, int32_t start_pos, float* logits_out, void* stream);

int mk_get_info(const mk_ctx* ctx, mk_info* out);

/* Greedy token over a caller's fp32 logits without allocating anything (the
 * pages have no counterpart: this serves callers that cannot call cudaMalloc,
 * e.g. engines that reserve all device memory up front and hand out pointers
 * into their own pool, or latency-critical code that must not allocate).
 * logits: device fp32 [n]; out_token: device int32, receives the index of the
 * largest finite logit (lowest index on ties), or -1 if none is finite.
 * The scratch (one partial result per block) is a fixed device array inside
 * the library, MK_NOALLOC_ARGMAX_BLOCKS * 8 bytes, held by every GPU that
 * loads the library until the process exits.  n > MK_NOALLOC_ARGMAX_MAX_N (or
 * n < 1, or a NULL pointer) returns MK_ERR_INVALID_ARG without launching.
 * The first call on a device looks up the array's device address (with that
 * device current) and keeps it for the life of the process; make that first
 * call before any stream capture, and do not use this entry point on a device
 * after cudaDeviceReset (the reset unloads the array, and the kept address is
 * then stale).  Every call shares the array: calls whose kernels overlap on
 * the GPU (e.g. two streams at once) race and must be serialized by the
 * caller.  -0.0 and +0.0 count as equal (the lower index wins).  A launch
 * that fails returns MK_ERR_CUDA (mk_last_cuda_error names the kernel).
 * Runs on the calling thread's current device; asynchronous on `stream`. */
#define MK_NOALLOC_ARGMAX_BLOCKS 1024
#define MK_NOALLOC_ARGMAX_MAX_N (MK_NOALLOC_ARGMAX_BLOCKS * 4096)
int mk_argmax_f32_noalloc(const float* logits, int32_t n, int32_t* out_token, void* stream);

/* Debug knobs (off by default).  MK_DBG_SKIP_ARRIVAL: value = cta * 65536 + sync_id
 * makes that CTA skip one flag arrival, so every CTA waiting on it runs into its
 * bounded wait (used by the failure-detection test; -1 = off).  sync_id = 4 * layer
 * + {0: q/k/v ready, 1: attention partials ready, 2: attention block done,
 * 3: FFN block done}.  MK_DBG_WAIT_LIMIT_NS: limit of every device-side wait
 * (default 1e9 ns). */
#define MK_DBG_SKIP_ARRIVAL 1
#define MK_DBG_WAIT_LIMIT_NS 2
/* MK_DBG_TRACE: value = device address of a uint64 buffer [grid_ctas][4096]
 * (0 = off).  Each step then records per CTA the %globaltimer (ns) at the end
 * of every segment: slot 16*layer + e for e = 0 layer start, 1 RMSNorm,
 * 2 QKV GEMV, 3 RoPE/KV append, 4 q/k/v flag seen, 5 attention partials,
 * 6 partials flag seen, 7 combine, 8 O-proj, 9 attention-block flag seen,
 * 10 RMSNorm, 11 gate/up, 12 down, 13 FFN-block flag seen; slot 16*L + 0
 * final RMSNorm, +1 LM head, +2 end, +3 start; slot 1024 + 8*layer + phase
 * (0 QKV, 1 attention, 2 O-proj, 3 gate/up, 4 down; 8*L + 5 LM head): ns the
 * consumers waited for ring data; slot 1536 + k/16: cumulative ns the copy
 * producer waited for a free slot after its k-th tile; slot 1535: producer done;
 * slot 2048 + k (k < 256): thread 0 got LM-head tile k; for the first 512
 * tiles of the step's stream: 2560 + k issue time, 3072 + k time a reader got
 * it, 3584 + k time a reader released it. */
#define MK_DBG_TRACE 3
/* MK_DBG_TRACE_DETAIL: 1 (default) = the trace also records the per-tile and
 * ring-wait slots; 0 = segment ends only (the least perturbed timing); 2 =
 * segment ends, and the detail marks as SM clock counts (for durations within
 * a CTA) without the per-tile records.  Detail marks (thread 0, layers < 24)
 * sit at slot 1600 + 16*layer + m: m = 7 attention segment entered, 0 q polled,
 * 1 q ready for every warp, 5 first K/V block taken, 6 its scores done, 2 all
 * blocks done, 3 first partials seen, 4 every thread's first partials seen,
 * 10 combine weights done, 11 its share of o written, 8 first O-proj tile
 * taken, 9 O-proj tiles done, 12 attention-block arrival issued. */
#define MK_DBG_TRACE_DETAIL 5
/* MK_DBG_INFLIGHT: value = most weight tiles each CTA keeps in flight (issued,
 * not yet landed) at once during the streaming segments, 1..16 (0 = the
 * default, 3).  Fewer bytes in
 * flight per SM shorten the queues every other global access of the step
 * (flags, activations) waits in, at the same streaming bandwidth. */
#define MK_DBG_INFLIGHT 6
/* MK_DBG_INFLIGHT_LAT: the same limit while the consumers are in a
 * latency-bound segment (norms, QKV, attention, O-proj, flag waits); the first
 * limit applies during the streaming segments (gate/up, down, LM head).
 * 0 = the default (1). */
#define MK_DBG_INFLIGHT_LAT 7
/* MK_DBG_PF_LEAD: the L2 warmer (tuning l2_prefetch_kib > 0) leaves the first
 * `value` tiles past the copy producer's cursor alone (the ring fetches those
 * as soon as slots free up) and warms the tiles after them; 0..64, -1 = the
 * default (the ring's slot count). */
#define MK_DBG_PF_LEAD 8
/* MK_DBG_PF_DEPTH: tiles of warming loads the L2 warmer keeps in flight,
 * 1 or 2 (0 = the default, 1). */
#define MK_DBG_PF_DEPTH 9
/* MK_DBG_ATTN_BUILD: which build a step launches: 0 (default) by context length
 * (attn_tc_min_ctx), 1 the lane-parallel attention always, 2 the tensor-core
 * attention always (MK_ERR_INVALID_ARG without attn_tc).  MK_DBG_ATTN_TC_MIN:
 * positions per CTA from which the default picks the tensor-core build
 * (default 0: every step; 0 .. max_seq). */
#define MK_DBG_ATTN_BUILD 10
#define MK_DBG_ATTN_TC_MIN 11
/* MK_DBG_ATTN_CTAS: value = CTAs of each KV group that run every step's
 * attention, 1 .. ctas_per_group (0 = by context length, the default).
 * MK_DBG_ATTN_POS_PER_CTA: positions per attention CTA of the default split
 * (1 .. max_seq; the default is mk_info.attn_pos_per_cta). */
#define MK_DBG_ATTN_CTAS 12
#define MK_DBG_ATTN_POS_PER_CTA 13
/* MK_DBG_STREAM_TAIL: where a layer's streaming segment (the copy producer's
 * larger in-flight limit) ends: 0 (default) after the down projection's tiles,
 * 1 after the FFN-block flag wait, 2 after the next layer's QKV GEMV. */
#define MK_DBG_STREAM_TAIL 14
/* MK_DBG_PREFILL_GEMM: the engines of mk_prefill: 0 (default) tcgen05 GEMMs
 * (TMA tiles, TMEM accumulators) and the causal attention on the tensor cores
 * (mma.sync, up to 8 query heads per KV group); 1 the warp-level mma.sync GEMMs
 * and the CUDA-core attention (the ablation). */
#define MK_DBG_PREFILL_GEMM 15
int mk_set_debug(mk_ctx* ctx, int32_t knob, int64_t value);

const char* mk_strerror(int code);
/* Text of the last CUDA error seen by this thread's calls into the library. */
const char* mk_last_cuda_error(void);
void mk_destroy(mk_ctx* ctx);

/* Host-only layout utilities (no GPU needed).  mk_arena_bytes: size of the
 * re-laid-out weight arena for `grid_ctas` CTAs, for the tuning's weight form
 * (bf16, weight_int8 or weight_int4); -1 for an invalid shape, grid or tuning
 * (both weight forms at once).  mk_relayout_host: build that arena on the host
 * from host weights (the same layout mk_load_weights writes on the device;
 * bf16 only). */
int64_t mk_arena_bytes(const mk_config* cfg, const mk_tuning* tuning, int32_t grid_ctas);
int mk_relayout_host(const mk_config* cfg, const mk_tuning* tuning, int32_t grid_ctas, const mk_weights* w,
                     void* arena_out);

#ifdef __cplusplus
}
#endif

#endif /* MK_H */
