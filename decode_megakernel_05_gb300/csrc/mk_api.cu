// mk_api.cu - host runtime and C ABI of the decode megakernel library (see
// include/mk.h for the contract of every entry point).
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <string>
#include <vector>

#include "../../include/mk.h"
#include "mk_aux.h"
#include "mk_internal.h"
#include "mk_perop.h"
#include "mk_prefill.h"

// One object per kernel variant: mk_kernel.cu compiled with -DMK_HD_V=<head_dim>
// -DMK_G_V=<q heads per kv head> -DMK_MH_V=<hidden / 256> (-DMK_LC_V=1 for the
// long-context builds, whose attention runs on the tensor cores); keep in sync
// with VARIANTS in build.py.
#define MK_VARIANTS(X) \
    X(64, 2, 1) X(64, 4, 2) X(64, 4, 4) X(64, 4, 8) X(64, 4, 16) X(128, 4, 4) X(128, 4, 8) X(128, 4, 16)
#define MK_LC_VARIANTS(X) X(64, 4, 2) X(64, 4, 8) X(128, 4, 4) X(128, 4, 16)
// Weight-only INT8 builds (-DMK_WB_V=1; keep in sync with Q8_VARIANTS and
// Q8_LC_VARIANTS in build.py).
#define MK_Q8_VARIANTS(X) X(64, 2, 1) X(64, 4, 8) X(128, 4, 16)
#define MK_Q8_LC_VARIANTS(X) X(64, 4, 8)
// Weight-only INT4 builds (-DMK_WB_V=0; keep in sync with Q4_VARIANTS and
// Q4_LC_VARIANTS in build.py).
#define MK_Q4_VARIANTS(X) X(64, 2, 1) X(64, 4, 8) X(128, 4, 16)
#define MK_Q4_LC_VARIANTS(X) X(64, 4, 8) X(128, 4, 16)
// Each variant exists twice: without trace code (launched normally) and with
// it (launched while a segment trace is requested).
#define MK_DECL(hd, g, mh)                                         \
    extern "C" const void* mk_kernel_ptr_##hd##_##g##_##mh(void); \
    extern "C" const void* mk_kernel_trace_ptr_##hd##_##g##_##mh(void);
#define MK_DECL_LC(hd, g, mh)                                          \
    extern "C" const void* mk_kernel_ptr_##hd##_##g##_##mh##_lc(void); \
    extern "C" const void* mk_kernel_trace_ptr_##hd##_##g##_##mh##_lc(void);
#define MK_DECL_Q8(hd, g, mh)                                          \
    extern "C" const void* mk_kernel_ptr_##hd##_##g##_##mh##_q8(void); \
    extern "C" const void* mk_kernel_trace_ptr_##hd##_##g##_##mh##_q8(void);
#define MK_DECL_LC_Q8(hd, g, mh)                                          \
    extern "C" const void* mk_kernel_ptr_##hd##_##g##_##mh##_lc_q8(void); \
    extern "C" const void* mk_kernel_trace_ptr_##hd##_##g##_##mh##_lc_q8(void);
#define MK_DECL_Q4(hd, g, mh)                                          \
    extern "C" const void* mk_kernel_ptr_##hd##_##g##_##mh##_q4(void); \
    extern "C" const void* mk_kernel_trace_ptr_##hd##_##g##_##mh##_q4(void);
#define MK_DECL_LC_Q4(hd, g, mh)                                          \
    extern "C" const void* mk_kernel_ptr_##hd##_##g##_##mh##_lc_q4(void); \
    extern "C" const void* mk_kernel_trace_ptr_##hd##_##g##_##mh##_lc_q4(void);
MK_VARIANTS(MK_DECL)
MK_LC_VARIANTS(MK_DECL_LC)
MK_Q8_VARIANTS(MK_DECL_Q8)
MK_Q8_LC_VARIANTS(MK_DECL_LC_Q8)
MK_Q4_VARIANTS(MK_DECL_Q4)
MK_Q4_LC_VARIANTS(MK_DECL_LC_Q4)
#undef MK_DECL
#undef MK_DECL_LC
#undef MK_DECL_Q8
#undef MK_DECL_LC_Q8
#undef MK_DECL_Q4
#undef MK_DECL_LC_Q4

// The kernel for a shape and weight form (wb = 2 bf16, 1 weight-only INT8, 0 INT4);
// with long_ctx, its long-context (tensor-core attention) build where one
// exists.  Returns 1 for a long-context build, 0 for the standard one, -1 if
// none fits.
static int mk_kernel_variant(int hd, int G, int H, int wb, bool long_ctx, const void** fn, const void** fn_trace) {
#define MK_PICK(hd_, g_, mh_, wb_, lc_, sfx)                                  \
    if ((!lc_ || long_ctx) && wb == wb_ && hd == hd_ && G == g_ && H == 256 * mh_) { \
        *fn = mk_kernel_ptr_##hd_##_##g_##_##mh_##sfx();                      \
        *fn_trace = mk_kernel_trace_ptr_##hd_##_##g_##_##mh_##sfx();          \
        return lc_;                                                           \
    }
#define MK_PICK_LC(hd_, g_, mh_) MK_PICK(hd_, g_, mh_, 2, 1, _lc)
#define MK_PICK_STD(hd_, g_, mh_) MK_PICK(hd_, g_, mh_, 2, 0, )
#define MK_PICK_LC_Q8(hd_, g_, mh_) MK_PICK(hd_, g_, mh_, 1, 1, _lc_q8)
#define MK_PICK_Q8(hd_, g_, mh_) MK_PICK(hd_, g_, mh_, 1, 0, _q8)
#define MK_PICK_LC_Q4(hd_, g_, mh_) MK_PICK(hd_, g_, mh_, 0, 1, _lc_q4)
#define MK_PICK_Q4(hd_, g_, mh_) MK_PICK(hd_, g_, mh_, 0, 0, _q4)
    MK_LC_VARIANTS(MK_PICK_LC)
    MK_Q8_LC_VARIANTS(MK_PICK_LC_Q8)
    MK_Q4_LC_VARIANTS(MK_PICK_LC_Q4)
    MK_VARIANTS(MK_PICK_STD)
    MK_Q8_VARIANTS(MK_PICK_Q8)
    MK_Q4_VARIANTS(MK_PICK_Q4)
#undef MK_PICK_LC
#undef MK_PICK_STD
#undef MK_PICK_LC_Q8
#undef MK_PICK_Q8
#undef MK_PICK_LC_Q4
#undef MK_PICK_Q4
#undef MK_PICK
    *fn = *fn_trace = nullptr;
    return -1;
}

namespace {

thread_local std::string g_cuda_err;

int cuda_fail(cudaError_t e, const char* what) {
    char buf[256];
    snprintf(buf, sizeof buf, "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
    g_cuda_err = buf;
    return e == cudaErrorMemoryAllocation ? MK_ERR_OOM : MK_ERR_CUDA;
}

}  // namespace

int mk_record_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }

namespace {

#define MK_CU(call)                                   \
    do {                                              \
        cudaError_t e_ = (call);                      \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
    } while (0)

// Where each weight goes in the arena: row copies (with, for int8 streams,
// where the row's scale goes), column blocks of W_down, and for int8 the
// W_down column scales kept in the GU tiles.
struct Maps {
    std::vector<std::vector<MkRowCopyQ>> q, k, v, o, gate, up;
    std::vector<std::vector<MkColCopy>> down;
    std::vector<std::vector<MkScaleCopy>> down_scale;
    std::vector<MkRowCopyQ> lm;
};

std::vector<MkRowCopy> plain_rows(const std::vector<MkRowCopyQ>& v) {
    std::vector<MkRowCopy> r;
    r.reserve(v.size());
    for (const MkRowCopyQ& o : v) r.push_back(MkRowCopy{o.dst_off, o.src_row, o.col0, o.ncols});
    return r;
}

// Tuning with defaults applied (grid size needs the SM count).
struct Tune {
    int ns_req, slot, l2pf, grid, wb;
};

Tune resolve_tuning(const mk_tuning* t) {
    Tune r;
    r.wb = (t && t->weight_int4) ? 0 : (t && t->weight_int8) ? 1 : 2;
    // the same 192 KB ring in 6 slots of 32 KB, or for INT4 in 8 of 24 KB:
    // a 32 KB tile holds 30 int4 rows of 2048 codes, so a CTA's QKV rows
    // make one tile for one consumer group and gate/up too few tiles for
    // three; 22-row tiles measured 1.9 % faster on the 1B shape (16 KB ones
    // 1.5 % slower)
    const int slot_kib = r.wb == 0 ? 24 : 32;
    r.ns_req = (t && t->ring_stages > 0) ? t->ring_stages : 192 / slot_kib;
    r.slot = (t && t->slot_kib > 0) ? t->slot_kib * 1024 : slot_kib * 1024;
    r.l2pf = (t && t->l2_prefetch_kib > 0) ? t->l2_prefetch_kib * 1024 : 0;   // default off (measured slower)
    r.grid = (t && t->grid_ctas > 0) ? t->grid_ctas : 0;
    return r;
}

// Shape checks shared by mk_create and the host layout utilities; the fused
// kernel must also be built for the shape when need_kernel is set.
int check_shape(const mk_config* c, bool need_kernel = true, int wb = 2) {
    if (!c) return MK_ERR_INVALID_ARG;
    if (c->n_layers < 1 || c->hidden < 8 || c->n_q_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 2 ||
        c->ffn < 1 || c->vocab < 1 || c->max_seq < 1 || !(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f))
        return MK_ERR_INVALID_ARG;
    if (c->n_q_heads % c->n_kv_heads) return MK_ERR_INVALID_ARG;
    if (c->head_dim != 64 && c->head_dim != 128) return MK_ERR_UNSUPPORTED;
    const int G = c->n_q_heads / c->n_kv_heads;
    const void *fn = nullptr, *fn_trace = nullptr;
    if (need_kernel && mk_kernel_variant(c->head_dim, G, c->hidden, wb, false, &fn, &fn_trace) < 0)
        return MK_ERR_UNSUPPORTED;
    // GEMV row length K: 8-column chunks spread over min(32, K/8) lanes, so
    // K/8 divides 32 (short rows) or K is a multiple of 256 (long rows).
    auto width_ok = [](int K) {
        if (K % 8) return false;
        const int n = K / 8;
        return n < 32 ? (32 % n == 0) : (K % 256 == 0);
    };
    if (!width_ok(c->hidden) || !width_ok(G * c->head_dim) || c->hidden < 256 || c->hidden > MK_MAX_H)
        return MK_ERR_UNSUPPORTED;
    return MK_OK;
}

int build_geom(const mk_config* c, const Tune& tu, int grid, int ns, MkGeom& g) {
    if (!mk_geom_init(g, c->n_layers, c->hidden, c->n_q_heads, c->n_kv_heads, c->head_dim, c->ffn, c->vocab,
                      c->max_seq, grid, tu.slot, ns, tu.wb))
        return MK_ERR_INVALID_ARG;
    if (g.TRh < 2 || g.TRq < 2 || g.TRo < 2 || g.JD < 1 || g.KB < 1 || tu.slot % 16) return MK_ERR_INVALID_ARG;
    if (ns < 1 || ns > 16) return MK_ERR_INVALID_ARG;
    if (g.max_rows > 4096 || g.max_nj > 8192) return MK_ERR_UNSUPPORTED;
    if (g.CPG * g.G > MK_MAX_CPG_G) return MK_ERR_UNSUPPORTED;
    mk_smem_layout(g);
    return MK_OK;
}

void build_plans(const MkGeom& g, std::vector<MkCtaPlan>& plans, int64_t& arena) {
    plans.resize(g.nC);
    int64_t off = 0;
    for (int c = 0; c < g.nC; ++c) {
        mk_cta_plan(g, c, plans[c]);
        plans[c].stream_off = off;
        off += mk_cta_stream_bytes(g, plans[c]);
    }
    arena = off;
}

void build_maps(const MkGeom& g, const std::vector<MkCtaPlan>& plans, Maps& m) {
    const int L = g.L, H = g.H, KO = g.G * g.hd, wb = g.wb;
    m.q.assign(L, {}); m.k.assign(L, {}); m.v.assign(L, {}); m.o.assign(L, {});
    m.gate.assign(L, {}); m.up.assign(L, {}); m.down.assign(L, {}); m.down_scale.assign(L, {}); m.lm.clear();
    // rows of tiles of at most TR rows of K weights from `off` on: row i of a
    // tile of R rows at tile + i * rb (rb = the row's bytes), its scale (int8,
    // int4) at tile + R * rb + 4 i
    auto row_tiles = [&](int64_t& off, int nrows, int TR, int K, auto&& emit) {
        const int64_t rb = mk_wbytes(K, wb);
        for (int r = 0; r < nrows; r += TR) {
            const int R = std::min(TR, nrows - r);
            for (int i = 0; i < R; ++i)
                emit(r + i, off + (int64_t)i * rb, off + (int64_t)R * rb + 4LL * i);
            off += mk_row_tile_bytes(R, K, wb, 0);
        }
    };
    for (int c = 0; c < g.nC; ++c) {
        const MkCtaPlan& p = plans[c];
        for (int l = 0; l < L; ++l) {
            int64_t off = p.stream_off + (int64_t)l * p.layer_bytes;
            row_tiles(off, 2 * p.npairs, g.TRq, H, [&](int r, int64_t d, int64_t so) {
                int mat, row;
                mk_qkv_row(g, p.g, p.pair0 + r / 2, r % 2, mat, row);
                (mat == 0 ? m.q : mat == 1 ? m.k : m.v)[l].push_back(MkRowCopyQ{d, row, 0, H, so});
            });
            row_tiles(off, p.norows, g.TRo, KO, [&](int r, int64_t d, int64_t so) {
                m.o[l].push_back(MkRowCopyQ{d, (int64_t)(p.orow0 + r), p.g * KO, KO, so});
            });
            // a GU tile: n gate rows, n up rows (then for int8 / int4 their 2n
            // scales and the n W_down column scales of the same j's)
            const int64_t hb = mk_wbytes(H, wb);
            for (int j = 0; j < p.nj; j += g.JT) {
                const int n = std::min(g.JT, p.nj - j);
                const int64_t sc = off + (int64_t)2 * n * hb;
                for (int jj = 0; jj < n; ++jj) {
                    const int64_t src = p.j0 + j + jj;
                    m.gate[l].push_back(MkRowCopyQ{off + (int64_t)jj * hb, src, 0, H, sc + 4LL * jj});
                    m.up[l].push_back(MkRowCopyQ{off + (int64_t)(n + jj) * hb, src, 0, H, sc + 4LL * (n + jj)});
                    if (wb != 2) m.down_scale[l].push_back(MkScaleCopy{sc + 4LL * (2 * n + jj), src});
                }
                off += mk_row_tile_bytes(2 * n, H, wb, n);
            }
            if (p.nj > 0) m.down[l].push_back(MkColCopy{off, p.j0, p.nj});
        }
        int64_t off = p.stream_off + (int64_t)L * p.layer_bytes;
        row_tiles(off, p.nv, g.TRh, H, [&](int r, int64_t d, int64_t so) {
            m.lm.push_back(MkRowCopyQ{d, (int64_t)(p.v0 + r), 0, H, so});
        });
    }
}

// Walks every CTA's tile stream (as the kernel will) for a few positions and
// checks that every bulk copy stays inside its buffer, is 16-byte aligned and
// sized, fits a ring slot, and that the weight tiles cover each CTA's stream.
bool check_schedule(const MkGeom& g, const std::vector<MkCtaPlan>& plans, int64_t arena_bytes) {
    const uint8_t* A = reinterpret_cast<const uint8_t*>((uintptr_t)1 << 40);   // fake, aligned bases
    const uint16_t* K = reinterpret_cast<const uint16_t*>((uintptr_t)1 << 41);
    const uint16_t* Vc = reinterpret_cast<const uint16_t*>((uintptr_t)3 << 41);
    const int64_t kv_bytes = (int64_t)g.L * g.kvh * g.max_seq * g.hd * 2;
    const int poss[4] = {0, 1, g.max_seq / 2, g.max_seq - 1};
    const int nas[4] = {1, 3, (g.CPG + 1) / 2, g.CPG};   // attention CTAs per group
    for (int ci = 0; ci < 16; ++ci) {
        const int pos = poss[ci / 4], na = nas[ci % 4];
        if (pos < 0 || pos >= g.max_seq || na > g.CPG) continue;
        for (int c = 0; c < g.nC; ++c) {
            const MkCtaPlan& pl = plans[c];
            const int64_t lo = pl.stream_off, hi = pl.stream_off + mk_cta_stream_bytes(g, pl);
            int64_t wbytes = 0;
            bool ok = true;
            mk_walk_tiles(g, pl, A, K, Vc, pos, na, [&](const void* src, uint32_t bytes) {
                const uint8_t* s = reinterpret_cast<const uint8_t*>(src);
                if (bytes == 0 || bytes % 16 || (int64_t)bytes > g.slot || ((uintptr_t)s & 15)) ok = false;
                const uint8_t* kb = reinterpret_cast<const uint8_t*>(K);
                const uint8_t* vb = reinterpret_cast<const uint8_t*>(Vc);
                if (s >= kb && s < kb + kv_bytes) {
                    if (s + bytes > kb + kv_bytes) ok = false;
                } else if (s >= vb && s < vb + kv_bytes) {
                    if (s + bytes > vb + kv_bytes) ok = false;
                } else {
                    const int64_t off = s - A;
                    if (off < lo || off + bytes > hi || off + bytes > arena_bytes) ok = false;
                    wbytes += bytes;
                }
            });
            if (!ok || wbytes != (int64_t)g.L * pl.layer_bytes + mk_lm_bytes(g, pl)) return false;
        }
    }
    return true;
}

// Weight bytes one step must read: every matrix once (bf16, or int8 / int4
// codes plus one fp32 scale per row / W_down column), the norm gains and one
// embedding row (counted at 2 bytes per value).
int64_t weight_bytes_per_token(const mk_config* c, int wb) {
    const int64_t H = c->hidden, qd = (int64_t)c->n_q_heads * c->head_dim, kvd = (int64_t)c->n_kv_heads * c->head_dim;
    const int64_t F = c->ffn, V = c->vocab, L = c->n_layers;
    const int64_t mat = L * (qd * H + 2 * kvd * H + H * qd + 3 * F * H) + V * H;
    const int64_t scales = wb != 2 ? 4 * (L * (qd + 2 * kvd + H + 3 * F) + V) : 0;
    return mk_wbytes(mat, wb) + scales + 2 * (L * 2 * H + H + H);
}

}  // namespace

struct mk_ctx {
    mk_config cfg;
    Tune tune;
    MkGeom geo;
    int device = 0, sm_count = 0;
    const void* kernel = nullptr;        // the fused step without trace code
    const void* kernel_trace = nullptr;  // the same with the segment trace compiled in
    // the build whose attention runs on the tensor cores (shapes with 4 query
    // heads of 64 dims per KV group; null otherwise) and the context length
    // per CTA from which a step launches it
    const void* kernel_tc = nullptr;
    const void* kernel_tc_trace = nullptr;
    int tc_min_per_cta = MK_ATTN_TC_MIN_PER_CTA;
    int attn_build = 0;                  // debug: 0 by context length, 1 lane-parallel, 2 tensor cores
    // the length-adaptive split: A = ceil(ctx / attn_pos_per_cta) CTAs of each
    // KV group (at most all of them) run a step's attention, or attn_ctas_force
    int attn_pos_per_cta = MK_ATTN_POS_PER_CTA;
    int attn_ctas_force = 0;
    std::vector<MkCtaPlan> plans;
    int64_t arena_bytes = 0, device_bytes = 0;
    bool weights_loaded = false;
    cudaStream_t last_stream = nullptr;
    std::vector<void*> allocs;
    // device buffers
    uint8_t* arena = nullptr;
    MkCtaPlan* d_plans = nullptr;
    uint16_t *embed = nullptr, *kc = nullptr, *vc = nullptr;
    float *attn_norm = nullptr, *ffn_norm = nullptr, *final_norm = nullptr, *rope_cos = nullptr, *rope_sin = nullptr;
    uint64_t *qll = nullptr, *kvll = nullptr, *partll = nullptr;
    float *xacc = nullptr, *hidden = nullptr;
    uint32_t *cnt = nullptr, *status = nullptr, *seq = nullptr;
    unsigned long long* amax = nullptr;
    int32_t *next_token = nullptr, *tokens_dev = nullptr, *prompt_dev = nullptr;
    int32_t* stop = nullptr;             // generation stopped (mk_generate with a stop token)
    float* lgs = nullptr;                // [V] logits scratch of top-p steps
    MkTopP* tp = nullptr;                // top-p threshold-search scratch
    float top_p = 1.f;                   // nucleus mass of sampled steps (mk_set_top_p); 1 = every token
    uint32_t* status_host = nullptr;     // pinned copy of the status word (read behind generate calls)
    // debug
    int dbg_skip_cta = -1, dbg_skip_sync = -1;
    int trace_detail = 1;
    int inflight = 0, inflight_lat = 0;
    int stream_tail = 0;
    int pf_lead_tiles = -1, pf_depth = 0;  // L2 warmer (debug knobs; -1 / 0 = defaults)
    int64_t wait_limit_ns = 1000000000LL;
    unsigned long long* trace = nullptr;
    // per-operator baseline
    bool perop_enabled = false, perop_ready = false;
    MkPerOp perop{};
    // batched prefill workspace (rows of capacity pf_rows), grown on demand
    int pf_rows = 0;
    float *pf_x = nullptr, *pf_xn = nullptr, *pf_qkv = nullptr, *pf_att = nullptr, *pf_gu = nullptr, *pf_u = nullptr;
    uint16_t* pf_parts = nullptr;        // the GEMM activations' three bf16 parts (tcgen05 path)
    int prefill_gemm = 0;                // debug: 0 tcgen05 GEMMs + tensor-core attention, 1 the mma.sync GEMMs and CUDA-core attention

    template <class T>
    int dalloc(T** p, size_t bytes) {
        void* q = nullptr;
        cudaError_t e = cudaMalloc(&q, bytes ? bytes : 16);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
        allocs.push_back(q);
        device_bytes += (int64_t)bytes;
        *p = reinterpret_cast<T*>(q);
        return MK_OK;
    }
};

namespace {

MkParams base_params(const mk_ctx* c) {
    MkParams p;
    memset(&p, 0, sizeof p);
    p.geo = c->geo;
    p.eps = c->cfg.rms_eps;
    p.l2_pf_bytes = c->tune.l2pf;
    p.arena = c->arena;
    p.plans = c->d_plans;
    p.embed = c->embed;
    p.attn_norm = c->attn_norm;
    p.ffn_norm = c->ffn_norm;
    p.final_norm = c->final_norm;
    p.kc = c->kc;
    p.vc = c->vc;
    p.rope_cos = c->rope_cos;
    p.rope_sin = c->rope_sin;
    p.qll = c->qll;
    p.kvll = c->kvll;
    p.partll = c->partll;
    p.xacc = c->xacc;
    p.hidden = c->hidden;
    p.cnt = c->cnt;
    p.amax = c->amax;
    p.next_token = c->next_token;
    p.status = c->status;
    p.seq = c->seq;
    p.dbg_skip_cta = c->dbg_skip_cta;
    p.dbg_skip_sync = c->dbg_skip_sync;
    p.trace_detail = c->trace_detail;
    p.inflight = c->inflight > 0 ? c->inflight : 3;
    p.inflight_lat = c->inflight_lat > 0 ? c->inflight_lat : 1;
    p.stream_tail = c->stream_tail;
    p.pf_lead_bytes = (c->pf_lead_tiles >= 0 ? c->pf_lead_tiles : c->geo.ns) * c->geo.slot;
    p.pf_depth = c->pf_depth > 0 ? c->pf_depth : 1;
    p.wait_limit_ns = c->wait_limit_ns;
    p.trace = c->trace;
    p.out_idx = 0;
    p.top_p = 1.f;   // sampled steps set the context's value
    p.lgs = c->lgs;
    p.tp = c->tp;
    return p;
}

// The attention plan of the step at position pos: how many CTAs of each KV
// group split the positions (the length-adaptive split) and whether the
// tensor-core build runs it (from tc_min_per_cta positions per attention CTA;
// default 0: always, where it exists).
void attn_plan(const mk_ctx* c, int pos, int* A, bool* tc) {
    const int64_t ctx = (int64_t)pos + 1, cpg = c->geo.CPG;
    int64_t a = c->attn_ctas_force > 0 ? c->attn_ctas_force : (ctx + c->attn_pos_per_cta - 1) / c->attn_pos_per_cta;
    a = a < 1 ? 1 : a > cpg ? cpg : a;
    *A = (int)a;
    *tc = c->kernel_tc && (c->attn_build == 2 ||
                           (c->attn_build == 0 && ctx >= (int64_t)c->tc_min_per_cta * a));
}

// Context length from which steps launch the tensor-core attention build (-1: never).
int64_t mk_tc_min_ctx(const mk_ctx* c) {
    for (int pos = 0; pos < c->geo.max_seq; ++pos) {
        int a;
        bool tc;
        attn_plan(c, pos, &a, &tc);
        if (tc) return pos + 1;
    }
    return -1;
}

int launch_step(mk_ctx* c, MkParams& p, cudaStream_t st) {
    cudaLaunchConfig_t lc;
    memset(&lc, 0, sizeof lc);
    lc.gridDim = dim3(c->geo.nC);
    lc.blockDim = dim3(MK_BLOCK);
    lc.dynamicSmemBytes = c->geo.smem_bytes;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    void* args[] = {&p};
    // attention CTAs per group and attention build by context length
    bool tc = false;
    attn_plan(c, p.pos, &p.attn_ctas, &tc);
    const void* fn = tc ? (c->trace ? c->kernel_tc_trace : c->kernel_tc) : (c->trace ? c->kernel_trace : c->kernel);
    MK_CU(cudaLaunchKernelExC(&lc, fn, args));
    c->last_stream = st;
    return MK_OK;
}

int copy_matrix_to_device(const void* src, int on_device, size_t bytes, uint16_t* staging, const uint16_t** out,
                          cudaStream_t st) {
    if (on_device) { *out = reinterpret_cast<const uint16_t*>(src); return MK_OK; }
    MK_CU(cudaMemcpyAsync(staging, src, bytes, cudaMemcpyHostToDevice, st));
    *out = staging;
    return MK_OK;
}

template <class T>
int upload_ops(const std::vector<T>& v, T** d, size_t* cap, cudaStream_t st) {
    if (v.empty()) return MK_OK;
    if (v.size() > *cap) {
        MK_CU(cudaStreamSynchronize(st));
        if (*d) cudaFree(*d);
        *d = nullptr;
        MK_CU(cudaMalloc(reinterpret_cast<void**>(d), v.size() * sizeof(T)));
        *cap = v.size();
    }
    MK_CU(cudaMemcpyAsync(*d, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice, st));
    // the host vector must outlive the copy: callers synchronize before reusing it
    return MK_OK;
}

}  // namespace

extern "C" {

const char* mk_strerror(int code) {
    switch (code) {
        case MK_OK: return "ok";
        case MK_ERR_INVALID_ARG: return "invalid argument";
        case MK_ERR_OOM: return "out of memory";
        case MK_ERR_CUDA: return "CUDA runtime error";
        case MK_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case MK_ERR_NUMERIC: return "non-finite logit";
        case MK_ERR_STATE: return "call out of order";
        case MK_ERR_UNSUPPORTED: return "shape not supported by the kernels";
        default: return "unknown error";
    }
}

const char* mk_last_cuda_error(void) { return g_cuda_err.c_str(); }

int64_t mk_arena_bytes(const mk_config* cfg, const mk_tuning* tuning, int32_t grid_ctas) {
    if (check_shape(cfg, false) != MK_OK || grid_ctas < 1) return -1;
    if (tuning && tuning->weight_int8 && tuning->weight_int4) return -1;   // one weight form
    Tune tu = resolve_tuning(tuning);
    MkGeom g;
    if (build_geom(cfg, tu, grid_ctas, 1, g) != MK_OK) return -1;
    std::vector<MkCtaPlan> plans;
    int64_t arena = 0;
    build_plans(g, plans, arena);
    return arena;
}

int mk_relayout_host(const mk_config* cfg, const mk_tuning* tuning, int32_t grid_ctas, const mk_weights* w,
                     void* arena_out) {
    int rc = check_shape(cfg, false);
    if (rc != MK_OK) return rc;
    if (!w || !arena_out || grid_ctas < 1 || w->on_device) return MK_ERR_INVALID_ARG;
    if (!cfg->tie_embeddings && !w->lm_head) return MK_ERR_INVALID_ARG;
    Tune tu = resolve_tuning(tuning);
    if (tuning && tuning->weight_int8 && tuning->weight_int4) return MK_ERR_INVALID_ARG;
    if (tu.wb != 2) return MK_ERR_UNSUPPORTED;   // int8 / int4 streams are quantized on the device only
    MkGeom g;
    if ((rc = build_geom(cfg, tu, grid_ctas, 1, g)) != MK_OK) return rc;
    std::vector<MkCtaPlan> plans;
    int64_t arena = 0;
    build_plans(g, plans, arena);
    Maps m;
    build_maps(g, plans, m);
    uint8_t* A = reinterpret_cast<uint8_t*>(arena_out);
    memset(A, 0, (size_t)arena);
    auto rows = [&](const std::vector<MkRowCopyQ>& ops, const void* src, int64_t cols) {
        const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
        for (const MkRowCopyQ& op : ops) memcpy(A + op.dst_off, s + op.src_row * cols + op.col0, (size_t)op.ncols * 2);
    };
    const int64_t H = g.H, qd = (int64_t)g.qh * g.hd;
    for (int l = 0; l < g.L; ++l) {
        rows(m.q[l], w->wq[l], H);
        rows(m.k[l], w->wk[l], H);
        rows(m.v[l], w->wv[l], H);
        rows(m.o[l], w->wo[l], qd);
        rows(m.gate[l], w->w_gate[l], H);
        rows(m.up[l], w->w_up[l], H);
        const uint16_t* d = reinterpret_cast<const uint16_t*>(w->w_down[l]);
        for (const MkColCopy& op : m.down[l]) {
            uint16_t* dst = reinterpret_cast<uint16_t*>(A + op.dst_off);
            for (int jj = 0; jj < op.nj; ++jj)
                for (int64_t r = 0; r < H; ++r) dst[jj * H + r] = d[r * g.F + op.j0 + jj];
        }
    }
    rows(m.lm, cfg->tie_embeddings ? w->embed : w->lm_head, H);
    return MK_OK;
}

int mk_create(const mk_config* cfg, const mk_tuning* tuning, int device, mk_ctx** out) {
    if (!out) return MK_ERR_INVALID_ARG;
    *out = nullptr;
    if (tuning && tuning->weight_int8 && tuning->weight_int4) return MK_ERR_INVALID_ARG;   // one weight form
    int rc = check_shape(cfg, true, resolve_tuning(tuning).wb);
    if (rc != MK_OK) return rc;
    mk_ctx* c = new mk_ctx();
    c->cfg = *cfg;
    c->tune = resolve_tuning(tuning);
    c->device = device;
    auto fail = [&](int code) { mk_destroy(c); return code; };
    cudaError_t e = cudaSetDevice(device);
    if (e != cudaSuccess) return fail(cuda_fail(e, "cudaSetDevice"));
    int smem_optin = 0;
    if ((e = cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device)) != cudaSuccess)
        return fail(cuda_fail(e, "cudaDeviceGetAttribute"));
    const int kvh = cfg->n_kv_heads;
    int grid = c->tune.grid ? c->tune.grid : kvh * (c->sm_count / kvh);
    if (grid < kvh || grid % kvh || grid > c->sm_count) return fail(MK_ERR_INVALID_ARG);
    // ring stages: as many as requested that fit the opt-in shared memory
    int ns = std::min(c->tune.ns_req, 16);
    for (;; --ns) {
        if (ns < 1) return fail(MK_ERR_UNSUPPORTED);
        MkGeom g;
        if ((rc = build_geom(cfg, c->tune, grid, ns, g)) != MK_OK) return fail(rc);
        if (g.smem_bytes + 1024 <= smem_optin) { c->geo = g; break; }
    }
    const int wb = c->tune.wb;
    if (mk_kernel_variant(cfg->head_dim, cfg->n_q_heads / kvh, cfg->hidden, wb, false, &c->kernel,
                          &c->kernel_trace) < 0)
        return fail(MK_ERR_UNSUPPORTED);
    if (mk_kernel_variant(cfg->head_dim, cfg->n_q_heads / kvh, cfg->hidden, wb, true, &c->kernel_tc,
                          &c->kernel_tc_trace) != 1)
        c->kernel_tc = c->kernel_tc_trace = nullptr;
    // both builds of a tensor-core shape read (and append) chunk-permuted K/V rows
    c->geo.kv_swz = mk_attn_tc(cfg->head_dim, cfg->n_q_heads / kvh) ? 1 : 0;
    for (const void* k : {c->kernel, c->kernel_trace, c->kernel_tc, c->kernel_tc_trace}) {
        if (!k) continue;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, c->geo.smem_bytes)) !=
            cudaSuccess)
            return fail(cuda_fail(e, "cudaFuncSetAttribute"));
        int per_sm = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, MK_BLOCK, c->geo.smem_bytes)) !=
            cudaSuccess)
            return fail(cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor"));
        if (per_sm < 1) return fail(MK_ERR_UNSUPPORTED);
    }
    build_plans(c->geo, c->plans, c->arena_bytes);
    if (!check_schedule(c->geo, c->plans, c->arena_bytes)) return fail(MK_ERR_STATE);

    const MkGeom& g = c->geo;
    const size_t L = g.L, H = g.H, V = g.V;
    const size_t kv_elems = L * g.kvh * (size_t)g.max_seq * g.hd;
    const size_t qll_bytes = L * g.qh * (size_t)g.hd * 8, kvll_bytes = L * g.kvh * 2 * (size_t)g.hd * 8;
    const size_t partll_bytes = L * g.kvh * g.CPG * ((size_t)g.G * g.hd + 2 * g.G) * 8;
    if ((rc = c->dalloc(&c->arena, (size_t)c->arena_bytes)) ||
        (rc = c->dalloc(&c->d_plans, sizeof(MkCtaPlan) * g.nC)) ||
        (rc = c->dalloc(&c->embed, V * H * 2)) || (rc = c->dalloc(&c->kc, kv_elems * 2)) ||
        (rc = c->dalloc(&c->vc, kv_elems * 2)) || (rc = c->dalloc(&c->attn_norm, L * H * 4)) ||
        (rc = c->dalloc(&c->ffn_norm, L * H * 4)) || (rc = c->dalloc(&c->final_norm, H * 4)) ||
        (rc = c->dalloc(&c->rope_cos, (size_t)g.max_seq * (g.hd / 2) * 4)) ||
        (rc = c->dalloc(&c->rope_sin, (size_t)g.max_seq * (g.hd / 2) * 4)) ||
        (rc = c->dalloc(&c->qll, qll_bytes)) || (rc = c->dalloc(&c->kvll, kvll_bytes)) ||
        (rc = c->dalloc(&c->partll, partll_bytes)) ||
        (rc = c->dalloc(&c->xacc, 2 * 2 * L * H * 4)) || (rc = c->dalloc(&c->hidden, H * 4)) ||
        (rc = c->dalloc(&c->cnt, (size_t)mk_cnt_total(g) * 4)) || (rc = c->dalloc(&c->status, 4)) ||
        (rc = c->dalloc(&c->seq, 4)) || (rc = c->dalloc(&c->amax, 8)) || (rc = c->dalloc(&c->next_token, 4)) ||
        (rc = c->dalloc(&c->tokens_dev, (size_t)g.max_seq * 4)) ||
        (rc = c->dalloc(&c->prompt_dev, (size_t)g.max_seq * 4)) || (rc = c->dalloc(&c->stop, 4)) ||
        (rc = c->dalloc(&c->lgs, V * 4)) || (rc = c->dalloc(&c->tp, sizeof(MkTopP))))
        return fail(rc);
    if ((e = cudaHostAlloc(reinterpret_cast<void**>(&c->status_host), 4, cudaHostAllocDefault)) != cudaSuccess)
        return fail(cuda_fail(e, "cudaHostAlloc"));
    *c->status_host = 0;
    cudaStream_t st = nullptr;
    if ((e = cudaMemcpy(c->d_plans, c->plans.data(), sizeof(MkCtaPlan) * g.nC, cudaMemcpyHostToDevice)) ||
        (e = cudaMemset(c->kc, 0, kv_elems * 2)) || (e = cudaMemset(c->vc, 0, kv_elems * 2)) ||
        (e = cudaMemset(c->xacc, 0, 2 * 2 * L * H * 4)) || (e = cudaMemset(c->qll, 0, qll_bytes)) ||
        (e = cudaMemset(c->kvll, 0, kvll_bytes)) || (e = cudaMemset(c->partll, 0, partll_bytes)) || (e = cudaMemset(c->cnt, 0, (size_t)mk_cnt_total(g) * 4)) ||
        (e = cudaMemset(c->status, 0, 4)) || (e = cudaMemset(c->seq, 0, 4)) || (e = cudaMemset(c->amax, 0, 8)) ||
        (e = cudaMemset(c->next_token, 0, 4)) || (e = cudaMemset(c->tokens_dev, 0, (size_t)g.max_seq * 4)) ||
        (e = cudaMemset(c->stop, 0, 4)) || (e = cudaMemset(c->tp, 0, sizeof(MkTopP))))
        return fail(cuda_fail(e, "context init"));
    if ((e = mk_launch_rope_table(c->rope_cos, c->rope_sin, g.max_seq, g.hd, (double)cfg->rope_theta, st)) ||
        (e = cudaDeviceSynchronize()))
        return fail(cuda_fail(e, "rope table"));
    *out = c;
    return MK_OK;
}

void mk_destroy(mk_ctx* c) {
    if (!c) return;
    cudaSetDevice(c->device);
    for (void* p : c->allocs) cudaFree(p);
    for (float* p : {c->pf_x, c->pf_xn, c->pf_qkv, c->pf_att, c->pf_gu, c->pf_u})
        if (p) cudaFree(p);
    if (c->pf_parts) cudaFree(c->pf_parts);
    if (c->status_host) cudaFreeHost(c->status_host);
    for (uint16_t* p : c->perop.wqkv) cudaFree(p);
    for (uint16_t* p : c->perop.wo) cudaFree(p);
    for (uint16_t* p : c->perop.wgu) cudaFree(p);
    for (uint16_t* p : c->perop.wd) cudaFree(p);
    delete c;
}

int mk_enable_perop(mk_ctx* c, int32_t keep_rowmajor) {
    if (!c) return MK_ERR_INVALID_ARG;
    if (keep_rowmajor && c->geo.wb != 2) return MK_ERR_UNSUPPORTED;   // the per-operator kernels read bf16
    if (c->weights_loaded && keep_rowmajor && !c->perop_ready) return MK_ERR_STATE;
    c->perop_enabled = keep_rowmajor != 0;
    return MK_OK;
}

int mk_load_weights(mk_ctx* c, const mk_weights* w, void* stream) {
    if (!c || !w) return MK_ERR_INVALID_ARG;
    const mk_config& cfg = c->cfg;
    if (!w->embed || !w->final_norm || !w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo || !w->ffn_norm ||
        !w->w_gate || !w->w_up || !w->w_down)
        return MK_ERR_INVALID_ARG;
    if (cfg.tie_embeddings ? (w->lm_head != nullptr) : (w->lm_head == nullptr)) return MK_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    MK_CU(cudaSetDevice(c->device));
    const MkGeom& g = c->geo;
    const size_t H = g.H, F = g.F, V = g.V, qd = (size_t)g.qh * g.hd, kvd = (size_t)g.kvh * g.hd;
    const int on_dev = w->on_device ? 1 : 0;
    if (on_dev) {   // the device gathers copy 16-byte chunks
        auto al = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
        bool ok = al(w->embed) && (!w->lm_head || al(w->lm_head));
        for (int l = 0; l < g.L && ok; ++l)
            ok = al(w->wq[l]) && al(w->wk[l]) && al(w->wv[l]) && al(w->wo[l]) && al(w->w_gate[l]) &&
                 al(w->w_up[l]) && al(w->w_down[l]);
        if (!ok) return MK_ERR_INVALID_ARG;
    }
    Maps m;
    build_maps(g, c->plans, m);

    const bool q8 = g.wb != 2;              // int8 or int4 codes
    const int qbits = g.wb == 0 ? 4 : 8;
    const size_t max_elems = std::max({V * H, F * H, qd * H, kvd * H, H});
    uint16_t* staging = nullptr;
    if (!on_dev) MK_CU(cudaMalloc(&staging, max_elems * 2));
    MkRowCopy* d_rows = nullptr;
    MkColCopy* d_cols = nullptr;
    MkRowCopyQ* d_rowsq = nullptr;
    MkScaleCopy* d_scl = nullptr;
    size_t cap_rows = 0, cap_cols = 0, cap_rowsq = 0, cap_scl = 0;
    uint16_t* gain_tmp = nullptr;
    int8_t* q_tmp = nullptr;     // int8 streams: one matrix's codes and scales
    float* s_tmp = nullptr;
    int rc = MK_OK;
    auto cleanup = [&]() {
        cudaStreamSynchronize(st);
        if (staging) cudaFree(staging);
        if (d_rows) cudaFree(d_rows);
        if (d_cols) cudaFree(d_cols);
        if (d_rowsq) cudaFree(d_rowsq);
        if (d_scl) cudaFree(d_scl);
        if (gain_tmp) cudaFree(gain_tmp);
        if (q_tmp) cudaFree(q_tmp);
        if (s_tmp) cudaFree(s_tmp);
    };
#define MK_TRY(x)                       \
    do {                                \
        rc = (x);                       \
        if (rc != MK_OK) { cleanup(); return rc; } \
    } while (0)
#define MK_TRYCU(x)                     \
    do {                                \
        cudaError_t e_ = (x);           \
        if (e_ != cudaSuccess) { rc = cuda_fail(e_, #x); cleanup(); return rc; } \
    } while (0)

    if (q8) {
        cudaError_t e = cudaMalloc(&q_tmp, max_elems);
        if (e == cudaSuccess) e = cudaMalloc(&s_tmp, std::max({V, F, H, qd, kvd}) * 4);
        if (e != cudaSuccess) { rc = cuda_fail(e, "int8/int4 staging"); cleanup(); return rc; }
    }
    // bf16 streams copy the rows; int8 / int4 streams quantize the matrix (per
    // row) and copy (int4: pack) codes and row scales
    auto gather_rows = [&](const std::vector<MkRowCopyQ>& ops, const void* src, size_t rows, size_t cols) -> int {
        const uint16_t* d = nullptr;
        int r = copy_matrix_to_device(src, on_dev, rows * cols * 2, staging, &d, st);
        if (r != MK_OK) return r;
        cudaError_t e;
        if (q8) {
            e = mk_launch_quantize(d, (int64_t)rows, (int64_t)cols, 0, qbits, q_tmp, s_tmp, st);
            if (e != cudaSuccess) return cuda_fail(e, "quantize rows");
            r = upload_ops(ops, &d_rowsq, &cap_rowsq, st);
            if (r != MK_OK) return r;
            e = qbits == 4
                    ? mk_launch_relayout_rows_q4(c->arena, q_tmp, (int64_t)cols, s_tmp, d_rowsq, (int)ops.size(), st)
                    : mk_launch_relayout_rows_q8(c->arena, q_tmp, (int64_t)cols, s_tmp, d_rowsq, (int)ops.size(), st);
        } else {
            const std::vector<MkRowCopy> plain = plain_rows(ops);
            r = upload_ops(plain, &d_rows, &cap_rows, st);
            if (r != MK_OK) return r;
            e = mk_launch_relayout_rows(c->arena, d, (int64_t)cols, d_rows, (int)ops.size(), st);
            if (e == cudaSuccess) e = cudaStreamSynchronize(st);   // `plain` must outlive its copy
        }
        if (e != cudaSuccess) return cuda_fail(e, "relayout rows");
        e = cudaStreamSynchronize(st);   // staging and the op buffer are reused by the next matrix
        return e == cudaSuccess ? MK_OK : cuda_fail(e, "relayout rows sync");
    };
    // per-operator copies (plain row-major) of the same weights, when enabled
    auto keep_rowmajor = [&](uint16_t** dst, const void* src, size_t elems, size_t dst_off_elems) -> int {
        cudaError_t e = cudaMemcpyAsync(*dst + dst_off_elems, src, elems * 2, cudaMemcpyDefault, st);
        return e == cudaSuccess ? MK_OK : cuda_fail(e, "row-major copy");
    };
    if (c->perop_enabled && !c->perop_ready) {
        MkPerOp& P = c->perop;
        P.wqkv.assign(g.L, nullptr); P.wo.assign(g.L, nullptr); P.wgu.assign(g.L, nullptr); P.wd.assign(g.L, nullptr);
        for (int l = 0; l < g.L; ++l) {
            MK_TRYCU(cudaMalloc(&P.wqkv[l], (qd + 2 * kvd) * H * 2));
            MK_TRYCU(cudaMalloc(&P.wo[l], H * qd * 2));
            MK_TRYCU(cudaMalloc(&P.wgu[l], 2 * F * H * 2));
            MK_TRYCU(cudaMalloc(&P.wd[l], H * F * 2));
        }
    }

    for (int l = 0; l < g.L; ++l) {
        MK_TRY(gather_rows(m.q[l], w->wq[l], qd, H));
        MK_TRY(gather_rows(m.k[l], w->wk[l], kvd, H));
        MK_TRY(gather_rows(m.v[l], w->wv[l], kvd, H));
        MK_TRY(gather_rows(m.o[l], w->wo[l], H, qd));
        MK_TRY(gather_rows(m.gate[l], w->w_gate[l], F, H));
        MK_TRY(gather_rows(m.up[l], w->w_up[l], F, H));
        {
            const uint16_t* d = nullptr;
            MK_TRY(copy_matrix_to_device(w->w_down[l], on_dev, H * F * 2, staging, &d, st));
            MK_TRY(upload_ops(m.down[l], &d_cols, &cap_cols, st));
            if (q8) {   // per-column scales, kept in the GU tiles of the same j's
                MK_TRYCU(mk_launch_quantize(d, (int64_t)H, (int64_t)F, 1, qbits, q_tmp, s_tmp, st));
                if (qbits == 4)
                    MK_TRYCU(mk_launch_relayout_cols_q4(c->arena, q_tmp, (int)H, (int)F, d_cols,
                                                        (int)m.down[l].size(), st));
                else
                    MK_TRYCU(mk_launch_relayout_cols_q8(c->arena, q_tmp, (int)H, (int)F, d_cols,
                                                        (int)m.down[l].size(), st));
                MK_TRY(upload_ops(m.down_scale[l], &d_scl, &cap_scl, st));
                MK_TRYCU(mk_launch_scatter_scales(c->arena, s_tmp, d_scl, (int)m.down_scale[l].size(), st));
            } else {
                MK_TRYCU(mk_launch_relayout_cols(c->arena, d, (int)H, (int)F, d_cols, (int)m.down[l].size(), st));
            }
            MK_TRYCU(cudaStreamSynchronize(st));
        }
        if (c->perop_enabled && !c->perop_ready) {
            MkPerOp& P = c->perop;
            MK_TRY(keep_rowmajor(&P.wqkv[l], w->wq[l], qd * H, 0));
            MK_TRY(keep_rowmajor(&P.wqkv[l], w->wk[l], kvd * H, qd * H));
            MK_TRY(keep_rowmajor(&P.wqkv[l], w->wv[l], kvd * H, (qd + kvd) * H));
            MK_TRY(keep_rowmajor(&P.wo[l], w->wo[l], H * qd, 0));
            MK_TRY(keep_rowmajor(&P.wgu[l], w->w_gate[l], F * H, 0));
            MK_TRY(keep_rowmajor(&P.wgu[l], w->w_up[l], F * H, F * H));
            MK_TRY(keep_rowmajor(&P.wd[l], w->w_down[l], H * F, 0));
            MK_TRYCU(cudaStreamSynchronize(st));
        }
    }
    MK_TRY(gather_rows(m.lm, cfg.tie_embeddings ? w->embed : w->lm_head, V, H));
    MK_TRYCU(cudaMemcpyAsync(c->embed, w->embed, V * H * 2, cudaMemcpyDefault, st));
    // norm gains: bf16 -> fp32 on the device
    MK_TRYCU(cudaMalloc(&gain_tmp, H * 2));
    auto gain = [&](const void* src, float* dst) -> int {
        cudaError_t e = cudaMemcpyAsync(gain_tmp, src, H * 2, cudaMemcpyDefault, st);
        if (e == cudaSuccess) e = mk_launch_bf16_to_f32(gain_tmp, dst, (int64_t)H, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        return e == cudaSuccess ? MK_OK : cuda_fail(e, "norm gains");
    };
    for (int l = 0; l < g.L; ++l) {
        MK_TRY(gain(w->attn_norm[l], c->attn_norm + (size_t)l * H));
        MK_TRY(gain(w->ffn_norm[l], c->ffn_norm + (size_t)l * H));
    }
    MK_TRY(gain(w->final_norm, c->final_norm));
    if (c->perop_enabled && !c->perop_ready) {
        MkPerOp& P = c->perop;
        P.L = g.L; P.H = g.H; P.qh = g.qh; P.kvh = g.kvh; P.hd = g.hd; P.F = g.F; P.V = g.V; P.max_seq = g.max_seq;
        P.eps = cfg.rms_eps;
        P.attn_chunk = 1024;
        P.amax_blocks = 256;
        P.embed = c->embed;
        if (cfg.tie_embeddings) {
            P.lm = c->embed;
        } else {
            uint16_t* lm = nullptr;
            MK_TRYCU(cudaMalloc(&lm, V * H * 2));
            c->allocs.push_back(lm);
            MK_TRYCU(cudaMemcpyAsync(lm, w->lm_head, V * H * 2, cudaMemcpyDefault, st));
            P.lm = lm;
        }
        P.attn_norm = c->attn_norm; P.ffn_norm = c->ffn_norm; P.final_norm = c->final_norm;
        P.rope_cos = c->rope_cos; P.rope_sin = c->rope_sin; P.kc = c->kc; P.vc = c->vc; P.kv_swz = c->geo.kv_swz;
        const size_t nsplit_max = ((size_t)g.max_seq + P.attn_chunk - 1) / P.attn_chunk;
        MK_TRY(c->dalloc(&P.x, H * 4)); MK_TRY(c->dalloc(&P.xn, H * 4));
        MK_TRY(c->dalloc(&P.qkv, (qd + 2 * kvd) * 4)); MK_TRY(c->dalloc(&P.attn, qd * 4));
        MK_TRY(c->dalloc(&P.u, F * 4));
        P.hidden = c->hidden;   // mk_get_hidden reads the same buffer for both paths
        MK_TRY(c->dalloc(&P.pml, (size_t)g.qh * nsplit_max * 2 * 4));
        MK_TRY(c->dalloc(&P.pacc, (size_t)g.qh * nsplit_max * g.hd * 4));
        MK_TRY(c->dalloc(&P.logits_tmp, V * 4));
        MK_TRY(c->dalloc(&P.amax_part, (size_t)P.amax_blocks * 8));
        P.next_token = c->next_token;
        P.status = c->status;
        const int smem_need = (int)std::max({H, F, qd, (size_t)(g.hd + P.attn_chunk)}) * 4;
        MK_TRYCU(mk_perop_prepare(smem_need));
        c->perop_ready = true;
    }
    cleanup();
    c->weights_loaded = true;
    c->last_stream = st;
#undef MK_TRY
#undef MK_TRYCU
    return MK_OK;
}

// A device buffer that lives for one call.
struct MkDevTmp {
    void* p = nullptr;
    ~MkDevTmp() { if (p) cudaFree(p); }
};

int mk_set_kv(mk_ctx* c, int32_t layer, const void* k, const void* v, int32_t n_pos, void* stream) {
    if (!c || !k || !v || layer < 0 || layer >= c->geo.L || n_pos < 0 || n_pos > c->geo.max_seq)
        return MK_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    MK_CU(cudaSetDevice(c->device));
    const MkGeom& g = c->geo;
    const size_t row = (size_t)n_pos * g.hd * 2;
    const size_t lay = ((size_t)layer * g.kvh * g.max_seq) * g.hd;
    if (g.kv_swz) {
        // rows chunk-permuted in the cache: stage the plain rows on the device, then permute
        if (n_pos == 0) return MK_OK;
        MkDevTmp tmp;
        const size_t bytes = row * g.kvh;
        MK_CU(cudaMalloc(&tmp.p, 2 * bytes));
        uint16_t* tk = static_cast<uint16_t*>(tmp.p);
        uint16_t* tv = tk + bytes / 2;
        MK_CU(cudaMemcpyAsync(tk, k, bytes, cudaMemcpyDefault, st));
        MK_CU(cudaMemcpyAsync(tv, v, bytes, cudaMemcpyDefault, st));
        MK_CU(mk_launch_kv_rows(tk, c->kc + lay, g.kvh, n_pos, 0, g.max_seq, g.hd, 1, 1, st));
        MK_CU(mk_launch_kv_rows(tv, c->vc + lay, g.kvh, n_pos, 0, g.max_seq, g.hd, 1, 1, st));
        MK_CU(cudaStreamSynchronize(st));
        return MK_OK;
    }
    for (int h = 0; h < g.kvh; ++h) {
        const size_t dst = lay + ((size_t)h * g.max_seq) * g.hd;
        MK_CU(cudaMemcpyAsync(c->kc + dst, (const uint8_t*)k + h * row, row, cudaMemcpyDefault, st));
        MK_CU(cudaMemcpyAsync(c->vc + dst, (const uint8_t*)v + h * row, row, cudaMemcpyDefault, st));
    }
    MK_CU(cudaStreamSynchronize(st));
    return MK_OK;
}

int mk_read_arena(mk_ctx* c, int64_t offset, int64_t bytes, void* out, void* stream) {
    if (!c || !out || offset < 0 || bytes < 0 || offset > c->arena_bytes || bytes > c->arena_bytes - offset)
        return MK_ERR_INVALID_ARG;
    if (!c->weights_loaded) return MK_ERR_STATE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    MK_CU(cudaSetDevice(c->device));
    if (bytes > 0) MK_CU(cudaMemcpyAsync(out, c->arena + offset, (size_t)bytes, cudaMemcpyDefault, st));
    MK_CU(cudaStreamSynchronize(st));
    return MK_OK;
}

int mk_get_kv(mk_ctx* c, int32_t layer, int32_t pos0, int32_t n_pos, void* k_out, void* v_out, void* stream) {
    if (!c || !k_out || !v_out || layer < 0 || layer >= c->geo.L || pos0 < 0 || n_pos < 0 ||
        (int64_t)pos0 + n_pos > c->geo.max_seq)
        return MK_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    MK_CU(cudaSetDevice(c->device));
    const MkGeom& g = c->geo;
    const size_t row = (size_t)n_pos * g.hd * 2;
    const size_t lay = ((size_t)layer * g.kvh * g.max_seq) * g.hd;
    if (g.kv_swz) {
        if (n_pos == 0) return MK_OK;
        MkDevTmp tmp;
        const size_t bytes = row * g.kvh;
        MK_CU(cudaMalloc(&tmp.p, 2 * bytes));
        uint16_t* tk = static_cast<uint16_t*>(tmp.p);
        uint16_t* tv = tk + bytes / 2;
        MK_CU(mk_launch_kv_rows(tk, c->kc + lay, g.kvh, n_pos, pos0, g.max_seq, g.hd, 1, 0, st));
        MK_CU(mk_launch_kv_rows(tv, c->vc + lay, g.kvh, n_pos, pos0, g.max_seq, g.hd, 1, 0, st));
        MK_CU(cudaMemcpyAsync(k_out, tk, bytes, cudaMemcpyDefault, st));
        MK_CU(cudaMemcpyAsync(v_out, tv, bytes, cudaMemcpyDefault, st));
        MK_CU(cudaStreamSynchronize(st));
        return MK_OK;
    }
    for (int h = 0; h < g.kvh; ++h) {
        const size_t src = lay + ((size_t)h * g.max_seq + pos0) * g.hd;
        MK_CU(cudaMemcpyAsync((uint8_t*)k_out + h * row, c->kc + src, row, cudaMemcpyDefault, st));
        MK_CU(cudaMemcpyAsync((uint8_t*)v_out + h * row, c->vc + src, row, cudaMemcpyDefault, st));
    }
    MK_CU(cudaStreamSynchronize(st));
    return MK_OK;
}

int mk_decode_step(mk_ctx* c, int32_t token, int32_t pos, float* logits_out, void* stream) {
    if (!c) return MK_ERR_INVALID_ARG;
    if (!c->weights_loaded) return MK_ERR_STATE;
    if (token < 0 || token >= c->geo.V || pos < 0 || pos >= c->geo.max_seq) return MK_ERR_INVALID_ARG;
    MkParams p = base_params(c);
    p.pos = pos;
    p.token = token;
    p.token_ptr = nullptr;
    p.logits = logits_out;
    p.tokens_out = nullptr;
    return launch_step(c, p, reinterpret_cast<cudaStream_t>(stream));
}

int mk_decode_step_greedy(mk_ctx* c, int32_t pos, float* logits_out, void* stream) {
    if (!c) return MK_ERR_INVALID_ARG;
    if (!c->weights_loaded) return MK_ERR_STATE;
    if (pos < 0 || pos >= c->geo.max_seq) return MK_ERR_INVALID_ARG;
    MkParams p = base_params(c);
    p.pos = pos;
    p.token_ptr = c->next_token;
    p.logits = logits_out;
    p.tokens_out = nullptr;
    return launch_step(c, p, reinterpret_cast<cudaStream_t>(stream));
}

static int sync_status(mk_ctx* c, cudaStream_t st, int* dev_rc);

int mk_generate_greedy(mk_ctx* c, const int32_t* prompt, int32_t n_prompt, int32_t start_pos, int32_t n_new,
                       int32_t* out_tokens, void* stream) {
    if (!c || !prompt || !out_tokens || n_prompt < 1 || n_new < 1 || start_pos < 0) return MK_ERR_INVALID_ARG;
    if (!c->weights_loaded) return MK_ERR_STATE;
    const int64_t steps = (int64_t)n_prompt + n_new - 1;
    if (start_pos + steps > c->geo.max_seq) return MK_ERR_INVALID_ARG;
    for (int i = 0; i < n_prompt; ++i)
        if (prompt[i] < 0 || prompt[i] >= c->geo.V) return MK_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    MK_CU(cudaMemcpyAsync(c->prompt_dev, prompt, (size_t)n_prompt * 4, cudaMemcpyHostToDevice, st));
    for (int64_t k = 0; k < steps; ++k) {
        MkParams p = base_params(c);
        p.pos = (int32_t)(start_pos + k);
        p.token = 0;
        p.token_ptr = (k < n_prompt) ? c->prompt_dev + k : c->next_token;
        p.logits = nullptr;
        p.tokens_out = (k >= n_prompt - 1) ? c->tokens_dev : nullptr;
        p.out_idx = (int32_t)(k - (n_prompt - 1));
        int rc = launch_step(c, p, st);
        if (rc != MK_OK) return rc;
    }
    MK_CU(cudaMemcpyAsync(out_tokens, c->tokens_dev, (size_t)n_new * 4, cudaMemcpyDeviceToHost, st));
    int dev = MK_OK;
    const int rc = sync_status(c, st, &dev);
    return rc != MK_OK ? rc : dev;
}

int mk_decode_step_sample(mk_ctx* c, int32_t token, int32_t pos, float temperature, uint64_t seed,
                          float* logits_out, void* stream) {
    if (!c) return MK_ERR_INVALID_ARG;
    if (!c->weights_loaded) return MK_ERR_STATE;
    if (token < -1 || token >= c->geo.V || pos < 0 || pos >= c->geo.max_seq || !(temperature == temperature))
        return MK_ERR_INVALID_ARG;
    MkParams p = base_params(c);
    p.pos = pos;
    p.token = token < 0 ? 0 : token;
    p.token_ptr = token < 0 ? c->next_token : nullptr;
    p.logits = logits_out;
    p.tokens_out = nullptr;
    p.inv_temp = temperature > 0.f ? 1.0f / temperature : 0.f;
    p.top_p = c->top_p;
    p.seed = seed;
    return launch_step(c, p, reinterpret_cast<cudaStream_t>(stream));
}

int mk_generate(mk_ctx* c, const int32_t* prompt, int32_t n_prompt, int32_t start_pos, int32_t n_new,
                float temperature, uint64_t seed, int32_t eos_id, int32_t* out_tokens, int32_t* n_out, void* stream) {
    if (!c || !prompt || !out_tokens || n_prompt < 1 || n_new < 1 || start_pos < 0 || !(temperature == temperature))
        return MK_ERR_INVALID_ARG;
    if (!c->weights_loaded) return MK_ERR_STATE;
    const int64_t steps = (int64_t)n_prompt + n_new - 1;
    if (start_pos + steps > c->geo.max_seq) return MK_ERR_INVALID_ARG;
    for (int i = 0; i < n_prompt; ++i)
        if (prompt[i] < 0 || prompt[i] >= c->geo.V) return MK_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    MK_CU(cudaMemcpyAsync(c->prompt_dev, prompt, (size_t)n_prompt * 4, cudaMemcpyHostToDevice, st));
    MK_CU(cudaMemsetAsync(c->stop, 0, 4, st));
    const float inv_temp = temperature > 0.f ? 1.0f / temperature : 0.f;
    for (int64_t k = 0; k < steps; ++k) {
        MkParams p = base_params(c);
        p.pos = (int32_t)(start_pos + k);
        p.token = 0;
        p.token_ptr = (k < n_prompt) ? c->prompt_dev + k : c->next_token;
        p.logits = nullptr;
        p.tokens_out = (k >= n_prompt - 1) ? c->tokens_dev : nullptr;
        p.out_idx = (int32_t)(k - (n_prompt - 1));
        p.inv_temp = inv_temp;
        p.top_p = c->top_p;
        p.seed = seed;
        p.eos_id = eos_id;
        p.stop = eos_id >= 0 ? c->stop : nullptr;
        int rc = launch_step(c, p, st);
        if (rc != MK_OK) return rc;
    }
    MK_CU(cudaMemcpyAsync(out_tokens, c->tokens_dev, (size_t)n_new * 4, cudaMemcpyDeviceToHost, st));
    int dev = MK_OK;
    const int rc = sync_status(c, st, &dev);
    if (rc != MK_OK) return rc;
    // the tokens up to and including the first stop token; the launches after it returned at once
    int32_t n = n_new;
    if (eos_id >= 0)
        for (int32_t i = 0; i < n_new; ++i)
            if (out_tokens[i] == eos_id) { n = i + 1; break; }
    for (int32_t i = n; i < n_new; ++i) out_tokens[i] = -1;
    if (n_out) *n_out = n;
    return dev;
}

int mk_set_top_p(mk_ctx* c, float top_p) {
    if (!c || !(top_p > 0.f) || !(top_p <= 1.f)) return MK_ERR_INVALID_ARG;
    c->top_p = top_p;
    return MK_OK;
}

int mk_get_hidden(mk_ctx* c, float* out, void* stream) {
    if (!c || !out) return MK_ERR_INVALID_ARG;
    MK_CU(cudaMemcpyAsync(out, c->hidden, (size_t)c->geo.H * 4, cudaMemcpyDeviceToDevice,
                          reinterpret_cast<cudaStream_t>(stream)));
    return MK_OK;
}

int mk_get_argmax(mk_ctx* c, int32_t* out, void* stream) {
    if (!c || !out) return MK_ERR_INVALID_ARG;
    MK_CU(cudaMemcpyAsync(out, c->next_token, 4, cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)));
    return MK_OK;
}

// The error a device status word stands for.
static int status_code(uint32_t st) {
    if (st & (MK_ST_TIMEOUT | MK_ST_SCHEDULE)) return MK_ERR_DEVICE_TIMEOUT;
    if (st & MK_ST_NUMERIC) return MK_ERR_NUMERIC;
    if (st & MK_ST_BADTOKEN) return MK_ERR_INVALID_ARG;
    return MK_OK;
}

int mk_status(mk_ctx* c) {
    if (!c) return MK_ERR_INVALID_ARG;
    MK_CU(cudaSetDevice(c->device));
    MK_CU(cudaStreamSynchronize(c->last_stream));
    uint32_t st = 0;
    MK_CU(cudaMemcpy(&st, c->status, 4, cudaMemcpyDeviceToHost));
    MK_CU(cudaMemset(c->status, 0, 4));
    return status_code(st);
}

// mk_status for the generate calls: the status word is copied to pinned host
// memory behind the work already queued on st, so one synchronization covers
// the tokens and the status; the word is cleared only when it is set.  The
// return value is the CUDA outcome (the queued work is complete when it is
// MK_OK); *dev_rc receives the device status as mk_status reports it.
static int sync_status(mk_ctx* c, cudaStream_t st, int* dev_rc) {
    *dev_rc = MK_OK;
    MK_CU(cudaMemcpyAsync(c->status_host, c->status, 4, cudaMemcpyDeviceToHost, st));
    MK_CU(cudaStreamSynchronize(st));
    const uint32_t v = *c->status_host;
    if (v == 0) return MK_OK;
    MK_CU(cudaMemsetAsync(c->status, 0, 4, st));
    MK_CU(cudaStreamSynchronize(st));
    *dev_rc = status_code(v);
    return MK_OK;
}

int mk_decode_step_perop(mk_ctx* c, int32_t token, int32_t pos, float* logits_out, void* stream,
                         int32_t* n_launches) {
    if (!c) return MK_ERR_INVALID_ARG;
    if (!c->weights_loaded || !c->perop_ready) return MK_ERR_STATE;
    if (token < 0 || token >= c->geo.V || pos < 0 || pos >= c->geo.max_seq) return MK_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    const int n = mk_perop_step(c->perop, token, nullptr, pos, logits_out, st, &e);
    if (e != cudaSuccess) return cuda_fail(e, "per-operator step");
    if (n_launches) *n_launches = n;
    c->last_stream = st;
    return MK_OK;
}

int mk_prefill(mk_ctx* c, const int32_t* tokens, int32_t n, int32_t start_pos, float* logits_out, void* stream) {
    if (!c || !tokens || n < 1 || start_pos < 0) return MK_ERR_INVALID_ARG;
    if (c->geo.wb != 2) return MK_ERR_UNSUPPORTED;   // the prefill GEMMs read the bf16 row-major copies
    if (!c->weights_loaded || !c->perop_ready) return MK_ERR_STATE;
    const MkGeom& g = c->geo;
    if ((int64_t)start_pos + n > g.max_seq) return MK_ERR_INVALID_ARG;
    if (g.F % 8 || g.H % 8) return MK_ERR_UNSUPPORTED;   // 16-byte weight pieces along K
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= g.V) return MK_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    MK_CU(cudaSetDevice(c->device));
    const size_t H = g.H, F = g.F, nqkv = (size_t)(g.qh + 2 * g.kvh) * g.hd, qd = (size_t)g.qh * g.hd;
    if (n > c->pf_rows) {   // grow the workspace (the buffers of a shorter prompt are freed first)
        MK_CU(cudaStreamSynchronize(st));
        if (c->pf_rows == 0) MK_CU(mk_prefill_prepare());
        for (float** p : {&c->pf_x, &c->pf_xn, &c->pf_qkv, &c->pf_att, &c->pf_gu, &c->pf_u})
            if (*p) { cudaFree(*p); *p = nullptr; }
        if (c->pf_parts) { cudaFree(c->pf_parts); c->pf_parts = nullptr; }
        c->pf_rows = 0;
        const size_t rows = (size_t)n;
        MK_CU(cudaMalloc(&c->pf_x, rows * H * 4));
        MK_CU(cudaMalloc(&c->pf_xn, rows * H * 4));
        MK_CU(cudaMalloc(&c->pf_qkv, rows * nqkv * 4));
        MK_CU(cudaMalloc(&c->pf_att, rows * qd * 4));
        MK_CU(cudaMalloc(&c->pf_gu, rows * 2 * F * 4));
        MK_CU(cudaMalloc(&c->pf_u, rows * F * 4));
        // [3][rows rounded up to 128][widest K]: the longest K a GEMM reads is H, F or qh*hd
        const size_t mp = (rows + 127) / 128 * 128, kmax = std::max({H, F, qd});
        MK_CU(cudaMalloc(&c->pf_parts, 3 * mp * kmax * 2));
        c->pf_rows = n;
    }
    MK_CU(cudaMemcpyAsync(c->prompt_dev, tokens, (size_t)n * 4, cudaMemcpyHostToDevice, st));
    const MkPerOp& P = c->perop;
    MkPrefillArgs a{};
    a.L = g.L; a.H = g.H; a.qh = g.qh; a.kvh = g.kvh; a.hd = g.hd; a.F = g.F; a.V = g.V; a.max_seq = g.max_seq;
    a.eps = c->cfg.rms_eps;
    a.n = n; a.start = start_pos; a.swz = g.kv_swz;
    a.tokens = c->prompt_dev;
    std::vector<const uint16_t*> wqkv(P.wqkv.begin(), P.wqkv.end()), wo(P.wo.begin(), P.wo.end()),
        wgu(P.wgu.begin(), P.wgu.end()), wd(P.wd.begin(), P.wd.end());
    a.wqkv = wqkv.data(); a.wo = wo.data(); a.wgu = wgu.data(); a.wd = wd.data();
    a.embed = P.embed; a.lm = P.lm;
    a.attn_norm = c->attn_norm; a.ffn_norm = c->ffn_norm; a.final_norm = c->final_norm;
    a.rope_cos = c->rope_cos; a.rope_sin = c->rope_sin; a.kc = c->kc; a.vc = c->vc;
    a.x = c->pf_x; a.xn = c->pf_xn; a.qkv = c->pf_qkv; a.att = c->pf_att; a.gu = c->pf_gu; a.u = c->pf_u;
    // tcgen05 GEMMs and the tensor-core attention (which writes the O-proj input's parts) go together
    const bool tc = c->prefill_gemm == 0 && g.G <= 8;
    a.parts = tc ? c->pf_parts : nullptr;
    a.parts_rows = c->pf_rows;
    a.attn_tc = tc ? 1 : 0;
    a.hidden = c->hidden;
    a.logits = logits_out ? logits_out : P.logits_tmp;
    a.amax_part = P.amax_part; a.amax_blocks = P.amax_blocks;
    a.next_token = c->next_token; a.status = c->status;
    cudaError_t e = cudaSuccess;
    mk_prefill_launch(a, st, &e);
    if (e != cudaSuccess) return cuda_fail(e, "prefill");
    c->last_stream = st;
    return MK_OK;
}

int mk_get_info(const mk_ctx* c, mk_info* o) {
    if (!c || !o) return MK_ERR_INVALID_ARG;
    memset(o, 0, sizeof *o);
    o->grid_ctas = c->geo.nC;
    o->ctas_per_group = c->geo.CPG;
    o->block_threads = MK_BLOCK;
    o->ring_stages = c->geo.ns;
    o->slot_bytes = c->geo.slot;
    o->smem_bytes = c->geo.smem_bytes;
    o->sm_count = c->sm_count;
    o->l2_prefetch_bytes = c->tune.l2pf;
    o->arena_bytes = c->arena_bytes;
    o->weight_bytes_per_token = weight_bytes_per_token(&c->cfg, c->geo.wb);
    o->kv_bytes_per_position = (int64_t)2 * c->geo.L * c->geo.kvh * c->geo.hd * 2;
    o->device_bytes = c->device_bytes;
    o->attn_tc = c->kernel_tc ? 1 : 0;
    o->attn_tc_min_ctx = c->kernel_tc ? (int32_t)mk_tc_min_ctx(c) : -1;
    o->attn_pos_per_cta = c->attn_ctas_force > 0 ? 0 : c->attn_pos_per_cta;
    o->weight_int8 = c->geo.wb == 1 ? 1 : 0;
    o->weight_int4 = c->geo.wb == 0 ? 1 : 0;
    return MK_OK;
}

int mk_set_debug(mk_ctx* c, int32_t knob, int64_t value) {
    if (!c) return MK_ERR_INVALID_ARG;
    if (knob == MK_DBG_SKIP_ARRIVAL) {
        if (value < 0) { c->dbg_skip_cta = -1; c->dbg_skip_sync = -1; }
        else { c->dbg_skip_cta = (int)(value >> 16); c->dbg_skip_sync = (int)(value & 0xFFFF); }
        return MK_OK;
    }
    if (knob == MK_DBG_TRACE) {
        if (value != 0 && c->geo.L > MK_TRACE_MAX_LAYERS) return MK_ERR_UNSUPPORTED;
        c->trace = reinterpret_cast<unsigned long long*>((uintptr_t)value);
        return MK_OK;
    }
    if (knob == MK_DBG_INFLIGHT || knob == MK_DBG_INFLIGHT_LAT) {
        if (value < 0 || value > 16) return MK_ERR_INVALID_ARG;
        (knob == MK_DBG_INFLIGHT ? c->inflight : c->inflight_lat) = (int)value;
        return MK_OK;
    }
    if (knob == MK_DBG_PF_LEAD) {
        if (value < -1 || value > 64) return MK_ERR_INVALID_ARG;
        c->pf_lead_tiles = (int)value;
        return MK_OK;
    }
    if (knob == MK_DBG_PF_DEPTH) {
        if (value < 0 || value > 2) return MK_ERR_INVALID_ARG;
        c->pf_depth = (int)value;
        return MK_OK;
    }
    if (knob == MK_DBG_TRACE_DETAIL) {
        if (value < 0 || value > 2) return MK_ERR_INVALID_ARG;
        c->trace_detail = (int)value;
        return MK_OK;
    }
    if (knob == MK_DBG_ATTN_BUILD) {
        if (value < 0 || value > 2 || (value == 2 && !c->kernel_tc)) return MK_ERR_INVALID_ARG;
        c->attn_build = (int)value;
        return MK_OK;
    }
    if (knob == MK_DBG_PREFILL_GEMM) {
        if (value < 0 || value > 1) return MK_ERR_INVALID_ARG;
        c->prefill_gemm = (int)value;
        return MK_OK;
    }
    if (knob == MK_DBG_STREAM_TAIL) {
        if (value < 0 || value > 2) return MK_ERR_INVALID_ARG;
        c->stream_tail = (int)value;
        return MK_OK;
    }
    if (knob == MK_DBG_ATTN_CTAS) {
        if (value < 0 || value > c->geo.CPG) return MK_ERR_INVALID_ARG;
        c->attn_ctas_force = (int)value;
        return MK_OK;
    }
    if (knob == MK_DBG_ATTN_POS_PER_CTA) {
        if (value < 1 || value > (int64_t)c->geo.max_seq) return MK_ERR_INVALID_ARG;
        c->attn_pos_per_cta = (int)value;
        return MK_OK;
    }
    if (knob == MK_DBG_ATTN_TC_MIN) {
        if (value < 0 || value > (int64_t)c->geo.max_seq) return MK_ERR_INVALID_ARG;
        c->tc_min_per_cta = (int)value;
        return MK_OK;
    }
    if (knob == MK_DBG_WAIT_LIMIT_NS) {
        if (value < 1000) return MK_ERR_INVALID_ARG;
        c->wait_limit_ns = value;
        return MK_OK;
    }
    return MK_ERR_INVALID_ARG;
}

}  // extern "C"
