// mk_internal.h - layout and launch description shared by the host runtime and
// the decode megakernel.  Nothing here is part of the public ABI.
//
// Weight arena layout (the offline re-layout, "lay weights out in memory-access
// order ahead of time", cloud.baidu.com/article/9434380, section 9).
//
//   nC  = CTAs of the persistent grid, kvh | nC, CPG = nC / kvh CTAs per KV group
//   G   = qh / kvh query heads per KV group, hd2 = hd / 2
//   CTA c belongs to KV group g = c / CPG and has index i = c % CPG in it.
//   split(n, parts, k) = [floor(k n / parts), floor((k+1) n / parts))
//
// Each CTA owns one contiguous byte stream (256-byte aligned start) holding
// every weight tile it reads during one decode step, in consumption order:
//   for layer l:
//     QKV : pairs p in split(NP, CPG, i), NP = (G + 2) * hd2.  Pair p is head
//           slot s = p / hd2 (s < G: query head g*G + s; s == G: key head g;
//           s == G + 1: value head g) and dim d = p % hd2; it is stored as the
//           two rows (d, d + hd2) of that head, each H bf16, so a RoPE pair
//           never leaves the CTA.
//     O   : rows r in split(H, CPG, i) of W_o, columns [g*G*hd, (g+1)*G*hd):
//           each stored row is the G*hd slice this KV group's heads feed.
//     GU  : j in split(F, nC, c) = [j0, j0 + nj), in groups of JT: the gate rows
//           of the group, then the up rows of the same j's.
//     D   : columns j0 .. j0 + nj - 1 of W_down, each stored as H contiguous bf16.
//   LM    : rows v in split(V, nC, c) of the LM head (the embedding when tied).
// A tile is TRq rows (QKV), TRh rows (LM), TRo rows (O), one GU group, or JD columns (D);
// the last tile of a block may be short.  Every tile is a multiple of 16 bytes.
//
// Weight-only INT8 streams (wb = 1) store each weight's code q as the byte
// q + 128, with a float scale per output row (QKV, O, gate, up, LM head) or per input
// column (W_down): a row tile is its R rows of K bytes, then the R rows'
// scales; a GU tile is its n gate rows and n up rows, then their 2n scales,
// then the n column scales of W_down for the same j's (the down projection
// folds them into SiLU(gate) * up); a D tile is columns of H bytes.  Each tile
// is padded to 16 bytes.
//
// Weight-only INT4 streams (wb = 0) have the same tiles and scales with two
// codes a byte, each stored as the nibble q + 8: every group of 8 consecutive
// weights of a row (or of a W_down column) is 4 bytes, byte k holding weight k
// in its low nibble and weight k + 4 in its high one, so the low nibbles of
// the word are the group's first four weights and the high nibbles its last
// four -- the same halves as an int8 group's two words.
#pragma once
#include <stdint.h>

#define MK_NCW 12                    // consumer warps
#define MK_WIDE_GROUPS 3             // consumer groups that take the hidden-width GEMVs' tiles in turn
#define MK_NCT (MK_NCW * 32)         // consumer threads
#define MK_PRODUCER_WARP MK_NCW      // bulk-copy producer
#define MK_PREFETCH_WARP (MK_NCW + 1)// L2 prefetch walker
#define MK_BLOCK ((MK_NCW + 2) * 32) // 448 threads: at most 4 warps per SM sub-partition (128 registers)

#define MK_MAX_CPG_G 640               // CTAs per group x query heads per group (combine weights)
#define MK_COMBINE_LOADS 5            // float4 loads per thread in the attention combine
#define MK_MISC_BYTES 6656
#define MK_MAX_H 8192                 // largest hidden size the kernels take
// Positions per CTA from which a step runs the tensor-core attention build.
// Measured on the 1B shape (19 CTAs per KV group) it is as fast as the
// lane-parallel build at 13 positions per CTA and faster from there on (2% at
// 54, 6% at 216), so every step of a shape that has it runs it.
#define MK_ATTN_TC_MIN_PER_CTA 0
// Length-adaptive attention split: a step at context ctx runs its attention on
// ceil(ctx / MK_ATTN_POS_PER_CTA) CTAs of each KV group (at most all of them).
// 192 is one 16-position chunk for each of the 12 consumer warps of the
// tensor-core build: below a full group, fewer CTAs take the same time per
// chunk and the combine waits on fewer partials.
#define MK_ATTN_POS_PER_CTA 192

// Top-p sampling inside the launch: rounds of the 33-way bisection for the
// nucleus threshold (each one grid-wide reduction of 33 masses); the boundary
// is resolved to 104 / 32^MK_TP_ITERS in logit / temperature.
#define MK_TP_ITERS 7
#define MK_TP_BINS 33

// Global scratch of the top-p threshold search, zeroed by the launch's last
// CTA after a top-p step (and once at context creation).
struct MkTopP {
    unsigned long long mkey;               // packed maximum of logit / temperature
    float hist[MK_TP_ITERS][MK_TP_BINS];   // per round: mass of each candidate interval
};

// Device status word bits.
#define MK_ST_TIMEOUT 0x1u
#define MK_ST_NUMERIC 0x2u
#define MK_ST_BADTOKEN 0x4u
#define MK_ST_SCHEDULE 0x8u
#define MK_ST_ABORT 0x80000000u

#ifdef __CUDACC__
#define MK_HD __host__ __device__ __forceinline__
#else
#define MK_HD inline
#endif

MK_HD int64_t mk_split(int64_t n, int64_t parts, int64_t k) { return (k * n) / parts; }

// Stream bytes of K weights: 2 each (bf16, wb = 2), 1 (int8, wb = 1) or half
// a byte (int4, wb = 0: two codes a byte).
MK_HD int64_t mk_wbytes(int64_t K, int wb) { return wb == 0 ? K / 2 : K * wb; }

// Bytes of a row tile: R rows of K weights, and for int8 / int4 (wb < 2) the R
// row scales plus `extra` more scales, padded to 16 bytes.
MK_HD int mk_row_tile_bytes(int R, int K, int wb, int extra) {
    int64_t b = (int64_t)R * mk_wbytes(K, wb);
    if (wb != 2) b += 4LL * (R + extra);
    return (int)((b + 15) & ~(int64_t)15);
}

// Rows per tile for a row-major GEMV tile of K columns: as many as fill a
// ring slot, even (QKV pairs and gate/up groups never straddle a tile).  For
// int8 the tile also holds the scales: gu_extra adds the half-as-many W_down
// column scales of a GU tile.
MK_HD int mk_tile_rows_wb(int K, int slot_bytes, int wb, bool gu_extra) {
    if (wb == 2) return (slot_bytes / (2 * K)) & ~1;
    int r = (int)(slot_bytes / mk_wbytes(K, wb)) & ~1;
    while (r > 2 && mk_row_tile_bytes(r, K, wb, gu_extra ? r / 2 : 0) > slot_bytes) r -= 2;
    return r;
}
MK_HD int mk_tile_rows(int K, int slot_bytes) { return mk_tile_rows_wb(K, slot_bytes, 2, false); }

// Column blocks of the hidden-width GEMV (QKV, gate/up): rows of H = 256 * MH
// columns are split into min(4, MH) blocks, one per consumer warp of a row slot.
MK_HD int mk_wide_nkb(int H) { return H / 256 < 4 ? H / 256 : 4; }

struct MkCtaPlan {
    int64_t stream_off;   // byte offset of this CTA's stream in the arena
    int64_t layer_bytes;  // bytes of one layer's tiles in the stream
    int32_t g, i;         // KV group, index in the group
    int32_t pair0, npairs;
    int32_t orow0, norows;
    int32_t j0, nj;
    int32_t v0, nv;
};

struct MkGeom {
    int32_t L, H, qh, kvh, hd, F, V, max_seq;
    int32_t G, CPG, nC, NP;
    int32_t slot, ns;            // ring slot bytes, ring stages
    int32_t TRh, TRq, TRo, JT, JD, KB;
    int32_t max_rows, max_nj;    // per-CTA maxima (QKV rows, FFN slice)
    int32_t smem_bytes;
    int32_t kv_swz;              // K/V cache rows chunk-permuted (mk_kv_index); set with the long-context build
    int32_t wb;                  // weight form in the stream: 2 bf16, 1 int8, 0 int4 (weight-only INT8 / INT4)
    // shared-memory carve-up (byte offsets from the dynamic smem base)
    int32_t off_full, off_empty, off_xv, off_ov, off_part, off_u, off_xres, off_xres2, off_rope,
        off_red, off_sc, off_misc;
};

// Element index of dim d of position pos in one KV head's rows of the cache
// ([max_seq][hd] bf16).  With swz, the 16-byte chunk index of a row is XORed
// with pos mod 8 (hd >= 64): eight consecutive positions then keep a given
// chunk in eight different shared-memory bank groups once a block of rows is
// copied into shared memory, which the long-context attention's 8x8 matrix
// loads (one chunk of eight consecutive positions each) need to be free of
// bank conflicts.
MK_HD int64_t mk_kv_index(int64_t pos, int d, int hd, int swz) {
    const int c = d >> 3;
    return pos * hd + ((int64_t)((swz ? (c ^ (int)(pos & 7)) : c) << 3) | (d & 7));
}

// Shapes whose attention can run on the tensor cores (4 query heads of 64 or
// 128 dims per KV group); their K/V cache rows are chunk-permuted (mk_kv_index).
MK_HD constexpr bool mk_attn_tc(int hd, int G) { return (hd == 64 || hd == 128) && G == 4; }

// Fills everything but smem offsets from the shape; returns false if the
// shape is outside what the kernels support.
MK_HD bool mk_geom_init(MkGeom& g, int L, int H, int qh, int kvh, int hd, int F, int V, int max_seq, int nC,
                        int slot_bytes, int ns, int wb = 2) {
    g.L = L; g.H = H; g.qh = qh; g.kvh = kvh; g.hd = hd; g.F = F; g.V = V; g.max_seq = max_seq;
    g.kv_swz = 0;
    g.wb = wb;
    if (wb < 0 || wb > 2) return false;
    if (L < 1 || H < 8 || qh < 1 || kvh < 1 || F < 1 || V < 1 || max_seq < 1 || nC < 1) return false;
    if (qh % kvh != 0 || nC % kvh != 0) return false;
    g.G = qh / kvh;
    g.CPG = nC / kvh;
    g.nC = nC;
    g.NP = (g.G + 2) * (hd / 2);
    g.slot = slot_bytes;
    g.ns = ns;
    // a consumer lane holds its share of a hidden-width tile in registers
    // (16 chunks of 16 bytes at most): slots of 32 KB at most
    if (slot_bytes > 32768) return false;
    g.TRh = mk_tile_rows_wb(H, slot_bytes, wb, true);
    g.TRo = mk_tile_rows_wb(g.G * hd, slot_bytes, wb, false);
    g.JT = g.TRh / 2;
    g.JD = (int32_t)(slot_bytes / mk_wbytes(H, wb));
    g.KB = slot_bytes / (2 * hd);
    g.max_rows = 2 * (int)((g.NP + g.CPG - 1) / g.CPG);
    // QKV tiles: TRh rows, or for int8 / int4 rows (which fit 1.75x / 2.75x
    // as many rows in a slot) few enough that a CTA's QKV rows make a tile
    // for each consumer group: one group on all of them was the longest
    // segment of the int4 layer
    g.TRq = g.TRh;
    if (wb != 2) {
        int t = (g.max_rows + MK_WIDE_GROUPS - 1) / MK_WIDE_GROUPS;
        t = (t + 1) & ~1;
        if (t < 2) t = 2;
        if (t < g.TRq) g.TRq = t;
    }
    g.max_nj = (F + nC - 1) / nC;
    return true;
}

// Shared-memory carve-up; returns total bytes.
MK_HD int mk_smem_layout(MkGeom& g) {
    int o = g.ns * g.slot;                    // ring (1024-aligned base)
    g.off_full = o; o += 8 * g.ns;
    g.off_empty = o; o += 8 * g.ns;
    o = (o + 15) & ~15;
    // normalised GEMV input; between QKV and the FFN norm also the attention
    // position-group partials (8 floats per consumer thread); the down-proj fold
    g.off_xv = o; o += 4 * (g.H > 8 * MK_NCT ? g.H : 8 * MK_NCT);
    g.off_ov = o; o += 4 * g.G * g.hd;        // o (O-proj input, split order)
    {   // per-column-block partial sums of the QKV / gate-up rows
        const int rows = g.max_rows > 2 * g.max_nj ? g.max_rows : 2 * g.max_nj;
        g.off_part = o; o += 4 * ((rows * mk_wide_nkb(g.H) + 3) & ~3);
    }
    g.off_u = o; o += 4 * ((g.max_nj + 3) & ~3);
    g.off_xres = o; o += 4 * ((g.H / g.CPG + 4) & ~3);
    g.off_xres2 = o; o += 4 * ((g.H / g.nC + 4) & ~3);
    g.off_rope = o; o += 4 * g.hd;
    o = (o + 15) & ~15;                       // 16-byte loads of the tensor-core attention's q fragments
    g.off_red = o; o += 4 * 2 * MK_NCT;       // double-buffered row partials; the q fragments during attention
    g.off_sc = o; o += 4 * 2 * (8 * MK_NCT / g.hd);   // attention (m, l) per position group and head
    g.off_misc = o; o += MK_MISC_BYTES;       // softmax state, staging, flags
    g.smem_bytes = o;
    return o;
}

// Kernel parameters (passed by value, __grid_constant__).
struct MkParams {
    MkGeom geo;
    float eps;
    int32_t l2_pf_bytes;
    const uint8_t* arena;
    const MkCtaPlan* plans;
    const uint16_t* embed;       // [V][H] bf16
    const float* attn_norm;      // [L][H]
    const float* ffn_norm;       // [L][H]
    const float* final_norm;     // [H]
    uint16_t* kc;                // [L][kvh][max_seq][hd] bf16
    uint16_t* vc;
    const float* rope_cos;       // [max_seq][hd/2]
    const float* rope_sin;
    // Tagged words (low 32 bits: fp32 value, high 32 bits: launch tag = seq + 1).
    // A reader polls the words it needs until every tag is this launch's: the
    // data carries its own ready flag (no fence, counter or separate poll).
    uint64_t* qll;               // [L][qh*hd] rotated q
    uint64_t* kvll;              // [L][kvh][2][hd] K (rotated) and V of the current position, bf16-rounded
    uint64_t* partll;            // [L][kvh][CPG][G*hd + 2G] attention partials: acc[G][hd], then (m, l) per head
    float* xacc;                 // [2][2L][H] residual states (parity double-buffered)
    float* hidden;               // [H]
    uint32_t* cnt;               // flag counters (see mk_cnt_*) then the done counter
    unsigned long long* amax;    // packed argmax key
    int32_t* next_token;
    uint32_t* status;
    uint32_t* seq;               // launch sequence number (selects the xacc parity)
    int32_t pos;
    int32_t attn_ctas;           // A: CTAs of each KV group that run this step's attention (1..CPG)
    int32_t token;               // used when token_ptr == nullptr
    const int32_t* token_ptr;
    float* logits;               // [V] or nullptr
    int32_t* tokens_out;         // greedy output buffer or nullptr
    int32_t out_idx;
    // sampling (cloud.baidu.com/article/9434380, section 5, steps 1 and 5: temperature
    // as a fixed sampling parameter; sampling and the stop condition on the fused path)
    float inv_temp;              // 1 / temperature; 0 = greedy
    uint64_t seed;               // noise generator seed
    int32_t eos_id;              // with stop: a generated token equal to it sets *stop
    int32_t* stop;               // nullptr, or a flag that makes every later launch return at once
    float top_p;                 // nucleus mass (sampling only); >= 1 keeps every token
    float* lgs;                  // [V] logits scratch of a top-p step
    MkTopP* tp;                  // threshold-search scratch of a top-p step
    int32_t dbg_skip_cta, dbg_skip_sync;
    int32_t trace_detail;        // with trace: also per-tile and ring-wait slots
    int32_t inflight;            // most tiles in flight per CTA in streaming segments (>= ns: no limit)
    int32_t inflight_lat;        // the same in latency-bound segments
    int32_t stream_tail;         // where a layer's streaming mode ends: 0 after the down loop, 1 after
                                 // the FFN-block flag wait, 2 after the next layer's QKV GEMV
    int32_t pf_lead_bytes;       // L2 warmer: bytes past the copy cursor it leaves to the ring
    int32_t pf_depth;            // L2 warmer: tiles of warming loads in flight (1 or 2)
    int64_t wait_limit_ns;
    // Optional segment trace (%globaltimer ns), nullptr = off.  Per CTA
    // MK_TRACE_STRIDE slots: consumer events 16*l + e (e = MK_EV_*), end
    // events at 16*L + k, consumer ring-wait ns per layer at 1024 + l,
    // producer ring-wait ns per layer at 1536 + l.
    unsigned long long* trace;
};
#define MK_TRACE_STRIDE 4096
#define MK_TRACE_MAX_LAYERS 63

MK_HD int mk_cnt_A(const MkGeom& g, int l, int grp) { return l * g.kvh + grp; }
MK_HD int mk_cnt_B(const MkGeom& g, int l, int grp) { return g.L * g.kvh + l * g.kvh + grp; }
MK_HD int mk_cnt_C(const MkGeom& g, int l) { return 2 * g.L * g.kvh + l; }
MK_HD int mk_cnt_E(const MkGeom& g, int l) { return 2 * g.L * g.kvh + g.L + l; }
// grid-wide syncs of a top-p step's threshold search: k < MK_TP_ITERS + 1
MK_HD int mk_cnt_tp(const MkGeom& g, int k) { return 2 * g.L * g.kvh + 2 * g.L + k; }
MK_HD int mk_cnt_done(const MkGeom& g) { return 2 * g.L * g.kvh + 2 * g.L + MK_TP_ITERS + 1; }
MK_HD int mk_cnt_total(const MkGeom& g) { return mk_cnt_done(g) + 1; }

MK_HD int mk_imin(int a, int b) { return a < b ? a : b; }

// Bytes of the weight tiles of one layer of a CTA's stream (QKV, O, GU, D).
MK_HD int64_t mk_layer_bytes(const MkGeom& g, const MkCtaPlan& p) {
    int64_t b = 0;
    const int nr = 2 * p.npairs, KO = g.G * g.hd;
    for (int r = 0; r < nr; r += g.TRq) b += mk_row_tile_bytes(mk_imin(g.TRq, nr - r), g.H, g.wb, 0);
    for (int r = 0; r < p.norows; r += g.TRo) b += mk_row_tile_bytes(mk_imin(g.TRo, p.norows - r), KO, g.wb, 0);
    for (int j = 0; j < p.nj; j += g.JT) {
        const int n = mk_imin(g.JT, p.nj - j);
        b += mk_row_tile_bytes(2 * n, g.H, g.wb, n);
    }
    for (int j = 0; j < p.nj; j += g.JD) b += (int64_t)mk_imin(g.JD, p.nj - j) * mk_wbytes(g.H, g.wb);
    return b;
}

// Per-CTA plan; stream offsets are filled by the caller.
MK_HD void mk_cta_plan(const MkGeom& g, int c, MkCtaPlan& p) {
    p.g = c / g.CPG;
    p.i = c % g.CPG;
    int64_t a = mk_split(g.NP, g.CPG, p.i), b = mk_split(g.NP, g.CPG, p.i + 1);
    p.pair0 = (int)a; p.npairs = (int)(b - a);
    a = mk_split(g.H, g.CPG, p.i); b = mk_split(g.H, g.CPG, p.i + 1);
    p.orow0 = (int)a; p.norows = (int)(b - a);
    a = mk_split(g.F, g.nC, c); b = mk_split(g.F, g.nC, c + 1);
    p.j0 = (int)a; p.nj = (int)(b - a);
    a = mk_split(g.V, g.nC, c); b = mk_split(g.V, g.nC, c + 1);
    p.v0 = (int)a; p.nv = (int)(b - a);
    p.layer_bytes = mk_layer_bytes(g, p);
    p.stream_off = 0;
}

MK_HD int64_t mk_lm_bytes(const MkGeom& g, const MkCtaPlan& p) {
    int64_t b = 0;
    for (int r = 0; r < p.nv; r += g.TRh) b += mk_row_tile_bytes(mk_imin(g.TRh, p.nv - r), g.H, g.wb, 0);
    return b;
}

MK_HD int64_t mk_cta_stream_bytes(const MkGeom& g, const MkCtaPlan& p) {
    int64_t b = (int64_t)g.L * p.layer_bytes + mk_lm_bytes(g, p);
    return (b + 255) & ~(int64_t)255;
}

// The share of attended positions [0, pos] of CTA i of a KV group when the
// first A CTAs of each group run the attention (the length-adaptive split:
// cloud.baidu.com/article/9434380, section 8, problems 3 and 5): CTA i < A
// takes split(pos + 1, A, i); the past positions of it, [*ka, *ke) clipped to
// [0, pos), come from the cache, and CTA A - 1 also takes the current
// position, which it reads from the step's own K/V.  CTAs i >= A take none.
MK_HD void mk_attn_share(int pos, int A, int i, int* ka, int* ke, bool* has_cur) {
    const int ctx = pos + 1;
    int a = 0, e = 0;
    if (i < A) {
        a = (int)mk_split(ctx, A, i);
        const int b = (int)mk_split(ctx, A, i + 1);
        e = b < pos ? b : pos;
    }
    *ka = a;
    *ke = e;
    *has_cur = (i == A - 1);
}

// Walks every tile CTA `pl` consumes during the step at position `pos`, in
// consumption order, calling f(src, bytes): per layer the QKV rows, then the
// K and V blocks of its share of positions [0, pos) (mk_attn_share with A
// attention CTAs per group; the current position is read directly, not
// streamed), then the O, gate/up and down tiles; then the LM-head rows.
template <class F>
MK_HD void mk_walk_tiles(const MkGeom& g, const MkCtaPlan& pl, const uint8_t* arena, const uint16_t* kc,
                         const uint16_t* vc, int pos, int A, F&& f) {
    const uint8_t* cur = arena + pl.stream_off;
    const int H = g.H;
    int a, e;
    bool hc;
    mk_attn_share(pos, A, pl.i, &a, &e, &hc);
    const int KO = g.G * g.hd;
    for (int l = 0; l < g.L; ++l) {
        const int nr = 2 * pl.npairs;
        for (int r = 0; r < nr; r += g.TRq) {
            uint32_t by = (uint32_t)mk_row_tile_bytes(mk_imin(g.TRq, nr - r), H, g.wb, 0);
            f((const void*)cur, by); cur += by;
        }
        const int64_t kvoff = ((int64_t)l * g.kvh + pl.g) * g.max_seq * g.hd;
        for (int q = a; q < e; q += g.KB) {
            uint32_t by = (uint32_t)(mk_imin(g.KB, e - q) * g.hd * 2);
            f((const void*)(kc + kvoff + (int64_t)q * g.hd), by);
            f((const void*)(vc + kvoff + (int64_t)q * g.hd), by);
        }
        for (int r = 0; r < pl.norows; r += g.TRo) {
            uint32_t by = (uint32_t)mk_row_tile_bytes(mk_imin(g.TRo, pl.norows - r), KO, g.wb, 0);
            f((const void*)cur, by); cur += by;
        }
        for (int j = 0; j < pl.nj; j += g.JT) {
            const int n = mk_imin(g.JT, pl.nj - j);
            uint32_t by = (uint32_t)mk_row_tile_bytes(2 * n, H, g.wb, n);
            f((const void*)cur, by); cur += by;
        }
        for (int j = 0; j < pl.nj; j += g.JD) {
            uint32_t by = (uint32_t)(mk_imin(g.JD, pl.nj - j) * mk_wbytes(H, g.wb));
            f((const void*)cur, by); cur += by;
        }
    }
    for (int r = 0; r < pl.nv; r += g.TRh) {
        uint32_t by = (uint32_t)mk_row_tile_bytes(mk_imin(g.TRh, pl.nv - r), H, g.wb, 0);
        f((const void*)cur, by); cur += by;
    }
}

// Source row of QKV stored row k (0 .. 2*npairs-1) of a CTA in group grp:
// which matrix (0 q, 1 k, 2 v) and the row inside it.
MK_HD void mk_qkv_row(const MkGeom& g, int grp, int pair, int half, int& mat, int& row) {
    int hd2 = g.hd / 2;
    int s = pair / hd2, d = pair % hd2 + half * hd2;
    if (s < g.G) { mat = 0; row = (grp * g.G + s) * g.hd + d; }
    else if (s == g.G) { mat = 1; row = grp * g.hd + d; }
    else { mat = 2; row = grp * g.hd + d; }
}
