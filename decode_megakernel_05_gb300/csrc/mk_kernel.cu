// mk_kernel.cu - one instantiation of the decode megakernel per translation
// unit: the build compiles this file once for every (head_dim, query heads per
// KV group, hidden/256) triple it supports, with -DMK_HD_V=<hd> -DMK_G_V=<G>
// -DMK_MH_V=<H/256>, so the variants compile in parallel.
#include "mk_kernel.cuh"

#if !defined(MK_HD_V) || !defined(MK_G_V) || !defined(MK_MH_V)
#error "compile with -DMK_HD_V=<head_dim> -DMK_G_V=<q heads per kv head> -DMK_MH_V=<hidden/256>"
#endif

#ifndef MK_LC_V
#define MK_LC_V 0   // 1: the long-context build (see mk_decode_kernel)
#endif
#ifndef MK_WB_V
#define MK_WB_V 2   // streamed weight form: 2 bf16, 1 weight-only INT8, 0 weight-only INT4
#endif
#if MK_LC_V && MK_WB_V == 1
#define MK_SFX _lc_q8
#elif MK_LC_V && MK_WB_V == 0
#define MK_SFX _lc_q4
#elif MK_LC_V
#define MK_SFX _lc
#elif MK_WB_V == 1
#define MK_SFX _q8
#elif MK_WB_V == 0
#define MK_SFX _q4
#else
#define MK_SFX
#endif
#define MK_CAT2(a, b, c, d, e) a##b##_##c##_##d##e
#define MK_CAT(a, b, c, d, e) MK_CAT2(a, b, c, d, e)

// Built twice per variant: with -DMK_NO_TRACE (the production kernel, no trace
// code at all: a smaller instruction footprint per layer) and without (the
// kernel launched while a segment trace is requested).
#ifdef MK_NO_TRACE
extern "C" const void* MK_CAT(mk_kernel_ptr_, MK_HD_V, MK_G_V, MK_MH_V, MK_SFX)(void) {
    return (const void*)&mk::mk_decode_kernel<MK_HD_V, MK_G_V, MK_MH_V, MK_LC_V, MK_WB_V>;
}
#else
extern "C" const void* MK_CAT(mk_kernel_trace_ptr_, MK_HD_V, MK_G_V, MK_MH_V, MK_SFX)(void) {
    return (const void*)&mk::mk_decode_kernel<MK_HD_V, MK_G_V, MK_MH_V, MK_LC_V, MK_WB_V>;
}
#endif
