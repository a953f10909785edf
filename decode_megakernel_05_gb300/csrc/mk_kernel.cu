// mk_kernel.cu - one instantiation of the decode megakernel per translation
// unit: the build compiles this file once for every (head_dim, query heads per
// KV group) pair it supports, with -DMK_HD_V=<hd> -DMK_G_V=<G>, so the
// variants compile in parallel.
#include "mk_kernel.cuh"

#if !defined(MK_HD_V) || !defined(MK_G_V)
#error "compile with -DMK_HD_V=<head_dim> -DMK_G_V=<q heads per kv head>"
#endif

#define MK_CAT2(a, b, c) a##b##_##c
#define MK_CAT(a, b, c) MK_CAT2(a, b, c)

extern "C" const void* MK_CAT(mk_kernel_ptr_, MK_HD_V, MK_G_V)(void) {
    return (const void*)&mk::mk_decode_kernel<MK_HD_V, MK_G_V>;
}
