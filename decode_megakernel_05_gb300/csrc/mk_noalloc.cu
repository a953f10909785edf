// mk_noalloc.cu - greedy argmax over a caller's logits that allocates nothing.
//
// Some callers cannot call cudaMalloc: engines that reserve all device memory
// up front and hand out only pointers into their own pool, and code on a
// latency-critical path where an allocation (and the device synchronization it
// may imply) is not allowed.  mk_argmax_f32_noalloc serves them: the caller
// passes the logits and the output slot, and the only scratch the two kernels
// need (one partial key per block) lives in the file-scope device array below,
// which every GPU that loads this library holds until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents; each call writes every slot it later reads, so nothing needs
// clearing.  Calls whose kernels overlap on the GPU (two streams at once)
// race on the array and must be serialized by the caller.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/mk.h"
#include "mk_aux.h"

namespace {

constexpr int kThreads = 256;
constexpr int kItemsPerThread = 16;
constexpr int kPerBlock = kThreads * kItemsPerThread;   // logits one block scans
static_assert((long long)MK_NOALLOC_ARGMAX_MAX_N == (long long)MK_NOALLOC_ARGMAX_BLOCKS * kPerBlock,
              "the size limit must match the scratch array");

static __device__ __align__(256) unsigned long long g_argmax_scratch[MK_NOALLOC_ARGMAX_BLOCKS];

// Order-preserving key: larger float -> larger key; on equal values the lower
// index wins (its complement is larger).  -0.0 and +0.0 compare equal as
// floats, so both take the key of +0.0 (the lower index then wins, as in a
// float comparison).
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    if (v == 0.0f) v = 0.0f;
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)idx);
}

__global__ void noalloc_argmax_partial(const float* __restrict__ lg, int n, unsigned long long* part) {
    __shared__ unsigned long long red[kThreads / 32];
    unsigned long long best = 0ull;   // 0 = no finite value seen
    const int base = blockIdx.x * kPerBlock;
    for (int k = 0; k < kItemsPerThread; ++k) {
        const int i = base + k * kThreads + threadIdx.x;
        if (i < n) {
            const float v = lg[i];
            if (isfinite(v)) {
                const unsigned long long key = argmax_key(v, i);
                best = key > best ? key : best;
            }
        }
    }
    for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = other > best ? other : best;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kThreads / 32; ++w) best = red[w] > best ? red[w] : best;
        part[blockIdx.x] = best;
    }
}

__global__ void noalloc_argmax_final(const unsigned long long* part, int nblocks, int32_t* out) {
    __shared__ unsigned long long red[kThreads / 32];
    unsigned long long best = 0ull;
    for (int b = threadIdx.x; b < nblocks; b += kThreads) best = part[b] > best ? part[b] : best;
    for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = other > best ? other : best;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kThreads / 32; ++w) best = red[w] > best ? red[w] : best;
        *out = best == 0ull ? -1 : (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
    }
}

// Device address of the scratch array, looked up once per device (the
// array's host-side name is only a handle for the runtime, not an address).
// The address stays valid for the life of the device's context; after a
// cudaDeviceReset the cached address is stale (the entry point is not for use
// on that device afterwards).
constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_scratch_addr[kMaxDevices] = {};

int scratch_for_current_device(unsigned long long** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return mk_record_cuda_error(e, "mk_argmax_f32_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return MK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_argmax_scratch);
        if (e != cudaSuccess) return mk_record_cuda_error(e, "mk_argmax_f32_noalloc: cudaGetSymbolAddress");
        if (!p) return MK_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = reinterpret_cast<unsigned long long*>(g_scratch_addr[dev]);
    return MK_OK;
}

}  // namespace

extern "C" int mk_argmax_f32_noalloc(const float* logits, int32_t n, int32_t* out_token, void* stream) {
    if (!logits || !out_token || n < 1) return MK_ERR_INVALID_ARG;
    if ((int64_t)n > (int64_t)MK_NOALLOC_ARGMAX_MAX_N) return MK_ERR_INVALID_ARG;
    unsigned long long* scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != MK_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int nblocks = (n + kPerBlock - 1) / kPerBlock;
    // cudaLaunchKernel returns the outcome of this launch itself, so an error
    // an earlier, unrelated call left pending is neither taken for this
    // call's nor cleared; a failure names the kernel that did not launch
    void* a1[] = {(void*)&logits, (void*)&n, (void*)&scratch};
    cudaError_t e = cudaLaunchKernel((const void*)noalloc_argmax_partial, dim3(nblocks), dim3(kThreads), a1, 0, st);
    if (e != cudaSuccess) return mk_record_cuda_error(e, "mk_argmax_f32_noalloc: partial-argmax launch");
    const unsigned long long* part = scratch;
    int nb = nblocks;
    void* a2[] = {(void*)&part, (void*)&nb, (void*)&out_token};
    e = cudaLaunchKernel((const void*)noalloc_argmax_final, dim3(1), dim3(kThreads), a2, 0, st);
    if (e != cudaSuccess) return mk_record_cuda_error(e, "mk_argmax_f32_noalloc: final-argmax launch");
    return MK_OK;
}
