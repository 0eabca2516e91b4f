// kda_noalloc.cu -- a prefill entry point that allocates nothing.
//
// kda_prefill needs a small device workspace that the caller allocates.  Some
// callers cannot do that: code that runs where device allocation is not
// allowed or not wanted -- plug-ins inside engines that own every byte of
// device memory, serving loops that must not allocate after start-up, hosts
// without their own allocator.  kda_prefill_noalloc serves them with scratch
// that lives in this library instead: a file-scope __device__ array of
// kNoAllocScratchBytes in the library's module.  The caller still passes every
// input and output.
//
// Set-up: in host code the array's name is only a host-side stand-in, not a
// device address.  The first call in each CUDA context looks the address up
// with cudaGetSymbolAddress; with CUDA's lazy module loading that is also when
// the module, with the array, and on first launch the prefill kernels' modules
// are loaded into the context, which takes device memory.  So the first call
// per context belongs at start-up, before any stream capture; later calls in
// that context allocate nothing.  The address is cached per context (keyed on
// the driver's unique context ID), so a context created after
// cudaDeviceReset, or a non-primary context on the same device, gets its own
// lookup and never the address of another context's copy.
//
// Every call on a device shares the one array and finds the previous call's
// contents in it; kda_prefill clears the status word at the start of each
// call.  Calls whose work overlaps on the GPU (other streams, no ordering)
// race on the array.
#include <cuda.h>

#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 65536;   // 64 KiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// the scratch address per CUDA context, keyed on the context's unique ID
constexpr int kMaxContexts = 64;
struct CtxEntry {
    unsigned long long id;
    void *addr;
};
CtxEntry g_scratch[kMaxContexts] = {};
int g_scratch_n = 0;
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <class F>
F driver_fn(const char *name) {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<F>(p);
    return nullptr;
}

// the unique ID of the calling thread's current context; a thread with none
// current gets the current device's primary context, as any runtime call would
bool current_context_id(unsigned long long *id) {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (get_current == nullptr || get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return false;
    if (ctx == nullptr) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return false;
        if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    }
    return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

extern "C" kda_status kda_prefill_noalloc(const void *q, const void *k, const void *v,
                                          const float *g, const float *beta,
                                          const float *init_state, const int32_t *cu_seqlens,
                                          int32_t N, int64_t T, kda_dims dims, void *out,
                                          float *final_state, int32_t *status_out,
                                          void *stream) {
    // the scratch always holds the status word; up to 16,320 documents it
    // also holds their dispatch order (larger batches run in document order)
    unsigned long long ctx_id = 0;
    if (!current_context_id(&ctx_id)) {
        kda::set_last_error(KDA_ERR_CUDA, "kda_prefill_noalloc: no usable current CUDA context");
        return KDA_ERR_CUDA;
    }
    void *scratch = nullptr;
    cudaError_t err;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        for (int i = 0; i < g_scratch_n; ++i)
            if (g_scratch[i].id == ctx_id) scratch = g_scratch[i].addr;
        if (scratch == nullptr) {
            if (g_scratch_n == kMaxContexts) {
                kda::set_last_error(KDA_ERR_CUDA, "kda_prefill_noalloc: more than 64 CUDA contexts");
                return KDA_ERR_CUDA;
            }
            err = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
            if (err != cudaSuccess || scratch == nullptr) {
                kda::set_last_error(KDA_ERR_CUDA,
                                    "kda_prefill_noalloc: cudaGetSymbolAddress of the static "
                                    "scratch failed");
                return KDA_ERR_CUDA;
            }
            g_scratch[g_scratch_n++] = CtxEntry{ctx_id, scratch};
        }
    }
    const kda_status st = kda_prefill(q, k, v, g, beta, init_state, cu_seqlens, N, T, dims, out,
                                      final_state, scratch, kNoAllocScratchBytes, stream);
    if (st != KDA_OK || status_out == nullptr) return st;
    err = cudaMemcpyAsync(status_out, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                          static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) {
        kda::set_last_error(KDA_ERR_CUDA, "kda_prefill_noalloc: copying the status word failed");
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}
