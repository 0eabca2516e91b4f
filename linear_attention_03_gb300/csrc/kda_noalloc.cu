// kda_noalloc.cu -- a prefill entry point that allocates nothing.
//
// kda_prefill needs a small device workspace that the caller allocates.  Some
// callers cannot do that: code that runs where device allocation is not
// allowed or not wanted -- plug-ins inside engines that own every byte of
// device memory, serving loops that must not allocate after start-up, hosts
// without their own allocator.  kda_prefill_noalloc serves them with scratch
// that lives in this library instead: a file-scope __device__ array of
// kNoAllocScratchBytes, which every GPU that loads the library holds until the
// process exits.  The caller still passes every input and output.
//
// Set-up: in host code the array's name is only a host-side stand-in, not a
// device address, so the first call on each device (with that device
// current) looks its address up with cudaGetSymbolAddress and caches it.
// That first call should therefore happen before any stream capture.
//
// Every call on a device shares the one array and finds the previous call's
// contents in it; kda_prefill clears the status word at the start of each
// call.  Calls whose work overlaps on the GPU (other streams, no ordering)
// race on the array.
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 65536;   // 64 KiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace

extern "C" kda_status kda_prefill_noalloc(const void *q, const void *k, const void *v,
                                          const float *g, const float *beta,
                                          const float *init_state, const int32_t *cu_seqlens,
                                          int32_t N, int64_t T, kda_dims dims, void *out,
                                          float *final_state, int32_t *status_out,
                                          void *stream) {
    // the scratch always holds the status word; up to 16,320 documents it
    // also holds their dispatch order (larger batches run in document order)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        kda::set_last_error(KDA_ERR_CUDA, "kda_prefill_noalloc: no usable current device");
        return KDA_ERR_CUDA;
    }
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (g_scratch_addr[dev] == nullptr) {
            err = cudaGetSymbolAddress(&g_scratch_addr[dev], g_noalloc_scratch);
            if (err != cudaSuccess) {
                g_scratch_addr[dev] = nullptr;
                kda::set_last_error(KDA_ERR_CUDA,
                                    "kda_prefill_noalloc: cudaGetSymbolAddress of the static "
                                    "scratch failed");
                return KDA_ERR_CUDA;
            }
        }
        scratch = g_scratch_addr[dev];
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
