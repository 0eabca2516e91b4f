// kda_schedule.cu -- the order in which the documents of a packed batch get
// their CTAs.
//
// The prefill gives every (document, head) one CTA, and a CTA's time grows
// with its document's chunk count (the chunk recurrence is serial inside a
// document).  CTAs start in block order, so with mixed lengths a long
// document that happens to come late runs alone at the end.  Dispatching the
// longest documents first (list scheduling in decreasing size) keeps that
// tail short.  This kernel sorts the documents by chunk count, decreasing,
// into an index array that the prefill kernels read through blockIdx.y.
//
// One CTA, counting sort over kBuckets buckets of the chunk count c: exact
// for c < 128, eight buckets per octave above (documents within ~12% of each
// other may come in either order).  Empty documents come last.  Offsets are
// clamped into [0, T] as in the prefill kernels (which report invalid ones
// through the status word); a negative length counts as empty.  The order
// changes no result, only when each CTA starts: the CTAs are independent.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kOrderThreads = 1024;
constexpr int kOrderBuckets = 288;
constexpr int kTokensPerChunk = 64;

__device__ __forceinline__ int chunk_bucket(int64_t chunks) {
    if (chunks < 128) return static_cast<int>(chunks);
    const int e = 63 - __clzll(static_cast<unsigned long long>(chunks));   // >= 7
    const int b = 128 + 8 * (e - 7) + static_cast<int>((chunks >> (e - 3)) & 7);
    return b < kOrderBuckets ? b : kOrderBuckets - 1;
}

__device__ __forceinline__ int64_t clamped_offset(const int32_t *cu, int n, int64_t T) {
    return min(static_cast<int64_t>(max(cu[n], 0)), T);
}

__global__ void __launch_bounds__(kOrderThreads)
doc_order_kernel(const int32_t *__restrict__ cu, int32_t N, int64_t T, int32_t *__restrict__ order) {
    __shared__ int count[kOrderBuckets];
    __shared__ int next[kOrderBuckets];
    for (int b = threadIdx.x; b < kOrderBuckets; b += kOrderThreads) count[b] = 0;
    __syncthreads();
    auto bucket_of_doc = [&](int n) {
        const int64_t len = max(clamped_offset(cu, n + 1, T) - clamped_offset(cu, n, T), int64_t{0});
        return chunk_bucket((len + kTokensPerChunk - 1) / kTokensPerChunk);
    };
    for (int n = threadIdx.x; n < N; n += kOrderThreads) atomicAdd(&count[bucket_of_doc(n)], 1);
    __syncthreads();
    if (threadIdx.x == 0) {            // first slot of each bucket, largest bucket first
        int run = 0;
        for (int b = kOrderBuckets - 1; b >= 0; --b) {
            next[b] = run;
            run += count[b];
        }
    }
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += kOrderThreads) order[atomicAdd(&next[bucket_of_doc(n)], 1)] = n;
}

}  // namespace

size_t doc_order_bytes(int32_t N) {
    return N > 1 ? (static_cast<size_t>(N) * sizeof(int32_t) + 255) / 256 * 256 : 0;
}

cudaError_t launch_doc_order(const int32_t *cu_seqlens, int32_t N, int64_t T, int32_t *order,
                             cudaStream_t stream) {
    doc_order_kernel<<<1, kOrderThreads, 0, stream>>>(cu_seqlens, N, T, order);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
