// kda_internal.cuh -- helpers shared by the KDA kernels and their launchers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "kda.h"

namespace kda {

// ------------------------------------------------------------ element access

template <typename T> struct Elem;

template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float *p) { return *p; }
    static __device__ __forceinline__ void store(float *p, float x) { *p = x; }
    // 8 consecutive elements (32 bytes, two 16-byte loads)
    static __device__ __forceinline__ void load8(const float *p, float (&x)[8]) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    static __device__ __forceinline__ void store8(float *p, const float (&x)[8]) {
        reinterpret_cast<float4 *>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
};

template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float x) {
        *p = __float2bfloat16_rn(x);
    }
    static __device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&x)[8]) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // bf16 -> fp32 is a 16-bit shift
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&x)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Offsets of document n, or false when they are out of order / out of range.
__device__ __forceinline__ bool doc_bounds(const int32_t *cu_seqlens, int32_t n,
                                           int32_t N, int64_t T, int64_t &bos,
                                           int64_t &eos) {
    if (cu_seqlens == nullptr) {
        bos = 0;
        eos = T;
        return true;
    }
    bos = cu_seqlens[n];
    eos = cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || eos > T) return false;
    if (n == 0 && bos != 0) return false;
    if (n == N - 1 && eos != T) return false;
    return true;
}

__device__ __forceinline__ void flag_status(int32_t *status, int32_t code) {
    if (status != nullptr) atomicCAS(status, KDA_DEVICE_OK, code);
}

// Prefix snapshots ("From GPT-2 to Kimi K3, from first principles", Chapter 14:
// the state kept at fixed token boundaries so that a later request with the
// same prefix resumes from it).  offsets[i] (strictly increasing, in the packed
// token axis) names the state of the document with bos < offsets[i] <= eos
// after its tokens [bos, offsets[i]); it goes to out[i] ([H, d_k, d_v] fp32,
// laid out as final_state).  A kernel writes the entries of its own document.
struct Snapshots {
    const int32_t *offsets = nullptr;
    int32_t n = 0;
    float *out = nullptr;
};

// the first snapshot index whose offset lies past bos (n when none)
__device__ __forceinline__ int32_t snap_first(const Snapshots &s, int64_t bos) {
    int32_t lo = 0, hi = s.n;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(s.offsets[mid]) <= bos) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Count of kernels queued by this library (kda_kernel_launches).
void count_launches(uint64_t n);

// Dynamic shared memory above the 48 KB default for `kernel`, set once per
// device: the attribute belongs to the current device's copy of the kernel.
// `done` is the call site's own set of devices already done (bit = device).
template <typename Kernel>
cudaError_t allow_dynamic_smem(Kernel *kernel, size_t bytes, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

// Record the thread's last-error text for kda_last_error().
void set_last_error(kda_status code, const char *msg);

// ------------------------------------------------------------ launchers
// Each returns the launch error (cudaSuccess when the kernels were queued).

cudaError_t launch_decode(const void *q, const void *k, const void *v,
                          const float *g, const float *beta, float *state,
                          void *out, int32_t N, int32_t H, int32_t D,
                          kda_dtype dt, cudaStream_t stream);

cudaError_t launch_prologue(const void *q_raw, const void *k_raw,
                            const void *v_raw, const float *conv_w,
                            const float *z_g, const float *z_beta,
                            const int32_t *cu_seqlens, int32_t N, int64_t T,
                            int32_t H, int32_t D, kda_dtype dt, void *q,
                            void *k, void *v, float *g, float *beta,
                            cudaStream_t stream);
// the same over tokens [t_begin, t_end) of the T-token inputs (the conv window
// reaches back before t_begin); outputs q, k, v, g, beta start at row t_begin
cudaError_t launch_prologue_range(const void *q_raw, const void *k_raw, const void *v_raw,
                                  const float *conv_w, const float *z_g, const float *z_beta,
                                  const int32_t *cu_seqlens, int32_t N, int64_t T, int64_t t_begin,
                                  int64_t t_end, int32_t H, int32_t D, kda_dtype dt, void *q,
                                  void *k, void *v, float *g, float *beta, cudaStream_t stream);

cudaError_t launch_prefill_recurrent(const void *q, const void *k,
                                     const void *v, const float *g,
                                     const float *beta, const float *init_state,
                                     const int32_t *cu_seqlens, int32_t N,
                                     int64_t T, int32_t H, int32_t D,
                                     kda_dtype dt, void *out,
                                     float *final_state, int32_t *status,
                                     cudaStream_t stream, const int32_t *order = nullptr,
                                     Snapshots snaps = {});

// checks snapshot offsets (in (0, T], strictly increasing, each a multiple of
// KDA_SNAPSHOT_ALIGN tokens into its document or that document's end) and sets
// KDA_DEVICE_BAD_SNAPSHOT in the status word when one is not
cudaError_t launch_snapshot_check(const int32_t *offsets, int32_t n, const int32_t *cu_seqlens,
                                  int32_t N, int64_t T, int32_t *status, cudaStream_t stream);

// the documents of a packed batch, longest first (chunk count, decreasing):
// order[i] is the document whose CTAs take grid row i.  doc_order_bytes(N) is
// the room it takes in a prefill workspace (0 when N <= 1).
size_t doc_order_bytes(int32_t N);
cudaError_t launch_doc_order(const int32_t *cu_seqlens, int32_t N, int64_t T, int32_t *order,
                             cudaStream_t stream);

cudaError_t launch_decode_conv(const void *q_raw, const void *k_raw, const void *v_raw,
                               const float *conv_w, void *conv_state, const float *z_g,
                               const float *z_beta, float *state, void *out, int32_t N,
                               int32_t H, int32_t D, kda_dtype dt, cudaStream_t stream);

cudaError_t launch_verify(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, const float *state_in, const int32_t *accept,
                          int32_t N, int32_t K, int32_t H, int32_t D, kda_dtype dt, void *out,
                          float *state_out, cudaStream_t stream);

cudaError_t launch_output_gate(const void *o, const void *z, const float *weight, int64_t rows,
                               int32_t D, kda_dtype dt, float eps, void *y, cudaStream_t stream);

cudaError_t launch_selftest_wait(uint64_t limit_ns, int32_t *status, cudaStream_t stream);

// Tensor-core chunked prefill (d = 128, bf16 q/k/v).  With out_f32 set, the
// outputs go there in fp32 (and `out` is not written).
bool chunk_prefill_supported(int32_t D, kda_dtype dt);
cudaError_t launch_prefill_chunk(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const float *init_state,
                                 const int32_t *cu_seqlens, int32_t N, int64_t T, int32_t H,
                                 void *out, float *final_state, int32_t *status,
                                 cudaStream_t stream, const int32_t *order = nullptr,
                                 float *out_f32 = nullptr, Snapshots snaps = {});

// prologue and prefill of one document, segment by segment, overlapped
size_t pipeline_workspace_size(int32_t H, int32_t D, kda_dtype dt, int64_t T, int64_t segment_tokens);
cudaError_t launch_prologue_prefill(const void *q_raw, const void *k_raw, const void *v_raw,
                                    const float *conv_w, const float *z_g, const float *z_beta,
                                    const float *init_state, int64_t T, int32_t H, int32_t D,
                                    kda_dtype dt, int64_t segment_tokens, void *out,
                                    float *final_state, void *workspace, bool use_chunk,
                                    cudaStream_t user, cudaStream_t pro);

// prefill of one document as independent segments joined by an exact scan
size_t segmented_workspace_size(int32_t H, int32_t D, kda_dtype dt, int64_t T, int32_t num_segments);
cudaError_t launch_prefill_segmented(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, const float *init_state, int64_t T, int32_t H,
                                     int32_t D, kda_dtype dt, int32_t num_segments, void *out,
                                     float *final_state, void *workspace, bool use_chunk,
                                     cudaStream_t s);

}  // namespace kda
