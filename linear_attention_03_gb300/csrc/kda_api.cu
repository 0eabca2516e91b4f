// kda_api.cu -- the C ABI declared in include/kda.h: argument checks,
// path selection and kernel launches.  No allocation happens here; every
// buffer belongs to the caller.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "kda_internal.cuh"

namespace {

thread_local char g_last_error[512] = "";
std::atomic<uint64_t> g_launches{0};

kda_status fail(kda_status code, const char *fmt, const char *what = "") {
    snprintf(g_last_error, sizeof(g_last_error), fmt, what);
    return code;
}

kda_status cuda_fail(cudaError_t err, const char *where) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, cudaGetErrorString(err));
    return KDA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status check_dims(const kda_dims &d) {
    if (d.H < 1) return fail(KDA_ERR_INVALID, "H must be >= 1%s");
    if (d.qkv_dtype != KDA_F32 && d.qkv_dtype != KDA_BF16)
        return fail(KDA_ERR_UNSUPPORTED, "qkv_dtype must be KDA_F32 or KDA_BF16%s");
    if (d.d_k != d.d_v)
        return fail(KDA_ERR_UNSUPPORTED, "d_k must equal d_v%s");
    if (d.d_k != 16 && d.d_k != 32 && d.d_k != 64 && d.d_k != 128)
        return fail(KDA_ERR_UNSUPPORTED, "head size must be 16, 32, 64 or 128%s");
    return KDA_OK;
}

// required pointer: non-null and 16-byte aligned; optional: null or aligned
kda_status need(const void *p, const char *name) {
    if (p == nullptr) return fail(KDA_ERR_INVALID, "%s must not be NULL", name);
    if (!aligned16(p)) return fail(KDA_ERR_INVALID, "%s must be 16-byte aligned", name);
    return KDA_OK;
}

// beta is read element by element: its natural 4-byte alignment suffices
kda_status need4(const void *p, const char *name) {
    if (p == nullptr) return fail(KDA_ERR_INVALID, "%s must not be NULL", name);
    if ((reinterpret_cast<uintptr_t>(p) & 3u) != 0)
        return fail(KDA_ERR_INVALID, "%s must be 4-byte aligned", name);
    return KDA_OK;
}

kda_status maybe(const void *p, const char *name) {
    if (p != nullptr && !aligned16(p))
        return fail(KDA_ERR_INVALID, "%s must be 16-byte aligned", name);
    return KDA_OK;
}

#define KDA_TRY(expr)                        \
    do {                                     \
        const kda_status _s = (expr);        \
        if (_s != KDA_OK) return _s;         \
    } while (0)

constexpr size_t kStatusBytes = 256;

// KDA_PREFILL_PATH=recurrent forces the CUDA-core prefill everywhere (used to
// cross-check the two prefill kernels on the same inputs); read once.
bool force_recurrent() {
    static const int v = [] {
        const char *e = getenv("KDA_PREFILL_PATH");
        return (e != nullptr && strcmp(e, "recurrent") == 0) ? 1 : 0;
    }();
    return v != 0;
}

}  // namespace

void kda::count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

void kda::set_last_error(kda_status code, const char *msg) { fail(code, "%s", msg); }

extern "C" {

const char *kda_last_error(void) { return g_last_error; }

uint64_t kda_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

size_t kda_prefill_workspace_size(kda_dims dims, int64_t T, int32_t N) {
    (void)dims;
    (void)T;
    // the status word, then (N > 1) the documents' dispatch order
    return kStatusBytes + kda::doc_order_bytes(N);
}

namespace {

kda_status prefill_impl(const void *q, const void *k, const void *v, const float *g,
                        const float *beta, const float *init_state, const int32_t *cu_seqlens,
                        int32_t N, int64_t T, kda_dims dims, void *out, float *final_state,
                        kda::Snapshots snaps, void *workspace, size_t workspace_bytes,
                        void *stream) {
    KDA_TRY(check_dims(dims));
    if (N < 1 || N > 65535) return fail(KDA_ERR_INVALID, "N must be in [1, 65535]%s");
    if (T < 0 || T > INT32_MAX) return fail(KDA_ERR_INVALID, "T must be in [0, 2^31)%s");
    if (cu_seqlens == nullptr && N != 1)
        return fail(KDA_ERR_INVALID, "cu_seqlens may be NULL only when N == 1%s");
    if (T > 0) {
        KDA_TRY(need(q, "q"));
        KDA_TRY(need(k, "k"));
        KDA_TRY(need(v, "v"));
        KDA_TRY(need(g, "g"));
        KDA_TRY(need4(beta, "beta"));
        KDA_TRY(need(out, "out"));
    }
    KDA_TRY(maybe(init_state, "init_state"));
    KDA_TRY(maybe(final_state, "final_state"));
    KDA_TRY(maybe(cu_seqlens, "cu_seqlens"));
    KDA_TRY(need(workspace, "workspace"));
    if (workspace_bytes < kStatusBytes)
        return fail(KDA_ERR_INVALID, "workspace too small (see kda_prefill_workspace_size)%s");

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t *status = static_cast<int32_t *>(workspace);
    cudaError_t err = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
    if (err != cudaSuccess) return cuda_fail(err, "clearing the status word");
    // several documents: their CTAs are dispatched longest first when the
    // workspace has room for the order (else in document order)
    const int32_t *order = nullptr;
    if (N > 1 && T > 0 && workspace_bytes >= kStatusBytes + kda::doc_order_bytes(N)) {
        int32_t *ord = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + kStatusBytes);
        err = kda::launch_doc_order(cu_seqlens, N, T, ord, s);
        if (err != cudaSuccess) return cuda_fail(err, "document order launch");
        order = ord;
    }
    if (snaps.n > 0) {
        err = kda::launch_snapshot_check(snaps.offsets, snaps.n, cu_seqlens, N, T, status, s);
        if (err != cudaSuccess) return cuda_fail(err, "snapshot offset check launch");
    }
    const kda_dtype dt = (kda_dtype)dims.qkv_dtype;
    if (T > 0 && kda::chunk_prefill_supported(dims.d_k, dt) && !force_recurrent())
        err = kda::launch_prefill_chunk(q, k, v, g, beta, init_state, cu_seqlens, N, T, dims.H,
                                        out, final_state, status, s, order, nullptr, snaps);
    else
        err = kda::launch_prefill_recurrent(q, k, v, g, beta, init_state, cu_seqlens, N, T,
                                            dims.H, dims.d_k, dt, out, final_state, status, s,
                                            order, snaps);
    if (err != cudaSuccess) return cuda_fail(err, "prefill launch");
    return KDA_OK;
}

}  // namespace

kda_status kda_prefill(const void *q, const void *k, const void *v,
                       const float *g, const float *beta,
                       const float *init_state, const int32_t *cu_seqlens,
                       int32_t N, int64_t T, kda_dims dims, void *out,
                       float *final_state, void *workspace,
                       size_t workspace_bytes, void *stream) {
    g_last_error[0] = '\0';
    return prefill_impl(q, k, v, g, beta, init_state, cu_seqlens, N, T, dims, out, final_state, {},
                        workspace, workspace_bytes, stream);
}

kda_status kda_prefill_snapshots(const void *q, const void *k, const void *v,
                                 const float *g, const float *beta,
                                 const float *init_state, const int32_t *cu_seqlens,
                                 int32_t N, int64_t T, kda_dims dims, void *out,
                                 float *final_state, const int32_t *snapshot_offsets,
                                 int32_t n_snapshots, float *snapshots, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    g_last_error[0] = '\0';
    if (n_snapshots < 0) return fail(KDA_ERR_INVALID, "n_snapshots must be >= 0%s");
    if (n_snapshots > 0) {
        KDA_TRY(need4(snapshot_offsets, "snapshot_offsets"));
        KDA_TRY(need(snapshots, "snapshots"));
    }
    kda::Snapshots snaps;
    snaps.offsets = n_snapshots > 0 ? snapshot_offsets : nullptr;
    snaps.n = n_snapshots;
    snaps.out = n_snapshots > 0 ? snapshots : nullptr;
    return prefill_impl(q, k, v, g, beta, init_state, cu_seqlens, N, T, dims, out, final_state, snaps,
                        workspace, workspace_bytes, stream);
}

size_t kda_prologue_prefill_workspace_size(kda_dims dims, int64_t T, int64_t segment_tokens) {
    if (check_dims(dims) != KDA_OK || T < 0 || segment_tokens < 1) return 0;
    return kda::pipeline_workspace_size(dims.H, dims.d_k, (kda_dtype)dims.qkv_dtype, T, segment_tokens);
}

kda_status kda_prologue_prefill(const void *q_raw, const void *k_raw, const void *v_raw,
                                const float *conv_w, const float *z_g, const float *z_beta,
                                const float *init_state, int64_t T, kda_dims dims,
                                int64_t segment_tokens, void *out, float *final_state,
                                void *workspace, size_t workspace_bytes, void *stream,
                                void *prologue_stream) {
    g_last_error[0] = '\0';
    KDA_TRY(check_dims(dims));
    if (T < 0 || T > INT32_MAX) return fail(KDA_ERR_INVALID, "T must be in [0, 2^31)%s");
    if (segment_tokens < 1) return fail(KDA_ERR_INVALID, "segment_tokens must be >= 1%s");
    if (T > 0) {
        KDA_TRY(need(q_raw, "q_raw"));
        KDA_TRY(need(k_raw, "k_raw"));
        KDA_TRY(need(v_raw, "v_raw"));
        KDA_TRY(need(conv_w, "conv_w"));
        KDA_TRY(need(z_g, "z_g"));
        KDA_TRY(need4(z_beta, "z_beta"));
        KDA_TRY(need(out, "out"));
    }
    KDA_TRY(maybe(init_state, "init_state"));
    KDA_TRY(maybe(final_state, "final_state"));
    KDA_TRY(need(workspace, "workspace"));
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(KDA_ERR_INVALID, "workspace must be 256-byte aligned%s");
    if (workspace_bytes < kda_prologue_prefill_workspace_size(dims, T, segment_tokens))
        return fail(KDA_ERR_INVALID, "workspace too small (see kda_prologue_prefill_workspace_size)%s");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t sbytes = (size_t)dims.H * dims.d_k * dims.d_v * sizeof(float);
    if (T == 0) {
        cudaError_t err = cudaMemsetAsync(workspace, 0, sizeof(int32_t), s);
        if (err == cudaSuccess && final_state != nullptr && final_state != init_state)
            err = init_state ? cudaMemcpyAsync(final_state, init_state, sbytes, cudaMemcpyDeviceToDevice, s)
                             : cudaMemsetAsync(final_state, 0, sbytes, s);
        return err == cudaSuccess ? KDA_OK : cuda_fail(err, "prologue + prefill (T = 0)");
    }
    const kda_dtype dt = (kda_dtype)dims.qkv_dtype;
    const bool chunk = kda::chunk_prefill_supported(dims.d_k, dt) && !force_recurrent();
    cudaError_t err = kda::launch_prologue_prefill(q_raw, k_raw, v_raw, conv_w, z_g, z_beta, init_state, T,
                                                   dims.H, dims.d_k, dt, segment_tokens, out, final_state,
                                                   workspace, chunk, s,
                                                   static_cast<cudaStream_t>(prologue_stream));
    if (err != cudaSuccess) return cuda_fail(err, "prologue + prefill launch");
    return KDA_OK;
}

size_t kda_prefill_segmented_workspace_size(kda_dims dims, int64_t T, int32_t num_segments) {
    if (check_dims(dims) != KDA_OK || T < 0 || num_segments < 1) return 0;
    return kda::segmented_workspace_size(dims.H, dims.d_k, (kda_dtype)dims.qkv_dtype, T, num_segments);
}

kda_status kda_prefill_segmented(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const float *init_state, int64_t T,
                                 kda_dims dims, int32_t num_segments, void *out,
                                 float *final_state, void *workspace, size_t workspace_bytes,
                                 void *stream) {
    g_last_error[0] = '\0';
    KDA_TRY(check_dims(dims));
    if (T < 0 || T > INT32_MAX) return fail(KDA_ERR_INVALID, "T must be in [0, 2^31)%s");
    if (num_segments < 1 || num_segments > 65535)
        return fail(KDA_ERR_INVALID, "num_segments must be in [1, 65535]%s");
    if (T > 0) {
        KDA_TRY(need(q, "q"));
        KDA_TRY(need(k, "k"));
        KDA_TRY(need(v, "v"));
        KDA_TRY(need(g, "g"));
        KDA_TRY(need4(beta, "beta"));
        KDA_TRY(need(out, "out"));
    }
    KDA_TRY(maybe(init_state, "init_state"));
    KDA_TRY(maybe(final_state, "final_state"));
    KDA_TRY(need(workspace, "workspace"));
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(KDA_ERR_INVALID, "workspace must be 256-byte aligned%s");
    if (workspace_bytes < kda_prefill_segmented_workspace_size(dims, T, num_segments))
        return fail(KDA_ERR_INVALID, "workspace too small (see kda_prefill_segmented_workspace_size)%s");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t err = cudaMemsetAsync(workspace, 0, sizeof(int32_t), s);
        const size_t bytes = (size_t)dims.H * dims.d_k * dims.d_v * sizeof(float);
        if (err == cudaSuccess && final_state != nullptr && final_state != init_state)
            err = init_state ? cudaMemcpyAsync(final_state, init_state, bytes, cudaMemcpyDeviceToDevice, s)
                             : cudaMemsetAsync(final_state, 0, bytes, s);
        return err == cudaSuccess ? KDA_OK : cuda_fail(err, "segmented prefill (T = 0)");
    }
    const kda_dtype dt = (kda_dtype)dims.qkv_dtype;
    const bool chunk = kda::chunk_prefill_supported(dims.d_k, dt) && !force_recurrent();
    cudaError_t err = kda::launch_prefill_segmented(q, k, v, g, beta, init_state, T, dims.H, dims.d_k, dt,
                                                    num_segments, out, final_state, workspace, chunk, s);
    if (err != cudaSuccess) return cuda_fail(err, "segmented prefill launch");
    return KDA_OK;
}

kda_status kda_decode_step(const void *q, const void *k, const void *v,
                           const float *g, const float *beta, float *state,
                           void *out, int32_t N, kda_dims dims, void *stream) {
    g_last_error[0] = '\0';
    KDA_TRY(check_dims(dims));
    if (N < 0) return fail(KDA_ERR_INVALID, "N must be >= 0%s");
    if ((int64_t)N * dims.H > INT32_MAX) return fail(KDA_ERR_INVALID, "N * H too large%s");
    if (N == 0) return KDA_OK;
    KDA_TRY(need(q, "q"));
    KDA_TRY(need(k, "k"));
    KDA_TRY(need(v, "v"));
    KDA_TRY(need(g, "g"));
    KDA_TRY(need4(beta, "beta"));
    KDA_TRY(need(state, "state"));
    KDA_TRY(need(out, "out"));
    cudaError_t err = kda::launch_decode(q, k, v, g, beta, state, out, N, dims.H, dims.d_k,
                                         (kda_dtype)dims.qkv_dtype,
                                         static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "decode launch");
    return KDA_OK;
}

kda_status kda_prologue(const void *q_raw, const void *k_raw,
                        const void *v_raw, const float *conv_w,
                        const float *z_g, const float *z_beta,
                        const int32_t *cu_seqlens, int32_t N, int64_t T,
                        kda_dims dims, void *q, void *k, void *v, float *g,
                        float *beta, void *stream) {
    g_last_error[0] = '\0';
    KDA_TRY(check_dims(dims));
    if (N < 1) return fail(KDA_ERR_INVALID, "N must be >= 1%s");
    if (T < 0 || T > INT32_MAX) return fail(KDA_ERR_INVALID, "T must be in [0, 2^31)%s");
    if (cu_seqlens == nullptr && N != 1)
        return fail(KDA_ERR_INVALID, "cu_seqlens may be NULL only when N == 1%s");
    if (T == 0) return KDA_OK;
    KDA_TRY(need(q_raw, "q_raw"));
    KDA_TRY(need(k_raw, "k_raw"));
    KDA_TRY(need(v_raw, "v_raw"));
    KDA_TRY(need(conv_w, "conv_w"));
    KDA_TRY(need(q, "q"));
    KDA_TRY(need(k, "k"));
    KDA_TRY(need(v, "v"));
    KDA_TRY(maybe(z_g, "z_g"));
    if (z_beta != nullptr) KDA_TRY(need4(z_beta, "z_beta"));
    KDA_TRY(maybe(cu_seqlens, "cu_seqlens"));
    if (z_g != nullptr) KDA_TRY(need(g, "g"));
    if (z_beta != nullptr) KDA_TRY(need4(beta, "beta"));
    cudaError_t err = kda::launch_prologue(q_raw, k_raw, v_raw, conv_w, z_g, z_beta,
                                           cu_seqlens, N, T, dims.H, dims.d_k,
                                           (kda_dtype)dims.qkv_dtype, q, k, v, g, beta,
                                           static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "prologue launch");
    return KDA_OK;
}

kda_status kda_decode_step_conv(const void *q_raw, const void *k_raw, const void *v_raw,
                                const float *conv_w, void *conv_state, const float *z_g,
                                const float *z_beta, float *state, void *out, int32_t N,
                                kda_dims dims, void *stream) {
    g_last_error[0] = '\0';
    KDA_TRY(check_dims(dims));
    if (N < 0) return fail(KDA_ERR_INVALID, "N must be >= 0%s");
    if ((int64_t)N * dims.H > INT32_MAX) return fail(KDA_ERR_INVALID, "N * H too large%s");
    if (N == 0) return KDA_OK;
    KDA_TRY(need(q_raw, "q_raw"));
    KDA_TRY(need(k_raw, "k_raw"));
    KDA_TRY(need(v_raw, "v_raw"));
    KDA_TRY(need(conv_w, "conv_w"));
    KDA_TRY(need(conv_state, "conv_state"));
    KDA_TRY(need(z_g, "z_g"));
    KDA_TRY(need4(z_beta, "z_beta"));
    KDA_TRY(need(state, "state"));
    KDA_TRY(need(out, "out"));
    cudaError_t err = kda::launch_decode_conv(q_raw, k_raw, v_raw, conv_w, conv_state, z_g, z_beta,
                                              state, out, N, dims.H, dims.d_k,
                                              (kda_dtype)dims.qkv_dtype,
                                              static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "decode-with-conv launch");
    return KDA_OK;
}

kda_status kda_decode_verify(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const float *state_in, const int32_t *accept,
                             int32_t N, int32_t K, kda_dims dims, void *out, float *state_out,
                             void *stream) {
    g_last_error[0] = '\0';
    KDA_TRY(check_dims(dims));
    if (N < 0 || K < 1) return fail(KDA_ERR_INVALID, "N must be >= 0 and K >= 1%s");
    if ((int64_t)N * K * dims.H > INT32_MAX) return fail(KDA_ERR_INVALID, "N * K * H too large%s");
    // up to two CTAs per (sequence, head)
    if ((int64_t)N * dims.H * 2 > INT32_MAX) return fail(KDA_ERR_INVALID, "N * H too large%s");
    if (N == 0) return KDA_OK;
    KDA_TRY(need(q, "q"));
    KDA_TRY(need(k, "k"));
    KDA_TRY(need(v, "v"));
    KDA_TRY(need(g, "g"));
    KDA_TRY(need4(beta, "beta"));
    KDA_TRY(need(state_in, "state_in"));
    KDA_TRY(need4(accept, "accept"));
    KDA_TRY(need(out, "out"));
    KDA_TRY(need(state_out, "state_out"));
    if (state_in == state_out) return fail(KDA_ERR_INVALID, "state_out must not alias state_in%s");
    cudaError_t err = kda::launch_verify(q, k, v, g, beta, state_in, accept, N, K, dims.H,
                                         dims.d_k, (kda_dtype)dims.qkv_dtype, out, state_out,
                                         static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "verify launch");
    return KDA_OK;
}

kda_status kda_output_gate(const void *o, const void *z, const float *weight, int64_t T,
                           kda_dims dims, float eps, void *y, void *stream) {
    g_last_error[0] = '\0';
    KDA_TRY(check_dims(dims));
    if (T < 0) return fail(KDA_ERR_INVALID, "T must be >= 0%s");
    if (!(eps >= 0.f)) return fail(KDA_ERR_INVALID, "eps must be >= 0%s");
    if (T == 0) return KDA_OK;
    KDA_TRY(need(o, "o"));
    KDA_TRY(need(z, "z"));
    KDA_TRY(maybe(weight, "weight"));
    KDA_TRY(need(y, "y"));
    cudaError_t err = kda::launch_output_gate(o, z, weight, T * dims.H, dims.d_k,
                                              (kda_dtype)dims.qkv_dtype, eps, y,
                                              static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "output gate launch");
    return KDA_OK;
}

kda_status kda_selftest_wait(int64_t limit_ns, void *workspace, size_t workspace_bytes,
                             void *stream) {
    g_last_error[0] = '\0';
    if (limit_ns < 0 || limit_ns > 1000000000)
        return fail(KDA_ERR_INVALID, "limit_ns must be in [0, 1e9]%s");
    KDA_TRY(need(workspace, "workspace"));
    if (workspace_bytes < kStatusBytes) return fail(KDA_ERR_INVALID, "workspace too small%s");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t *status = static_cast<int32_t *>(workspace);
    cudaError_t err = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
    if (err == cudaSuccess) err = kda::launch_selftest_wait((uint64_t)limit_ns, status, s);
    if (err != cudaSuccess) return cuda_fail(err, "self-test launch");
    return KDA_OK;
}

kda_status kda_get_device_status(const void *workspace, int32_t *status_out,
                                 void *stream) {
    g_last_error[0] = '\0';
    if (workspace == nullptr || status_out == nullptr)
        return fail(KDA_ERR_INVALID, "workspace and status_out must not be NULL%s");
    int32_t word = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess) err = cudaStreamSynchronize(s);
    if (err != cudaSuccess) return cuda_fail(err, "reading the status word");
    *status_out = word;
    if (word == KDA_DEVICE_OK) return KDA_OK;
    if (word == KDA_DEVICE_TIMEOUT)
        return fail(KDA_ERR_TIMEOUT, "a device-side wait gave up%s");
    if (word == KDA_DEVICE_RANGE)
        return fail(KDA_ERR_DEVICE, "a value held in fp16 operands reached 65504 in magnitude%s");
    if (word == KDA_DEVICE_BAD_SNAPSHOT)
        return fail(KDA_ERR_DEVICE, "a snapshot offset is out of range, out of order or misaligned%s");
    return fail(KDA_ERR_DEVICE, "the device rejected cu_seqlens (not 0..T, non-decreasing)%s");
}

}  // extern "C"
