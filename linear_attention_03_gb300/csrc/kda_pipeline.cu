// kda_pipeline.cu -- the KDA layer's input path and recurrence for one long
// document, segment by segment: the prologue of segment s + 1 (ShortConv,
// Swish, L2 norm and the gates of "An infra-oriented diagram of Kimi K3",
// KDA card) runs while the prefill of segment s ("From GPT-2 to Kimi K3",
// Chapter 6, chunk mode) runs, and the fp32 state is carried from segment to
// segment.  The prefill of one head is a serial chain that leaves SMs idle;
// the prologue, which streams HBM, fills them.  The intermediate q, k, v, g
// and beta live in two segment-sized buffers instead of T-sized ones.
//
// Ordering: two library streams per device, the prefills on the higher
// priority one.  Both start after the work already queued on the caller's
// stream, and the caller's stream waits for the last prefill.
#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Ring {
    size_t q, k, v, g, beta, bytes;
};

Ring ring_layout(int32_t H, int32_t D, kda_dtype dt, int64_t L) {
    const size_t esz = dt == KDA_BF16 ? 2 : 4;
    const size_t tok = static_cast<size_t>(L) * H * D;
    Ring r{};
    size_t off = 0;
    r.q = off; off += up(tok * esz);
    r.k = off; off += up(tok * esz);
    r.v = off; off += up(tok * esz);
    r.g = off; off += up(tok * sizeof(float));
    r.beta = off; off += up(static_cast<size_t>(L) * H * sizeof(float));
    r.bytes = off;
    return r;
}

int64_t seg_tokens_of(int64_t T, int64_t segment_tokens) {
    int64_t L = segment_tokens < 64 ? 64 : segment_tokens;
    L = (L + 63) / 64 * 64;
    return T > 0 && L > T ? (T + 63) / 64 * 64 : L;
}

// library streams and events of one device, created on first use; a call
// holds the device's lock while it enqueues, so calls from several host
// threads do not interleave on them
struct DeviceQueues {
    std::mutex mu;
    cudaStream_t pro = nullptr, pre = nullptr;
    cudaEvent_t start = nullptr, end = nullptr, pro_done[2] = {}, pre_done[2] = {};
    bool ready = false;
};

DeviceQueues g_queues[64];

// with q.mu held
cudaError_t queues_ready(DeviceQueues &q) {
    if (!q.ready) {
        int lo = 0, hi = 0;
        cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&q.pro, cudaStreamNonBlocking, lo);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&q.pre, cudaStreamNonBlocking, hi);
        cudaEvent_t *evs[6] = {&q.start, &q.end, &q.pro_done[0], &q.pro_done[1], &q.pre_done[0],
                               &q.pre_done[1]};
        for (int i = 0; i < 6 && e == cudaSuccess; ++i)
            e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        q.ready = true;
    }
    return cudaSuccess;
}

}  // namespace

size_t pipeline_workspace_size(int32_t H, int32_t D, kda_dtype dt, int64_t T, int64_t segment_tokens) {
    const int64_t L = seg_tokens_of(T, segment_tokens);
    return kAlign + 2 * ring_layout(H, D, dt, L).bytes + up(static_cast<size_t>(H) * D * D * sizeof(float));
}

cudaError_t launch_prologue_prefill(const void *q_raw, const void *k_raw, const void *v_raw,
                                    const float *conv_w, const float *z_g, const float *z_beta,
                                    const float *init_state, int64_t T, int32_t H, int32_t D,
                                    kda_dtype dt, int64_t segment_tokens, void *out,
                                    float *final_state, void *workspace, bool use_chunk,
                                    cudaStream_t user) {
    const int64_t L = seg_tokens_of(T, segment_tokens);
    const Ring R = ring_layout(H, D, dt, L);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    uint8_t *ring[2] = {ws + kAlign, ws + kAlign + R.bytes};
    float *state = reinterpret_cast<float *>(ws + kAlign + 2 * R.bytes);
    const size_t sbytes = static_cast<size_t>(H) * D * D * sizeof(float);
    const size_t esz = dt == KDA_BF16 ? 2 : 4;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DeviceQueues *Q = &g_queues[dev];
    std::lock_guard<std::mutex> lock(Q->mu);
    if ((e = queues_ready(*Q)) != cudaSuccess) return e;

    if ((e = cudaMemsetAsync(status, 0, 4, user)) != cudaSuccess) return e;
    e = init_state ? cudaMemcpyAsync(state, init_state, sbytes, cudaMemcpyDeviceToDevice, user)
                   : cudaMemsetAsync(state, 0, sbytes, user);
    if (e != cudaSuccess) return e;
    if ((e = cudaEventRecord(Q->start, user)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(Q->pro, Q->start, 0)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(Q->pre, Q->start, 0)) != cudaSuccess) return e;

    const int64_t nseg = (T + L - 1) / L;
    for (int64_t s = 0; s < nseg; ++s) {
        const int b = static_cast<int>(s & 1);
        const int64_t tb = s * L, te = tb + L < T ? tb + L : T;
        uint8_t *r = ring[b];
        // the prologue of segment s into buffer b, once segment s - 2's prefill has read it
        if (s >= 2 && (e = cudaStreamWaitEvent(Q->pro, Q->pre_done[b], 0)) != cudaSuccess) return e;
        e = launch_prologue_range(q_raw, k_raw, v_raw, conv_w, z_g, z_beta, nullptr, 1, T, tb, te, H, D,
                                  dt, r + R.q, r + R.k, r + R.v, reinterpret_cast<float *>(r + R.g),
                                  reinterpret_cast<float *>(r + R.beta), Q->pro);
        if (e != cudaSuccess) return e;
        if ((e = cudaEventRecord(Q->pro_done[b], Q->pro)) != cudaSuccess) return e;
        // its prefill, continuing the state
        if ((e = cudaStreamWaitEvent(Q->pre, Q->pro_done[b], 0)) != cudaSuccess) return e;
        void *o = static_cast<uint8_t *>(out) + static_cast<size_t>(tb) * H * D * esz;
        const float *gp = reinterpret_cast<const float *>(r + R.g);
        const float *bp = reinterpret_cast<const float *>(r + R.beta);
        e = use_chunk ? launch_prefill_chunk(r + R.q, r + R.k, r + R.v, gp, bp, state, nullptr, 1, te - tb,
                                             H, o, state, status, Q->pre)
                      : launch_prefill_recurrent(r + R.q, r + R.k, r + R.v, gp, bp, state, nullptr, 1,
                                                 te - tb, H, D, dt, o, state, status, Q->pre);
        if (e != cudaSuccess) return e;
        if ((e = cudaEventRecord(Q->pre_done[b], Q->pre)) != cudaSuccess) return e;
    }
    if (final_state != nullptr &&
        (e = cudaMemcpyAsync(final_state, state, sbytes, cudaMemcpyDeviceToDevice, Q->pre)) != cudaSuccess)
        return e;
    if ((e = cudaEventRecord(Q->end, Q->pre)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(user, Q->end, 0);
}

}  // namespace kda
