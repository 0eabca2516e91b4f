// kda_pipeline.cu -- the KDA layer's input path and recurrence for one long
// document, segment by segment: the prologue of segment s + 1 (ShortConv,
// Swish, L2 norm and the gates of "An infra-oriented diagram of Kimi K3",
// KDA card) runs while the prefill of segment s ("From GPT-2 to Kimi K3",
// Chapter 6, chunk mode) runs, and the fp32 state is carried from segment to
// segment.  The prefill of one head is a serial chain that leaves SMs idle;
// the prologue, which streams HBM, fills them.  The intermediate q, k, v, g
// and beta live in two segment-sized buffers instead of T-sized ones.
//
// Ordering: the caller owns both streams.  The prefills run on the caller's
// `stream`, the prologues on `pro` (the caller's second stream, normally of
// lower priority); `pro` starts after the work already queued on `stream`, and
// since the last prefill waits for the last prologue, `stream` holds the end
// of the whole call.  The cross-stream events are created by the call and
// destroyed before it returns (CUDA releases them once their work is done),
// so nothing outlives the call.  With pro == stream the segments run one
// after another.
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

// the call's events, destroyed when the call returns
struct CallEvents {
    cudaEvent_t ev[5] = {};   // start, pro_done[2], pre_done[2]
    cudaError_t create() {
        for (auto &e : ev) {
            const cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
            if (r != cudaSuccess) return r;
        }
        return cudaSuccess;
    }
    ~CallEvents() {
        for (auto e : ev)
            if (e != nullptr) cudaEventDestroy(e);
    }
};

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
                                    cudaStream_t user, cudaStream_t pro) {
    const int64_t L = seg_tokens_of(T, segment_tokens);
    const Ring R = ring_layout(H, D, dt, L);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    uint8_t *ring[2] = {ws + kAlign, ws + kAlign + R.bytes};
    float *state = reinterpret_cast<float *>(ws + kAlign + 2 * R.bytes);
    const size_t sbytes = static_cast<size_t>(H) * D * D * sizeof(float);
    const size_t esz = dt == KDA_BF16 ? 2 : 4;

    CallEvents E;
    cudaError_t e = E.create();
    if (e != cudaSuccess) return e;
    cudaEvent_t start = E.ev[0], pro_done[2] = {E.ev[1], E.ev[2]}, pre_done[2] = {E.ev[3], E.ev[4]};

    if ((e = cudaMemsetAsync(status, 0, 4, user)) != cudaSuccess) return e;
    e = init_state ? cudaMemcpyAsync(state, init_state, sbytes, cudaMemcpyDeviceToDevice, user)
                   : cudaMemsetAsync(state, 0, sbytes, user);
    if (e != cudaSuccess) return e;
    if ((e = cudaEventRecord(start, user)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(pro, start, 0)) != cudaSuccess) return e;

    const int64_t nseg = (T + L - 1) / L;
    for (int64_t s = 0; s < nseg; ++s) {
        const int b = static_cast<int>(s & 1);
        const int64_t tb = s * L, te = tb + L < T ? tb + L : T;
        uint8_t *r = ring[b];
        // the prologue of segment s into buffer b, once segment s - 2's prefill has read it
        if (s >= 2 && (e = cudaStreamWaitEvent(pro, pre_done[b], 0)) != cudaSuccess) return e;
        e = launch_prologue_range(q_raw, k_raw, v_raw, conv_w, z_g, z_beta, nullptr, 1, T, tb, te, H, D,
                                  dt, r + R.q, r + R.k, r + R.v, reinterpret_cast<float *>(r + R.g),
                                  reinterpret_cast<float *>(r + R.beta), pro);
        if (e != cudaSuccess) return e;
        if ((e = cudaEventRecord(pro_done[b], pro)) != cudaSuccess) return e;
        // its prefill, continuing the state
        if ((e = cudaStreamWaitEvent(user, pro_done[b], 0)) != cudaSuccess) return e;
        void *o = static_cast<uint8_t *>(out) + static_cast<size_t>(tb) * H * D * esz;
        const float *gp = reinterpret_cast<const float *>(r + R.g);
        const float *bp = reinterpret_cast<const float *>(r + R.beta);
        e = use_chunk ? launch_prefill_chunk(r + R.q, r + R.k, r + R.v, gp, bp, state, nullptr, 1, te - tb,
                                             H, o, state, status, user)
                      : launch_prefill_recurrent(r + R.q, r + R.k, r + R.v, gp, bp, state, nullptr, 1,
                                                 te - tb, H, D, dt, o, state, status, user);
        if (e != cudaSuccess) return e;
        if ((e = cudaEventRecord(pre_done[b], user)) != cudaSuccess) return e;
    }
    if (final_state != nullptr &&
        (e = cudaMemcpyAsync(final_state, state, sbytes, cudaMemcpyDeviceToDevice, user)) != cudaSuccess)
        return e;
    return cudaSuccess;
}

}  // namespace kda
