// kda_prefill_recurrent.cu -- token-serial KDA prefill on CUDA cores, fp32.
//
// This is the fused-recurrent form of the recurrence ("Kimi K3 Architecture
// Explained", Step 3; "From GPT-2 to Kimi K3, from first principles",
// Chapter 6 names it fused_recurrent).  It serves every head size and fp32
// inputs (where tensor-core bf16 operands would not meet fp32 accuracy), and
// is the exact-arithmetic companion of the tensor-core chunked prefill.
//
// One CTA per (head, document); thread j owns column j of the d x d state
// in D registers, so both column reductions of a token are private to the
// thread (no synchronisation inside the token loop):
//     a_j = sum_i alpha_i k_i S_ij,  b_j = sum_i alpha_i q_i S_ij   (old S)
//     u_j = beta (v_j - a_j),  o_j = b_j + u_j (k . q),
//     S_ij <- alpha_i S_ij + k_i u_j.
// Token inputs are staged through shared memory TT tokens at a time; every
// thread then reads the same address (broadcast).  Prefix snapshots are
// written from the registers at stage boundaries (every snapshot offset is
// a multiple of 64 tokens into its document, or its end).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kStage = 16;   // tokens staged per pass

template <typename Tin, int D>
__global__ void __launch_bounds__(D)
recurrent_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                 const Tin *__restrict__ v, const float *__restrict__ g,
                 const float *__restrict__ beta, const float *init_state,
                 const int32_t *__restrict__ cu, int32_t N, int64_t T, int32_t H,
                 Tin *__restrict__ out, float *final_state,
                 int32_t *__restrict__ status, const int32_t *__restrict__ order, Snapshots snaps) {
    constexpr int NW = (D + 31) / 32;
    constexpr int LANES = D < 32 ? D : 32;           // lanes of a (partial) warp
    constexpr unsigned MASK = D < 32 ? ((1u << D) - 1u) : 0xffffffffu;
    const int h = blockIdx.x;
    const int n = order ? order[blockIdx.y] : static_cast<int>(blockIdx.y);   // longest first
    const int j = threadIdx.x;
    int64_t bos, eos;
    if (!doc_bounds(cu, n, N, T, bos, eos)) {
        if (j == 0) flag_status(status, KDA_DEVICE_BAD_OFFSETS);
        return;
    }

    __shared__ __align__(16) float s_ka[kStage][D];
    __shared__ __align__(16) float s_qa[kStage][D];
    __shared__ __align__(16) float s_al[kStage][D];
    __shared__ __align__(16) float s_k[kStage][D];
    __shared__ float s_v[kStage][D];
    __shared__ float s_beta[kStage];
    __shared__ float s_kqp[kStage][NW];

    const size_t unit = (size_t)n * H + h;
    float S[D];
#pragma unroll
    for (int i = 0; i < D; ++i)
        S[i] = init_state ? init_state[unit * D * D + (size_t)i * D + j] : 0.f;
    // the document's next snapshot: its state after the tokens before offsets[snap]
    int32_t snap = snaps.n > 0 ? snap_first(snaps, bos) : 0;
    auto take_snapshot = [&](int64_t at) {
        if (snap < snaps.n && static_cast<int64_t>(snaps.offsets[snap]) == at) {
            float *dst = snaps.out + ((size_t)snap * H + h) * D * D + j;
#pragma unroll
            for (int i = 0; i < D; ++i) dst[(size_t)i * D] = S[i];
            ++snap;
        }
    };

    for (int64_t t0 = bos; t0 < eos; t0 += kStage) {
        const int cnt = (int)((eos - t0) < kStage ? (eos - t0) : kStage);
        if (t0 > bos) take_snapshot(t0);
        __syncthreads();
        for (int tt = 0; tt < cnt; ++tt) {
            const size_t row = (size_t)(t0 + tt) * H + h;
            const float kk = Elem<Tin>::load(k + row * D + j);
            const float qq = Elem<Tin>::load(q + row * D + j);
            const float a = __expf(g[row * D + j]);
            s_k[tt][j] = kk;
            s_ka[tt][j] = a * kk;
            s_qa[tt][j] = a * qq;
            s_al[tt][j] = a;
            s_v[tt][j] = Elem<Tin>::load(v + row * D + j);
            float p = kk * qq;
#pragma unroll
            for (int o = LANES / 2; o > 0; o >>= 1) p += __shfl_xor_sync(MASK, p, o, LANES);
            if ((j & 31) == 0) s_kqp[tt][j >> 5] = p;
            if (j == 0) s_beta[tt] = beta[row];
        }
        __syncthreads();
        for (int tt = 0; tt < cnt; ++tt) {
            float kq = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) kq += s_kqp[tt][w];
            float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
            for (int i = 0; i < D; i += 4) {
                const float4 ka = *reinterpret_cast<const float4 *>(&s_ka[tt][i]);
                const float4 qa = *reinterpret_cast<const float4 *>(&s_qa[tt][i]);
                a0 += ka.x * S[i] + ka.y * S[i + 1];
                a1 += ka.z * S[i + 2] + ka.w * S[i + 3];
                b0 += qa.x * S[i] + qa.y * S[i + 1];
                b1 += qa.z * S[i + 2] + qa.w * S[i + 3];
            }
            const float u = s_beta[tt] * (s_v[tt][j] - (a0 + a1));
            const size_t row = (size_t)(t0 + tt) * H + h;
            Elem<Tin>::store(out + row * D + j, (b0 + b1) + u * kq);
#pragma unroll
            for (int i = 0; i < D; i += 4) {
                const float4 al = *reinterpret_cast<const float4 *>(&s_al[tt][i]);
                const float4 kk = *reinterpret_cast<const float4 *>(&s_k[tt][i]);
                S[i] = al.x * S[i] + kk.x * u;
                S[i + 1] = al.y * S[i + 1] + kk.y * u;
                S[i + 2] = al.z * S[i + 2] + kk.z * u;
                S[i + 3] = al.w * S[i + 3] + kk.w * u;
            }
        }
    }
    if (eos > bos) take_snapshot(eos);
    if (final_state) {
#pragma unroll
        for (int i = 0; i < D; ++i) final_state[unit * D * D + (size_t)i * D + j] = S[i];
    }
}

template <typename Tin, int D>
cudaError_t run(const void *q, const void *k, const void *v, const float *g,
                const float *beta, const float *init_state, const int32_t *cu,
                int32_t N, int64_t T, int32_t H, void *out, float *final_state,
                int32_t *status, cudaStream_t stream, const int32_t *order, Snapshots snaps) {
    recurrent_kernel<Tin, D><<<dim3(H, N), D, 0, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k),
        static_cast<const Tin *>(v), g, beta, init_state, cu, N, T, H,
        static_cast<Tin *>(out), final_state, status, order, snaps);
    count_launches(1);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t run_d(const void *q, const void *k, const void *v, const float *g,
                  const float *beta, const float *init_state, const int32_t *cu,
                  int32_t N, int64_t T, int32_t H, int32_t D, void *out,
                  float *final_state, int32_t *status, cudaStream_t stream, const int32_t *order,
                  Snapshots snaps) {
    switch (D) {
    case 16: return run<Tin, 16>(q, k, v, g, beta, init_state, cu, N, T, H, out, final_state, status, stream, order, snaps);
    case 32: return run<Tin, 32>(q, k, v, g, beta, init_state, cu, N, T, H, out, final_state, status, stream, order, snaps);
    case 64: return run<Tin, 64>(q, k, v, g, beta, init_state, cu, N, T, H, out, final_state, status, stream, order, snaps);
    case 128: return run<Tin, 128>(q, k, v, g, beta, init_state, cu, N, T, H, out, final_state, status, stream, order, snaps);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prefill_recurrent(const void *q, const void *k,
                                     const void *v, const float *g,
                                     const float *beta, const float *init_state,
                                     const int32_t *cu_seqlens, int32_t N,
                                     int64_t T, int32_t H, int32_t D,
                                     kda_dtype dt, void *out,
                                     float *final_state, int32_t *status,
                                     cudaStream_t stream, const int32_t *order, Snapshots snaps) {
    if (dt == KDA_BF16)
        return run_d<__nv_bfloat16>(q, k, v, g, beta, init_state, cu_seqlens, N, T, H, D,
                                    out, final_state, status, stream, order, snaps);
    return run_d<float>(q, k, v, g, beta, init_state, cu_seqlens, N, T, H, D, out,
                        final_state, status, stream, order, snaps);
}

namespace {

// one thread per offset: in (0, T], above its predecessor, and a multiple of
// KDA_SNAPSHOT_ALIGN into the document with bos < p <= eos, or that eos
__global__ void snapshot_check_kernel(const int32_t *__restrict__ offsets, int32_t n,
                                      const int32_t *__restrict__ cu, int32_t N, int64_t T,
                                      int32_t *__restrict__ status) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int64_t p = offsets[i];
    bool ok = p > 0 && p <= T && (i == 0 || static_cast<int64_t>(offsets[i - 1]) < p);
    if (ok) {
        int64_t bos = 0, eos = T;
        if (cu != nullptr) {
            // the first document end at or past p: its document holds p
            int32_t lo = 0, hi = N;
            while (lo < hi) {
                const int32_t mid = (lo + hi) >> 1;
                if (static_cast<int64_t>(cu[mid + 1]) < p) lo = mid + 1; else hi = mid;
            }
            if (lo >= N) {
                ok = false;
            } else {
                bos = cu[lo];
                eos = cu[lo + 1];
            }
        }
        ok = ok && bos < p && p <= eos && ((p - bos) % KDA_SNAPSHOT_ALIGN == 0 || p == eos);
    }
    if (!ok) flag_status(status, KDA_DEVICE_BAD_SNAPSHOT);
}

}  // namespace

cudaError_t launch_snapshot_check(const int32_t *offsets, int32_t n, const int32_t *cu_seqlens,
                                  int32_t N, int64_t T, int32_t *status, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    snapshot_check_kernel<<<(n + 255) / 256, 256, 0, stream>>>(offsets, n, cu_seqlens, N, T, status);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
