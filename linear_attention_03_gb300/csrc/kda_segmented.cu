// kda_segmented.cu -- prefill of one long document as independent segments,
// joined by an exact scan of their affine state maps.
//
// "From GPT-2 to Kimi K3, from first principles", Chapter 6 (context
// parallelism): over a segment the state evolves as S_out = P S_in + R, with
// P the product of the segment's transitions (I - beta k k^T) Diag(alpha) and
// R the state reached from zero, and such maps compose as
// (P2, R2) o (P1, R1) = (P2 P1, P2 R1 + R2).  The recurrence is linear in the
// pair (v, S_in), so every quantity comes out of plain prefills of the
// segments, each an independent document:
//   1. v as given, segment 0 from init_state and the others from 0:
//      outputs o^0 and the states R_s;
//   2. v = 0 from the identity: the states P_s;
//   3. the scan S_1 = R_0, S_{s+1} = P_s S_s + R_s (S_end = final state);
//   4. v = 0 from S_s: the outputs the incoming state adds, o = o^0 + o^S.
// With the tensor-core prefill (bf16 q/k/v) o^0 and o^S are kept in fp32 and
// the sum is rounded to bf16 once.
// It costs three prefills instead of one, spread over segments x heads CTAs:
// it pays off when heads x documents alone cannot fill the GPU.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct SegLayout {
    int32_t nseg;
    int64_t seg_len;
    size_t status, cu, v0, init0, ident, R, P, Sin, ocorr, o0f, total;
};

// fp32 partial outputs: the tensor-core prefill (bf16 inputs, d = 128)
bool f32_partials(int32_t D, kda_dtype dt) { return chunk_prefill_supported(D, dt); }

SegLayout layout(int32_t H, int32_t D, kda_dtype dt, int64_t T, int32_t num_segments) {
    SegLayout L{};
    const int64_t chunks = (T + 63) / 64;
    int64_t per = num_segments > 0 ? (chunks + num_segments - 1) / num_segments : chunks;
    if (per < 1) per = 1;
    L.seg_len = per * 64;
    L.nseg = T > 0 ? static_cast<int32_t>((T + L.seg_len - 1) / L.seg_len) : 1;
    const size_t esz = dt == KDA_BF16 ? 2 : 4;
    const size_t tok = static_cast<size_t>(T) * H * D * esz;
    const size_t st = static_cast<size_t>(L.nseg) * H * D * D * sizeof(float);
    size_t off = 0;
    L.status = off; off += up(4);
    L.cu = off; off += up(static_cast<size_t>(L.nseg + 1) * sizeof(int32_t));
    L.v0 = off; off += up(tok);
    L.init0 = off; off += up(st);
    L.ident = off; off += up(st);
    L.R = off; off += up(st);
    L.P = off; off += up(st);
    L.Sin = off; off += up(st);
    const size_t tokf = static_cast<size_t>(T) * H * D * sizeof(float);
    L.ocorr = off; off += up(f32_partials(D, dt) ? tokf : tok);
    L.o0f = off; off += f32_partials(D, dt) ? up(tokf) : 0;
    L.total = off;
    return L;
}

// segment offsets and identity states
__global__ void seg_setup_kernel(int32_t *cu, int32_t nseg, int64_t seg_len, int64_t T, float *ident,
                                 int64_t nmat, int32_t D) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i <= nseg) {
        const int64_t o = i * seg_len;
        cu[i] = static_cast<int32_t>(o < T ? o : T);
    }
    const int64_t n = nmat * D * D;
    for (int64_t e = i; e < n; e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = (e / D) % D, c = e % D;
        ident[e] = r == c ? 1.f : 0.f;
    }
}

// Per head: S = R_0; for s >= 1: Sin_s = S, S = P_s S + R_s; final = S.
// One CTA of 256 threads per head, each thread an 8x8 block of the product;
// P_s is staged transposed and S row-major in shared memory (2 x D x D fp32).
template <int D>
__global__ void __launch_bounds__(256) seg_scan_kernel(const float *__restrict__ R,
                                                       const float *__restrict__ P, float *Sin,
                                                       float *final_state, int32_t nseg, int32_t H) {
    extern __shared__ float smem[];
    float *Pt = smem;          // Pt[k * D + i] = P[i][k]
    float *S = smem + D * D;   // S[k * D + j]
    const int h = blockIdx.x, tid = threadIdx.x;
    constexpr int TB = D / 8;  // thread blocks of 8 x 8 per dimension (D = 128: 16)
    const size_t mat = static_cast<size_t>(D) * D;
    const float *R0 = R + static_cast<size_t>(h) * mat;
    for (int e = tid; e < D * D; e += 256) S[e] = R0[e];
    __syncthreads();
    for (int s = 1; s < nseg; ++s) {
        const float *Ps = P + (static_cast<size_t>(s) * H + h) * mat;
        const float *Rs = R + (static_cast<size_t>(s) * H + h) * mat;
        float *Sout = Sin + (static_cast<size_t>(s) * H + h) * mat;
        for (int e = tid; e < D * D; e += 256) {
            Sout[e] = S[e];                           // the state entering segment s
            Pt[e] = Ps[(e % D) * D + e / D];          // contiguous shared-memory writes
        }
        __syncthreads();
        const bool act = tid < TB * TB;
        const int i0 = 8 * (tid / TB), j0 = 8 * (tid % TB);
        float acc[8][8];
        if (act) {
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) acc[a][b] = Rs[(i0 + a) * D + j0 + b];
            for (int k = 0; k < D; ++k) {
                float pc[8], sr[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) pc[a] = Pt[k * D + i0 + a];
#pragma unroll
                for (int b = 0; b < 8; ++b) sr[b] = S[k * D + j0 + b];
#pragma unroll
                for (int a = 0; a < 8; ++a)
#pragma unroll
                    for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(pc[a], sr[b], acc[a][b]);
            }
        }
        __syncthreads();   // every read of S is done: the new state replaces it
        if (act) {
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) S[(i0 + a) * D + j0 + b] = acc[a][b];
        }
        __syncthreads();
    }
    if (final_state != nullptr) {
        float *F = final_state + static_cast<size_t>(h) * mat;
        for (int e = tid; e < D * D; e += 256) F[e] = S[e];
    }
}

// out = bf16(o^0 + o^S), the partial outputs in fp32
__global__ void sum_partials_kernel(__nv_bfloat16 *out, const float *o0, const float *os, int64_t n) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t e = 4 * i; e < n; e += 4 * static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 a = *reinterpret_cast<const float4 *>(o0 + e);
        const float4 b = *reinterpret_cast<const float4 *>(os + e);
        __nv_bfloat162 lo = __floats2bfloat162_rn(a.x + b.x, a.y + b.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(a.z + b.z, a.w + b.w);
        *reinterpret_cast<__nv_bfloat162 *>(out + e) = lo;
        *reinterpret_cast<__nv_bfloat162 *>(out + e + 2) = hi;
    }
}

// out += o^S for the tokens after segment 0 (segment 0's correction is zero)
template <typename T>
__global__ void add_correction_kernel(T *out, const T *corr, int64_t begin, int64_t n) {
    const int64_t i = begin + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t e = i; e < n; e += static_cast<int64_t>(gridDim.x) * blockDim.x)
        Elem<T>::store(out + e, Elem<T>::load(out + e) + Elem<T>::load(corr + e));
}

}  // namespace

size_t segmented_workspace_size(int32_t H, int32_t D, kda_dtype dt, int64_t T, int32_t num_segments) {
    return layout(H, D, dt, T, num_segments).total;
}

cudaError_t launch_prefill_segmented(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, const float *init_state, int64_t T, int32_t H,
                                     int32_t D, kda_dtype dt, int32_t num_segments, void *out,
                                     float *final_state, void *workspace, bool use_chunk,
                                     cudaStream_t s) {
    const SegLayout L = layout(H, D, dt, T, num_segments);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    int32_t *cu = reinterpret_cast<int32_t *>(ws + L.cu);
    void *v0 = ws + L.v0;
    float *init0 = reinterpret_cast<float *>(ws + L.init0);
    float *ident = reinterpret_cast<float *>(ws + L.ident);
    float *R = reinterpret_cast<float *>(ws + L.R);
    float *P = reinterpret_cast<float *>(ws + L.P);
    float *Sin = reinterpret_cast<float *>(ws + L.Sin);
    void *ocorr = ws + L.ocorr;
    const size_t esz = dt == KDA_BF16 ? 2 : 4;
    const size_t tokbytes = static_cast<size_t>(T) * H * D * esz;
    const size_t mat = static_cast<size_t>(D) * D * sizeof(float);
    const size_t st = static_cast<size_t>(L.nseg) * H * mat;
    const int32_t n = L.nseg;

    cudaError_t e;
    if ((e = cudaMemsetAsync(status, 0, 4, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(v0, 0, tokbytes, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(init0, 0, st, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(Sin, 0, st, s)) != cudaSuccess) return e;
    if (init_state != nullptr &&
        (e = cudaMemcpyAsync(init0, init_state, static_cast<size_t>(H) * mat, cudaMemcpyDeviceToDevice,
                             s)) != cudaSuccess)
        return e;
    seg_setup_kernel<<<592, 256, 0, s>>>(cu, n, L.seg_len, T, ident, static_cast<int64_t>(n) * H, D);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const bool f32p = use_chunk && f32_partials(D, dt);
    float *o0f = f32p ? reinterpret_cast<float *>(ws + L.o0f) : nullptr;
    auto prefill = [&](const void *vv, const float *init, void *o, float *fin, float *of) {
        return use_chunk ? launch_prefill_chunk(q, k, vv, g, beta, init, cu, n, T, H, o, fin, status, s,
                                                nullptr, of)
                         : launch_prefill_recurrent(q, k, vv, g, beta, init, cu, n, T, H, D, dt, o, fin,
                                                    status, s);
    };
    // 1. outputs from zero state (segment 0 from init_state) and the states R_s
    if ((e = prefill(v, init0, out, R, n > 1 ? o0f : nullptr)) != cudaSuccess) return e;
    if (n == 1) {
        if (final_state != nullptr &&
            (e = cudaMemcpyAsync(final_state, R, static_cast<size_t>(H) * mat, cudaMemcpyDeviceToDevice,
                                 s)) != cudaSuccess)
            return e;
        return cudaSuccess;
    }
    // 2. the transition maps P_s (v = 0 from the identity); the outputs are scratch
    if ((e = prefill(v0, ident, ocorr, P, f32p ? static_cast<float *>(ocorr) : nullptr)) != cudaSuccess)
        return e;
    // 3. the states entering each segment, and the final state
    const size_t scan_smem = 2 * mat;
    switch (D) {
    case 16: seg_scan_kernel<16><<<H, 256, scan_smem, s>>>(R, P, Sin, final_state, n, H); break;
    case 32: seg_scan_kernel<32><<<H, 256, scan_smem, s>>>(R, P, Sin, final_state, n, H); break;
    case 64: seg_scan_kernel<64><<<H, 256, scan_smem, s>>>(R, P, Sin, final_state, n, H); break;
    case 128: {
        static std::atomic<uint64_t> smem_set{0};
        if ((e = allow_dynamic_smem(seg_scan_kernel<128>, scan_smem, smem_set)) != cudaSuccess) return e;
        seg_scan_kernel<128><<<H, 256, scan_smem, s>>>(R, P, Sin, final_state, n, H);
        break;
    }
    default: return cudaErrorInvalidValue;
    }
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 4. what the incoming states add to the outputs (v = 0 from S_s), then the sum
    if ((e = prefill(v0, Sin, ocorr, nullptr, f32p ? static_cast<float *>(ocorr) : nullptr)) != cudaSuccess)
        return e;
    const int64_t begin = L.seg_len * H * D, total = T * H * D;
    if (f32p)
        sum_partials_kernel<<<2048, 256, 0, s>>>(static_cast<__nv_bfloat16 *>(out), o0f,
                                                 static_cast<const float *>(ocorr), total);
    else if (dt == KDA_BF16)
        add_correction_kernel<__nv_bfloat16><<<2048, 256, 0, s>>>(
            static_cast<__nv_bfloat16 *>(out), static_cast<const __nv_bfloat16 *>(ocorr), begin, total);
    else
        add_correction_kernel<float><<<2048, 256, 0, s>>>(static_cast<float *>(out),
                                                          static_cast<const float *>(ocorr), begin, total);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
