// kda_decode.cu -- single-token KDA step for N independent sequences
// ("fused_recurrent" mode, "From GPT-2 to Kimi K3, from first principles",
// Chapter 6), bandwidth-bound: each fp32 state is read once and written once.
//
// With R = Diag(alpha) S the recurrence of "Kimi K3 Architecture Explained",
// Step 3, multiplies out to S' = R + k u^T with u = beta (v - R^T k), and the
// read after the update is o = S'^T q = R^T q + u (k . q).  Both column
// reductions, a_j = sum_i alpha_i k_i S_ij and b_j = sum_i alpha_i q_i S_ij,
// use the OLD state, so one pass over S yields everything:
//     u_j = beta (v_j - a_j),  o_j = b_j + u_j (k . q),
//     S_ij <- alpha_i S_ij + k_i u_j      (written in place)
//
// Layout: one CTA per (sequence, head).  Thread (r, c) owns float4 column
// group c (columns 4c..4c+3) of rows r*ROWS .. r*ROWS+ROWS-1, so a warp
// reads whole 512-byte rows (D = 128): fully coalesced 16-byte accesses.
// Per-thread partial sums are combined across row groups in shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

template <typename Tin, int D>
struct DecodeCfg {
    static constexpr int COLG = D / 4;                 // float4 column groups
    static constexpr int RG = 8;                       // row groups
    static constexpr int ROWS = D / RG;                // rows per thread
    static constexpr int THREADS = COLG * RG;
};

template <typename Tin, int D>
__global__ void __launch_bounds__(DecodeCfg<Tin, D>::THREADS)
decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
              const Tin *__restrict__ v, const float *__restrict__ g,
              const float *__restrict__ beta, float *__restrict__ state,
              Tin *__restrict__ out, int32_t H) {
    using C = DecodeCfg<Tin, D>;
    const int unit = blockIdx.x;             // sequence * H + head
    const int tid = threadIdx.x;
    const int c = tid % C::COLG;             // column group
    const int r = tid / C::COLG;             // row group

    __shared__ float s_ka[D];                // alpha_i k_i
    __shared__ float s_qa[D];                // alpha_i q_i
    __shared__ float s_alpha[D];
    __shared__ float s_k[D];
    __shared__ float s_kq[C::THREADS / 32];
    __shared__ float4 s_part[2][C::RG][C::COLG];

    float *S = state + (size_t)unit * D * D;
    const size_t vec = (size_t)unit * D;

    // issue the state loads first: 16-byte, coalesced, ROWS of them in flight
    float4 s[C::ROWS];
#pragma unroll
    for (int i = 0; i < C::ROWS; ++i)
        s[i] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)(r * C::ROWS + i) * D) + c);

    float kq = 0.f;
    for (int i = tid; i < D; i += C::THREADS) {
        const float ki = Elem<Tin>::load(k + vec + i);
        const float qi = Elem<Tin>::load(q + vec + i);
        const float a = __expf(g[vec + i]);
        s_alpha[i] = a;
        s_k[i] = ki;
        s_ka[i] = a * ki;
        s_qa[i] = a * qi;
        kq += ki * qi;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
    if ((tid & 31) == 0) s_kq[tid >> 5] = kq;
    __syncthreads();

    float4 pa = make_float4(0.f, 0.f, 0.f, 0.f), pb = pa;
#pragma unroll
    for (int i = 0; i < C::ROWS; ++i) {
        const int row = r * C::ROWS + i;
        const float ka = s_ka[row], qa = s_qa[row];
        pa.x += ka * s[i].x; pa.y += ka * s[i].y; pa.z += ka * s[i].z; pa.w += ka * s[i].w;
        pb.x += qa * s[i].x; pb.y += qa * s[i].y; pb.z += qa * s[i].z; pb.w += qa * s[i].w;
    }
    s_part[0][r][c] = pa;
    s_part[1][r][c] = pb;
    __syncthreads();

    // every thread needs u for its own 4 columns: sum the row groups
    float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f), b4 = a4;
#pragma unroll
    for (int j = 0; j < C::RG; ++j) {
        const float4 x = s_part[0][j][c], y = s_part[1][j][c];
        a4.x += x.x; a4.y += x.y; a4.z += x.z; a4.w += x.w;
        b4.x += y.x; b4.y += y.y; b4.z += y.z; b4.w += y.w;
    }
    float kq_all = 0.f;
#pragma unroll
    for (int w = 0; w < C::THREADS / 32; ++w) kq_all += s_kq[w];

    const float bt = beta[unit];
    float vv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) vv[j] = Elem<Tin>::load(v + vec + 4 * c + j);
    float4 u;
    u.x = bt * (vv[0] - a4.x); u.y = bt * (vv[1] - a4.y);
    u.z = bt * (vv[2] - a4.z); u.w = bt * (vv[3] - a4.w);

    if (r == 0) {
        Elem<Tin>::store(out + vec + 4 * c + 0, b4.x + u.x * kq_all);
        Elem<Tin>::store(out + vec + 4 * c + 1, b4.y + u.y * kq_all);
        Elem<Tin>::store(out + vec + 4 * c + 2, b4.z + u.z * kq_all);
        Elem<Tin>::store(out + vec + 4 * c + 3, b4.w + u.w * kq_all);
    }

#pragma unroll
    for (int i = 0; i < C::ROWS; ++i) {
        const int row = r * C::ROWS + i;
        const float a = s_alpha[row], ki = s_k[row];
        float4 x = s[i];
        x.x = a * x.x + ki * u.x; x.y = a * x.y + ki * u.y;
        x.z = a * x.z + ki * u.z; x.w = a * x.w + ki * u.w;
        __stcs(reinterpret_cast<float4 *>(S + (size_t)row * D) + c, x);
    }
}

template <typename Tin, int D>
cudaError_t run(const void *q, const void *k, const void *v, const float *g,
                const float *beta, float *state, void *out, int32_t N, int32_t H,
                cudaStream_t stream) {
    const unsigned units = (unsigned)N * (unsigned)H;
    if (units == 0) return cudaSuccess;
    decode_kernel<Tin, D><<<units, DecodeCfg<Tin, D>::THREADS, 0, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k),
        static_cast<const Tin *>(v), g, beta, state, static_cast<Tin *>(out), H);
    count_launches(1);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t run_d(const void *q, const void *k, const void *v, const float *g,
                  const float *beta, float *state, void *out, int32_t N,
                  int32_t H, int32_t D, cudaStream_t stream) {
    switch (D) {
    case 16: return run<Tin, 16>(q, k, v, g, beta, state, out, N, H, stream);
    case 32: return run<Tin, 32>(q, k, v, g, beta, state, out, N, H, stream);
    case 64: return run<Tin, 64>(q, k, v, g, beta, state, out, N, H, stream);
    case 128: return run<Tin, 128>(q, k, v, g, beta, state, out, N, H, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v,
                          const float *g, const float *beta, float *state,
                          void *out, int32_t N, int32_t H, int32_t D,
                          kda_dtype dt, cudaStream_t stream) {
    if (dt == KDA_BF16)
        return run_d<__nv_bfloat16>(q, k, v, g, beta, state, out, N, H, D, stream);
    return run_d<float>(q, k, v, g, beta, state, out, N, H, D, stream);
}

}  // namespace kda
