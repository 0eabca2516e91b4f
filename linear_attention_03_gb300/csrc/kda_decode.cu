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

// ---------------------------------------------------------------------------
// Shared pieces of the one-pass update used by the decode-with-conv and the
// multi-token verify kernels: the per-thread state tile is 16 rows x 4
// columns (D = 128) held as float4, the column reductions over the old state
// go through shared memory, and the update is written back in registers.

template <int D>
struct TokenSmem {
    float2 kqa[D];    // (alpha_i k_i, alpha_i q_i): one 8-byte read per state row
    float2 ak[D];     // (alpha_i, k_i)
    float v[D];
    float red[24];    // per-warp partial sums (k.q and the L2 norms)
    float kq, beta;
};

// Given a staged token (sm), produce o (written by row group 0) and update
// the register tile s in place.
template <typename Tin, int D>
__device__ __forceinline__ void token_update(float4 (&s)[DecodeCfg<Tin, D>::ROWS],
                                             const TokenSmem<D> &sm,
                                             float4 (&part)[2][DecodeCfg<Tin, D>::RG]
                                                           [DecodeCfg<Tin, D>::COLG],
                                             int r, int c, Tin *out_vec) {
    using C = DecodeCfg<Tin, D>;
    float4 pa = make_float4(0.f, 0.f, 0.f, 0.f), pb = pa;
#pragma unroll
    for (int i = 0; i < C::ROWS; ++i) {
        const int row = r * C::ROWS + i;
        const float2 w = sm.kqa[row];
        const float ka = w.x, qa = w.y;
        pa.x += ka * s[i].x; pa.y += ka * s[i].y; pa.z += ka * s[i].z; pa.w += ka * s[i].w;
        pb.x += qa * s[i].x; pb.y += qa * s[i].y; pb.z += qa * s[i].z; pb.w += qa * s[i].w;
    }
    part[0][r][c] = pa;
    part[1][r][c] = pb;
    __syncthreads();
    float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f), b4 = a4;
#pragma unroll
    for (int j = 0; j < C::RG; ++j) {
        const float4 x = part[0][j][c], y = part[1][j][c];
        a4.x += x.x; a4.y += x.y; a4.z += x.z; a4.w += x.w;
        b4.x += y.x; b4.y += y.y; b4.z += y.z; b4.w += y.w;
    }
    const float bt = sm.beta, kq = sm.kq;
    float4 u;
    u.x = bt * (sm.v[4 * c + 0] - a4.x); u.y = bt * (sm.v[4 * c + 1] - a4.y);
    u.z = bt * (sm.v[4 * c + 2] - a4.z); u.w = bt * (sm.v[4 * c + 3] - a4.w);
    if (r == 0) {
        Elem<Tin>::store(out_vec + 4 * c + 0, b4.x + u.x * kq);
        Elem<Tin>::store(out_vec + 4 * c + 1, b4.y + u.y * kq);
        Elem<Tin>::store(out_vec + 4 * c + 2, b4.z + u.z * kq);
        Elem<Tin>::store(out_vec + 4 * c + 3, b4.w + u.w * kq);
    }
#pragma unroll
    for (int i = 0; i < C::ROWS; ++i) {
        const int row = r * C::ROWS + i;
        const float2 f = sm.ak[row];
        const float a = f.x, ki = f.y;
        s[i].x = a * s[i].x + ki * u.x; s[i].y = a * s[i].y + ki * u.y;
        s[i].z = a * s[i].z + ki * u.z; s[i].w = a * s[i].w + ki * u.w;
    }
}

// Block-wide sums of three values per thread in one pass (all threads call it).
template <int THREADS>
__device__ __forceinline__ float3 block_sum3(float3 x, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        x.x += __shfl_xor_sync(0xffffffffu, x.x, o);
        x.y += __shfl_xor_sync(0xffffffffu, x.y, o);
        x.z += __shfl_xor_sync(0xffffffffu, x.z, o);
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        red[3 * (threadIdx.x >> 5)] = x.x;
        red[3 * (threadIdx.x >> 5) + 1] = x.y;
        red[3 * (threadIdx.x >> 5) + 2] = x.z;
    }
    __syncthreads();
    float3 t = make_float3(0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) {
        t.x += red[3 * w]; t.y += red[3 * w + 1]; t.z += red[3 * w + 2];
    }
    return t;
}

// Block-wide sum of one value per thread (all threads call it).
template <int THREADS>
__device__ __forceinline__ float block_sum(float x, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) t += red[w];
    return t;
}

// One decode step with the ShortConv cache ("From GPT-2 to Kimi K3",
// Chapter 5: the short convolution "is a short local preprocessor whose
// state must also be cached during decoding").  The prologue of the
// infra diagram's KDA card runs on the token's raw projections against the
// cached last three raw inputs, then the same one-pass update as
// decode_kernel.  conv_state [N, 3 taps (t-3, t-2, t-1), 3 (q,k,v), H, D] in
// the raw dtype is shifted in place.
template <typename Tin, int D>
__global__ void __launch_bounds__(DecodeCfg<Tin, D>::THREADS)
decode_conv_kernel(const Tin *__restrict__ q_raw, const Tin *__restrict__ k_raw,
                   const Tin *__restrict__ v_raw, const float *__restrict__ conv_w,
                   Tin *__restrict__ conv_state, const float *__restrict__ z_g,
                   const float *__restrict__ z_beta, float *__restrict__ state,
                   Tin *__restrict__ out, int32_t H) {
    using C = DecodeCfg<Tin, D>;
    const int unit = blockIdx.x;             // sequence * H + head
    const int n = unit / H, h = unit % H;
    const int tid = threadIdx.x;
    const int c = tid % C::COLG, r = tid / C::COLG;
    __shared__ TokenSmem<D> sm;
    __shared__ float4 s_part[2][C::RG][C::COLG];

    float *S = state + (size_t)unit * D * D;
    const size_t vec = (size_t)unit * D;
    const int64_t HD = (int64_t)H * D;
    // the token's small inputs first (cached window, raw projections, taps,
    // gate logits), so that they arrive ahead of the 64 KB state behind them
    // and the prologue runs while the state streams in
    Tin win[3][3], xr[3];
    float4 wt[3];
    float zg = 0.f;
    if (tid < D) {
        const Tin *raws[3] = {q_raw, k_raw, v_raw};
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            wt[i] = __ldg(reinterpret_cast<const float4 *>(conv_w + ((int64_t)i * HD + (int64_t)h * D + tid) * 4));
            const Tin *cs = conv_state + ((size_t)n * 9 + i) * HD + (size_t)h * D + tid;  // tap 0
            win[i][0] = cs[0]; win[i][1] = cs[3 * HD]; win[i][2] = cs[6 * HD];
            xr[i] = raws[i][vec + tid];
        }
        zg = z_g[vec + tid];
    }
    float4 s[C::ROWS];
#pragma unroll
    for (int i = 0; i < C::ROWS; ++i)
        s[i] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)(r * C::ROWS + i) * D) + c);

    // prologue for channel ch = tid (tid < D): conv over the cached window
    float yq = 0.f, yk = 0.f, yv = 0.f;
    if (tid < D) {
        const int ch = tid;
        float y3[3];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const float4 w = wt[i];
            Tin *cs = conv_state + ((size_t)n * 9 + i) * HD + (size_t)h * D + ch;  // tap 0
            const float yv2 = w.x * Elem<Tin>::load(&win[i][0]) + w.y * Elem<Tin>::load(&win[i][1]) +
                              w.z * Elem<Tin>::load(&win[i][2]) + w.w * Elem<Tin>::load(&xr[i]);
            y3[i] = __fdividef(yv2, 1.f + __expf(-yv2));
            cs[0] = win[i][1];               // shift the window: t-2 -> t-3, ...
            cs[3 * HD] = win[i][2];
            cs[6 * HD] = xr[i];
        }
        yq = y3[0]; yk = y3[1]; yv = y3[2];
    }
    // |q|^2, |k|^2 and q.k of the unnormalised head vectors in one pass;
    // k.q of the normalised vectors is then iq * ik * (q.k)
    const float3 sums = block_sum3<C::THREADS>(make_float3(yq * yq, yk * yk, yq * yk), sm.red);
    const float iq = rsqrtf(sums.x + 1e-6f), ik = rsqrtf(sums.y + 1e-6f);
    const float kq = iq * ik * sums.z;
    if (tid < D) {
        const float qq = yq * iq, kk = yk * ik;
        const float a = __expf(-5.f / (1.f + __expf(-zg)));
        sm.ak[tid] = make_float2(a, kk);
        sm.kqa[tid] = make_float2(a * kk, a * qq);
        sm.v[tid] = yv;
    }
    if (tid == 0) {
        sm.kq = kq;
        sm.beta = 1.f / (1.f + __expf(-z_beta[unit]));
    }
    __syncthreads();
    token_update<Tin, D>(s, sm, s_part, r, c, out + vec);
#pragma unroll
    for (int i = 0; i < C::ROWS; ++i)
        __stcs(reinterpret_cast<float4 *>(S + (size_t)(r * C::ROWS + i) * D) + c, s[i]);
}

// Multi-token verify with a rollback point: K draft tokens of one sequence
// run from a read-only state (the snapshot semantics of "From GPT-2 to Kimi
// K3", Chapter 14: cached KDA states are read-only, a hit works on a private
// copy); every draft token's output is written and state_out receives the
// state after the first accept[n] tokens (the accepted prefix).
//
// Two draft tokens share each pass over the state.  Both column reductions of
// token t+1 run on the state before token t:
//   (D_{t+1} S_t)^T x = (alpha_{t+1} alpha_t x)^T S + ((alpha_{t+1} x) . k_t) u_t
// for x = k_{t+1} (its error term) and x = q_{t+1} (its read), so one pass over
// S gives four column sums, two scalars fix them up once u_t is known, and one
// pass applies S <- D_{t+1} (D_t S + k_t u_t^T) + k_{t+1} u_{t+1}^T.  An odd
// last draft runs as a pair whose second token is neutral (alpha = 1,
// k = q = v = beta = 0: u = 0 and the state passes through), with no output.
template <int D>
struct PairSmem {
    // per state row, one 16-byte read each: the four reduction weights
    // (alpha_t k_t, alpha_t q_t, alpha_{t+1} alpha_t k_{t+1}, alpha_{t+1} alpha_t q_{t+1})
    // and the four update factors (alpha_t, alpha_{t+1}, k_t, k_{t+1})
    float4 red_w[D], upd[D];
    float v1[D], v2[D];
    float red[8][4];          // per-warp partial sums of the four scalars
    float sc[4];              // k_t.q_t, k_{t+1}.q_{t+1}, (alpha_{t+1} k_{t+1}).k_t, (alpha_{t+1} q_{t+1}).k_t
    float beta1, beta2;
};

// The state's columns are independent here too (the column sums, the update
// and the scalars k.q, (alpha k').k need no other column), so for d >= 64
// verify gives each (sequence, head) SPLIT = 2 CTAs of half the columns.
// Each thread keeps its 16 rows x 4 columns; a CTA has half the warps behind
// each of its barriers, and four 128-thread CTAs fit an SM where two 256-thread
// ones did, so one CTA's barrier wait is covered by three others (the top
// stall of the one-CTA form).  Each CTA stages the token vectors whole, one
// thread per channel.
template <typename Tin, int D>
struct VerifyCfg {
    static constexpr int SPLIT = D >= 64 ? 2 : 1;
    static constexpr int COLG = D / 4 / SPLIT;         // float4 column groups of a CTA
    static constexpr int RG = 8;
    static constexpr int ROWS = D / RG;
    static constexpr int THREADS = COLG * RG;
};

template <typename Tin, int D>
__global__ void __launch_bounds__(VerifyCfg<Tin, D>::THREADS)
verify_pair_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                   const float *__restrict__ g, const float *__restrict__ beta,
                   const float *__restrict__ state_in, const int32_t *__restrict__ accept,
                   int32_t K, int32_t H, Tin *__restrict__ out, float *__restrict__ state_out) {
    using C = VerifyCfg<Tin, D>;
    static_assert(C::THREADS / 32 <= 8, "per-warp partials");
    static_assert(C::THREADS >= D, "one thread per channel stages the vectors");
    const int unit = blockIdx.x / C::SPLIT;  // sequence * H + head
    const int col0 = (blockIdx.x % C::SPLIT) * (D / C::SPLIT);   // this CTA's first column
    const int n = unit / H, h = unit % H;
    const int tid = threadIdx.x;
    const int c = tid % C::COLG, r = tid / C::COLG;
    __shared__ PairSmem<D> pm;
    __shared__ float4 s_part[4][C::RG][C::COLG];
    __shared__ float4 s_sum[4][C::COLG];     // the four column sums of a pair
    static_assert(C::RG >= 4, "row groups 0..3 finish the four sums");

    const float *S0 = state_in + (size_t)unit * D * D;
    float *S1 = state_out + (size_t)unit * D * D;
    float4 s[C::ROWS];
#pragma unroll
    for (int i = 0; i < C::ROWS; ++i)
        s[i] = __ldcs(reinterpret_cast<const float4 *>(S0 + (size_t)(r * C::ROWS + i) * D + col0) + c);
    int acc = accept[n];
    acc = acc < 0 ? 0 : (acc > K ? K : acc);

    auto store_state = [&]() {
#pragma unroll
        for (int i = 0; i < C::ROWS; ++i)
            __stcs(reinterpret_cast<float4 *>(S1 + (size_t)(r * C::ROWS + i) * D + col0) + c, s[i]);
    };
    // one pass over the state for drafts t and t + 1; two = false: t is the
    // last draft and the second token is neutral.  (A compile-time flag, with
    // the pass inlined twice, took 127 registers and ran 3% slower.)
    auto pass = [&](const int t, const bool two) {
        if (t == acc) store_state();
        const size_t vec1 = ((size_t)(n * K + t) * H + h) * D, vec2 = vec1 + (size_t)H * D;
        float4 sc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (tid < D) {
            const float k1 = Elem<Tin>::load(k + vec1 + tid), q1 = Elem<Tin>::load(q + vec1 + tid);
            const float k2 = two ? Elem<Tin>::load(k + vec2 + tid) : 0.f;
            const float q2 = two ? Elem<Tin>::load(q + vec2 + tid) : 0.f;
            const float a1 = __expf(g[vec1 + tid]), a2 = two ? __expf(g[vec2 + tid]) : 1.f;
            pm.red_w[tid] = make_float4(a1 * k1, a1 * q1, a2 * a1 * k2, a2 * a1 * q2);
            pm.upd[tid] = make_float4(a1, a2, k1, k2);
            pm.v1[tid] = Elem<Tin>::load(v + vec1 + tid);
            pm.v2[tid] = two ? Elem<Tin>::load(v + vec2 + tid) : 0.f;
            sc = make_float4(k1 * q1, k2 * q2, a2 * k2 * k1, a2 * q2 * k1);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sc.x += __shfl_xor_sync(0xffffffffu, sc.x, o);
            sc.y += __shfl_xor_sync(0xffffffffu, sc.y, o);
            sc.z += __shfl_xor_sync(0xffffffffu, sc.z, o);
            sc.w += __shfl_xor_sync(0xffffffffu, sc.w, o);
        }
        if ((tid & 31) == 0) {
            pm.red[tid >> 5][0] = sc.x; pm.red[tid >> 5][1] = sc.y;
            pm.red[tid >> 5][2] = sc.z; pm.red[tid >> 5][3] = sc.w;
        }
        if (tid == 0) {
            pm.beta1 = beta[(size_t)(n * K + t) * H + h];
            pm.beta2 = two ? beta[(size_t)(n * K + t + 1) * H + h] : 0.f;
        }
        __syncthreads();
        if (tid < 4) {
            float x = 0.f;
#pragma unroll
            for (int w = 0; w < C::THREADS / 32; ++w) x += pm.red[w][tid];
            pm.sc[tid] = x;
        }
        // the four column sums over the old state
        float4 p[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) p[m] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < C::ROWS; ++i) {
            const int row = r * C::ROWS + i;
            const float4 fw = pm.red_w[row];
            const float f[4] = {fw.x, fw.y, fw.z, fw.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                p[m].x += f[m] * s[i].x; p[m].y += f[m] * s[i].y;
                p[m].z += f[m] * s[i].z; p[m].w += f[m] * s[i].w;
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) s_part[m][r][c] = p[m];
        __syncthreads();
        // row group m (< 4) finishes sum m of its column group; everyone reads the four
        if (r < 4) {
            float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < C::RG; ++j) {
                const float4 x = s_part[r][j][c];
                x4.x += x.x; x4.y += x.y; x4.z += x.z; x4.w += x.w;
            }
            s_sum[r][c] = x4;
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < 4; ++m) p[m] = s_sum[m][c];
        const float kq1 = pm.sc[0], kq2 = pm.sc[1], ck = pm.sc[2], cq = pm.sc[3];
        const float b1 = pm.beta1, b2 = pm.beta2;
        const float a1v[4] = {p[0].x, p[0].y, p[0].z, p[0].w}, r1v[4] = {p[1].x, p[1].y, p[1].z, p[1].w};
        const float a2v[4] = {p[2].x, p[2].y, p[2].z, p[2].w}, r2v[4] = {p[3].x, p[3].y, p[3].z, p[3].w};
        float u1[4], u2[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = col0 + 4 * c + j;
            u1[j] = b1 * (pm.v1[col] - a1v[j]);
            u2[j] = b2 * (pm.v2[col] - (a2v[j] + ck * u1[j]));
        }
        if (r == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                Elem<Tin>::store(out + vec1 + col0 + 4 * c + j, r1v[j] + u1[j] * kq1);
                if (two)
                    Elem<Tin>::store(out + vec2 + col0 + 4 * c + j, r2v[j] + cq * u1[j] + u2[j] * kq2);
            }
        }
        // the state after token t alone, when that is the accepted prefix
        if (t + 1 == acc) {
#pragma unroll
            for (int i = 0; i < C::ROWS; ++i) {
                const int row = r * C::ROWS + i;
                const float4 up = pm.upd[row];
                const float a = up.x, ki = up.z;
                const float4 x = make_float4(a * s[i].x + ki * u1[0], a * s[i].y + ki * u1[1],
                                             a * s[i].z + ki * u1[2], a * s[i].w + ki * u1[3]);
                __stcs(reinterpret_cast<float4 *>(S1 + (size_t)row * D + col0) + c, x);
            }
        }
#pragma unroll
        for (int i = 0; i < C::ROWS; ++i) {
            const int row = r * C::ROWS + i;
            const float4 up = pm.upd[row];
            const float a1 = up.x, a2 = up.y, k1 = up.z, k2 = up.w;
            s[i].x = a2 * (a1 * s[i].x + k1 * u1[0]) + k2 * u2[0];
            s[i].y = a2 * (a1 * s[i].y + k1 * u1[1]) + k2 * u2[1];
            s[i].z = a2 * (a1 * s[i].z + k1 * u1[2]) + k2 * u2[2];
            s[i].w = a2 * (a1 * s[i].w + k1 * u1[3]) + k2 * u2[3];
        }
        __syncthreads();   // the next pair restages the shared inputs
    };
    for (int t = 0; t < K; t += 2) pass(t, t + 1 < K);
    // all K drafts accepted: for odd K the last pass stored it already
    if (acc == K && (K & 1) == 0) store_state();
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

template <typename Tin, int D>
cudaError_t run_conv(const void *q_raw, const void *k_raw, const void *v_raw, const float *conv_w,
                     void *conv_state, const float *z_g, const float *z_beta, float *state,
                     void *out, int32_t N, int32_t H, cudaStream_t stream) {
    const unsigned units = (unsigned)N * (unsigned)H;
    if (units == 0) return cudaSuccess;
    decode_conv_kernel<Tin, D><<<units, DecodeCfg<Tin, D>::THREADS, 0, stream>>>(
        static_cast<const Tin *>(q_raw), static_cast<const Tin *>(k_raw),
        static_cast<const Tin *>(v_raw), conv_w, static_cast<Tin *>(conv_state), z_g, z_beta,
        state, static_cast<Tin *>(out), H);
    count_launches(1);
    return cudaGetLastError();
}

template <typename Tin, int D>
cudaError_t run_verify(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, const float *state_in, const int32_t *accept,
                       int32_t N, int32_t K, int32_t H, void *out, float *state_out,
                       cudaStream_t stream) {
    using C = VerifyCfg<Tin, D>;
    const uint64_t ctas = (uint64_t)N * (uint64_t)H * C::SPLIT;
    if (ctas == 0) return cudaSuccess;
    if (ctas > 0x7fffffffu) return cudaErrorInvalidValue;
    verify_pair_kernel<Tin, D><<<(unsigned)ctas, C::THREADS, 0, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v), g,
        beta, state_in, accept, K, H, static_cast<Tin *>(out), state_out);
    count_launches(1);
    return cudaGetLastError();
}

#define KDA_DISPATCH_D(D, CALL)                   \
    switch (D) {                                  \
    case 16: { constexpr int DD = 16; return CALL; }   \
    case 32: { constexpr int DD = 32; return CALL; }   \
    case 64: { constexpr int DD = 64; return CALL; }   \
    case 128: { constexpr int DD = 128; return CALL; } \
    default: return cudaErrorInvalidValue;        \
    }

}  // namespace

cudaError_t launch_decode_conv(const void *q_raw, const void *k_raw, const void *v_raw,
                               const float *conv_w, void *conv_state, const float *z_g,
                               const float *z_beta, float *state, void *out, int32_t N,
                               int32_t H, int32_t D, kda_dtype dt, cudaStream_t stream) {
    if (dt == KDA_BF16)
        KDA_DISPATCH_D(D, (run_conv<__nv_bfloat16, DD>(q_raw, k_raw, v_raw, conv_w, conv_state,
                                                       z_g, z_beta, state, out, N, H, stream)))
    KDA_DISPATCH_D(D, (run_conv<float, DD>(q_raw, k_raw, v_raw, conv_w, conv_state, z_g, z_beta,
                                           state, out, N, H, stream)))
}

cudaError_t launch_verify(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, const float *state_in, const int32_t *accept,
                          int32_t N, int32_t K, int32_t H, int32_t D, kda_dtype dt, void *out,
                          float *state_out, cudaStream_t stream) {
    if (dt == KDA_BF16)
        KDA_DISPATCH_D(D, (run_verify<__nv_bfloat16, DD>(q, k, v, g, beta, state_in, accept, N, K,
                                                         H, out, state_out, stream)))
    KDA_DISPATCH_D(D, (run_verify<float, DD>(q, k, v, g, beta, state_in, accept, N, K, H, out,
                                             state_out, stream)))
}

cudaError_t launch_decode(const void *q, const void *k, const void *v,
                          const float *g, const float *beta, float *state,
                          void *out, int32_t N, int32_t H, int32_t D,
                          kda_dtype dt, cudaStream_t stream) {
    if (dt == KDA_BF16)
        return run_d<__nv_bfloat16>(q, k, v, g, beta, state, out, N, H, D, stream);
    return run_d<float>(q, k, v, g, beta, state, out, N, H, D, stream);
}

}  // namespace kda
