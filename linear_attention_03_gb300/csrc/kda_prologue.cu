// kda_prologue.cu -- the KDA input path of "An infra-oriented diagram of
// Kimi K3" (KDA card: "q, k, v ... ShortConv, Swish; q and k then L2Norm";
// "scaled sigmoid bounds log-decay to (-5, 0)"; "beta ... followed by
// sigmoid"), and the lower-bounded decay of "From GPT-2 to Kimi K3, from
// first principles", Chapter 5 (g = gmin * sigmoid(z), gmin = -5).
//
// Kernel 1 (conv_swish_norm): one pass over a raw q, k or v tensor.  A CTA
// covers 256 consecutive tokens of a group of heads whose channels are one
// contiguous slice of each token row (2,048 elements); the slices stream
// through a shared-memory ring by 1-D bulk copies, two halves of several
// tokens each, so that many bytes are in flight without holding registers.
// Each thread owns 8 consecutive channels of one head and keeps the last
// three raw inputs of its channels in registers as the causal window:
//     y_t = w0 x_{t-3} + w1 x_{t-2} + w2 x_{t-1} + w3 x_t     (fp32, two
// channels per instruction)
// History is zero before each document start (cu_seqlens).  Then
// s = y * sigmoid(y); for q and k the head's d channels are scaled by
// 1 / sqrt(sum s^2 + 1e-6), the sum taken with shuffles among the d/8 lanes
// that own the head.  HBM-bound: every raw element is read once (plus a
// three-token halo per tile) and every output written once.
//
// Kernel 2 (gates): elementwise g = -5 sigmoid(z_g), beta = sigmoid(z_beta).
#include <type_traits>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kTileTokens = 256;  // tokens per CTA
constexpr int kSliceElems = kThreads * 8;   // one token's channels of a CTA's heads
// tokens per half of the shared-memory ring (each half is 32 KB)
template <typename Tin> constexpr int ring_half() { return sizeof(Tin) == 2 ? 8 : 4; }
template <typename Tin> constexpr size_t ring_bytes() {
    return 2 * ring_half<Tin>() * kSliceElems * sizeof(Tin) + 16;   // + two mbarriers
}
constexpr float kL2Eps = 1e-6f;
constexpr float kGmin = -5.0f;

// index of the document holding token t (largest n with cu[n] <= t), with
// every offset clamped into [0, T] so bad offsets stay in bounds
__device__ __forceinline__ int find_doc(const int32_t *cu, int N, int64_t T, int64_t t) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const int64_t c = min((int64_t)max(cu[mid], 0), T);
        if (c <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int64_t clamp_off(const int32_t *cu, int n, int N, int64_t T) {
    if (cu == nullptr) return n == 0 ? 0 : T;
    if (n > N) return T;
    return min((int64_t)max(cu[n], 0), T);
}

// Raw row of 8 channels kept packed until used (bf16: one uint4; fp32: two).
template <typename Tin> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
        u = __ldcs(reinterpret_cast<const uint4 *>(p));
    }
    __device__ __forceinline__ void load_shared(const __nv_bfloat16 *p) {
        u = *reinterpret_cast<const uint4 *>(p);
    }
    __device__ __forceinline__ void zero() { u = make_uint4(0, 0, 0, 0); }
    __device__ __forceinline__ void get(float (&x)[8]) const {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float *p) {
        a = __ldcs(reinterpret_cast<const float4 *>(p));
        b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ __forceinline__ void load_shared(const float *p) {
        a = reinterpret_cast<const float4 *>(p)[0];
        b = reinterpret_cast<const float4 *>(p)[1];
    }
    __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ void get(float (&x)[8]) const {
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
};

// Two fp32 lanes in one instruction (the paired FMA and multiply of sm_100
// and later): a thread's 8 channels are 4 pairs, so the conv taps, the
// Swish, the sum of squares and the scaling issue half the instructions.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)),
          "l"(*reinterpret_cast<unsigned long long *>(&c)));
    return *reinterpret_cast<float2 *>(&d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}
__device__ __forceinline__ float ex2_approx(float x) {   // 2^x, the special-function unit
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {   // 1/x, the special-function unit
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Swish s = y sigmoid(y) on a pair, y / (1 + e^-y) for either output type:
// e^-y = 2^(-y log2 e) and the reciprocal on the special-function unit (each a
// few fp32 ulps), the multiplies and the add paired.  (The hardware tanh form
// 0.5 y (1 + tanh(y / 2)), one special-function op, has an error of ~5e-4 of
// s: below bf16's rounding step, but it moves about one bf16 rounding in
// sixteen to the neighbouring value, and the prefill carries those changed
// inputs into every later output.)
constexpr float kLog2e = 1.4426950408889634f;
template <typename Tin>
__device__ __forceinline__ float2 swish2(float2 y) {
    const float2 t = mul2(y, make_float2(-kLog2e, -kLog2e));
    const float2 d = add2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), make_float2(1.f, 1.f));
    return mul2(y, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads, 2)
conv_swish_norm_kernel(const Tin *__restrict__ x0, const Tin *__restrict__ x1,
                       const Tin *__restrict__ x2, const float *__restrict__ conv_w,
                       const int32_t *__restrict__ cu, int32_t N, int64_t T, int32_t H,
                       int64_t t_begin, int64_t t_end,
                       Tin *__restrict__ y0, Tin *__restrict__ y1, Tin *__restrict__ y2) {
    // tokens [t_begin, t_end) of the T-token inputs; output row 0 is token t_begin
    constexpr int TPH = D / 8;                     // lanes per head
    constexpr int HPB = kThreads / TPH;            // heads per CTA
    const int which = blockIdx.z;                  // 0 = q, 1 = k, 2 = v
    const Tin *x = which == 0 ? x0 : (which == 1 ? x1 : x2);
    Tin *y = which == 0 ? y0 : (which == 1 ? y1 : y2);
    const bool normalise = which < 2;

    const int h = blockIdx.y * HPB + threadIdx.x / TPH;
    const int sub = threadIdx.x % TPH;
    const bool live = h < H;
    const int64_t row_stride = (int64_t)H * D;
    const int64_t ch = (int64_t)(live ? h : 0) * D + 8 * sub;   // first channel

    // weights [3, H*D, 4]: the 4 taps of a channel are one float4; held as
    // tap x channel pair
    float2 w[4][4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
        const float4 wa = live ? __ldg(reinterpret_cast<const float4 *>(
                                     conv_w + ((int64_t)which * row_stride + ch + 2 * e2) * 4))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 wb = live ? __ldg(reinterpret_cast<const float4 *>(
                                     conv_w + ((int64_t)which * row_stride + ch + 2 * e2 + 1) * 4))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        w[0][e2] = make_float2(wa.x, wb.x); w[1][e2] = make_float2(wa.y, wb.y);
        w[2][e2] = make_float2(wa.z, wb.z); w[3][e2] = make_float2(wa.w, wb.w);
    }

    const int64_t t0 = t_begin + (int64_t)blockIdx.x * kTileTokens;
    const int64_t t1 = min(t_end, t0 + kTileTokens);
    int n = cu ? find_doc(cu, N, T, t0) : 0;
    int64_t start = clamp_off(cu, n, N, T);
    int64_t next = clamp_off(cu, n + 1, N, T);

    float2 hist[3][4];                             // x_{t-3}, x_{t-2}, x_{t-1}
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int64_t tj = t0 - 3 + j;
        Raw8<Tin> r;
        if (live && tj >= start && tj >= 0) r.load(x + tj * row_stride + ch); else r.zero();
        float hv[8];
        r.get(hv);
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) hist[j][e2] = make_float2(hv[2 * e2], hv[2 * e2 + 1]);
    }

    // the ring: two halves of HB token slices; thread 0 refills a half once
    // every thread has read it
    constexpr int HB = ring_half<Tin>();
    extern __shared__ __align__(128) uint8_t ring_raw[];
    const Tin *ring = reinterpret_cast<const Tin *>(ring_raw);
    const uint32_t ring_s = tc::smem_u32(ring_raw);
    const uint32_t bar = ring_s + 2 * HB * kSliceElems * (uint32_t)sizeof(Tin);
    const int h0 = blockIdx.y * HPB;
    const uint32_t slice_bytes = (uint32_t)(min(HPB, H - h0) * D * (int)sizeof(Tin));
    const Tin *xs = x + (int64_t)h0 * D;            // token t's slice at xs + t * row_stride
    if (threadIdx.x == 0) {
        tc::mbar_init(bar, 1);
        tc::mbar_init(bar + 8, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    auto fill = [&](int half, int64_t tb) {       // thread 0: tokens tb .. tb+HB-1 into a half
        const int64_t cnt = min((int64_t)HB, t1 - tb);
        if (cnt <= 0) return;
        const uint32_t hb = bar + 8 * half;
        tc::mbar_expect_tx(hb, (uint32_t)cnt * slice_bytes);
        for (int b = 0; b < cnt; ++b)
            tc::bulk_load(ring_s + (uint32_t)((half * HB + b) * kSliceElems * sizeof(Tin)),
                          xs + (tb + b) * row_stride, slice_bytes, hb);
    };
    if (threadIdx.x == 0) {
        fill(0, t0);
        fill(1, t0 + HB);
    }
    const int local = (threadIdx.x / TPH) * D + 8 * sub;   // this thread's channels in a slice
    uint32_t ph0 = 0, ph1 = 0;
    int half = 0;
    for (int64_t tb = t0; tb < t1; tb += HB, half ^= 1) {
        // a lost copy ends the wait after the time limit; the outputs are then
        // wrong but nothing hangs
        tc::mbar_wait(bar + 8 * half, half ? ph1 : ph0);
        if (half) ph1 ^= 1; else ph0 ^= 1;
#pragma unroll
        for (int b = 0; b < HB; ++b) {
            const int64_t t = tb + b;
            if (t >= t1) break;                     // uniform across the CTA
            while (t >= next && n < N - 1) {        // entered a new document
                ++n;
                start = clamp_off(cu, n, N, T);
                next = clamp_off(cu, n + 1, N, T);
#pragma unroll
                for (int j = 0; j < 3; ++j)
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) hist[j][e2] = make_float2(0.f, 0.f);
            }
            float cur[8];
            Raw8<Tin> r;
            r.load_shared(ring + (half * HB + b) * kSliceElems + local);
            r.get(cur);
            float2 s2[4];
            float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                const float2 c2 = make_float2(cur[2 * e2], cur[2 * e2 + 1]);
                float2 yv = mul2(w[0][e2], hist[0][e2]);
                yv = fma2(w[1][e2], hist[1][e2], yv);
                yv = fma2(w[2][e2], hist[2][e2], yv);
                yv = fma2(w[3][e2], c2, yv);
                s2[e2] = swish2<Tin>(yv);
                ss2 = fma2(s2[e2], s2[e2], ss2);
                hist[0][e2] = hist[1][e2];
                hist[1][e2] = hist[2][e2];
                hist[2][e2] = c2;
            }
            if (normalise) {
                float ss = ss2.x + ss2.y;
#pragma unroll
                for (int o = TPH / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float inv = rsqrtf(ss + kL2Eps);
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) s2[e2] = mul2(s2[e2], make_float2(inv, inv));
            }
            float s[8];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) { s[2 * e2] = s2[e2].x; s[2 * e2 + 1] = s2[e2].y; }
            if (live) Elem<Tin>::store8(y + (t - t_begin) * row_stride + ch, s);
        }
        __syncthreads();                            // this half is read
        if (threadIdx.x == 0) fill(half, tb + 2 * HB);
    }
}

__global__ void gates_kernel(const float *__restrict__ z_g, const float *__restrict__ z_beta,
                             float *__restrict__ g, float *__restrict__ beta,
                             int64_t n_g4, int64_t n_b) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_g4; i += stride) {
        float4 z = __ldcs(reinterpret_cast<const float4 *>(z_g) + i);
        z.x = kGmin / (1.f + __expf(-z.x));
        z.y = kGmin / (1.f + __expf(-z.y));
        z.z = kGmin / (1.f + __expf(-z.z));
        z.w = kGmin / (1.f + __expf(-z.w));
        __stcs(reinterpret_cast<float4 *>(g) + i, z);
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_b; i += stride)
        beta[i] = 1.f / (1.f + __expf(-z_beta[i]));
}

template <typename Tin, int D>
cudaError_t run_conv(const void *q_raw, const void *k_raw, const void *v_raw,
                     const float *conv_w, const int32_t *cu, int32_t N, int64_t T,
                     int64_t t_begin, int64_t t_end, int32_t H, void *q, void *k, void *v,
                     cudaStream_t stream) {
    constexpr int HPB = kThreads / (D / 8);
    const dim3 grid((unsigned)((t_end - t_begin + kTileTokens - 1) / kTileTokens),
                    (unsigned)((H + HPB - 1) / HPB), 3);
    static std::atomic<uint64_t> smem_set{0};   // per instantiation
    cudaError_t e = allow_dynamic_smem(conv_swish_norm_kernel<Tin, D>, ring_bytes<Tin>(), smem_set);
    if (e != cudaSuccess) return e;
    conv_swish_norm_kernel<Tin, D><<<grid, kThreads, ring_bytes<Tin>(), stream>>>(
        static_cast<const Tin *>(q_raw), static_cast<const Tin *>(k_raw),
        static_cast<const Tin *>(v_raw), conv_w, cu, N, T, H, t_begin, t_end,
        static_cast<Tin *>(q), static_cast<Tin *>(k), static_cast<Tin *>(v));
    count_launches(1);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t run_conv_d(const void *q_raw, const void *k_raw, const void *v_raw,
                       const float *conv_w, const int32_t *cu, int32_t N, int64_t T,
                       int64_t tb, int64_t te, int32_t H, int32_t D, void *q, void *k, void *v,
                       cudaStream_t stream) {
    switch (D) {
    case 16: return run_conv<Tin, 16>(q_raw, k_raw, v_raw, conv_w, cu, N, T, tb, te, H, q, k, v, stream);
    case 32: return run_conv<Tin, 32>(q_raw, k_raw, v_raw, conv_w, cu, N, T, tb, te, H, q, k, v, stream);
    case 64: return run_conv<Tin, 64>(q_raw, k_raw, v_raw, conv_w, cu, N, T, tb, te, H, q, k, v, stream);
    case 128: return run_conv<Tin, 128>(q_raw, k_raw, v_raw, conv_w, cu, N, T, tb, te, H, q, k, v, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prologue_range(const void *q_raw, const void *k_raw, const void *v_raw,
                                  const float *conv_w, const float *z_g, const float *z_beta,
                                  const int32_t *cu_seqlens, int32_t N, int64_t T, int64_t t_begin,
                                  int64_t t_end, int32_t H, int32_t D, kda_dtype dt, void *q,
                                  void *k, void *v, float *g, float *beta, cudaStream_t stream) {
    cudaError_t err = cudaSuccess;
    const int64_t n = t_end - t_begin;
    if (n > 0) {
        err = dt == KDA_BF16
                  ? run_conv_d<__nv_bfloat16>(q_raw, k_raw, v_raw, conv_w, cu_seqlens, N, T,
                                              t_begin, t_end, H, D, q, k, v, stream)
                  : run_conv_d<float>(q_raw, k_raw, v_raw, conv_w, cu_seqlens, N, T, t_begin,
                                      t_end, H, D, q, k, v, stream);
        if (err != cudaSuccess) return err;
    }
    const int64_t n_g4 = z_g ? n * H * D / 4 : 0;
    const int64_t n_b = z_beta ? n * H : 0;
    if (n_g4 + n_b > 0) {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t most = n_g4 > n_b ? n_g4 : n_b;
        int64_t blocks = (most + 255) / 256;
        if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
        if (blocks < 1) blocks = 1;
        gates_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
            z_g ? z_g + t_begin * H * D : nullptr, z_beta ? z_beta + t_begin * H : nullptr, g, beta,
            n_g4, n_b);
        count_launches(1);
        err = cudaGetLastError();
    }
    return err;
}

cudaError_t launch_prologue(const void *q_raw, const void *k_raw,
                            const void *v_raw, const float *conv_w,
                            const float *z_g, const float *z_beta,
                            const int32_t *cu_seqlens, int32_t N, int64_t T,
                            int32_t H, int32_t D, kda_dtype dt, void *q,
                            void *k, void *v, float *g, float *beta,
                            cudaStream_t stream) {
    return launch_prologue_range(q_raw, k_raw, v_raw, conv_w, z_g, z_beta, cu_seqlens, N, T, 0, T, H,
                                 D, dt, q, k, v, g, beta, stream);
}

}  // namespace kda
