// kda_prefill_chunk.cu -- chunkwise KDA prefill on the tcgen05 tensor cores
// (d_k = d_v = 128, bf16 q/k/v, fp32 g/beta/state), for sm_103a.
//
// What it computes is the recurrence of "Kimi K3 Architecture Explained",
// Step 3 (S_t = (I - b k k^T) Diag(alpha_t) S_{t-1} + b k v^T, o_t = S_t^T q_t),
// re-associated over chunks of C = 64 tokens the way "From GPT-2 to Kimi K3,
// from first principles", Chapter 6, describes it: recurrent across chunks,
// dense matrix products within a chunk, through a UT transform and a
// pseudo-value term.  Per chunk with incoming state S and G_t = sum_{s<=t} g_s:
//
//   L  = strict_lower(diag(b) [k_t . k_j e^{G_t - G_j}])    (64 x 64)
//   P  = lower_with_diag([q_t . k_j e^{G_t - G_j}])         (64 x 64)
//   T  = (I + L)^-1,  Tb = T diag(b)
//   W  = Tb (e^{G} * K),  Ut = Tb V                          (UT transform)
//   U  = Ut - W S                                            (pseudo-values)
//   O  = (e^{G} * Q) S + P U                                 (read after update)
//   S' = Diag(e^{G_63}) S + Khat^T U,  Khat_j = e^{G_63 - G_j} k_j
//
// Rescaling ("From GPT-2 to Kimi K3", Chapter 5, K3's lower-bounded decay):
// with g >= -5 a 16-token tile accumulates at most -80 of log-decay, so
// every factor below stays inside fp32/bf16 range.  For a row t in tile a
// and a column j in tile b <= a, with s_a = G before tile a and e_b = G at
// the end of tile b:
//   e^{G_t - G_j} = e^{G_t - s_a} * e^{s_a - e_b} * e^{e_b - G_j}
//                     (<= 1)        (<= e^80)       (<= 1)
// so the Gram matrices are one dense MMA per row tile a:
//   [k E; q E] (128 x 128) times R^(a) (16(a+1) x 128),
//   E_t = e^{G_t - s_a},  R^(a)_j = k_j e^{e_b - G_j} e^{s_a - e_b}.
// Only 2 exponentials per (token, channel) are taken; the rest are products
// with per-channel tile vectors.
//
// Data path (one CTA of 256 threads per (document, head), chunks in order):
//   TMA (128B swizzle) -> shared memory tiles of q, k, v (bf16) and g (fp32)
//   CUDA cores: cumulative G, decay factors, bf16 operands in shared memory
//   tcgen05.mma (bf16 x bf16 -> fp32 in TMEM) for every matrix product
//   CUDA cores: UT solve in fp32 (16x16 diagonal blocks by forward
//               substitution, off-diagonal blocks by block recursion)
//   the fp32 state lives in registers (64 values per thread); its bf16 copy
//   in shared memory is the B operand of the next chunk's W S / Q+ S.
// All waits are bounded: a lost arrival sets KDA_DEVICE_TIMEOUT and the CTA
// leaves after draining its own outstanding copies.
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kC = 64;         // tokens per chunk
constexpr int kD = 128;        // d_k = d_v
constexpr int kThreads = 256;  // 8 warps

// ---- shared memory map (bytes from a 1024-aligned base) ----
// A1: [-W ; Q+] K-major, two K halves of [128 rows][128 B]; the q tile of
//     the chunk is loaded by TMA into rows 64..127 and scaled in place.
constexpr uint32_t OFF_A1 = 0;
// k tile (TMA, channel halves of [64 rows][128 B]) -> K+ in place (MN-major B)
constexpr uint32_t OFF_K = 32768;
// v tile (TMA) -- used directly as the MN-major B operand of Ut = Tb V
constexpr uint32_t OFF_V = 49152;
// g tile fp32 [64][128] (TMA, no swizzle) -> G in place -> Khat (MN-major A,
// channel halves of [64 rows][128 B]) after the operand pass
constexpr uint32_t OFF_G = 65536;
// Gram region: operands of the Gram MMAs, then P / L / Tb / U
constexpr uint32_t OFF_GR = 98304;
constexpr uint32_t GR_GA = 0;          // [kE; qE] K-major, 2 halves x 16384
constexpr uint32_t GR_RT = 32768;      // R^(a), a = 0..3 (4K, 8K, 12K, 16K)
constexpr uint32_t GR_P = 0;           // [0; P] K-major [128][128 B]
constexpr uint32_t GR_L = 16384;       // L, then T, fp32 [64][64]
constexpr uint32_t GR_TB = 32768;      // [Tb; 0] K-major [128][128 B]
constexpr uint32_t GR_U = 49152;       // U MN-major, 2 halves of [64][128 B]
constexpr uint32_t GR_Y = 65536;       // fp32 [16][48] scratch of the UT solve
// bf16 state, MN-major B: two N halves of [128 rows][128 B]
constexpr uint32_t OFF_S = 172032;
// per-channel fp32 vectors of the chunk
constexpr uint32_t OFF_VEC = 204800;
constexpr uint32_t VEC_GS = 0;                 // [4][128] e^{s_a}
constexpr uint32_t VEC_KH = 4 * 512;           // [4][128] e^{G_63 - e_a}
constexpr uint32_t VEC_PV = 8 * 512;           // [10][128] e^{s_a - e_b}, b <= a
constexpr uint32_t VEC_DEC = 18 * 512;         // [128] e^{G_63}
constexpr uint32_t OFF_BETA = OFF_VEC + 19 * 512;   // [64] fp32
constexpr uint32_t OFF_BAR = OFF_BETA + 256;        // mbarriers
constexpr uint32_t OFF_MISC = OFF_BAR + 64;         // tmem base, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;   // + alignment slack

constexpr uint32_t BAR_Q = 0, BAR_K = 8, BAR_V = 16, BAR_G = 24, BAR_MMA = 32;

// TMEM columns
constexpr uint32_t TM_D1 = 0;     // [U ; O] accumulator
constexpr uint32_t TM_D3 = 128;   // Khat^T U
constexpr uint32_t TM_G = 256;    // Gram blocks (160 columns), then W (128)
constexpr uint32_t TM_COLS = 512;

__device__ __forceinline__ uint32_t gram_col(int a) { return 8u * a * (a + 1); }  // 0,16,48,96
__device__ __forceinline__ uint32_t rt_off(int a) { return 2048u * a * (a + 1); }  // 0,4K,12K,24K

struct Maps {
    CUtensorMap q, k, v, g;
};

__global__ void __launch_bounds__(kThreads, 1)
chunk_kernel(const __grid_constant__ Maps maps, const float *__restrict__ beta,
             const float *init_state, const int32_t *__restrict__ cu, int32_t N, int64_t T,
             int32_t H, __nv_bfloat16 *__restrict__ out, float *final_state,
             int32_t *__restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sp = warp & 3;          // TMEM sub-partition (lanes 32*sp .. 32*sp+31)
    const int hh = warp >> 2;         // which 64-column half this warp handles
    const int h = blockIdx.x, n = blockIdx.y;
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + OFF_MISC);
    // plain shared-memory accesses (the compiler may schedule them) by address
#define SM_F(a) (*reinterpret_cast<float *>(smem + ((a) - sb)))
#define SM_F4(a) (*reinterpret_cast<float4 *>(smem + ((a) - sb)))
#define SM_U4(a) (*reinterpret_cast<uint4 *>(smem + ((a) - sb)))

    int64_t bos, eos;
    if (!doc_bounds(cu, n, N, T, bos, eos)) {
        if (tid == 0) flag_status(status, KDA_DEVICE_BAD_OFFSETS);
        return;
    }
    const int64_t len = eos - bos;
    const int nchunks = static_cast<int>((len + kC - 1) / kC);
    const size_t unit = static_cast<size_t>(n) * H + h;

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(sb + OFF_BAR + 8 * i, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(sb + OFF_MISC, TM_COLS);

    // state rows r = 32*sp + lane, columns 64*hh .. 64*hh+63, fp32 registers
    const int srow = 32 * sp + lane;
    float S[64];
    {
        const float *src = init_state ? init_state + unit * kD * kD + (size_t)srow * kD + 64 * hh
                                      : nullptr;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
            float4 x = src ? *reinterpret_cast<const float4 *>(src + j)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
        }
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = S[8 * c8 + e];
            (SM_U4(sb + OFF_S + hh * 16384 + sw128_off(srow, c8)) = pack_bf16x8(x));
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    auto issue_q = [&](int64_t t0) {
        mbar_expect_tx(sb + OFF_BAR + BAR_Q, 16384);
        tma_load_2d(sb + OFF_A1 + 8192, &maps.q, h * kD, (int32_t)t0, sb + OFF_BAR + BAR_Q);
        tma_load_2d(sb + OFF_A1 + 16384 + 8192, &maps.q, h * kD + 64, (int32_t)t0,
                    sb + OFF_BAR + BAR_Q);
    };
    auto issue_k = [&](int64_t t0) {
        mbar_expect_tx(sb + OFF_BAR + BAR_K, 16384);
        tma_load_2d(sb + OFF_K, &maps.k, h * kD, (int32_t)t0, sb + OFF_BAR + BAR_K);
        tma_load_2d(sb + OFF_K + 8192, &maps.k, h * kD + 64, (int32_t)t0, sb + OFF_BAR + BAR_K);
    };
    auto issue_v = [&](int64_t t0) {
        mbar_expect_tx(sb + OFF_BAR + BAR_V, 16384);
        tma_load_2d(sb + OFF_V, &maps.v, h * kD, (int32_t)t0, sb + OFF_BAR + BAR_V);
        tma_load_2d(sb + OFF_V + 8192, &maps.v, h * kD + 64, (int32_t)t0, sb + OFF_BAR + BAR_V);
    };
    auto issue_g = [&](int64_t t0) {
        mbar_expect_tx(sb + OFF_BAR + BAR_G, 32768);
        tma_load_2d(sb + OFF_G, &maps.g, h * kD, (int32_t)t0, sb + OFF_BAR + BAR_G);
    };

    // chunk index of the last load issued on each TMA barrier (thread 0 only),
    // so an aborting CTA can drain its own copies before it exits
    int issued[4] = {-1, -1, -1, -1};
    if (tid == 0 && nchunks > 0) {
        issue_q(bos);
        issue_k(bos);
        issue_v(bos);
        issue_g(bos);
        issued[0] = issued[1] = issued[2] = issued[3] = 0;
    }

    uint32_t mma_phase = 0;
    // all threads wait on the MMA barrier; a timeout raises the abort flag
    auto wait_mma = [&]() {
        if (!mbar_wait(sb + OFF_BAR + BAR_MMA, mma_phase)) misc[1] = 1;
        mma_phase ^= 1;
        tc_fence_after();
    };
    auto wait_tma = [&](uint32_t bar, int c) {
        if (!mbar_wait(sb + OFF_BAR + bar, c & 1)) misc[1] = 1;
    };

    const uint32_t gr = sb + OFF_GR;
    int c = 0;
    for (; c < nchunks; ++c) {
        const int64_t t0 = bos + (int64_t)c * kC;
        const int lenc = (eos - t0) < kC ? static_cast<int>(eos - t0) : kC;

        // ---------------- step 1: inputs, beta, cumulative log-decay
        wait_tma(BAR_Q, c);
        wait_tma(BAR_K, c);
        wait_tma(BAR_G, c);
        if (tid < kC)
            (SM_F(sb + OFF_BETA + 4 * tid) = tid < lenc ? beta[(size_t)(t0 + tid) * H + h] : 0.f);
        {
            // G in place: thread = (channel, half of the tokens); 32 loads in flight
            const int ch = tid & 127, half = tid >> 7;
            float gv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int t = 32 * half + i;
                gv[i] = (t < lenc) ? SM_F(sb + OFF_G + (uint32_t)(t * kD + ch) * 4) : 0.f;
            }
#pragma unroll
            for (int i = 1; i < 32; ++i) gv[i] += gv[i - 1];
            if (half == 0) {
#pragma unroll
                for (int i = 0; i < 32; ++i) SM_F(sb + OFF_G + (uint32_t)(i * kD + ch) * 4) = gv[i];
            }
            __syncthreads();
            if (half == 1) {
                const float base = SM_F(sb + OFF_G + (uint32_t)(31 * kD + ch) * 4);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    SM_F(sb + OFF_G + (uint32_t)((32 + i) * kD + ch) * 4) = gv[i] + base;
            }
        }
        __syncthreads();
        if (misc[1]) break;

        // ---------------- per-channel tile vectors
        {
            const int ch = tid & 127;
            auto G = [&](int t) {
                return t < 0 ? 0.f : SM_F(sb + OFF_G + (uint32_t)(t * kD + ch) * 4);
            };
            const float g63 = G(63);
            if (tid < 128) {
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    (SM_F(sb + OFF_VEC + VEC_GS + a * 512 + ch * 4) = __expf(G(16 * a - 1)));
                    (SM_F(sb + OFF_VEC + VEC_KH + a * 512 + ch * 4) = __expf(g63 - G(16 * a + 15)));
                }
                (SM_F(sb + OFF_VEC + VEC_DEC + ch * 4) = __expf(g63));
            } else {
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b <= a; ++b)
                        (SM_F(sb + OFF_VEC + VEC_PV + (a * (a + 1) / 2 + b) * 512 + ch * 4) = __expf(G(16 * a - 1) - G(16 * b + 15)));
            }
        }
        __syncthreads();

        // ---------------- step 2: operands (thread: channel chunk cc, one row per tile)
        uint4 khat[4];
        {
            const int cc = tid & 15;                 // 8-channel chunk
            const int half = cc >> 3, c8 = cc & 7;   // channel half, chunk in the half
            const int c0 = 8 * cc;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int t = (tid >> 4) + 16 * a;
                const bool live = t < lenc;
                float Gt[8], Gs[8], Ge[8];
                {
                    const uint32_t rt = sb + OFF_G + (uint32_t)(t * kD + c0) * 4;
                    float4 x0 = SM_F4(rt), x1 = SM_F4(rt + 16);
                    Gt[0] = x0.x; Gt[1] = x0.y; Gt[2] = x0.z; Gt[3] = x0.w;
                    Gt[4] = x1.x; Gt[5] = x1.y; Gt[6] = x1.z; Gt[7] = x1.w;
                    const uint32_t re = sb + OFF_G + (uint32_t)((16 * a + 15) * kD + c0) * 4;
                    x0 = SM_F4(re); x1 = SM_F4(re + 16);
                    Ge[0] = x0.x; Ge[1] = x0.y; Ge[2] = x0.z; Ge[3] = x0.w;
                    Ge[4] = x1.x; Ge[5] = x1.y; Ge[6] = x1.z; Ge[7] = x1.w;
                    if (a == 0) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) Gs[e] = 0.f;
                    } else {
                        const uint32_t rs = sb + OFF_G + (uint32_t)((16 * a - 1) * kD + c0) * 4;
                        x0 = SM_F4(rs); x1 = SM_F4(rs + 16);
                        Gs[0] = x0.x; Gs[1] = x0.y; Gs[2] = x0.z; Gs[3] = x0.w;
                        Gs[4] = x1.x; Gs[5] = x1.y; Gs[6] = x1.z; Gs[7] = x1.w;
                    }
                }
                const uint32_t kaddr = sb + OFF_K + half * 8192 + sw128_off(t, c8);
                const uint32_t qaddr = sb + OFF_A1 + half * 16384 + sw128_off(64 + t, c8);
                float kv[8], qv[8];
                unpack_bf16x8(SM_U4(kaddr), kv);
                unpack_bf16x8(SM_U4(qaddr), qv);
                if (!live) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) kv[e] = qv[e] = 0.f;
                }
                float E[8], Eb[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    E[e] = __expf(Gt[e] - Gs[e]);
                    Eb[e] = __expf(Ge[e] - Gt[e]);
                }
                // Gram left operand rows t (k) and 64 + t (q)
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = kv[e] * E[e];
                (SM_U4(gr + GR_GA + half * 16384 + sw128_off(t, c8)) = pack_bf16x8(x));
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = qv[e] * E[e];
                (SM_U4(gr + GR_GA + half * 16384 + sw128_off(64 + t, c8)) = pack_bf16x8(x));
                // Gram right operands R^(a') for every row tile a' >= a
                float kb[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) kb[e] = kv[e] * Eb[e];
#pragma unroll
                for (int ap = a; ap < 4; ++ap) {
                    const uint32_t pv = sb + OFF_VEC + VEC_PV + (ap * (ap + 1) / 2 + a) * 512 + c0 * 4;
                    const float4 p0 = SM_F4(pv), p1 = SM_F4(pv + 16);
                    const float pvv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = kb[e] * pvv[e];
                    const uint32_t nrows = 16u * (ap + 1);
                    (SM_U4(gr + GR_RT + rt_off(ap) + half * nrows * 128 + sw128_off(t, c8)) = pack_bf16x8(x));
                }
                // Q+ and K+ in place: scale by e^{G_t} = E_t e^{s_a}
                {
                    const uint32_t gs = sb + OFF_VEC + VEC_GS + a * 512 + c0 * 4;
                    const float4 p0 = SM_F4(gs), p1 = SM_F4(gs + 16);
                    const float gsv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float at = E[e] * gsv[e];
                        x[e] = qv[e] * at;
                        y[e] = kv[e] * at;
                    }
                    (SM_U4(qaddr) = pack_bf16x8(x));
                    (SM_U4(kaddr) = pack_bf16x8(y));
                }
                // Khat = k e^{G_63 - G_t} = (k Eb) e^{G_63 - e_a}; stored after the barrier
                {
                    const uint32_t kh = sb + OFF_VEC + VEC_KH + a * 512 + c0 * 4;
                    const float4 p0 = SM_F4(kh), p1 = SM_F4(kh + 16);
                    const float khv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = kb[e] * khv[e];
                    khat[a] = pack_bf16x8(x);
                }
            }
            __syncthreads();   // every read of G is done: the g buffer now takes Khat
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int t = (tid >> 4) + 16 * a;
                (SM_U4(sb + OFF_G + half * 8192 + sw128_off(t, c8)) = khat[a]);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ---------------- step 3: Gram MMAs
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const uint32_t nrows = 16u * (a + 1);
                const uint32_t id = idesc_bf16(128, nrows, 0, 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad =
                        sw128_desc(gr + GR_GA + (kk >> 2) * 16384 + (kk & 3) * 32, 0, 1024);
                    const uint64_t bd = sw128_desc(
                        gr + GR_RT + rt_off(a) + (kk >> 2) * nrows * 128 + (kk & 3) * 32, 0, 1024);
                    mma_bf16(tmem + TM_G + gram_col(a), ad, bd, id, kk > 0);
                }
            }
            mma_commit(sb + OFF_BAR + BAR_MMA);
        }
        wait_mma();

        // ---------------- step 4: L (k rows) and P (q rows) out of TMEM
        {
            // warp -> row tile a: sub-partition sp covers tokens 32*(sp&1)..+31
            const int a = 2 * (sp & 1) + hh;
            const bool mine = (lane >> 4) == hh;     // lanes of tile a
            const int t = 32 * (sp & 1) + lane;      // token of this lane
            float G[64];
            tmem_ld64(tmem + ((uint32_t)(32 * sp) << 16) + TM_G + gram_col(a), G);
            if (mine) {
                if (sp < 2) {
                    const float bt = SM_F(sb + OFF_BETA + 4 * t);
#pragma unroll
                    for (int j = 0; j < 64; j += 4) {
                        float4 v;
                        v.x = (j + 0 < t) ? bt * G[j + 0] : 0.f;
                        v.y = (j + 1 < t) ? bt * G[j + 1] : 0.f;
                        v.z = (j + 2 < t) ? bt * G[j + 2] : 0.f;
                        v.w = (j + 3 < t) ? bt * G[j + 3] : 0.f;
                        (SM_F4(gr + GR_L + (uint32_t)(t * 64 + j) * 4) = v);
                    }
                } else {
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = (8 * c8 + e <= t) ? G[8 * c8 + e] : 0.f;
                        (SM_U4(gr + GR_P + sw128_off(64 + t, c8)) = pack_bf16x8(x));
                    }
                }
            }
            // rows 0..63 of [0; P] are zero
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int i = tid; i < 512; i += kThreads)
                (SM_U4(gr + GR_P + sw128_off(i >> 3, i & 7)) = z);
        }
        tc_fence_before();
        __syncthreads();

        // ---------------- step 5: T = (I + L)^-1 in fp32, then Tb = T diag(beta)
        {
            const uint32_t Lb = gr + GR_L;
            // 5a: diagonal 16x16 blocks, thread = (block a, column col)
            float xcol[16];
            const int a5 = tid >> 4, col = tid & 15;
            if (tid < 64) {
                float acc[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    xcol[i] = (i == col ? 1.f : 0.f) - acc[i];
#pragma unroll
                    for (int k = i + 1; k < 16; ++k)
                        acc[k] += SM_F(Lb + (uint32_t)((16 * a5 + k) * 64 + 16 * a5 + i) * 4) *
                                  xcol[i];
                }
            }
            __syncthreads();
            if (tid < 64) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    (SM_F(Lb + (uint32_t)((16 * a5 + i) * 64 + 16 * a5 + col) * 4) = xcol[i]);
            }
            __syncthreads();
            // 5b: block rows a = 1..3: T_ab = -T_aa sum_{m=b}^{a-1} L_am T_mb
            const int i5 = tid >> 4, jj = tid & 15;
            const uint32_t Yb = gr + GR_Y;
#pragma unroll
            for (int a = 1; a < 4; ++a) {
                for (int b = 0; b < a; ++b) {
                    float y = 0.f;
                    for (int m = b; m < a; ++m)
#pragma unroll
                        for (int l = 0; l < 16; ++l)
                            y += SM_F(Lb + (uint32_t)((16 * a + i5) * 64 + 16 * m + l) * 4) *
                                 SM_F(Lb + (uint32_t)((16 * m + l) * 64 + 16 * b + jj) * 4);
                    (SM_F(Yb + (uint32_t)(i5 * 48 + 16 * b + jj) * 4) = y);
                }
                __syncthreads();
                for (int b = 0; b < a; ++b) {
                    float y = 0.f;
#pragma unroll
                    for (int l = 0; l < 16; ++l)
                        y += SM_F(Lb + (uint32_t)((16 * a + i5) * 64 + 16 * a + l) * 4) *
                             SM_F(Yb + (uint32_t)(l * 48 + 16 * b + jj) * 4);
                    (SM_F(Lb + (uint32_t)((16 * a + i5) * 64 + 16 * b + jj) * 4) = -y);
                }
                __syncthreads();
            }
            // 5c: [Tb; 0], thread = (row t, 16-column quarter)
            {
                const int t = tid >> 2, qc = tid & 3;
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    const int c8 = 2 * qc + hc;
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 8 * c8 + e;
                        x[e] = (j <= t) ? SM_F(Lb + (uint32_t)(t * 64 + j) * 4) *
                                              SM_F(sb + OFF_BETA + 4 * j)
                                        : 0.f;
                    }
                    (SM_U4(gr + GR_TB + sw128_off(t, c8)) = pack_bf16x8(x));
                    (SM_U4(gr + GR_TB + sw128_off(64 + t, c8)) = make_uint4(0, 0, 0, 0));
                }
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ---------------- step 6: W = Tb K+ and Ut = Tb V (Ut lands in D1 rows 0..63)
        if (tid == 0) {
            tc_fence_after();
            wait_tma(BAR_V, c);
            const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sw128_desc(gr + GR_TB + kk * 32, 0, 1024);
                mma_bf16(tmem + TM_G, ad, sw128_desc(sb + OFF_K + kk * 2048, 8192, 1024), id, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sw128_desc(gr + GR_TB + kk * 32, 0, 1024);
                mma_bf16(tmem + TM_D1, ad, sw128_desc(sb + OFF_V + kk * 2048, 8192, 1024), id, kk > 0);
            }
            mma_commit(sb + OFF_BAR + BAR_MMA);
        }
        wait_mma();
        // -W -> rows 0..63 of A1 (warps of sub-partitions 0 and 1)
        if (sp < 2) {
            const int t = 32 * sp + lane;
            float v64[64];
            tmem_ld64(tmem + ((uint32_t)(32 * sp) << 16) + TM_G + 64 * hh, v64);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = -v64[8 * c8 + e];
                (SM_U4(sb + OFF_A1 + hh * 16384 + sw128_off(t, c8)) = pack_bf16x8(x));
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ---------------- step 7: D1 += [-W; Q+] S  ->  [U ; Q+ S]
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = sw128_desc(sb + OFF_A1 + (kk >> 2) * 16384 + (kk & 3) * 32, 0, 1024);
                const uint64_t bd = sw128_desc(sb + OFF_S + kk * 2048, 16384, 1024);
                mma_bf16(tmem + TM_D1, ad, bd, id, 1);
            }
            mma_commit(sb + OFF_BAR + BAR_MMA);
        }
        wait_mma();
        // q, k and v of this chunk are consumed: prefetch the next chunk's
        if (tid == 0 && c + 1 < nchunks) {
            issue_q(t0 + kC);
            issue_k(t0 + kC);
            issue_v(t0 + kC);
            issued[0] = issued[1] = issued[2] = c + 1;
        }

        // ---------------- step 8: U (D1 rows 0..63) -> bf16 MN-major B operand
        if (sp < 2) {
            const int t = 32 * sp + lane;
            float v64[64];
            tmem_ld64(tmem + ((uint32_t)(32 * sp) << 16) + TM_D1 + 64 * hh, v64);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = v64[8 * c8 + e];
                (SM_U4(gr + GR_U + hh * 8192 + sw128_off(t, c8)) = pack_bf16x8(x));
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ---------------- step 9: O = Q+ S + P U (D1 rows 64..127), D3 = Khat^T U
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id2 = idesc_bf16(128, 128, 0, 1);
            const uint32_t id3 = idesc_bf16(128, 128, 1, 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = sw128_desc(gr + GR_U + kk * 2048, 8192, 1024);
                mma_bf16(tmem + TM_D1, sw128_desc(gr + GR_P + kk * 32, 0, 1024), bd, id2, 1);
                mma_bf16(tmem + TM_D3, sw128_desc(sb + OFF_G + kk * 2048, 8192, 1024), bd, id3, kk > 0);
            }
            mma_commit(sb + OFF_BAR + BAR_MMA);
        }
        wait_mma();
        if (tid == 0 && c + 1 < nchunks) {
            issue_g(t0 + kC);
            issued[3] = c + 1;
        }

        // ---------------- step 10: outputs and the state update
        {
            const uint32_t lanebase = tmem + ((uint32_t)(32 * sp) << 16);
            if (sp >= 2) {
                const int t = 32 * (sp - 2) + lane;
                float v64[64];
                tmem_ld64(lanebase + TM_D1 + 64 * hh, v64);
                if (t < lenc) {
                    uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)(t0 + t) * H + h) * kD + 64 * hh);
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = v64[8 * c8 + e];
                        dst[c8] = pack_bf16x8(x);
                    }
                }
            }
            const float dec = SM_F(sb + OFF_VEC + VEC_DEC + 4 * srow);
            {
                float v64[64];
                tmem_ld64(lanebase + TM_D3 + 64 * hh, v64);
#pragma unroll
                for (int j = 0; j < 64; ++j) S[j] = dec * S[j] + v64[j];
            }
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = S[8 * c8 + e];
                (SM_U4(sb + OFF_S + hh * 16384 + sw128_off(srow, c8)) = pack_bf16x8(x));
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (misc[1]) break;
    }

    if (misc[1]) {
        // a wait gave up: report, let this CTA's own copies and MMAs drain
        if (tid == 0) {
            flag_status(status, KDA_DEVICE_TIMEOUT);
            mbar_wait(sb + OFF_BAR + BAR_MMA, mma_phase, 100000000ull);
            const uint32_t bars[4] = {BAR_Q, BAR_K, BAR_V, BAR_G};
            for (int i = 0; i < 4; ++i)
                if (issued[i] >= c)   // issued for this chunk or the next, maybe not landed
                    mbar_wait(sb + OFF_BAR + bars[i], issued[i] & 1, 100000000ull);
        }
    } else if (final_state != nullptr) {
        float *dst = final_state + unit * kD * kD + (size_t)srow * kD + 64 * hh;
#pragma unroll
        for (int j = 0; j < 64; j += 4)
            *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D view [T rows][H*128 elements] of a [T, H, 128] tensor, box 64 tokens tall
bool make_map(CUtensorMap *map, const void *base, int64_t T, int32_t H, bool fp32) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint32_t esz = fp32 ? 4 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)H * kD, (cuuint64_t)(T > 0 ? T : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)H * kD * esz};
    cuuint32_t box[2] = {fp32 ? 128u : 64u, (cuuint32_t)kC};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     fp32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool chunk_prefill_supported(int32_t D, kda_dtype dt) { return D == kD && dt == KDA_BF16; }

cudaError_t launch_prefill_chunk(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const float *init_state,
                                 const int32_t *cu_seqlens, int32_t N, int64_t T, int32_t H,
                                 void *out, float *final_state, int32_t *status,
                                 cudaStream_t stream) {
    Maps maps;
    if (!make_map(&maps.q, q, T, H, false) || !make_map(&maps.k, k, T, H, false) ||
        !make_map(&maps.v, v, T, H, false) || !make_map(&maps.g, g, T, H, true))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    chunk_kernel<<<dim3(H, N), kThreads, SMEM_BYTES, stream>>>(
        maps, beta, init_state, cu_seqlens, N, T, H, static_cast<__nv_bfloat16 *>(out),
        final_state, status);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
