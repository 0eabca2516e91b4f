// kda_prefill_chunk.cu -- chunkwise KDA prefill on the tcgen05 tensor cores
// (d_k = d_v = 128, bf16 q/k/v, fp32 g/beta/state), for sm_103a.
//
// What it computes is the recurrence of "Kimi K3 Architecture Explained",
// Step 3 (S_t = (I - b k k^T) Diag(alpha_t) S_{t-1} + b k v^T, o_t = S_t^T q_t),
// re-associated over chunks of C = 32 tokens the way "From GPT-2 to Kimi K3,
// from first principles", Chapter 6, describes it: recurrent across chunks,
// dense matrix products within a chunk, through a UT transform and a
// pseudo-value term.  Per chunk with incoming state S and G_t = sum_{s<=t} g_s:
//
//   L  = strict_lower(diag(b) [k_t . k_j e^{G_t - G_j}])    (32 x 32)
//   P  = lower_with_diag([q_t . k_j e^{G_t - G_j}])         (32 x 32)
//   T  = (I + L)^-1,  Tb = T diag(b)                         (UT transform)
//   U  = Tb V + Tb (-K+ S),  K+ = e^{G} * K                  (pseudo-values: the
//        pages' Ut = Tb V and W = Tb K+, with U = Ut - W S, as Tb V + Tb (-K+ S))
//   O  = Q+ S + P U,  Q+ = e^{G} * Q                         (read after update)
//   S' = Diag(e^{G_31}) S + Khat^T U,  Khat_j = e^{G_31 - G_j} k_j
//
// Layout: the state is held transposed in TMEM (lane = value channel v,
// column = key channel), fp32.  Every product of the state chain then has the
// value channels on the 128 accumulator lanes, and its left operand (the
// state, -K+ S and U, each rounded to fp16) is read by the MMA straight from
// TMEM.  The chunk's right operands (-K+, Q+, Khat, Tb, P, V) are fp16 tiles
// in shared memory.  fp16 (11 significant bits) keeps every element of the
// outputs and states within 2e-2 of their RMS of the exact recurrence where
// bf16 (8 bits) does not; it needs |v|, |state|, |U| < 65504, and a value
// beyond that is reported as KDA_DEVICE_RANGE.
//
// The Gram matrices: with g >= -5 ("From GPT-2 to Kimi K3", Chapter 5, K3's
// lower-bounded decay) a 16-token tile accumulates at most -80 of log-decay.
// Row tile a uses its start s_a as reference point: left rows k_t e^{G_t - s_a}
// (<= 1) and right rows k_j e^{s_a - G_j} (<= e^80 on the diagonal tile, <= 1
// before it), so one bf16 MMA (M = 128, N = 80) gives both matrices.  P's
// diagonal 16 x 16 blocks carry most of the output's sensitivity and are
// formed from hi + lo bf16 splits of both operands (hi.hi + hi.lo + lo.hi): the
// left operand's rows are [k; q hi; q lo] and the right operand's 80 rows [the
// off-diagonal tile; diagonal hi; diagonal lo].
//
// Warp-specialized pipeline, one CTA of 512 threads per (document, head); the
// roles run concurrently on different chunks and hand over through mbarriers:
//   warps 8..15  the operand pass of chunk x + 2: q, k by ldmatrix, g by
//                loads a chunk ahead; a lane owns one channel and two
//                consecutive tokens; every decay-scaled operand out by a
//                transposed stmatrix (8-channel groups as a loop: three per
//                warp on warps 8..11, one on warps 12..15).  Warps 12..15
//                also take the second half (key channels 64..127) of the
//                chain's state pass
//   warp 7       the Gram MMA of chunk x + 1, then the q/k load of chunk x + 3
//                into the slot that chunk x + 1's pass has read
//   warps 4..6   chunk x + 1's L and P out of TMEM, the 32 x 32 inverse (warp 4:
//                the diagonal blocks; warp 5: the off-diagonal block, a chunk
//                behind), v to fp16 (warp 6)
//   warps 0..3   the state chain of chunk x: the state's fp16 copy and its
//                decay (first half; see warps 12..15), -(K+ S) and Q+ S,
//                Tb V + Tb (-K+ S), S += Khat^T U and O += P U, the outputs of
//                chunk x - 1 out under chunk x's first MMA
// Prefix snapshots (every offset 64 tokens into a document, or its end) are
// written from the state's fp32 TMEM copy by the warps of the state pass as
// they read it at the top of a chunk, and by the chain warps at the end.
// All waits are bounded: a lost arrival sets KDA_DEVICE_TIMEOUT, every later
// wait of the CTA returns at once, and the CTA leaves after draining its own
// outstanding copies and MMAs.
#include <cuda.h>
#include <cuda_fp16.h>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kC = 32;         // tokens per chunk
constexpr int kD = 128;        // d_k = d_v
constexpr int kThreads = 512;  // 16 warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kF16Max = 65504.f;

// ---- shared memory map (bytes from a 1024-aligned base) ----
// q and k tiles, two slots: a tile is two 64-channel halves of [32 rows][128 B], 128-byte swizzle
constexpr uint32_t OFF_QK = 0, QK_SLOT = 16384, K_IN_SLOT = 8192, TILE_HALF = 4096;
// v tiles, three slots (bf16 as loaded, fp16 once the pass has converted them)
constexpr uint32_t OFF_V = 32768, V_SLOT = 8192;
// Gram left operand, K-major, two K halves of [128 rows][128 B]: k, q hi, q lo (rows 96.. unused)
constexpr uint32_t OFF_GL = 57344, GL_HALF = 16384;
// Gram right operand, K-major, two K halves of [80 rows][128 B]: off-diagonal tile, diag hi, diag lo
constexpr uint32_t OFF_R = 90112, R_HALF = 10240;
// [-K+; Q+] (fp16), three slots, K-major, two K halves of [64 rows][128 B]
constexpr uint32_t OFF_AQ = 110592, AQ_SLOT = 16384, AQ_HALF = 8192;
// Khat (fp16), three slots, token-major (MN-major B), two channel halves of [32 rows][128 B]
constexpr uint32_t OFF_KH = 159744, KH_SLOT = 8192, KH_HALF = 4096;
// Tb and P (fp16), two slots each: row t holds columns j = 0..31 in the first 64 B of 128 B
constexpr uint32_t OFF_TB = 184320, OFF_PM = 192512, SQ_SLOT = 4096;
// the output tile (bf16, two channel halves of [32 rows][128 B])
constexpr uint32_t OFF_STG = 200704;
// L, then T: fp32, transposed, element (t, j) at [j * LST + t]; two buffers
constexpr uint32_t OFF_L = 208896, LST = 36, L_BUF = 4608;
// lo-row partial sums of P's diagonal blocks: [32][LOS] fp32
constexpr uint32_t OFF_LO = 218112, LOS = 17;
// inverse scratch: M10 = L10 T00, 16 x 16 fp32, row stride 20
constexpr uint32_t OFF_X = 220288, XS = 20;
// e^{G_31} per channel, three slots; beta of a chunk, two slots
constexpr uint32_t OFF_VEC = 221568, VEC_D = 0, VEC_BETA = 1536;
// mbarriers.  Loads: BAR_QK[2], BAR_V[3] (transaction bytes).  MMA completion
// (tcgen05.commit): BAR_G, BAR_1, BAR_2, BAR_3 (the state), BAR_O (the outputs), and the slot releases EMPTY_B[3]
// (MMA3 of the chunk done: its -K+/Q+/Khat slot), TB_FREE[2], PM_FREE[2].
// Hand-overs: FULL_B[3] (8 pass warps stored a chunk's operands), TB_FULL[2]
// (Tb complete and v converted: 2 warps), TG_FREE (3 readout warps read the
// Gram), T_READY[2] (the diagonal blocks of T), L_FREE[2] (T's buffer read).
constexpr uint32_t OFF_BAR = OFF_VEC + 2048;
constexpr uint32_t BAR_QK = 0, BAR_V = 16, BAR_G = 40, BAR_1 = 48, BAR_2 = 56, BAR_3 = 64,
                   FULL_B = 72, EMPTY_B = 96, TB_FULL = 120, TB_FREE = 136, PM_FREE = 152,
                   TG_FREE = 168, BAR_DR0 = 176, BAR_DR1 = 184, T_READY = 192, L_FREE = 208,
                   BAR_O = 224, NUM_BARS = 29;
// tmem base, abort flag, then the last chunk whose load went to each q/k and v slot
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * NUM_BARS;
constexpr uint32_t MISC_TMEM = 0, MISC_ABORT = 1, MISC_QK = 2, MISC_V = 4;
constexpr uint32_t SMEM_USED = OFF_MISC + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;   // + alignment slack

// TMEM columns
constexpr uint32_t TM_S = 0;      // S^T fp32 (lane v, column key channel)
constexpr uint32_t TM_SB = 128;   // S^T fp16, two per column (A operand, K = 128)
constexpr uint32_t TM_XO = 192;   // two buffers of 64: [-(K+ S)^T | O^T] fp32, 32 tokens each
constexpr uint32_t TM_U = 320;    // U^T fp32, 32 columns
constexpr uint32_t TM_XB = 352;   // -(K+ S)^T fp16 (A operand, K = 32)
constexpr uint32_t TM_UB = 368;   // U^T fp16 (A operand, K = 32)
constexpr uint32_t TM_G = 384;    // Gram, 80 columns
constexpr uint32_t TM_UL = 464;   // U^T - fp16(U^T), fp16 (the low half of U for O += P U)
constexpr uint32_t TM_COLS = 512;

// ---- the map checked at compile time ----
constexpr bool kA1K(uint32_t off) { return off % 1024 == 0; }
static_assert(kA1K(OFF_QK) && kA1K(QK_SLOT) && kA1K(K_IN_SLOT) && kA1K(TILE_HALF) && kA1K(OFF_V) &&
              kA1K(V_SLOT) && kA1K(OFF_GL) && kA1K(GL_HALF) && kA1K(OFF_R) && kA1K(R_HALF) &&
              kA1K(OFF_AQ) && kA1K(AQ_SLOT) && kA1K(AQ_HALF) && kA1K(OFF_KH) && kA1K(KH_SLOT) &&
              kA1K(KH_HALF) && kA1K(OFF_TB) && kA1K(OFF_PM) && kA1K(SQ_SLOT) && kA1K(OFF_STG),
              "swizzled tiles on 1 KB");
static_assert(OFF_QK + 2 * QK_SLOT <= OFF_V && OFF_V + 3 * V_SLOT <= OFF_GL, "q/k and v slots");
static_assert(OFF_GL + 2 * GL_HALF <= OFF_R && GL_HALF >= 128 * 128, "Gram left: 128 rows per K half");
static_assert(OFF_R + 2 * R_HALF <= OFF_AQ && R_HALF >= 80 * 128, "Gram right: 80 rows per K half");
static_assert(OFF_AQ + 3 * AQ_SLOT <= OFF_KH && AQ_HALF >= 64 * 128, "[-K+; Q+]: 64 rows per K half");
static_assert(OFF_KH + 3 * KH_SLOT <= OFF_TB && KH_HALF >= 32 * 128, "Khat: 32 rows per half");
static_assert(OFF_TB + 2 * SQ_SLOT <= OFF_PM && OFF_PM + 2 * SQ_SLOT <= OFF_STG, "Tb, P");
static_assert(OFF_STG + 2 * TILE_HALF <= OFF_L, "output tile");
static_assert(L_BUF >= kC * LST * 4 && OFF_L + 2 * L_BUF <= OFF_LO && OFF_LO + kC * LOS * 4 <= OFF_X,
              "L, lo partials");
static_assert(OFF_X + 16 * XS * 4 <= OFF_VEC && VEC_BETA >= 3 * kD * 4 && VEC_BETA + 2 * kC * 4 <= 2048,
              "scratch, vectors");
static_assert(L_FREE + 16 <= BAR_O && BAR_O + 8 <= 8 * NUM_BARS, "mbarriers");
static_assert(SMEM_BYTES <= 232448, "227 KB of dynamic shared memory per CTA");
static_assert(TM_XO + 128 <= TM_U && TM_U + 32 <= TM_XB && TM_XB + 16 <= TM_UB && TM_UB + 16 <= TM_G &&
              TM_G + 80 <= TM_UL && TM_UL + 16 <= TM_COLS, "TMEM columns");

struct Maps {
    CUtensorMap q, k, v, g, o;
};

// ---- 16x16x16 products for the inverse's off-diagonal block, one warp each, on
// the warp-synchronous tensor-core path (mma.sync m16n8k8, tf32 in, fp32 out).
// Fragment layout (g = lane / 4, t = lane % 4): A rows g and g+8, columns t and
// t+4 of each 8-wide K slice; B K-rows t and t+4, column g; D rows g and g+8,
// columns 2t and 2t+1 of each 8-wide N tile.
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// acc += A B for 16x16 fp32 blocks in shared memory: A(r, k) at A[r sa + k]
// (or A[k sa + r] when AT), B(k, n) at B[k sb + n] (or B[n sb + k] when BT)
template <bool AT, bool BT>
__device__ __forceinline__ void gemm16(float (&acc)[2][4], const float *A, int sa, const float *B, int sb,
                                       int lane) {
    const int g = lane >> 2, t = lane & 3;
    auto Ael = [&](int r, int k) { return AT ? A[k * sa + r] : A[r * sa + k]; };
    auto Bel = [&](int k, int n) { return BT ? B[n * sb + k] : B[k * sb + n]; };
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const uint32_t a[4] = {to_tf32(Ael(g, 8 * ks + t)), to_tf32(Ael(g + 8, 8 * ks + t)),
                               to_tf32(Ael(g, 8 * ks + t + 4)), to_tf32(Ael(g + 8, 8 * ks + t + 4))};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b[2] = {to_tf32(Bel(8 * ks + t, 8 * nt + g)), to_tf32(Bel(8 * ks + t + 4, 8 * nt + g))};
            mma_tf32(acc[nt], a, b);
        }
    }
}

// running max of |x| that keeps a NaN (an fp16 overflow anywhere upstream of
// -K+ S or U reaches them as an infinity or a NaN)
__device__ __forceinline__ float max_abs_nan(float m, float x) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(x)));
    return r;
}

// kMode 0: every option; 1: no prefix snapshots and bf16 outputs, so that those
// paths are not in its code; 2: as 1, for one document of whole chunks
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
chunk_kernel(const __grid_constant__ Maps maps, const float *__restrict__ g, const float *__restrict__ beta,
             const float *init_state, const int32_t *__restrict__ cu, int32_t N, int64_t T, int32_t H,
             __nv_bfloat16 *__restrict__ out, float *final_state, int32_t *__restrict__ status,
             const int32_t *__restrict__ order, float *__restrict__ out_f32_arg, const Snapshots snaps_arg) {
    constexpr bool kPlain = kMode >= 1, kWhole = kMode == 2;
    float *const out_f32 = kPlain ? nullptr : out_f32_arg;
    Snapshots snaps = snaps_arg;
    if (kPlain) snaps.n = 0;
    extern __shared__ uint8_t smem_raw[];
    // 1024-aligned base, derived from the shared array so accesses stay in the shared window
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // warp-uniform by construction (a shuffle from lane 0), so that the compiler
    // keeps them, and what is derived from them, in uniform registers
    const uint32_t sb = __shfl_sync(0xffffffffu, smem_u32(smem), 0);
    const int tid = threadIdx.x, lane = tid & 31;
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    const int sp = warp & 3;          // TMEM sub-partition (lanes 32 sp .. 32 sp + 31)
    const int h = blockIdx.x;
    const int n = order ? order[blockIdx.y] : static_cast<int>(blockIdx.y);   // longest first
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + OFF_MISC);
#define SM_F(o) (*reinterpret_cast<float *>(smem + (o)))
#define SM_U32(o) (*reinterpret_cast<uint32_t *>(smem + (o)))
#define SM_U4(o) (*reinterpret_cast<uint4 *>(smem + (o)))
#define SM_H(o) (*reinterpret_cast<__half *>(smem + (o)))

    int64_t bos, eos;
    if (!doc_bounds(cu, n, N, T, bos, eos)) {
        if (tid == 0) flag_status(status, KDA_DEVICE_BAD_OFFSETS);
        return;
    }
    const int64_t len = eos - bos;
    const int nchunks = static_cast<int>((len + kC - 1) / kC);
    const size_t unit = static_cast<size_t>(n) * H + h;
    const int64_t row_stride = static_cast<int64_t>(H) * kD;   // elements between tokens

    if (tid == 0) {
        for (int i = 0; i < (int)NUM_BARS; ++i) {
            const uint32_t off = 8u * i;
            const uint32_t cnt = (off >= FULL_B && off < FULL_B + 24) ? 8u
                               : off == TG_FREE ? 3u : (off == TB_FULL || off == TB_FULL + 8) ? 2u : 1u;
            mbar_init(sb + OFF_BAR + off, cnt);
        }
        for (int i = 1; i < 16; ++i) misc[i] = 0;
        misc[MISC_QK] = misc[MISC_QK + 1] = 0xffffffffu;
        misc[MISC_V] = misc[MISC_V + 1] = misc[MISC_V + 2] = 0xffffffffu;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(sb + OFF_MISC + 4 * MISC_TMEM, TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, misc[MISC_TMEM], 0);
    const uint32_t tlane = tmem + ((uint32_t)(32 * sp) << 16);   // this warp's lanes

    auto bar = [&](uint32_t b) { return sb + OFF_BAR + b; };
    // a bounded wait that gives up at once after any earlier wait of the CTA gave up
    auto wait_bar = [&](uint32_t b, uint32_t parity) {
        if (misc[MISC_ABORT]) return;
        if (!mbar_wait(sb + OFF_BAR + b, parity)) misc[MISC_ABORT] = 1;
    };
    auto chunk_t0 = [&](int x) { return bos + (int64_t)x * kC; };
    auto chunk_len = [&](int x) {
        if (kWhole) return kC;
        const int64_t r = eos - chunk_t0(x);
        return r < kC ? static_cast<int>(r) : kC;
    };

    // ---- loads: q/k of chunk x into slot x & 1, v into slot x % 3
    auto issue_qk = [&](int x) {
        const uint32_t s = x & 1, dst = sb + OFF_QK + s * QK_SLOT, b = bar(BAR_QK + 8 * s);
        const int32_t y = (int32_t)chunk_t0(x);
        mbar_expect_tx(b, 2 * 2 * TILE_HALF);
        tma_load_2d(dst, &maps.q, h * kD, y, b);
        tma_load_2d(dst + TILE_HALF, &maps.q, h * kD + 64, y, b);
        tma_load_2d(dst + K_IN_SLOT, &maps.k, h * kD, y, b);
        tma_load_2d(dst + K_IN_SLOT + TILE_HALF, &maps.k, h * kD + 64, y, b);
        misc[MISC_QK + s] = x;
    };
    auto issue_v = [&](int x) {
        const uint32_t s = x % 3, dst = sb + OFF_V + s * V_SLOT, b = bar(BAR_V + 8 * s);
        const int32_t y = (int32_t)chunk_t0(x);
        mbar_expect_tx(b, 2 * TILE_HALF);
        tma_load_2d(dst, &maps.v, h * kD, y, b);
        tma_load_2d(dst + TILE_HALF, &maps.v, h * kD + 64, y, b);
        misc[MISC_V + s] = x;
    };

    // the state, transposed: warps 0..3, lane v = 32 sp + lane, all 128 key channels
    if (warp < 4) {
        const int v = 32 * sp + lane;
        const float *src = init_state ? init_state + unit * kD * kD + v : nullptr;
#pragma unroll 1
        for (int q4b = 0; q4b < 4; ++q4b) {
            float S[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) S[e] = src ? src[(size_t)(32 * q4b + e) * kD] : 0.f;
            tmem_st32_nowait(tlane + TM_S + 32 * q4b, S);
        }
        tmem_wait_st();
    }
    if (tid == 0 && nchunks > 0) {
        issue_qk(0);
        issue_v(0);
        if (nchunks > 1) { issue_qk(1); issue_v(1); }
        if (nchunks > 2) issue_v(2);
    }
    uint32_t range_bad = 0;   // a value beyond the fp16 range met by this thread
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // The state pass over the 32-column pieces [q0, q1) of chunk c: the fp16 copy
    // of the state (the A operand of -(K+ S) and Q+ S), then S <- Diag(e^{G_31}) S
    // in place (before S += Khat^T U); the state before chunk c goes to a
    // snapshot when one is asked for.  Pieces 0-1 by the chain warps, 2-3 by
    // warps 12..15 (each warp its own 32 lanes).
    auto state_pass = [&](int c, int q0, int q1, int32_t &snap) {
        const uint32_t dvec = sb + OFF_VEC + VEC_D + (c % 3) * 512;
        float *snap_dst = nullptr;
        if (c > 0 && snap < snaps.n && static_cast<int64_t>(snaps.offsets[snap]) == chunk_t0(c))
            snap_dst = snaps.out + (static_cast<size_t>(snap++) * H + h) * kD * kD + 32 * sp + lane;
#pragma unroll 1
        for (int q4b = q0; q4b < q1; ++q4b) {
            float xs[32];
            tmem_ld32(tlane + TM_S + 32 * q4b, xs);
            if (snap_dst != nullptr) {
#pragma unroll
                for (int e = 0; e < 32; ++e) snap_dst[(size_t)(32 * q4b + e) * kD] = xs[e];
            }
            uint32_t y[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) y[e] = pack_f16x2(xs[2 * e], xs[2 * e + 1]);
            tmem_st16_nowait(tlane + TM_SB + 16 * q4b, y);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 d = ld_shared_f4(dvec + 4 * (32 * q4b + e));
                const float2 a2 = f2mul(make_float2(xs[e], xs[e + 1]), make_float2(d.x, d.y));
                const float2 b2 = f2mul(make_float2(xs[e + 2], xs[e + 3]), make_float2(d.z, d.w));
                xs[e] = a2.x; xs[e + 1] = a2.y; xs[e + 2] = b2.x; xs[e + 3] = b2.y;
            }
            tmem_st32_nowait(tlane + TM_S + 32 * q4b, xs);
        }
    };

    if (warp >= 8) {
        // ====================================================== operand pass
        // 8-channel groups: warps 8..11 take three each (0..11), warps 12..15 one
        // each (12..15), so that the helpers are free early for the state pass.
        // A lane owns channel 8 grp + lane / 4 and tokens 8 m + 2 (lane & 3) + {0, 1}
        // (m = 0..3) of each group
        const int pw = warp - 8, q4 = lane & 3;
        const int ng = pw < 4 ? 3 : 1, gb = pw < 4 ? 3 * pw : 8 + pw;
        float gnext[3][8];
        auto load_g = [&](int x) {
            const int64_t t0 = chunk_t0(x);
            const int lc = chunk_len(x);
#pragma unroll
            for (int gi = 0; gi < 3; ++gi) {
                if (gi >= ng) break;
                const float *gp = g + h * kD + 8 * (gb + gi) + (lane >> 2);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int tk = 8 * (i >> 1) + 2 * q4 + (i & 1);
                    gnext[gi][i] = tk < lc ? __ldg(gp + (t0 + tk) * row_stride) : 0.f;
                }
            }
        };
        if (nchunks > 0) load_g(0);
        // warps 12..15: the second half of chunk c's state pass, beside the chain's
        int32_t hsnap = snaps.n > 0 ? snap_first(snaps, bos) : 0;
        auto help = [&](int c) {
            if (c >= 1) wait_bar(BAR_3, (c - 1) & 1);
            wait_bar(FULL_B + 8 * (c % 3), (c / 3) & 1);
            __syncwarp();
            tc_fence_after();
            state_pass(c, 2, 4, hsnap);
            tmem_wait_st();
            tc_fence_before();
            asm volatile("bar.sync 5, 256;" ::: "memory");
        };
#pragma unroll 1
        for (int x = 0; x < nchunks; ++x) {
            const int lenx = chunk_len(x);
            const bool full = lenx == kC;
            if (warp >= 12 && x >= 2) help(x - 2);
            wait_bar(BAR_QK + 8 * (x & 1), (x >> 1) & 1);
#pragma unroll 1
            for (int gi = 0; gi < ng; ++gi) {
                const int grp = gb + gi;
                const int chalf = grp >> 3;
                // this group's q, k (ldmatrix) and gates (selected from the prefetch)
                uint32_t qg[4], kg[4];
                {
                    const uint32_t a = sb + OFF_QK + (x & 1) * QK_SLOT + (grp >> 3) * TILE_HALF +
                                       sw128_off(lane, grp & 7);
                    ldsm_x4_trans(a, qg);
                    ldsm_x4_trans(a + K_IN_SLOT, kg);
                }
                float gg[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) gg[i] = gi == 0 ? gnext[0][i] : (gi == 1 ? gnext[1][i] : gnext[2][i]);
                const uint32_t co = sw128_off(lane, grp & 7);
                // G in log2 units per token pair: pair sums, a prefix over the quad
                // (the 8 tokens of a matrix), group totals
                float2 G[4];
                float e0 = 0.f, e1;
                {
                    float O = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float2 gp = f2mul(make_float2(gg[2 * m], gg[2 * m + 1]),
                                                make_float2(kLog2e, kLog2e));
                        float xs = gp.x + gp.y;
                        float ys = __shfl_up_sync(0xffffffffu, xs, 1, 4);
                        if (q4 >= 1) xs += ys;
                        ys = __shfl_up_sync(0xffffffffu, xs, 2, 4);
                        if (q4 >= 2) xs += ys;
                        const float tot = __shfl_sync(0xffffffffu, xs, 3, 4);
                        G[m] = make_float2(O + xs - gp.y, O + xs);
                        O += tot;
                        if (m == 1) e0 = O;
                    }
                    e1 = O;   // G after tile 0 (= s_1) and after tile 1 (= G_31)
                }
                if (gi == ng - 1 && x + 1 < nchunks) load_g(x + 1);   // the next chunk's gates, a chunk ahead
                const float fd0 = ex2(-e0), fd1 = ex2(e0 - e1);   // e^{s_a - e_a}, diagonal right rows
                const float gs1 = ex2(e0);                         // e^{s_1}: K+ and Q+ of tile 1
                const float kh0 = ex2(e1 - e0);                    // e^{G_31 - e_0}: Khat of tile 0
                const float dch = ex2(e1);                         // e^{G_31}: the chunk's state decay
                // per token pair: kE = k e^{G - s_a}, qE = q e^{G - s_a} (<= 1), B = k e^{e_a - G} (<= 1)
                float2 kE[4], qE[4], B[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int a = m >> 1;                      // 16-token tile
                    const float sa = a ? e0 : 0.f, ea = a ? e1 : e0;
                    float2 k2 = unpack_bf16x2(kg[m]), q2 = unpack_bf16x2(qg[m]);
                    if (!full) {
                        const int t0k = 8 * m + 2 * q4;
                        if (t0k >= lenx) { k2.x = 0.f; q2.x = 0.f; }
                        if (t0k + 1 >= lenx) { k2.y = 0.f; q2.y = 0.f; }
                    }
                    const float2 ea2 = f2sub(make_float2(ea, ea), G[m]);
                    const float2 sa2 = f2sub(G[m], make_float2(sa, sa));
                    const float2 E = make_float2(ex2(sa2.x), ex2(sa2.y));
                    const float2 Eb = make_float2(ex2(ea2.x), ex2(ea2.y));
                    kE[m] = f2mul(k2, E);
                    qE[m] = f2mul(q2, E);
                    B[m] = f2mul(k2, Eb);
                }
                if (gi == 0) {
                    // the slots this chunk writes are free: its -K+/Q+/Khat/decay slot
                    // (MMA3 of chunk x - 3 done) and the Gram operands (Gram of x - 1 done)
                    if (x >= 3) wait_bar(EMPTY_B + 8 * (x % 3), ((x / 3) - 1) & 1);
                    if (x >= 1) wait_bar(BAR_G, (x - 1) & 1);
                }
                if (q4 == 0) SM_F(OFF_VEC + VEC_D + (x % 3) * 512 + 4 * (8 * grp + (lane >> 2))) = dch;
                // each operand family packed and stored in turn: stored row = token,
                // this group's 16-byte channel chunk
                const uint32_t gl_b = sb + OFF_GL + chalf * GL_HALF + co;
                const uint32_t r_b = sb + OFF_R + chalf * R_HALF + co;
                const uint32_t aq_b = sb + OFF_AQ + (x % 3) * AQ_SLOT + chalf * AQ_HALF + co;
                {
                    uint32_t w[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) w[m] = pack_bf16x2(kE[m].x, kE[m].y);
                    stsm_x4_trans(gl_b, w[0], w[1], w[2], w[3]);                  // k: rows t
                }
                {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        hi[m] = pack_bf16x2(qE[m].x, qE[m].y);
                        const float2 r = f2sub(qE[m], unpack_bf16x2(hi[m]));
                        lo[m] = pack_bf16x2(r.x, r.y);
                    }
                    stsm_x4_trans(gl_b + 4096, hi[0], hi[1], hi[2], hi[3]);       // q hi: 32 + t
                    stsm_x4_trans(gl_b + 8192, lo[0], lo[1], lo[2], lo[3]);       // q lo: 64 + t
                }
                {
                    uint32_t w[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float2 kp = (m >> 1) ? f2mul(kE[m], make_float2(-gs1, -gs1))
                                                   : make_float2(-kE[m].x, -kE[m].y);
                        w[m] = pack_f16x2(kp.x, kp.y);
                    }
                    stsm_x4_trans(aq_b, w[0], w[1], w[2], w[3]);                  // -K+: rows t
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float2 qp = (m >> 1) ? f2mul(qE[m], make_float2(gs1, gs1)) : qE[m];
                        w[m] = pack_f16x2(qp.x, qp.y);
                    }
                    stsm_x4_trans(aq_b + 4096, w[0], w[1], w[2], w[3]);           // Q+: 32 + t
                }
                {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float fd = (m >> 1) ? fd1 : fd0;
                        const float2 Rd = f2mul(B[m], make_float2(fd, fd));
                        hi[m] = pack_bf16x2(Rd.x, Rd.y);
                        const float2 r = f2sub(Rd, unpack_bf16x2(hi[m]));
                        lo[m] = pack_bf16x2(r.x, r.y);
                    }
                    stsm_x2_trans(r_b, pack_bf16x2(B[0].x, B[0].y), pack_bf16x2(B[1].x, B[1].y));  // rows t < 16
                    stsm_x4_trans(r_b + 2048, hi[0], hi[1], hi[2], hi[3]);        // diag hi: 16 + t
                    stsm_x4_trans(r_b + 6144, lo[0], lo[1], lo[2], lo[3]);        // diag lo: 48 + t
                }
                {
                    uint32_t w[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float2 kh = (m >> 1) ? B[m] : f2mul(B[m], make_float2(kh0, kh0));
                        w[m] = pack_f16x2(kh.x, kh.y);
                    }
                    stsm_x4_trans(sb + OFF_KH + (x % 3) * KH_SLOT + chalf * KH_HALF + co, w[0], w[1], w[2], w[3]);
                }
            }
            // this chunk's operands are stored and its q/k slot is read (the Gram
            // warp refills the slot with chunk x + 2 once all eight warps are here)
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(FULL_B + 8 * (x % 3)));
        }
        if (warp >= 12) {
#pragma unroll 1
            for (int c = nchunks > 2 ? nchunks - 2 : 0; c < nchunks; ++c) help(c);
        }
    } else if (warp == 7) {
        // ====================================================== the Gram MMAs (one elected lane)
        const uint32_t id = idesc_bf16(128, 80, 0, 0);
#pragma unroll 1
        for (int x = 0; x < nchunks; ++x) {
            wait_bar(FULL_B + 8 * (x % 3), (x / 3) & 1);
            if (x >= 1) wait_bar(TG_FREE, (x - 1) & 1);
            __syncwarp();
            tc_fence_after();
            constexpr uint64_t dk = sw128_hi(0, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_w(tmem + TM_G, dk | sw128_lo(sb + OFF_GL + (kk >> 2) * GL_HALF + (kk & 3) * 32),
                           dk | sw128_lo(sb + OFF_R + (kk >> 2) * R_HALF + (kk & 3) * 32), id, kk > 0);
            mma_commit_w(bar(BAR_G));
            // every pass warp has read chunk x's q/k slot (FULL_B): load chunk x + 2 into it
            if (lane == 0 && x + 2 < nchunks && !misc[MISC_ABORT]) issue_qk(x + 2);
            __syncwarp();
        }
    } else if (warp >= 4) {
        // ====================================================== L, P, the inverse, v
        // Warp 4: k rows (L: off-diagonal block, diagonal hi.hi), then the inverse's
        // diagonal blocks.  Warp 5: q hi rows (P: off-diagonal block, diagonal
        // hi.hi + hi.lo), and a chunk behind, the inverse's off-diagonal block.
        // Warp 6: q lo rows (P's diagonal lo.hi partials), then v to fp16.
        const int t = lane, a = t >> 4;
        float beta_next = 0.f;
        auto load_beta = [&](int x) {
            beta_next = lane < chunk_len(x) ? __ldg(beta + (chunk_t0(x) + lane) * H + h) : 0.f;
        };
        if (warp == 4 && nchunks > 0) load_beta(0);
        // warp 5: T10 = -T11 L10 T00 of chunk x, as Tb10 = T10 diag(beta)
        auto offdiag = [&](int x) {
            wait_bar(T_READY + 8 * (x & 1), (x >> 1) & 1);
            float *Lf = reinterpret_cast<float *>(smem + OFF_L + (x & 1) * L_BUF);
            const float *betas = reinterpret_cast<const float *>(smem + OFF_VEC + VEC_BETA + (x & 1) * 128);
            const uint32_t tb = OFF_TB + (x & 1) * SQ_SLOT;
            // block (a, b) of L or T in the transposed storage: element (r, k) at [k LST + r]
            auto LB = [&](int ra, int rb) { return Lf + 16 * rb * LST + 16 * ra; };
            float *X = reinterpret_cast<float *>(smem + OFF_X);
            const int fg = lane >> 2, ft = lane & 3;
            {
                float acc[2][4] = {};
                gemm16<true, true>(acc, LB(1, 0), LST, LB(0, 0), LST, lane);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    *reinterpret_cast<float2 *>(X + fg * XS + 8 * nt + 2 * ft) = make_float2(acc[nt][0], acc[nt][1]);
                    *reinterpret_cast<float2 *>(X + (fg + 8) * XS + 8 * nt + 2 * ft) = make_float2(acc[nt][2], acc[nt][3]);
                }
            }
            __syncwarp();
            {
                float acc[2][4] = {};
                gemm16<true, false>(acc, LB(1, 1), LST, X, XS, lane);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int col = 8 * nt + 2 * ft;
                    const float b0 = betas[col], b1 = betas[col + 1];
                    SM_U32(tb + sw128_off(16 + fg, nt) + 4 * ft) = pack_f16x2(-acc[nt][0] * b0, -acc[nt][1] * b1);
                    SM_U32(tb + sw128_off(24 + fg, nt) + 4 * ft) = pack_f16x2(-acc[nt][2] * b0, -acc[nt][3] * b1);
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(TB_FULL + 8 * (x & 1)));
                mbar_arrive(bar(L_FREE + 8 * (x & 1)));
            }
        };
#pragma unroll 1
        for (int x = 0; x < nchunks; ++x) {
            if (warp == 5 && x >= 1) offdiag(x - 1);
            const uint32_t lb = OFF_L + (x & 1) * L_BUF;
            const uint32_t bvec = OFF_VEC + VEC_BETA + (x & 1) * 128;
            float beta_cur = 0.f;
            if (warp == 4) {
                beta_cur = beta_next;
                if (x + 1 < nchunks) load_beta(x + 1);
                if (x >= 2) wait_bar(L_FREE + 8 * (x & 1), ((x >> 1) - 1) & 1);
                SM_F(bvec + 4 * t) = beta_cur;
            }
            if (warp == 5 && x >= 2) wait_bar(PM_FREE + 8 * (x & 1), ((x >> 1) - 1) & 1);
            wait_bar(BAR_G, x & 1);
            tc_fence_after();
            if (warp == 4) {
                // L, scaled by beta_t, stored transposed for the inverse.  Columns of
                // row t: [0, 16) the off-diagonal block (tile 1's rows), [16, 32) /
                // [32, 48) the diagonal of tile 0 / 1
                float c[64];
                tmem_ld64(tlane + TM_G, c);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(TG_FREE));
#pragma unroll
                for (int j = 0; j < 16; ++j) SM_F(lb + 4 * (j * LST + t)) = beta_cur * (a ? c[j] : c[16 + j]);
#pragma unroll
                for (int j = 0; j < 16; ++j) SM_F(lb + 4 * ((16 + j) * LST + t)) = a ? beta_cur * c[32 + j] : 0.f;
                // ---------------- the diagonal 16x16 blocks of T = (I + L)^-1 in fp32,
                // column-oriented forward substitution (once x_i is known every later
                // partial sum takes one FMA); lane = (block a5, column col).  Written
                // out as Tb = T diag(beta), fp16
                if (x >= 2) wait_bar(TB_FREE + 8 * (x & 1), ((x >> 1) - 1) & 1);
                __syncwarp();
                float *Lf = reinterpret_cast<float *>(smem + lb);
                const float *betas = reinterpret_cast<const float *>(smem + bvec);
                const uint32_t tb = OFF_TB + (x & 1) * SQ_SLOT;
                const int a5 = lane >> 4, col = lane & 15;
                float *blk = Lf + 16 * a5 * LST + 16 * a5;   // blk[i LST + k] = L[16 a5 + k][16 a5 + i]
                float xs[16], accs[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) accs[i] = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    xs[i] = ((i == col) ? 1.f : 0.f) - accs[i];
                    float lc[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (4 * q + 3 <= i) continue;
                        const float4 v = *reinterpret_cast<const float4 *>(blk + i * LST + 4 * q);
                        lc[4 * q] = v.x; lc[4 * q + 1] = v.y; lc[4 * q + 2] = v.z; lc[4 * q + 3] = v.w;
                    }
#pragma unroll
                    for (int k = i + 1; k < 16; ++k) accs[k] += lc[k] * xs[i];
                }
                __syncwarp();
                // T_aa column col in place (transposed storage, as L) and its Tb column
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<float4 *>(blk + col * LST + 4 * q) =
                        make_float4(xs[4 * q], xs[4 * q + 1], xs[4 * q + 2], xs[4 * q + 3]);
                const int j = 16 * a5 + col;
                const float bj = betas[j];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    SM_H(tb + sw128_off(16 * a5 + i, j >> 3) + (j & 7) * 2) = __float2half_rn(xs[i] * bj);
                // the block above the diagonal, T01 = 0 (rows 0..15, columns 16..31)
                SM_U4(tb + sw128_off(lane >> 1, 2 + (lane & 1))) = make_uint4(0, 0, 0, 0);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(T_READY + 8 * (x & 1)));
            } else {
                if (warp == 6) {
                    float c[32];
                    tmem_ld32(tlane + TM_G + 16, c);   // columns 16..47: the diagonal hi right rows
#pragma unroll
                    for (int j = 0; j < 16; ++j) SM_F(OFF_LO + 4 * (t * LOS + j)) = a ? c[16 + j] : c[j];
                }
                asm volatile("bar.sync 2, 64;" ::: "memory");
                if (warp == 5) {
                    // P: the off-diagonal block, and on the diagonal hi.hi ([16, 48)) +
                    // hi.lo ([48, 80)) + lo.hi (the partials); lower with the diagonal, fp16
                    float c[64], d16[16];
                    tmem_ld64(tlane + TM_G, c);
                    tmem_ld16w(tlane + TM_G + 64, d16);
                    const uint32_t pm = OFF_PM + (x & 1) * SQ_SLOT;
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float v2[2];
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const int j = 2 * e + i;       // P column
                            float pv;
                            if (j < 16) {
                                const float dg = c[16 + j] + c[48 + j] + SM_F(OFF_LO + 4 * (t * LOS + j));
                                pv = a ? c[j] : (j <= t ? dg : 0.f);
                            } else {
                                const float dg = c[32 + (j - 16)] + d16[j - 16] + SM_F(OFF_LO + 4 * (t * LOS + j - 16));
                                pv = (a && j <= t) ? dg : 0.f;
                            }
                            v2[i] = pv;
                        }
                        w[e] = pack_f16x2(v2[0], v2[1]);
                    }
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        SM_U4(pm + sw128_off(t, q8)) = make_uint4(w[4 * q8], w[4 * q8 + 1], w[4 * q8 + 2], w[4 * q8 + 3]);
                    fence_proxy_async();
                }
                tc_fence_before();
                asm volatile("bar.sync 2, 64;" ::: "memory");   // the Gram and the partials are read
                if (lane == 0) mbar_arrive(bar(TG_FREE));
                if (warp == 6) {
                    // v of chunk x to fp16 in place (rows beyond the chunk zeroed); an fp16
                    // overflow here shows up in U and is reported where U is converted
                    wait_bar(BAR_V + 8 * (x % 3), (x / 3) & 1);
                    const int lenx = chunk_len(x);
                    auto cv = [](uint32_t w2) { const float2 f = unpack_bf16x2(w2); return pack_f16x2(f.x, f.y); };
#pragma unroll 4
                    for (int cc = 0; cc < 16; ++cc) {
                        const uint32_t va = OFF_V + (x % 3) * V_SLOT + (cc >> 3) * TILE_HALF + sw128_off(lane, cc & 7);
                        uint4 v4 = SM_U4(va);
                        if (lane >= lenx) v4 = make_uint4(0, 0, 0, 0);
                        SM_U4(va) = make_uint4(cv(v4.x), cv(v4.y), cv(v4.z), cv(v4.w));
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(TB_FULL + 8 * (x & 1)));
                }
            }
        }
        if (warp == 5 && nchunks > 0) offdiag(nchunks - 1);
    } else {
        // ====================================================== the state chain
        // lane v = 32 sp + lane of every TMEM product; thread 0 issues the MMAs
        auto txo = [&](int c) { return TM_XO + 64u * (c & 1); };   // [-(K+ S)^T | O^T] of chunk c
        auto out_conv = [&](int c) {
            // the outputs of chunk c: O^T (lane v, column t) through 16x256b
            // fragments and a transposed stmatrix into the token-major output tile
            const int lenc = chunk_len(c);
            const int64_t t0 = chunk_t0(c);
            const uint32_t to = txo(c) + 32;
            if (out_f32 != nullptr) {
                // fp32 outputs (the segment scan's partial outputs): lane v, one token a store
                float xo[32];
                tmem_ld32(tlane + to, xo);
                float *dst = out_f32 + (t0 * H + h) * kD + 32 * sp + lane;
#pragma unroll
                for (int t = 0; t < kC; ++t)
                    if (t < lenc) dst[(int64_t)t * row_stride] = xo[t];
                return;
            }
            uint32_t r2[32];
            tmem_ld16x256b_x4x2(tlane + to, tlane + (16u << 16) + to, r2);
#pragma unroll
            for (int h16 = 0; h16 < 2; ++h16) {
                uint32_t w[8];
#pragma unroll
                for (int rep = 0; rep < 4; ++rep) {
                    const uint32_t *r = r2 + 16 * h16 + 4 * rep;
                    w[2 * rep] = pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1]));
                    w[2 * rep + 1] = pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3]));
                }
#pragma unroll
                for (int k2 = 0; k2 < 2; ++k2) {
                    // matrices: (rep 2 k2, v rows 0-7), (rep 2 k2, rows 8-15), (rep 2 k2 + 1, ...)
                    const int mi = lane >> 3, rr = lane & 7;
                    const int rep = 2 * k2 + (mi >> 1);
                    const int v0 = 32 * sp + 16 * h16 + 8 * (mi & 1);
                    const uint32_t dst = sb + OFF_STG + (v0 >> 6) * TILE_HALF + sw128_off(8 * rep + rr, (v0 & 63) >> 3);
                    stsm_x4_trans(dst, w[4 * k2], w[4 * k2 + 1], w[4 * k2 + 2], w[4 * k2 + 3]);
                }
            }
            fence_proxy_async();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (lenc == kC) {
                if (tid == 0) {
                    tma_store_2d(&maps.o, h * kD, (int32_t)t0, sb + OFF_STG);
                    tma_store_2d(&maps.o, h * kD + 64, (int32_t)t0, sb + OFF_STG + TILE_HALF);
                    bulk_commit();
                }
            } else {
                // the document's ragged last chunk: only its own rows
                for (int idx = tid; idx < kC * 16; idx += 128) {
                    const int rw = idx >> 4, cc = idx & 15;
                    if (rw < lenc)
                        *reinterpret_cast<uint4 *>(out + ((t0 + rw) * H + h) * kD + 8 * cc) =
                            SM_U4(OFF_STG + (cc >> 3) * TILE_HALF + sw128_off(rw, cc & 7));
                }
            }
        };
        // fp32 -> fp16 copy of 32 TMEM columns (a [-K+ S | U]^T block), with the range check
        auto to_f16 = [&](uint32_t src, uint32_t dst) {
            float xv[32];
            tmem_ld32(tlane + src, xv);
            uint32_t y[16];
            float mx = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                mx = max_abs_nan(max_abs_nan(mx, xv[2 * e]), xv[2 * e + 1]);
                y[e] = pack_f16x2(xv[2 * e], xv[2 * e + 1]);
            }
            range_bad |= !(mx <= kF16Max);
            tmem_st16_nowait(tlane + dst, y);
        };
        // the document's next snapshot: its state after the tokens before offsets[snap]
        int32_t snap = snaps.n > 0 ? snap_first(snaps, bos) : 0;
        // U^T (32 columns) to fp16 high and low parts, with the range check
        auto to_f16_hilo = [&](uint32_t src, uint32_t dst_hi, uint32_t dst_lo) {
            float xv[32];
            tmem_ld32(tlane + src, xv);
            uint32_t hi[16], lo[16];
            float mx = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                mx = max_abs_nan(max_abs_nan(mx, xv[2 * e]), xv[2 * e + 1]);
                hi[e] = pack_f16x2(xv[2 * e], xv[2 * e + 1]);
                const float2 h2 = __half22float2(*reinterpret_cast<const __half2 *>(&hi[e]));
                lo[e] = pack_f16x2(xv[2 * e] - h2.x, xv[2 * e + 1] - h2.y);
            }
            range_bad |= !(mx <= kF16Max);
            tmem_st16_nowait(tlane + dst_hi, hi);
            tmem_st16_nowait(tlane + dst_lo, lo);
        };
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            if (c >= 1) wait_bar(BAR_3, (c - 1) & 1);
            wait_bar(FULL_B + 8 * (c % 3), (c / 3) & 1);
            tc_fence_after();
            state_pass(c, 0, 2, snap);   // the first half; warps 12..15 take the second
            tmem_wait_st();
            if (tid == 0) bulk_wait_read_all();    // the previous output tile has been read
            tc_fence_before();
            asm volatile("bar.sync 5, 256;" ::: "memory");   // both halves of the state pass
            if (warp == 0) {
                // [-(K+ S)^T | (Q+ S)^T] of chunk c
                tc_fence_after();
                const uint32_t id = idesc_f16(128, 64, 0, 0);
                const uint32_t aq = sb + OFF_AQ + (c % 3) * AQ_SLOT;
                const uint32_t dx = tmem + txo(c);
                constexpr uint64_t dk = sw128_hi(0, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_tmem_a_w(dx, tmem + TM_SB + 8 * kk, dk | sw128_lo(aq + (kk >> 2) * AQ_HALF + (kk & 3) * 32),
                                 id, kk > 0);
                mma_commit_w(bar(BAR_1));
            }
            // the previous chunk's outputs, under this chunk's MMA
            if (c >= 1) {
                wait_bar(BAR_O, (c - 1) & 1);
                tc_fence_after();
                out_conv(c - 1);
            }
            // -(K+ S)^T to fp16, then U = Tb V + Tb (-K+ S)
            wait_bar(BAR_1, c & 1);
            tc_fence_after();
            to_f16(txo(c), TM_XB);
            tmem_wait_st();
            tc_fence_before();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (warp == 0) {
                tc_fence_after();
                wait_bar(TB_FULL + 8 * (c & 1), (c >> 1) & 1);
                __syncwarp();
                tc_fence_after();
                const uint32_t id = idesc_f16(128, 32, 1, 0), id2 = idesc_f16(128, 32, 0, 0);
                const uint32_t tbs = sb + OFF_TB + (c & 1) * SQ_SLOT;
                const uint32_t vs = sb + OFF_V + (c % 3) * V_SLOT;
                constexpr uint64_t dk = sw128_hi(0, 1024), dmn = sw128_hi(TILE_HALF, 1024);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_bf16_w(tmem + TM_U, dmn | sw128_lo(vs + kk * 2048), dk | sw128_lo(tbs + kk * 32), id, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_tmem_a_w(tmem + TM_U, tmem + TM_XB + 8 * kk, dk | sw128_lo(tbs + kk * 32), id2, 1);
                mma_commit_w(bar(BAR_2));
                mma_commit_w(bar(TB_FREE + 8 * (c & 1)));
            }
            // U^T to fp16, then S += Khat^T U and O += P U
            wait_bar(BAR_2, c & 1);
            tc_fence_after();
            if (tid == 0 && c + 3 < nchunks) issue_v(c + 3);   // Tb V of chunk c has read its slot
            to_f16_hilo(TM_U, TM_UB, TM_UL);
            tmem_wait_st();
            tc_fence_before();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (warp == 0) {
                tc_fence_after();
                const uint32_t is = idesc_f16(128, 128, 0, 1), io = idesc_f16(128, 32, 0, 0);
                const uint32_t kh = sb + OFF_KH + (c % 3) * KH_SLOT, pmb = sb + OFF_PM + (c & 1) * SQ_SLOT;
                constexpr uint64_t dk = sw128_hi(0, 1024), dmn = sw128_hi(KH_HALF, 1024);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_tmem_a_w(tmem + TM_S, tmem + TM_UB + 8 * kk, dmn | sw128_lo(kh + kk * 2048), is, 1);
                mma_commit_w(bar(BAR_3));   // the state first: the next chunk waits on it
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_tmem_a_w(tmem + txo(c) + 32, tmem + TM_UB + 8 * kk, dk | sw128_lo(pmb + kk * 32), io, 1);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_tmem_a_w(tmem + txo(c) + 32, tmem + TM_UL + 8 * kk, dk | sw128_lo(pmb + kk * 32), io, 1);
                mma_commit_w(bar(BAR_O));
                mma_commit_w(bar(EMPTY_B + 8 * (c % 3)));
                mma_commit_w(bar(PM_FREE + 8 * (c & 1)));
            }
        }
        if (nchunks > 0) {
            wait_bar(BAR_3, (nchunks - 1) & 1);
            wait_bar(BAR_O, (nchunks - 1) & 1);
            tc_fence_after();
            if (tid == 0) bulk_wait_read_all();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            out_conv(nchunks - 1);
        }
    }

    // ---------------- the end: final state, or drain after a wait gave up
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool aborted = misc[MISC_ABORT] != 0;
    if (range_bad) flag_status(status, KDA_DEVICE_RANGE);
    if (aborted) {
        // report, then let this CTA's own MMAs and copies drain
        if (tid == 0) {
            flag_status(status, KDA_DEVICE_TIMEOUT);
            mma_commit(bar(BAR_DR0));
            mbar_wait(bar(BAR_DR0), 0, 100000000ull);
        }
        if (tid == 224) {
            mma_commit(bar(BAR_DR1));
            mbar_wait(bar(BAR_DR1), 0, 100000000ull);
        }
        if (tid == 32) {
            for (int s = 0; s < 2; ++s)
                if (misc[MISC_QK + s] != 0xffffffffu)
                    mbar_wait(bar(BAR_QK + 8 * s), (misc[MISC_QK + s] >> 1) & 1, 100000000ull);
            for (int s = 0; s < 3; ++s)
                if (misc[MISC_V + s] != 0xffffffffu)
                    mbar_wait(bar(BAR_V + 8 * s), (misc[MISC_V + s] / 3) & 1, 100000000ull);
        }
    } else if (warp < 4) {
        // S^T lane v, columns i  ->  final_state[i][v], and the snapshot at the
        // document's end when one is asked for
        const int v = 32 * sp + lane;
        float *dst = final_state != nullptr ? final_state + unit * kD * kD + v : nullptr;
        float *sdst = nullptr;
        if (nchunks > 0 && snaps.n > 0) {
            const int32_t i = snap_first(snaps, eos - 1);
            if (i < snaps.n && static_cast<int64_t>(snaps.offsets[i]) == eos)
                sdst = snaps.out + (static_cast<size_t>(i) * H + h) * kD * kD + v;
        }
        if (dst != nullptr || sdst != nullptr) {
#pragma unroll 1
            for (int q4b = 0; q4b < 4; ++q4b) {
                float S[32];
                tmem_ld32(tlane + TM_S + 32 * q4b, S);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    if (dst != nullptr) dst[(size_t)(32 * q4b + e) * kD] = S[e];
                    if (sdst != nullptr) sdst[(size_t)(32 * q4b + e) * kD] = S[e];
                }
            }
        }
    }
    if (tid == 0) bulk_wait_all();   // the output stores of thread 0 are complete
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
#undef SM_F
#undef SM_U32
#undef SM_U4
#undef SM_H
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

// 2-D view [T rows][H*128 elements] of a [T, H, 128] tensor, box one chunk tall:
// bf16 64 elements wide (128-byte swizzle), fp32 128 wide (no swizzle; L2 prefetch only)
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
                                 cudaStream_t stream, const int32_t *order, float *out_f32,
                                 Snapshots snaps) {
    Maps maps;
    if (!make_map(&maps.q, q, T, H, false) || !make_map(&maps.k, k, T, H, false) ||
        !make_map(&maps.v, v, T, H, false) || !make_map(&maps.g, g, T, H, true) ||
        !make_map(&maps.o, out, T, H, false))
        return cudaErrorInvalidValue;
    static std::atomic<uint64_t> smem_set[3] = {};
    const int mode = !(snaps.n == 0 && out_f32 == nullptr) ? 0
                     : (N == 1 && cu_seqlens == nullptr && T % kC == 0) ? 2 : 1;
    auto kern = mode == 0 ? chunk_kernel<0> : mode == 1 ? chunk_kernel<1> : chunk_kernel<2>;
    cudaError_t e = allow_dynamic_smem(kern, SMEM_BYTES, smem_set[mode]);
    if (e != cudaSuccess) return e;
    kern<<<dim3(H, N), kThreads, SMEM_BYTES, stream>>>(
        maps, g, beta, init_state, cu_seqlens, N, T, H, static_cast<__nv_bfloat16 *>(out),
        final_state, status, order, out_f32, snaps);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
