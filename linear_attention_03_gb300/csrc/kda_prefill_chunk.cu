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
//   T  = (I + L)^-1,  Tb = T diag(b)                         (UT transform)
//   U  = Tb (V - K+ S),  K+ = e^{G} * K                      (pseudo-values; the
//        pages' W = Tb K+ and Ut = Tb V, with U = Ut - W S, re-associated)
//   O  = Q+ S + P U,  Q+ = e^{G} * Q                         (read after update)
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
// Data path (one CTA of 512 threads per (document, head), chunks in order):
//   TMA (128B swizzle) -> shared memory tiles of q, k, v (bf16) and g (fp32)
//   CUDA cores: cumulative G, decay factors, bf16 operands in shared memory
//   tcgen05.mma (bf16 x bf16 -> fp32 in TMEM) for every matrix product
//   CUDA cores: UT solve in fp32 (16x16 diagonal blocks by forward
//               substitution, off-diagonal blocks by block recursion)
//   the fp32 state lives in TMEM; its bf16 copy in shared memory is the B
//   operand of the chunk's [K+; Q+] S, which runs alongside the block inverse,
//   so that after it only U = Tb (V - K+ S), the read of U and the chunk's last
//   MMAs (O += P U, S += Khat^T U) remain.
// Decay factors are 2^x of log2-scaled G on the special-function unit.  The
// Gram left operand, Q+ and K+ are scaled in fp32 and rounded to bf16 once; the
// Gram right operand rows and Khat, which multiply one bf16 row by several
// per-channel factors, are packed bf16x2 products (two roundings).
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
constexpr int kThreads = 512;  // 16 warps: 4 per TMEM sub-partition
constexpr float kLog2e = 1.4426950408889634f;

// ---- shared memory map (bytes from a 1024-aligned base) ----
// A1: [K+ ; Q+] K-major, two K halves of [128 rows][128 B]: the A operand of
//     [K+; Q+] S.  The q tile of a chunk is loaded by TMA into rows 64..127 and
//     scaled in place; rows 0..63 receive K+.
constexpr uint32_t OFF_A1 = 0;
// two tile buffers that alternate roles: chunk c loads k into BUF[c & 1]
// (turned into Khat in place, the MN-major A operand of Khat^T U) and v into
// BUF[(c + 1) & 1] (overwritten by V - K+ S, the MN-major B operand of U = Tb (V - K+ S))
constexpr uint32_t OFF_BUF0 = 32768;
constexpr uint32_t OFF_BUF1 = 49152;
// g tile fp32 [64][128] (TMA, no swizzle); once scanned, the staging tile of the
// previous chunk's outputs (bf16, two 64-column halves, 128-byte swizzle) for a
// bulk tensor store
constexpr uint32_t OFF_G = 65536;
// Gram region: cumsum scratch, the Gram operands, afterwards P / L / Tb / U
constexpr uint32_t OFF_GR = 98304;
constexpr uint32_t GR_GA = 0;          // [kE; qE] K-major, 2 halves x 16384
constexpr uint32_t GR_RT = 32768;      // R rows 0..159 K-major, 2 halves x 20480
constexpr uint32_t RT_HALF = 20480;
constexpr uint32_t GR_P = 0;           // [0; P] K-major [128][128 B]
constexpr uint32_t GR_L = 16384;       // L, then T: fp32, stored transposed ([column][row], stride LST)
constexpr uint32_t LST = 72;           // padded stride (floats)
constexpr uint32_t GR_TB = 34816;      // [Tb; 0] K-major [128][128 B]
constexpr uint32_t GR_U = 51200;       // U MN-major, 2 halves of [64][128 B]; first the
                                       // block-inverse scratch (11 fp32 16x16 blocks)
// bf16 copy of the state, MN-major B: two N halves of [128 rows][128 B]
constexpr uint32_t OFF_S = 172032;
// per-channel vectors of the chunk
constexpr uint32_t OFF_VEC = 204800;
constexpr uint32_t VEC_SEG = 0;         // fp32 [8][128]  sums of g over the 8-token segments
constexpr uint32_t VEC_DEC = 4096;      // fp32 [128]     e^{G_63} of the chunk
constexpr uint32_t OFF_BETA = OFF_VEC + 4608;       // [64] fp32
constexpr uint32_t OFF_BAR = OFF_BETA + 256;        // mbarriers
// tmem base, abort flag, then the chunk index of the last g, v, k, q load issued
constexpr uint32_t OFF_MISC = OFF_BAR + 64;
constexpr uint32_t SMEM_USED = OFF_MISC + 32;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;   // + alignment slack

constexpr uint32_t BAR_Q = 0, BAR_K = 8, BAR_V = 16, BAR_G = 24, BAR_MMA = 32;
// a chunk's last two MMA groups are issued by two threads, each committing here
constexpr uint32_t BAR_MMA2 = 40;
// [K+; Q+] S, issued during the block inverse
constexpr uint32_t BAR_MMA1 = 48;

// TMEM columns
constexpr uint32_t TM_D1 = 0;     // [K+ S ; Q+ S], then [U ; O]
constexpr uint32_t TM_G = 128;    // Gram blocks (160 columns)
constexpr uint32_t TM_S = 288;    // fp32 state, 128 columns; Khat^T U accumulates into it
constexpr uint32_t TM_COLS = 512;

// ---- the map checked at compile time ----
// 128-byte-swizzled operand tiles (MMA descriptors, TMA tiles) start on 1 KB
constexpr bool kAligned1K(uint32_t off) { return off % 1024 == 0; }
static_assert(kAligned1K(OFF_A1) && kAligned1K(OFF_BUF0) && kAligned1K(OFF_BUF1) &&
              kAligned1K(OFF_G) && kAligned1K(OFF_S), "tile bases on 1 KB");
static_assert(kAligned1K(OFF_GR + GR_GA) && kAligned1K(OFF_GR + GR_RT) && kAligned1K(RT_HALF) &&
              kAligned1K(OFF_GR + GR_P) && kAligned1K(OFF_GR + GR_TB) && kAligned1K(OFF_GR + GR_U),
              "Gram-region tiles on 1 KB");
// regions in order, none running into the next
static_assert(OFF_A1 + 2 * 16384 <= OFF_BUF0, "A1: [K+; Q+], two K halves of 128 x 128 B");
static_assert(OFF_BUF0 + 16384 <= OFF_BUF1 && OFF_BUF1 + 16384 <= OFF_G, "k / v buffers, 64 x 256 B");
static_assert(OFF_G + kC * kD * 4 <= OFF_GR, "g tile fp32 [64][128]");
static_assert(2 * 8192 <= kC * kD * 4, "output staging (two 64-column bf16 halves) fits the g tile");
static_assert(OFF_GR + GR_RT + 2 * RT_HALF <= OFF_S && RT_HALF >= 160 * 128,
              "Gram right operand: 160 rows x 128 B per K half");
static_assert(GR_GA + 2 * 16384 <= GR_RT, "Gram left operand [kE; qE], two K halves");
static_assert(GR_P + 16384 <= GR_L && GR_L + kC * LST * 4 <= GR_TB && LST >= kC,
              "P, then L / T transposed with a padded stride");
static_assert(GR_TB + 16384 <= GR_U && OFF_GR + GR_U + 16384 <= OFF_S, "[Tb; 0], then U");
static_assert(11 * 16 * 20 * 4 <= 16384, "block-inverse scratch (11 blocks, row stride 20) inside U");
static_assert(OFF_S + 2 * 16384 <= OFF_VEC, "bf16 state copy, two N halves");
static_assert(VEC_DEC + kD * 4 <= OFF_BETA - OFF_VEC && VEC_SEG + 8 * kD * 4 <= VEC_DEC,
              "segment sums and chunk decay");
static_assert(OFF_BETA + kC * 4 <= OFF_BAR, "beta of a chunk");
static_assert(BAR_MMA1 + 8 <= OFF_MISC - OFF_BAR, "seven mbarriers");
static_assert(SMEM_BYTES <= 232448, "227 KB of dynamic shared memory per CTA");
// TMEM: D1 (128 columns), the Gram result (N = 160), the fp32 state (128)
static_assert(TM_D1 + 128 <= TM_G && TM_G + 160 <= TM_S && TM_S + kD <= TM_COLS && TM_COLS <= 512,
              "TMEM columns");

// first row / column of row tile a inside the stacked Gram operand / result
__device__ __forceinline__ uint32_t gram_off(int a) { return 8u * a * (a + 1); }  // 0,16,48,96
__device__ __forceinline__ uint32_t buf_off(int i) { return (i & 1) ? OFF_BUF1 : OFF_BUF0; }

struct Maps {
    CUtensorMap q, k, v, g, o;
};

// ---- 16x16x16 products for the block inverse, one warp each, on the
// warp-synchronous tensor-core path (mma.sync m16n8k8, tf32 in, fp32 out).
// Operands are rounded to tf32 (10-bit mantissa, 3 bits more than the bf16
// Tb they produce).  Fragment layout (g = lane / 4, t = lane % 4): A rows g
// and g+8, columns t and t+4 of each 8-wide K slice; B K-rows t and t+4,
// column g; D rows g and g+8, columns 2t and 2t+1 of each 8-wide N tile.
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
// acc += sign * A B for 16x16 fp32 blocks in shared memory: A(r, k) at A[r sa + k]
// (or A[k sa + r] when AT), B(k, n) at B[k sb + n] (or B[n sb + k] when BT)
template <bool NEG, bool AT, bool BT>
__device__ __forceinline__ void gemm16(float (&acc)[2][4], const float *A, int sa, const float *B, int sb,
                                       int lane) {
    const int g = lane >> 2, t = lane & 3;
    auto Ael = [&](int r, int k) { return AT ? A[k * sa + r] : A[r * sa + k]; };
    auto Bel = [&](int k, int n) { return BT ? B[n * sb + k] : B[k * sb + n]; };
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const float av[4] = {Ael(g, 8 * ks + t), Ael(g + 8, 8 * ks + t), Ael(g, 8 * ks + t + 4),
                             Ael(g + 8, 8 * ks + t + 4)};
        uint32_t a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = to_tf32(NEG ? -av[i] : av[i]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b[2] = {to_tf32(Bel(8 * ks + t, 8 * nt + g)), to_tf32(Bel(8 * ks + t + 4, 8 * nt + g))};
            mma_tf32(acc[nt], a, b);
        }
    }
}
// D-layout fragments from / to a row-major 16x16 fp32 block (row stride sc)
__device__ __forceinline__ void load_c16(float (&acc)[2][4], const float *C, int sc, int lane, float scale) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const float2 lo = *reinterpret_cast<const float2 *>(C + g * sc + 8 * nt + 2 * t);
        const float2 hi = *reinterpret_cast<const float2 *>(C + (g + 8) * sc + 8 * nt + 2 * t);
        acc[nt][0] = scale * lo.x; acc[nt][1] = scale * lo.y;
        acc[nt][2] = scale * hi.x; acc[nt][3] = scale * hi.y;
    }
}
__device__ __forceinline__ void store_c16(const float (&acc)[2][4], float *C, int sc, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2 *>(C + g * sc + 8 * nt + 2 * t) = make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2 *>(C + (g + 8) * sc + 8 * nt + 2 * t) = make_float2(acc[nt][2], acc[nt][3]);
    }
}

// element-wise product of two bf16 pairs, rounded to nearest
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&a), y = *reinterpret_cast<__nv_bfloat162 *>(&b);
    __nv_bfloat162 z = __hmul2(x, y);
    return *reinterpret_cast<uint32_t *>(&z);
}

// barrier 1: the six warps of the block inverse only
__device__ __forceinline__ void ut_sync() { asm volatile("bar.sync 1, 192;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1)
chunk_kernel(const __grid_constant__ Maps maps, const float *__restrict__ beta,
             const float *init_state, const int32_t *__restrict__ cu, int32_t N, int64_t T,
             int32_t H, __nv_bfloat16 *__restrict__ out, float *final_state,
             int32_t *__restrict__ status, const int32_t *__restrict__ order) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-aligned base, derived from the shared array so accesses stay in the shared window
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sp = warp & 3;          // TMEM sub-partition (lanes 32*sp .. 32*sp+31)
    const int qq = warp >> 2;         // which 32-column quarter this warp handles
    const int h = blockIdx.x;
    const int n = order ? order[blockIdx.y] : static_cast<int>(blockIdx.y);   // longest first
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + OFF_MISC);
#define SM_F(o) (*reinterpret_cast<float *>(smem + (o)))
#define SM_F4(o) (*reinterpret_cast<float4 *>(smem + (o)))
#define SM_U4(o) (*reinterpret_cast<uint4 *>(smem + (o)))
#define SM_H(o) (*reinterpret_cast<__nv_bfloat16 *>(smem + (o)))

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
        mbar_init(sb + OFF_BAR + BAR_MMA2, 2);
        mbar_init(sb + OFF_BAR + BAR_MMA1, 1);
        misc[1] = 0;
        for (int i = 2; i < 6; ++i) misc[i] = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(sb + OFF_MISC, TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const uint32_t tlane = tmem + ((uint32_t)(32 * sp) << 16);   // this warp's lanes

    // the state: row r = 32*sp + lane, columns 32*qq .. 32*qq+31, fp32 in TMEM
    // and bf16 in shared memory (N half qq >> 1, 16-byte chunks 4*(qq & 1) + i)
    const int srow = 32 * sp + lane;
    const uint32_t s_smem = OFF_S + (qq >> 1) * 16384;
    {
        float S[32];
        const float *src = init_state ? init_state + unit * kD * kD + (size_t)srow * kD + 32 * qq
                                      : nullptr;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float4 x = src ? *reinterpret_cast<const float4 *>(src + j)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
        }
        tmem_st32(tlane + TM_S + 32 * qq, S);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = S[8 * i + e];
            SM_U4(s_smem + sw128_off(srow, 4 * (qq & 1) + i)) = pack_bf16x8(x);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    auto issue_q = [&](int64_t t0) {
        mbar_expect_tx(sb + OFF_BAR + BAR_Q, 16384);
        tma_load_2d(sb + OFF_A1 + 8192, &maps.q, h * kD, (int32_t)t0, sb + OFF_BAR + BAR_Q);
        tma_load_2d(sb + OFF_A1 + 16384 + 8192, &maps.q, h * kD + 64, (int32_t)t0,
                    sb + OFF_BAR + BAR_Q);
    };
    auto issue_k = [&](int64_t t0, uint32_t buf) {
        mbar_expect_tx(sb + OFF_BAR + BAR_K, 16384);
        tma_load_2d(sb + buf, &maps.k, h * kD, (int32_t)t0, sb + OFF_BAR + BAR_K);
        tma_load_2d(sb + buf + 8192, &maps.k, h * kD + 64, (int32_t)t0, sb + OFF_BAR + BAR_K);
    };
    auto issue_v = [&](int64_t t0, uint32_t buf) {
        mbar_expect_tx(sb + OFF_BAR + BAR_V, 16384);
        tma_load_2d(sb + buf, &maps.v, h * kD, (int32_t)t0, sb + OFF_BAR + BAR_V);
        tma_load_2d(sb + buf + 8192, &maps.v, h * kD + 64, (int32_t)t0, sb + OFF_BAR + BAR_V);
    };
    auto issue_g = [&](int64_t t0) {
        mbar_expect_tx(sb + OFF_BAR + BAR_G, 32768);
        tma_load_2d(sb + OFF_G, &maps.g, h * kD, (int32_t)t0, sb + OFF_BAR + BAR_G);
    };

    // the loads are issued by threads of different warps (a TMA issue holds its
    // thread for a while); each records the chunk index in misc[2..5] (g, v, k,
    // q) so an aborting CTA can drain its own copies before it exits
    if (tid == 0 && nchunks > 0) {
        issue_q(bos);
        issue_k(bos, buf_off(0));
        issue_v(bos, buf_off(1));
        issue_g(bos);
    }
    // beta of the first chunk, held in a register by threads 0..63
    float beta_next = 0.f;
    if (tid < kC && nchunks > 0 && tid < len) beta_next = beta[(size_t)(bos + tid) * H + h];

    uint32_t mma_phase = 0, mma2_phase = 0, mma1_phase = 0;
    // all threads wait on the MMA barrier; a timeout raises the abort flag
    auto wait_mma = [&]() {
        if (!mbar_wait(sb + OFF_BAR + BAR_MMA, mma_phase)) misc[1] = 1;
        mma_phase ^= 1;
        tc_fence_after();
    };
    auto wait_mma2 = [&]() {
        if (!mbar_wait(sb + OFF_BAR + BAR_MMA2, mma2_phase)) misc[1] = 1;
        mma2_phase ^= 1;
        tc_fence_after();
    };
    auto wait_tma = [&](uint32_t bar, int c) {
        if (!mbar_wait(sb + OFF_BAR + bar, c & 1)) misc[1] = 1;
    };

    const uint32_t gr = sb + OFF_GR;    // shared address of the Gram region (descriptors)
    int c = 0;
    for (; c < nchunks; ++c) {
        const int64_t t0 = bos + (int64_t)c * kC;
        const int lenc = (eos - t0) < kC ? static_cast<int>(eos - t0) : kC;
        const uint32_t kbuf = buf_off(c), vbuf = buf_off(c + 1);

        // ---------------- step 1: this chunk's q/k/g tiles and beta
        if (tid < kC) {
            SM_F(OFF_BETA + 4 * tid) = beta_next;
            // the next chunk's beta: a whole chunk ahead, so that its latency is hidden
            if (c + 1 < nchunks)
                beta_next = (tid < eos - (t0 + kC)) ? beta[(size_t)(t0 + kC + tid) * H + h] : 0.f;
        }
        wait_tma(BAR_Q, c);
        wait_tma(BAR_K, c);
        wait_tma(BAR_G, c);
        __syncthreads();
        if (misc[1]) break;

        // ---------------- step 2: G and every decay-scaled operand, one pass.
        // warp = (channel half hh, row tile a, 8-token segment s8 of the tile),
        // lane = channel pair ch, ch+1: the running sum over the segment is
        // sequential in registers, the segment offsets go through shared memory,
        // and each operand row is stored as 32 bf16 pairs (one full 128-byte row).
        {
            const int hh = warp & 1, a = (warp >> 1) & 3, s8 = warp >> 3;
            const int ch = 64 * hh + 2 * lane;
            const int seg = 2 * a + s8, tb = 8 * seg;
            const uint32_t cw = sw128_off(0, lane >> 2) + 4 * (lane & 3);   // row-0 byte offset
            auto rowoff = [&](int row) { return (uint32_t)(row * 128) + (cw ^ ((row & 7) << 4)); };
            float2 G[8];
            {
                float2 run = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int t = tb + i;
                    const float2 gv = (t < lenc) ? *reinterpret_cast<const float2 *>(smem + OFF_G + (uint32_t)(t * kD + ch) * 4)
                                                 : make_float2(0.f, 0.f);
                    run.x += gv.x; run.y += gv.y;
                    G[i] = run;
                }
                *reinterpret_cast<float2 *>(smem + OFF_VEC + VEC_SEG + (uint32_t)(seg * kD + ch) * 4) = run;
            }
            __syncthreads();
            // the previous chunk's last MMAs (O += P U, S += Khat^T U) have run
            // while this chunk loaded and scanned: its P, U and Khat are free now
            if (c > 0) wait_mma2();
            // this chunk's v goes into the buffer that held the previous Khat (warp
            // 15 writes the fewest Gram rows in the pass below)
            if (tid == 480 && c > 0) {
                issue_v(t0, vbuf);
                misc[3] = c;
            }
            // segment boundaries (log2 units), as predicated running sums so that no
            // array is indexed at run time: G before this segment, before tile a
            // (s_a), after tile a (e_a), before every tile (for the Gram rows), G_63
            float2 base = make_float2(0.f, 0.f), sa = base, ea = base, g63 = base;
            float2 tile0[4];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                if ((m & 1) == 0) tile0[m >> 1] = make_float2(g63.x * kLog2e, g63.y * kLog2e);
                const float2 sv = *reinterpret_cast<const float2 *>(smem + OFF_VEC + VEC_SEG + (uint32_t)(m * kD + ch) * 4);
                if (m < seg) { base.x += sv.x; base.y += sv.y; }
                if (m < 2 * a) { sa.x += sv.x; sa.y += sv.y; }
                if (m < 2 * a + 2) { ea.x += sv.x; ea.y += sv.y; }
                g63.x += sv.x; g63.y += sv.y;
            }
            base.x *= kLog2e; base.y *= kLog2e;
            sa.x *= kLog2e; sa.y *= kLog2e;
            ea.x *= kLog2e; ea.y *= kLog2e;
            g63.x *= kLog2e; g63.y *= kLog2e;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                G[i].x = base.x + G[i].x * kLog2e;
                G[i].y = base.y + G[i].y * kLog2e;
            }
            if (warp >= 14)   // e^{G_63}, the state decay of the chunk
                *reinterpret_cast<float2 *>(smem + OFF_VEC + VEC_DEC + 4 * ch) = make_float2(ex2(g63.x), ex2(g63.y));
            // e^{s_ap - e_a} for the Gram right operand rows of tiles ap >= a
            uint32_t pv[4];
#pragma unroll
            for (int ap = 0; ap < 4; ++ap)
                pv[ap] = pack_bf16x2(ex2(tile0[ap].x - ea.x), ex2(tile0[ap].y - ea.y));
            const float2 gs = make_float2(ex2(sa.x), ex2(sa.y));                    // e^{s_a}
            const uint32_t kh = pack_bf16x2(ex2(g63.x - ea.x), ex2(g63.y - ea.y));    // e^{G_63 - e_a}
            float2 kE[8], qE[8];
            uint32_t kB[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = tb + i;
                uint32_t kraw = *reinterpret_cast<const uint32_t *>(smem + kbuf + hh * 8192 + rowoff(t));
                uint32_t qraw = *reinterpret_cast<const uint32_t *>(smem + OFF_A1 + hh * 16384 + rowoff(64 + t));
                if (t >= lenc) kraw = qraw = 0u;
                const float2 k2 = unpack_bf16x2(kraw), q2 = unpack_bf16x2(qraw);
                const float2 E = make_float2(ex2(G[i].x - sa.x), ex2(G[i].y - sa.y));
                const float2 Eb = make_float2(ex2(ea.x - G[i].x), ex2(ea.y - G[i].y));
                kE[i] = make_float2(k2.x * E.x, k2.y * E.y);
                qE[i] = make_float2(q2.x * E.x, q2.y * E.y);
                kB[i] = pack_bf16x2(k2.x * Eb.x, k2.y * Eb.y);
                // Gram left operand rows t (k) and 64 + t (q)
                *reinterpret_cast<uint32_t *>(smem + OFF_GR + GR_GA + hh * 16384 + rowoff(t)) =
                    pack_bf16x2(kE[i].x, kE[i].y);
                *reinterpret_cast<uint32_t *>(smem + OFF_GR + GR_GA + hh * 16384 + rowoff(64 + t)) =
                    pack_bf16x2(qE[i].x, qE[i].y);
                // Gram right operand: row gram_off(ap) + t for every row tile ap >= a
#pragma unroll
                for (int ap = 0; ap < 4; ++ap) {
                    if (ap < a) continue;
                    *reinterpret_cast<uint32_t *>(smem + OFF_GR + GR_RT + hh * RT_HALF + rowoff(gram_off(ap) + t)) =
                        mul_bf16x2(kB[i], pv[ap]);
                }
            }
            fence_proxy_async();
            __syncthreads();
            // ---------------- step 3: Gram MMAs (8 instructions, N = 160), issued
            // while the remaining operands are written
            if (tid == 0) {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 160, 0, 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = sw128_desc(gr + GR_GA + (kk >> 2) * 16384 + (kk & 3) * 32, 0, 1024);
                    const uint64_t bd = sw128_desc(gr + GR_RT + (kk >> 2) * RT_HALF + (kk & 3) * 32, 0, 1024);
                    mma_bf16(tmem + TM_G, ad, bd, id, kk > 0);
                }
                mma_commit(sb + OFF_BAR + BAR_MMA);
            }
            // Q+ = q e^{G} in place, K+ = k e^{G} into rows 0..63 of A1, Khat = k e^{G_63 - G} in place of k
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = tb + i;
                *reinterpret_cast<uint32_t *>(smem + OFF_A1 + hh * 16384 + rowoff(64 + t)) =
                    pack_bf16x2(qE[i].x * gs.x, qE[i].y * gs.y);
                *reinterpret_cast<uint32_t *>(smem + OFF_A1 + hh * 16384 + rowoff(t)) =
                    pack_bf16x2(kE[i].x * gs.x, kE[i].y * gs.y);
                *reinterpret_cast<uint32_t *>(smem + kbuf + hh * 8192 + rowoff(t)) = mul_bf16x2(kB[i], kh);
            }
        }
        fence_proxy_async();
        wait_mma();

        // ---------------- step 4: L (k rows) and P (q rows) out of TMEM
        {
            const int a = 2 * (sp & 1) + (qq >> 1);   // row tile this warp reads
            const int ch2 = qq & 1;                   // 32-column half of the tile's columns
            const bool mine = (lane >> 4) == (qq >> 1);
            const int t = 32 * (sp & 1) + lane;       // token of this lane
            float G[32];
            tmem_ld32(tlane + TM_G + gram_off(a) + 32 * ch2, G);
            if (mine) {
                if (sp < 2) {
                    // L stored transposed: L[t][j] at (j LST + t).  Unmasked: the
                    // block inverse reads only the strictly lower part of the
                    // diagonal blocks and the blocks below them
                    const float bt = SM_F(OFF_BETA + 4 * t);
                    float *Lt = reinterpret_cast<float *>(smem + OFF_GR + GR_L) + t;
#pragma unroll
                    for (int j = 0; j < 32; ++j) Lt[(32 * ch2 + j) * LST] = bt * G[j];
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int jj = 32 * ch2 + 8 * i + e;
                            x[e] = (jj <= t) ? G[8 * i + e] : 0.f;
                        }
                        SM_U4(OFF_GR + GR_P + sw128_off(64 + t, 4 * ch2 + i)) = pack_bf16x8(x);
                    }
                }
            }
            // rows 0..63 of [0; P] are zero
            SM_U4(OFF_GR + GR_P + sw128_off(tid >> 3, tid & 7)) = make_uint4(0, 0, 0, 0);
        }
        tc_fence_before();
        __syncthreads();

        // ---------------- step 5: T = (I + L)^-1 in fp32, written out as [Tb; 0], Tb = T diag(beta)
        if (warp < 6) {
            float *Lf = reinterpret_cast<float *>(smem + OFF_GR + GR_L);
            const float *betas = reinterpret_cast<const float *>(smem + OFF_BETA);
            // 5a: diagonal 16x16 blocks by forward substitution, column-oriented:
            // once x_i is known every later partial sum takes one FMA, so the
            // dependency chain is one FMA per row.  thread = (block a, column col)
            if (tid < 64) {
                const int a5 = tid >> 4, col = tid & 15;
                // the block in transposed storage: blk[i LST + k] = L[16 a5 + k][16 a5 + i]
                float *blk = Lf + 16 * a5 * LST + 16 * a5;
                float x[16], acc[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    x[i] = ((i == col) ? 1.f : 0.f) - acc[i];
                    // column i of the block is one contiguous row of the transposed storage
                    float lc[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (4 * q + 3 <= i) continue;
                        const float4 v = *reinterpret_cast<const float4 *>(blk + i * LST + 4 * q);
                        lc[4 * q] = v.x; lc[4 * q + 1] = v.y; lc[4 * q + 2] = v.z; lc[4 * q + 3] = v.w;
                    }
#pragma unroll
                    for (int k = i + 1; k < 16; ++k) acc[k] += lc[k] * x[i];
                }
                __syncwarp();
                // every thread of this warp has read its block: T_aa column col goes in
                // place (transposed storage, as L), and its Tb column (zero above the
                // diagonal, as x_i = 0 for i < col)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<float4 *>(blk + col * LST + 4 * q) =
                        make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
                const int j = 16 * a5 + col;
                const float bj = betas[j];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    SM_H(OFF_GR + GR_TB + sw128_off(16 * a5 + i, j >> 3) + (j & 7) * 2) =
                        __float2bfloat16_rn(x[i] * bj);

            }
            ut_sync();
            // 5b: off-diagonal blocks.  With D = blockdiag(T_aa) and N the
            // strictly block-lower part of L, (I + L) = (I + N D) D^-1, so
            // T = D (I + M)^-1 = D (I - M + M^2 - M^3) with M = N D (block
            // nilpotent).  Stage 1 forms the six M_ab = L_ab T_bb; stage 2 gives
            //   T_{a,a-1} = -T_aa M_{a,a-1},  V20 = M21 M10 - M20,
            //   V31 = M32 M21 - M31,  Y30 = M31 M10 - M30;
            // stage 3: T20 = T22 V20, T31 = T33 V31 and, with T32 = -T33 M32,
            //   T30 = T33 (Y30 - M32 V20) = T33 Y30 + T32 V20.
            // One warp per output block (T30's second product on warp 0, which is
            // free in stage 3); scratch blocks fp32, row stride 20.
            constexpr int XS = 20;
            float *X = reinterpret_cast<float *>(smem + OFF_GR + GR_U);
            auto XB = [&](int i) { return X + i * 16 * XS; };
            // block (a, b) of L or T in the transposed storage: element (r, k) at [k LST + r]
            auto LB = [&](int a, int b) { return Lf + 16 * b * LST + 16 * a; };
            enum { M10 = 0, M21, M32, M20, M31, M30, V20, V31, Y30, T32F, P30 };
            // Tb block (ta, tb) = sgn * acc, column-scaled by beta, in bf16:
            // rows 16 ta + g (+8), columns 16 tb + 8 nt + 2t (+1)
            auto tb_store = [&](int ta, int tb, float sgn, const float (&acc)[2][4]) {
                const int g = lane >> 2, t = lane & 3;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int col = 16 * tb + 8 * nt + 2 * t;
                    const float2 bb = *reinterpret_cast<const float2 *>(betas + col);
                    *reinterpret_cast<uint32_t *>(smem + OFF_GR + GR_TB + sw128_off(16 * ta + g, 2 * tb + nt) + 4 * t) =
                        pack_bf16x2(sgn * acc[nt][0] * bb.x, sgn * acc[nt][1] * bb.y);
                    *reinterpret_cast<uint32_t *>(smem + OFF_GR + GR_TB + sw128_off(16 * ta + g + 8, 2 * tb + nt) + 4 * t) =
                        pack_bf16x2(sgn * acc[nt][2] * bb.x, sgn * acc[nt][3] * bb.y);
                }
            };
            {
                // stage 1, (a, b) = (1,0) (2,1) (3,2) (2,0) (3,1) (3,0)
                const int a = warp < 3 ? warp + 1 : (warp == 3 ? 2 : 3);
                const int b = warp < 3 ? warp : (warp == 4 ? 1 : 0);
                float acc[2][4] = {};
                gemm16<false, true, true>(acc, LB(a, b), LST, LB(b, b), LST, lane);
                store_c16(acc, XB(warp), XS, lane);
            }
            ut_sync();
            {
                // stage 2
                float acc[2][4] = {};
                if (warp < 3) {
                    const int a = warp + 1;
                    gemm16<false, true, false>(acc, LB(a, a), LST, XB(M10 + warp), XS, lane);
                    tb_store(a, a - 1, -1.f, acc);
                    if (warp == 2) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i >> 2][i & 3] = -acc[i >> 2][i & 3];
                        store_c16(acc, XB(T32F), XS, lane);
                    }
                } else {
                    // V20 = M21 M10 - M20, V31 = M32 M21 - M31, Y30 = M31 M10 - M30
                    const int left = warp == 3 ? M21 : (warp == 4 ? M32 : M31);
                    const int right = warp == 4 ? M21 : M10;
                    const int sub = warp == 3 ? M20 : (warp == 4 ? M31 : M30);
                    load_c16(acc, XB(sub), XS, lane, -1.f);
                    gemm16<false, false, false>(acc, XB(left), XS, XB(right), XS, lane);
                    store_c16(acc, XB(V20 + (warp - 3)), XS, lane);
                }
            }
            ut_sync();
            if (warp == 0) {
                // stage 3, the second half of T30: T32 V20 -> scratch, handed to warp 5
                float acc[2][4] = {};
                gemm16<false, false, false>(acc, XB(T32F), XS, XB(V20), XS, lane);
                store_c16(acc, XB(P30), XS, lane);
                asm volatile("bar.arrive 4, 64;" ::: "memory");
            } else if (warp >= 3) {
                // stage 3
                float acc[2][4] = {};
                if (warp == 3) {
                    gemm16<false, true, false>(acc, LB(2, 2), LST, XB(V20), XS, lane);
                    tb_store(2, 0, 1.f, acc);
                } else if (warp == 4) {
                    gemm16<false, true, false>(acc, LB(3, 3), LST, XB(V31), XS, lane);
                    tb_store(3, 1, 1.f, acc);
                } else {
                    gemm16<false, true, false>(acc, LB(3, 3), LST, XB(Y30), XS, lane);
                    asm volatile("bar.sync 4, 64;" ::: "memory");
                    float part[2][4];
                    load_c16(part, XB(P30), XS, lane, 1.f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i >> 2][i & 3] += part[i >> 2][i & 3];
                    tb_store(3, 0, 1.f, acc);
                }
            }
        } else {
            // warps 6..15, alongside the block inverse: the previous chunk's outputs
            // out of D1, the incoming state's bf16 copy and pre-scale, [K+; Q+] S
            // into D1 and V - K+ S; then the zero parts of [Tb; 0].  First the next
            // chunk's tiles into L2, so that their loads, issued late in this chunk,
            // hit L2
            if (tid == 224 && c + 1 < nchunks) {
                const int32_t y1 = (int32_t)(t0 + kC);
                tma_prefetch_2d(&maps.q, h * kD, y1);
                tma_prefetch_2d(&maps.q, h * kD + 64, y1);
                tma_prefetch_2d(&maps.g, h * kD, y1);
                tma_prefetch_2d(&maps.k, h * kD, y1);
                tma_prefetch_2d(&maps.k, h * kD + 64, y1);
                tma_prefetch_2d(&maps.v, h * kD, y1);
                tma_prefetch_2d(&maps.v, h * kD + 64, y1);
            }
            const int w6 = warp - 6;   // 0..9
            if (w6 == 0 || w6 == 1) {
                // warps 6 (lanes 64..95) and 7 (lanes 96..127): the previous chunk's
                // outputs, one token row per lane, into the staging tile (the g tile
                // is scanned), then out with two bulk tensor stores
                if (c > 0) {
                    const int t = 32 * (sp - 2) + lane;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        float v32[32];
                        tmem_ld32(tlane + TM_D1 + 32 * q4, v32);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float x[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) x[e] = v32[8 * i + e];
                            SM_U4(OFF_G + (q4 >> 1) * 8192 + sw128_off(t, 4 * (q4 & 1) + i)) = pack_bf16x8(x);
                        }
                    }
                    fence_proxy_async();
                }
                asm volatile("bar.sync 3, 64;" ::: "memory");
                if (tid == 192 && c > 0) {
                    tma_store_2d(&maps.o, h * kD, (int32_t)(t0 - kC), sb + OFF_G);
                    tma_store_2d(&maps.o, h * kD + 64, (int32_t)(t0 - kC), sb + OFF_G + 8192);
                    bulk_commit();
                }
            } else {
                // warps 8..15: the incoming state (rows 32 sp .., 64 columns each):
                // its bf16 copy for this chunk's K+ S and Q+ S, then S <- Diag(e^{G_63}) S
                // in TMEM so that the chunk's Khat^T U accumulates into it
                const int c64 = (w6 - 2) >> 2;          // column half
                const int row = 32 * sp + lane;
                const uint32_t sdst = OFF_S + c64 * 16384;
                const float dec = SM_F(OFF_VEC + VEC_DEC + 4 * row);
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    float v32[32];
                    tmem_ld32(tlane + TM_S + 64 * c64 + 32 * q2, v32);
                    if (c > 0) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float x[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) x[e] = v32[8 * i + e];
                            SM_U4(sdst + sw128_off(row, 4 * q2 + i)) = pack_bf16x8(x);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) v32[j] *= dec;
                    tmem_st32_nowait(tlane + TM_S + 64 * c64 + 32 * q2, v32);
                }
                tmem_wait_st();
                fence_proxy_async();
            }
            // [K+; Q+] S into D1 once the outputs have left it and the copy is in place:
            // rows 0..63 K+ S, rows 64..127 Q+ S (to which P U is added later)
            tc_fence_before();
            asm volatile("bar.sync 5, 320;" ::: "memory");
            if (tid == 192) {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = sw128_desc(sb + OFF_A1 + (kk >> 2) * 16384 + (kk & 3) * 32, 0, 1024);
                    const uint64_t bd = sw128_desc(sb + OFF_S + kk * 2048, 16384, 1024);
                    mma_bf16(tmem + TM_D1, ad, bd, id, kk > 0);
                }
                mma_commit(sb + OFF_BAR + BAR_MMA1);
                // the stores have read the staging tile: the next chunk's g tile goes there
                if (c + 1 < nchunks) {
                    bulk_wait_read_all();
                    issue_g(t0 + kC);
                    misc[2] = c + 1;
                }
            }
            if (w6 >= 2 && sp < 2) {
                // warps 8, 9, 12, 13 (TMEM lanes 0..63): V - K+ S into the v buffer as
                // the B operand of U = Tb (V - K+ S), and D1 rows 0..63 cleared for it
                if (!mbar_wait(sb + OFF_BAR + BAR_MMA1, mma1_phase)) misc[1] = 1;
                tc_fence_after();
                wait_tma(BAR_V, c);
                const int c64 = (w6 - 2) >> 2;
                const int t = 32 * sp + lane;
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    float y32[32];
                    tmem_ld32(tlane + TM_D1 + 64 * c64 + 32 * q2, y32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t off = vbuf + c64 * 8192 + sw128_off(t, 4 * q2 + i);
                        float xv[8];
                        unpack_bf16x8(SM_U4(off), xv);
#pragma unroll
                        for (int e = 0; e < 8; ++e) xv[e] -= y32[8 * i + e];
                        SM_U4(off) = pack_bf16x8(xv);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) y32[j] = 0.f;
                    tmem_st32_nowait(tlane + TM_D1 + 64 * c64 + 32 * q2, y32);
                }
                tmem_wait_st();
                fence_proxy_async();
            } else if (w6 == 9) {
                // warp 15: q of the next chunk once [K+; Q+] S has read A1
                if (!mbar_wait(sb + OFF_BAR + BAR_MMA1, mma1_phase)) misc[1] = 1;
                if (tid == 480 && c + 1 < nchunks) {
                    issue_q(t0 + kC);
                    misc[5] = c + 1;
                }
            }
            // rows 64..127, and the blocks above the diagonal (row tile a, 16-byte
            // chunks 2(a+1)..7)
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int i = tid - 192; i < 512 + 192; i += kThreads - 192) {
                if (i < 512) {
                    SM_U4(OFF_GR + GR_TB + sw128_off(64 + (i >> 3), i & 7)) = z;
                } else {
                    const int j = i - 512;
                    const int row = j < 96 ? j / 6 : (j < 160 ? 16 + (j - 96) / 4 : 32 + (j - 160) / 2);
                    const int ch = j < 96 ? 2 + j % 6 : (j < 160 ? 4 + (j - 96) % 4 : 6 + (j - 160) % 2);
                    SM_U4(OFF_GR + GR_TB + sw128_off(row, ch)) = z;
                }
            }
        }
        mma1_phase ^= 1;
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ---------------- step 6: D1 rows 0..63 += Tb (V - K+ S) = U; rows 64..127 keep Q+ S
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sw128_desc(gr + GR_TB + kk * 32, 0, 1024);
                mma_bf16(tmem + TM_D1, ad, sw128_desc(sb + vbuf + kk * 2048, 8192, 1024), id, 1);
            }
            mma_commit(sb + OFF_BAR + BAR_MMA);
        }
        wait_mma();
        // v is consumed: the next chunk's k goes into its buffer
        if (tid == 448 && c + 1 < nchunks) {
            issue_k(t0 + kC, vbuf);
            misc[4] = c + 1;
        }

        // ---------------- step 7: U (D1 rows 0..63) -> bf16 MN-major B operand
        if (sp < 2) {
            const int t = 32 * sp + lane;
            float v32[32];
            tmem_ld32(tlane + TM_D1 + 32 * qq, v32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = v32[8 * i + e];
                SM_U4(OFF_GR + GR_U + (qq >> 1) * 8192 + sw128_off(t, 4 * (qq & 1) + i)) = pack_bf16x8(x);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ---------------- step 8: O = Q+ S + P U (D1 rows 64..127), S += Khat^T U.
        // Not waited for here: the next chunk's loads and scan run meanwhile.
        // Two issuing threads (warps 0 and 1), one per accumulator.
        if (tid == 0 || tid == 32) {
            tc_fence_after();
            const bool o_part = tid == 0;
            const uint32_t id = o_part ? idesc_bf16(128, 128, 0, 1) : idesc_bf16(128, 128, 1, 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = sw128_desc(gr + GR_U + kk * 2048, 8192, 1024);
                const uint64_t ad = o_part ? sw128_desc(gr + GR_P + kk * 32, 0, 1024)
                                           : sw128_desc(sb + kbuf + kk * 2048, 8192, 1024);
                mma_bf16(tmem + (o_part ? TM_D1 : TM_S), ad, bd, id, 1);
            }
            mma_commit(sb + OFF_BAR + BAR_MMA2);
        }
    }

    // the last chunk: its outputs once its last MMAs are done
    if (!misc[1] && nchunks > 0) {
        wait_mma2();
        if (sp >= 2) {
            const int64_t tl = bos + (int64_t)(nchunks - 1) * kC;
            const int t = 32 * (sp - 2) + lane;
            float v32[32];
            tmem_ld32(tlane + TM_D1 + 32 * qq, v32);
            if (tl + t < eos) {
                uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)(tl + t) * H + h) * kD + 32 * qq);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = v32[8 * i + e];
                    dst[i] = pack_bf16x8(x);
                }
            }
        }
    }

    if (misc[1]) {
        // a wait gave up: report, let this CTA's own copies and MMAs drain
        if (tid == 0) {
            flag_status(status, KDA_DEVICE_TIMEOUT);
            mbar_wait(sb + OFF_BAR + BAR_MMA, mma_phase, 100000000ull);
            mbar_wait(sb + OFF_BAR + BAR_MMA2, mma2_phase, 100000000ull);
            mbar_wait(sb + OFF_BAR + BAR_MMA1, mma1_phase, 100000000ull);
            const int issued[4] = {(int)misc[5], (int)misc[4], (int)misc[3], (int)misc[2]};
            const uint32_t bars[4] = {BAR_Q, BAR_K, BAR_V, BAR_G};
            for (int i = 0; i < 4; ++i)
                if (issued[i] >= c)   // issued for this chunk or the next, maybe not landed
                    mbar_wait(sb + OFF_BAR + bars[i], issued[i] & 1, 100000000ull);
        }
    } else if (final_state != nullptr) {
        tc_fence_after();
        float S[32];
        tmem_ld32(tlane + TM_S + 32 * qq, S);
        float *dst = final_state + unit * kD * kD + (size_t)srow * kD + 32 * qq;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    if (tid == 192) bulk_wait_all();   // the output stores of thread 192 are complete
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
#undef SM_F
#undef SM_F4
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
                                 cudaStream_t stream, const int32_t *order) {
    Maps maps;
    if (!make_map(&maps.q, q, T, H, false) || !make_map(&maps.k, k, T, H, false) ||
        !make_map(&maps.v, v, T, H, false) || !make_map(&maps.g, g, T, H, true) ||
        !make_map(&maps.o, out, T, H, false))
        return cudaErrorInvalidValue;
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = allow_dynamic_smem(chunk_kernel, SMEM_BYTES, smem_set);
    if (e != cudaSuccess) return e;
    chunk_kernel<<<dim3(H, N), kThreads, SMEM_BYTES, stream>>>(
        maps, beta, init_state, cu_seqlens, N, T, H, static_cast<__nv_bfloat16 *>(out),
        final_state, status, order);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
