// kda_epilogue.cu -- the step after the recurrent read: head-wise RMSNorm and
// the full-rank output gate ("From GPT-2 to Kimi K3, from first principles",
// Chapter 5 "A third gate: control what leaves the module"; "Kimi K3
// Architecture Explained", "Inside a KDA Layer": the result is normalised and
// multiplied element-wise by an output gate; infra diagram KDA card "Head
// RMSNorm + gate").  The gate logits W_g x are an input (the projection needs
// trained weights):
//     y[r, c] = o[r, c] / sqrt(mean_c o[r, c]^2 + eps) * w[c] * sigmoid(z[r, c])
// d/8 lanes per row (token, head), 8 channels per lane; HBM-bound: o and z
// read once, y written once.  The bf16 kernel keeps its two 16-byte loads as
// packed pairs and reads the weights inside the loop, so that it fits 32
// registers and eight 256-thread blocks fill an SM: the loads in flight per SM
// are what sets its bandwidth.
#include "kda_internal.cuh"

#include <type_traits>

namespace kda {
namespace {

template <typename Tin, int D>
__global__ void __launch_bounds__(256)
output_gate_kernel(const Tin *__restrict__ o, const Tin *__restrict__ z,
                   const float *__restrict__ weight, int64_t rows, float eps,
                   Tin *__restrict__ y) {
    // 8 channels (one 16-byte load for bf16) per lane; LPR lanes per row
    constexpr int LPR = D / 8;
    constexpr int RPW = 32 / LPR;                       // rows per warp
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR, slot = lane / LPR;
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5) * RPW;
    float w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = weight ? weight[sub * 8 + e] : 1.f;
    for (int64_t row = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW + slot;
         row - slot < rows; row += stride) {
        const bool live = row < rows;
        float ov[8], zv[8];
        float ss = 0.f;
        if (live) {
            Elem<Tin>::load8(o + row * D + sub * 8, ov);
            Elem<Tin>::load8(z + row * D + sub * 8, zv);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss += ov[e] * ov[e];
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = rsqrtf(ss / D + eps);
        if (live) {
            float yv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                yv[e] = ov[e] * inv * w[e] * __fdividef(1.f, 1.f + __expf(-zv[e]));
            Elem<Tin>::store8(y + row * D + sub * 8, yv);
        }
    }
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

template <int D>
__global__ void __launch_bounds__(256, 8)
output_gate_bf16_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ z,
                        const float *__restrict__ weight, int64_t rows, float eps,
                        __nv_bfloat16 *__restrict__ y) {
    constexpr int LPR = D / 8;
    constexpr int RPW = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR, slot = lane / LPR;
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5) * RPW;
    const float4 *w4 = reinterpret_cast<const float4 *>(weight + sub * 8);
    for (int64_t row = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW + slot;
         row - slot < rows; row += stride) {
        const bool live = row < rows;
        uint4 ro = make_uint4(0u, 0u, 0u, 0u), rz = ro;
        if (live) {
            ro = __ldg(reinterpret_cast<const uint4 *>(o + row * D + sub * 8));
            rz = __ldg(reinterpret_cast<const uint4 *>(z + row * D + sub * 8));
        }
        const uint32_t po[4] = {ro.x, ro.y, ro.z, ro.w}, pz[4] = {rz.x, rz.y, rz.z, rz.w};
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 a = bf16x2_to_float2(po[e]);
            ss += a.x * a.x;
            ss += a.y * a.y;
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = rsqrtf(ss / D + eps);
        if (live) {
            float4 wa = make_float4(1.f, 1.f, 1.f, 1.f), wb = wa;
            if (weight) {
                wa = __ldg(w4);
                wb = __ldg(w4 + 1);
            }
            const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
            uint32_t packed[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a = bf16x2_to_float2(po[e]), b = bf16x2_to_float2(pz[e]);
                const float y0 = a.x * inv * wv[2 * e] * __fdividef(1.f, 1.f + __expf(-b.x));
                const float y1 = a.y * inv * wv[2 * e + 1] * __fdividef(1.f, 1.f + __expf(-b.y));
                const __nv_bfloat162 pr = __floats2bfloat162_rn(y0, y1);
                packed[e] = *reinterpret_cast<const uint32_t *>(&pr);
            }
            *reinterpret_cast<uint4 *>(y + row * D + sub * 8) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
    }
}

template <typename Tin, int D>
cudaError_t run(const void *o, const void *z, const float *weight, int64_t rows, float eps,
                void *y, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t rows_per_block = 8 * (32 / (D / 8));
    int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        // four waves of eight resident blocks per SM
        if (blocks > (int64_t)sms * 32) blocks = (int64_t)sms * 32;
        output_gate_bf16_kernel<D><<<(unsigned)blocks, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(z), weight,
            rows, eps, static_cast<__nv_bfloat16 *>(y));
    } else {
        if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
        output_gate_kernel<Tin, D><<<(unsigned)blocks, 256, 0, stream>>>(
            static_cast<const Tin *>(o), static_cast<const Tin *>(z), weight, rows, eps,
            static_cast<Tin *>(y));
    }
    count_launches(1);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t run_d(const void *o, const void *z, const float *weight, int64_t rows, int32_t D,
                  float eps, void *y, cudaStream_t stream) {
    switch (D) {
    case 16: return run<Tin, 16>(o, z, weight, rows, eps, y, stream);
    case 32: return run<Tin, 32>(o, z, weight, rows, eps, y, stream);
    case 64: return run<Tin, 64>(o, z, weight, rows, eps, y, stream);
    case 128: return run<Tin, 128>(o, z, weight, rows, eps, y, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_output_gate(const void *o, const void *z, const float *weight, int64_t rows,
                               int32_t D, kda_dtype dt, float eps, void *y, cudaStream_t stream) {
    if (dt == KDA_BF16) return run_d<__nv_bfloat16>(o, z, weight, rows, D, eps, y, stream);
    return run_d<float>(o, z, weight, rows, D, eps, y, stream);
}

}  // namespace kda
