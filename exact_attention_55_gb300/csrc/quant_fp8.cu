// quant_fp8.cu -- per-block FP8-E4M3 quantisation of a bf16 [BH, N, d] tensor.
//
// "Warp Group Cluster 优化：Flash Attention V3 在 H100 上的 FP8 融合计算实践",
// §3 FP8 量化与精度保持: a scale factor computed per block maps the block's range
// onto the FP8 range (largest E4M3 magnitude 448); "大模型加速-核心网络算子-
// Flash Attention V3", §1 item 3 / §1.5: block quantisation into E4M3.
//
// For each (head, block of 128 rows, all d columns):
//   amax  = max |x|;  scale = amax / 448 (IEEE fp32 division), or 1 when amax == 0
//   x8    = e4m3_rn_satfinite(x / scale)   (IEEE fp32 division, one rounding to E4M3)
// The kernel is HBM-bound: it reads each bf16 element once (kept in registers for
// the second pass) and writes one byte per element plus one float per block.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_params.h"
#include "ptx.cuh"

namespace gb300 {

constexpr int kQuantThreads = 256;
constexpr int kQuantRows = 128;
// 16-element groups per thread: 128 rows * 256 cols / 16 / 256 threads
constexpr int kQuantGroupsPerThread = 8;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(kQuantThreads) quant_fp8_kernel(const QuantParams p)
{
    __shared__ float warp_max[kQuantThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = p.BH * p.nblk;
    for (int blk = blockIdx.x; blk < total; blk += gridDim.x) {
        const int bh = blk / p.nblk, b = blk % p.nblk;
        const int r0 = b * kQuantRows;
        const int rows = min(kQuantRows, p.N - r0);
        const size_t base = ((size_t)bh * p.N + r0) * p.d;  // element offset of the block
        const int ngroups = rows * p.d / 16;
        const uint4* src = reinterpret_cast<const uint4*>(
            reinterpret_cast<const __nv_bfloat16*>(p.x) + base);
        uint4 raw[kQuantGroupsPerThread][2];
        float amax = 0.0f;
#pragma unroll
        for (int v = 0; v < kQuantGroupsPerThread; ++v) {
            const int g = threadIdx.x + v * kQuantThreads;
            if (g < ngroups) {
                raw[v][0] = __ldcs(src + 2 * g);
                raw[v][1] = __ldcs(src + 2 * g + 1);
                const uint32_t* w = reinterpret_cast<const uint32_t*>(raw[v]);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
            }
        }
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, s));
        if (lane == 0) warp_max[warp] = amax;
        __syncthreads();
        amax = warp_max[0];
#pragma unroll
        for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
        const float scale = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;

        uint4* dst = reinterpret_cast<uint4*>(p.x8 + base);
#pragma unroll
        for (int v = 0; v < kQuantGroupsPerThread; ++v) {
            const int g = threadIdx.x + v * kQuantThreads;
            if (g < ngroups) {
                const uint32_t* w = reinterpret_cast<const uint32_t*>(raw[v]);
                uint32_t out[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t lo = pack_e4m3x2(__fdiv_rn(bf16_lo(w[2 * e]), scale),
                                                    __fdiv_rn(bf16_hi(w[2 * e]), scale));
                    const uint32_t hi = pack_e4m3x2(__fdiv_rn(bf16_lo(w[2 * e + 1]), scale),
                                                    __fdiv_rn(bf16_hi(w[2 * e + 1]), scale));
                    out[e] = lo | (hi << 16);
                }
                __stcs(dst + g, make_uint4(out[0], out[1], out[2], out[3]));
            }
        }
        if (threadIdx.x == 0) p.scales[blk] = scale;
        __syncthreads();  // warp_max is reused by the next block
    }
}

cudaError_t launch_quant_fp8(const QuantParams& p, int sm_count, cudaStream_t stream)
{
    const int total = p.BH * p.nblk;
    int grid = sm_count * (2048 / kQuantThreads);
    if (grid > total) grid = total;
    quant_fp8_kernel<<<grid, kQuantThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gb300
