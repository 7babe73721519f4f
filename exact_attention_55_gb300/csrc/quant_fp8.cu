// quant_fp8.cu -- per-block FP8 quantisation (E4M3, or E5M2) of a bf16 [BH, N, d] tensor.
//
// "Warp Group Cluster 优化：Flash Attention V3 在 H100 上的 FP8 融合计算实践",
// §3 FP8 量化与精度保持: a scale factor computed per block maps the block's range
// onto the FP8 range (largest E4M3 magnitude 448); "大模型加速-核心网络算子-
// Flash Attention V3", §1 item 3 / §1.5: block quantisation into E4M3.
//
// For each (head, block of 128 rows -- or 64, the head-dim-aware block of Q and K at
// d = 64 -- all d columns):
//   amax  = max |x|;  scale = amax / 448 (IEEE fp32 division), or 1 when amax == 0
//   x8    = e4m3_rn_satfinite(x / scale)   (IEEE fp32 quotient, one rounding to E4M3)
// The E5M2 variant (the pages' wider-range format, "大模型加速-核心网络算子-Flash
// Attention V3" §1.5) divides amax by 57344, its largest finite value, and rounds
// the same quotient to E5M2.  The power-of-two variant keeps E4M3 codes but takes the
// smallest power of two at or above amax / 448 as the block's scale (a shared exponent),
// so that the quotient is exact and ratios of two blocks' scales are powers of two.
//
// HBM-bound design: persistent CTAs, as many per SM as fit (two at d = 128),
// each stream whole blocks (one contiguous run of rows * d * 2 bytes) into a
// 3-stage shared-memory ring with cp.async.bulk, so several blocks are in flight
// per SM while the threads reduce and convert the current one.  Each element is
// read from HBM once and written as one byte.
//
// With rotation (incoherent processing, "大模型加速-核心网络算子-Flash Attention
// V3" §1 item 3: 块量化和无相关处理), each row is first multiplied by the
// orthonormal Walsh-Hadamard matrix H_d / sqrt(d), computed in fp32 as the
// radix-2 butterfly sweep h = 1, 2, ..., d/2 -- each pair (i, i + h), (i & h) == 0,
// becomes (a + b, a - b) -- followed by one multiply by c = fp32(1 / sqrt(d)); the
// block's amax and codes are then taken over the rotated values.  TPR threads
// share a row (TPR = 4): thread q holds the 16-byte
// chunks q, q + TPR, q + 2 TPR, ... of it, so element index bits 0-2 and the bits
// above the chunk-lane bits are inside a thread, while the stages h = 8 .. 4 TPR
// exchange with lanes q ^ 1 and q ^ 2 by shuffles.  Every butterfly rounds
// exactly as in the sweep, so the codes do not depend on the split.
//
// The quotient x / scale is formed from the correctly rounded reciprocal
// y = RN(1/scale) with one residual correction, q = RN(x*y), r = x - scale*q
// (exact with an FMA), q' = RN(q + r*y) -- Markstein's final division step
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990), which gives the correctly
// rounded quotient without a per-element divide.  The GPU tests compare the
// result bit for bit with the oracle's IEEE division over every pair of bf16
// mantissas.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_params.h"
#include "ptx.cuh"

namespace gb300 {

constexpr int kQuantRows = 128;
constexpr int kQuantStages = 3;

// Dynamic shared memory: alignment slack, kQuantStages blocks of 128 * d bf16, barriers.
__host__ __device__ constexpr int quant_smem_bytes(int d)
{
    return 128 + kQuantStages * kQuantRows * d * 2 + 64;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Per half: the larger of two bf16 values (a NaN loses to the other operand, as in fmaxf).
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// RN(x / s) for two values at once, s > 0 finite and the quotients normal, from
// y = RN(1/s) and s_neg = -s: q = RN(x y), r = x - q s (exact), RN(q + r y).
__device__ __forceinline__ float2 div2_by_scale(float2 x, float2 s_neg, float2 y)
{
    const float2 q = __fmul2_rn(x, y);
    const float2 r = __ffma2_rn(q, s_neg, x);  // x - q s, exact
    const float2 c = __ffma2_rn(r, y, q);
    // c equals q when r == 0, except that q = -0 (x = -0) would come back as +0;
    // the quotient's sign is x's in every case
    return make_float2(copysignf(c.x, x.x), copysignf(c.y, x.y));
}

// a + b and a - b of two pairs, each rounded once (a - b as fma(b, -1, a)).
__device__ __forceinline__ void butterfly2(float& a0, float& a1, float& b0, float& b1)
{
    const float2 a = make_float2(a0, a1), b = make_float2(b0, b1);
    const float2 sum = __fadd2_rn(a, b);
    const float2 dif = __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
    a0 = sum.x; a1 = sum.y;
    b0 = dif.x; b1 = dif.y;
}

// Launch shape per variant: plain, 512 threads; rotated, a 128-row block with one thread
// per row at d = 64 (all butterflies in registers, no shuffles), two at d = 128 (one
// shuffle stage) and four at d = 256.  Measured per B16 H16 N8192 tensor: one thread per
// row was 24 % faster than four at d = 64 but 12 % slower at d = 128 (254 registers a
// thread leave two 4-warp CTAs per SM); two were 2 % faster than four at d = 128.
// Rotated d <= 128: two or more CTAs per SM.
template <int DR> struct QuantShape {
    static constexpr int TPR = (DR == 64) ? 1 : (DR == 128 ? 2 : 4);
    static constexpr int kThreads = (DR == 0) ? 512 : kQuantRows * TPR;
    static constexpr int kMinBlocks = (DR > 0 && DR <= 128) ? 2 : 1;
};

// DR = 0: plain per-block quantisation (any d); DR = d in {64, 128, 256}: rotate first.
// FMT = 0: E4M3; FMT = 1: E5M2; FMT = 2: E4M3 with power-of-two scales (plain only).

// The smallest power of two >= s (s > 0 finite), normal or subnormal.
__device__ __forceinline__ float pow2_at_least(float s)
{
    const uint32_t b = __float_as_uint(s);
    if ((b & 0x7F800000u) == 0) {  // subnormal: 2^k >= m * 2^-149 from m's highest bit
        const uint32_t m = b & 0x7FFFFFu;
        return __uint_as_float((m & (m - 1)) == 0 ? m : (1u << (32 - __clz(m))));
    }
    return (b & 0x7FFFFFu) == 0 ? s : __uint_as_float((b & 0x7F800000u) + 0x00800000u);
}
template <int DR, int FMT = 0>
__global__ void __launch_bounds__(QuantShape<DR>::kThreads, QuantShape<DR>::kMinBlocks)
    quant_fp8_kernel(const QuantParams p)
{
    constexpr int kThreads = QuantShape<DR>::kThreads;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                               ~uintptr_t(127));
    const int stage_bytes = kQuantRows * p.d * 2;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQuantStages * stage_bytes);
    __shared__ float warp_max[kThreads / 32];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = p.BH * p.nblk;
    const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(p.x);

    // blocks of p.rows rows (128, or 64); a stage holds the largest block, 128 rows
    auto block_rows = [&](int blk) { return min(p.rows, p.N - (blk % p.nblk) * p.rows); };
    auto block_base = [&](int blk) {  // element offset of the block
        return ((size_t)(blk / p.nblk) * p.N + (size_t)(blk % p.nblk) * p.rows) * p.d;
    };
    // load the block of iteration `j` of this CTA into its stage (the test hook withholds
    // one iteration's load: its wait then runs out)
    auto issue = [&](int j) {
        if (j + 1 == p.withhold) return;
        const int blk = blockIdx.x + j * gridDim.x, stage = j % kQuantStages;
        const uint32_t bytes = (uint32_t)block_rows(blk) * p.d * 2;
        const uint32_t bar = smem_u32(&full[stage]);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(smem_u32(smem + stage * stage_bytes), x + block_base(blk), bytes, bar);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQuantStages; ++s) mbar_init(smem_u32(&full[s]), 1);
        abort_flag = 0;
        fence_mbar_init();
        for (int s = 0; s < kQuantStages; ++s)
            if (blockIdx.x + s * gridDim.x < total) issue(s);
    }
    __syncthreads();

    int it = 0;
    for (int blk = blockIdx.x; blk < total; blk += gridDim.x, ++it) {
        const int stage = it % kQuantStages;
        const uint32_t parity = (it / kQuantStages) & 1;
        bool ok = mbar_wait(smem_u32(&full[stage]), parity, &abort_flag, p.timeout_ns);
        if (!__syncthreads_and(ok)) {
            if (threadIdx.x == 0) {
                abort_flag = 1;
                atomicExch(p.status, kStatusTimeout);
            }
            break;
        }
        const uint8_t* st = smem + stage * stage_bytes;
        // block amax over all threads (every thread passes its own partial)
        auto block_amax = [&](float amax) {
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, s));
            if (lane == 0) warp_max[warp] = amax;
            __syncthreads();
            amax = warp_max[0];
#pragma unroll
            for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
            return amax;
        };
        float scale;
        if constexpr (DR == 0) {
            const int nchunk = block_rows(blk) * p.d / 8;  // 16-byte chunks of 8 bf16
            // amax on packed bf16 pairs: |x| is x with the sign bit cleared, and the
            // maximum of bf16 values is exact (NaN ignored, as by fmaxf)
            uint32_t mag2 = 0;
            for (int g = threadIdx.x; g < nchunk; g += kThreads) {
                const uint4 v = *reinterpret_cast<const uint4*>(st + g * 16);
                mag2 = max_bf16x2(mag2, max_bf16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu));
                mag2 = max_bf16x2(mag2, max_bf16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
            }
            const float amax = block_amax(fmaxf(bf16_lo(mag2), bf16_hi(mag2)));
            scale = (amax > 0.0f) ? __fdiv_rn(amax, FMT == 1 ? 57344.0f : 448.0f) : 1.0f;
            if (FMT == 2 && amax > 0.0f) scale = pow2_at_least(scale);
            const float y = __frcp_rn(scale);
            const float2 y2 = make_float2(y, y), sn2 = make_float2(-scale, -scale);
            auto pack2 = [](float2 t) -> uint32_t {
                return FMT == 1 ? pack_e5m2x2(t.x, t.y) : pack_e4m3x2(t.x, t.y);
            };

            uint2* dst = reinterpret_cast<uint2*>(p.x8 + block_base(blk));
            for (int g = threadIdx.x; g < nchunk; g += kThreads) {
                const uint4 v = *reinterpret_cast<const uint4*>(st + g * 16);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t out[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float2 a = div2_by_scale(make_float2(bf16_lo(w[2 * e]), bf16_hi(w[2 * e])), sn2, y2);
                    const float2 b = div2_by_scale(make_float2(bf16_lo(w[2 * e + 1]), bf16_hi(w[2 * e + 1])),
                                                   sn2, y2);
                    out[e] = pack2(a) | (pack2(b) << 16);
                }
                __stcs(dst + g, make_uint2(out[0], out[1]));
            }
        } else {
            static_assert(DR == 64 || DR == 128 || DR == 256, "rotated head dim");
            constexpr int TPR = QuantShape<DR>::TPR;  // threads per row
            if constexpr (TPR == 1) {
                // One thread per row.  Register block b (8 elements) holds the row's 16-byte
                // chunk b ^ z, z = r & 7: the eight rows of a quarter-warp then read eight
                // different 16-byte slots of their 128-byte lines (rows 2 * DR bytes apart would
                // otherwise hit the same banks).  The butterflies over chunk bits 0-2 (h = 8, 16,
                // 32) pair register blocks b and b ^ 2^k whose chunks are swapped where bit k of
                // z is set; there x' = fma(x, -1, y) = a - b and y' = fma(y, 1, x) = a + b land
                // in the right chunks, each rounded once as in the sweep (sign sg = -1 for a
                // swapped pair, +1 otherwise: x' = fma(x, sg, y), y' = fma(y, -sg, x)).
                constexpr int NCH = DR / 8;               // chunks per row
                const int r = threadIdx.x, z = r & 7;
                const bool live = r < block_rows(blk);
                float v[DR];
#pragma unroll
                for (int b = 0; b < NCH; ++b) {
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (live) w = *reinterpret_cast<const uint4*>(st + ((size_t)r * DR + 8 * (b ^ z)) * 2);
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[8 * b + 2 * e] = bf16_lo(ww[e]);
                        v[8 * b + 2 * e + 1] = bf16_hi(ww[e]);
                    }
                }
                // h = 1: neighbours inside a pair of registers
#pragma unroll
                for (int e = 0; e < DR; e += 2) {
                    const float a = v[e], bb = v[e + 1];
                    v[e] = __fadd_rn(a, bb);
                    v[e + 1] = __fsub_rn(a, bb);
                }
                // h = 2, 4: inside each chunk
#pragma unroll
                for (int h = 2; h < 8; h <<= 1)
#pragma unroll
                    for (int b = 0; b < NCH; ++b)
#pragma unroll
                        for (int j = 0; j < 8; j += 2)
                            if (!(j & h)) butterfly2(v[8 * b + j], v[8 * b + j + 1], v[8 * b + j + h], v[8 * b + j + h + 1]);
                // h = 8, 16, 32: chunk bits 0-2, swapped per row by z
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const float sg = ((z >> k) & 1) ? -1.0f : 1.0f;
                    const float2 sg2 = make_float2(sg, sg), nsg2 = make_float2(-sg, -sg);
#pragma unroll
                    for (int b = 0; b < NCH; ++b) {
                        if (b & (1 << k)) continue;
                        const int b2 = b | (1 << k);
#pragma unroll
                        for (int j = 0; j < 8; j += 2) {
                            const float2 x = make_float2(v[8 * b + j], v[8 * b + j + 1]);
                            const float2 y = make_float2(v[8 * b2 + j], v[8 * b2 + j + 1]);
                            const float2 xn = __ffma2_rn(x, sg2, y);
                            const float2 yn = __ffma2_rn(y, nsg2, x);
                            v[8 * b + j] = xn.x; v[8 * b + j + 1] = xn.y;
                            v[8 * b2 + j] = yn.x; v[8 * b2 + j + 1] = yn.y;
                        }
                    }
                }
                // chunk bits from 3 up (none at d = 64), not swapped
#pragma unroll
                for (int hm = 8; hm < NCH; hm <<= 1)
#pragma unroll
                    for (int b = 0; b < NCH; ++b)
                        if (!(b & hm))
#pragma unroll
                            for (int j = 0; j < 8; j += 2)
                                butterfly2(v[8 * b + j], v[8 * b + j + 1], v[8 * (b + hm) + j], v[8 * (b + hm) + j + 1]);
                float amax = 0.0f;
                const float2 c2 = make_float2(p.rot_c, p.rot_c);
#pragma unroll
                for (int e = 0; e < DR; e += 2) {
                    const float2 t = __fmul2_rn(make_float2(v[e], v[e + 1]), c2);
                    v[e] = t.x;
                    v[e + 1] = t.y;
                    amax = fmax3(amax, fabsf(t.x), fabsf(t.y));
                }
                amax = block_amax(amax);
                scale = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
                const float y = __frcp_rn(scale);
                const float2 y2 = make_float2(y, y), sn2 = make_float2(-scale, -scale);
                if (live) {
                    uint8_t* row8 = p.x8 + block_base(blk) + (size_t)r * DR;
#pragma unroll
                    for (int b = 0; b < NCH; ++b) {
                        uint32_t out[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float* u = v + 8 * b + 4 * e;
                            const float2 a = div2_by_scale(make_float2(u[0], u[1]), sn2, y2);
                            const float2 bq = div2_by_scale(make_float2(u[2], u[3]), sn2, y2);
                            out[e] = (uint32_t)pack_e4m3x2(a.x, a.y) | ((uint32_t)pack_e4m3x2(bq.x, bq.y) << 16);
                        }
                        __stcs(reinterpret_cast<uint2*>(row8 + 8 * (b ^ z)), make_uint2(out[0], out[1]));
                    }
                }
            } else {
                constexpr int E = DR / TPR;               // elements per thread
                constexpr int NCH = E / 8;                // 16-byte chunks per thread
                const int r = threadIdx.x / TPR, q = threadIdx.x % TPR;
                const bool live = r < block_rows(blk);
                // v[8 m + j] holds element 8 (TPR (m ^ zr) + q) + j of row r: the 8 / TPR rows of a
                // quarter-warp take their chunk groups in orders XORed by zr = r mod (8 / TPR), so
                // they read different slots of their lines instead of the same banks
                constexpr int ZB = (TPR == 4) ? 1 : 2;    // group bits swapped per row
                const int zr = r & ((1 << ZB) - 1);
                float v[E];
#pragma unroll
                for (int m = 0; m < NCH; ++m) {
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (live)
                        w = *reinterpret_cast<const uint4*>(st + ((size_t)r * DR + 8 * (TPR * (m ^ zr) + q)) * 2);
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[8 * m + 2 * e] = bf16_lo(ww[e]);
                        v[8 * m + 2 * e + 1] = bf16_hi(ww[e]);
                    }
                }
                // h = 1: neighbours inside a pair of registers
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    const float a = v[e], b = v[e + 1];
                    v[e] = __fadd_rn(a, b);
                    v[e + 1] = __fsub_rn(a, b);
                }
                // h = 2, 4: inside each chunk, two butterflies per packed instruction
#pragma unroll
                for (int h = 2; h < 8; h <<= 1)
#pragma unroll
                    for (int m = 0; m < NCH; ++m)
#pragma unroll
                        for (int j = 0; j < 8; j += 2)
                            if (!(j & h)) butterfly2(v[8 * m + j], v[8 * m + j + 1], v[8 * m + j + h], v[8 * m + j + h + 1]);
                // h = 8, 16, ..., 4 TPR: across the row's lanes; the lower lane keeps v + o
                // and the upper one o - v, both as fma(v, +-1, o)
#pragma unroll
                for (int lb = 0; (1 << lb) < TPR; ++lb) {
                    const float sg = ((q >> lb) & 1) ? -1.0f : 1.0f;
                    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
                    for (int e = 0; e < E; e += 2) {
                        const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, v[e], 1 << lb),
                                                     __shfl_xor_sync(0xffffffffu, v[e + 1], 1 << lb));
                        const float2 t = __ffma2_rn(make_float2(v[e], v[e + 1]), sg2, o);
                        v[e] = t.x;
                        v[e + 1] = t.y;
                    }
                }
                // h = 8 TPR, ...: chunk-group bits below ZB, swapped in rows with that bit of zr
                // set: there the pair's registers hold (b, a), and x' = fma(x, -1, y) = a - b,
                // y' = fma(y, 1, x) = a + b land in the right groups, each rounded once as in the sweep
#pragma unroll
                for (int k = 0; k < ZB; ++k) {
                    const int hm = 1 << k;
                    const float sg = ((zr >> k) & 1) ? -1.0f : 1.0f;
                    const float2 sg2 = make_float2(sg, sg), nsg2 = make_float2(-sg, -sg);
#pragma unroll
                    for (int m = 0; m < NCH; ++m) {
                        if (m & hm) continue;
#pragma unroll
                        for (int j = 0; j < 8; j += 2) {
                            const float2 x = make_float2(v[8 * m + j], v[8 * m + j + 1]);
                            const float2 y = make_float2(v[8 * (m + hm) + j], v[8 * (m + hm) + j + 1]);
                            const float2 xn = __ffma2_rn(x, sg2, y);
                            const float2 yn = __ffma2_rn(y, nsg2, x);
                            v[8 * m + j] = xn.x; v[8 * m + j + 1] = xn.y;
                            v[8 * (m + hm) + j] = yn.x; v[8 * (m + hm) + j + 1] = yn.y;
                        }
                    }
                }
                // the other chunk-group bits, not swapped
#pragma unroll
                for (int hm = 1 << ZB; hm < NCH; hm <<= 1)
#pragma unroll
                    for (int m = 0; m < NCH; ++m)
                        if (!(m & hm))
#pragma unroll
                            for (int j = 0; j < 8; j += 2)
                                butterfly2(v[8 * m + j], v[8 * m + j + 1], v[8 * (m + hm) + j], v[8 * (m + hm) + j + 1]);
                float amax = 0.0f;
                const float2 c2 = make_float2(p.rot_c, p.rot_c);
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    const float2 t = __fmul2_rn(make_float2(v[e], v[e + 1]), c2);
                    v[e] = t.x;
                    v[e + 1] = t.y;
                    amax = fmax3(amax, fabsf(t.x), fabsf(t.y));
                }
                amax = block_amax(amax);
                scale = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
                const float y = __frcp_rn(scale);
                const float2 y2 = make_float2(y, y), sn2 = make_float2(-scale, -scale);
                if (live) {
                    uint8_t* row8 = p.x8 + block_base(blk) + (size_t)r * DR + 8 * q;  // chunk TPR m + q
#pragma unroll
                    for (int m = 0; m < NCH; ++m) {
                        uint32_t out[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float* u = v + 8 * m + 4 * e;
                            const float2 a = div2_by_scale(make_float2(u[0], u[1]), sn2, y2);
                            const float2 b = div2_by_scale(make_float2(u[2], u[3]), sn2, y2);
                            out[e] = (uint32_t)pack_e4m3x2(a.x, a.y) | ((uint32_t)pack_e4m3x2(b.x, b.y) << 16);
                        }
                        __stcs(reinterpret_cast<uint2*>(row8 + 8 * TPR * (m ^ zr)), make_uint2(out[0], out[1]));
                    }
                }
            }
        }
        if (threadIdx.x == 0) p.scales[blk] = scale;
        // every thread is done with this stage (and with warp_max) before it is refilled
        __syncthreads();
        if (threadIdx.x == 0) {
            if (blk + kQuantStages * gridDim.x < total) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(it + kQuantStages);
            }
        }
    }
    // Let every copy this CTA issued land before its shared memory is released (copies
    // end on their own: the fixed cleanup bound, not the per-wait limit).
    if (threadIdx.x == 0 && abort_flag) {
        for (int k = 0; k < kQuantStages; ++k) {
            const int j = it + k;  // loads issued for iterations it .. it+stages-1
            const int blk = blockIdx.x + j * gridDim.x;
            if (blk < total && j + 1 != p.withhold)
                mbar_wait(smem_u32(&full[j % kQuantStages]), (j / kQuantStages) & 1, nullptr,
                          kCleanupTimeoutNs);
        }
    }
}

template <int DR, int FMT = 0>
static cudaError_t launch_quant(const QuantParams& p, int sm_count, cudaStream_t stream)
{
    const int total = p.BH * p.nblk;
    const int smem = quant_smem_bytes(p.d);
    auto kernel = quant_fp8_kernel<DR, FMT>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 1;  // CTAs that fit on one SM (two at d = 128, four at d = 64)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, QuantShape<DR>::kThreads,
                                                      smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const long long want = (long long)sm_count * per_sm;
    const int grid = total < want ? total : (int)want;
    kernel<<<grid, QuantShape<DR>::kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

// Diagnostic: the FP8 conversion the quantiser uses (pack_e4m3x2 / pack_e5m2x2), applied to
// the fp32 bit patterns first .. first + count - 1 (count a multiple of 8): codes[i] is the
// code of the float whose bits are first + i.  Lets a test compare the device conversion
// with an independent encoder over every fp32 pattern.
template <int FMT>
__global__ void __launch_bounds__(256) fp8_convert_kernel(uint32_t first, size_t count8, uint2* codes)
{
    for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < count8;
         g += (size_t)gridDim.x * blockDim.x) {
        const uint32_t b0 = first + (uint32_t)(8 * g);
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float f[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) f[k] = __uint_as_float(b0 + 4 * h + k);
            const uint32_t lo = FMT == 1 ? pack_e5m2x2(f[0], f[1]) : pack_e4m3x2(f[0], f[1]);
            const uint32_t hi = FMT == 1 ? pack_e5m2x2(f[2], f[3]) : pack_e4m3x2(f[2], f[3]);
            w[h] = lo | (hi << 16);
        }
        codes[g] = make_uint2(w[0], w[1]);
    }
}

cudaError_t launch_fp8_convert(uint32_t first, size_t count, int fmt, void* codes, int sm_count,
                               cudaStream_t stream)
{
    const size_t count8 = count / 8;
    size_t blocks = (count8 + 255) / 256;
    const size_t cap = (size_t)sm_count * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (fmt == 1)
        fp8_convert_kernel<1><<<(unsigned)blocks, 256, 0, stream>>>(first, count8, static_cast<uint2*>(codes));
    else
        fp8_convert_kernel<0><<<(unsigned)blocks, 256, 0, stream>>>(first, count8, static_cast<uint2*>(codes));
    return cudaGetLastError();
}

cudaError_t launch_quant_fp8(const QuantParams& p, int sm_count, cudaStream_t stream)
{
    if (!p.rotate) {
        if (p.fmt == 1) return launch_quant<0, 1>(p, sm_count, stream);
        if (p.fmt == 2) return launch_quant<0, 2>(p, sm_count, stream);
        return launch_quant<0, 0>(p, sm_count, stream);
    }
    if (p.fmt) return cudaErrorInvalidValue;    // the rotated variant writes E4M3 only
    switch (p.d) {
    case 64: return launch_quant<64>(p, sm_count, stream);
    case 128: return launch_quant<128>(p, sm_count, stream);
    case 256: return launch_quant<256>(p, sm_count, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300
