// decode.cu -- one decoding step of attention over a paged KV cache, split over keys.
//
// "大模型加速-核心网络算子-Flash Attention V3" §3 总结: decoding produces tokens one at
// a time and keeps the keys and values of earlier positions in a KV cache; "Warp
// Group Cluster 优化：Flash Attention V3 在 H100 上的 FP8 融合计算实践", 局限性与后续方向
// item 2: KV-cache management with PagedAttention.  For sequence b with L_b cached
// tokens (its nq newest included) and head h, query i sits at position L_b - nq + i
// and attends to keys 0 .. L_b - nq + i.  Key t is row t % page_size of page
// page_table[b][t / page_size] of a cache laid out [num_pages, H, page_size, D].
//
// HBM-bound: every cached byte is read once per step for nq/2 FLOP per byte, so the
// arithmetic runs on the CUDA cores and the design is about the loads.  Grid
// (splits, B*H); a CTA takes a contiguous range of the sequence's pages and its four
// warps take groups of G keys in turn.  Lane l holds D/32 consecutive elements of
// every row (coalesced 4-16 byte streaming loads, K and V of a group issued
// together), dot products are summed across the warp with shuffles, and each warp
// keeps an online softmax (max, sum, its O slice) per query.  The warps merge in
// shared memory; with one split the CTA writes O and LSE, otherwise (O / l, log2 of
// the sum) goes to the workspace and decode_combine_kernel merges the splits with
// weights 2^(lse_s - lse).  Page numbers and lengths are clamped to the cache, so a
// bad table gives wrong values, never an access outside the tensors.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_params.h"
#include "ptx.cuh"

namespace gb300 {

constexpr int kDecWarps = 4;
constexpr int kDecG = 8;  // keys per warp per step

template <int E>
struct RowVec;  // E consecutive bf16 of a row, one lane's share
template <> struct RowVec<2> { using T = uint32_t; };
template <> struct RowVec<4> { using T = uint2; };
template <> struct RowVec<8> { using T = uint4; };

template <int E>
__device__ __forceinline__ void unpack_bf16(const typename RowVec<E>::T& w, float* out)
{
    const uint32_t* u = reinterpret_cast<const uint32_t*>(&w);
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
        out[2 * k] = __uint_as_float(u[k] << 16);
        out[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
    }
}

template <int E>
__device__ __forceinline__ typename RowVec<E>::T load_row(const __nv_bfloat16* p)
{
    return __ldcs(reinterpret_cast<const typename RowVec<E>::T*>(p));
}

// Sum each of the NV values over the 32 lanes and give every lane every sum.  A
// reduce-scatter first (at each shuffle distance a lane keeps half of its values and
// adds the partner's copy of that half, while more than one value is left), then a
// butterfly on the last value, then one broadcast shuffle per value: NV=8 takes 17
// shuffles instead of 40, and all lanes see bit-identical sums.
template <int NV>
__device__ __forceinline__ void warp_sum_all(float* v, int lane)
{
    float cur[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) cur[j] = v[j];
    int c = NV;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        if (c > 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int j = 0; j < NV / 2; ++j) {
                if (j < c / 2) {
                    const float send = upper ? cur[j] : cur[j + c / 2];
                    const float keep = upper ? cur[j + c / 2] : cur[j];
                    cur[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            c >>= 1;
        } else {
            cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], o);
        }
    }
    // value idx now sits in slot idx % SLOTS of lane (idx / SLOTS) * (32 / GROUPS)
    constexpr int SLOTS = NV > 32 ? NV / 32 : 1;
    constexpr int GROUPS = NV / SLOTS;
#pragma unroll
    for (int idx = 0; idx < NV; ++idx)
        v[idx] = __shfl_sync(0xffffffffu, cur[idx % SLOTS], (idx / SLOTS) * (32 / GROUPS));
}

template <int D, int NQ>
__global__ void __launch_bounds__(kDecWarps * 32) decode_split_kernel(const DecodeParams p)
{
    constexpr int E = D / 32;
    using V = typename RowVec<E>::T;
    __shared__ float sm_m[kDecWarps][NQ], sm_l[kDecWarps][NQ];
    __shared__ float sm_acc[kDecWarps][NQ][D];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.H, h = bh - b * p.H;
    const int nq = p.nq;
    const int ps_mask = (1 << p.log2_ps) - 1;
    const int cap = p.max_pages << p.log2_ps;
    const int L = min(max(__ldg(p.seq_lens + b), 0), cap);
    const int k_begin = (split * p.pages_per_split) << p.log2_ps;
    const int k_end = min(L, ((split + 1) * p.pages_per_split) << p.log2_ps);
    const float NEG_INF = -__int_as_float(0x7f800000);

    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* kc = reinterpret_cast<const __nv_bfloat16*>(p.kc);
    const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(p.vc);
    const int* ptab = p.page_table + (size_t)b * p.max_pages;

    // this lane's slice of every query, pre-multiplied by scale * log2(e)
    float qv[NQ][E];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        float t[E];
        if (i < nq) {
            unpack_bf16<E>(load_row<E>(qb + (((size_t)bh * nq + i) * D + lane * E)), t);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) t[e] = 0.0f;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) qv[i][e] = t[e] * p.c_log2;
    }
    float m[NQ], l[NQ], acc[NQ][E];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        m[i] = NEG_INF;
        l[i] = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[i][e] = 0.0f;
    }

    // groups start at multiples of kDecG inside a split that starts on a page, so with
    // pages of at least kDecG keys a group never crosses a page
    const bool group_in_page = p.log2_ps >= 3;
    for (int t0 = k_begin + warp * kDecG; t0 < k_end; t0 += kDecWarps * kDecG) {
        // edge groups: the split's or the sequence's end falls inside (needs masks)
        const bool edge = (t0 + kDecG > k_end) || (t0 + kDecG - 1 > L - nq);
        V kr[kDecG], vr[kDecG];
        if (group_in_page && !edge) {
            int page = __ldg(ptab + (t0 >> p.log2_ps));
            page = min(max(page, 0), p.num_pages - 1);
            const size_t row0 = (((size_t)page * p.H + h) << p.log2_ps) + (t0 & ps_mask);
            const __nv_bfloat16* kp = kc + row0 * D + lane * E;
            const __nv_bfloat16* vp = vc + row0 * D + lane * E;
#pragma unroll
            for (int g = 0; g < kDecG; ++g) {
                kr[g] = load_row<E>(kp + g * D);
                vr[g] = load_row<E>(vp + g * D);
            }
        } else {
#pragma unroll
            for (int g = 0; g < kDecG; ++g) {
                const int t = t0 + g;
                if (t < k_end) {
                    int page = __ldg(ptab + (t >> p.log2_ps));
                    page = min(max(page, 0), p.num_pages - 1);
                    const size_t row = (((size_t)page * p.H + h) << p.log2_ps) + (t & ps_mask);
                    kr[g] = load_row<E>(kc + row * D + lane * E);
                    vr[g] = load_row<E>(vc + row * D + lane * E);
                } else {
                    kr[g] = V{};
                    vr[g] = V{};
                }
            }
        }
        // scores in log2 units: s[g][i] = c * q_i . k_t
        float s[kDecG][NQ];
#pragma unroll
        for (int g = 0; g < kDecG; ++g) {
            float kf[E];
            unpack_bf16<E>(kr[g], kf);
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                float a = 0.0f;
#pragma unroll
                for (int e = 0; e < E; ++e) a = fmaf(qv[i][e], kf[e], a);
                s[g][i] = a;
            }
        }
        warp_sum_all<kDecG * NQ>(&s[0][0], lane);
        // mask: query slots past nq, keys past this split's range, and the end-aligned
        // causal limit (the last two only in edge groups)
#pragma unroll
        for (int g = 0; g < kDecG; ++g)
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                const int t = t0 + g;
                if (i >= nq || (edge && (t >= k_end || t > L - nq + i))) s[g][i] = NEG_INF;
            }
        // online softmax: new maxima and rescaling first, then the scores become weights
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            float mx = s[0][i];
#pragma unroll
            for (int g = 1; g < kDecG; ++g) mx = fmaxf(mx, s[g][i]);
            if (mx > m[i]) {                       // never true when the group is all masked
                const float alpha = ex2(m[i] - mx);  // ex2(-inf) = 0 on the first group
                l[i] *= alpha;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[i][e] *= alpha;
                m[i] = mx;
            }
            const float mb = (m[i] == NEG_INF) ? 0.0f : m[i];
#pragma unroll
            for (int g = 0; g < kDecG; ++g) {
                s[g][i] = ex2(s[g][i] - mb);       // masked keys: ex2(-inf) = 0
                l[i] += s[g][i];
            }
        }
        // O slice += p V, one V row at a time
#pragma unroll
        for (int g = 0; g < kDecG; ++g) {
            float vf[E];
            unpack_bf16<E>(vr[g], vf);
#pragma unroll
            for (int i = 0; i < NQ; ++i)
#pragma unroll
                for (int e = 0; e < E; ++e) acc[i][e] = fmaf(s[g][i], vf[e], acc[i][e]);
        }
    }

    // merge the warps
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        if (lane == 0) {
            sm_m[warp][i] = m[i];
            sm_l[warp][i] = l[i];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) sm_acc[warp][i][lane * E + e] = acc[i][e];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < NQ * D; idx += kDecWarps * 32) {
        const int i = idx / D, e = idx - i * D;
        if (i >= nq) continue;
        float M = sm_m[0][i];
#pragma unroll
        for (int w = 1; w < kDecWarps; ++w) M = fmaxf(M, sm_m[w][i]);
        float lsum = 0.0f, o = 0.0f;
        if (M != NEG_INF) {
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) {
                const float f = ex2(sm_m[w][i] - M);
                lsum = fmaf(sm_l[w][i], f, lsum);
                o = fmaf(sm_acc[w][i][e], f, o);
            }
        }
        const float val = lsum > 0.0f ? o / lsum : 0.0f;
        const float lse2 = lsum > 0.0f ? M + __log2f(lsum) : NEG_INF;
        const size_t qi = (size_t)bh * nq + i;
        if (p.splits == 1) {
            reinterpret_cast<__nv_bfloat16*>(p.o)[qi * D + e] = __float2bfloat16_rn(val);
            if (e == 0) p.lse[qi] = lse2 * 0.69314718055994531f;
        } else {
            float* w = p.ws + (((size_t)bh * p.splits + split) * nq + i) * (D + 1);
            w[e] = val;
            if (e == 0) w[D] = lse2;
        }
    }
}

// Merge the splits of one (head, query) per warp: O = sum_s 2^(lse_s - lse) O_s / S.
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p)
{
    constexpr int E = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t qi = (size_t)blockIdx.x * 4 + warp;  // (bh, i) flattened
    if (qi >= (size_t)p.B * p.H * p.nq) return;
    const size_t bh = qi / p.nq, i = qi - bh * p.nq;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const float* base = p.ws + (bh * p.splits * p.nq + i) * (D + 1);
    const size_t sstride = (size_t)p.nq * (D + 1);
    float M = NEG_INF;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, base[s * sstride + D]);
    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.0f;
    float wsum = 0.0f;
    if (M != NEG_INF) {
        for (int s = 0; s < p.splits; ++s) {
            const float* w = base + s * sstride;
            const float f = ex2(w[D] - M);  // empty split: ex2(-inf) = 0
            wsum += f;
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = fmaf(f, w[lane * E + e], o[e]);
        }
    }
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + qi * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) orow[e] = __float2bfloat16_rn(wsum > 0.0f ? o[e] / wsum : 0.0f);
    if (lane == 0) p.lse[qi] = wsum > 0.0f ? (M + __log2f(wsum)) * 0.69314718055994531f : NEG_INF;
}

// Merge the split partials in p.ws into o and lse (also used by the tensor-core kernel).
cudaError_t launch_decode_combine(const DecodeParams& p, int d, cudaStream_t stream)
{
    const long long rows = (long long)p.B * p.H * p.nq;
    const unsigned grid = (unsigned)((rows + 3) / 4);
    switch (d) {
    case 64: decode_combine_kernel<64><<<grid, 128, 0, stream>>>(p); break;
    case 128: decode_combine_kernel<128><<<grid, 128, 0, stream>>>(p); break;
    case 256: decode_combine_kernel<256><<<grid, 128, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int D, int NQ>
static cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream)
{
    dim3 grid(p.splits, p.B * p.H);
    decode_split_kernel<D, NQ><<<grid, kDecWarps * 32, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.splits == 1) return e;
    return launch_decode_combine(p, D, stream);
}

template <int D>
static cudaError_t launch_decode_d(const DecodeParams& p, cudaStream_t stream)
{
    if (p.nq == 1) return launch_decode_t<D, 1>(p, stream);
    if (p.nq == 2) return launch_decode_t<D, 2>(p, stream);
    if (p.nq <= 4) return launch_decode_t<D, 4>(p, stream);
    return launch_decode_t<D, 8>(p, stream);
}

cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t stream)
{
    switch (d) {
    case 64: return launch_decode_d<64>(p, stream);
    case 128: return launch_decode_d<128>(p, stream);
    case 256: return launch_decode_d<256>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300
