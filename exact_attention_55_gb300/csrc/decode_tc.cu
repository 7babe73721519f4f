// decode_tc.cu -- a decoding step over a paged KV cache on the tensor cores, for 2 to 8
// new tokens per sequence (speculative or multi-token decoding) at head dims 64 and 128.
//
// "大模型加速-核心网络算子-Flash Attention V3" §3 总结: tokens are produced one at a time
// over a cache of earlier keys and values; "Warp Group Cluster 优化：Flash Attention V3 在
// H100 上的 FP8 融合计算实践", 局限性与后续方向 item 2: PagedAttention KV-cache
// management.  Same result as decode.cu's CUDA-core kernel (query i of sequence b sits at
// position L_b - nq + i and sees keys 0 .. L_b - nq + i), computed as a small forward pass:
//
//   * a persistent CTA per SM walks units (head, split of the sequence's keys);
//   * warp 1 (one lane) loads the unit's nq query rows with TMA into a 128-row tile whose
//     other rows stay zero, then streams K and V tiles of 128 keys through a ring of
//     shared-memory slots, one TMA box per page (or per 128 keys of a larger page);
//   * warp 2 issues tcgen05.mma: S = Q K^T (M 128, N 128, K d) into one of two TMEM
//     buffers, and O += P V with P read back from TMEM;
//   * warp 0 owns TMEM lanes 0-31, i.e. query rows 0-31: it reads S, masks, keeps the
//     running max and sum (lazy rescale, threshold 2^8 as the forward's bf16 path), writes
//     P as bf16 over S, and at the end of a unit writes O / l and the log-sum-exp (or the
//     split's partials for decode_combine_kernel).
//
// The tensor core does 128-row work for nq rows, but a decoding step is HBM-bound: a
// 128-key tile is 32 KB of K and V (d = 128) per 1 M FLOP of useful work, so the padded
// MMAs (8.4 M FLOP per tile) and the one softmax warp still finish well inside the time
// HBM needs to deliver the tile.  Keys past the sequence end inside the last tile come
// from whatever pages the (clamped) table names there: their scores are masked, and
// their V rows are zeroed in shared memory before P V so that a non-finite value in an
// unused page can never reach O through 0 * NaN.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_params.h"
#include "ptx.cuh"

namespace gb300 {

cudaError_t launch_decode_combine(const DecodeParams& p, int d, cudaStream_t stream);

template <int D>
struct DecTcCfg {
    static constexpr int BM = 128;                        // query rows of the MMA (nq used)
    static constexpr int BN = 128;                        // keys per tile
    static constexpr int NCB = D / 64;                    // 128-byte column blocks of a row
    static constexpr int CB_BYTES = 128 * 128;            // one column block of a 128-row tile
    static constexpr int Q_BYTES = NCB * CB_BYTES;
    static constexpr int KV_BYTES = NCB * CB_BYTES;
    static constexpr int SMEM_CAP = 227 * 1024;
    static constexpr int BAR_BYTES = 1024;
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int NSLOT_FIT = (SMEM_CAP - BAR_BYTES - ALIGN_SLACK - Q_BYTES) / KV_BYTES;
    static constexpr int NSLOT = NSLOT_FIT < 8 ? NSLOT_FIT : 8;
    static constexpr int SMEM_BYTES = ALIGN_SLACK + Q_BYTES + NSLOT * KV_BYTES + BAR_BYTES;
    static constexpr int O_COL = 2 * BN;                  // S buffers at 0 and BN, O after
    static constexpr int TMEM_COLS = 512;
    static constexpr int NUM_THREADS = 128;               // softmax, producer, MMA, spare
    static constexpr float TAU = 8.0f;                    // lazy-rescale threshold (log2)
    static_assert(D == 64 || D == 128, "tensor-core decoding: head dim 64 or 128");
    static_assert(O_COL + D <= TMEM_COLS, "TMEM");
    static_assert(NSLOT >= 4, "ring");
    static_assert(SMEM_BYTES <= SMEM_CAP, "shared memory");
};

struct alignas(8) DecTcBars {
    uint64_t q_full, q_empty;
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2], p_full[2];
    uint64_t pv_done, o_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Unit u = (head bh, split): keys [k0, k1) of sequence b; n tiles of 128 keys (0 when the
// split starts past the sequence end).
struct DecTcUnit {
    int bh, b, h, split;
    int L;        // cached length (clamped)
    int k0, k1;   // this split's keys
    int n;        // tiles
};

__device__ __forceinline__ void dec_tc_unit(const DecodeParams& p, int u, DecTcUnit& w)
{
    w.bh = u / p.splits;
    w.split = u - w.bh * p.splits;
    w.b = w.bh / p.H;
    w.h = w.bh - w.b * p.H;
    const int cap = p.max_pages << p.log2_ps;
    w.L = min(max(__ldg(p.seq_lens + w.b), 0), cap);
    const int kps = p.pages_per_split << p.log2_ps;   // a multiple of 128
    w.k0 = w.split * kps;
    w.k1 = min(w.L, w.k0 + kps);
    w.n = w.k1 > w.k0 ? (w.k1 - w.k0 + 127) / 128 : 0;
}

__device__ __forceinline__ void dec_tc_timeout(const DecodeParams& p, DecTcBars* bars)
{
    atomicExch(p.status, kStatusTimeout);
    *reinterpret_cast<volatile int*>(&bars->abort_flag) = 1;
}

template <int D>
__global__ void __launch_bounds__(DecTcCfg<D>::NUM_THREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const DecodeParams p)
{
    using C = DecTcCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* q_smem = smem;
    uint8_t* kv_smem = smem + C::Q_BYTES;
    DecTcBars* bars = reinterpret_cast<DecTcBars*>(kv_smem + C::NSLOT * C::KV_BYTES);
    const volatile int* abort_flag = &bars->abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = p.B * p.H * p.splits;
    const int R = p.log2_ps < 7 ? (1 << p.log2_ps) : 128;   // rows per TMA box (a page, or 128)

    // Q rows nq .. 127 stay zero for the whole kernel (the unit's TMA writes rows 0 .. nq-1)
    for (int i = threadIdx.x; i < C::Q_BYTES / 16; i += C::NUM_THREADS)
        reinterpret_cast<uint4*>(q_smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->q_full), 1);
        mbar_init(smem_u32(&bars->q_empty), 1);
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(smem_u32(&bars->kv_full[s]), 1);
            mbar_init(smem_u32(&bars->kv_empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars->s_full[i]), 1);
            mbar_init(smem_u32(&bars->p_full[i]), 1);
        }
        mbar_init(smem_u32(&bars->pv_done), 1);
        mbar_init(smem_u32(&bars->o_empty), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(&bars->tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 1) {
        // ------------------------------------------------------------ TMA producer
        // The whole warp walks the tiles; lane 0 waits for free slots and arms the barriers,
        // then lane i issues box i of the tile (its page number loaded by that lane), so the
        // up to 16 boxes of a tile of small pages go out together.
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        const uint64_t pol = l2_policy_evict_first();
        uint32_t ring = 0, uc = 0, q_armed = 0;
        bool ok = true;
        const int nbox = 128 / R;                                   // 1 .. 16 boxes per tile
        auto wait_lane0 = [&](uint64_t* bar, uint32_t parity) -> bool {
            int r = 1;
            if (lane == 0) r = mbar_wait(smem_u32(bar), parity, abort_flag, p.timeout_ns) ? 1 : 0;
            r = __shfl_sync(0xffffffffu, r, 0);
            if (!r) ok = false;
            return r != 0;
        };
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            DecTcUnit w;
            dec_tc_unit(p, u, w);
            if (w.n == 0) continue;
            if (!wait_lane0(&bars->q_empty, (uc & 1) ^ 1)) break;
            if (lane == 0) {
                const uint32_t qb = smem_u32(&bars->q_full);
                mbar_arrive_expect_tx(qb, (uint32_t)(p.nq * 128 * C::NCB));
#pragma unroll
                for (int cb = 0; cb < C::NCB; ++cb)
                    tma_load_3d(smem_u32(q_smem + cb * C::CB_BYTES), &tmQ, qb, cb * 64, 0, w.bh, pol);
            }
            ++q_armed;
            const int* ptab = p.page_table + (size_t)w.b * p.max_pages;
            for (int jj = 0; jj < w.n && ok; ++jj) {
                const int t = w.k0 + jj * 128 + lane * R;               // first key of lane's box
                int pg = 0, r0 = 0;
                if (lane < nbox) {
                    const int pi = min(t >> p.log2_ps, p.max_pages - 1);
                    pg = min(max(__ldg(ptab + pi), 0), p.num_pages - 1);
                    r0 = t & ((1 << p.log2_ps) - 1);                    // 0 unless a page holds 128+
                }
#pragma unroll
                for (int which = 0; which < 2; ++which) {   // K then V
                    const uint32_t slot = ring % C::NSLOT;
                    if (!wait_lane0(&bars->kv_empty[slot], ((ring / C::NSLOT) & 1) ^ 1)) break;
                    const uint32_t fb = smem_u32(&bars->kv_full[slot]);
                    if (lane == 0) mbar_arrive_expect_tx(fb, C::KV_BYTES);
                    __syncwarp();
                    if (lane < nbox) {
                        const uint32_t dst = smem_u32(kv_smem + slot * C::KV_BYTES) + lane * R * 128;
                        const CUtensorMap* map = which == 0 ? &tmK : &tmV;
#pragma unroll
                        for (int cb = 0; cb < C::NCB; ++cb)
                            tma_load_3d(dst + cb * C::CB_BYTES, map, fb, cb * 64, r0, pg * p.H + w.h, pol);
                    }
                    ++ring;
                }
            }
            ++uc;
        }
        if (!ok && lane == 0) dec_tc_timeout(p, bars);
        // every copy issued lands before shared memory is released
        if (lane == 0) {
            const uint32_t armed = ring < C::NSLOT ? ring : C::NSLOT;
            for (uint32_t k = ring - armed; k < ring; ++k)
                mbar_wait(smem_u32(&bars->kv_full[k % C::NSLOT]), (k / C::NSLOT) & 1, nullptr,
                          kCleanupTimeoutNs);
            if (q_armed > 0)
                mbar_wait(smem_u32(&bars->q_full), (q_armed - 1) & 1, nullptr, kCleanupTimeoutNs);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc_s = idesc_f32acc(1, 0, C::BM, C::BN);   // bf16, K-major B
        constexpr uint32_t idesc_o = idesc_f32acc(1, 1, C::BM, D);       // V MN-major
        const uint64_t q_desc = sdesc_sw128(smem_u32(q_smem), 16, 1024);
        const uint64_t kv_desc0 = sdesc_sw128(smem_u32(kv_smem), 16, 1024);
        const uint64_t v_desc0 = sdesc_sw128(smem_u32(kv_smem), C::CB_BYTES, 1024);
        uint32_t ring = 0, uc = 0, p_phase = 0;
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool r = ok && mbar_wait(smem_u32(bar), parity, abort_flag, p.timeout_ns);
            r = __all_sync(0xffffffffu, r);
            if (!r) ok = false;
            return r;
        };
        auto commit = [&](uint64_t* bar) { mma_commit_warp(smem_u32(bar)); };
        auto issue_s = [&](int sb, uint32_t slot) {
            const uint64_t kb = kv_desc0 + (uint64_t)((slot * C::KV_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (((kk * 32) / 128) * C::CB_BYTES + (kk * 32) % 128) >> 4;
                mma_ss_warp<false>(tmem + sb * C::BN, q_desc + off, kb + off, idesc_s, kk > 0 ? 1u : 0u);
            }
        };
        auto issue_pv = [&](int sb, uint32_t slot, bool acc) {
            const uint64_t vb = v_desc0 + (uint64_t)((slot * C::KV_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < C::BN / 16; ++kk)
                mma_ts_warp<false>(tmem + C::O_COL, tmem + sb * C::BN + kk * 8, vb + ((kk * 16 * 128) >> 4),
                                   idesc_o, (kk > 0 || acc) ? 1u : 0u);
        };
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            DecTcUnit w;
            dec_tc_unit(p, u, w);
            if (w.n == 0) continue;
            if (!wait(&bars->q_full, uc & 1)) break;
            tc_fence_after_sync();
            for (int jj = 0; jj <= w.n && ok; ++jj) {
                if (jj < w.n) {   // S(jj) = Q K(jj)^T
                    const uint32_t rk = ring + 2 * jj;
                    if (!wait(&bars->kv_full[rk % C::NSLOT], (rk / C::NSLOT) & 1)) break;
                    issue_s(jj & 1, rk % C::NSLOT);
                    commit(&bars->s_full[jj & 1]);
                    if (jj == w.n - 1) commit(&bars->q_empty);
                }
                if (jj > 0) {     // O (+)= P(jj-1) V(jj-1)
                    const uint32_t rv = ring + 2 * (jj - 1) + 1;
                    const int sp = (jj - 1) & 1;
                    if (!wait(&bars->kv_full[rv % C::NSLOT], (rv / C::NSLOT) & 1)) break;
                    if (!wait(&bars->p_full[sp], (p_phase >> sp) & 1)) break;
                    p_phase ^= 1u << sp;
                    if (jj == 1 && !wait(&bars->o_empty, (uc & 1) ^ 1)) break;
                    tc_fence_after_sync();
                    issue_pv(sp, rv % C::NSLOT, jj > 1);
                    commit(&bars->pv_done);
                    commit(&bars->kv_empty[rv % C::NSLOT]);
                    commit(&bars->kv_empty[(rv - 1) % C::NSLOT]);   // K(jj-1)
                }
            }
            if (!ok) break;
            ring += 2 * w.n;
            ++uc;
        }
        if (!ok && lane == 0) dec_tc_timeout(p, bars);
        commit(&bars->drain);
        mbar_wait(smem_u32(&bars->drain), 0, nullptr, kCleanupTimeoutNs);
        __syncwarp();
    } else if (warp == 0) {
        // ------------------------------------------------------------ softmax (rows 0-31)
        const int r = lane;                       // query row of this thread
        const float NEG_INF = -__int_as_float(0x7f800000);
        uint32_t s_phase = 0, pv_phase = 0, uc = 0, ring = 0;
        bool ok = true;
        auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool res = ok && mbar_wait(smem_u32(bar), parity, abort_flag, p.timeout_ns);
            res = __all_sync(0xffffffffu, res);
            if (!res) ok = false;
            return res;
        };
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            DecTcUnit w;
            dec_tc_unit(p, u, w);
            const int last = w.L - p.nq + r;      // this row's last allowed key
            float m_used = NEG_INF, l = 0.0f;
            for (int jj = 0; jj < w.n; ++jj) {
                const int sb = jj & 1;
                const int t0 = w.k0 + jj * 128;
                if (!wait_all(&bars->s_full[sb], (s_phase >> sb) & 1)) break;
                s_phase ^= 1u << sb;
                tc_fence_after_sync();
                uint32_t sr[128];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) tmem_ld32p(tmem + sb * C::BN + ch * 32, sr + ch * 32);
                tmem_wait_ld_only();
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) reg_fence32(sr + ch * 32);
                float* s = reinterpret_cast<float*>(sr);
                // keys t0 + e allowed for this row: t < k1 (the split) and t <= last
                const int lim = r < p.nq ? min(w.k1 - 1, last) - t0 : -1;   // allowed e <= lim
                if (lim < 127) {
#pragma unroll
                    for (int e = 0; e < 128; ++e)
                        if (e > lim) s[e] = NEG_INF;
                }
                float mx[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float m = s[k];
#pragma unroll
                    for (int u2 = 1; u2 + 1 < 16; u2 += 2) m = fmax3(m, s[k + 8 * u2], s[k + 8 * u2 + 8]);
                    mx[k] = fmaxf(m, s[k + 8 * 15]);
                }
                const float tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                         fmaxf(mx[6], mx[7]));
                const float m_cand = tmax * p.c_log2;
                const bool resc = m_cand > m_used + C::TAU;
                const float alpha = resc ? ex2(m_used - m_cand) : 1.0f;   // ex2(-inf) = 0
                if (resc) {
                    l *= alpha;
                    m_used = m_cand;
                }
                const float mb = (m_used == NEG_INF) ? 0.0f : m_used;
                const float2 c2 = make_float2(p.c_log2, p.c_log2), b2 = make_float2(-mb, -mb);
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int i0 = ch * 64 + 2 * e;
                        const float2 x = __ffma2_rn(make_float2(s[i0], s[i0 + 1]), c2, b2);
                        const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                        acc = __fadd2_rn(acc, pp);
                        pk[e] = pack_bf16x2(pp.x, pp.y);
                    }
                    tmem_st32p(tmem + sb * C::BN + ch * 32, pk);
                }
                l += acc.x + acc.y;
                // V rows of keys past the sequence end (last tile only) are zeroed, so that
                // whatever the table's unused pages hold cannot reach O
                const uint32_t rv = ring + 2 * jj + 1;
                if (t0 + 128 > w.L) {
                    if (!wait_all(&bars->kv_full[rv % C::NSLOT], (rv / C::NSLOT) & 1)) break;
                    uint8_t* vt = kv_smem + (rv % C::NSLOT) * C::KV_BYTES;
                    const int first = max(w.L - t0, 0);
                    for (int e = first + lane; e < 128; e += 32)
#pragma unroll
                        for (int cb = 0; cb < C::NCB; ++cb)
#pragma unroll
                            for (int q4 = 0; q4 < 8; ++q4)
                                reinterpret_cast<uint4*>(vt + cb * C::CB_BYTES + e * 128)[q4] =
                                    make_uint4(0u, 0u, 0u, 0u);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                if (jj > 0) {
                    // O holds P(jj-1) V once that MMA is done; rescale it if a row's max moved
                    if (!wait_all(&bars->pv_done, pv_phase & 1)) break;
                    ++pv_phase;
                    if (__any_sync(0xffffffffu, resc)) {
                        tc_fence_after_sync();
                        const float2 f2 = make_float2(alpha, alpha);
#pragma unroll
                        for (int ch = 0; ch < D / 32; ++ch) {
                            uint32_t o[32];
                            tmem_ld32(tmem + C::O_COL + ch * 32, o);
                            tmem_wait_ld(o);
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float2 v2 = __fmul2_rn(
                                    make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), f2);
                                o[2 * e] = __float_as_uint(v2.x);
                                o[2 * e + 1] = __float_as_uint(v2.y);
                            }
                            tmem_st32p(tmem + C::O_COL + ch * 32, o);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[sb]));
            }
            if (!ok) break;
            // epilogue: O / l and the log2-sum-exp of this row over the split's keys
            float inv_l = 0.0f;
            if (w.n > 0) {
                if (!wait_all(&bars->pv_done, pv_phase & 1)) break;
                ++pv_phase;
                tc_fence_after_sync();
                inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
            }
            const float lse2 = (l > 0.0f) ? m_used + __log2f(l) : NEG_INF;
            const size_t qi = (size_t)w.bh * p.nq + r;
            float* wrow = p.splits > 1 ? p.ws + (((size_t)w.bh * p.splits + w.split) * p.nq + r) * (D + 1)
                                       : nullptr;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t o[32];
                if (w.n > 0) {
                    tmem_ld32(tmem + C::O_COL + ch * 32, o);
                    tmem_wait_ld(o);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                if (r < p.nq) {
                    if (wrow != nullptr) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) wrow[ch * 32 + e] = __uint_as_float(o[e]) * inv_l;
                    } else {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l,
                                                __uint_as_float(o[2 * e + 1]) * inv_l);
                        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                                              qi * D + ch * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                    }
                }
            }
            if (r < p.nq) {
                if (wrow != nullptr) wrow[D] = lse2;
                else p.lse[qi] = lse2 * 0.69314718055994531f;
            }
            if (w.n > 0) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->o_empty));
                ring += 2 * w.n;
                ++uc;
            }
        }
        if (!ok) dec_tc_timeout(p, bars);
        tmem_wait_st();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 2) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D>
static cudaError_t launch_decode_tc_d(const CUtensorMap& mq, const CUtensorMap& mk,
                                      const CUtensorMap& mv, const DecodeParams& p, int sm_count,
                                      cudaStream_t stream)
{
    using C = DecTcCfg<D>;
    auto kernel = decode_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long units = (long long)p.B * p.H * p.splits;
    const int grid = units < sm_count ? (int)units : sm_count;
    kernel<<<grid, C::NUM_THREADS, C::SMEM_BYTES, stream>>>(mq, mk, mv, p);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.splits == 1) return e;
    return launch_decode_combine(p, D, stream);
}

cudaError_t launch_decode_tc(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                             const DecodeParams& p, int d, int sm_count, cudaStream_t stream)
{
    switch (d) {
    case 64: return launch_decode_tc_d<64>(mq, mk, mv, p, sm_count, stream);
    case 128: return launch_decode_tc_d<128>(mq, mk, mv, p, sm_count, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300
