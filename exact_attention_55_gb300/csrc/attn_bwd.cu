// attn_bwd.cu -- backward pass of the fused exact attention: dQ, dK, dV.
//
// The gradients of O = softmax(scale * Q K^T + mask) V for an upstream gradient dO,
// with P recomputed from the forward's per-row log-sum-exp (P = exp(s - LSE), already
// normalised):
//     D_i = dO_i . O_i,   dP = dO V^T,   dS = P * (dP - D),
//     dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO.
// The pages name the backward pass only in passing ("FlashAttention V3：优化框架吞吐量
// 的关键技术实践" §2.3.2: micro-batches' forward and backward passes overlapped in
// pipeline training, and its introduction: training as well as inference; "大模型加速-
// 核心网络算子-Flash Attention V3" §2.3-2.4 call the kernel they describe the forward
// pass); the formulas are the chain rule through the forward definition.
//
// Three launches, no atomics and no fp32 accumulation buffer:
//   bwd_dot_kernel          D_i, one warp per row;
//   bwd_kernel<D, true>     (dQ pass) per 128-row query tile, in steps of 128 keys:
//                           S = Q K_j^T and dP = dO V_j^T into TMEM, the compute
//                           warpgroups turn them into dS (bf16, over S), then
//                           dQ += dS K_j with K_j as the MN-major operand;
//   bwd_kernel<D, false>    (dK/dV pass) per 128-key tile, in steps of 64 queries, the
//                           transposed products: S^T = K Q_i^T and dP^T = V dO_i^T,
//                           then dV += P^T dO_i and dK += dS^T Q_i.
// S is recomputed in both passes (7 matmuls per tile pair instead of 5) to keep dQ in
// TMEM rather than in a global fp32 buffer updated by atomics.
//
// Software pipelines.  dQ pass: S(j) goes to one of two TMEM S buffers and dP(j) to one
// dP buffer that the compute warps release as soon as they have loaded it, so the MMA
// warp issues dP(j), then the accumulation of step j-1, then S(j+1), and the tensor pipe
// computes dP(j) and S(j+1) while both compute warpgroups work on steps j-1 and j (64 keys
// each).  dK/dV pass: S^T and dP^T of a 64-query step live in one of two TMEM step buffers,
// the MMA warp issues step h's products before step h-1's accumulations, and the two
// compute warpgroups ping-pong over the buffers (warpgroup b takes the steps of buffer b).
//
// Roles per CTA (persistent over units): warps 0-7 compute (two warpgroups, one thread
// per tile row), warp 8 streams tiles with TMA through an mbarrier ring, warp 9 issues
// the tcgen05.mma, warps 10-11 only complete the control warpgroup (registers move from
// it to the compute warpgroups).  Every wait is bounded and gives up with
// ATTN_ERR_TIMEOUT.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "attn_params.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace gb300 {

template <int D, bool kDQ>
struct BwdCfg {
    static constexpr int BT = 128;                 // rows of a unit's tile (query or key)
    static constexpr int BC = kDQ ? 128 : 64;      // columns of a step (the other index)
    static constexpr int NCB = D / 64;             // 128-byte column blocks of a bf16 row
    static constexpr int FIX_CB = BT * 128;        // one column block of a fixed tile
    static constexpr int FIX_BYTES = NCB * FIX_CB;
    static constexpr int RING_CB = BC * 128;       // one column block of a ring tile
    static constexpr int RING_BYTES = NCB * RING_CB;
    static constexpr int SMEM_CAP = 227 * 1024;
    // barriers (+ dK/dV: per-warp LSE / D at +512), then the packed-sequence schedule table
    static constexpr int TAB_OFF = kDQ ? 256 : 512 + 4096;
    static constexpr int BAR_BYTES = TAB_OFF + 1792;
    static constexpr int ALIGN_SLACK = 1024;
    // A ring slot holds one tile (dQ pass: V_j and K_j have different lifetimes) or a
    // step's two tiles under one barrier pair (dK/dV pass: Q_i and dO_i are used alike).
    static constexpr int TILES_PER_SLOT = kDQ ? 1 : 2;
    static constexpr int SLOT_BYTES = TILES_PER_SLOT * RING_BYTES;
    static constexpr int NSLOT_FIT = (SMEM_CAP - BAR_BYTES - ALIGN_SLACK - 2 * FIX_BYTES) / SLOT_BYTES;
    static constexpr int NSLOT = NSLOT_FIT < 8 ? NSLOT_FIT : 8;
    static constexpr int SMEM_BYTES = ALIGN_SLACK + 2 * FIX_BYTES + NSLOT * SLOT_BYTES + BAR_BYTES;
    // TMEM.  dQ pass: S of step h in buffer h & 1 at 128 (h & 1) (then dS, packed), dP at
    // DQ_DP_COL, dQ at ACC_COL.  dK/dV pass: step buffer h & 1 at 128 (h & 1) holds S^T at
    // +S_OFF (then P^T) and dP^T at +DP_OFF (then dS^T); dV at ACC_COL, dK at ACC_COL + D.
    static constexpr int BUF_COLS = 128;
    static constexpr int S_OFF = 0;
    static constexpr int DP_OFF = 64;
    static constexpr int DQ_DP_COL = 256;
    static constexpr int ACC_COL = kDQ ? 384 : 256;
    static constexpr int TMEM_COLS = 512;
    static constexpr int COMPUTE_WARPS = 8;        // two warpgroups, one per step buffer
    static constexpr int NUM_THREADS = 384;        // + one control warpgroup (2 spare warps)
    static constexpr int PRODUCER_WARP = 8;
    static constexpr int MMA_WARP = 9;
    // Register split: the compute warpgroups grow to REG_COMPUTE, the control warpgroup
    // shrinks to REG_CONTROL; needs REG_POOL <= registers per thread at launch * NUM_THREADS.
    static constexpr int REG_COMPUTE = 208;
    static constexpr int REG_CONTROL = 88;
    static constexpr int REG_POOL = 256 * REG_COMPUTE + 128 * REG_CONTROL;
    static_assert(D == 64 || D == 128, "backward head dim");
    static_assert(kDQ ? ACC_COL + D <= TMEM_COLS : ACC_COL + 2 * D <= TMEM_COLS, "TMEM budget");
    static_assert(NSLOT >= (kDQ ? 5 : 4), "ring too small");
    static_assert(SMEM_BYTES <= SMEM_CAP, "shared memory");
    static_assert(sizeof(SortTab) <= 1792, "schedule table");
};

struct alignas(16) BwdBars {
    uint64_t fix_full, fix_empty;        // the unit's two fixed tiles
    uint64_t ring_full[8], ring_empty[8];
    uint64_t s_full[2], p_full[2];       // dK/dV: per TMEM step buffer (and compute warpgroup);
                                         // dQ: [0] only, one phase per step
    uint64_t dp_free;                    // dQ: the compute warps have read the step's dP
    uint64_t acc_done, acc_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(BwdBars) <= 512, "barrier block");
// dK/dV pass: after the barriers, each compute warp's copy of the LSE (log2 units, [w][0])
// and D ([w][1]) of its current step's 64 query columns: float [8][2][64].

__device__ __forceinline__ void bwd_timeout(const BwdParams& p, BwdBars* bars)
{
    atomicExch(p.status, kStatusTimeout);
    *reinterpret_cast<volatile int*>(&bars->abort_flag) = 1;
}

// One unit of work: tile t of one head of one sequence, with where its rows live.
// Batched layout: head bh, rows r at TMA coordinates (r, bh), LSE / D at bh N + r, output
// row bh N + r.  Packed sequences: head h of tokens [y0, y0 + N), row r at TMA coordinates
// (h, y0 + r), LSE / D at h T + y0 + r, output row (y0 + r) H + h.
struct BwdUnit {
    int t;            // tile (128 rows) within the sequence
    int N;            // rows of the sequence
    int c1, c2;       // TMA coordinates of row 0: (row offset, head) or (head, token)
    bool packed;
};

// LSE / D index of row r of the unit's sequence: batched [BH, N]; packed [H, T].
__device__ __forceinline__ size_t bwd_vidx(const BwdParams& p, const BwdUnit& u, int r)
{
    return u.packed ? (size_t)u.c1 * p.T + (size_t)(u.c2 + r) : (size_t)u.c2 * p.N + r;
}

// Output row (of d elements) of row r: batched [BH, N, d]; packed [T, H, d].
__device__ __forceinline__ size_t bwd_orow(const BwdParams& p, const BwdUnit& u, int r)
{
    return u.packed ? (size_t)(u.c2 + r) * p.H + u.c1 : (size_t)u.c2 * p.N + r;
}

__device__ __forceinline__ void bwd_coords(const BwdUnit& u, int r, int& c1, int& c2)
{
    c1 = u.packed ? u.c1 : u.c1 + r;
    c2 = u.packed ? u.c2 + r : u.c2;
}

// Steps (blocks of `bc` columns of the other operand, bc = 128 or 64) that tile t (rows
// [128 t, 128 t + 128)) of a sequence of N rows meets under the mask: for a query tile,
// the key blocks [lo, hi); for a key tile (transposed), the query blocks.  Computed on
// 128-column tiles, then (bc = 64) split in two and cut at the sequence end.
__device__ __forceinline__ void bwd_steps(const BwdParams& p, const BwdUnit& u, bool key_tile, int bc,
                                          int& lo, int& hi)
{
    const int t = u.t, N = u.N;
    const int a = t * 128, last = min(N, a + 128) - 1;
    lo = 0;
    hi = (N + 127) / 128;
    if (!key_tile) {
        if (p.causal) hi = min(hi, last / 128 + 1);
        else if (p.window > 0) hi = min(hi, (last + p.window) / 128 + 1);
        if (p.window > 0) lo = max(0, (a - p.window) / 128);
    } else {
        // queries i with some allowed key j in [a, last]: causal i >= j, window |i - j| <= w
        if (p.causal) lo = a / 128;
        else if (p.window > 0) lo = max(0, (a - p.window) / 128);
        if (p.window > 0) hi = min(hi, (last + p.window) / 128 + 1);
    }
    if (lo >= hi) hi = lo + 1;  // never empty (cannot happen for the masks above)
    if (bc == 64) {
        lo *= 2;
        hi = min(2 * hi, (N + 63) / 64);
    }
}

// Work order.  A pass's units are the 128-row tiles t of every head; under a causal mask
// tile t of the dQ pass meets t + 1 key tiles and tile t of the dK/dV pass nt - t query
// tiles, so units differ in cost and a round-robin over them leaves the busiest CTA ~12 %
// above the mean.  Units are therefore handed out in complementary pairs (nt - 1 - k, k)
// whose costs add up to the same nt + 1 tiles for every k; a CTA takes both halves of a
// pair, pairs go round-robin, and pairs of one head are adjacent so CTAs that run at the
// same time share that head's operands in L2.  Sub-unit s is half (s & 1) of pair s >> 1;
// the middle tile of an odd tile count appears once.  Packed sequences: pair slots are
// laid out for the longest sequence and a shorter one skips the slots it does not have;
// offsets are clamped to [0, T] so a unit never addresses a token outside the tensors.
// With up to kSortMaxSeqs packed sequences the pairs are instead dealt longest sequence
// first in snake order from the table each CTA sorts (sched.cuh).
template <bool kPacked>
__device__ __forceinline__ bool bwd_unit(const BwdParams& p, int s, BwdUnit& u, const SortTab* tab)
{
    const int npair = (p.nt + 1) >> 1;
    const int pair = s >> 1;
    int sh = pair / npair;                       // batched: bh; packed: sequence * H + head
    int k = pair - sh * npair;
    u.packed = kPacked;
    if (kPacked && tab != nullptr) {
        int seq, rem, a, b;
        sorted_pair(tab, p.num_seqs, pair, seq, rem);
        seq_span(p.cu_seqlens, seq, p.T, a, b);
        const int np = (((b - a + 127) / 128) + 1) >> 1;   // > 0 for a sequence that holds pairs
        const int h = rem / np;
        k = rem - h * np;
        sh = seq * p.H + h;
    }
    if (!u.packed) {
        u.N = p.N;
        u.c1 = 0;
        u.c2 = sh;
    } else {
        const int seq = sh / p.H, h = sh - seq * p.H;
        const int a = min(max(__ldg(p.cu_seqlens + seq), 0), p.T);
        const int b = min(max(__ldg(p.cu_seqlens + seq + 1), a), p.T);
        u.N = b - a;
        u.c1 = h;
        u.c2 = a;
    }
    const int nt = (u.N + 127) / 128;
    if (k >= ((nt + 1) >> 1)) return false;      // beyond this sequence's pairs (or empty)
    u.t = (s & 1) ? k : nt - 1 - k;
    return !((s & 1) && k == nt - 1 - k);
}

__device__ __forceinline__ int bwd_next(int s, const SortTab* tab)
{
    if (!(s & 1)) return s + 1;
    return tab != nullptr ? snake_next_sub(s) : s + 2 * (int)gridDim.x - 1;
}

// True when every (query, key) pair of the block of queries [q0, q0 + nq) and keys
// [k0, k0 + nk) lies inside the sequence and is allowed by the mask, so the step needs
// no per-element test: causal needs the last key at or before the first query, a window
// the first key within w of the last query (and, without causal, the last key within
// w after the first query).
__device__ __forceinline__ bool bwd_block_full(const BwdParams& p, int N, int q0, int nq, int k0, int nk)
{
    if (q0 + nq > N || k0 + nk > N) return false;
    if (p.causal && k0 + nk - 1 > q0) return false;
    if (p.window > 0) {
        if (k0 < q0 + nq - 1 - p.window) return false;
        if (!p.causal && k0 + nk - 1 > q0 + p.window) return false;
    }
    return true;
}

// D_i = dO_i . O_i in fp32, one warp per row.
template <int D>
__global__ void __launch_bounds__(256) bwd_dot_kernel(const BwdParams p)
{
    constexpr int E = D / 32;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    // batched: rows bh N + r, D at the same index; packed: rows token H + h, D at h T + token
    const long long nrows = p.cu_seqlens ? (long long)p.T * p.H : (long long)p.BH * p.N;
    if (row >= nrows) return;
    const __nv_bfloat16* o = reinterpret_cast<const __nv_bfloat16*>(p.o) + row * D + lane * E;
    const __nv_bfloat16* g = reinterpret_cast<const __nv_bfloat16*>(p.dout) + row * D + lane * E;
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc = fmaf(__bfloat162float(o[e]), __bfloat162float(g[e]), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) p.delta[p.cu_seqlens ? (row % p.H) * p.T + row / p.H : row] = acc;
}

// One pass (kPacked: packed variable-length sequences).  `kDQ` selects it: the dQ pass's unit is a query tile (fixed tiles Q, dO;
// ring V then K of each 128-key step, 128-row boxes), the dK/dV pass's unit is a key tile
// (fixed tiles K, V; ring Q then dO of each 64-query step, 64-row boxes).  The fixed maps
// have 128-row boxes.
template <int D, bool kDQ, bool kPacked>
__global__ void __launch_bounds__(BwdCfg<D, kDQ>::NUM_THREADS, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmFixA, const __grid_constant__ CUtensorMap tmFixB,
               const __grid_constant__ CUtensorMap tmRingA, const __grid_constant__ CUtensorMap tmRingB,
               const BwdParams p)
{
    using C = BwdCfg<D, kDQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* fix = smem;                                   // 2 fixed tiles
    uint8_t* ring = smem + 2 * C::FIX_BYTES;               // NSLOT ring tiles
    BwdBars* bars = reinterpret_cast<BwdBars*>(ring + C::NSLOT * C::SLOT_BYTES);
    const volatile int* abort_flag = &bars->abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int nsub = 2 * ((p.nt + 1) >> 1) * p.BH;         // sub-units (see bwd_unit)

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->fix_full), 1);
        mbar_init(smem_u32(&bars->fix_empty), 1);
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(smem_u32(&bars->ring_full[s]), 1);
            mbar_init(smem_u32(&bars->ring_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars->s_full[b]), 1);
            // dQ pass: all eight compute warps arrive per step; dK/dV: one warpgroup
            mbar_init(smem_u32(&bars->p_full[b]), kDQ ? C::COMPUTE_WARPS : C::COMPUTE_WARPS / 2);
        }
        mbar_init(smem_u32(&bars->dp_free), C::COMPUTE_WARPS);
        mbar_init(smem_u32(&bars->acc_done), 1);
        mbar_init(smem_u32(&bars->acc_empty), C::COMPUTE_WARPS);
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == C::MMA_WARP) {
        tmem_alloc(smem_u32(&bars->tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    // packed sequences: the sorted schedule (every thread takes part; same in all CTAs)
    const SortTab* tab = nullptr;
    if constexpr (kPacked) {
        if (p.num_seqs <= kSortMaxSeqs) {
            SortTab* t = reinterpret_cast<SortTab*>(reinterpret_cast<uint8_t*>(bars) + C::TAB_OFF);
            build_sort_tab<128>(p.cu_seqlens, p.num_seqs, p.T, p.H, t);
            tab = t;
            nsub = 2 * t->total;
        }
    }

    if (warp == C::PRODUCER_WARP) {
        regs_decrease<C::REG_CONTROL>();
        if (lane == 0) {
            const uint64_t pol_fix = l2_policy_evict_first();
            const uint64_t pol_ring = l2_policy_evict_last();
            uint32_t rc = 0, uc = 0, armed = 0;
            bool ok = true;
            for (int su = 2 * (int)blockIdx.x; su < nsub && ok; su = bwd_next(su, tab)) {
                BwdUnit un;
                if (!bwd_unit<kPacked>(p, su, un, tab)) continue;
                const int t = un.t;
                int lo, hi;
                bwd_steps(p, un, !kDQ, C::BC, lo, hi);
                if (!mbar_wait(smem_u32(&bars->fix_empty), (uc & 1) ^ 1, abort_flag, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&bars->fix_full);
                mbar_arrive_expect_tx(fb, 2 * C::FIX_BYTES);
                ++armed;
                int f1, f2;
                bwd_coords(un, t * 128, f1, f2);
#pragma unroll
                for (int cb = 0; cb < C::NCB; ++cb) {
                    tma_load_3d(smem_u32(fix + cb * C::FIX_CB), &tmFixA, fb, cb * 64, f1, f2, pol_fix);
                    tma_load_3d(smem_u32(fix + C::FIX_BYTES + cb * C::FIX_CB), &tmFixB, fb, cb * 64,
                                f1, f2, pol_fix);
                }
                for (int s = lo; s < hi && ok; ++s) {
#pragma unroll
                    for (int which = 0; which < 2; ++which) {
                        // dQ pass: V_j then K_j, a slot each; dK/dV pass: Q_i then dO_i, one slot
                        const uint32_t slot = rc % C::NSLOT;
                        const uint32_t rb = smem_u32(&bars->ring_full[slot]);
                        if (kDQ || which == 0) {
                            if (!mbar_wait(smem_u32(&bars->ring_empty[slot]), ((rc / C::NSLOT) & 1) ^ 1,
                                           abort_flag, p.timeout_ns)) {
                                ok = false;
                                break;
                            }
                            if (rc + 1 == (uint32_t)p.withhold_ring) {  // test hook: never arrives
                                ++rc;
                                if (!kDQ) break;    // the slot's second tile is not loaded either
                                continue;
                            }
                            mbar_arrive_expect_tx(rb, C::SLOT_BYTES);
                        }
                        const CUtensorMap* map = (which == 0) == kDQ ? &tmRingB : &tmRingA;
                        uint8_t* dst = ring + slot * C::SLOT_BYTES + (kDQ ? 0 : which * C::RING_BYTES);
                        int r1, r2;
                        bwd_coords(un, s * C::BC, r1, r2);
#pragma unroll
                        for (int cb = 0; cb < C::NCB; ++cb)
                            tma_load_3d(smem_u32(dst + cb * C::RING_CB), map, rb, cb * 64, r1, r2, pol_ring);
                        if (kDQ || which == 1) ++rc;
                    }
                }
                ++uc;
            }
            if (!ok) bwd_timeout(p, bars);
            // Every copy this producer issued lands before shared memory is released (after
            // an abort by another role they may still be in flight even when this loop
            // ended normally); copies end on their own, hence the fixed cleanup bound.
            const uint32_t n = rc < C::NSLOT ? rc : C::NSLOT;
            for (uint32_t k = rc - n; k < rc; ++k) {
                if (k + 1 == (uint32_t)p.withhold_ring) continue;  // never issued
                mbar_wait(smem_u32(&bars->ring_full[k % C::NSLOT]), (k / C::NSLOT) & 1, nullptr,
                          kCleanupTimeoutNs);
            }
            if (armed > 0)
                mbar_wait(smem_u32(&bars->fix_full), (armed - 1) & 1, nullptr, kCleanupTimeoutNs);
        }
    } else if (warp == C::MMA_WARP) {
      if constexpr (kDQ) {
        // ---------------------------------------------------------------- MMA, dQ pass
        // Step j (128 keys): S(j) = Q K_j^T into S buffer j & 1, dP(j) = dO V_j^T into the
        // dP columns, then dQ += dS(j) K_j.  Order per step: dP(j) once the compute warps
        // have read dP(j-1); the accumulation of step j-1; S(j+1) into the other S buffer.
        // The tensor core thus computes dP(j) while step j-1's ALU work is still running,
        // and S(j+1) while step j's is.  Ring tiles: V_j then K_j of every step.
        regs_decrease<C::REG_CONTROL>();
        constexpr uint32_t idesc_s = idesc_f32acc(1, 0, 128, 128);   // bf16, both K-major, N = 128
        constexpr uint32_t idesc_acc = idesc_f32acc(1, 1, 128, D);    // B MN-major, N = D
        const uint64_t fixA_k = sdesc_sw128(smem_u32(fix), 16, 1024);                    // Q
        const uint64_t fixB_k = sdesc_sw128(smem_u32(fix + C::FIX_BYTES), 16, 1024);     // dO
        const uint64_t ring_k = sdesc_sw128(smem_u32(ring), 16, 1024);
        const uint64_t ring_mn = sdesc_sw128(smem_u32(ring), C::RING_CB, 1024);
        uint32_t rc = 0, uc = 0, hs = 0;
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool r = ok && mbar_wait(smem_u32(bar), parity, abort_flag, p.timeout_ns);
            r = __all_sync(0xffffffffu, r);
            if (!r) ok = false;
            return r;
        };
        auto commit = [&](uint64_t* bar) { mma_commit_warp(smem_u32(bar)); };
        auto slot = [&](uint32_t n) { return n % C::NSLOT; };
        auto full = [&](uint32_t n) -> bool { return wait(&bars->ring_full[n % C::NSLOT], (n / C::NSLOT) & 1); };
        // D[128 x 128] = A[128 x D] (fixed tile) B[128 x D]^T (ring tile in slot sl), K = D
        auto mm_kk = [&](uint32_t d_col, uint64_t a0, uint32_t sl) {
            const uint64_t b0 = ring_k + (uint64_t)((sl * C::SLOT_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int byte = kk * 32;
                const uint32_t offa = ((byte / 128) * C::FIX_CB + (byte % 128)) >> 4;
                const uint32_t offb = ((byte / 128) * C::RING_CB + (byte % 128)) >> 4;
                mma_ss_warp<false>(tmem + d_col, a0 + offa, b0 + offb, idesc_s, kk > 0 ? 1u : 0u);
            }
        };
        // dQ (+)= dS (TMEM: bf16 pairs of keys 0-63 at a + [0, 32), keys 64-127 at
        // a + [64, 96), one run per compute warpgroup) * K_j (slot sl as MN-major, K = 128)
        auto mm_acc = [&](uint32_t a_col, uint32_t sl, bool accumulate) {
            const uint64_t b0 = ring_mn + (uint64_t)((sl * C::SLOT_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < C::BC / 16; ++kk)
                mma_ts_warp<false>(tmem + C::ACC_COL, tmem + a_col + (kk / 4) * 64 + (kk % 4) * 8,
                                   b0 + ((kk * 16 * 128) >> 4), idesc_acc, (kk > 0 || accumulate) ? 1u : 0u);
        };
        for (int su = 2 * (int)blockIdx.x; su < nsub && ok; su = bwd_next(su, tab)) {
            BwdUnit un;
            if (!bwd_unit<kPacked>(p, su, un, tab)) continue;
            int lo, hi;
            bwd_steps(p, un, false, C::BC, lo, hi);
            const uint32_t r0 = rc, h0 = hs;            // tiles: V_j at r0 + 2(j-lo), K_j next
            if (!wait(&bars->fix_full, uc & 1)) break;
            tc_fence_after_sync();
            if (!full(r0 + 1)) break;                   // K_lo
            tc_fence_after_sync();
            mm_kk((h0 & 1) * C::BUF_COLS, fixA_k, slot(r0 + 1));          // S(lo)
            bool acc_started = false;
            for (int j = lo; j < hi && ok; ++j) {
                const uint32_t hj = h0 + (uint32_t)(j - lo);
                const uint32_t nv = r0 + 2u * (uint32_t)(j - lo), nk = nv + 1;
                if (!full(nv)) break;                                      // V_j
                if (hj > 0 && !wait(&bars->dp_free, (hj - 1) & 1)) break;  // dP(j-1) read
                tc_fence_after_sync();
                mm_kk(C::DQ_DP_COL, fixB_k, slot(nv));                     // dP(j) = dO V_j^T
                commit(&bars->ring_empty[slot(nv)]);
                if (j == hi - 1) commit(&bars->fix_empty);                 // last use of Q, dO
                if (j > lo) {
                    // s_full(j) is committed only after p_full(j-1) is seen: the compute warps
                    // cannot start step j before finishing j-1 anyway, and so p_full never
                    // runs a phase ahead of this wait.  It precedes the accumulation, so it
                    // tracks S(j) and dP(j) only.
                    if (!wait(&bars->p_full[0], (hj - 1) & 1)) break;
                    commit(&bars->s_full[0]);
                    if (!acc_started && !wait(&bars->acc_empty, (uc & 1) ^ 1)) break;
                    tc_fence_after_sync();
                    mm_acc(((hj - 1) & 1) * C::BUF_COLS, slot(nk - 2), acc_started);   // dQ += dS(j-1) K_{j-1}
                    acc_started = true;
                    commit(&bars->ring_empty[slot(nk - 2)]);
                } else {
                    commit(&bars->s_full[0]);     // the previous step's p_full was seen at its unit's end
                }
                if (j + 1 < hi) {
                    // S buffer (j+1) & 1 was last read by the accumulation just issued
                    if (!full(nk + 2)) break;                              // K_{j+1}
                    tc_fence_after_sync();
                    mm_kk(((hj + 1) & 1) * C::BUF_COLS, fixA_k, slot(nk + 2));
                }
            }
            if (!ok) break;
            const uint32_t hl = h0 + (uint32_t)(hi - 1 - lo);              // the unit's last step
            if (!wait(&bars->p_full[0], hl & 1)) break;
            if (!acc_started && !wait(&bars->acc_empty, (uc & 1) ^ 1)) break;
            tc_fence_after_sync();
            mm_acc((hl & 1) * C::BUF_COLS, slot(r0 + 2u * (uint32_t)(hi - 1 - lo) + 1), acc_started);
            commit(&bars->ring_empty[slot(r0 + 2u * (uint32_t)(hi - 1 - lo) + 1)]);
            commit(&bars->acc_done);
            rc = r0 + 2u * (uint32_t)(hi - lo);
            hs = h0 + (uint32_t)(hi - lo);
            ++uc;
        }
        if (!ok && lane == 0) bwd_timeout(p, bars);
        commit(&bars->drain);
        mbar_wait(smem_u32(&bars->drain), 0, nullptr, kCleanupTimeoutNs);
        __syncwarp();
      } else {
        // ---------------------------------------------------------------- MMA, dK/dV pass
        regs_decrease<C::REG_CONTROL>();
        constexpr uint32_t idesc_kk = idesc_f32acc(1, 0, 128, C::BC);  // bf16, both K-major, N = 64
        constexpr uint32_t idesc_acc = idesc_f32acc(1, 1, 128, D);     // B MN-major, N = D
        const uint64_t fixA_k = sdesc_sw128(smem_u32(fix), 16, 1024);
        const uint64_t fixB_k = sdesc_sw128(smem_u32(fix + C::FIX_BYTES), 16, 1024);
        const uint64_t ring_k = sdesc_sw128(smem_u32(ring), 16, 1024);
        const uint64_t ring_mn = sdesc_sw128(smem_u32(ring), C::RING_CB, 1024);
        uint32_t rc = 0, uc = 0, hs = 0;
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool r = ok && mbar_wait(smem_u32(bar), parity, abort_flag, p.timeout_ns);
            r = __all_sync(0xffffffffu, r);
            if (!r) ok = false;
            return r;
        };
        auto commit = [&](uint64_t* bar) { mma_commit_warp(smem_u32(bar)); };
        // D[128 x 64] = A[128 x D] (fixed tile) B[64 x D]^T (ring tile), both K-major, K = D
        auto mm_kk = [&](uint32_t d_col, uint64_t a0, uint64_t b0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int byte = kk * 32;
                const uint32_t offa = ((byte / 128) * C::FIX_CB + (byte % 128)) >> 4;
                const uint32_t offb = ((byte / 128) * C::RING_CB + (byte % 128)) >> 4;
                mma_ss_warp<false>(tmem + d_col, a0 + offa, b0 + offb, idesc_kk, kk > 0 ? 1u : 0u);
            }
        };
        // acc[128 x D] (+)= A (TMEM, 128 x 64 bf16 as 32 columns of pairs at a_col) * B (ring
        // tile as MN-major, K = 64 rows)
        auto mm_acc = [&](uint32_t acc_col, uint32_t a_col, uint64_t bmn, bool accumulate) {
#pragma unroll
            for (int kk = 0; kk < C::BC / 16; ++kk)
                mma_ts_warp<false>(tmem + acc_col, tmem + a_col + kk * 8, bmn + ((kk * 16 * 128) >> 4),
                                   idesc_acc, (kk > 0 || accumulate) ? 1u : 0u);
        };
        for (int su = 2 * (int)blockIdx.x; su < nsub && ok; su = bwd_next(su, tab)) {
            BwdUnit un;
            if (!bwd_unit<kPacked>(p, su, un, tab)) continue;
            int lo, hi;
            bwd_steps(p, un, !kDQ, C::BC, lo, hi);
            if (!wait(&bars->fix_full, uc & 1)) break;
            tc_fence_after_sync();
            bool acc_started = false;
            // accumulation of step h (its P / dS are in TMEM once p_full fires), then the
            // step's two ring tiles are free
            auto issue_acc = [&](uint32_t h, uint32_t sa) -> bool {
                if (!wait(&bars->p_full[h & 1], (h >> 1) & 1)) return false;
                if (!acc_started && !wait(&bars->acc_empty, (uc & 1) ^ 1)) return false;
                tc_fence_after_sync();
                const uint64_t ma = ring_mn + (uint64_t)((sa * C::SLOT_BYTES) >> 4);               // Q_i
                const uint64_t mb = ring_mn + (uint64_t)((sa * C::SLOT_BYTES + C::RING_BYTES) >> 4);  // dO_i
                const uint32_t bc = (h & 1) * C::BUF_COLS;
                if constexpr (kDQ) {
                    mm_acc(C::ACC_COL, bc + C::S_OFF, ma, acc_started);          // dQ += dS K
                } else {
                    mm_acc(C::ACC_COL, bc + C::S_OFF, mb, acc_started);          // dV += P^T dO
                    mm_acc(C::ACC_COL + D, bc + C::DP_OFF, ma, acc_started);     // dK += dS^T Q
                }
                acc_started = true;
                commit(&bars->ring_empty[sa]);
                return true;
            };
            uint32_t psa = 0;
            bool pend = false;
            for (int s = lo; s < hi; ++s) {
                const uint32_t sa = rc % C::NSLOT;       // Q_i and dO_i of this step
                if (!wait(&bars->ring_full[sa], (rc / C::NSLOT) & 1)) break;
                tc_fence_after_sync();
                // buffer hs & 1 was last read by step hs - 2's accumulation, issued earlier
                const uint32_t bc = (hs & 1) * C::BUF_COLS;
                mm_kk(bc + C::S_OFF, fixA_k, ring_k + (uint64_t)((sa * C::SLOT_BYTES) >> 4));                 // S^T
                mm_kk(bc + C::DP_OFF, fixB_k, ring_k + (uint64_t)((sa * C::SLOT_BYTES + C::RING_BYTES) >> 4));  // dP^T
                commit(&bars->s_full[hs & 1]);
                if (s == hi - 1) commit(&bars->fix_empty);
                if (pend && !issue_acc(hs - 1, psa)) break;
                psa = sa;
                pend = true;
                ++hs;
                rc += 1;
            }
            if (!ok) break;
            if (!issue_acc(hs - 1, psa)) break;
            commit(&bars->acc_done);
            ++uc;
        }
        if (!ok && lane == 0) bwd_timeout(p, bars);
        commit(&bars->drain);
        mbar_wait(smem_u32(&bars->drain), 0, nullptr, kCleanupTimeoutNs);
        __syncwarp();
      }
    } else if (warp < C::COMPUTE_WARPS) {
        // ---------------------------------------------------------------- compute warpgroups
        // warpgroup wg takes the steps whose global index h has h & 1 == wg (TMEM buffer
        // wg); a warp reaches the TMEM lanes of its index within the warpgroup
        regs_increase<C::REG_COMPUTE>();
        const int wg = warp >> 2;
        const int trow = (warp & 3) * 32 + lane;        // row of this thread in the tile
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t buf = tmem + lane_addr + (uint32_t)wg * C::BUF_COLS;
        const float LOG2E = 1.4426950408889634f;
        uint32_t h = 0, uc = 0;
        bool ok = true;
        auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool r = ok && mbar_wait(smem_u32(bar), parity, abort_flag, p.timeout_ns);
            r = __all_sync(0xffffffffu, r);
            if (!r) ok = false;
            return r;
        };
        // dK/dV pass: lane l holds the LSE (log2 units) and D of columns c + 2l, c + 2l + 1
        // of a step; each warp keeps its own copy in shared memory while it works on it
        float* my_lse2 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 512) + warp * 128;
        float* my_delta = my_lse2 + 64;
        auto col_load = [&](const BwdUnit& cu, int c, float2& l2v, float2& dv) {
            const size_t base = bwd_vidx(p, cu, 0);
            const int c0 = min(c + 2 * lane, cu.N - 1), c1 = min(c + 2 * lane + 1, cu.N - 1);
            l2v = make_float2(__ldg(p.lse + base + c0) * LOG2E, __ldg(p.lse + base + c1) * LOG2E);
            dv = make_float2(__ldg(p.delta + base + c0), __ldg(p.delta + base + c1));
        };
        for (int su = 2 * (int)blockIdx.x; su < nsub && ok; su = bwd_next(su, tab)) {
            BwdUnit un;
            if (!bwd_unit<kPacked>(p, su, un, tab)) continue;
            const int t = un.t, NS = un.N;              // tile and sequence length
            int lo, hi;
            bwd_steps(p, un, !kDQ, C::BC, lo, hi);
            const int my = t * 128 + trow;              // this thread's row (query or key)
            const bool valid = my < NS;
            float lse2 = 0.0f, dlt = 0.0f;              // dQ pass: per-row LSE and D
            if constexpr (kDQ) {
                lse2 = valid ? p.lse[bwd_vidx(p, un, my)] * LOG2E : 0.0f;
                dlt = valid ? p.delta[bwd_vidx(p, un, my)] : 0.0f;
            }
            // The columns (the other index) the mask allows for this thread's row form one
            // interval [m_lo, m_hi]: for a query row, keys from i - w (w > 0) or 0 to i
            // (causal) or i + w (window) or N - 1; for a key row, queries from j (causal) or
            // j - w (window) or 0, to j + w (window) or N - 1.  One unsigned compare per
            // element tests it.  A row past N gets some interval: its values stay finite and
            // are never stored (row r of a product depends on row r of its TMEM operand only).
            int m_lo, m_hi;
            if constexpr (kDQ) {
                m_lo = p.window > 0 ? my - p.window : 0;
                m_hi = p.causal ? my : (p.window > 0 ? my + p.window : NS - 1);
            } else {
                m_lo = p.causal ? my : (p.window > 0 ? my - p.window : 0);
                m_hi = p.window > 0 ? my + p.window : NS - 1;
            }
            m_hi = min(m_hi, NS - 1);   // packed: the next sequence's tokens in a tile are masked
            const uint32_t m_span = (uint32_t)(m_hi - m_lo);
          if constexpr (kDQ) {
            // dQ pass: both warpgroups work on every step, warpgroup wg on keys
            // [64 wg, 64 wg + 64) of it; dP is released as soon as it is in registers
            const uint32_t h0 = h;                      // global index of step lo
            h = h0 + (uint32_t)(hi - lo);
            for (int j = lo; j < hi; ++j) {
                const uint32_t hj = h0 + (uint32_t)(j - lo);
                const int c0 = j * C::BC + wg * 64;     // this warpgroup's first key
                if (!wait_all(&bars->s_full[0], hj & 1)) break;
                tc_fence_after_sync();
                const uint32_t sb = tmem + lane_addr + (hj & 1) * C::BUF_COLS + (uint32_t)wg * 64;
                const uint32_t db = tmem + lane_addr + C::DQ_DP_COL + (uint32_t)wg * 64;
                uint32_t sra[64], dra[64];
                tmem_ld32p(sb, sra);
                tmem_ld32p(sb + 32, sra + 32);
                tmem_ld32p(db, dra);
                tmem_ld32p(db + 32, dra + 32);
                tmem_wait_ld_only();
                reg_fence32(sra);
                reg_fence32(sra + 32);
                reg_fence32(dra);
                reg_fence32(dra + 32);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->dp_free));
                // dS = P * (dP - D) of this thread's row over the warpgroup's 64 keys, packed to
                // bf16 pairs over the first 32 of its S columns (already in registers)
                auto stepq = [&](auto masked_tag) {
                    constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float dsv[2];
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const int i = ch * 32 + 2 * e + h2;
                                float pr = ex2(fmaf(__uint_as_float(sra[i]), p.c_log2, -lse2));
                                if constexpr (kMasked) {
                                    // key c0 + i is allowed iff it lies in [m_lo, m_hi]
                                    const uint32_t off = (uint32_t)(c0 - m_lo) + (uint32_t)i;
                                    pr = off <= m_span ? pr : 0.0f;
                                }
                                dsv[h2] = pr * (__uint_as_float(dra[i]) - dlt);
                            }
                            pk[e] = pack_bf16x2(dsv[0], dsv[1]);
                        }
                        tmem_st16p(sb + ch * 16, pk);
                    }
                };
                if (bwd_block_full(p, NS, t * 128, 128, j * C::BC, C::BC))
                    stepq(std::false_type{});
                else
                    stepq(std::true_type{});
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[0]));
            }
          } else {
            const uint32_t h0 = h;                      // global index of step lo
            h = h0 + (uint32_t)(hi - lo);
            int s = lo + (int)((h0 ^ (uint32_t)wg) & 1u);   // this warpgroup's first step
            [[maybe_unused]] float2 nl2 = make_float2(0.f, 0.f), nd = nl2;
            if constexpr (!kDQ) {
                if (s < hi) col_load(un, s * C::BC, nl2, nd);
            }
            for (; s < hi; s += 2) {
                const uint32_t hh = h0 + (uint32_t)(s - lo);
                const int c0 = s * C::BC;               // first column (key / query) of the step
                if constexpr (!kDQ) {
                    // publish this step's column values to the warp's copy, then prefetch
                    // the warpgroup's next step (two on) into registers
                    __syncwarp();                       // the previous step's reads are done
                    *reinterpret_cast<float2*>(my_lse2 + 2 * lane) = nl2;
                    *reinterpret_cast<float2*>(my_delta + 2 * lane) = nd;
                    __syncwarp();
                    if (s + 2 < hi) col_load(un, c0 + 2 * C::BC, nl2, nd);
                }
                if (!wait_all(&bars->s_full[wg], (hh >> 1) & 1)) break;
                tc_fence_after_sync();
                // P and dS of this thread's row over the step's 64 columns, 32 at a time; the
                // mask is evaluated only on blocks that cross the diagonal, a window edge or
                // the sequence end
                auto step = [&](auto masked_tag) {
                    constexpr bool kMasked = decltype(masked_tag)::value;
                    uint32_t sra[64], dra[64];              // the step's S and dP row, one wait
                    tmem_ld32p(buf + C::S_OFF, sra);
                    tmem_ld32p(buf + C::S_OFF + 32, sra + 32);
                    tmem_ld32p(buf + C::DP_OFF, dra);
                    tmem_ld32p(buf + C::DP_OFF + 32, dra + 32);
                    tmem_wait_ld_only();
                    reg_fence32(sra);
                    reg_fence32(sra + 32);
                    reg_fence32(dra);
                    reg_fence32(dra + 32);
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        const int cc = ch * 32;
                        const uint32_t* sr = sra + cc;
                        const uint32_t* dr = dra + cc;
                        uint32_t pk[16];
                        [[maybe_unused]] uint32_t pkp[16];
                        [[maybe_unused]] float4 l4, d4;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            if constexpr (!kDQ) {
                                if ((e & 1) == 0) {   // four columns' LSE and D per vector load
                                    l4 = *reinterpret_cast<const float4*>(my_lse2 + cc + 2 * e);
                                    d4 = *reinterpret_cast<const float4*>(my_delta + cc + 2 * e);
                                }
                            }
                            float pv[2], dsv[2];
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                float l2 = lse2, dl = dlt;
                                if constexpr (!kDQ) {
                                    l2 = (e & 1) ? (h2 ? l4.w : l4.z) : (h2 ? l4.y : l4.x);
                                    dl = (e & 1) ? (h2 ? d4.w : d4.z) : (h2 ? d4.y : d4.x);
                                }
                                const float sv = __uint_as_float(sr[2 * e + h2]);
                                float pr = ex2(fmaf(sv, p.c_log2, -l2));
                                if constexpr (kMasked) {
                                    // column c0 + cc + 2e + h2 is allowed iff it lies in [m_lo, m_hi]
                                    const uint32_t off = (uint32_t)(c0 + cc - m_lo) + (uint32_t)(2 * e + h2);
                                    pr = off <= m_span ? pr : 0.0f;
                                }
                                pv[h2] = pr;
                                dsv[h2] = pr * (__uint_as_float(dr[2 * e + h2]) - dl);
                            }
                            pk[e] = pack_bf16x2(dsv[0], dsv[1]);
                            if constexpr (!kDQ) pkp[e] = pack_bf16x2(pv[0], pv[1]);
                        }
                        // bf16 pairs: chunk ch fills packed TMEM columns [16 ch, 16 ch + 16) of
                        // the buffer's S (dP) columns, already loaded above
                        if constexpr (kDQ) {
                            tmem_st16p(buf + C::S_OFF + ch * 16, pk);             // dS over S
                        } else {
                            tmem_st16p(buf + C::S_OFF + ch * 16, pkp);            // P^T over S^T
                            tmem_st16p(buf + C::DP_OFF + ch * 16, pk);            // dS^T over dP^T
                        }
                    }
                };
                if (bwd_block_full(p, NS, kDQ ? t * 128 : c0, kDQ ? 128 : C::BC, kDQ ? c0 : t * 128,
                                   kDQ ? C::BC : 128))
                    step(std::false_type{});
                else
                    step(std::true_type{});
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[wg]));
            }
          }
            if (!ok) break;
            // epilogue: dQ (or dV, dK) from TMEM, times scale where it applies, to bf16.
            // dQ pass: each warpgroup writes half of dQ's columns; dK/dV pass: warpgroup 0
            // writes dV, warpgroup 1 dK
            if (!wait_all(&bars->acc_done, uc & 1)) break;
            tc_fence_after_sync();
            {
                const int which = kDQ ? 0 : wg;
                const float f = kDQ ? p.scale : (which == 0 ? 1.0f : p.scale);
                __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(kDQ ? p.dq : (which == 0 ? p.dv : p.dk));
                out += bwd_orow(p, un, my) * D;
                constexpr int NCH = kDQ ? D / 64 : D / 32;     // 32-column chunks per warpgroup
                const int ch0 = kDQ ? wg * NCH : 0;
#pragma unroll
                for (int ci = 0; ci < NCH; ++ci) {
                    const int ch = ch0 + ci;
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_addr + C::ACC_COL + which * D + ch * 32, r);
                    tmem_wait_ld(r);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * f, __uint_as_float(r[2 * e + 1]) * f);
                    if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(out + ch * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty));
            ++uc;
        }
        if (!ok) bwd_timeout(p, bars);
        tmem_wait_st();  // an aborted step may have left a P or dS store in flight
    } else {
        regs_decrease<C::REG_CONTROL>();                // spare warps of the control warpgroup
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == C::MMA_WARP) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, bool kPacked>
cudaError_t launch_bwd_t(const BwdMaps& m, const BwdParams& p, int sm_count, cudaStream_t stream)
{
    using CQ = BwdCfg<D, true>;
    using CKV = BwdCfg<D, false>;
    const long long rows = p.cu_seqlens ? (long long)p.T * p.H : (long long)p.BH * p.N;
    bwd_dot_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int pairs = ((p.nt + 1) >> 1) * p.BH;     // units go out in pairs (bwd_unit)
    const int grid = pairs < sm_count ? pairs : sm_count;
    auto kq = bwd_kernel<D, true, kPacked>;
    auto kkv = bwd_kernel<D, false, kPacked>;
    if ((e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, CQ::SMEM_BYTES)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, CKV::SMEM_BYTES)) != cudaSuccess)
        return e;
    // setmaxnreg.inc would wait forever if the launch pool were smaller than the split
    for (const void* f : {reinterpret_cast<const void*>(kq), reinterpret_cast<const void*>(kkv)}) {
        cudaFuncAttributes attr;
        if ((e = cudaFuncGetAttributes(&attr, f)) != cudaSuccess) return e;
        if (attr.numRegs * CQ::NUM_THREADS < CQ::REG_POOL) return cudaErrorInvalidConfiguration;
    }
    // dQ pass: ring K and V with 128-row boxes; dK/dV pass: ring Q and dO with 64-row boxes
    kq<<<grid, CQ::NUM_THREADS, CQ::SMEM_BYTES, stream>>>(m.q, m.dout, m.k, m.v, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kkv<<<grid, CKV::NUM_THREADS, CKV::SMEM_BYTES, stream>>>(m.k, m.v, m.q64, m.dout64, p);
    return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdMaps& m, const BwdParams& p, int d, int sm_count, cudaStream_t stream)
{
    const bool packed = p.cu_seqlens != nullptr;
    if (d == 64) return packed ? launch_bwd_t<64, true>(m, p, sm_count, stream)
                               : launch_bwd_t<64, false>(m, p, sm_count, stream);
    if (d == 128) return packed ? launch_bwd_t<128, true>(m, p, sm_count, stream)
                                : launch_bwd_t<128, false>(m, p, sm_count, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gb300
