// attn_fwd.cuh -- fused exact-attention forward for sm_103a (tcgen05 + TMA + TMEM).
//
// Computes, per head, O = softmax(scale * Q K^T + mask) V and the per-row
// log-sum-exp, block by block with an online softmax so the N x N scores never
// leave the SM.  Pages it follows (titles as published):
//   [WGC] "Warp Group Cluster 优化：Flash Attention V3 在 H100 上的 FP8 融合计算实践"
//         §2 GEMM-Softmax 融合流水线 (local max/sum, running statistics, rescale,
//         straight into the next GEMM), §3 FP8 量化与精度保持 (per-block scaling,
//         FP32 accumulation, 16-bit output), 运行时调优 (128-row Q tiles, 3-4 stage pipeline)
//   [JJ]  "大模型加速-核心网络算子-Flash Attention V3"
//         §2.1 producer/consumer warp specialisation and ping-pong of two softmax
//         groups against the GEMMs, §2.2 softmax overlapped with the asynchronous
//         GEMMs, §1.1 TMA block copies, §2.4 (first) transaction-count barriers
//   [YT]  "FlashAttention V3：优化框架吞吐量的关键技术实践"
//         §1.2 mask fused with matmul and softmax, §2.1.2 band-mask zero-region skipping
//
// Blackwell design (not a port of the Hopper one on the pages):
//   * one persistent CTA per SM walks work units (head, 128*NQ query rows);
//   * warp PRODUCER (one lane) streams Q tiles and K/V tiles with TMA into a
//     ring of NSLOT shared-memory slots, each guarded by a full/empty mbarrier;
//   * warp MMA (one lane) issues tcgen05.mma: S = Q K^T into tensor memory, and
//     O += P V with P read back from tensor memory (it overwrites S in place);
//   * NQ softmax warpgroups (one thread = one query row) read S from TMEM,
//     apply the mask on edge tiles, update the running max with a lazy
//     threshold, exponentiate with ex2, keep the running sum, write P to TMEM
//     and, only when the stale maximum would let P exceed 2^tau, rescale their
//     O rows in TMEM; at the end they normalise O, write the LSE and (d = 128) send
//     their O rows out through a small shared-memory slab per warp with TMA stores, so
//     they go on to the next unit without waiting for global stores (d = 64 and 256,
//     and packed rows that run past their sequence, store directly).
//   With NQ = 2 the two Q tiles ping-pong: one group's softmax runs while the
//   tensor core works on the other tile's GEMMs.  With NQ = 1 (d = 256) S is
//   double-buffered so QK^T of the next block overlaps the current softmax.
#pragma once

#include <cuda_bf16.h>

#include "attn_params.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace gb300 {

template <int D, bool F8, bool PK = false, bool Q64 = false>
struct FwdCfg {
    static constexpr bool PACKED = PK;                   // packed variable-length sequences
    // fp8: Q and K scaled per 64-row block (two K descales per 128-key tile); otherwise 128
    static constexpr bool QK64 = Q64;
    static constexpr int BM = 128;                       // query rows per Q tile (MMA M)
    static constexpr int NQ = (D <= 128) ? 2 : 1;        // Q tiles per work unit
    static constexpr int BN = (D == 256 && !F8) ? 64 : 128;  // keys per K/V tile
    static constexpr int EB = F8 ? 1 : 2;                // bytes per operand element
    // swizzle span: 128 bytes, or 64 when a whole row is 64 bytes (fp8, d = 64)
    static constexpr int SWZ = D * EB < 128 ? D * EB : 128;
    static constexpr int SWE = SWZ / EB;                 // elements per swizzle row
    static constexpr int NCB = D / SWE;                  // swizzle-row column blocks per row
    static constexpr int CB_Q_BYTES = BM * SWZ;
    static constexpr int CB_KV_BYTES = BN * SWZ;
    static constexpr int Q_BYTES = NCB * CB_Q_BYTES;
    static constexpr int KV_BYTES = NCB * CB_KV_BYTES;
    static constexpr int SMEM_CAP = 227 * 1024;
    // barriers (FwdBars, 256 bytes at most) followed by the packed-sequence schedule table
    static constexpr int BAR_BYTES = 2048;
    static constexpr int ALIGN_SLACK = 1024;
    // d = 128: each softmax warp's 32 O rows leave through its own 4 KB slab of shared memory
    // (32 rows x 64 bf16, 128-byte swizzled, the layout a TMA store reads), one 64-column half
    // at a time, by TMA stores its lane 0 issues; the warp waits only for its own previous
    // store.  (d = 64 measured 1 % slower with it; d = 256 has no shared memory to spare.)
    static constexpr bool OSTAGE = D == 128;
    static constexpr int O_SLAB_BYTES = 32 * 128;
    static constexpr int OSTAGE_BYTES = OSTAGE ? 4 * NQ * O_SLAB_BYTES : 0;
    static constexpr int NSLOT_FIT =
        (SMEM_CAP - BAR_BYTES - ALIGN_SLACK - NQ * Q_BYTES - OSTAGE_BYTES) / KV_BYTES;
    static constexpr int NSLOT = NSLOT_FIT < 8 ? NSLOT_FIT : 8;
    static constexpr int SMEM_BYTES = ALIGN_SLACK + NQ * Q_BYTES + NSLOT * KV_BYTES + OSTAGE_BYTES + BAR_BYTES;
    static constexpr int K_STEP = F8 ? 32 : 16;          // K per tcgen05.mma
    static constexpr int NSB = 2;                        // S/P buffers in TMEM
    static constexpr int S_COL0 = 0;                     // S buffer b at columns [b*BN, b*BN+BN)
    static constexpr int O_COL0 = NSB * BN;              // O of Q tile i at [O_COL0 + i*D, +D)
    static constexpr int TMEM_COLS = 512;
    static constexpr int P_COLS = BN * EB / 4;           // packed P columns (2 bf16 / 4 e4m3 per col)
    static constexpr int NUM_SOFTMAX_WARPS = 4 * NQ;
    static constexpr int PRODUCER_WARP = NUM_SOFTMAX_WARPS;   // first warp of the last warpgroup
    static constexpr int MMA_WARP = NUM_SOFTMAX_WARPS + 1;
    static constexpr int NUM_THREADS = 32 * (NUM_SOFTMAX_WARPS + 4);  // whole warpgroups
    // Register split (NQ = 2 only): softmax warpgroups grow, the control warpgroup
    // shrinks.  Needs REG_POOL <= registers per thread at launch * NUM_THREADS.
    static constexpr bool SPLIT_REGS = NQ == 2;
    static constexpr int REG_SOFTMAX = 208;
    static constexpr int REG_CONTROL = 88;
    static constexpr int REG_POOL = NQ * 128 * REG_SOFTMAX + 128 * REG_CONTROL;
    // bf16: lazy-rescale threshold in log2 units (P <= 2^TAU while the max is stale).
    // fp8: the running max is always exact (P <= 1) and O is rescaled every key tile
    // anyway, because the V descale of tile t is applied to O, not folded into P.
    static constexpr float TAU = 8.0f;
    // fp8: P is stored as e4m3(p * 2^P8_SHIFT); a power of two keeps p = 1 exact.
    static constexpr int P8_SHIFT = 8;

    static_assert(D == 64 || D == 128 || D == 256, "head dim");
    static_assert(SWZ == 128 || SWZ == 64, "swizzle span");
    static_assert(!F8 || BN == 128, "fp8: one 128-row V scale block per key tile");
    static_assert(NSLOT >= 3, "ring too small");
    static_assert(O_COL0 + NQ * D <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= SMEM_CAP, "shared memory budget");
    static_assert(BN % 32 == 0 && D % 32 == 0, "chunking");
};

// Shared-memory barrier block (lives in the last BAR_BYTES of dynamic smem).
struct alignas(8) FwdBars {
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t kv_full[8];
    uint64_t kv_empty[8];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t pv_done[2];
    uint64_t o_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Packed sequences: the schedule table (sched.cuh) sits in the barrier block.
constexpr int kSortTabOffset = 256;  // bytes into the barrier block
static_assert(kSortTabOffset + sizeof(SortTab) <= 2048, "schedule table must fit the barrier block");
static_assert(sizeof(FwdBars) <= kSortTabOffset, "barriers must end before the schedule table");

struct Unit {
    int z;       // batched: flattened (batch, head); packed sequences: the head
    int y0;      // packed sequences: first token of the sequence (0 when batched)
    int N;       // rows (= keys) of this unit's sequence
    int q0;      // first query row of the unit, relative to its sequence
    int t0;      // first key tile
    int n;       // key tiles visited
};

// Work decomposition.  A work unit is (head, query block of NQ*128 rows).  The
// query blocks of a head are handed out in complementary pairs (nq-1-k, k): under
// a causal mask the two halves' key ranges add up to the same count for every k,
// so giving pairs to CTAs round-robin balances the persistent grid without a
// runtime scheduler ("dynamic load balancing" is what the pages ask for; here the
// balance is built into the order).  Pairs of one head are adjacent, so CTAs that
// run at the same time share that head's K/V in L2.  Sub-unit s is half (s & 1)
// of pair s >> 1, the heavy half first; a CTA walks 2c, 2c+1, 2c+2G, 2c+2G+1, ...
// Without a causal mask the units of a head cost the same (with a window, all but those
// near the sequence's ends), and when whole pairs would leave part of the grid a round
// short (512 pairs on 152 CTAs: 4 rounds for some, 3 for the rest) the CTAs walk single
// units in rotated rounds instead (unit_walk, chosen by the host; see first_sub).
// Returns false for the empty second half of the middle pair when nq is odd.
// Packed sequences ("FlashAttention V3：优化框架吞吐量的关键技术实践" §1.1, variable
// sequence lengths): pair slots are laid out for the longest sequence and a
// shorter one skips the slots it does not have; offsets are clamped to [0, T] so
// a unit never addresses a token outside the tensors.
template <class C>
__device__ __forceinline__ bool unit_of(int s, const FwdParams& p, Unit& w, const SortTab* tab)
{
    const int npair = (p.num_qblk + 1) >> 1;
    const int pair = s >> 1;
    int k = pair % npair;
    int nq = p.num_qblk;
    if constexpr (!C::PACKED) {
        w.z = pair / npair;
        w.y0 = 0;
        w.N = p.N;
    } else if (tab != nullptr) {
        // sorted packed sequences (sched.cuh)
        int seq, rem, a, b;
        sorted_pair(tab, p.num_seqs, pair, seq, rem);
        seq_span(p.cu_seqlens, seq, p.T, a, b);
        w.y0 = a;
        w.N = b - a;
        nq = (w.N + C::NQ * C::BM - 1) / (C::NQ * C::BM);
        const int np = (nq + 1) >> 1;                 // > 0: empty sequences hold no pairs
        w.z = rem / np;
        k = rem - w.z * np;
    } else {
        // more sequences than the table holds: round-robin over pair slots laid out
        // for the longest sequence; a shorter one skips the slots it does not have
        const int sh = pair / npair;
        const int seq = sh / p.H;
        w.z = sh - seq * p.H;
        int a, b;
        seq_span(p.cu_seqlens, seq, p.T, a, b);
        w.y0 = a;
        w.N = b - a;
        nq = (w.N + C::NQ * C::BM - 1) / (C::NQ * C::BM);
        if (k >= ((nq + 1) >> 1)) return false;  // beyond this sequence's pairs
    }
    const int qb = (s & 1) ? k : nq - 1 - k;
    if ((s & 1) && qb == nq - 1 - k) return false;
    w.q0 = qb * (C::NQ * C::BM);
    const int r_last = min(w.N, w.q0 + C::NQ * C::BM) - 1;
    int lo = 0, hi = w.N;  // keys [lo, hi) that some row of the unit may use
    if (p.window > 0) lo = max(0, w.q0 - p.window);
    if (p.causal) hi = r_last + 1;
    else if (p.window > 0) hi = min(w.N, r_last + p.window + 1);
    w.t0 = lo / C::BN;
    w.n = (hi + C::BN - 1) / C::BN - w.t0;
    return true;
}

__device__ __forceinline__ int next_sub(int s) { return (s & 1) ? s + 2 * (int)gridDim.x - 1 : s + 1; }

// The next sub-unit of this CTA: the second half of its pair, or the first half of its
// pair in the next round -- round-robin, or snake order over the sorted table.
__device__ __forceinline__ int next_sub(int s, const SortTab* tab)
{
    if (tab == nullptr || !(s & 1)) return next_sub(s);
    return snake_next_sub(s);
}

// This CTA's first sub-unit and its next one after s: packed sequences walk pairs (round-
// robin or snake); batched launches walk pairs round-robin, or single units with a plain
// stride (no mask: every unit costs the same), or under a window single units in rotated
// rounds: in round r CTA c takes unit r*G + (c + r) mod G.  Each round covers the same
// G units as a plain stride, but a CTA moves one position along a head's units per
// round; with a plain stride and G a multiple of a head's unit count, every CTA would
// meet the same position (under a window, the same cost) in every head.
// The batched walks are one rule whose constants the launch writes: pairs step +1 from
// the first half to the second and +(2G - 1) to the next pair; plain-stride units +G;
// rotated units +(G + 1), or +1 where (c + r + 1) mod G wraps to 0.
template <class C>
__device__ __forceinline__ int first_sub(const FwdParams& p)
{
    if constexpr (C::PACKED) return 2 * (int)blockIdx.x;
    else return (int)blockIdx.x * p.walk_first;
}
template <class C>
__device__ __forceinline__ int next_sub(int s, const FwdParams& p, const SortTab* tab)
{
    if constexpr (C::PACKED) return next_sub(s, tab);
    else return s + 1 + (((s + p.walk_a) % p.walk_m == 0) ? 0 : p.walk_step);
}

// Sub-units [0, 2 * pairs) exist: pair slots of the layout, or the table's exact count.
__device__ __forceinline__ int num_subs(const FwdParams& p, const SortTab* tab)
{
    return 2 * (tab != nullptr ? tab->total : p.num_units);
}

// Steps [L, R) of the unit's key-tile range that Q tile i needs: a key tile is
// skipped for a Q tile when every (row, key) pair of it is masked (causal: all
// keys after the tile's last row; band: all keys before its first row's window,
// or after its last row's).  Never empty; with one Q tile the whole range.
template <class C>
__device__ __forceinline__ void tile_steps(const Unit& w, int i, const FwdParams& p, int& L, int& R)
{
    L = 0;
    R = w.n;
    if constexpr (C::NQ == 2) {
        const int a = w.q0 + i * C::BM, last = a + C::BM - 1;
        int lo_t = w.t0, hi_t = w.t0 + w.n;
        if (p.causal) hi_t = min(hi_t, last / C::BN + 1);
        else if (p.window > 0) hi_t = min(hi_t, (last + p.window) / C::BN + 1);
        if (p.window > 0 && a - p.window > 0) lo_t = max(lo_t, (a - p.window) / C::BN);
        if (lo_t >= hi_t) {
            lo_t = w.t0 + w.n - 1;
            hi_t = w.t0 + w.n;
        }
        L = lo_t - w.t0;
        R = hi_t - w.t0;
    }
}

// Whether the 32 O rows of softmax warp wq of the Q tile starting at row a leave through the
// warp's slab and TMA stores: batched rows past N are clipped by the tensor map; packed rows
// that run past their sequence's end would write into the next sequence, so such a warp (and
// every warp at d = 64 or 256) stores its rows directly.
template <class C>
__device__ __forceinline__ bool slab_staged(const Unit& w, int a, int wq)
{
    if constexpr (!C::OSTAGE) return false;
    const int r0 = a + wq * 32;
    if (r0 >= w.N) return false;
    if constexpr (C::PACKED) return r0 + 32 <= w.N;
    return true;
}

__device__ __forceinline__ void raise_timeout(const FwdParams& p, FwdBars* bars)
{
    atomicExch(p.status, kStatusTimeout);
    *reinterpret_cast<volatile int*>(&bars->abort_flag) = 1;
}

template <int D, bool F8, bool PK = false, bool QK64 = false>
__global__ void __launch_bounds__(FwdCfg<D, F8>::NUM_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const FwdParams p)
{
    using C = FwdCfg<D, F8, PK, QK64>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* q_smem = smem;                                   // NQ tiles
    uint8_t* kv_smem = smem + C::NQ * C::Q_BYTES;             // NSLOT tiles
    uint8_t* ostage = kv_smem + C::NSLOT * C::KV_BYTES;       // O slabs, one per softmax warp
    FwdBars* bars = reinterpret_cast<FwdBars*>(ostage + C::OSTAGE_BYTES);
    const volatile int* abort_flag = &bars->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // packed sequences: the sorted schedule (every thread takes part; same result in all CTAs)
    const SortTab* tab = nullptr;
    if constexpr (C::PACKED) {
        if (p.num_seqs <= kSortMaxSeqs) {
            SortTab* t = reinterpret_cast<SortTab*>(reinterpret_cast<uint8_t*>(bars) + kSortTabOffset);
            build_sort_tab<C::NQ * C::BM>(p.cu_seqlens, p.num_seqs, p.T, p.H, t);
            tab = t;
        }
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars->q_full[i]), 1);
            mbar_init(smem_u32(&bars->q_empty[i]), 1);
            mbar_init(smem_u32(&bars->s_full[i]), 1);
            mbar_init(smem_u32(&bars->p_full[i]), 4);
            mbar_init(smem_u32(&bars->pv_done[i]), 1);
            mbar_init(smem_u32(&bars->o_empty[i]), 4);
        }
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(smem_u32(&bars->kv_full[s]), 1);
            mbar_init(smem_u32(&bars->kv_empty[s]), 1);
        }
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == C::PRODUCER_WARP && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        if constexpr (C::OSTAGE) tma_prefetch_desc(&tmO);
    }
    if (warp == C::MMA_WARP) {
        tmem_alloc(smem_u32(&bars->tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    if (warp == C::PRODUCER_WARP) {
        // ------------------------------------------------------------ TMA producer
        if constexpr (C::SPLIT_REGS) regs_decrease<C::REG_CONTROL>();
        if (lane == 0) {
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            uint32_t ring = 0, uc = 0;
            uint32_t q_armed[2] = {0, 0};
            bool ok = true;
            for (int su = first_sub<C>(p); su < num_subs(p, tab) && ok; su = next_sub<C>(su, p, tab)) {
                Unit w;
                if (!unit_of<C>(su, p, w, tab)) continue;
                for (int i = 0; i < C::NQ && ok; ++i) {
                    const uint32_t fb = smem_u32(&bars->q_full[i]);
                    if (!mbar_wait(smem_u32(&bars->q_empty[i]), (uc & 1) ^ 1, abort_flag,
                                   p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(fb, C::Q_BYTES);
                    ++q_armed[i];
                    const uint32_t dst = smem_u32(q_smem + i * C::Q_BYTES);
                    const int row = w.q0 + i * C::BM;
#pragma unroll
                    for (int cb = 0; cb < C::NCB; ++cb) {
                        if constexpr (!C::PACKED)  // map (d, N, BH)
                            tma_load_3d(dst + cb * C::CB_Q_BYTES, &tmQ, fb, cb * C::SWE, row, w.z, pol_q);
                        else                          // map (d, H, T)
                            tma_load_3d(dst + cb * C::CB_Q_BYTES, &tmQ, fb, cb * C::SWE, w.z, w.y0 + row, pol_q);
                    }
                }
                for (int jj = 0; jj < w.n && ok; ++jj) {
                    const int c0 = (w.t0 + jj) * C::BN;
#pragma unroll
                    for (int which = 0; which < 2; ++which) {  // K then V
                        const uint32_t slot = ring % C::NSLOT;
                        const uint32_t par = ((ring / C::NSLOT) & 1) ^ 1;
                        if (!mbar_wait(smem_u32(&bars->kv_empty[slot]), par, abort_flag,
                                       p.timeout_ns)) {
                            ok = false;
                            break;
                        }
                        if (ring + 1 == (uint32_t)p.withhold_kv) {  // test hook: never arrives
                            ++ring;
                            continue;
                        }
                        const uint32_t fb = smem_u32(&bars->kv_full[slot]);
                        mbar_arrive_expect_tx(fb, C::KV_BYTES);
                        const uint32_t dst = smem_u32(kv_smem + slot * C::KV_BYTES);
                        const CUtensorMap* map = which == 0 ? &tmK : &tmV;
#pragma unroll
                        for (int cb = 0; cb < C::NCB; ++cb) {
                            if constexpr (!C::PACKED)
                                tma_load_3d(dst + cb * C::CB_KV_BYTES, map, fb, cb * C::SWE, c0, w.z, pol_kv);
                            else
                                tma_load_3d(dst + cb * C::CB_KV_BYTES, map, fb, cb * C::SWE, w.z, w.y0 + c0, pol_kv);
                        }
                        ++ring;
                    }
                }
                ++uc;
            }
            if (!ok) raise_timeout(p, bars);
            // Every copy this producer issued lands before shared memory is released:
            // wait for the latest arming of each ring slot and of each Q buffer.  On
            // the normal path the consumers have waited for them too; after an abort
            // by another role (which may come after this loop ended normally) they
            // may still be in flight.  Copies end on their own, so the bound is the
            // fixed cleanup one, not the per-wait limit.
            const uint32_t armed = ring < C::NSLOT ? ring : C::NSLOT;
            for (uint32_t k = ring - armed; k < ring; ++k) {
                if (k + 1 == (uint32_t)p.withhold_kv) continue;  // never issued
                mbar_wait(smem_u32(&bars->kv_full[k % C::NSLOT]), (k / C::NSLOT) & 1,
                          nullptr, kCleanupTimeoutNs);
            }
            for (int i = 0; i < C::NQ; ++i)
                if (q_armed[i] > 0)
                    mbar_wait(smem_u32(&bars->q_full[i]), (q_armed[i] - 1) & 1, nullptr,
                              kCleanupTimeoutNs);
        }
    } else if (warp == C::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop in lock-step with warp-uniform values; one
        // elected lane issues each tcgen05 instruction.  Descriptors are built once
        // and every MMA only adds a compile-time offset, so issue keeps pace with
        // the tensor core.
        if constexpr (C::SPLIT_REGS) regs_decrease<C::REG_CONTROL>();
        constexpr uint32_t fmt = F8 ? 0u : 1u;
        // fp8: Q and K may both be E5M2 (format 1 of kind::f8f6f4); V and P stay E4M3, so
        // each MMA's two operands always share one type
        const uint32_t idesc_s = F8 ? idesc_f32acc(p.qk_fmt ? 1u : 0u, 0, C::BM, C::BN)
                                    : idesc_f32acc(fmt, 0, C::BM, C::BN);
        constexpr uint32_t idesc_o = idesc_f32acc(fmt, 1, C::BM, D);
        const uint64_t q_desc0 = sdesc_sw<C::SWZ>(smem_u32(q_smem), 16, 8 * C::SWZ);
        const uint64_t k_desc0 = sdesc_sw<C::SWZ>(smem_u32(kv_smem), 16, 8 * C::SWZ);
        const uint64_t v_desc0 = sdesc_sw<C::SWZ>(smem_u32(kv_smem), C::CB_KV_BYTES, 8 * C::SWZ);
        uint32_t ring = 0, uc = 0;
        uint32_t p_phase = 0;  // bit b: parity of the next p_full[b] completion
        bool ok = true;

        auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool r = ok && mbar_wait(smem_u32(bar), parity, abort_flag, p.timeout_ns);
            r = __all_sync(0xffffffffu, r);
            if (!r) ok = false;
            return r;
        };
        auto commit = [&](uint64_t* bar) { mma_commit_warp(smem_u32(bar)); };
        // S[sb] = Q_i K^T with K in ring slot `slot`
        auto issue_s = [&](int i, int sb, uint32_t slot) {
            const uint64_t qa = q_desc0 + (uint64_t)((i * C::Q_BYTES) >> 4);
            const uint64_t kb = k_desc0 + (uint64_t)((slot * C::KV_BYTES) >> 4);
            const uint32_t d_t = tmem + C::S_COL0 + sb * C::BN;
#pragma unroll
            for (int kk = 0; kk < D / C::K_STEP; ++kk) {
                constexpr int step_bytes = C::K_STEP * C::EB;  // along the row
                const int byte = kk * step_bytes;
                const uint32_t off_a = ((byte / C::SWZ) * C::CB_Q_BYTES + (byte % C::SWZ)) >> 4;
                const uint32_t off_b = ((byte / C::SWZ) * C::CB_KV_BYTES + (byte % C::SWZ)) >> 4;
                mma_ss_warp<F8>(d_t, qa + off_a, kb + off_b, idesc_s, kk > 0 ? 1u : 0u);
            }
        };
        // O_i (+)= P[sb] V with V in ring slot `slot` (V is MN-major: d contiguous)
        auto issue_pv = [&](int i, int sb, uint32_t slot, bool accumulate) {
            const uint64_t vb = v_desc0 + (uint64_t)((slot * C::KV_BYTES) >> 4);
            const uint32_t d_t = tmem + C::O_COL0 + i * D;
            const uint32_t a_t = tmem + C::S_COL0 + sb * C::BN;
            const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < C::BN / C::K_STEP; ++kk) {
                const uint32_t off_b = (kk * C::K_STEP * C::SWZ) >> 4;  // K_STEP key rows of SWZ bytes
                mma_ts_warp<F8>(d_t, a_t + kk * (C::K_STEP * C::EB / 4), vb + off_b, idesc_o,
                                kk > 0 ? 1u : acc0);
            }
        };

        for (int su = first_sub<C>(p); su < num_subs(p, tab) && ok; su = next_sub<C>(su, p, tab)) {
            Unit w;
            if (!unit_of<C>(su, p, w, tab)) continue;
#pragma unroll
            for (int i = 0; i < C::NQ; ++i) wait(&bars->q_full[i], uc & 1);
            tc_fence_after_sync();
            int Lr[C::NQ], Rr[C::NQ];  // per-Q-tile step ranges
#pragma unroll
            for (int i = 0; i < C::NQ; ++i) tile_steps<C>(w, i, p, Lr[i], Rr[i]);
            // step 0: S(0) for every Q tile that needs key tile 0
            {
                const uint32_t slot = ring % C::NSLOT;
                if (!wait(&bars->kv_full[slot], (ring / C::NSLOT) & 1)) break;
#pragma unroll
                for (int i = 0; i < C::NQ; ++i) {
                    if (Lr[i] != 0) continue;
                    issue_s(i, i, slot);
                    commit(&bars->s_full[i]);
                    if (Rr[i] == 1) commit(&bars->q_empty[i]);
                }
                commit(&bars->kv_empty[slot]);
                ++ring;
            }
            for (int jj = 1; jj < w.n && ok; ++jj) {
                const uint32_t slot_v = ring % C::NSLOT;         // V_{jj-1}
                const uint32_t slot_k = (ring + 1) % C::NSLOT;   // K_jj
                const uint32_t par_v = (ring / C::NSLOT) & 1;
                const uint32_t par_k = ((ring + 1) / C::NSLOT) & 1;
                if constexpr (C::NQ == 2) {
                    if (!wait(&bars->kv_full[slot_v], par_v)) break;
                    if (!wait(&bars->kv_full[slot_k], par_k)) break;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int jp = jj - 1;  // step whose P . V is due
                        if (jp >= Lr[i] && jp < Rr[i]) {
                            if (!wait(&bars->p_full[i], (p_phase >> i) & 1)) break;
                            p_phase ^= 1u << i;
                            if (jp == Lr[i] && !wait(&bars->o_empty[i], (uc & 1) ^ 1)) break;
                            tc_fence_after_sync();
                            // the s_full commit below also covers this PV; only the
                            // tile's last PV gets its own commit (for the epilogue)
                            issue_pv(i, i, slot_v, jp > Lr[i]);
                            if (jp == Rr[i] - 1) commit(&bars->pv_done[i]);
                        }
                        if (jj >= Lr[i] && jj < Rr[i]) {
                            issue_s(i, i, slot_k);
                            commit(&bars->s_full[i]);
                            if (jj == Rr[i] - 1) commit(&bars->q_empty[i]);
                        }
                    }
                } else {
                    const int sb = jj & 1, sp = (jj - 1) & 1;
                    if (!wait(&bars->kv_full[slot_k], par_k)) break;
                    issue_s(0, sb, slot_k);
                    commit(&bars->s_full[sb]);
                    if (jj == w.n - 1) commit(&bars->q_empty[0]);
                    if (!wait(&bars->kv_full[slot_v], par_v)) break;
                    if (!wait(&bars->p_full[sp], (p_phase >> sp) & 1)) break;
                    p_phase ^= 1u << sp;
                    if (jj == 1 && !wait(&bars->o_empty[0], (uc & 1) ^ 1)) break;
                    tc_fence_after_sync();
                    issue_pv(0, sp, slot_v, jj > 1);
                    commit(&bars->pv_done[0]);
                }
                if (!ok) break;
                commit(&bars->kv_empty[slot_v]);
                commit(&bars->kv_empty[slot_k]);
                ring += 2;
            }
            if (!ok) break;
            // tail: P(n-1) V_{n-1}
            {
                const uint32_t slot_v = ring % C::NSLOT;
                if (!wait(&bars->kv_full[slot_v], (ring / C::NSLOT) & 1)) break;
                const int sp = (C::NQ == 2) ? 0 : ((w.n - 1) & 1);
#pragma unroll
                for (int i = 0; i < C::NQ; ++i) {
                    const int sb = (C::NQ == 2) ? i : sp;
                    const int jp = w.n - 1;
                    if (jp < Lr[i] || jp >= Rr[i]) continue;  // this tile finished earlier
                    if (!wait(&bars->p_full[sb], (p_phase >> sb) & 1)) break;
                    p_phase ^= 1u << sb;
                    if (jp == Lr[i] && !wait(&bars->o_empty[i], (uc & 1) ^ 1)) break;
                    tc_fence_after_sync();
                    issue_pv(i, sb, slot_v, jp > Lr[i]);
                    commit(&bars->pv_done[i]);
                }
                if (!ok) break;
                commit(&bars->kv_empty[slot_v]);
                ++ring;
            }
            ++uc;
        }
        if (!ok && lane == 0) raise_timeout(p, bars);
        // Drain: every MMA this warp issued has finished before TMEM is freed (the
        // fixed cleanup bound: issued MMAs end on their own).
        commit(&bars->drain);
        mbar_wait(smem_u32(&bars->drain), 0, nullptr, kCleanupTimeoutNs);
        __syncwarp();
    } else if (warp < C::NUM_SOFTMAX_WARPS) {
        // ------------------------------------------------------------ softmax groups
        if constexpr (C::SPLIT_REGS) regs_increase<C::REG_SOFTMAX>();
        const int grp = warp >> 2;           // Q tile of this warpgroup
        const int wq = warp & 3;             // TMEM lane quarter
        const int row_in_tile = wq * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        const float NEG_INF = -__int_as_float(0x7f800000);
        uint32_t s_phase = 0, pv_phase = 0;  // per-buffer / per-tile parities
        uint32_t uc = 0;
        bool ok = true;

        auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool r = ok && mbar_wait(smem_u32(bar), parity, abort_flag, p.timeout_ns);
            r = __all_sync(0xffffffffu, r);
            if (!r) ok = false;
            return r;
        };

        for (int su = first_sub<C>(p); su < num_subs(p, tab) && ok; su = next_sub<C>(su, p, tab)) {
            Unit w;
            if (!unit_of<C>(su, p, w, tab)) continue;
            const int a = w.q0 + grp * C::BM;    // first row of this Q tile
            const int row = a + row_in_tile;     // this thread's query row
            // keys allowed for row r: [jlo(r), jhi(r)] (positions inside the sequence); both
            // bounds grow with r, so this warp's 32 rows span jlo in [lo_min, lo_max] and jhi
            // in [hi_min, hi_max], the bounds of its first and last row (warp-uniform)
            auto key_bounds = [&](int r, int& lo, int& hi) {
                lo = 0;
                hi = w.N - 1;
                if (p.causal) hi = min(hi, r);
                if (p.window > 0) {
                    lo = r - p.window;
                    if (!p.causal) hi = min(hi, r + p.window);
                }
            };
            int jlo, jhi;
            key_bounds(row, jlo, jhi);
            // fp8: O is kept in units of the current key tile's V descale: before
            // P(t) V8(t) is added, O *= alpha * dv(t-1) / dv(t).  When every V block scale
            // is a power of two (v_pow2), O is kept in units of the largest V scale seen so
            // far instead, dv_ref, and tile t's ratio dv(t) / dv_ref = 2^k (k <= 0, exact)
            // goes into P's exponent: P = e4m3(p * 2^(P8_SHIFT + k)).  O is then rescaled only
            // when the row max or dv_ref grows.
            // fp8: Q and K descales come per block of 2^qk_shift rows (64 or 128; N is a
            // multiple of 128), V's per 128-row block (one per key tile).  This thread's row
            // has one Q descale; a key tile's two 64-key halves may have different K
            // descales, so the score scale c is kept per half (equal when the block is 128).
            float dv_cur = 1.0f, cq = p.c_log2;
            const float* dk_head = p.dk;
            constexpr int QS = C::QK64 ? 6 : 7;   // log2 of the Q / K block rows
            if constexpr (F8) {
                const size_t qk_base = (size_t)w.z * (size_t)(p.N >> QS);
                cq = p.c_log2 * p.dq[qk_base + (row >> QS)];
                dk_head = p.dk + qk_base;
            }

            int L, R;  // key steps this Q tile needs
            tile_steps<C>(w, grp, p, L, R);
            float m_used = NEG_INF, l = 0.0f;
            for (int jj = L; jj < R; ++jj) {
                const int t = w.t0 + jj;
                const int c0 = t * C::BN;
                const int sb = (C::NQ == 2) ? grp : (jj & 1);
                float c = p.c_log2;      // bf16; fp8: c_lo for keys c0 .. c0+63, c_hi above
                float c_hi = c;
                float dv_ratio = 1.0f;  // fp8: factor on O before P(t) V8(t) is added
                int pshift = 0;          // fp8, v_pow2: k = log2(dv(t) / dv_ref) <= 0
                bool dv_up = false;      // fp8, v_pow2: dv_ref grew at this tile
                if constexpr (F8) {
                    const int nkb = p.N >> 7;
                    c = cq * dk_head[c0 >> QS];
                    if constexpr (C::QK64) c_hi = cq * dk_head[(c0 + 64) >> QS];
                    else c_hi = c;
                    const float dv_t = p.dv[(size_t)w.z * nkb + t];
                    if (!p.v_pow2) {
                        dv_ratio = dv_cur / dv_t;
                        dv_cur = dv_t;
                    } else if (jj == L || dv_t > dv_cur) {
                        dv_ratio = (jj == L) ? 1.0f : dv_cur / dv_t;  // O is empty on the first step
                        dv_up = jj > L;
                        dv_cur = dv_t;
                    } else {
                        // both are powers of two: the exponent difference is exact
                        pshift = (int)((__float_as_uint(dv_t) >> 23) & 0xFFu) -
                                 (int)((__float_as_uint(dv_cur) >> 23) & 0xFFu);
                        pshift = max(pshift, -100);  // P underflows to 0 long before
                    }
                }
                if (!wait_all(&bars->s_full[sb], (s_phase >> sb) & 1)) break;
                s_phase ^= 1u << sb;
                tc_fence_after_sync();

                // S row -> registers: issue every load, then one wait
                uint32_t sr[C::BN];
                const uint32_t s_addr = tmem + lane_addr + C::S_COL0 + sb * C::BN;
#pragma unroll
                for (int ch = 0; ch < C::BN / 32; ++ch) tmem_ld32p(s_addr + ch * 32, sr + ch * 32);
                tmem_wait_ld_only();
#pragma unroll
                for (int ch = 0; ch < C::BN / 32; ++ch) reg_fence32(sr + ch * 32);
                float* s = reinterpret_cast<float*>(sr);

                // mask only on tiles that cross a boundary of some row's allowed set
                const bool edge = (c0 + C::BN > w.N) || (p.causal && c0 + C::BN - 1 > a) ||
                                  (p.window > 0 &&
                                   (c0 < a + C::BM - 1 - p.window ||
                                    (!p.causal && c0 + C::BN - 1 > a + p.window)));
                if (edge) {
                    // per 32-key chunk, for this warp's rows: allowed for every row (skipped)
                    // or not; key c0 + e is allowed iff c0 + e - jlo lies in [0, jhi - jlo],
                    // and a chunk masked for every row takes an offset that fails every test
                    int lo_min, hi_min, lo_max, hi_max;
                    key_bounds(a + wq * 32, lo_min, hi_min);
                    key_bounds(a + wq * 32 + 31, lo_max, hi_max);
                    const uint32_t span = (uint32_t)(jhi - jlo);
#pragma unroll
                    for (int ch = 0; ch < C::BN / 32; ++ch) {
                        const int x0 = c0 + ch * 32, x1 = x0 + 31;
                        if (!(x0 >= lo_max && x1 <= hi_min)) {
                            const int base = (x1 < lo_min || x0 > hi_max) ? -(1 << 30) : x0 - jlo;
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if ((uint32_t)(base + e) > span) s[ch * 32 + e] = NEG_INF;
                        }
                    }
                }
                // row max: 8 independent chains of 3-input maxima, then a small tree
                // (fp8: one maximum per 64-key half, each scaled by its own c)
                float m_cand;
                if constexpr (!C::QK64) {
                    float mx[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        constexpr int PER = C::BN / 8;
                        float m = s[k];
#pragma unroll
                        for (int u2 = 1; u2 + 1 < PER; u2 += 2) m = fmax3(m, s[k + 8 * u2], s[k + 8 * u2 + 8]);
                        if constexpr (PER % 2 == 0) m = fmaxf(m, s[k + 8 * (PER - 1)]);
                        mx[k] = m;
                    }
                    const float tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                             fmaxf(mx[6], mx[7]));
                    m_cand = tmax * c;
                } else {
                    float mx[2][8];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float* sh = s + 64 * hf;
                            mx[hf][k] = fmaxf(fmax3(fmax3(sh[k], sh[k + 8], sh[k + 16]), sh[k + 24], sh[k + 32]),
                                              fmax3(sh[k + 40], sh[k + 48], sh[k + 56]));
                        }
                    float hmax[2];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
                        hmax[hf] = fmax3(fmax3(mx[hf][0], mx[hf][1], mx[hf][2]),
                                         fmax3(mx[hf][3], mx[hf][4], mx[hf][5]), fmaxf(mx[hf][6], mx[hf][7]));
                    m_cand = fmaxf(hmax[0] * c, hmax[1] * c_hi);  // c, c_hi > 0
                }
                const float m_new = fmaxf(m_used, m_cand);
                // bf16: move the max only when it grew by more than TAU; fp8: always
                const bool resc = F8 ? (m_new > m_used) : (m_cand > m_used + C::TAU);
                const float alpha = resc ? ex2(m_used - m_new) : 1.0f;  // ex2(-inf) = 0
                if (resc) {
                    l *= alpha;
                    m_used = m_new;
                }
                // P = 2^(s*c - m) (fp8: times 2^P8_SHIFT, folded into the exponent)
                const float mb = (m_used == NEG_INF) ? 0.0f : m_used;
                const float2 c2 = make_float2(c, c);
                const float2 c2_hi = C::QK64 ? make_float2(c_hi, c_hi) : c2;
                const float bias = F8 ? float(C::P8_SHIFT + pshift) - mb : -mb;
                const float2 b2 = make_float2(bias, bias);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                const uint32_t p_addr = tmem + lane_addr + C::S_COL0 + sb * C::BN;
                if constexpr (!F8) {
#pragma unroll
                    for (int ch = 0; ch < C::BN / 64; ++ch) {
                        uint32_t pk[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int i0 = ch * 64 + 2 * e;
                            const float2 x = __ffma2_rn(make_float2(s[i0], s[i0 + 1]), c2, b2);
                            const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                            acc[e & 3] = __fadd2_rn(acc[e & 3], pp);
                            pk[e] = pack_bf16x2(pp.x, pp.y);
                        }
                        tmem_st32p(p_addr + ch * 32, pk);
                    }
                } else {
#pragma unroll
                    for (int ch = 0; ch < C::BN / 128; ++ch) {
                        uint32_t pk[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int i0 = ch * 128 + 4 * e;
                            const float2 ce = (e < 16) ? c2 : c2_hi;  // key half of i0
                            const float2 x0 = __ffma2_rn(make_float2(s[i0], s[i0 + 1]), ce, b2);
                            const float2 x1 = __ffma2_rn(make_float2(s[i0 + 2], s[i0 + 3]), ce, b2);
                            const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
                            const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
                            acc[(2 * e) & 3] = __fadd2_rn(acc[(2 * e) & 3], p0);
                            acc[(2 * e + 1) & 3] = __fadd2_rn(acc[(2 * e + 1) & 3], p1);
                            pk[e] = (uint32_t)pack_e4m3x2(p0.x, p0.y) |
                                    ((uint32_t)pack_e4m3x2(p1.x, p1.y) << 16);
                        }
                        tmem_st32p(p_addr + ch * 32, pk);
                    }
                }
                const float2 a01 = __fadd2_rn(acc[0], acc[1]);
                const float2 a23 = __fadd2_rn(acc[2], acc[3]);
                float rowsum = (a01.x + a01.y) + (a23.x + a23.y);
                if constexpr (F8)   // undo the 2^(P8_SHIFT + k) of P (an exact power of two)
                    rowsum *= __uint_as_float((uint32_t)(127 - C::P8_SHIFT - pshift) << 23);
                l += rowsum;

                if (jj > L) {
                    // O must hold P(jj-1) V before it is rescaled.  With two Q tiles the
                    // s_full commit of this step was issued after PV(jj-1) of this tile,
                    // so its completion already implies that PV's; with one Q tile S(jj)
                    // runs ahead of PV(jj-1) and this group waits for it explicitly.
                    if constexpr (C::NQ == 1) {
                        if (!wait_all(&bars->pv_done[grp], (pv_phase >> grp) & 1)) break;
                        pv_phase ^= 1u << grp;
                    }
                    const bool any_resc = (F8 && !p.v_pow2) ? true : (__any_sync(0xffffffffu, resc) || dv_up);
                    if (any_resc) {
                        tc_fence_after_sync();
                        const float f = alpha * dv_ratio;
                        const float2 f2 = make_float2(f, f);
                        const uint32_t o_addr = tmem + lane_addr + C::O_COL0 + grp * D;
                        constexpr int CH = D / 32 < 4 ? D / 32 : 4;  // chunks per batch
#pragma unroll
                        for (int c0 = 0; c0 < D / 32; c0 += CH) {
                            uint32_t r[CH * 32];
#pragma unroll
                            for (int ch = 0; ch < CH; ++ch) tmem_ld32p(o_addr + (c0 + ch) * 32, r + ch * 32);
                            tmem_wait_ld_only();
#pragma unroll
                            for (int ch = 0; ch < CH; ++ch) reg_fence32(r + ch * 32);
#pragma unroll
                            for (int e = 0; e < CH * 16; ++e) {
                                const float2 v2 = __fmul2_rn(
                                    make_float2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])), f2);
                                r[2 * e] = __float_as_uint(v2.x);
                                r[2 * e + 1] = __float_as_uint(v2.y);
                            }
#pragma unroll
                            for (int ch = 0; ch < CH; ++ch) tmem_st32p(o_addr + (c0 + ch) * 32, r + ch * 32);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[sb]));
            }
            if (!ok) break;
            // epilogue: O / l -> bf16, LSE
            if (!wait_all(&bars->pv_done[grp], (pv_phase >> grp) & 1)) break;
            pv_phase ^= 1u << grp;
            tc_fence_after_sync();
            float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
            if constexpr (F8) inv_l *= dv_cur * (1.0f / float(1u << C::P8_SHIFT));
            const uint32_t o_addr = tmem + lane_addr + C::O_COL0 + grp * D;
            if (slab_staged<C>(w, a, wq)) {
                // O's row as bf16 pairs in registers, TMEM released, then the warp's 32 rows
                // leave in 64-column halves through its own 4 KB slab of the staging area
                // (row r's 16-byte chunk c at r * 128 + ((c ^ (r & 7)) * 16): the 128-byte
                // swizzle of the tensor map): lane 0 waits until its previous store has read
                // the slab, the lanes write it, lane 0 issues the TMA store
                uint32_t pk[D / 2];
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t r[32];
                    tmem_ld32(o_addr + ch * 32, r);
                    tmem_wait_ld(r);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[ch * 16 + e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l,
                                                      __uint_as_float(r[2 * e + 1]) * inv_l);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->o_empty[grp]));
                uint8_t* slab = ostage + warp * C::O_SLAB_BYTES;
#pragma unroll
                for (int hc = 0; hc < D / 64; ++hc) {
                    if (lane == 0) bulk_wait_group_read0();
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(slab + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                            make_uint4(pk[hc * 32 + 4 * c], pk[hc * 32 + 4 * c + 1], pk[hc * 32 + 4 * c + 2],
                                       pk[hc * 32 + 4 * c + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int r0 = a + wq * 32;
                        if constexpr (!C::PACKED)  // map (d, N, BH)
                            tma_store_3d(&tmO, smem_u32(slab), hc * 64, r0, w.z);
                        else                       // map (d, H, T)
                            tma_store_3d(&tmO, smem_u32(slab), hc * 64, w.z, w.y0 + r0);
                        bulk_commit_group();
                    }
                }
            } else {
                // batched: o[z][row]; packed: o[y0 + row][z] ([T, H, D])
                const size_t orow_idx = (!C::PACKED)
                                            ? (size_t)w.z * p.N + row
                                            : ((size_t)w.y0 + row) * p.H + w.z;
                __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + orow_idx * D;
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t r[32];
                    tmem_ld32(o_addr + ch * 32, r);
                    tmem_wait_ld(r);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l,
                                            __uint_as_float(r[2 * e + 1]) * inv_l);
                    if (row < w.N) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->o_empty[grp]));
            }
            if (row < w.N) {
                const float lse2 = (l > 0.0f) ? m_used + __log2f(l) : NEG_INF;
                const size_t li = (!C::PACKED) ? (size_t)w.z * p.N + row
                                                            : (size_t)w.z * p.T + w.y0 + row;
                p.lse[li] = lse2 * 0.69314718055994531f;
            }
            ++uc;
        }
        if (!ok) raise_timeout(p, bars);
        tmem_wait_st();  // an aborted step may have left a P or O store in flight
        if constexpr (C::OSTAGE) {
            if (lane == 0) bulk_wait_group0();  // this warp's O stores have landed
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ spare warps
        if constexpr (C::SPLIT_REGS) regs_decrease<C::REG_CONTROL>();
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == C::MMA_WARP) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace gb300

namespace gb300 {

// Defined once per (D, F8) instantiation in attn_fwd_inst.cu.
template <int D, bool F8>
cudaError_t launch_attn_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const CUtensorMap& tmO, const FwdParams& p, int sm_count, cudaStream_t stream);

}  // namespace gb300
