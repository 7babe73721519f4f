// attn_params.h -- launch parameters shared by the host launcher and the kernels.
#pragma once

#include <cstdint>

#include <cuda.h>

namespace gb300 {

// Status codes written to the device status word (same values as attn_status_t).
enum : int {
    kStatusOk = 0,
    kStatusTimeout = 5,
};

// Bound on the waits that only let work already issued finish before shared memory or
// tensor memory is released after an abort: TMA copies in flight and issued MMAs.
// Those end within microseconds, so this bound is fixed and independent of the
// per-wait limit a call sets (which a test may make very short).
constexpr unsigned long long kCleanupTimeoutNs = 2000000000ull;

struct FwdParams {
    void* o;              // bf16 [BH, N, D]
    float* lse;           // fp32 [BH, N], natural log
    const float* dq;      // fp8 path: Q descale per (head, 128-row block), else null
    const float* dk;      // fp8 path: K descale
    const float* dv;      // fp8 path: V descale
    int* status;          // device status word (timeouts)
    int BH;               // batch * heads
    int N;                // sequence length (queries = keys)
    int num_qblk;         // query blocks per head (NQ * 128 rows each)
    int num_units;        // BH * ceil(num_qblk / 2): pairs of query blocks
    int unit_walk;        // batched walk, chosen by the host: 0 whole pairs, 1 single units
                          // with a plain stride (non-causal), 2 single units in rotated
                          // rounds (windowed)
    int walk_first;       // the batched walk for the launch's grid G, set at launch: CTA c
    int walk_a;           // starts at sub-unit c * walk_first, and after s goes to s + 1
    int walk_m;           // when (s + walk_a) % walk_m == 0, else to s + 1 + walk_step
    int walk_step;        // (pairs: 2, 0, 2, 2G - 2; plain stride: 1, 1, 2^31 - 1, G - 1;
                          // rotated: 1, 1, G, G)
    int causal;           // 1: key j allowed only for j <= i
    int window;           // > 0: band of that half-width (left edge only when causal)
    float c_log2;         // softmax scale * log2(e)
    unsigned long long timeout_ns;  // bound on every mbarrier wait
    int withhold_kv;      // test hook, 0 in every normal call: k > 0 makes each CTA's
                          // producer skip its K/V load number k - 1 (neither armed nor
                          // issued), so the waits on it run out and the CTA aborts
    int qk_fmt;           // fp8 path: format of the Q and K codes, 0 E4M3, 1 E5M2 (V is E4M3)
    int v_pow2;           // fp8 path: V's block scales are powers of two (see the softmax)
    int qk_shift;         // fp8 path: log2 of the rows per Q and K scale block, 6 or 7 (V: 128)
    // Packed variable-length sequences (null cu_seqlens: the batched [BH, N, D] layout).
    // q, k, v, o are [T, H, D]; lse is [H, T]; sequence s is tokens [cu[s], cu[s+1]).
    // Units are (sequence, head, pair of query blocks) with num_qblk from max_seqlen.
    const int* cu_seqlens;
    int num_seqs;
    int H;
    int T;
};

// Grid of a forward launch on sm_count SMs (one CTA per SM): pairs, or single units under
// the single-unit walks, whichever the CTAs stride over, at most one per SM.
inline int fwd_grid(const FwdParams& p, int sm_count)
{
    const int items = p.unit_walk ? 2 * p.num_units : p.num_units;
    return items < sm_count ? items : sm_count;
}

// The batched walk's constants for a launch of `grid` CTAs: CTA c starts at sub-unit
// c * walk_first and after s goes to s + 1 when (s + walk_a) % walk_m == 0, else to
// s + 1 + walk_step (the kernel's first_sub / next_sub).
inline void set_fwd_walk(FwdParams& p, int grid)
{
    if (p.unit_walk == 0) {          // pairs: 2c, 2c + 1, 2c + 2G, 2c + 2G + 1, ...
        p.walk_first = 2, p.walk_a = 0, p.walk_m = 2, p.walk_step = 2 * grid - 2;
    } else if (p.unit_walk == 1) {   // single units, plain stride: c, c + G, ...
        p.walk_first = 1, p.walk_a = 1, p.walk_m = 0x7fffffff, p.walk_step = grid - 1;
    } else {                         // single units, rotated rounds
        p.walk_first = 1, p.walk_a = 1, p.walk_m = grid, p.walk_step = grid;
    }
}

// Backward pass (attn_bwd.cu).  Tensors [BH, N, D] bf16; lse / delta [BH, N] fp32.
struct BwdParams {
    const void* o;        // forward output
    const void* dout;     // upstream gradient dO
    const float* lse;     // forward LSE (natural log)
    float* delta;         // D_i = dO_i . O_i, written by the pre-pass
    void* dq;
    void* dk;
    void* dv;
    int* status;          // device status word (timeouts)
    int BH, N;
    int nt;               // 128-row tiles per head
    int causal, window;
    float c_log2;         // scale * log2(e)
    float scale;
    unsigned long long timeout_ns;
    int withhold_ring;    // test hook, 0 in every normal call: k > 0 makes each CTA's
                          // producer skip its ring load number k - 1, so the waits run out
    // Packed variable-length sequences (null cu_seqlens: the batched layout).  Tensors
    // are [T, H, D], lse / delta [H, T]; BH = num_seqs * H, N = max_seqlen, nt from N.
    const int* cu_seqlens;
    int num_seqs;
    int H;
    int T;
};

// Tensor maps of the backward pass: 128-row boxes for a unit's fixed tiles, 64-row
// boxes for the ring tiles of a step.
struct BwdMaps {
    CUtensorMap q, k, v, dout;
    CUtensorMap q64, k64, v64, dout64;
};

// One decoding step over a paged KV cache (decode.cu).
struct DecodeParams {
    const void* q;        // bf16 [B, H, nq, D]
    const void* kc;       // bf16 [num_pages, H, page_size, D]
    const void* vc;       // bf16 [num_pages, H, page_size, D]
    const int* page_table;  // int32 [B, max_pages]
    const int* seq_lens;  // int32 [B]
    void* o;              // bf16 [B, H, nq, D]
    float* lse;           // fp32 [B, H, nq], natural log
    float* ws;            // fp32 [B*H, splits, nq, D + 1] when splits > 1
    int B, H, nq;
    int log2_ps;          // page_size = 1 << log2_ps
    int num_pages, max_pages;
    int splits, pages_per_split;
    float c_log2;         // softmax scale * log2(e)
    int* status;          // device status word (the tensor-core kernel's bounded waits)
    unsigned long long timeout_ns;
};

struct QuantParams {
    const void* x;        // bf16 [BH, N, d]
    uint8_t* x8;          // e4m3 or e5m2 codes [BH, N, d]
    float* scales;        // fp32 [BH, ceil(N/rows)]
    int* status;          // device status word (timeouts)
    int BH, N, d;
    int rows;             // rows per block: 128, or 64 (head-dim-aware scaling at d = 64)
    int nblk;             // ceil(N / rows)
    int rotate;           // 1: Walsh-Hadamard rotation of each row before quantising
    int fmt;              // 0: E4M3 codes, scale = amax / 448; 1: E5M2, scale = amax / 57344;
                          // 2: E4M3, scale = the smallest power of two >= amax / 448
    float rot_c;          // rotation normalisation fp32(1 / sqrt(d))
    unsigned long long timeout_ns;  // bound on each wait for a block's load
    int withhold;         // test hook, 0 in every normal call: k > 0 makes each CTA skip
                          // the load of its iteration k - 1, so the wait on it runs out
};

}  // namespace gb300
