// sched.cuh -- the work order over packed variable-length sequences, shared by the forward
// and the backward kernels.
//
// "FlashAttention V3：优化框架吞吐量的关键技术实践" §1.2 asks for dynamic load balancing
// across uneven work, and §1.1 for variable sequence lengths.  Over packed sequences a
// unit of work is a pair of query (or key) tiles of one (sequence, head), and its cost
// grows with its sequence's length, so a plain round-robin over units leaves some CTAs
// with much more work than others.  Here every CTA builds the same table in shared
// memory at start: the sequences sorted by length (descending, ties by index) and, per
// sorted position, the number of pairs before it.  Pair u of the sorted list goes to
// CTA c in snake order -- round r = u / G gives pair r G + c to CTA c when r is even and
// r G + G - 1 - c when r is odd -- which deals the costliest pairs first and evens out
// the sums, while CTAs running at the same time still work on neighbouring pairs of the
// same head (shared K/V in L2).  No global state, no host synchronisation.  Up to
// kSortMaxSeqs sequences; a call with more falls back to the caller's round-robin.
#pragma once

#include <cstdint>

namespace gb300 {

constexpr int kSortMaxSeqs = 220;

struct SortTab {
    int seq[kSortMaxSeqs];      // sequence at each sorted position
    int prefix[kSortMaxSeqs];   // pairs before each sorted position (over all heads)
    int total;                  // pairs in all
};

// Sequence s spans tokens [cu[s], cu[s+1]) clamped to [0, T].
__device__ __forceinline__ void seq_span(const int* cu, int s, int T, int& a, int& b)
{
    a = min(max(__ldg(cu + s), 0), T);
    b = min(max(__ldg(cu + s + 1), a), T);
}

// Build the table (all threads of the CTA; ends with __syncthreads).  A sequence of n
// tokens holds H * ceil(ceil(n / ROWS) / 2) pairs, ROWS being the rows of one tile.
template <int ROWS>
__device__ __forceinline__ void build_sort_tab(const int* cu, int S, int T, int H, SortTab* tab)
{
    for (int i = threadIdx.x; i < S; i += blockDim.x) {  // lengths, in the prefix slots for now
        int a, b;
        seq_span(cu, i, T, a, b);
        tab->prefix[i] = b - a;
    }
    __syncthreads();
    constexpr int R = (kSortMaxSeqs + 127) / 128;
    int rank[R];
#pragma unroll
    for (int t = 0; t < R; ++t) {
        const int i = threadIdx.x + t * 128;
        rank[t] = -1;
        if (threadIdx.x < 128 && i < S) {
            const int li = tab->prefix[i];
            int r = 0;
            for (int j = 0; j < S; ++j) {
                const int lj = tab->prefix[j];
                r += (lj > li || (lj == li && j < i)) ? 1 : 0;
            }
            rank[t] = r;
        }
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < R; ++t)
        if (rank[t] >= 0) tab->seq[rank[t]] = threadIdx.x + t * 128;
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int r = 0; r < S; ++r) {
            int a, b;
            seq_span(cu, tab->seq[r], T, a, b);
            const int nt = (b - a + ROWS - 1) / ROWS;
            tab->prefix[r] = acc;
            acc += H * ((nt + 1) >> 1);
        }
        tab->total = acc;
    }
    __syncthreads();
}

// Pair `pair` of the sorted list: its sequence and its index among that sequence's pairs
// (over all heads, head-major).  Empty sequences sort last and hold no pairs, so the
// search never lands on one for pair < total.
__device__ __forceinline__ void sorted_pair(const SortTab* tab, int S, int pair, int& seq, int& rem)
{
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tab->prefix[mid] <= pair) lo = mid;
        else hi = mid - 1;
    }
    seq = tab->seq[lo];
    rem = pair - tab->prefix[lo];
}

// The first sub-unit of a pair in the next round (snake order), after sub-unit s.
__device__ __forceinline__ int snake_next_sub(int s)
{
    const int G = (int)gridDim.x;
    const int r = (s >> 1) / G + 1;
    return 2 * (r * G + ((r & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x));
}

}  // namespace gb300
