// api.cu -- the C ABI: argument checks, tensor-map encoding and kernel launches.
//
// No entry point allocates device memory or synchronises (except
// attn_get_device_status, which exists to synchronise).  Tensor maps are encoded
// on the host for every call (a few microseconds) and passed by value as
// __grid_constant__ kernel parameters.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/attn.h"
#include "attn_fwd.cuh"
#include "attn_params.h"

namespace gb300 {

cudaError_t launch_quant_fp8(const QuantParams& p, int sm_count, cudaStream_t stream);
cudaError_t launch_fp8_convert(uint32_t first, size_t count, int fmt, void* codes, int sm_count,
                               cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t stream);
cudaError_t launch_decode_tc(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                             const DecodeParams& p, int d, int sm_count, cudaStream_t stream);
cudaError_t launch_bwd(const BwdMaps& m, const BwdParams& p, int d, int sm_count, cudaStream_t stream);

// One status word per device: kernels write kStatusTimeout here when they give up.
__device__ int g_device_status;

// Device-wide scratch for attn_decode_bf16_paged_noalloc, the entry point for callers
// that cannot allocate device memory when they decode: the split partials of a
// decoding step live here instead of in a caller-provided workspace.  16 MiB, held
// by every device that loads the library until the process exits.  Host code never
// passes the symbol itself to a kernel (on the host it names a host-side stand-in);
// device_info() looks up its device address once per device and caches it.  Every
// split writes all of its partials before the merge reads them, so nothing here has
// to start at zero; calls that overlap on the GPU race on it.
constexpr size_t kDecodeScratchFloats = size_t(1) << 22;
static __device__ __align__(256) float g_decode_scratch[kDecodeScratchFloats];

// A bounded wait on a barrier that no thread arrives on: exercises the timeout
// path (give up, record the status, return) without faulting or hanging.
__global__ void wait_timeout_kernel(int* status, unsigned long long timeout_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        if (!mbar_wait(smem_u32(&bar), 0, nullptr, timeout_ns)) atomicExch(status, kStatusTimeout);
    }
}

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kWaitTimeoutNs = 4000000000ull;  // 4 s per mbarrier wait

struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int* status = nullptr;
    float* decode_scratch = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device facts, looked up once with that device current.
attn_status_t device_info(DeviceInfo** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return ATTN_ERR_CUDA;
        void* scratch = nullptr;
        if (cudaGetSymbolAddress(&scratch, g_decode_scratch) != cudaSuccess) return ATTN_ERR_CUDA;
        d.sm_count = sms;
        d.status = static_cast<int*>(addr);
        d.decode_scratch = static_cast<float*>(scratch);
        d.ready = true;
    }
    if (g_encode == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return ATTN_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = &d;
    return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 3-D map over a [BH, N, d] tensor: dims (d, N, BH) innermost first, 128-byte
// swizzled boxes of (128 bytes of d) x box_rows x 1.  Rows past N read as zero.
bool encode_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, int d,
               int N, int BH, int box_rows, int swz = 128)
{
    // swz: swizzle span in bytes, 128 or (rows of exactly 64 bytes) 64
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * elem_bytes, (cuuint64_t)N * d * elem_bytes};
    cuuint32_t box[3] = {(cuuint32_t)(swz / elem_bytes), (cuuint32_t)box_rows, 1};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swz == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D map over a packed [T, H, d] tensor: dims (d, H, T) innermost first (strides
// grow outward), boxes of (128 bytes of d) x 1 head x box_rows tokens -- the same
// shared-memory layout as the batched map's boxes.  Tokens past T read as zero.
bool encode_3d_packed(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes,
                      int d, int H, int T, int box_rows)
{
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)d * elem_bytes, (cuuint64_t)H * d * elem_bytes};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes), 1, (cuuint32_t)box_rows};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// How the batched forward's CTAs walk the work: 0 complementary pairs, 1 single units
// with a plain stride, 2 single units in rotated rounds.  Pairs balance a causal mask.  Without one the units of a head cost
// the same, and single units end in fewer rounds whenever whole pairs leave part of the
// grid a round short (for example 512 pairs on 152 SMs: 4 pair rounds = 8 unit times,
// against 7 unit rounds).  With a window the units within a window of the sequence's
// ends are lighter; pairs then land on the same positions of every head round after
// round (152 is a multiple of 4 and 8), while the rotated rounds move each CTA along a
// head's units, so a window takes rotated single units unless they need more rounds.
// (Without a window the plain stride measured slightly faster than the rotated one.)  A
// window of N - 1 keys or more masks nothing beyond the causal mask (or nothing at all),
// and is walked as that mask is (for a causal one, complementary pairs balance exactly).
int single_unit_walk(int causal, int window, int N, long long pairs, int sm_count)
{
    if (window >= N - 1) window = 0;
    if (causal && window <= 0) return 0;
    const long long G = sm_count > 0 ? sm_count : 1;
    const long long pair_times = 2 * ((pairs + G - 1) / G);   // in units of one unit's time
    const long long unit_times = (2 * pairs + G - 1) / G;
    if (window > 0) return unit_times <= pair_times ? 2 : 0;
    return unit_times < pair_times ? 1 : 0;
}

template <int D>
attn_status_t run_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int* cu_seqlens, int num_seqs, int max_seqlen, int T, int H,
                             float scale, int causal, int window, cudaStream_t stream)
{
    using C = FwdCfg<D, false>;
    DeviceInfo* dev = nullptr;
    attn_status_t st = device_info(&dev);
    if (st != ATTN_OK) return st;
    const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    alignas(64) CUtensorMap mq, mk, mv, mo;
    if (!encode_3d_packed(&mq, q, dt, C::EB, D, H, T, C::BM) ||
        !encode_3d_packed(&mk, k, dt, C::EB, D, H, T, C::BN) ||
        !encode_3d_packed(&mv, v, dt, C::EB, D, H, T, C::BN) ||
        !encode_3d_packed(&mo, o, dt, 2, D, H, T, 32))  // O leaves by TMA stores of 32-row boxes
        return ATTN_ERR_CUDA;
    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.o = o;
    p.lse = lse;
    p.status = dev->status;
    p.BH = num_seqs * H;
    p.N = max_seqlen;
    p.num_qblk = (max_seqlen + C::NQ * C::BM - 1) / (C::NQ * C::BM);
    const long long units = (long long)num_seqs * H * ((p.num_qblk + 1) / 2);
    // sub-unit indices, and a walk's step past the last one (< 4 * grid), stay in int
    if (2 * units + 4LL * dev->sm_count > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    p.num_units = (int)units;
    p.causal = causal ? 1 : 0;
    p.window = window > 0 ? window : 0;
    p.c_log2 = (float)((double)scale * 1.4426950408889634);
    p.timeout_ns = kWaitTimeoutNs;
    p.cu_seqlens = cu_seqlens;
    p.num_seqs = num_seqs;
    p.H = H;
    p.T = T;
    if (launch_attn_fwd<D, false>(mq, mk, mv, mo, p, dev->sm_count, stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

template <int D, bool F8>
attn_status_t run_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                      const float* dq, const float* dk, const float* dv, int BH, int N, float scale,
                      int causal, int window, cudaStream_t stream, int qk_fmt = 0, int v_pow2 = 0,
                      unsigned long long timeout_ns = kWaitTimeoutNs, int withhold_kv = 0,
                      int qk_block = 128)
{
    using C = FwdCfg<D, F8>;
    DeviceInfo* dev = nullptr;
    attn_status_t st = device_info(&dev);
    if (st != ATTN_OK) return st;
    const CUtensorMapDataType dt =
        F8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    alignas(64) CUtensorMap mq, mk, mv, mo;
    if (!encode_3d(&mq, q, dt, C::EB, D, N, BH, C::BM, C::SWZ) ||
        !encode_3d(&mk, k, dt, C::EB, D, N, BH, C::BN, C::SWZ) ||
        !encode_3d(&mv, v, dt, C::EB, D, N, BH, C::BN, C::SWZ) ||
        // O is bf16 in both paths and leaves by TMA stores of 64-column x 32-row boxes
        !encode_3d(&mo, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, N, BH, 32, 128))
        return ATTN_ERR_CUDA;
    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.o = o;
    p.lse = lse;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.status = dev->status;
    p.BH = BH;
    p.N = N;
    p.num_qblk = (N + C::NQ * C::BM - 1) / (C::NQ * C::BM);
    const long long units = (long long)BH * ((p.num_qblk + 1) / 2);
    // sub-unit indices, and a walk's step past the last one (< 4 * grid), stay in int
    if (2 * units + 4LL * dev->sm_count > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    p.num_units = (int)units;
    p.unit_walk = single_unit_walk(causal, window, N, units, dev->sm_count);
    p.causal = causal ? 1 : 0;
    p.window = window > 0 ? window : 0;
    p.c_log2 = (float)((double)scale * 1.4426950408889634);
    p.timeout_ns = timeout_ns;
    p.withhold_kv = withhold_kv;
    p.qk_fmt = qk_fmt;
    p.v_pow2 = v_pow2;
    p.qk_shift = qk_block == 64 ? 6 : 7;
    if (launch_attn_fwd<D, F8>(mq, mk, mv, mo, p, dev->sm_count, stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status_t check_common(int B, int H, int N, float scale, long long* BH)
{
    if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    *BH = (long long)B * H;
    if (*BH > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// Split plan of a decoding step: requested > 0 is taken as is (at most max_pages).
// 0 aims at about 24 four-warp CTAs per SM -- enough loads in flight to keep HBM busy
// -- but keeps at least 512 keys per split, so the per-split start, merge and the
// combine stay small against the streaming (measured on B16 H16 L8192 and
// B1 H16 L65536 decode steps).  Returns the splits and pages per split.
void decode_plan(int BH, int max_pages, int log2_ps, int requested, int sm_count, int* splits,
                 int* pps)
{
    long long want = (24LL * sm_count + BH - 1) / BH;
    const long long keys_cap = ((long long)max_pages << log2_ps) / 512;
    if (want > keys_cap) want = keys_cap;
    if (requested > 0) want = requested;
    if (want < 1) want = 1;
    if (want > max_pages) want = max_pages;
    *pps = (int)((max_pages + want - 1) / want);
    *splits = (max_pages + *pps - 1) / *pps;
}

// The tensor-core decoding kernel (decode_tc.cu) takes steps of 2 to 8 queries at head dims
// 64 and 128 with pages of at least 8 rows (one TMA box per page); nq = 1, d = 256 and tiny
// pages stay on the CUDA-core kernel.
bool decode_uses_tc(int nq, int d, int log2_ps)
{
    return nq >= 2 && (d == 64 || d == 128) && log2_ps >= 3;
}

// Split plan of the tensor-core kernel: splits hold whole 128-key tiles; 0 aims at about
// eight (head, split) units per CTA of the persistent grid with at least two tiles each;
// requested > 0 is honoured up to whole tiles (never more splits than requested).
void decode_plan_tc(int BH, int max_pages, int log2_ps, int requested, int sm_count, int* splits,
                    int* pps)
{
    const long long tiles = (((long long)max_pages << log2_ps) + 127) / 128;
    long long want = (8LL * sm_count + BH - 1) / BH;
    if (want > (tiles + 1) / 2) want = (tiles + 1) / 2;
    if (requested > 0) want = requested;
    if (want < 1) want = 1;
    if (want > tiles) want = tiles;
    const long long tps = (tiles + want - 1) / want;                  // tiles per split
    long long pages = log2_ps >= 7 ? (tps * 128 + (1LL << log2_ps) - 1) >> log2_ps
                                   : tps << (7 - log2_ps);            // keys: a multiple of 128
    if (pages > max_pages) pages = max_pages;                          // then one split
    if (pages < 1) pages = 1;
    *pps = (int)pages;
    *splits = (int)((max_pages + pages - 1) / pages);
}

void decode_plan_any(int BH, int nq, int d, int max_pages, int log2_ps, int requested,
                     int sm_count, int* splits, int* pps)
{
    if (decode_uses_tc(nq, d, log2_ps))
        decode_plan_tc(BH, max_pages, log2_ps, requested, sm_count, splits, pps);
    else
        decode_plan(BH, max_pages, log2_ps, requested, sm_count, splits, pps);
}

int page_log2(int page_size)
{
    int lg = 0;
    while ((1 << lg) < page_size) ++lg;
    return lg;
}

size_t decode_ws_bytes(long long BH, int splits, int nq, int d)
{
    return splits > 1 ? (size_t)BH * splits * nq * (d + 1) * sizeof(float) : 0;
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" attn_status_t attn_fwd_bf16(const void* q, const void* k, const void* v, void* o,
                                       float* lse, int B, int H, int N, int d, float scale,
                                       int causal, int window, void* stream)
{
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    long long BH = 0;
    attn_status_t st = check_common(B, H, N, scale, &BH);
    if (st != ATTN_OK) return st;
    if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
        !aligned(lse, 4))
        return ATTN_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (d) {
        case 64: return run_fwd<64, false>(q, k, v, o, lse, nullptr, nullptr, nullptr, (int)BH, N, scale, causal, window, s);
        case 128: return run_fwd<128, false>(q, k, v, o, lse, nullptr, nullptr, nullptr, (int)BH, N, scale, causal, window, s);
        default: return run_fwd<256, false>(q, k, v, o, lse, nullptr, nullptr, nullptr, (int)BH, N, scale, causal, window, s);
    }
}

extern "C" attn_status_t attn_fwd_bf16_varlen(const void* q, const void* k, const void* v, void* o,
                                              float* lse, const int* cu_seqlens, int num_seqs,
                                              int max_seqlen, int total_tokens, int H, int d,
                                              float scale, int causal, int window, void* stream)
{
    if (num_seqs < 1 || H < 1 || total_tokens < 0 || max_seqlen < 0) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
    if ((long long)num_seqs * H > 0x7fffffffLL || max_seqlen > total_tokens)
        return ATTN_ERR_INVALID_ARG;
    if (total_tokens == 0 || max_seqlen == 0) return ATTN_OK;  // nothing to compute
    if (!q || !k || !v || !o || !lse || !cu_seqlens) return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
        !aligned(lse, 4) || !aligned(cu_seqlens, 4))
        return ATTN_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (d) {
        case 64: return run_fwd_varlen<64>(q, k, v, o, lse, cu_seqlens, num_seqs, max_seqlen, total_tokens, H, scale, causal, window, s);
        case 128: return run_fwd_varlen<128>(q, k, v, o, lse, cu_seqlens, num_seqs, max_seqlen, total_tokens, H, scale, causal, window, s);
        default: return run_fwd_varlen<256>(q, k, v, o, lse, cu_seqlens, num_seqs, max_seqlen, total_tokens, H, scale, causal, window, s);
    }
}

static attn_status_t fwd_fp8(const void* q8, const void* k8, const void* v8,
                             const float* descale_q, const float* descale_k,
                             const float* descale_v, void* o, float* lse, int B, int H, int N,
                             int d, float scale, int causal, int window, int qk_format,
                             int v_format, int qk_block, void* stream)
{
    if (!q8 || !k8 || !v8 || !descale_q || !descale_k || !descale_v || !o || !lse)
        return ATTN_ERR_INVALID_ARG;
    if (qk_format != ATTN_FP8_E4M3 && qk_format != ATTN_FP8_E5M2 && qk_format != ATTN_FP8_E4M3_POW2)
        return ATTN_ERR_INVALID_ARG;
    if (v_format != ATTN_FP8_E4M3 && v_format != ATTN_FP8_E4M3_POW2) return ATTN_ERR_INVALID_ARG;
    if (qk_block != 64 && qk_block != 128) return ATTN_ERR_UNSUPPORTED;
    const int qk_fmt = qk_format == ATTN_FP8_E5M2 ? 1 : 0;   // the codes' type in the QK^T MMA
    const int v_pow2 = v_format == ATTN_FP8_E4M3_POW2 ? 1 : 0;
    long long BH = 0;
    attn_status_t st = check_common(B, H, N, scale, &BH);
    if (st != ATTN_OK) return st;
    if ((d != 64 && d != 128 && d != 256) || N % 128 != 0) return ATTN_ERR_UNSUPPORTED;
    if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(v8, 16) || !aligned(o, 16) ||
        !aligned(lse, 4) || !aligned(descale_q, 4) || !aligned(descale_k, 4) ||
        !aligned(descale_v, 4))
        return ATTN_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const unsigned long long t = kWaitTimeoutNs;
    switch (d) {
        case 64: return run_fwd<64, true>(q8, k8, v8, o, lse, descale_q, descale_k, descale_v, (int)BH, N, scale, causal, window, s, qk_fmt, v_pow2, t, 0, qk_block);
        case 128: return run_fwd<128, true>(q8, k8, v8, o, lse, descale_q, descale_k, descale_v, (int)BH, N, scale, causal, window, s, qk_fmt, v_pow2, t, 0, qk_block);
        default: return run_fwd<256, true>(q8, k8, v8, o, lse, descale_q, descale_k, descale_v, (int)BH, N, scale, causal, window, s, qk_fmt, v_pow2, t, 0, qk_block);
    }
}

extern "C" attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* v8,
                                      const float* descale_q, const float* descale_k,
                                      const float* descale_v, void* o, float* lse, int B, int H,
                                      int N, int d, float scale, int causal, int window,
                                      void* stream)
{
    return fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, o, lse, B, H, N, d, scale, causal,
                   window, ATTN_FP8_E4M3, ATTN_FP8_E4M3, 128, stream);
}

extern "C" attn_status_t attn_fwd_fp8_fmt(const void* q8, const void* k8, const void* v8,
                                          const float* descale_q, const float* descale_k,
                                          const float* descale_v, void* o, float* lse, int B, int H,
                                          int N, int d, float scale, int causal, int window,
                                          int qk_format, int v_format, void* stream)
{
    return fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, o, lse, B, H, N, d, scale, causal,
                   window, qk_format, v_format, 128, stream);
}

extern "C" attn_status_t attn_fwd_fp8_blocks(const void* q8, const void* k8, const void* v8,
                                             const float* descale_q, const float* descale_k,
                                             const float* descale_v, void* o, float* lse, int B,
                                             int H, int N, int d, float scale, int causal,
                                             int window, int qk_format, int v_format,
                                             int qk_block, void* stream)
{
    return fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, o, lse, B, H, N, d, scale, causal,
                   window, qk_format, v_format, qk_block, stream);
}

extern "C" int attn_fp8_qk_block_rows(int d)
{
    if (d < 1) return 0;
    return d < 128 ? d : 128;
}

extern "C" attn_status_t attn_fwd_schedule(int B, int H, int N, int d, int causal, int window,
                                           int sm_count, int* out)
{
    if (out == nullptr || sm_count < 1) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
    const int unit_rows = d == 256 ? FwdCfg<256, false>::NQ * FwdCfg<256, false>::BM
                                   : FwdCfg<128, false>::NQ * FwdCfg<128, false>::BM;
    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.num_qblk = (N + unit_rows - 1) / unit_rows;
    const long long pairs = (long long)B * H * ((p.num_qblk + 1) / 2);
    if (2 * pairs + 4LL * sm_count > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    p.num_units = (int)pairs;
    p.unit_walk = single_unit_walk(causal, window, N, pairs, sm_count);
    const int grid = fwd_grid(p, sm_count);
    set_fwd_walk(p, grid);
    out[0] = p.unit_walk;
    out[1] = grid;
    out[2] = 2 * p.num_units;
    out[3] = p.walk_first;
    out[4] = p.walk_a;
    out[5] = p.walk_m;
    out[6] = p.walk_step;
    out[7] = p.num_qblk;
    return ATTN_OK;
}

static attn_status_t quantize(const void* x, void* x8, float* scales, int B, int H, int N, int d,
                              int block, bool rotate, void* stream, int fmt = ATTN_FP8_E4M3,
                              unsigned long long timeout_ns = kWaitTimeoutNs, int withhold = 0)
{
    if (!x || !x8 || !scales) return ATTN_ERR_INVALID_ARG;
    if (fmt != ATTN_FP8_E4M3 && fmt != ATTN_FP8_E5M2 && fmt != ATTN_FP8_E4M3_POW2)
        return ATTN_ERR_INVALID_ARG;
    if (rotate && fmt != ATTN_FP8_E4M3) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
    if ((block != 64 && block != 128) || d % 16 != 0 || d > 256) return ATTN_ERR_UNSUPPORTED;
    if (rotate && d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
    if (!aligned(x, 16) || !aligned(x8, 16) || !aligned(scales, 4)) return ATTN_ERR_MISALIGNED;
    const long long BH = (long long)B * H;
    const long long nblk = (N + block - 1) / block;
    if (BH * nblk > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    DeviceInfo* dev = nullptr;
    attn_status_t st = device_info(&dev);
    if (st != ATTN_OK) return st;
    QuantParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = x;
    p.x8 = static_cast<uint8_t*>(x8);
    p.scales = scales;
    p.status = dev->status;
    p.BH = (int)BH;
    p.N = N;
    p.d = d;
    p.nblk = (int)nblk;
    p.rows = block;
    p.rotate = rotate ? 1 : 0;
    p.rot_c = (float)(1.0 / sqrt((double)d));
    p.fmt = fmt;
    p.timeout_ns = timeout_ns;
    p.withhold = withhold;
    if (launch_quant_fp8(p, dev->sm_count, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

extern "C" attn_status_t attn_quantize_fp8_blockwise(const void* x, void* x8, float* scales, int B,
                                                     int H, int N, int d, int block, void* stream)
{
    return quantize(x, x8, scales, B, H, N, d, block, false, stream);
}

extern "C" attn_status_t attn_quantize_fp8_blockwise_fmt(const void* x, void* x8, float* scales,
                                                         int B, int H, int N, int d, int block,
                                                         int format, void* stream)
{
    return quantize(x, x8, scales, B, H, N, d, block, false, stream, format);
}

extern "C" attn_status_t attn_quantize_fp8_hadamard(const void* x, void* x8, float* scales, int B,
                                                    int H, int N, int d, int block, void* stream)
{
    return quantize(x, x8, scales, B, H, N, d, block, true, stream);
}

extern "C" const char* attn_status_string(attn_status_t status)
{
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported shape or parameter";
        case ATTN_ERR_MISALIGNED: return "misaligned pointer";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_TIMEOUT: return "kernel gave up on an internal wait";
        default: return "unknown status";
    }
}

extern "C" attn_status_t attn_get_device_status(void* stream)
{
    DeviceInfo* dev = nullptr;
    attn_status_t st = device_info(&dev);
    if (st != ATTN_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    int value = 0;
    if (cudaMemcpy(&value, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return value == 0 ? ATTN_OK : static_cast<attn_status_t>(value);
}

extern "C" attn_status_t attn_selftest_wait_timeout(unsigned long long timeout_ns, void* stream)
{
    if (timeout_ns == 0 || timeout_ns > 2000000000ull) return ATTN_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    attn_status_t st = device_info(&dev);
    if (st != ATTN_OK) return st;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->status, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

static attn_status_t bwd_batched(const void* q, const void* k, const void* v, const void* o,
                                 const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                 void* workspace, size_t workspace_bytes, int B, int H, int N,
                                 int d, float scale, int causal, int window, void* stream,
                                 unsigned long long timeout_ns, int withhold_ring);

extern "C" attn_status_t attn_selftest_fp8_convert(unsigned int first, size_t count, int format,
                                                   void* codes, void* stream)
{
    if (!codes || count == 0 || count % 8 != 0) return ATTN_ERR_INVALID_ARG;
    if (format != ATTN_FP8_E4M3 && format != ATTN_FP8_E5M2) return ATTN_ERR_INVALID_ARG;
    if ((unsigned long long)first + count > (1ull << 32)) return ATTN_ERR_INVALID_ARG;
    if (!aligned(codes, 16)) return ATTN_ERR_MISALIGNED;
    DeviceInfo* dev = nullptr;
    attn_status_t st = device_info(&dev);
    if (st != ATTN_OK) return st;
    if (launch_fp8_convert(first, count, format == ATTN_FP8_E5M2 ? 1 : 0, codes, dev->sm_count,
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

// The real kernels with one load withheld (the test hooks in their parameters) and a
// short per-wait limit: the waits on the missing load run out, the CTA aborts through
// its normal failure path and the status word reads ATTN_ERR_TIMEOUT.
static bool selftest_args_ok(int withheld, unsigned long long timeout_ns)
{
    return withheld >= 0 && withheld < 0x7ffffffe && timeout_ns > 0 && timeout_ns <= 2000000000ull;
}

extern "C" attn_status_t attn_selftest_fwd_withheld_load(const void* q, const void* k,
                                                        const void* v, void* o, float* lse, int B,
                                                        int H, int N, int d, int causal,
                                                        int withheld,
                                                        unsigned long long timeout_ns,
                                                        void* stream)
{
    if (!selftest_args_ok(withheld, timeout_ns)) return ATTN_ERR_INVALID_ARG;
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    long long BH = 0;
    attn_status_t st = check_common(B, H, N, 1.0f, &BH);
    if (st != ATTN_OK) return st;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
        !aligned(lse, 4))
        return ATTN_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const float scale = 1.0f / sqrtf((float)d);
    switch (d) {
        case 64: return run_fwd<64, false>(q, k, v, o, lse, nullptr, nullptr, nullptr, (int)BH, N, scale, causal, 0, s, 0, 0, timeout_ns, withheld + 1);
        case 128: return run_fwd<128, false>(q, k, v, o, lse, nullptr, nullptr, nullptr, (int)BH, N, scale, causal, 0, s, 0, 0, timeout_ns, withheld + 1);
        case 256: return run_fwd<256, false>(q, k, v, o, lse, nullptr, nullptr, nullptr, (int)BH, N, scale, causal, 0, s, 0, 0, timeout_ns, withheld + 1);
        default: return ATTN_ERR_UNSUPPORTED;
    }
}

extern "C" attn_status_t attn_selftest_quant_withheld_load(const void* x, void* x8, float* scales,
                                                          int B, int H, int N, int d,
                                                          int withheld,
                                                          unsigned long long timeout_ns,
                                                          void* stream)
{
    if (!selftest_args_ok(withheld, timeout_ns)) return ATTN_ERR_INVALID_ARG;
    return quantize(x, x8, scales, B, H, N, d, 128, false, stream, ATTN_FP8_E4M3, timeout_ns,
                    withheld + 1);
}

extern "C" attn_status_t attn_selftest_bwd_withheld_load(
    const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
    void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N,
    int d, int causal, int withheld, unsigned long long timeout_ns, void* stream)
{
    if (!selftest_args_ok(withheld, timeout_ns)) return ATTN_ERR_INVALID_ARG;
    return bwd_batched(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d,
                       1.0f / sqrtf((float)d), causal, 0, stream, timeout_ns, withheld + 1);
}

extern "C" size_t attn_decode_workspace_bytes(int B, int H, int nq, int d, int page_size,
                                             int max_pages, int num_splits)
{
    if (B < 1 || H < 1 || nq < 1 || d < 1 || max_pages < 1 || page_size < 1) return 0;
    DeviceInfo* dev = nullptr;
    if (device_info(&dev) != ATTN_OK) return 0;
    int splits = 1, pps = 1;
    decode_plan_any(B * H, nq, d, max_pages, page_log2(page_size), num_splits, dev->sm_count,
                    &splits, &pps);
    return decode_ws_bytes((long long)B * H, splits, nq, d);
}

static attn_status_t decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                  const int* page_table, const int* seq_lens, void* o, float* lse,
                                  int B, int H, int nq, int d, int page_size, int num_pages,
                                  int max_pages, float scale, int num_splits, void* workspace,
                                  size_t workspace_bytes, bool use_scratch, void* stream)
{
    if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !o || !lse)
        return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || nq < 1 || num_pages < 1 || max_pages < 1 || num_splits < 0)
        return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
    if (nq > 8 || (long long)B * H > 65535) return ATTN_ERR_UNSUPPORTED;
    if (page_size < 1 || page_size > 65536 || (page_size & (page_size - 1)) != 0)
        return ATTN_ERR_UNSUPPORTED;
    if ((long long)max_pages * page_size > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
        !aligned(lse, 4) || !aligned(page_table, 4) || !aligned(seq_lens, 4) ||
        (workspace && !aligned(workspace, 16)))
        return ATTN_ERR_MISALIGNED;
    DeviceInfo* dev = nullptr;
    attn_status_t st = device_info(&dev);
    if (st != ATTN_OK) return st;
    if (use_scratch) {
        workspace = dev->decode_scratch;
        workspace_bytes = kDecodeScratchFloats * sizeof(float);
    }
    const long long BH = (long long)B * H;
    const int lg = page_log2(page_size);
    const bool tc = decode_uses_tc(nq, d, lg);
    if (tc && (long long)num_pages * H > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;  // TMA rows
    int splits = 1, pps = 1;
    decode_plan_any((int)BH, nq, d, max_pages, lg, num_splits, dev->sm_count, &splits, &pps);
    if (decode_ws_bytes(BH, splits, nq, d) > (workspace ? workspace_bytes : 0)) {
        if (num_splits > 0) return ATTN_ERR_INVALID_ARG;   // asked for more than fits
        // automatic plan: fall back to as many splits as the workspace holds
        const long long per = BH * nq * (d + 1) * (long long)sizeof(float);
        const long long fit = workspace ? (long long)(workspace_bytes / per) : 1;
        decode_plan_any((int)BH, nq, d, max_pages, lg, fit > 1 ? (int)fit : 1, dev->sm_count,
                        &splits, &pps);
    }
    if (tc && BH * splits > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;   // (head, split) units
    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q;
    p.kc = k_cache;
    p.vc = v_cache;
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.o = o;
    p.lse = lse;
    p.ws = static_cast<float*>(workspace);
    p.B = B;
    p.H = H;
    p.nq = nq;
    p.log2_ps = lg;
    p.num_pages = num_pages;
    p.max_pages = max_pages;
    p.splits = splits;
    p.pages_per_split = pps;
    p.c_log2 = (float)((double)scale * 1.4426950408889634);
    p.status = dev->status;
    p.timeout_ns = kWaitTimeoutNs;
    if (tc) {
        // Q as (d, nq, B*H) with nq-row boxes; the caches as (d, page_size, pages * H) with
        // boxes of one page (or 128 rows of a larger page): a page of one head is contiguous
        alignas(64) CUtensorMap mq, mk, mv;
        const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const int rows = page_size < 128 ? page_size : 128;
        if (!encode_3d(&mq, q, dt, 2, d, nq, (int)BH, nq) ||
            !encode_3d(&mk, k_cache, dt, 2, d, page_size, num_pages * H, rows) ||
            !encode_3d(&mv, v_cache, dt, 2, d, page_size, num_pages * H, rows))
            return ATTN_ERR_CUDA;
        if (launch_decode_tc(mq, mk, mv, p, d, dev->sm_count, static_cast<cudaStream_t>(stream)) !=
            cudaSuccess)
            return ATTN_ERR_CUDA;
        return ATTN_OK;
    }
    if (launch_decode(p, d, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

extern "C" attn_status_t attn_decode_bf16_paged(const void* q, const void* k_cache,
                                               const void* v_cache, const int* page_table,
                                               const int* seq_lens, void* o, float* lse, int B,
                                               int H, int nq, int d, int page_size,
                                               int num_pages, int max_pages, float scale,
                                               int num_splits, void* workspace,
                                               size_t workspace_bytes, void* stream)
{
    return decode_paged(q, k_cache, v_cache, page_table, seq_lens, o, lse, B, H, nq, d, page_size,
                        num_pages, max_pages, scale, num_splits, workspace, workspace_bytes, false,
                        stream);
}

extern "C" attn_status_t attn_decode_bf16_paged_noalloc(const void* q, const void* k_cache,
                                                       const void* v_cache,
                                                       const int* page_table,
                                                       const int* seq_lens, void* o, float* lse,
                                                       int B, int H, int nq, int d, int page_size,
                                                       int num_pages, int max_pages, float scale,
                                                       int num_splits, void* stream)
{
    return decode_paged(q, k_cache, v_cache, page_table, seq_lens, o, lse, B, H, nq, d, page_size,
                        num_pages, max_pages, scale, num_splits, nullptr, 0, true, stream);
}

extern "C" size_t attn_bwd_workspace_bytes(int B, int H, int N)
{
    if (B < 1 || H < 1 || N < 1) return 0;
    return (size_t)B * H * N * sizeof(float);
}

extern "C" attn_status_t attn_bwd_bf16_varlen(const void* q, const void* k, const void* v,
                                             const void* o, const void* dout, const float* lse,
                                             void* dq, void* dk, void* dv, void* workspace,
                                             size_t workspace_bytes, const int* cu_seqlens,
                                             int num_seqs, int max_seqlen, int total_tokens, int H,
                                             int d, float scale, int causal, int window,
                                             void* stream)
{
    if (num_seqs < 1 || H < 1 || total_tokens < 0 || max_seqlen < 0) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if ((long long)num_seqs * H > 0x7fffffffLL || max_seqlen > total_tokens)
        return ATTN_ERR_INVALID_ARG;
    if (total_tokens == 0 || max_seqlen == 0) return ATTN_OK;  // nothing to compute
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace || !cu_seqlens)
        return ATTN_ERR_INVALID_ARG;
    if (workspace_bytes < (size_t)H * total_tokens * sizeof(float)) return ATTN_ERR_INVALID_ARG;
    const long long BH = (long long)num_seqs * H;
    const long long nt = (max_seqlen + 127) / 128;
    if (BH * 2 * ((nt + 1) / 2) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;  // sub-units fit an int
    if ((long long)total_tokens * H > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
        !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
        !aligned(lse, 4) || !aligned(workspace, 4) || !aligned(cu_seqlens, 4))
        return ATTN_ERR_MISALIGNED;
    DeviceInfo* dev = nullptr;
    attn_status_t st = device_info(&dev);
    if (st != ATTN_OK) return st;
    const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // [T, H, d] maps: 128-token boxes for a unit's fixed tiles, 64-token boxes for the ring
    alignas(64) BwdMaps maps;
    const void* src[4] = {q, k, v, dout};
    CUtensorMap* big[4] = {&maps.q, &maps.k, &maps.v, &maps.dout};
    CUtensorMap* small[4] = {&maps.q64, &maps.k64, &maps.v64, &maps.dout64};
    for (int i = 0; i < 4; ++i)
        if (!encode_3d_packed(big[i], src[i], dt, 2, d, H, total_tokens, 128) ||
            !encode_3d_packed(small[i], src[i], dt, 2, d, H, total_tokens, 64))
            return ATTN_ERR_CUDA;
    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.o = o;
    p.dout = dout;
    p.lse = lse;
    p.delta = static_cast<float*>(workspace);
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.status = dev->status;
    p.BH = (int)BH;
    p.N = max_seqlen;
    p.nt = (int)nt;
    p.causal = causal ? 1 : 0;
    p.window = window > 0 ? window : 0;
    p.c_log2 = (float)((double)scale * 1.4426950408889634);
    p.scale = scale;
    p.timeout_ns = kWaitTimeoutNs;
    p.cu_seqlens = cu_seqlens;
    p.num_seqs = num_seqs;
    p.H = H;
    p.T = total_tokens;
    if (launch_bwd(maps, p, d, dev->sm_count, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

static attn_status_t bwd_batched(const void* q, const void* k, const void* v, const void* o,
                                 const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                 void* workspace, size_t workspace_bytes, int B, int H, int N,
                                 int d, float scale, int causal, int window, void* stream,
                                 unsigned long long timeout_ns, int withhold_ring)
{
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
        return ATTN_ERR_INVALID_ARG;
    long long BH = 0;
    attn_status_t st = check_common(B, H, N, scale, &BH);
    if (st != ATTN_OK) return st;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (workspace_bytes < (size_t)BH * N * sizeof(float)) return ATTN_ERR_INVALID_ARG;
    const long long nt = (N + 127) / 128;
    if (BH * 2 * ((nt + 1) / 2) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;  // sub-units fit an int
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
        !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
        !aligned(lse, 4) || !aligned(workspace, 4))
        return ATTN_ERR_MISALIGNED;
    DeviceInfo* dev = nullptr;
    st = device_info(&dev);
    if (st != ATTN_OK) return st;
    const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // 128-row boxes for a unit's fixed tiles, 64-row boxes for the ring tiles of a step
    alignas(64) BwdMaps maps;
    const void* src[4] = {q, k, v, dout};
    CUtensorMap* big[4] = {&maps.q, &maps.k, &maps.v, &maps.dout};
    CUtensorMap* small[4] = {&maps.q64, &maps.k64, &maps.v64, &maps.dout64};
    for (int i = 0; i < 4; ++i)
        if (!encode_3d(big[i], src[i], dt, 2, d, N, (int)BH, 128) ||
            !encode_3d(small[i], src[i], dt, 2, d, N, (int)BH, 64))
            return ATTN_ERR_CUDA;
    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.o = o;
    p.dout = dout;
    p.lse = lse;
    p.delta = static_cast<float*>(workspace);
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.status = dev->status;
    p.BH = (int)BH;
    p.N = N;
    p.nt = (int)nt;
    p.causal = causal ? 1 : 0;
    p.window = window > 0 ? window : 0;
    p.c_log2 = (float)((double)scale * 1.4426950408889634);
    p.scale = scale;
    p.timeout_ns = timeout_ns;
    p.withhold_ring = withhold_ring;
    if (launch_bwd(maps, p, d, dev->sm_count, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

extern "C" attn_status_t attn_bwd_bf16(const void* q, const void* k, const void* v, const void* o,
                                      const void* dout, const float* lse, void* dq, void* dk,
                                      void* dv, void* workspace, size_t workspace_bytes, int B,
                                      int H, int N, int d, float scale, int causal, int window,
                                      void* stream)
{
    return bwd_batched(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d,
                       scale, causal, window, stream, kWaitTimeoutNs, 0);
}
