// attn_fwd_inst.cu -- one (head dim, operand type) instantiation of the forward
// kernel and its launcher.  The build compiles this file once per pair with
// -DGB300_ATTN_D=<64|128|256> -DGB300_ATTN_F8=<0|1> so the instantiations build in parallel.
#include <cuda_runtime.h>

#include "attn_fwd.cuh"

#ifndef GB300_ATTN_D
#error "GB300_ATTN_D must be defined"
#endif
#ifndef GB300_ATTN_F8
#error "GB300_ATTN_F8 must be defined"
#endif

namespace gb300 {

template <int D, bool F8>
cudaError_t launch_attn_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const CUtensorMap& tmO, const FwdParams& p, int sm_count, cudaStream_t stream)
{
    using C = FwdCfg<D, F8>;
    // packed variable-length sequences run their own instantiation (bf16 only), so the
    // batched kernel carries none of their scheduling code
    auto kernel = attn_fwd_kernel<D, F8, false, false>;
    if constexpr (!F8) {
        if (p.cu_seqlens != nullptr) kernel = attn_fwd_kernel<D, F8, true, false>;
    } else {
        // 64-row Q/K scale blocks: two K descales per key tile (head-dim-aware scaling)
        if (p.qk_shift == 6) kernel = attn_fwd_kernel<D, F8, false, true>;
    }
    // The attribute is per device; setting it is cheap and idempotent.
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if constexpr (C::SPLIT_REGS) {
        // setmaxnreg.inc would wait forever if the launch pool were smaller than the split.
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, kernel);
        if (e != cudaSuccess) return e;
        if (attr.numRegs * C::NUM_THREADS < C::REG_POOL) return cudaErrorInvalidConfiguration;
    }
    const int grid = fwd_grid(p, sm_count);
    FwdParams q = p;
    set_fwd_walk(q, grid);
    kernel<<<grid, C::NUM_THREADS, C::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, tmO, q);
    return cudaGetLastError();
}

template cudaError_t launch_attn_fwd<GB300_ATTN_D, (GB300_ATTN_F8 != 0)>(
    const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const FwdParams&,
    int, cudaStream_t);

}  // namespace gb300
