// Instantiations of the NF4-B GEMM variants.
#include "lm_gemm_nf4.cuh"
#include "lm_internal.h"

namespace lm {

template <bool B_MN, int EPI>
static cudaError_t launch_nf4_variant(const Params& p, int grid, cudaStream_t st) {
    constexpr int smem = Nf4Cfg<B_MN>::SMEM_BYTES;
    auto k = gemm_nf4_kernel<B_MN, EPI>;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    k<<<grid, kNf4Threads, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_gemm_nf4(GemmKind k, const Params& p, int grid, cudaStream_t st) {
    switch (k) {
        case G_NF4_GLU_FWD: return launch_nf4_variant<false, EPI_GLU_FWD>(p, grid, st);
        case G_NF4_STORE_K: return launch_nf4_variant<false, EPI_STORE>(p, grid, st);
        case G_NF4_GLU_BWD: return launch_nf4_variant<true, EPI_GLU_BWD>(p, grid, st);
        case G_NF4_STORE_MN: return launch_nf4_variant<true, EPI_STORE>(p, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lm
