// Instantiations of the one-CTA split-K GEMM for the rank-r input projections (X A^T, h A^T):
// a 64-wide B stage (eight 24 KB stages) when the projection is at most 64 wide, else 256-wide.
#include "lm_internal.h"

namespace lm {

template <int BN_MAX, bool A_MN, bool B_MN, int EPI>
static cudaError_t launch_variant(const Params& p, int grid, cudaStream_t st) {
    constexpr int smem = GemmCfg<BN_MAX, A_MN, B_MN>::SMEM_BYTES;
    auto k = gemm_kernel<BN_MAX, A_MN, B_MN, EPI>;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    return launch_pdl(k, dim3(grid), dim3(kNumThreads), smem, st, nullptr, 0, p);
}

cudaError_t launch_gemm_fwd(GemmKind k, const Params& p, int grid, cudaStream_t st) {
    switch (k) {
        case G_PART_KK: return launch_variant<256, false, false, EPI_PARTIAL>(p, grid, st);
        case G_PART_KK64: return launch_variant<64, false, false, EPI_PARTIAL>(p, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lm
