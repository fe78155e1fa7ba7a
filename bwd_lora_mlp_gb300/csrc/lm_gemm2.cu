// Instantiations of the CTA-pair GEMM variants and their cluster launch.
#include "lm_gemm2.cuh"
#include "lm_internal.h"

namespace lm {

template <bool B_MN, int EPI>
static cudaError_t launch_pair_variant(const Params& p, int max_units, cudaStream_t st) {
    constexpr int smem = Gemm2Cfg<B_MN>::SMEM_BYTES;
    auto k = gemm2_kernel<B_MN, EPI>;
    static int clusters[64] = {0};  // co-resident CTA pairs per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dev < 64 && clusters[dev] == 0) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
        if (e != cudaSuccess) return e;
        clusters[dev] = n > 0 ? n : 1;
    }
    const int ncl = std::min(max_units, dev < 64 ? clusters[dev] : 1);
    e = launch_pdl(k, dim3(2 * ncl, 1, 1), cfg.blockDim, smem, st, attr, 1, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_gemm_pair(GemmKind k, const Params& p, int max_units, cudaStream_t st) {
    switch (k) {
        case G2_GLU_FWD: return launch_pair_variant<false, EPI_GLU_FWD>(p, max_units, st);
        case G2_STORE_K: return launch_pair_variant<false, EPI_STORE>(p, max_units, st);
        case G2_GLU_BWD: return launch_pair_variant<true, EPI_GLU_BWD>(p, max_units, st);
        case G2_STORE_MN: return launch_pair_variant<true, EPI_STORE>(p, max_units, st);
        case G2_ACT_FWD: return launch_pair_variant<false, EPI_ACT_FWD>(p, max_units, st);
        case G2_ACT_BWD: return launch_pair_variant<true, EPI_ACT_BWD>(p, max_units, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lm
