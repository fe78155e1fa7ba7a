// Instantiations of the CTA-pair NF4-B GEMM variants and their cluster launch.
#include "lm_gemm2_nf4.cuh"
#include "lm_internal.h"

namespace lm {

template <bool B_MN, int EPI>
static cudaLaunchConfig_t pair_nf4_config(cudaLaunchAttribute* attr, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kPairNf4Threads, 1, 1);
    cfg.dynamicSmemBytes = Gemm2Nf4Cfg::SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// resident clusters of the variant on the current device (queried once per device)
template <bool B_MN, int EPI>
static cudaError_t pair_nf4_variant_clusters(int* out) {
    auto k = gemm2_nf4_kernel<B_MN, EPI>;
    static int clusters[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || clusters[dev] == 0) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Gemm2Nf4Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = pair_nf4_config<B_MN, EPI>(attr, nullptr);
        cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
        if (e != cudaSuccess) return e;
        n = n > 0 ? n : 1;
        if (dev < 64) clusters[dev] = n;
        *out = n;
        return cudaSuccess;
    }
    *out = clusters[dev];
    return cudaSuccess;
}

template <bool B_MN, int EPI>
static cudaError_t launch_pair_nf4_variant(const Params& p, int max_units, cudaStream_t st) {
    int n = 0;
    cudaError_t e = pair_nf4_variant_clusters<B_MN, EPI>(&n);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_nf4_config<B_MN, EPI>(attr, st);
    const int ncl = std::min(max_units, n);
    e = launch_pdl(gemm2_nf4_kernel<B_MN, EPI>, dim3(2 * ncl, 1, 1), cfg.blockDim, cfg.dynamicSmemBytes, st, attr, 1,
                   p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t pair_nf4_clusters(GemmKind k, int* n) {
    switch (k) {
        case G2N_GLU_FWD: return pair_nf4_variant_clusters<false, EPI_GLU_FWD>(n);
        case G2N_STORE_K: return pair_nf4_variant_clusters<false, EPI_STORE>(n);
        case G2N_GLU_BWD: return pair_nf4_variant_clusters<true, EPI_GLU_BWD>(n);
        case G2N_STORE_MN: return pair_nf4_variant_clusters<true, EPI_STORE>(n);
        case G2N_ACT_FWD: return pair_nf4_variant_clusters<false, EPI_ACT_FWD>(n);
        case G2N_ACT_BWD: return pair_nf4_variant_clusters<true, EPI_ACT_BWD>(n);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm_pair_nf4(GemmKind k, const Params& p, int max_units, cudaStream_t st) {
    switch (k) {
        case G2N_GLU_FWD: return launch_pair_nf4_variant<false, EPI_GLU_FWD>(p, max_units, st);
        case G2N_STORE_K: return launch_pair_nf4_variant<false, EPI_STORE>(p, max_units, st);
        case G2N_GLU_BWD: return launch_pair_nf4_variant<true, EPI_GLU_BWD>(p, max_units, st);
        case G2N_STORE_MN: return launch_pair_nf4_variant<true, EPI_STORE>(p, max_units, st);
        case G2N_ACT_FWD: return launch_pair_nf4_variant<false, EPI_ACT_FWD>(p, max_units, st);
        case G2N_ACT_BWD: return launch_pair_nf4_variant<true, EPI_ACT_BWD>(p, max_units, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lm
