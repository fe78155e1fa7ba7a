// Host-side declarations shared by the translation units of liblora_mlp.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lm_dual.cuh"
#include "lm_gemm.cuh"

namespace lm {

// The GEMM variants built.  One-CTA split-K kernels (BN_MAX, A major, B major, epilogue):
enum GemmKind : int {
    G_PART_KK = 4,   // 256, K, K, PARTIAL    X A^T (rank-r input projection), split-K partials
    G_PART_KMN = 5,  //  64, K, MN, PARTIAL   dOut B (rank-r output-gradient projection)
    G_PART_MNK = 6,  //  64, MN, K, PARTIAL   column reductions over T for dA / dB
    G_PART_KK64 = 7, //  64, K, K, PARTIAL    G_PART_KK for projections at most 64 wide
    // bf16 base, CTA pair (cta_group::2), 256 x 256 tiles
    G2_GLU_FWD = 11,     // K-major B, GLU_FWD
    G2_STORE_K = 12,     // K-major B, STORE
    G2_GLU_BWD = 13,     // MN-major B, GLU_BWD
    G2_STORE_MN = 14,    // MN-major B, STORE
    G2_ACT_FWD = 15,     // K-major B, ACT_FWD (non-gated activation: u and act(u))
    G2_ACT_BWD = 16,     // MN-major B, ACT_BWD (du = dh * act'(u))
    // NF4 base decoded in the mainloop, CTA pair, 512 x 256 tiles
    G2N_GLU_FWD = 21,
    G2N_STORE_K = 22,
    G2N_GLU_BWD = 23,
    G2N_STORE_MN = 24,
    G2N_ACT_FWD = 25,
    G2N_ACT_BWD = 26,
    G_NUM_KINDS = 27
};

inline bool gemm_is_pair(GemmKind k) { return k >= G2_GLU_FWD && k <= G2_ACT_BWD; }
inline bool gemm_is_pair_nf4(GemmKind k) { return k >= G2N_GLU_FWD && k <= G2N_ACT_BWD; }
// Launch at most `max_units` CTA pairs (fewer if fewer pairs fit on the device at once).
cudaError_t launch_gemm_pair(GemmKind k, const Params& p, int max_units, cudaStream_t st);
cudaError_t launch_gemm_pair_nf4(GemmKind k, const Params& p, int max_units, cudaStream_t st);

cudaError_t launch_gemm(GemmKind k, const Params& p, int grid, cudaStream_t st);
// The dual rank-r reduction (lm_dual.cuh): `grid` CTAs, one per SM.
cudaError_t launch_dual_reduce(const DualParams& p, int grid, cudaStream_t st);


// Finalisation of split-K partials of rank-r projections:
//   out[t][c] = bf16(s[c / group] * sum_ks part[ks][t][c]), also written transposed to
//   outT[c][t] (row stride ldT).
struct FinRowJob {
    const float* part;
    int64_t split_stride;
    int32_t splits;
    int32_t ncols;
    int32_t group;
    float s[3];
    uint16_t* out;
    uint16_t* outT;
    int64_t ldT;
};

// Finalisation of split-K partials of the dA / dB column reductions:
//   dB layout (transposed == 0): out[c][j] = sum_ks part[ks][c][j], j < r
//   dA layout (transposed == 1): out[j][c] = sum_ks part[ks][c][j]
struct FinColJob {
    const float* part;       // column j of the job is part[ks][c][j] (the slice of a wider partial row)
    int64_t split_stride;
    int64_t C;
    int32_t splits;
    int32_t rp;
    int32_t r;
    int32_t transposed;
    float* out;
    int32_t ldp;             // floats per partial row: rp, or nb * rp when nb projections share Z
};
constexpr int kMaxFinColJobs = 6;  // jobs of one finalisation launch
cudaError_t launch_fin_colreduce(const FinColJob* jobs, int njobs, cudaStream_t st);

cudaError_t launch_nf4_pack(const uint16_t* W, int64_t numel, uint8_t* codes, int8_t* absmax_q,
                            float* scale, cudaStream_t st);
cudaError_t launch_nf4_dequant(const uint8_t* codes, const int8_t* absmax_q, const float* scale,
                               int64_t numel, bool bf16_out, void* out, cudaStream_t st);
// Finalisation of split tail tiles of a plain-store NF4 pair GEMM: out[m][n] = bf16(sum over parts
// in order of part[(t * splits + k) * 512 + row][col]) for the tiles tail_begin + t.
struct TailFin {
    const float* part;
    uint16_t* out;
    int64_t M, N, ld_out, out_col_step;
    int32_t ntail, splits, bn, tail_begin, tiles_m, tiles_n, group_m;
};
cudaError_t launch_tail_fin(const TailFin& f, cudaStream_t st);
// fp32 -> bf16 bits (RNE) of up to six matrices in one launch
struct CvtJob {
    const float* in;
    uint16_t* out;
    int64_t n;
};
struct CvtJobs {
    CvtJob j[6];
};
cudaError_t launch_f32_to_bf16(const CvtJobs& jobs, int njobs, cudaStream_t st);
// clusters the NF4 pair GEMM of kind k runs with on the current device
cudaError_t pair_nf4_clusters(GemmKind k, int* n);

// fp32 block scales of up to three NF4 weights in one launch, each K-block-major:
// table[kb * rows + row] = fp32(absmax_q[b] * scale[b / 256]), b = row * kblocks + kb
struct Nf4ScaleJob {
    const int8_t* absmax_q;
    const float* scale;
    int64_t rows, kblocks;
    float* table;
};
struct Nf4ScaleJobs {
    Nf4ScaleJob j[3];
};
// Independent work a row finalisation launch can carry in blocks of its own (blockIdx.y past the
// row jobs), in place of launches of their own: the block-diagonal rank-r operand [B_g 0; 0 B_u]
// (2n x 2rp, when bd_out is set) and NF4 block-scale tables (nf4_jobs of them).
struct FinSide {
    const uint16_t* bd_Bg = nullptr;
    const uint16_t* bd_Bu = nullptr;
    int64_t bd_n = 0;
    int32_t bd_r = 0, bd_rp = 0;
    uint16_t* bd_out = nullptr;
    Nf4ScaleJobs nf4{};
    int32_t nf4_jobs = 0;
};
cudaError_t launch_fin_rowproj(const FinRowJob* jobs, int njobs, int64_t T, cudaStream_t st,
                               const FinSide* side = nullptr);
void nf4_codebook_host(float* out16);
// int4 groupwise base: codes (rows * cols / 2 bytes) and (scale, zero) words sz[g * rows + row]
cudaError_t launch_int4_pack(const uint16_t* W, int64_t rows, int64_t cols, int group, uint8_t* codes,
                             uint32_t* sz, cudaStream_t st);
cudaError_t launch_int4_dequant(const uint8_t* codes, const uint32_t* sz, int64_t rows, int64_t cols, int group,
                                bool bf16_out, void* out, cudaStream_t st);
// NVFP4 weight-only base: codes (rows * cols / 2 bytes), E4M3 block scales sf (rows * cols / 16
// bytes, [cols / 64][rows][4]) and the fp32 tensor scale *gs (device)
cudaError_t launch_nvfp4_pack(const uint16_t* W, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* sf, float* gs,
                              cudaStream_t st);
cudaError_t launch_nvfp4_dequant(const uint8_t* codes, const uint8_t* sf, const float* gs, int64_t rows, int64_t cols,
                                 bool bf16_out, void* out, cudaStream_t st);

}  // namespace lm
