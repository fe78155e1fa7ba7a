// One pass over an output gradient for both of its rank-r reductions ("Avoid recomputing LoRA
// B-projected gradient in fused-LoRA backward", LoRA_MLP.backward: G = dOut B feeds dA and dX,
// and dB = dOut^T (X A^T); both read the same dOut).
//
// For each job j of a launch (Z: T x C bf16, row-major):
//     Gpart[cr][t][0..rp)  = sum over the columns c of unit (rr, cr) of  Z[t][c] B[c][.]
//     Dpart[rr][c][0..rp)  = sum over the rows    t of unit (rr, cr) of  Z[t][c] P[.][t]
// with B the projection's LoRA B (C x r, row-major; columns r..rp read as zeros) and P the rank
// block of s (X A^T)^T (rp rows of a K-major rows x T array).  Summing Gpart over cr gives the row
// reduction Z B, summing Dpart over rr the column reduction Z^T (s X A^T): the two finalisation
// kernels do that in fixed order.
//
// A work unit is a rectangle of RB x CB tiles of 128 x 128 elements.  Each tile reaches shared
// memory once (two 64-column TMA boxes, 128-byte swizzle) and feeds two sets of tcgen05 MMAs
// (M = 128, N = rp, K = 16): read K-major it is the A operand of Z B (M = rows, K = columns), read
// MN-major the A operand of Z^T P (M = columns, K = rows).  B comes as it is stored: its rows are
// the K index and its r columns the N index, an MN-major operand of 16-column boxes with 32-byte
// swizzle.  The G accumulator of a row block (rp TMEM columns, two alternating) is drained after
// the unit's last column block; the CB dB accumulators (CB x rp columns, two alternating sets)
// after the unit's last row block.
//
// Roles (192 threads): warp 0 lane 0 TMA producer, warp 1 MMA issuer (the whole warp runs the
// issue loop, lane 0 issues), warps 2-5 drain TMEM to the fp32 partials.  Every wait is bounded.
// This header holds the launch parameters; the kernel is in lm_dual.cu.
#pragma once

#include "lm_gemm.cuh"

namespace lm {

constexpr int kDualMaxJobs = 3;
constexpr int kDualThreads = 192;
constexpr int kDualMaxStages = 6;
constexpr int kDualSmemBytes = 220 * 1024;  // dynamic shared memory of one CTA (one per SM)

struct DualJob {
    int32_t z_map, b_map, p_map;   // tensor maps: Z (box 64 x 128), B (box 16 x 128, 32-byte swizzle),
                                   // P (box 64 x rp)
    int32_t p_row0;                // first row of this job's rank block in P
    int32_t T, C;
    int32_t nrb, ncb;              // 128-row / 128-column blocks
    int32_t RB, CB;                // blocks per unit
    int32_t nrr, ncr;              // row ranges, column ranges
    int32_t unit_begin;
    float* gpart;                  // [ncr][T][rp]
    float* dpart;                  // [nrr][C][rp]
};

struct DualParams {  // CUtensorMap members carry their own 128-byte alignment
    CUtensorMap maps[3 * kDualMaxJobs];
    DualJob job[kDualMaxJobs];
    int32_t njobs;
    int32_t total_units;
    int32_t rp;
    int32_t stages;
    int32_t stage_bytes;           // 32 KB of Z + 512 rp bytes of B and P
    int32_t* err;
    uint64_t wait_ns;
    int32_t inject;
    int32_t kernel_id;
};

}  // namespace lm
