// Persistent, warp-specialised tcgen05 GEMM for sm_103a with segmented K.
//
// One work unit computes a 128 x bn fp32 accumulator tile in TMEM:
//     D[m, j] = sum over segments  sum_k  A_seg[m, k] * B_seg[j, k]
// where each segment has its own TMA tensor maps.  The rank-r LoRA term of a projection is
// one more segment of the same accumulator (A = s * X A^T, B = LoRA B), so the low-rank
// product is added by extra K steps of the MMA instead of a separate matmul.
//
// Roles (320 threads):
//   warp 0 lane 0  TMA producer: fills a ring of shared-memory stages (A tile 128 x 64,
//                  B tile bn x 64, both 128-byte swizzled, K-major or MN-major).
//   warp 1         MMA issuer: tcgen05.mma kind::f16 (bf16 in, fp32 accumulate), commits
//                  each stage back to the producer and each finished tile to the epilogue.
//                  The whole warp runs the issue loop (warp-uniform operands) and lane 0
//                  issues; each stage is a fixed, unrolled four-MMA body.
//   warps 2..9     epilogue: TMEM -> registers (tcgen05.ld) -> fused epilogue -> global.
// Two TMEM accumulators alternate so the epilogue of one tile overlaps the mainloop of the
// next.  Every wait is bounded: on timeout the kernel records an error and returns.
#pragma once

#include "lm_ptx.cuh"

namespace lm {

enum : int { EPI_STORE = 0, EPI_GLU_FWD = 1, EPI_GLU_BWD = 2, EPI_PARTIAL = 3, EPI_ACT_FWD = 4, EPI_ACT_BWD = 5 };
enum : int { ACT_SWIGLU = 0, ACT_GEGLU = 1, ACT_RELU2 = 2 };

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kMaxMaps = 24;
constexpr int kMaxProbs = 6;
constexpr int kMaxSegs = 6;
constexpr int kNumEpiWarps = 8;
constexpr int kNumThreads = 64 + 32 * kNumEpiWarps;
constexpr int kErrTimeout = 8;  // == LM_ERR_TIMEOUT

// One K segment of a problem.
struct Seg {
    int32_t a_map;        // tensor map of A (K-major: box 64 x 128; MN-major: box 64 x 64)
    int32_t b_map[3];     // B tensor maps; -1 = unused.  MN-major B uses b_map[0] only.
    int32_t b_xoff[3];    // K-major B: added to the K coordinate of b_map[i]
    int32_t b_rows;       // K-major B: block i lands at smem row i * b_rows
    int32_t kext;         // K extent of the segment (elements)
    int32_t dual_split;   // > 0: K steps with k < dual_split use B block 0 and the first bn/2
                          // accumulator columns, the others B block 1 and the second half
    int32_t a_xoff;       // added to the K coordinate of A
    int32_t b_scale[2];   // packed 4-bit kernel: tensor map of the scales of the weight whose
                          // codes b_map[i] holds -- the fp32 block-scale table of an NF4 weight or
                          // the (scale, zero) words of an int4 one (-1: b_map[i] is a bf16
                          // operand loaded as is)
    int32_t b_rank_off;   // CTA-pair kernel: B rows (K-major) / columns (MN-major) CTA 1 adds
};

struct Prob {
    int32_t M, N;               // output rows; output columns (per half for GLU_FWD)
    int32_t tiles_m, tiles_n;
    int32_t splits, kb_per_split;  // split-K (single-segment problems only)
    int32_t unit_begin;
    int32_t nseg;
    int32_t bn;                 // accumulator columns per tile (multiple of 16, <= BN_MAX)
    int32_t n_step;             // B rows (K-major) / B columns (MN-major) per N tile
    int32_t out_col_step;       // output columns per N tile
    int32_t act;
    int32_t group_m;            // M tiles per raster group (units run M-fastest within a group)
    Seg seg[kMaxSegs];
    void* out0;
    void* out1;
    void* out2;
    const void* in0;
    const void* in1;
    int64_t ld_out, ld_in;      // elements
    int64_t split_stride;       // PARTIAL: elements between split slices
    // Tail splitting (NF4 pair kernel, plain-store epilogue): tiles from tail_begin on are each
    // run as tail_splits units over consecutive slices of their K-block sequence; each writes its
    // fp32 accumulator to tail_part[(tile - tail_begin) * tail_splits + part] (tile-sized
    // row-major blocks of rows x bn) and a finalisation kernel sums the parts in order.
    int32_t tail_begin, tail_splits;
    float* tail_part;
    // Packed pair kernel, GLU_BWD epilogue: tensor maps of in0 (e) and in1 (u), box 16 columns x
    // 128 rows with 32-byte swizzle, to stage them through shared memory; -1: plain global loads.
    int32_t in_map[2];
};

struct Params {  // CUtensorMap members carry their own 128-byte alignment
    CUtensorMap maps[kMaxMaps];
    uint32_t map_bytes[kMaxMaps];   // bytes one box of the map delivers
    int32_t map_w[kMaxMaps];        // inner (K or MN) extent of the map, elements
    int32_t map_group[kMaxMaps];    // scale map of a packed 4-bit weight: 0 NF4 block scales,
                                    // G > 0 int4 (scale, zero) words of groups of G elements,
                                    // -1 NVFP4 E4M3 block scales (four per 32-bit word)
    const float* map_gscale[kMaxMaps];  // NVFP4 scale map: the weight's fp32 tensor scale (device)
    Prob prob[kMaxProbs];
    float nf4_code[16];             // the NF4 values (NF4 kernel only)
    int32_t nprob;
    int32_t total_units;
    int32_t* err;
    uint64_t wait_ns;               // time limit of every pipeline wait (nanoseconds)
    int32_t inject;                 // test-only: nonzero = the producers issue no loads at all,
                                    // so every consumer wait runs out (see lm_debug_inject)
    int32_t kernel_id;              // recorded with an error: 1 split-K, 2 bf16 pair, 3 packed pair
};

template <int BN_MAX, bool A_MN, bool B_MN>
struct GemmCfg {
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = (BN_MAX < 64 ? 64 : BN_MAX) * kBK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // the narrow (rank-r wide) variants stream A through a tiny B: two CTAs per SM, two
    // independent load pipelines, the same bytes in flight per SM
    static constexpr int CTAS_PER_SM = BN_MAX <= 64 ? 2 : 1;
    static constexpr int STAGES = (196608 / CTAS_PER_SM / STAGE_BYTES) > 8 ? 8 : (196608 / CTAS_PER_SM / STAGE_BYTES);
    static constexpr int TMEM_COLS = 2 * BN_MAX < 32 ? 32 : 2 * BN_MAX;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024;
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM columns must be a power of two");
    static_assert(TMEM_COLS <= 512, "TMEM holds 512 columns");
};

struct Unit {
    int pi, mb, nb, ks;
    int tail;    // >= 0: index of a split tail tile (then ks is its part); -1 otherwise
};

// (mb, nb) of tile `t` of a problem: groups of `group_m` M tiles, M fastest within a group
__host__ __device__ inline void raster_tile(int t, int tiles_m, int tiles_n, int group_m, int& mb, int& nb) {
    const int GM = group_m > 0 ? group_m : 16;
    const int per_group = GM * tiles_n;
    const int g = t / per_group, w = t % per_group;
    const int gm = (tiles_m - g * GM) < GM ? (tiles_m - g * GM) : GM;
    mb = g * GM + w % gm;
    nb = w / gm;
}

__device__ __forceinline__ Unit decode_unit(const Params& p, int u) {
    Unit r;
    int pi = 0;
    while (pi + 1 < p.nprob && u >= p.prob[pi + 1].unit_begin) ++pi;
    const Prob& P = p.prob[pi];
    int local = u - P.unit_begin;
    r.pi = pi;
    r.tail = -1;
    if (P.tail_splits > 1 && local >= P.tail_begin) {
        const int q = local - P.tail_begin;
        r.tail = q / P.tail_splits;
        r.ks = q % P.tail_splits;
        local = P.tail_begin + r.tail;
    } else {
        r.ks = local % P.splits;
        local /= P.splits;
    }
    // rasterise in groups of group_m M tiles (M fastest): the tiles running at once share B
    // panels, and a group's A rows stay small enough to be re-read from L2 for every N column
    raster_tile(local, P.tiles_m, P.tiles_n, P.group_m, r.mb, r.nb);
    return r;
}

// K-block slice [g0, g1) of unit U over the concatenated K blocks of all its segments: all of
// them, or part U.ks of tail_splits for a split tail tile.
__device__ __forceinline__ void unit_kslice(const Prob& P, const Unit& U, int& g0, int& g1) {
    int total = 0;
    for (int si = 0; si < P.nseg; ++si) total += (P.seg[si].kext + kBK - 1) / kBK;
    if (U.tail >= 0) {
        g0 = (int)((int64_t)U.ks * total / P.tail_splits);
        g1 = (int)((int64_t)(U.ks + 1) * total / P.tail_splits);
    } else {
        g0 = 0;
        g1 = total;
    }
}

// error word: [0] status, [1] role that gave up (1 producer, 2 MMA issuer, 3 epilogue, 4 decoder,
// 5 drain of in-flight loads), [2] block, [3] kernel family (Params::kernel_id)
__device__ __forceinline__ void record_error(const Params& p, int code, int where) {
    if (p.err) {
        atomicExch(p.err, code);
        p.err[1] = where;
        p.err[2] = blockIdx.x;
        p.err[3] = p.kernel_id;
    }
}

// ---------------------------------------------------------------- activations
__device__ __forceinline__ float act_fwd(int act, float x) {
    // fast division (reciprocal times numerator, ~2 ulp), far below the bf16 rounding of the
    // outputs; for x below about -88 the denominator is inf and the quotient 0, the limit
    if (act == ACT_SWIGLU) return __fdividef(x, 1.0f + __expf(-x));
    if (act == ACT_RELU2) return x > 0.0f ? x * x : 0.0f;  // squared ReLU
    return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
}
// returns act(x) and act'(x)
__device__ __forceinline__ void act_fwd_bwd(int act, float x, float& f, float& df) {
    if (act == ACT_SWIGLU) {
        const float sg = __fdividef(1.0f, 1.0f + __expf(-x));
        f = x * sg;
        df = sg * (1.0f + x * (1.0f - sg));
    } else if (act == ACT_RELU2) {  // relu(x)^2 and 2 relu(x)
        const float rx = x > 0.0f ? x : 0.0f;
        f = rx * rx;
        df = 2.0f * rx;
    } else {
        const float cdf = 0.5f * (1.0f + erff(x * 0.70710678118654752f));
        const float pdf = 0.39894228040143268f * __expf(-0.5f * x * x);
        f = x * cdf;
        df = cdf + x * pdf;
    }
}

// ---------------------------------------------------------------- epilogues
// Columns [c_lo, c_hi) of the accumulator row this thread holds (GLU_FWD: the gate columns of
// that range and the matching up columns bn/2 further on).  PARTIAL takes every column with
// stride `c_step` starting at c_lo.
template <int EPI>
__device__ __forceinline__ void epilogue_cols(const Prob& P, const Unit& U, uint32_t tacc, int c_lo, int c_hi,
                                              int c_step, int64_t m, bool mvalid) {
    if constexpr (EPI == EPI_STORE) {
#pragma unroll 1
        for (int col = c_lo; col < c_hi; col += 32) {
            uint32_t a[16], b[16];
            tmem_ld_x16(tacc + col, a);
            tmem_ld_x16(tacc + col + 16, b);
            tmem_ld_wait32(a, b);
            const int64_t gcol = (int64_t)U.nb * P.out_col_step + col;
            if (mvalid && gcol < P.N) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    w[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
                    w[8 + i] = pack_bf16x2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1]));
                }
                uint16_t* dst = static_cast<uint16_t*>(P.out0) + m * P.ld_out + gcol;
                st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                st_global_v8(dst + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
            }
        }
    } else if constexpr (EPI == EPI_GLU_FWD) {
        // accumulator columns [0, bn/2) hold e (gate), [bn/2, bn) hold u (up) for the same
        // output columns; write e, u and h = act(e) * u, with h taken from the bf16 e and u.
        const int half = P.bn >> 1;
#pragma unroll 1
        for (int col = c_lo; col < c_hi; col += 16) {
            uint32_t g[16], u[16];
            tmem_ld_x16(tacc + col, g);
            tmem_ld_x16(tacc + half + col, u);
            tmem_ld_wait32(g, u);
            const int64_t gcol = (int64_t)U.nb * P.out_col_step + col;
            if (mvalid && gcol < P.N) {
                uint32_t eo[8], uo[8], ho[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    eo[i] = pack_bf16x2(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
                    uo[i] = pack_bf16x2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
                    const float e0 = bf16lo(eo[i]), e1 = bf16hi(eo[i]);
                    const float u0 = bf16lo(uo[i]), u1 = bf16hi(uo[i]);
                    ho[i] = pack_bf16x2(act_fwd(P.act, e0) * u0, act_fwd(P.act, e1) * u1);
                }
                const int64_t off = m * P.ld_out + gcol;
                st_global_v8(static_cast<uint16_t*>(P.out0) + off, eo[0], eo[1], eo[2], eo[3], eo[4], eo[5], eo[6], eo[7]);
                st_global_v8(static_cast<uint16_t*>(P.out1) + off, uo[0], uo[1], uo[2], uo[3], uo[4], uo[5], uo[6], uo[7]);
                st_global_v8(static_cast<uint16_t*>(P.out2) + off, ho[0], ho[1], ho[2], ho[3], ho[4], ho[5], ho[6], ho[7]);
            }
        }
    } else if constexpr (EPI == EPI_GLU_BWD) {
        // accumulator = dh; with the saved e, u:  de = dh * u * act'(e),  du = dh * act(e)
#pragma unroll 1
        for (int col = c_lo; col < c_hi; col += 16) {
            const int64_t gcol = (int64_t)U.nb * P.out_col_step + col;
            const bool ok = mvalid && gcol < P.N;
            uint32_t ev[8], uv[8];
            if (ok) {
                ld_global_nc_v8(static_cast<const uint16_t*>(P.in0) + m * P.ld_in + gcol, ev);
                ld_global_nc_v8(static_cast<const uint16_t*>(P.in1) + m * P.ld_in + gcol, uv);
            }
            uint32_t a[16];
            tmem_ld_x16(tacc + col, a);
            tmem_ld_wait16(a);
            if (ok) {
                uint32_t deo[8], duo[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float f0, df0, f1, df1;
                    const float e0 = bf16lo(ev[i]), e1 = bf16hi(ev[i]);
                    const float u0 = bf16lo(uv[i]), u1 = bf16hi(uv[i]);
                    act_fwd_bwd(P.act, e0, f0, df0);
                    act_fwd_bwd(P.act, e1, f1, df1);
                    const float h0 = __uint_as_float(a[2 * i]), h1 = __uint_as_float(a[2 * i + 1]);
                    deo[i] = pack_bf16x2(h0 * u0 * df0, h1 * u1 * df1);
                    duo[i] = pack_bf16x2(h0 * f0, h1 * f1);
                }
                const int64_t off = m * P.ld_out + gcol;
                st_global_v8(static_cast<uint16_t*>(P.out0) + off, deo[0], deo[1], deo[2], deo[3], deo[4], deo[5], deo[6],
                             deo[7]);
                st_global_v8(static_cast<uint16_t*>(P.out1) + off, duo[0], duo[1], duo[2], duo[3], duo[4], duo[5], duo[6],
                             duo[7]);
            }
        }
    } else if constexpr (EPI == EPI_ACT_FWD) {
        // non-gated activation: the accumulator is u; write u and h = act(u), h taken from the
        // bf16 u (the value the backward reads)
#pragma unroll 1
        for (int col = c_lo; col < c_hi; col += 16) {
            uint32_t a[16];
            tmem_ld_x16(tacc + col, a);
            tmem_ld_wait16(a);
            const int64_t gcol = (int64_t)U.nb * P.out_col_step + col;
            if (mvalid && gcol < P.N) {
                uint32_t uo[8], ho[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uo[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
                    ho[i] = pack_bf16x2(act_fwd(P.act, bf16lo(uo[i])), act_fwd(P.act, bf16hi(uo[i])));
                }
                const int64_t off = m * P.ld_out + gcol;
                st_global_v8(static_cast<uint16_t*>(P.out0) + off, uo[0], uo[1], uo[2], uo[3], uo[4], uo[5], uo[6], uo[7]);
                st_global_v8(static_cast<uint16_t*>(P.out1) + off, ho[0], ho[1], ho[2], ho[3], ho[4], ho[5], ho[6], ho[7]);
            }
        }
    } else if constexpr (EPI == EPI_ACT_BWD) {
        // accumulator = dh; with the saved u:  du = dh * act'(u)
#pragma unroll 1
        for (int col = c_lo; col < c_hi; col += 16) {
            const int64_t gcol = (int64_t)U.nb * P.out_col_step + col;
            const bool ok = mvalid && gcol < P.N;
            uint32_t uv[8];
            if (ok) ld_global_nc_v8(static_cast<const uint16_t*>(P.in0) + m * P.ld_in + gcol, uv);
            uint32_t a[16];
            tmem_ld_x16(tacc + col, a);
            tmem_ld_wait16(a);
            if (ok) {
                uint32_t duo[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float f0, df0, f1, df1;
                    act_fwd_bwd(P.act, bf16lo(uv[i]), f0, df0);
                    act_fwd_bwd(P.act, bf16hi(uv[i]), f1, df1);
                    duo[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * df0, __uint_as_float(a[2 * i + 1]) * df1);
                }
                st_global_v8(static_cast<uint16_t*>(P.out0) + m * P.ld_out + gcol, duo[0], duo[1], duo[2], duo[3], duo[4],
                             duo[5], duo[6], duo[7]);
            }
        }
    } else {  // EPI_PARTIAL: raw fp32 accumulator to out0[ks][m][0..bn)
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += c_step) {
            uint32_t a[16];
            tmem_ld_x16(tacc + c, a);
            tmem_ld_wait16(a);
            if (mvalid) {
                float* dst = static_cast<float*>(P.out0) + (int64_t)U.ks * P.split_stride + m * P.ld_out + c;
                st_global_v8(dst, a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7]);
                st_global_v8(dst + 8, a[8], a[9], a[10], a[11], a[12], a[13], a[14], a[15]);
            }
        }
    }
}

// The one-CTA kernel's split of a tile's columns between its two epilogue warp groups.
template <int EPI>
__device__ __forceinline__ void epilogue_tile(const Prob& P, const Unit& U, uint32_t tacc, int hh, int64_t m,
                                              bool mvalid) {
    const int half = P.bn >> 1;
    if constexpr (EPI == EPI_GLU_FWD) {
        const int per = half >> 1;
        epilogue_cols<EPI>(P, U, tacc, hh * per, hh * per + per, 16, m, mvalid);
    } else if constexpr (EPI == EPI_PARTIAL) {
        epilogue_cols<EPI>(P, U, tacc, hh * 16, P.bn, 32, m, mvalid);
    } else {
        epilogue_cols<EPI>(P, U, tacc, hh * half, hh * half + half, 0, m, mvalid);
    }
}

// ---------------------------------------------------------------- the kernel
template <int BN_MAX, bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(kNumThreads, BN_MAX <= 64 ? 2 : 1) gemm_kernel(const __grid_constant__ Params p) {
    using C = GemmCfg<BN_MAX, A_MN, B_MN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    griddep_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), kNumEpiWarps);
        }
        mbar_init(smem_u32(drain), 1);
        *s_abort = 0;
        fence_mbar_init();
        for (int i = 0; i < kMaxMaps; ++i)
            if (p.map_bytes[i]) tma_prefetch_map(&p.maps[i]);
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();  // the previous kernel of the stream has completed: its outputs are visible
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t nfill = 0;  // stage fills issued
            bool ok = true;
            for (int u = blockIdx.x; ok && !p.inject && u < p.total_units; u += gridDim.x) {
                const Unit U = decode_unit(p, u);
                const Prob& P = p.prob[U.pi];
                for (int si = 0; ok && si < P.nseg; ++si) {
                    const Seg& S = P.seg[si];
                    const int nkb = (S.kext + kBK - 1) / kBK;
                    int kb0 = 0, kb1 = nkb;
                    if (P.splits > 1) {
                        kb0 = U.ks * P.kb_per_split;
                        kb1 = min(nkb, kb0 + P.kb_per_split);
                    }
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, s_abort, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
                        const uint32_t sB = sA + C::A_BYTES;
                        const uint32_t fb = smem_u32(&full[stage]);
                        const int kx = kb * kBK;
                        // which B loads are issued (a box entirely outside the tensor is skipped;
                        // no MMA reads the stage region it would have filled)
                        uint32_t bytes = C::A_BYTES;
                        bool use_b[3] = {false, false, false};
                        int nch = 0;
                        if constexpr (B_MN) {
                            nch = (P.bn + 63) >> 6;
                            bytes += nch * 8192u;
                        } else {
#pragma unroll
                            for (int i = 0; i < 3; ++i) {
                                const int mi = S.b_map[i];
                                if (mi >= 0) {
                                    const int x = kx + S.b_xoff[i];
                                    use_b[i] = (x + kBK > 0) && (x < p.map_w[mi]);
                                    if (use_b[i]) bytes += p.map_bytes[mi];
                                }
                            }
                        }
                        mbar_expect_tx(fb, bytes);
                        if constexpr (A_MN) {
                            tma_load_2d(sA, &p.maps[S.a_map], fb, U.mb * kBM, kx);
                            tma_load_2d(sA + 8192, &p.maps[S.a_map], fb, U.mb * kBM + 64, kx);
                        } else {
                            tma_load_2d(sA, &p.maps[S.a_map], fb, kx + S.a_xoff, U.mb * kBM);
                        }
                        if constexpr (B_MN) {
                            for (int c = 0; c < nch; ++c)
                                tma_load_2d(sB + c * 8192, &p.maps[S.b_map[0]], fb, U.nb * P.n_step + c * 64, kx);
                        } else {
#pragma unroll
                            for (int i = 0; i < 3; ++i)
                                if (use_b[i])
                                    tma_load_2d(sB + i * S.b_rows * 128, &p.maps[S.b_map[i]], fb, kx + S.b_xoff[i],
                                                U.nb * P.n_step);
                        }
                        ++nfill;
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            if (!ok) {
                record_error(p, kErrTimeout, 1);
                *s_abort = 1;
            }
            // no load of this CTA may land after it exits (another role may have given up
            // before consuming the last fills)
            if (!drain_fills(smem_u32(&full[0]), C::STAGES, nfill, p.wait_ns)) record_error(p, kErrTimeout, 5);
        }
    } else if (warp == 1) {
        {  // ---------------- MMA issuer: the whole warp, lane 0 issues
            const bool leader = lane == 0;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t aphase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x) {
                const Unit U = decode_unit(p, u);
                const Prob& P = p.prob[U.pi];
                if (!mbar_wait_warp(smem_u32(&tempty[acc]), aphase ^ 1u, s_abort, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + acc * BN_MAX;
                const uint32_t idesc = make_idesc_bf16(kBM, P.bn, A_MN, B_MN);
                const uint32_t idesc_h = make_idesc_bf16(kBM, P.bn >> 1, A_MN, B_MN);
                uint32_t accum = 0;
                for (int si = 0; ok && si < P.nseg; ++si) {
                    const Seg& S = P.seg[si];
                    const int nkb = (S.kext + kBK - 1) / kBK;
                    int kb0 = 0, kb1 = nkb;
                    if (P.splits > 1) {
                        kb0 = U.ks * P.kb_per_split;
                        kb1 = min(nkb, kb0 + P.kb_per_split);
                    }
                    const bool dual = !B_MN && S.dual_split > 0;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait_warp(smem_u32(&full[stage]), phase, s_abort, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
                        const uint32_t sB = sA + C::A_BYTES;
                        const int rem = S.kext - kb * kBK;
                        const int nsteps = rem >= kBK ? 4 : (rem + 15) >> 4;
                        // fixed four-step body; a short last K block masks its tail steps.
                        // Descriptor addresses are in 16-byte units: a K step is 32 bytes along a
                        // K-major row or 16 rows (2048 bytes) of an MN-major tile.
                        const uint64_t ad0 = A_MN ? make_sdesc_sw128(sA, 8192, 1024) : make_sdesc_sw128(sA, 16, 1024);
                        const uint64_t bd0 = B_MN ? make_sdesc_sw128(sB, 8192, 1024) : make_sdesc_sw128(sB, 16, 1024);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint64_t ad = ad0 + (uint64_t)(A_MN ? ks * 128 : ks * 2);
                            const bool go = leader && ks < nsteps;
                            const uint32_t ac = ks == 0 ? accum : 1u;
                            if (dual) {
                                const int hf = (kb * kBK + ks * 16) >= S.dual_split ? 1 : 0;
                                const uint64_t bd = bd0 + (uint64_t)((hf * (P.bn >> 1) * 128) >> 4) + (uint64_t)(ks * 2);
                                umma_bf16_if(d0 + hf * (P.bn >> 1), ad, bd, idesc_h, ac, go);
                            } else {
                                const uint64_t bd = bd0 + (uint64_t)(B_MN ? ks * 128 : ks * 2);
                                umma_bf16_if(d0, ad, bd, idesc, ac, go);
                            }
                        }
                        accum = 1;
                        umma_commit_if(smem_u32(&empty[stage]), leader);
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                umma_commit_if(smem_u32(&tfull[acc]), leader);
                acc ^= 1;
                if (acc == 0) aphase ^= 1u;
            }
            if (!ok && leader) {
                record_error(p, kErrTimeout, 2);
                *s_abort = 1;
            }
            // wait until every MMA the leader issued has finished before TMEM is released
            umma_commit_if(smem_u32(drain), leader);
            volatile int never = 0;
            mbar_wait(smem_u32(drain), 0, &never, p.wait_ns);
            __syncwarp();
        }
    } else {  // ---------------- epilogue warps
        const int ew = warp - 2;
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int hh = ew >> 2;  // which half of the tile's columns
        int acc = 0;
        uint32_t aphase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
            const Unit U = decode_unit(p, u);
            const Prob& P = p.prob[U.pi];
            if (!mbar_wait(smem_u32(&tfull[acc]), aphase, s_abort, p.wait_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN_MAX;
            const int row = q * 32 + lane;
            const int64_t m = (int64_t)U.mb * kBM + row;
            epilogue_tile<EPI>(P, U, tacc, hh, m, m < P.M);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
            acc ^= 1;
            if (acc == 0) aphase ^= 1u;
        }
        if (!ok && lane == 0) {
            record_error(p, kErrTimeout, 3);
            *s_abort = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace lm
