// tcgen05 GEMM whose B operand is an NF4-packed frozen weight, decoded inside the mainloop
// ("loralei" README, QLoRA section: unpacking and double-scale reconstruction fused into the
// matmul; NF4 with 64-element blocks and block scales double-quantised per 256 blocks).
//
// A work unit is a 256 x 128 tile: two M = 128 MMAs share each decoded B tile, so every decoded
// weight element feeds 256 output rows.  Per stage the TMA producer brings the two 128-row A
// tiles and the raw code bytes of the B tile (4 KB instead of 16 KB of bf16); eight decode warps
// turn each 64-element NF4 block into bf16 -- fp32(code * fp32(q * c)) rounded to nearest-even,
// the same values nf4_dequant writes -- and store it as one 128-byte row of the 128-byte-
// swizzled layout the MMA reads (K-major for the forward, MN-major for dh / dX), then fence the
// generic-proxy writes to the async proxy and signal the MMA warp.  Rank-r segments (bf16 LoRA
// operands) go through the same pipeline unchanged.
//
// Roles (576 threads): warp 0 TMA producer, warp 1 MMA issuer, warps 2-9 decoders (two threads
// per NF4 block, half a block each), warps 10-17 epilogue (warp w reads TMEM lane quarter w % 4
// of M half (w - 10) / 4).  The decoders fetch the block scales of the stage after the one they
// decode, so the global-load latency of the scales stays off their critical path.
#pragma once

#include "lm_gemm.cuh"

namespace lm {

constexpr int kNf4DecodeWarps = 8;
constexpr int kNf4Threads = 64 + 32 * kNf4DecodeWarps + 32 * kNumEpiWarps;

template <bool B_MN>
struct Nf4Cfg {
    static constexpr int A_BYTES = 2 * kBM * kBK * 2;   // two 128 x 64 bf16 tiles
    static constexpr int B_BYTES = 128 * kBK * 2;       // 128 x 64 bf16, decoded
    static constexpr int C_BYTES = 4096;                // raw codes of the B tile
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + C_BYTES;
    static constexpr int STAGES = 4;
    static constexpr int TMEM_COLS = 512;               // 2 buffers x 2 M halves x 128 columns
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024;
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
};

// Decode half of a 64-element NF4 block (16 code bytes at `src`: elements 32*half .. +31) into
// 16-byte chunks 4*half .. 4*half+3 of a 128-byte swizzled smem row.
__device__ __forceinline__ void nf4_decode_half(const uint8_t* src, uint32_t dst_row, int half, int swz, float amax,
                                                bool valid, const float* cb) {
    const uint4 c = *reinterpret_cast<const uint4*>(src);
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t byte = (words[j] >> (8 * k)) & 0xFFu;
            const float v0 = __fmul_rn(cb[byte >> 4], amax);
            const float v1 = __fmul_rn(cb[byte & 15u], amax);
            o[k] = valid ? pack_bf16x2(v0, v1) : 0u;
        }
        const uint32_t addr = dst_row + ((uint32_t)((half * 4 + j) ^ swz) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                     "r"(o[3])
                     : "memory");
    }
}

// Walks the (work unit, K segment, K block) sequence every role of the kernel follows.
struct StageIter {
    int u, si, kb;
    Unit U;
    __device__ __forceinline__ bool valid(const Params& p) const { return u < p.total_units; }
    __device__ __forceinline__ void settle(const Params& p, int stride) {
        // skip to the first (unit, segment, block) that exists
        while (u < p.total_units) {
            const Prob& P = p.prob[U.pi];
            if (si < P.nseg && kb < (P.seg[si].kext + kBK - 1) / kBK) return;
            if (si < P.nseg) {
                ++si;
                kb = 0;
                continue;
            }
            u += stride;
            si = 0;
            kb = 0;
            if (u < p.total_units) U = decode_unit(p, u);
        }
    }
    __device__ __forceinline__ void start(const Params& p, int first, int stride) {
        u = first;
        si = 0;
        kb = 0;
        if (u < p.total_units) U = decode_unit(p, u);
        settle(p, stride);
    }
    __device__ __forceinline__ void next(const Params& p, int stride) {
        ++kb;
        settle(p, stride);
    }
};

// Which weight, row / column and block-scale index decoder thread `row` handles at stage `it`.
template <bool B_MN>
__device__ __forceinline__ float nf4_stage_amax(const Params& p, const StageIter& it, int row, bool& valid) {
    valid = false;
    if (!it.valid(p)) return 0.0f;
    const Prob& P = p.prob[it.U.pi];
    const Seg& S = P.seg[it.si];
    if (S.b_nf4[0] < 0) return 0.0f;
    int64_t b;
    const Nf4Src* W;
    if constexpr (B_MN) {
        const int kr = row & 63, c = row >> 6;
        W = &p.nf4[S.b_nf4[0]];
        const int64_t krow = (int64_t)it.kb * kBK + kr;
        const int64_t ncol = (int64_t)it.U.nb * P.n_step + c * 64;
        valid = krow < W->rows && ncol < W->cols;
        b = (krow * W->cols + ncol) >> 6;
    } else {
        const int blk = S.b_rows > 0 ? row / S.b_rows : 0;
        const int lr = row - blk * S.b_rows;
        W = &p.nf4[S.b_nf4[blk]];
        const int64_t r = (int64_t)it.U.nb * P.n_step + lr;
        valid = r < W->rows;
        b = r * (W->cols >> 6) + it.kb;
    }
    if (!valid) return 0.0f;
    return __fmul_rn((float)__ldg(W->absmax_q + b), __ldg(W->scale + (b >> 8)));
}

template <bool B_MN, int EPI>
__global__ void __launch_bounds__(kNf4Threads, 1) gemm_nf4_kernel(const __grid_constant__ Params p) {
    using C = Nf4Cfg<B_MN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* bready = full + C::STAGES;
    uint64_t* empty = bready + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* s_code = reinterpret_cast<float*>(tmem_slot + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&bready[s]), kNf4DecodeWarps);
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
    if (threadIdx.x < 16) s_code[threadIdx.x] = p.nf4_code[threadIdx.x];
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x) {
                const Unit U = decode_unit(p, u);
                const Prob& P = p.prob[U.pi];
                for (int si = 0; ok && si < P.nseg; ++si) {
                    const Seg& S = P.seg[si];
                    const int nkb = (S.kext + kBK - 1) / kBK;
                    const bool nf4 = S.b_nf4[0] >= 0;
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, s_abort)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
                        const uint32_t sB = sA + C::A_BYTES;
                        const uint32_t sC = sB + C::B_BYTES;
                        const uint32_t fb = smem_u32(&full[stage]);
                        const int kx = kb * kBK;
                        uint32_t bytes = C::A_BYTES;
                        bool use_b[3] = {false, false, false};
                        if (nf4) {
                            for (int i = 0; i < 3; ++i)
                                if (S.b_map[i] >= 0) bytes += p.map_bytes[S.b_map[i]];
                        } else if constexpr (B_MN) {
                            bytes += 2 * 8192u;
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
                        tma_load_2d(sA, &p.maps[S.a_map], fb, kx + S.a_xoff, U.mb * 256);
                        tma_load_2d(sA + 16384, &p.maps[S.a_map], fb, kx + S.a_xoff, U.mb * 256 + 128);
                        if (nf4) {
                            if constexpr (B_MN) {
                                // codes rows = K index, 64 bytes = the tile's 128 N elements
                                tma_load_2d(sC, &p.maps[S.b_map[0]], fb, U.nb * P.n_step / 2, kx);
                            } else {
                                for (int i = 0; i < 3; ++i)
                                    if (S.b_map[i] >= 0)
                                        tma_load_2d(sC + i * S.b_rows * 32, &p.maps[S.b_map[i]], fb, kx / 2,
                                                    U.nb * P.n_step);
                            }
                        } else if constexpr (B_MN) {
                            tma_load_2d(sB, &p.maps[S.b_map[0]], fb, U.nb * P.n_step, kx);
                            tma_load_2d(sB + 8192, &p.maps[S.b_map[0]], fb, U.nb * P.n_step + 64, kx);
                        } else {
#pragma unroll
                            for (int i = 0; i < 3; ++i)
                                if (use_b[i])
                                    tma_load_2d(sB + i * S.b_rows * 128, &p.maps[S.b_map[i]], fb, kx + S.b_xoff[i],
                                                U.nb * P.n_step);
                        }
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
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t aphase = 0;
            bool ok = true;
            const uint32_t idesc128 = make_idesc_bf16(kBM, 128, false, B_MN);
            const uint32_t idesc64 = make_idesc_bf16(kBM, 64, false, B_MN);
            for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x) {
                const Unit U = decode_unit(p, u);
                const Prob& P = p.prob[U.pi];
                if (!mbar_wait(smem_u32(&tempty[acc]), aphase ^ 1u, s_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + acc * 256;
                uint32_t accum = 0;
                for (int si = 0; ok && si < P.nseg; ++si) {
                    const Seg& S = P.seg[si];
                    const int nkb = (S.kext + kBK - 1) / kBK;
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!mbar_wait(smem_u32(&bready[stage]), phase, s_abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
                        const uint32_t sB = sA + C::A_BYTES;
                        const int rem = S.kext - kb * kBK;
                        const int nsteps = rem >= kBK ? 4 : (rem + 15) >> 4;
                        for (int ks = 0; ks < nsteps; ++ks) {
                            if (!B_MN && S.dual_split > 0) {
                                const int hf = (kb * kBK + ks * 16) >= S.dual_split ? 1 : 0;
                                const uint64_t bd = make_sdesc_sw128(sB + hf * 64 * 128 + ks * 32, 16, 1024);
#pragma unroll
                                for (int h = 0; h < 2; ++h)
                                    umma_bf16(d0 + h * 128 + hf * 64,
                                              make_sdesc_sw128(sA + h * 16384 + ks * 32, 16, 1024), bd, idesc64, accum);
                            } else {
                                const uint64_t bd = B_MN ? make_sdesc_sw128(sB + ks * 2048, 8192, 1024)
                                                         : make_sdesc_sw128(sB + ks * 32, 16, 1024);
#pragma unroll
                                for (int h = 0; h < 2; ++h)
                                    umma_bf16(d0 + h * 128, make_sdesc_sw128(sA + h * 16384 + ks * 32, 16, 1024), bd,
                                              idesc128, accum);
                            }
                            accum = 1;
                        }
                        umma_commit(smem_u32(&empty[stage]));
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&tfull[acc]));
                acc ^= 1;
                if (acc == 0) aphase ^= 1u;
            }
            if (!ok) {
                record_error(p, kErrTimeout, 2);
                *s_abort = 1;
            }
            umma_commit(smem_u32(drain));
            volatile int never = 0;
            mbar_wait(smem_u32(drain), 0, &never);
        }
    } else if (warp < 2 + kNf4DecodeWarps) {  // ---------------- NF4 decoders
        const int dt = threadIdx.x - 64;   // 0..255
        const int row = dt >> 1;           // B-tile row (K-major) or (K row, N chunk) pair (MN-major)
        const int half = dt & 1;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        StageIter it;
        it.start(p, blockIdx.x, gridDim.x);
        bool valid = false;
        float amax = nf4_stage_amax<B_MN>(p, it, row, valid);
        while (ok && it.valid(p)) {
            StageIter nx = it;
            nx.next(p, gridDim.x);
            bool nvalid = false;
            const float namax = nf4_stage_amax<B_MN>(p, nx, row, nvalid);  // in flight while decoding
            if (!mbar_wait(smem_u32(&full[stage]), phase, s_abort)) {
                ok = false;
                break;
            }
            const Seg& S = p.prob[it.U.pi].seg[it.si];
            if (S.b_nf4[0] >= 0) {
                uint8_t* stg = smem + stage * C::STAGE_BYTES;
                const uint32_t sB = smem_u32(stg + C::A_BYTES);
                const uint8_t* sC = stg + C::A_BYTES + C::B_BYTES;
                if constexpr (B_MN) {
                    const int kr = row & 63, c = row >> 6;
                    nf4_decode_half(sC + kr * 64 + c * 32 + half * 16, sB + c * 8192 + kr * 128, half, kr & 7, amax,
                                    valid, s_code);
                } else {
                    nf4_decode_half(sC + row * 32 + half * 16, sB + row * 128, half, row & 7, amax, valid, s_code);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bready[stage]));
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
            it = nx;
            amax = namax;
            valid = nvalid;
        }
        if (!ok && lane == 0) {
            record_error(p, kErrTimeout, 4);
            *s_abort = 1;
        }
    } else {  // ---------------- epilogue warps
        const int ew = warp - 2 - kNf4DecodeWarps;
        const int q = warp & 3;
        const int hh = ew >> 2;  // M half
        int acc = 0;
        uint32_t aphase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
            const Unit U = decode_unit(p, u);
            const Prob& P = p.prob[U.pi];
            if (!mbar_wait(smem_u32(&tfull[acc]), aphase, s_abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256 + hh * 128;
            const int64_t m = (int64_t)U.mb * 256 + hh * 128 + q * 32 + lane;
            if constexpr (EPI == EPI_GLU_FWD)
                epilogue_cols<EPI>(P, U, tacc, 0, P.bn >> 1, 16, m, m < P.M);
            else
                epilogue_cols<EPI>(P, U, tacc, 0, P.bn, 16, m, m < P.M);
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
