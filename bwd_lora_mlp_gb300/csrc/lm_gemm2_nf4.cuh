// The CTA-pair GEMM of lm_gemm2.cuh with an NF4-packed frozen B operand decoded in the mainloop
// ("loralei" README, QLoRA section: unpacking and double-scale reconstruction fused into the
// matmul).
//
// Each CTA of the pair holds 128 A rows and half of the 256-wide B tile per 64-deep K block.  TMA
// brings the A rows and the raw NF4 codes of that B half (4 KB) into the CTA's own stage and
// completes on the CTA's own stage barrier; decode warps turn every 64-element NF4 block into a
// 128-byte swizzled bf16 row of the B tile and then report to CTA 0's decoded barrier, which
// counts both CTAs' decoders, so CTA 0's MMA thread starts a K block only when both halves of B
// and both A halves are in place.
//
// Decoding keeps everything in registers: for a block with scale amax' = fp32(q * c) the thread
// forms the 16 products bf16(fp32(code_i * amax')) (the values nf4_dequant writes), splits them
// into low-byte and high-byte tables of four registers each, and assembles every output pair of
// bf16 with byte permutes (prmt) indexed by the code nibbles, choosing between the two halves of
// each table by the nibble's top bit.  No shared-memory table is read, which keeps the shared
// memory bandwidth for the MMA operands.
//
// Roles (576 threads): warp 0 TMA producer, warp 1 MMA issuer (CTA 0), warps 2-9 decoders in two
// groups of four that take alternate K blocks (one thread per NF4 block), warps 10-17 epilogue.
#pragma once

#include "lm_gemm2.cuh"
#include "lm_nf4_table.cuh"

namespace lm {

constexpr int kPairNf4DecodeWarps = 8;
constexpr int kPairNf4Threads = 64 + 32 * kPairNf4DecodeWarps + 32 * kNumEpiWarps;

struct Gemm2Nf4Cfg {
    static constexpr int A_BYTES = kBM * kBK * 2;   // this CTA's 128 A rows
    static constexpr int B_BYTES = 128 * kBK * 2;   // this CTA's half of B, decoded (or bf16 via TMA)
    static constexpr int C_BYTES = 4096;            // raw codes of that half
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + C_BYTES;
    static constexpr int STAGES = 6;
    static constexpr int TMEM_COLS = 512;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024;
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Decode one NF4 block (32 code bytes c0, c1; element 2i in the high nibble of byte i) with
// block scale amax into a 128-byte row of the swizzled B tile at dst_row (16-byte chunk j stored
// at chunk j ^ swz).
__device__ __forceinline__ void nf4_decode_block_regs(uint4 c0, uint4 c1, float amax, bool valid, uint32_t dst_row,
                                                      int swz) {
    uint32_t T[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        T[i] = valid ? pack_bf16x2(__fmul_rn(nf4_value(2 * i), amax), __fmul_rn(nf4_value(2 * i + 1), amax)) : 0u;
    // low / high bytes of the 16 bf16 products, four per register, in code order
    const uint32_t L0 = prmt(T[0], T[1], 0x6420), L1 = prmt(T[2], T[3], 0x6420);
    const uint32_t L2 = prmt(T[4], T[5], 0x6420), L3 = prmt(T[6], T[7], 0x6420);
    const uint32_t H0 = prmt(T[0], T[1], 0x7531), H1 = prmt(T[2], T[3], 0x7531);
    const uint32_t H2 = prmt(T[4], T[5], 0x7531), H3 = prmt(T[6], T[7], 0x7531);
    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // four nibbles n0..n3 (bits 4k..4k+3 of x): n0, n1 = elements 1, 0 and n2, n3 = 3, 2
            // of this half word
            const uint32_t x = h ? (words[j] >> 16) : words[j];
            const uint32_t sel = x & 0x7777u;                       // index within a table half
            const uint32_t z = prmt(x, 0u, 0x1100);                  // bytes x.b0 x.b0 x.b1 x.b1
            const uint32_t y = ((z << 4) & 0x00800080u) | (z & ~0x00800080u);  // bit 7 of byte k = bit 3 of n_k
            const uint32_t m = prmt(y, y, 0xBA98);                   // 0xFF where n_k >= 8
            const uint32_t lw = (prmt(L2, L3, sel) & m) | (prmt(L0, L1, sel) & ~m);
            const uint32_t hw = (prmt(H2, H3, sel) & m) | (prmt(H0, H1, sel) & ~m);
            o[2 * h] = prmt(lw, hw, 0x4051);      // bf16 of n1 (low half), n0 (high half)
            o[2 * h + 1] = prmt(lw, hw, 0x6273);  // bf16 of n3, n2
        }
        const uint32_t addr = dst_row + ((uint32_t)(j ^ swz) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                     "r"(o[3])
                     : "memory");
    }
}

template <bool B_MN, int EPI>
__global__ void __launch_bounds__(kPairNf4Threads, 1) gemm2_nf4_kernel(const __grid_constant__ Params p) {
    using C = Gemm2Nf4Cfg;
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

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = (int)cluster_id_x();
    const int ncl = (int)nclusters_x();

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&bready[s]), 2 * (kPairNf4DecodeWarps / 2));
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), 2 * kNumEpiWarps);
        }
        mbar_init(smem_u32(drain), 1);
        *s_abort = 0;
        fence_mbar_init();
        for (int i = 0; i < kMaxMaps; ++i)
            if (p.map_bytes[i]) tma_prefetch_map(&p.maps[i]);
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t bready0 = map_to_rank(smem_u32(&bready[0]), 0);
    const uint32_t tempty0 = map_to_rank(smem_u32(&tempty[0]), 0);

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer (both CTAs, own stage barriers)
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = cid; ok && u < p.total_units; u += ncl) {
                const Unit U = decode_unit(p, u);
                const Prob& P = p.prob[U.pi];
                for (int si = 0; ok && si < P.nseg; ++si) {
                    const Seg& S = P.seg[si];
                    const int nkb = (S.kext + kBK - 1) / kBK;
                    const bool nf4 = S.b_nf4[0] >= 0;
                    const int bmap = (rank == 1 && S.b_map[1] >= 0) ? S.b_map[1] : S.b_map[0];
                    const int brow = U.nb * P.n_step + (int)rank * S.b_rank_off;
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
                        mbar_expect_tx(fb, C::A_BYTES + (nf4 ? (uint32_t)p.map_bytes[bmap] : (uint32_t)C::B_BYTES));
                        tma_load_2d(sA, &p.maps[S.a_map], fb, kx + S.a_xoff, U.mb * 256 + (int)rank * kBM);
                        if (nf4) {
                            if constexpr (B_MN) tma_load_2d(sC, &p.maps[bmap], fb, brow / 2, kx);
                            else tma_load_2d(sC, &p.maps[bmap], fb, kx / 2, brow);
                        } else if constexpr (B_MN) {
                            tma_load_2d(sB, &p.maps[bmap], fb, brow, kx);
                            tma_load_2d(sB + 8192, &p.maps[bmap], fb, brow + 64, kx);
                        } else {
                            tma_load_2d(sB, &p.maps[bmap], fb, kx + S.b_xoff[0], brow);
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
        if (lane == 0 && rank == 0) {  // ---------------- MMA issuer (CTA 0 only)
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t aphase = 0;
            bool ok = true;
            for (int u = cid; ok && u < p.total_units; u += ncl) {
                const Unit U = decode_unit(p, u);
                const Prob& P = p.prob[U.pi];
                if (!mbar_wait(smem_u32(&tempty[acc]), aphase ^ 1u, s_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + acc * 256;
                const uint32_t idesc = make_idesc_bf16(256, P.bn, false, B_MN);
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
                            const uint64_t ad = make_sdesc_sw128(sA + ks * 32, 16, 1024);
                            const uint64_t bd = B_MN ? make_sdesc_sw128(sB + ks * 2048, 8192, 1024)
                                                     : make_sdesc_sw128(sB + ks * 32, 16, 1024);
                            umma_bf16_pair(d0, ad, bd, idesc, accum);
                            accum = 1;
                        }
                        umma_commit_pair(smem_u32(&empty[stage]), 0x3);
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                umma_commit_pair(smem_u32(&tfull[acc]), 0x3);
                acc ^= 1;
                if (acc == 0) aphase ^= 1u;
            }
            if (!ok) {
                record_error(p, kErrTimeout, 2);
                *s_abort = 1;
            }
            umma_commit_pair(smem_u32(drain), 0x1);
            volatile int never = 0;
            mbar_wait(smem_u32(drain), 0, &never);
        }
    } else if (warp < 2 + kPairNf4DecodeWarps) {  // ---------------- decoders (both CTAs)
        const int dw = warp - 2;
        const int group = dw >> 2;                 // takes K blocks with iteration parity `group`
        const int t = (dw & 3) * 32 + lane;        // 0..127: one NF4 block per stage
        int stage = 0;
        uint32_t phase = 0;
        uint32_t iter = 0;
        bool ok = true;
        for (int u = cid; ok && u < p.total_units; u += ncl) {
            const Unit U = decode_unit(p, u);
            const Prob& P = p.prob[U.pi];
            for (int si = 0; ok && si < P.nseg; ++si) {
                const Seg& S = P.seg[si];
                const int nkb = (S.kext + kBK - 1) / kBK;
                const bool nf4 = S.b_nf4[0] >= 0;
                const Nf4Src* W = nf4 ? &p.nf4[(rank == 1 && S.b_nf4[1] >= 0) ? S.b_nf4[1] : S.b_nf4[0]] : nullptr;
                const int bcol0 = U.nb * P.n_step + (int)rank * S.b_rank_off;
                for (int kb = 0; kb < nkb; ++kb, ++iter) {
                    if ((int)(iter & 1u) == group) {
                        // the block scale does not depend on the stage data: fetch it before waiting
                        bool valid = false;
                        float amax = 0.0f;
                        int64_t b = 0;
                        int kr = 0, c = 0;
                        if (nf4) {
                            if constexpr (B_MN) {
                                kr = t & 63;
                                c = t >> 6;
                                const int64_t krow = (int64_t)kb * kBK + kr;
                                const int64_t ncol = (int64_t)bcol0 + c * 64;
                                valid = krow < W->rows && ncol < W->cols;
                                b = (krow * W->cols + ncol) >> 6;
                            } else {
                                const int64_t row = (int64_t)bcol0 + t;
                                valid = row < W->rows;
                                b = row * (W->cols >> 6) + kb;
                            }
                            if (valid) amax = __fmul_rn((float)__ldg(W->absmax_q + b), __ldg(W->scale + (b >> 8)));
                        }
                        if (!mbar_wait(smem_u32(&full[stage]), phase, s_abort)) {
                            ok = false;
                            break;
                        }
                        if (nf4) {
                            uint8_t* stg = smem + stage * C::STAGE_BYTES;
                            const uint32_t sB = smem_u32(stg + C::A_BYTES);
                            const uint8_t* sC = stg + C::A_BYTES + C::B_BYTES;
                            if constexpr (B_MN) {
                                const uint4* src = reinterpret_cast<const uint4*>(sC + kr * 64 + c * 32);
                                nf4_decode_block_regs(src[0], src[1], amax, valid, sB + c * 8192 + kr * 128, kr & 7);
                            } else {
                                const uint4* src = reinterpret_cast<const uint4*>(sC + t * 32);
                                nf4_decode_block_regs(src[0], src[1], amax, valid, sB + t * 128, t & 7);
                            }
                            fence_proxy_async_smem();
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote(bready0 + stage * 8);
                    }
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (!ok && lane == 0) {
            record_error(p, kErrTimeout, 4);
            *s_abort = 1;
        }
    } else {  // ---------------- epilogue warps (both CTAs)
        const int ew = warp - 2 - kPairNf4DecodeWarps;
        const int q = warp & 3;
        const int hh = ew >> 2;
        int acc = 0;
        uint32_t aphase = 0;
        bool ok = true;
        for (int u = cid; u < p.total_units; u += ncl) {
            const Unit U = decode_unit(p, u);
            const Prob& P = p.prob[U.pi];
            if (!mbar_wait(smem_u32(&tfull[acc]), aphase, s_abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256;
            const int64_t m = (int64_t)U.mb * 256 + (int64_t)rank * kBM + q * 32 + lane;
            epilogue_tile<EPI>(P, U, tacc, hh, m, m < P.M);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(tempty0 + acc * 8);
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
    cluster_sync();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace lm
