// The bf16 GEMM of lm_gemm.cuh run by a CTA pair (cluster of 2) with tcgen05 cta_group::2.
//
// A work unit is a 256 x 256 tile.  CTA r of the pair loads rows [128 r, 128 r + 128) of the A
// tile and half of the B tile (the operand rows that feed accumulator columns
// [128 r, 128 r + 128)), 32 KB per 64-deep K block instead of the one-CTA kernel's 48 KB, so
// seven stages fit.  CTA 0 issues tcgen05.mma.cta_group::2 with M = 256: the hardware reads A and
// B from both CTAs' shared memory at the same offsets and writes each CTA's 128 accumulator rows
// into that CTA's TMEM.  Both CTAs' TMA loads complete on CTA 0's stage barrier (CTA 0 expects
// the pair's bytes); MMA completion is multicast to both CTAs' stage-free and tile-ready
// barriers; each CTA's epilogue reads its own TMEM and reports to CTA 0's accumulator-free
// barrier.  Per-CTA B rows come from a per-rank tensor map (b_map[rank]) or from one map with a
// per-rank row offset (b_rank_off).
#pragma once

#include "lm_gemm.cuh"

namespace lm {

template <bool B_MN>
struct Gemm2Cfg {
    static constexpr int A_BYTES = kBM * kBK * 2;   // this CTA's 128 A rows
    static constexpr int B_BYTES = 128 * kBK * 2;   // this CTA's half of the B tile
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = 7;
    static constexpr int TMEM_COLS = 512;           // two 256-column accumulators
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024;
};

template <bool B_MN, int EPI>
__global__ void __launch_bounds__(kNumThreads, 1) gemm2_kernel(const __grid_constant__ Params p) {
    using C = Gemm2Cfg<B_MN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // stage fills issued by each CTA's producer (both written into CTA 0's copy), read by CTA 0
    // when it waits out the pair's loads still in flight before either CTA leaves
    volatile uint32_t* s_fill = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    griddep_launch_dependents();
    const uint32_t rank = cluster_ctarank();
    const int cid = (int)cluster_id_x();
    const int ncl = (int)nclusters_x();

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
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
    cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    griddep_wait();  // the previous kernel of the stream has completed: its outputs are visible
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t full0 = map_to_rank(smem_u32(&full[0]), 0);      // CTA 0's stage barriers
    const uint32_t tempty0 = map_to_rank(smem_u32(&tempty[0]), 0);  // CTA 0's accumulator-free barriers

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t nfill = 0;  // stage fills issued by this CTA
            bool ok = true;
            for (int u = cid; ok && !p.inject && u < p.total_units; u += ncl) {
                const Unit U = decode_unit(p, u);
                const Prob& P = p.prob[U.pi];
                for (int si = 0; ok && si < P.nseg; ++si) {
                    const Seg& S = P.seg[si];
                    const int nkb = (S.kext + kBK - 1) / kBK;
                    const int bmap = (rank == 1 && S.b_map[1] >= 0) ? S.b_map[1] : S.b_map[0];
                    const int brow = U.nb * P.n_step + (int)rank * S.b_rank_off;
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, s_abort, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
                        const uint32_t sB = sA + C::A_BYTES;
                        const uint32_t fb = full0 + stage * 8;
                        const int kx = kb * kBK;
                        if (rank == 0) mbar_expect_tx(smem_u32(&full[stage]), 2u * (C::A_BYTES + C::B_BYTES));
                        tma_load_2d_pair(sA, &p.maps[S.a_map], fb, kx + S.a_xoff, U.mb * 256 + (int)rank * kBM);
                        if constexpr (B_MN) {
                            tma_load_2d_pair(sB, &p.maps[bmap], fb, brow, kx);
                            tma_load_2d_pair(sB + 8192, &p.maps[bmap], fb, brow + 64, kx);
                        } else {
                            tma_load_2d_pair(sB, &p.maps[bmap], fb, kx + S.b_xoff[0], brow);
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
            st_cluster_u32(map_to_rank(smem_u32(const_cast<uint32_t*>(&s_fill[rank])), 0), nfill);
        }
    } else if (warp == 1) {
        if (rank == 0) {  // ---------------- MMA issuer (CTA 0 only): the whole warp, lane 0 issues
            const bool leader = lane == 0;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t aphase = 0;
            bool ok = true;
            for (int u = cid; ok && u < p.total_units; u += ncl) {
                const Unit U = decode_unit(p, u);
                const Prob& P = p.prob[U.pi];
                if (!mbar_wait_warp(smem_u32(&tempty[acc]), aphase ^ 1u, s_abort, p.wait_ns)) {
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
                        if (!mbar_wait_warp(smem_u32(&full[stage]), phase, s_abort, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
                        const uint32_t sB = sA + C::A_BYTES;
                        const int rem = S.kext - kb * kBK;
                        const int nsteps = rem >= kBK ? 4 : (rem + 15) >> 4;
                        // a fixed four-step body (a short last K block of a segment masks its
                        // tail steps): a loop with a run-time trip count here starves the tensor pipe
                        const uint64_t ad0 = make_sdesc_sw128(sA, 16, 1024);
                        const uint64_t bd0 = B_MN ? make_sdesc_sw128(sB, 8192, 1024) : make_sdesc_sw128(sB, 16, 1024);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            // 16 K elements = 32 bytes along a K-major row or 16 rows (2048 bytes) of an
                            // MN-major tile; the descriptor holds the address in 16-byte units
                            const uint64_t ad = ad0 + (uint64_t)(ks * 2);
                            const uint64_t bd = bd0 + (uint64_t)(B_MN ? ks * 128 : ks * 2);
                            umma_bf16_pair_if(d0, ad, bd, idesc, ks == 0 ? accum : 1u, leader && ks < nsteps);
                        }
                        accum = 1;
                        umma_commit_pair_if(smem_u32(&empty[stage]), 0x3, leader);
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                umma_commit_pair_if(smem_u32(&tfull[acc]), 0x3, leader);
                acc ^= 1;
                if (acc == 0) aphase ^= 1u;
            }
            if (!ok && leader) {
                record_error(p, kErrTimeout, 2);
                *s_abort = 1;
            }
            umma_commit_pair_if(smem_u32(drain), 0x1, leader);
            volatile int never = 0;
            mbar_wait(smem_u32(drain), 0, &never, p.wait_ns);
            __syncwarp();
        }
    } else {  // ---------------- epilogue warps (both CTAs)
        const int ew = warp - 2;
        const int q = warp & 3;
        const int hh = ew >> 2;
        int acc = 0;
        uint32_t aphase = 0;
        bool ok = true;
        for (int u = cid; u < p.total_units; u += ncl) {
            const Unit U = decode_unit(p, u);
            const Prob& P = p.prob[U.pi];
            if (!mbar_wait(smem_u32(&tfull[acc]), aphase, s_abort, p.wait_ns)) {
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
    cluster_sync();  // neither CTA leaves while its peer may still signal its barriers
    if (rank == 0 && threadIdx.x == 0) {
        // Both CTAs' loads complete on CTA 0's stage barriers, so CTA 0 waits out the pair's
        // fills still in flight (a role that gave up may have left the last ones unconsumed).
        // The two producers issue the same fill sequence and neither can run a whole ring ahead
        // of the other, so only the last STAGES fills of the longer sequence can be pending.  A
        // fill CTA 0 armed for both CTAs but CTA 1 never issued has CTA 1's bytes completed here;
        // one CTA 1 issued but CTA 0 never armed is armed here with CTA 1's bytes.
        const uint32_t n0 = s_fill[0], n1 = s_fill[1], hi = n0 > n1 ? n0 : n1;
        const uint32_t S = (uint32_t)C::STAGES, half = (uint32_t)(C::A_BYTES + C::B_BYTES);
        volatile int never = 0;
        bool ok = true;
        for (uint32_t k = hi > S ? hi - S : 0u; k < hi; ++k) {
            const uint32_t bar = smem_u32(&full[k % S]);
            if (k < n0 && k >= n1) mbar_complete_tx(bar, half);
            else if (k >= n0 && k < n1) mbar_expect_tx(bar, half);
            ok = mbar_wait(bar, (k / S) & 1u, &never, p.wait_ns) && ok;
        }
        if (!ok) record_error(p, kErrTimeout, 5);
    }
    cluster_sync();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace lm
