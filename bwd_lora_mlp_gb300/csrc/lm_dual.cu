// The dual rank-r reduction kernel (parameters and description in lm_dual.cuh) and its launch:
// one CTA per SM, persistent.
#include "lm_internal.h"

namespace lm {

struct DualUnit {
    int j, rb0, rb1, cb0, cb1, rr, cr;
};

__device__ __forceinline__ DualUnit dual_unit(const DualParams& p, int u) {
    DualUnit U;
    int j = 0;
    while (j + 1 < p.njobs && u >= p.job[j + 1].unit_begin) ++j;
    const DualJob& J = p.job[j];
    const int local = u - J.unit_begin;
    U.j = j;
    U.rr = local / J.ncr;
    U.cr = local - U.rr * J.ncr;
    U.rb0 = U.rr * J.RB;
    U.rb1 = min(J.nrb, U.rb0 + J.RB);
    U.cb0 = U.cr * J.CB;
    U.cb1 = min(J.ncb, U.cb0 + J.CB);
    return U;
}

__device__ __forceinline__ void dual_error(const DualParams& p, int where) {
    if (p.err) {
        atomicExch(p.err, kErrTimeout);
        p.err[1] = where;
        p.err[2] = blockIdx.x;
        p.err[3] = p.kernel_id;
    }
}

__global__ void __launch_bounds__(kDualThreads, 1) dual_reduce_kernel(const __grid_constant__ DualParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kDualMaxStages;
    uint64_t* gfull = empty + kDualMaxStages;   // G accumulator ready (2)
    uint64_t* gempty = gfull + 2;               // G accumulator drained (2)
    uint64_t* dfull = gempty + 2;               // dB accumulator set ready (2)
    uint64_t* dempty = dfull + 2;               // dB accumulator set drained (2)
    uint64_t* drain = dempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint8_t* stages = smem + 1024;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rp = p.rp;
    const int S = p.stages;
    griddep_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&gfull[a]), 1);
            mbar_init(smem_u32(&gempty[a]), 4);
            mbar_init(smem_u32(&dfull[a]), 1);
            mbar_init(smem_u32(&dempty[a]), 4);
        }
        mbar_init(smem_u32(drain), 1);
        *s_abort = 0;
        fence_mbar_init();
        for (int i = 0; i < 3 * p.njobs; ++i) tma_prefetch_map(&p.maps[i]);
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();
    const uint32_t tmem_base = *tmem_slot;
    // TMEM columns: G accumulators at [0, rp) and [rp, 2 rp); dB accumulator set a, column block
    // k of the unit at 2 rp + (a * CBmax + k) rp, CBmax = (512 - 2 rp) / (2 rp)
    const int cbmax = (512 - 2 * rp) / (2 * rp);
    const uint32_t box_p = 128u * (uint32_t)rp;   // bytes of one 64-column box of P
    // B in a stage: rp / 16 boxes of 16 columns x 128 rows (4 KB each), the 16-wide N chunks of an
    // MN-major operand (32-byte swizzle); 256 rp bytes like P's two boxes

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0, nfill = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && !p.inject && u < p.total_units; u += gridDim.x) {
                const DualUnit U = dual_unit(p, u);
                const DualJob& J = p.job[U.j];
                for (int rb = U.rb0; ok && rb < U.rb1; ++rb)
                    for (int cb = U.cb0; cb < U.cb1; ++cb) {
                        if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, s_abort, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sz = smem_u32(stages + stage * p.stage_bytes);
                        const uint32_t sb = sz + 32768u, sp = sb + 2u * box_p;
                        const uint32_t fb = smem_u32(&full[stage]);
                        mbar_expect_tx(fb, (uint32_t)p.stage_bytes);
                        tma_load_2d(sz, &p.maps[J.z_map], fb, cb * 128, rb * 128);
                        tma_load_2d(sz + 16384u, &p.maps[J.z_map], fb, cb * 128 + 64, rb * 128);
                        for (int i = 0; i < (rp >> 4); ++i)
                            tma_load_2d(sb + 4096u * (uint32_t)i, &p.maps[J.b_map], fb, 16 * i, cb * 128);
                        tma_load_2d(sp, &p.maps[J.p_map], fb, rb * 128, J.p_row0);
                        tma_load_2d(sp + box_p, &p.maps[J.p_map], fb, rb * 128 + 64, J.p_row0);
                        ++nfill;
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
            }
            if (!ok) {
                dual_error(p, 1);
                *s_abort = 1;
            }
            if (!drain_fills(smem_u32(&full[0]), S, nfill, p.wait_ns)) dual_error(p, 5);
        }
    } else if (warp == 1) {  // ---------------- MMA issuer: the whole warp, lane 0 issues
        const bool leader = lane == 0;
        const uint32_t idg = make_idesc_bf16(128, rp, false, true);   // Z B: A K-major, B MN-major
        const uint32_t idd = make_idesc_bf16(128, rp, true, false);   // Z^T P: A MN-major
        int stage = 0;
        uint32_t phase = 0;
        uint32_t ga = 0, gph = 0;  // G accumulator in use and its phase
        uint32_t da = 0, dph = 0;  // dB accumulator set in use and its phase
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x) {
            const DualUnit U = dual_unit(p, u);
            if (!mbar_wait_warp(smem_u32(&dempty[da]), dph ^ 1u, s_abort, p.wait_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tdb = tmem_base + (uint32_t)(2 * rp) + da * (uint32_t)(cbmax * rp);
            for (int rb = U.rb0; ok && rb < U.rb1; ++rb) {
                if (!mbar_wait_warp(smem_u32(&gempty[ga]), gph ^ 1u, s_abort, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tg = tmem_base + ga * (uint32_t)rp;
                for (int cb = U.cb0; cb < U.cb1; ++cb) {
                    if (!mbar_wait_warp(smem_u32(&full[stage]), phase, s_abort, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sz = smem_u32(stages + stage * p.stage_bytes);
                    const uint32_t sb = sz + 32768u, sp = sb + 2u * box_p;
                    // The two products alternate, so consecutive MMAs write different accumulators.
                    // Z B: K = the tile's 128 columns, 4 steps of 16 per 64-column box of Z; B's
                    // 16 K rows of a step are 512 bytes of each 16-wide N chunk (4 KB apart).
                    // Z^T P: M = the tile's 128 columns (two 64-wide chunks 16 KB apart), K = its
                    // 128 rows, 16 rows (2048 bytes) per step.
                    const uint32_t td = tdb + (uint32_t)((cb - U.cb0) * rp);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t bx = (uint32_t)(ks >> 2);
                        const uint64_t ag = make_sdesc_sw128(sz + bx * 16384u, 16, 1024) + (uint64_t)((ks & 3) * 2);
                        const uint64_t bg = make_sdesc_sw32(sb + (uint32_t)ks * 512u, 4096, 256);
                        umma_bf16_if(tg, ag, bg, idg, (cb == U.cb0 && ks == 0) ? 0u : 1u, leader);
                        const uint64_t ad = make_sdesc_sw128(sz, 16384, 1024) + (uint64_t)(ks * 128);
                        const uint64_t bd = make_sdesc_sw128(sp + bx * box_p, 16, 1024) + (uint64_t)((ks & 3) * 2);
                        umma_bf16_if(td, ad, bd, idd, (rb == U.rb0 && ks == 0) ? 0u : 1u, leader);
                    }
                    umma_commit_if(smem_u32(&empty[stage]), leader);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_if(smem_u32(&gfull[ga]), leader);
                ga ^= 1u;
                if (ga == 0) gph ^= 1u;
            }
            if (!ok) break;
            umma_commit_if(smem_u32(&dfull[da]), leader);
            da ^= 1u;
            if (da == 0) dph ^= 1u;
        }
        if (!ok && leader) {
            dual_error(p, 2);
            *s_abort = 1;
        }
        umma_commit_if(smem_u32(drain), leader);
        volatile int never = 0;
        mbar_wait(smem_u32(drain), 0, &never, p.wait_ns);
        __syncwarp();
    } else {  // ---------------- drain warps: TMEM lane quarter q = warp & 3
        const int q = warp & 3;
        const int row = q * 32 + lane;  // accumulator lane: a tile row (G) or a tile column (dB)
        uint32_t ga = 0, gph = 0, da = 0, dph = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x) {
            const DualUnit U = dual_unit(p, u);
            const DualJob& J = p.job[U.j];
            for (int rb = U.rb0; rb < U.rb1; ++rb) {
                if (!mbar_wait_warp(smem_u32(&gfull[ga]), gph, s_abort, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int64_t t = (int64_t)rb * 128 + row;
                const uint32_t tg = tmem_base + ((uint32_t)(q * 32) << 16) + ga * (uint32_t)rp;
                float* dst = J.gpart + ((int64_t)U.cr * J.T + t) * rp;
#pragma unroll 1
                for (int c = 0; c < rp; c += 16) {
                    uint32_t a[16];
                    tmem_ld_x16(tg + c, a);
                    tmem_ld_wait16(a);
                    if (t < J.T) {
                        st_global_v8(dst + c, a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7]);
                        st_global_v8(dst + c + 8, a[8], a[9], a[10], a[11], a[12], a[13], a[14], a[15]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&gempty[ga]));
                ga ^= 1u;
                if (ga == 0) gph ^= 1u;
            }
            if (!ok) break;
            if (!mbar_wait_warp(smem_u32(&dfull[da]), dph, s_abort, p.wait_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tdb =
                tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(2 * rp) + da * (uint32_t)(cbmax * rp);
            for (int cb = U.cb0; cb < U.cb1; ++cb) {
                const int64_t c = (int64_t)cb * 128 + row;
                float* dst = J.dpart + ((int64_t)U.rr * J.C + c) * rp;
#pragma unroll 1
                for (int k = 0; k < rp; k += 16) {
                    uint32_t a[16];
                    tmem_ld_x16(tdb + (uint32_t)((cb - U.cb0) * rp + k), a);
                    tmem_ld_wait16(a);
                    if (c < J.C) {
                        st_global_v8(dst + k, a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7]);
                        st_global_v8(dst + k + 8, a[8], a[9], a[10], a[11], a[12], a[13], a[14], a[15]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&dempty[da]));
            da ^= 1u;
            if (da == 0) dph ^= 1u;
        }
        if (!ok && lane == 0) {
            dual_error(p, 3);
            *s_abort = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

cudaError_t launch_dual_reduce(const DualParams& p, int grid, cudaStream_t st) {
    const int smem = 2048 + p.stages * p.stage_bytes;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(dual_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDualSmemBytes);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    e = launch_pdl(dual_reduce_kernel, dim3(grid), dim3(kDualThreads), smem, st, nullptr, 0, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace lm
