// The CTA-pair GEMM of lm_gemm2.cuh with a 4-bit packed frozen B operand decoded in the mainloop
// ("loralei" README, QLoRA section: unpacking and double-scale reconstruction fused into the
// matmul, and the same section's groupwise int4 base; "LoRA Optimizations", FP32 LoRA gradients:
// weight-only NVFP4 bases).  The formats differ only in how a 64-element block of codes becomes
// bf16 -- NF4 code_i * amax' (a register table built per block), int4 (q - 8) * s + z with the
// bf16 scale and zero of the block's group (f16 magic-number arithmetic and one fp32 FMA per
// element), NVFP4 e2m1 * fp32(s_b * S_g) (the hardware E2M1 conversion) -- and in the scales a
// stage carries (see the producer).  The same kernel also
// runs plain bf16 GEMMs (every stage loaded as it is), which the MLPs use for their store GEMMs.
//
// A work unit is a 512 x 256 tile: per 64-deep K block each CTA of the pair holds 2 x 128 A rows
// (one set per M half) and half of the 256-wide B tile, and CTA 0 issues two M = 256 pair MMAs
// per K step that share the decoded B tile, so each decoded weight element feeds 512 output rows
// (decode work per MMA cycle is half that of a 256 x 256 tile).  The accumulator (2 M halves x 256
// columns) fills TMEM, so it is single-buffered.  TMA brings the A rows, the raw 4-bit codes of
// the CTA's B half (4 KB) and their scales (up to 1 KB: for NF4 128 fp32 block scales from a
// per-call table of fp32(q * c) laid out K-block-major; for int4 and NVFP4 the stored scale words
// themselves) into the CTA's own stage and completes on the CTA's own stage barrier; decode warps
// turn every 64-element block of codes into a 128-byte swizzled bf16 row of
// the B tile and then report to CTA 0's decoded barrier, which counts both CTAs' decoders, so
// CTA 0's MMA thread starts a K block only when both halves of B and both A halves are in place.
// The decode warps issue no global loads: their release-arrive would wait for them.
//
// Decoding keeps everything in registers.  NF4: for a block with scale amax' = fp32(q * c) the thread
// forms the 16 products bf16(fp32(code_i * amax')) (the values nf4_dequant writes), splits them
// into low-byte and high-byte tables of four registers each, and assembles every output pair of
// bf16 with byte permutes (prmt) indexed by the code nibbles, choosing between the two halves of
// each table by the nibble's top bit.  No shared-memory table is read, which keeps the shared
// memory bandwidth for the MMA operands.
//
// Roles (576 threads): warp 0 TMA producer, warp 1 MMA issuer (CTA 0), warps 2-9 decoders in
// kPairNf4DecodeGroups groups that take K blocks round-robin (with two groups of four warps, two K
// blocks are decoded at once and each thread decodes one 64-element block of each), warps 10-17
// epilogue.  The producer tags every stage for the decoders (bf16, NF4, int4 with its group size,
// NVFP4 with its scale map, or end of work), so they follow the stage ring without walking the
// work-unit sequence themselves.  The GLU backward epilogue (dh) may borrow the stage slot of its
// tile's last K block to stage e, u through shared memory (glu_bwd_staged); the producer then
// holds back the next load into that slot until the epilogue releases it.
#pragma once

#include "lm_gemm2.cuh"
#include "lm_nf4_table.cuh"

namespace lm {

constexpr int kPairNf4DecodeWarps = 8;
constexpr int kPairNf4DecodeGroups = 2;   // groups take K blocks round-robin
constexpr int kPairNf4GroupWarps = kPairNf4DecodeWarps / kPairNf4DecodeGroups;
constexpr int kPairNf4BlocksPerThread = 128 / (32 * kPairNf4GroupWarps);  // 64-element blocks per thread per K block
static_assert(kPairNf4BlocksPerThread == 1 || kPairNf4BlocksPerThread == 2, "decode split");
constexpr int kPairNf4Threads = 64 + 32 * kPairNf4DecodeWarps + 32 * kNumEpiWarps;

struct Gemm2Nf4Cfg {
    static constexpr int A_BYTES = 2 * kBM * kBK * 2;  // this CTA's 2 x 128 A rows (one per M half)
    static constexpr int B_BYTES = 128 * kBK * 2;      // this CTA's half of B, decoded (or bf16 via TMA)
    static constexpr int C_BYTES = 4096;               // raw codes of that half
    static constexpr int S_BYTES = 1024;               // their scales: 128 fp32 NF4 block scales,
                                                       // or up to 256 int4 (scale, zero) words
    static constexpr int S_OFF = A_BYTES + B_BYTES + C_BYTES;
    static constexpr int STAGE_BYTES = (S_OFF + S_BYTES + 1023) / 1024 * 1024;
    static constexpr int STAGES = 4;
    static constexpr int TMEM_COLS = 512;              // one accumulator: 2 M halves x 256 columns
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024;
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
    // Each stage slot must always be decoded by the same group: a group waits on a slot's full
    // barrier by phase parity, and if the slot's previous K block belonged to another group whose
    // TMA had not landed yet (loads of different stages complete in any order), the barrier would
    // still be one phase behind and the parity wait would pass at once.
    static_assert(STAGES % kPairNf4DecodeGroups == 0, "decode groups must divide the stage count");
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The 16 bf16 values of a 4-bit code as low-byte and high-byte tables of four registers each,
// in code order.
struct Q4Tab {
    uint32_t L0, L1, L2, L3, H0, H1, H2, H3;
};

// T[i] holds the bf16 values of codes 2i (low half) and 2i + 1 (high half)
__device__ __forceinline__ Q4Tab q4_tab(const uint32_t (&T)[8]) {
    Q4Tab t;
    t.L0 = prmt(T[0], T[1], 0x6420);
    t.L1 = prmt(T[2], T[3], 0x6420);
    t.L2 = prmt(T[4], T[5], 0x6420);
    t.L3 = prmt(T[6], T[7], 0x6420);
    t.H0 = prmt(T[0], T[1], 0x7531);
    t.H1 = prmt(T[2], T[3], 0x7531);
    t.H2 = prmt(T[4], T[5], 0x7531);
    t.H3 = prmt(T[6], T[7], 0x7531);
    return t;
}

// NF4 block with scale amax: code i -> bf16(fp32(nf4[i] * amax))
__device__ __forceinline__ Q4Tab nf4_tab(float amax) {
    uint32_t T[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        T[i] = pack_bf16x2(__fmul_rn(nf4_value(2 * i), amax), __fmul_rn(nf4_value(2 * i + 1), amax));
    return q4_tab(T);
}

// Decode the 16-byte output chunks J0..J1-1 (8 elements each, from code word j) of one 64-element
// block into a 128-byte row of the swizzled B tile at dst_row (chunk j stored at chunk j ^ swz).
// Code words hold element 2i in the high nibble of byte i.
template <int J0, int J1>
__device__ __forceinline__ void q4_decode_chunks(const Q4Tab& t, const uint32_t (&words)[8], uint32_t dst_row,
                                                 int swz) {
#pragma unroll
    for (int j = J0; j < J1; ++j) {
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
            const uint32_t lw = (prmt(t.L2, t.L3, sel) & m) | (prmt(t.L0, t.L1, sel) & ~m);
            const uint32_t hw = (prmt(t.H2, t.H3, sel) & m) | (prmt(t.H0, t.H1, sel) & ~m);
            o[2 * h] = prmt(lw, hw, 0x4051);      // bf16 of n1 (low half), n0 (high half)
            o[2 * h + 1] = prmt(lw, hw, 0x6273);  // bf16 of n3, n2
        }
        const uint32_t addr = dst_row + ((uint32_t)(j ^ swz) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                     "r"(o[3])
                     : "memory");
    }
}

__device__ __forceinline__ void q4_words(const uint4* src, uint32_t (&w)[8]) {
    const uint4 c0 = src[0], c1 = src[1];
    w[0] = c0.x; w[1] = c0.y; w[2] = c0.z; w[3] = c0.w;
    w[4] = c1.x; w[5] = c1.y; w[6] = c1.z; w[7] = c1.w;
}

// Decode one 64-element int4 block (8 code words, element 2i in the high nibble of byte i) into a
// 128-byte row of the swizzled B tile: w = bf16(fp32((q - 8) * s + z)), with (s, z) of word sz[0]
// for the first 32 elements and of sz[1] for the rest.  The nibbles become f16 values 1024 + q by
// OR-ing them into the mantissa of 1024 (two per instruction), an f16 subtraction of 1032 gives
// q - 8 exactly, and an fp32 fused multiply-add rounds (q - 8) * s + z once -- the arithmetic
// runs on the FMA pipe instead of a chain of byte permutes on the integer pipe.
__device__ __forceinline__ void int4_decode_block(const uint32_t (&words)[8], const uint32_t (&sz)[2],
                                                  uint32_t dst_row, int swz) {
    const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6408u),
                                        __ushort_as_half((unsigned short)0x6408u));  // 1032
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t wd = sz[j >> 2];
        const float s = __uint_as_float(wd << 16), z = __uint_as_float(wd & 0xFFFF0000u);
        const uint32_t w = words[j];
        // p_i holds nibbles i (low half) and i + 4 (high half); nibble 2k is element 2k + 1 and
        // nibble 2k + 1 is element 2k of the word
        float v[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t m = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;
            const float2 f = __half22float2(__hsub2(*reinterpret_cast<const __half2*>(&m), bias));
            const int e = (i & 1) ? i - 1 : i + 1;  // element of nibble i
            v[e] = __fmaf_rn(f.x, s, z);
            v[e + 4] = __fmaf_rn(f.y, s, z);
        }
        const uint32_t o0 = pack_bf16x2(v[0], v[1]), o1 = pack_bf16x2(v[2], v[3]);
        const uint32_t o2 = pack_bf16x2(v[4], v[5]), o3 = pack_bf16x2(v[6], v[7]);
        const uint32_t addr = dst_row + ((uint32_t)(j ^ swz) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o0), "r"(o1), "r"(o2), "r"(o3)
                     : "memory");
    }
}

// Two E4M3 bytes (low byte first) -> their values as f16x2 (exact: every E4M3 value is an f16)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t d;
    asm("{\n .reg .b16 h;\n mov.b32 {h, _}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}" : "=r"(d) : "r"(two));
    return d;
}

// Four bytes of E2M1 code pairs (element 2i in the low nibble) -> four f16x2 (exact)
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

__device__ __forceinline__ float f16lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu))); }
__device__ __forceinline__ float f16hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

// Decode one 64-element NVFP4 span (8 code words, word j = elements 8j..8j+7; E4M3 scales of its
// four 16-element blocks in the bytes of sc4) with tensor scale gs into a 128-byte row of the
// swizzled B tile: w = bf16(fp32(e2m1 * fp32(s_b * gs))).
__device__ __forceinline__ void nvfp4_decode_block(const uint32_t (&words)[8], uint32_t sc4, float gs,
                                                   uint32_t dst_row, int swz) {
    const uint32_t s01 = e4m3x2_to_f16x2(sc4), s23 = e4m3x2_to_f16x2(sc4 >> 16);
    const float S[4] = {__fmul_rn(f16lo(s01), gs), __fmul_rn(f16hi(s01), gs), __fmul_rn(f16lo(s23), gs),
                        __fmul_rn(f16hi(s23), gs)};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t h[4], o[4];
        e2m1x8_to_f16x2(words[j], h);
        const float Sj = S[j >> 1];
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = pack_bf16x2(__fmul_rn(f16lo(h[k]), Sj), __fmul_rn(f16hi(h[k]), Sj));
        const uint32_t addr = dst_row + ((uint32_t)(j ^ swz) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                     "r"(o[3])
                     : "memory");
    }
}

// GLU backward epilogue of a 512-row tile with e, u staged through shared memory.  The tile's
// single accumulator leaves its epilogue exposed, and with one accumulator row per thread each
// warp access to e, u in global memory would touch 32 rows of 32 bytes; here TMA brings them in
// chunks of 16 columns (this CTA's two 128-row halves of e and u: 16 KB) into three buffers of
// the stage slot that held the tile's last K block.  The producer does not refill that slot
// until every epilogue warp has arrived on `scrfree` (see the producer's gate).  Lane 0 of the
// first epilogue warp issues the loads, three chunks ahead; each warp releases a buffer as soon
// as it has read its row from it.  `qn` counts the chunks staged by this CTA so far (buffer
// qn % 3, phase qn / 3); *s_qi counts the chunks issued, which may run three ahead of qn, so that
// the loads still in flight can be waited out before the CTA leaves.  Returns false on a timed-out
// wait.
constexpr int kStageChunkBytes = 16384;
constexpr int kStageBuffers = 3;

__device__ __forceinline__ bool glu_bwd_staged(const Params& p, const Prob& P, const Unit& U, uint32_t tacc,
                                               int64_t m, uint32_t scr, uint32_t efull0, uint32_t eempty0,
                                               uint32_t rank, bool issuer, int hh, int r, uint32_t& qn,
                                               volatile uint32_t* s_qi, volatile int* s_abort) {
    const int nch = P.bn >> 4;
    const int32_t row0 = (int32_t)((int64_t)U.mb * 512 + (int64_t)rank * kBM);
    const int64_t col0 = (int64_t)U.nb * P.out_col_step;
    const CUtensorMap* me = &p.maps[P.in_map[0]];
    const CUtensorMap* mu = &p.maps[P.in_map[1]];
    const uint32_t q0 = qn;
    // chunk c of this tile into buffer (q0 + c) % 3, once every warp has released that buffer's
    // previous chunk
    auto issue = [&](int c) -> bool {
        const uint32_t q = q0 + (uint32_t)c, b = q % kStageBuffers;
        if (q >= kStageBuffers &&
            !mbar_wait(eempty0 + 8 * b, ((q - kStageBuffers) / kStageBuffers) & 1u, s_abort, p.wait_ns))
            return false;
        const uint32_t dst = scr + b * kStageChunkBytes, bar = efull0 + 8 * b;
        const int32_t x = (int32_t)(col0 + 16 * c);
        mbar_expect_tx(bar, kStageChunkBytes);
        tma_load_2d(dst, me, bar, x, row0);
        tma_load_2d(dst + 4096, me, bar, x, row0 + 256);
        tma_load_2d(dst + 8192, mu, bar, x, row0);
        tma_load_2d(dst + 12288, mu, bar, x, row0 + 256);
        *s_qi = q + 1;
        return true;
    };
    int fail = 0;
    if (issuer)
        for (int c = 0; c < kStageBuffers && c < nch && !fail; ++c) fail = !issue(c);
    if (__any_sync(0xffffffffu, fail)) return false;
    // this thread's row in a 128-row box: 32 bytes, 16-byte halves swapped on every other group
    // of four rows (the 32-byte swizzle)
    const uint32_t sw = (uint32_t)((r >> 2) & 1) << 4;
    const uint32_t roff = (uint32_t)hh * 4096 + (uint32_t)r * 32;
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
        const uint32_t q = q0 + (uint32_t)c, b = q % kStageBuffers;
        if (!mbar_wait_warp(efull0 + 8 * b, (q / kStageBuffers) & 1u, s_abort, p.wait_ns)) return false;
        const uint32_t base = scr + b * kStageChunkBytes + roff;
        uint32_t ev[8], uv[8];
        ld_shared_v4(base + sw, ev[0], ev[1], ev[2], ev[3]);
        ld_shared_v4(base + (sw ^ 16u), ev[4], ev[5], ev[6], ev[7]);
        ld_shared_v4(base + 8192 + sw, uv[0], uv[1], uv[2], uv[3]);
        ld_shared_v4(base + 8192 + (sw ^ 16u), uv[4], uv[5], uv[6], uv[7]);
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(eempty0 + 8 * b);
        uint32_t a[16];
        tmem_ld_x16(tacc + 16 * c, a);
        tmem_ld_wait16(a);
        const int64_t gcol = col0 + 16 * c;
        if (m < P.M && gcol < P.N) {
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
        if (issuer && c + kStageBuffers < nch) fail = !issue(c + kStageBuffers);
        if (__any_sync(0xffffffffu, fail)) return false;
    }
    qn = q0 + (uint32_t)nch;
    return true;
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
    uint64_t* efull = drain + 1;       // staged e, u chunks of the GLU backward epilogue
    uint64_t* eempty = efull + kStageBuffers;
    uint64_t* scrfree = eempty + kStageBuffers;  // the epilogue has released the slot it borrowed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(scrfree + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // what each stage holds, written by this CTA's producer before the stage's loads: 0 bf16 B
    // (nothing to decode), 1 NF4 codes, 3 | G << 8 int4 codes with groups of G, 4 | map << 8 NVFP4
    // codes (map: the scale map, whose tensor scale s_gscale holds), 2 no more K blocks (one such
    // stage per decode group)
    volatile int32_t* stage_kind = reinterpret_cast<volatile int32_t*>(tmem_slot + 2);
    // fp32 tensor scale of each NVFP4 scale map, read once at launch
    float* s_gscale = const_cast<float*>(reinterpret_cast<volatile float*>(stage_kind + C::STAGES));
    // e, u chunks the staged GLU backward epilogue has issued (its issuing thread writes it)
    volatile uint32_t* s_qi = reinterpret_cast<volatile uint32_t*>(s_gscale + kMaxMaps);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    griddep_launch_dependents();
    const uint32_t rank = cluster_ctarank();
    const int cid = (int)cluster_id_x();
    const int ncl = (int)nclusters_x();

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&bready[s]), 2 * kPairNf4GroupWarps);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), 2 * kNumEpiWarps);
        }
        mbar_init(smem_u32(drain), 1);
        for (int b = 0; b < kStageBuffers; ++b) {
            mbar_init(smem_u32(&efull[b]), 1);
            mbar_init(smem_u32(&eempty[b]), kNumEpiWarps);
        }
        mbar_init(smem_u32(scrfree), kNumEpiWarps);
        *s_abort = 0;
        *s_qi = 0;
        fence_mbar_init();
        for (int i = 0; i < kMaxMaps; ++i)
            if (p.map_bytes[i]) tma_prefetch_map(&p.maps[i]);
    }
    if (threadIdx.x >= 32 && threadIdx.x < 32 + kMaxMaps) {  // published by the cluster barrier below
        const int i = threadIdx.x - 32;
        griddep_wait();  // (a previous kernel of the stream may have written the scale)
        s_gscale[i] = p.map_gscale[i] ? __ldg(p.map_gscale[i]) : 0.0f;
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    griddep_wait();  // the previous kernel of the stream has completed: its outputs are visible
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t bready0 = map_to_rank(smem_u32(&bready[0]), 0);
    const uint32_t tempty0 = map_to_rank(smem_u32(&tempty[0]), 0);

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer (both CTAs, own stage barriers)
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // A GLU backward epilogue that stages e, u borrows the slot of its tile's last K block
            // (iteration E - 1, E = K blocks issued up to the end of the tile); iteration E + 3 is
            // the next load into that slot and waits until the epilogue has released it.  Every
            // unit of such a launch has at least four K blocks, so the gate falls inside the next
            // tile and the releases are waited for in order, one phase at a time.
            uint32_t it = 0, gate[4] = {0u, 0u, 0u, 0u}, gh = 0, gt = 0, nrel = 0;
            uint32_t nfill = 0;  // stage fills (loads and end-of-work marks) issued
            for (int u = cid; ok && !p.inject && u < p.total_units; u += ncl) {
                const Unit U = decode_unit(p, u);
                const Prob& P = p.prob[U.pi];
                int g0, g1;
                unit_kslice(P, U, g0, g1);
                for (int si = 0, g = 0; ok && si < P.nseg; ++si) {
                    const Seg& S = P.seg[si];
                    const int nkb = (S.kext + kBK - 1) / kBK;
                    const int kb0 = max(0, g0 - g), kb1 = min(nkb, g1 - g);
                    g += nkb;
                    const bool nf4 = S.b_scale[0] >= 0;
                    const int bmap = (rank == 1 && S.b_map[1] >= 0) ? S.b_map[1] : S.b_map[0];
                    const int smap = (rank == 1 && S.b_scale[1] >= 0) ? S.b_scale[1] : S.b_scale[0];
                    // int4 group size (0: NF4, -1: NVFP4); the decoders read the format, and the
                    // int4 group size or the NVFP4 scale map, from the stage tag
                    const int q4g = nf4 ? p.map_group[smap] : 0;
                    const int32_t tag = !nf4 ? 0 : q4g > 0 ? (3 | (q4g << 8)) : q4g < 0 ? (4 | (smap << 8)) : 1;
                    const int brow = U.nb * P.n_step + (int)rank * S.b_rank_off;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (gh != gt && gate[gh & 3] == it) {
                            if (!mbar_wait(smem_u32(scrfree), nrel & 1u, s_abort, p.wait_ns)) {
                                ok = false;
                                break;
                            }
                            ++nrel;
                            ++gh;
                        }
                        if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, s_abort, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        ++it;
                        const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
                        const uint32_t sB = sA + C::A_BYTES;
                        const uint32_t sC = sB + C::B_BYTES;
                        const uint32_t fb = smem_u32(&full[stage]);
                        const int kx = kb * kBK;
                        stage_kind[stage] = tag;
                        mbar_expect_tx(fb, C::A_BYTES + (nf4 ? (uint32_t)(p.map_bytes[bmap] + p.map_bytes[smap])
                                                             : (uint32_t)C::B_BYTES));
                        tma_load_2d(sA, &p.maps[S.a_map], fb, kx + S.a_xoff, U.mb * 512 + (int)rank * kBM);
                        tma_load_2d(sA + 16384, &p.maps[S.a_map], fb, kx + S.a_xoff, U.mb * 512 + 256 + (int)rank * kBM);
                        if (nf4) {
                            // NF4 scale table / NVFP4 scale words [64-column span][weight row]:
                            // K-major, the 128 rows of this K block; MN-major, 64 K rows of the
                            // two 64-wide column spans.  int4 (scale, zero) words [group][weight
                            // row]: the groups that the stage's 64 (K-major) or 128 (MN-major)
                            // weight columns fall in.
                            const uint32_t sS = sA + C::S_OFF;
                            if constexpr (B_MN) {
                                tma_load_2d(sC, &p.maps[bmap], fb, brow / 2, kx);
                                tma_load_2d(sS, &p.maps[smap], fb, kx, q4g > 0 ? brow / q4g : brow / 64);
                            } else {
                                tma_load_2d(sC, &p.maps[bmap], fb, kx / 2, brow);
                                tma_load_2d(sS, &p.maps[smap], fb, brow, q4g > 0 ? kx / q4g : kb);
                            }
                        } else if constexpr (B_MN) {
                            tma_load_2d(sB, &p.maps[bmap], fb, brow, kx);
                            tma_load_2d(sB + 8192, &p.maps[bmap], fb, brow + 64, kx);
                        } else {
                            tma_load_2d(sB, &p.maps[bmap], fb, kx + S.b_xoff[0], brow);
                        }
                        ++nfill;
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (EPI == EPI_GLU_BWD && P.in_map[0] >= 0) gate[gt++ & 3] = it + 3;
            }
            // one end-of-work stage for each decode group (the next stage in its round-robin)
            for (int g = 0; ok && !p.inject && g < kPairNf4DecodeGroups; ++g) {
                if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, s_abort, p.wait_ns)) {
                    ok = false;
                    break;
                }
                stage_kind[stage] = 2;
                mbar_arrive(smem_u32(&full[stage]));
                ++nfill;
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                record_error(p, kErrTimeout, 1);
                *s_abort = 1;
            }
            // this CTA's loads complete on its own stage barriers: wait out the ones in flight
            if (!drain_fills(smem_u32(&full[0]), C::STAGES, nfill, p.wait_ns)) record_error(p, kErrTimeout, 5);
        }
    } else if (warp == 1) {
        if (rank == 0) {  // ---------------- MMA issuer (CTA 0 only): the whole warp, lane 0 issues
            const bool leader = lane == 0;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t aphase = 0;  // one accumulator: its free / ready phases flip every tile
            bool ok = true;
            for (int u = cid; ok && u < p.total_units; u += ncl) {
                const Unit U = decode_unit(p, u);
                const Prob& P = p.prob[U.pi];
                if (!mbar_wait_warp(smem_u32(&tempty[0]), aphase ^ 1u, s_abort, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t idesc = make_idesc_bf16(256, P.bn, false, B_MN);
                uint32_t accum = 0;
                int g0, g1;
                unit_kslice(P, U, g0, g1);
                for (int si = 0, g = 0; ok && si < P.nseg; ++si) {
                    const Seg& S = P.seg[si];
                    const int nkb = (S.kext + kBK - 1) / kBK;
                    const int kb0 = max(0, g0 - g), kb1 = min(nkb, g1 - g);
                    g += nkb;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait_warp(smem_u32(&bready[stage]), phase, s_abort, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
                        const uint32_t sB = sA + C::A_BYTES;
                        const int rem = S.kext - kb * kBK;
                        const int nsteps = rem >= kBK ? 4 : (rem + 15) >> 4;
                        // fixed four-step body; a short last K block masks its tail steps
                        const uint64_t ad0 = make_sdesc_sw128(sA, 16, 1024);
                        const uint64_t bd0 = B_MN ? make_sdesc_sw128(sB, 8192, 1024) : make_sdesc_sw128(sB, 16, 1024);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint64_t bd = bd0 + (uint64_t)(B_MN ? ks * 128 : ks * 2);
#pragma unroll
                            for (int h = 0; h < 2; ++h)  // both M halves share the decoded B tile
                                umma_bf16_pair_if(tmem_base + h * 256, ad0 + (uint64_t)(h * 1024 + ks * 2), bd, idesc,
                                                  ks == 0 ? accum : 1u, leader && ks < nsteps);
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
                umma_commit_pair_if(smem_u32(&tfull[0]), 0x3, leader);
                aphase ^= 1u;
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
    } else if (warp < 2 + kPairNf4DecodeWarps) {  // ---------------- decoders (both CTAs)
        const int dw = warp - 2;
        const int group = dw / kPairNf4GroupWarps;  // takes the K blocks with iter % groups == group
        // blocks t0 (and t0 + 64 with two per thread) of each K block
        const int t0 = (dw % kPairNf4GroupWarps) * 32 + lane;
        bool ok = true;
        for (uint32_t iter = (uint32_t)group;; iter += kPairNf4DecodeGroups) {
            const int stage = (int)(iter % C::STAGES);
            const uint32_t phase = (iter / C::STAGES) & 1u;
            if (!mbar_wait(smem_u32(&full[stage]), phase, s_abort, p.wait_ns)) {
                ok = false;
                break;
            }
            const int kind = stage_kind[stage];
            if (kind == 2) break;
            if (kind == 1) {
                uint8_t* stg = smem + stage * C::STAGE_BYTES;
                const uint32_t sB = smem_u32(stg + C::A_BYTES);
                const uint8_t* sC = stg + C::A_BYTES + C::B_BYTES;
                // block t's scale sits at index t in both layouts (K-major: B row t; MN-major:
                // column block t >> 6, K row t & 63); rows outside the weight read 0
                const float* sS = reinterpret_cast<const float*>(stg + C::S_OFF);
#pragma unroll
                for (int j = 0; j < kPairNf4BlocksPerThread; ++j) {
                    const int t = t0 + 64 * j;
                    // MN-major: K row t & 63, 64-wide N chunk t >> 6 (32 code bytes of a 64-byte K
                    // row); K-major: B row t
                    const uint4* src = B_MN ? reinterpret_cast<const uint4*>(sC + (t & 63) * 64 + (t >> 6) * 32)
                                            : reinterpret_cast<const uint4*>(sC + t * 32);
                    const uint32_t dst = B_MN ? sB + (t >> 6) * 8192 + (t & 63) * 128 : sB + t * 128;
                    uint32_t words[8];
                    q4_words(src, words);
                    q4_decode_chunks<0, 8>(nf4_tab(sS[t]), words, dst, t & 7);
                }
                fence_proxy_async_smem();
            } else if ((kind & 0xFF) == 3) {
                // int4: the (scale, zero) words of this stage, [group][row] as loaded; a block's
                // first and second 32 elements share a word unless groups hold 32 elements
                uint8_t* stg = smem + stage * C::STAGE_BYTES;
                const uint32_t sB = smem_u32(stg + C::A_BYTES);
                const uint8_t* sC = stg + C::A_BYTES + C::B_BYTES;
                const uint32_t* sW = reinterpret_cast<const uint32_t*>(stg + C::S_OFF);
                const int gsh = 31 - __clz(kind >> 8);  // log2 of the group size
#pragma unroll
                for (int j = 0; j < kPairNf4BlocksPerThread; ++j) {
                    const int t = t0 + 64 * j;
                    const uint4* src = B_MN ? reinterpret_cast<const uint4*>(sC + (t & 63) * 64 + (t >> 6) * 32)
                                            : reinterpret_cast<const uint4*>(sC + t * 32);
                    const uint32_t dst = B_MN ? sB + (t >> 6) * 8192 + (t & 63) * 128 : sB + t * 128;
                    // MN-major: groups along the stage's 128 columns, 64 K rows each; K-major: one
                    // group per row (two when groups hold 32 elements), 128 rows each
                    const int lo = B_MN ? (((t >> 6) * 64) >> gsh) * 64 + (t & 63) : t;
                    const int hi = B_MN ? (((t >> 6) * 64 + 32) >> gsh) * 64 + (t & 63) : (gsh == 5 ? 128 + t : t);
                    uint32_t words[8];
                    q4_words(src, words);
                    const uint32_t sz[2] = {sW[lo], sW[hi]};
                    int4_decode_block(words, sz, dst, t & 7);
                }
                fence_proxy_async_smem();
            } else if ((kind & 0xFF) == 4) {
                // NVFP4: block t's four E4M3 scales (one per 16 elements) sit in word t in both
                // layouts, as the NF4 block scales do
                uint8_t* stg = smem + stage * C::STAGE_BYTES;
                const uint32_t sB = smem_u32(stg + C::A_BYTES);
                const uint8_t* sC = stg + C::A_BYTES + C::B_BYTES;
                const uint32_t* sW = reinterpret_cast<const uint32_t*>(stg + C::S_OFF);
                const float gs = s_gscale[kind >> 8];
#pragma unroll
                for (int j = 0; j < kPairNf4BlocksPerThread; ++j) {
                    const int t = t0 + 64 * j;
                    const uint4* src = B_MN ? reinterpret_cast<const uint4*>(sC + (t & 63) * 64 + (t >> 6) * 32)
                                            : reinterpret_cast<const uint4*>(sC + t * 32);
                    const uint32_t dst = B_MN ? sB + (t >> 6) * 8192 + (t & 63) * 128 : sB + t * 128;
                    uint32_t words[8];
                    q4_words(src, words);
                    nvfp4_decode_block(words, sW[t], gs, dst, t & 7);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_peer(bready0 + stage * 8);
        }
        if (!ok && lane == 0) {
            record_error(p, kErrTimeout, 4);
            *s_abort = 1;
        }
    } else {  // ---------------- epilogue warps (both CTAs)
        const int ew = warp - 2 - kPairNf4DecodeWarps;
        const int q = warp & 3;
        const int hh = ew >> 2;  // M half
        uint32_t aphase = 0;
        uint32_t kdone = 0;  // K blocks of this CTA's tiles so far: the stage ring's position
        uint32_t qn = 0;     // e, u chunks staged so far
        bool ok = true;
        for (int u = cid; u < p.total_units; u += ncl) {
            const Unit U = decode_unit(p, u);
            const Prob& P = p.prob[U.pi];
            int g0, g1;
            unit_kslice(P, U, g0, g1);
            kdone += (uint32_t)(g1 - g0);
            if (!mbar_wait(smem_u32(&tfull[0]), aphase, s_abort, p.wait_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + hh * 256;
            const int64_t m = (int64_t)U.mb * 512 + hh * 256 + (int64_t)rank * kBM + q * 32 + lane;
            if constexpr (EPI == EPI_GLU_BWD) {
                if (P.in_map[0] >= 0) {
                    // the slot of the tile's last K block: free once the MMAs behind tfull are done
                    const uint32_t scr = smem_u32(smem + ((kdone - 1u) % C::STAGES) * C::STAGE_BYTES);
                    if (!glu_bwd_staged(p, P, U, tacc, m, scr, smem_u32(&efull[0]), smem_u32(&eempty[0]), rank,
                                        ew == 0 && lane == 0, hh, q * 32 + lane, qn, s_qi, s_abort)) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(scrfree));
                } else {
                    epilogue_cols<EPI>(P, U, tacc, 0, P.bn, 16, m, m < P.M);
                }
            } else if constexpr (EPI == EPI_GLU_FWD) {
                epilogue_cols<EPI>(P, U, tacc, 0, P.bn >> 1, 16, m, m < P.M);
            } else if (EPI == EPI_STORE && U.tail >= 0) {
                // part U.ks of a split tail tile: the raw fp32 accumulator row to its block
                float* dst = P.tail_part +
                             ((int64_t)(U.tail * P.tail_splits + U.ks) * 512 + (m - (int64_t)U.mb * 512)) * P.bn;
#pragma unroll 1
                for (int c = 0; c < P.bn; c += 32) {
                    uint32_t a[16], b[16];
                    tmem_ld_x16(tacc + c, a);
                    tmem_ld_x16(tacc + c + 16, b);
                    tmem_ld_wait32(a, b);
                    st_global_v8(dst + c, a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7]);
                    st_global_v8(dst + c + 8, a[8], a[9], a[10], a[11], a[12], a[13], a[14], a[15]);
                    st_global_v8(dst + c + 16, b[0], b[1], b[2], b[3], b[4], b[5], b[6], b[7]);
                    st_global_v8(dst + c + 24, b[8], b[9], b[10], b[11], b[12], b[13], b[14], b[15]);
                }
            } else {
                epilogue_cols<EPI>(P, U, tacc, 0, P.bn, 16, m, m < P.M);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_peer(tempty0);  // this CTA's TMEM reads are complete (wait::ld)
            aphase ^= 1u;
        }
        if (!ok && lane == 0) {
            record_error(p, kErrTimeout, 3);
            *s_abort = 1;
        }
    }
    if constexpr (EPI == EPI_GLU_BWD) {
        // the thread that staged e, u chunks waits out its loads still in flight
        if (threadIdx.x == 32 * (2 + kPairNf4DecodeWarps) &&
            !drain_fills(smem_u32(&efull[0]), kStageBuffers, *s_qi, p.wait_ns))
            record_error(p, kErrTimeout, 5);
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
