// Memory-bound helper kernels: finalisation of split-K partials of the rank-r products, and
// NF4 pack / dequantise ("loralei" README, QLoRA section: NF4 with 64-element blocks and
// block scales double-quantised per 256 blocks).
#include <cmath>

#include "lm_internal.h"
#include "lm_nf4_table.cuh"

namespace lm {

// ------------------------------------------------------------------ split-K finalisation
struct FinRowJobs {
    FinRowJob j[3];
};

// Sum of split slices in slice order, with the loads of up to eight slices issued before their
// additions (the order of the additions, and so the result, is that of a plain loop).
__device__ __forceinline__ float4 sum_splits(const float* p0, int64_t stride, int splits) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < splits; k0 += 8) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (k0 + i < splits) v[i] = *reinterpret_cast<const float4*>(p0 + (int64_t)(k0 + i) * stride);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (k0 + i < splits) {
                acc.x += v[i].x;
                acc.y += v[i].y;
                acc.z += v[i].z;
                acc.w += v[i].w;
            }
    }
    return acc;
}

// One CTA per 32 rows of one job: the rows' partials are one contiguous span of 32 ncols floats
// per split, read with coalesced 16-byte loads; the row-major result is written the same way and
// the transposed one through a shared-memory tile, 32 contiguous values per output row.  ncols
// (at most kFinRowMaxCols) and group are multiples of 4.  The grid is flat: njobs x row_blocks
// blocks for the row jobs, then side_blocks blocks that loop over the launch's side work
// (FinSide), which depends on nothing the row jobs produce.
constexpr int kFinRowMaxCols = 192;
constexpr int kFinRowTile = 32;

__device__ void blockdiag_rows(const uint16_t* __restrict__ Bg, const uint16_t* __restrict__ Bu, int64_t n, int r,
                               int rp, uint16_t* __restrict__ out, int64_t first, int64_t stride);
__device__ void nf4_scale_tile(const Nf4ScaleJobs& jobs, int njobs, int t, float (*tile)[65]);
__host__ __device__ inline int64_t nf4_scale_tiles(const Nf4ScaleJobs& jobs, int njobs) {
    int64_t tiles = 0;
    for (int j = 0; j < njobs; ++j) tiles += ((jobs.j[j].rows + 63) / 64) * ((jobs.j[j].kblocks + 63) / 64);
    return tiles;
}

__global__ void __launch_bounds__(256) fin_rowproj_kernel(FinRowJobs jobs, int njobs, int64_t T, int64_t row_blocks,
                                                             int64_t side_blocks, FinSide side) {
    __shared__ union {
        uint16_t tileT[kFinRowMaxCols * (kFinRowTile + 2)];  // row jobs: [column][row], padded pitch
        float nf4[64][65];                                   // NF4 table tiles
    } sm;
    griddep_launch_dependents();
    griddep_wait();
    const int64_t bid = blockIdx.x;
    if (bid >= njobs * row_blocks) {  // side work: the block-diagonal operand, then NF4 tables
        const int64_t sb = bid - njobs * row_blocks;
        if (side.bd_out)
            blockdiag_rows(side.bd_Bg, side.bd_Bu, side.bd_n, side.bd_r, side.bd_rp, side.bd_out,
                           sb * blockDim.x + threadIdx.x, side_blocks * blockDim.x);
        const int64_t tiles = nf4_scale_tiles(side.nf4, side.nf4_jobs);
        for (int64_t t = sb; t < tiles; t += side_blocks) {  // (uniform across the CTA)
            nf4_scale_tile(side.nf4, side.nf4_jobs, (int)t, sm.nf4);
            __syncthreads();
        }
        return;
    }
    const FinRowJob& J = jobs.j[bid / row_blocks];
    const int nc = J.ncols;
    const int pitch = kFinRowTile + 2;
    const int64_t t0 = (bid % row_blocks) * kFinRowTile;
    if (t0 >= T) return;
    const int rows = T - t0 < kFinRowTile ? (int)(T - t0) : kFinRowTile;
    const int n4 = rows * nc / 4;
    const float* base = J.part + t0 * nc;
    uint16_t* tileT = sm.tileT;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const int e = 4 * i, row = e / nc, c0 = e - row * nc;
        const float4 a = sum_splits(base + e, J.split_stride, J.splits);
        const float sc = J.s[c0 / J.group];
        const uint32_t w0 = pack_bf16x2(a.x * sc, a.y * sc), w1 = pack_bf16x2(a.z * sc, a.w * sc);
        *reinterpret_cast<uint2*>(J.out + (t0 + row) * nc + c0) = make_uint2(w0, w1);
        tileT[(c0 + 0) * pitch + row] = (uint16_t)(w0 & 0xFFFFu);
        tileT[(c0 + 1) * pitch + row] = (uint16_t)(w0 >> 16);
        tileT[(c0 + 2) * pitch + row] = (uint16_t)(w1 & 0xFFFFu);
        tileT[(c0 + 3) * pitch + row] = (uint16_t)(w1 >> 16);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nc * kFinRowTile; i += blockDim.x) {
        const int c = i / kFinRowTile, row = i - c * kFinRowTile;
        if (row < rows) J.outT[(int64_t)c * J.ldT + t0 + row] = tileT[c * pitch + row];
    }
}

cudaError_t launch_fin_rowproj(const FinRowJob* jobs, int njobs, int64_t T, cudaStream_t st, const FinSide* side) {
    FinRowJobs js{};
    if (njobs < 0 || njobs > 3) return cudaErrorInvalidValue;
    for (int i = 0; i < njobs; ++i) {
        if (jobs[i].ncols > kFinRowMaxCols || jobs[i].ncols % 4 || jobs[i].group % 4) return cudaErrorInvalidValue;
        js.j[i] = jobs[i];
    }
    FinSide sd{};
    if (side) sd = *side;
    const int64_t row_blocks = (T + kFinRowTile - 1) / kFinRowTile;
    // side blocks: about one resident wave (three CTAs per SM at this kernel's register count), each
    // looping over its share
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 152;  // (a GB300's count; only the side blocks' number depends on it)
    int64_t side_blocks = 0;
    if (sd.bd_out) side_blocks = (2 * sd.bd_n * (2 * sd.bd_rp / 8) + 255) / 256;
    if (sd.nf4_jobs > 0) side_blocks = std::max<int64_t>(side_blocks, nf4_scale_tiles(sd.nf4, sd.nf4_jobs));
    side_blocks = std::min<int64_t>(side_blocks, 3 * (int64_t)sms);
    const int64_t blocks = njobs * row_blocks + side_blocks;
    if (blocks == 0) return cudaSuccess;
    // (the kernel divides by row_blocks only for blocks below njobs * row_blocks, so 0 is safe)
    return launch_pdl(fin_rowproj_kernel, dim3((unsigned)blocks), dim3(256), 0, st, nullptr, 0, js, njobs, T, row_blocks,
                      side_blocks, sd);
}

struct FinColJobs {
    FinColJob j[kMaxFinColJobs];
};

// One CTA per 32 columns of one job.  The columns' partial rows are read with coalesced 16-byte
// loads (4-wide chunk of j fastest; rp and ldp are multiples of 4) and summed over the splits in
// split order.  The dB layout out[c][j] of 32 columns is one contiguous span, written directly;
// the dA layout out[j][c] goes through a shared-memory tile so that each output row gets 32
// contiguous values.
constexpr int kFinColTile = 32;
constexpr int kFinColMaxRp = 64;
__global__ void __launch_bounds__(256) fin_colreduce_kernel(FinColJobs jobs) {
    __shared__ float tile[kFinColMaxRp * (kFinColTile + 1)];  // [j][column], padded pitch
    griddep_launch_dependents();
    griddep_wait();
    const FinColJob& J = jobs.j[blockIdx.y];
    const int64_t c0 = (int64_t)blockIdx.x * kFinColTile;
    if (c0 >= J.C) return;
    const int cols = J.C - c0 < kFinColTile ? (int)(J.C - c0) : kFinColTile;
    const int nchunk = J.rp / 4;
    const int pitch = kFinColTile + 1;
    for (int i = threadIdx.x; i < cols * nchunk; i += blockDim.x) {
        const int cl = i / nchunk, j0 = 4 * (i - cl * nchunk);
        if (j0 >= J.r) continue;
        const int64_t c = c0 + cl;
        const float4 a = sum_splits(J.part + c * J.ldp + j0, J.split_stride, J.splits);
        const float v[4] = {a.x, a.y, a.z, a.w};
        const int nj = min(4, J.r - j0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k < nj) {
                if (J.transposed) tile[(j0 + k) * pitch + cl] = v[k];
                else J.out[c * J.r + j0 + k] = v[k];  // out[c][j]
            }
    }
    if (!J.transposed) return;  // (uniform across the CTA: one job per blockIdx.y)
    __syncthreads();
    for (int i = threadIdx.x; i < J.r * kFinColTile; i += blockDim.x) {
        const int j = i / kFinColTile, cl = i - j * kFinColTile;
        if (cl < cols) J.out[(int64_t)j * J.C + c0 + cl] = tile[j * pitch + cl];  // out[j][c]
    }
}

cudaError_t launch_fin_colreduce(const FinColJob* jobs, int njobs, cudaStream_t st) {
    if (njobs < 1 || njobs > kMaxFinColJobs) return cudaErrorInvalidValue;
    FinColJobs js{};
    int64_t most = 0;
    for (int i = 0; i < njobs; ++i) {
        if (jobs[i].rp > kFinColMaxRp || jobs[i].rp % 4 || jobs[i].ldp % 4 || jobs[i].r > jobs[i].rp)
            return cudaErrorInvalidValue;
        js.j[i] = jobs[i];
        most = std::max<int64_t>(most, jobs[i].C);
    }
    const int64_t blocks = (most + kFinColTile - 1) / kFinColTile;
    return launch_pdl(fin_colreduce_kernel, dim3((unsigned)std::max<int64_t>(blocks, 1), njobs), dim3(256), 0, st, nullptr,
                      0, js);
}

// ------------------------------------------------------------------ fp32 LoRA parameters
// fp32 -> bf16 bits, round to nearest even (the GEMM input precision of fp32 LoRA parameters);
// blockIdx.y picks the matrix
__global__ void __launch_bounds__(256) f32_to_bf16_kernel(CvtJobs jobs) {
    griddep_launch_dependents();
    griddep_wait();
    const CvtJob& J = jobs.j[blockIdx.y];
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < J.n; i += (int64_t)gridDim.x * blockDim.x) {
        const __nv_bfloat16 b = __float2bfloat16_rn(J.in[i]);
        J.out[i] = *reinterpret_cast<const uint16_t*>(&b);
    }
}

cudaError_t launch_f32_to_bf16(const CvtJobs& jobs, int njobs, cudaStream_t st) {
    int64_t most = 0;
    for (int i = 0; i < njobs; ++i) most = std::max<int64_t>(most, jobs.j[i].n);
    if (njobs == 0 || most == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((most + 255) / 256, 256);
    return launch_pdl(f32_to_bf16_kernel, dim3((unsigned)blocks, (unsigned)njobs), dim3(256), 0, st, nullptr, 0, jobs);
}

// ------------------------------------------------------------------ split tail tiles
// One thread per 4 columns of a tail-tile row; 512-row tiles, bn and N multiples of 4.
__global__ void __launch_bounds__(256) tail_fin_kernel(TailFin f) {
    griddep_launch_dependents();
    griddep_wait();
    const int c4n = f.bn / 4;
    const int64_t total = (int64_t)f.ntail * 512 * c4n;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int c4 = (int)(idx % c4n);
        const int64_t rt = idx / c4n;
        const int row = (int)(rt % 512);
        const int t = (int)(rt / 512);
        int mb, nb;
        raster_tile(f.tail_begin + t, f.tiles_m, f.tiles_n, f.group_m, mb, nb);
        const int64_t m = (int64_t)mb * 512 + row;
        const int64_t gcol = (int64_t)nb * f.out_col_step + c4 * 4;
        if (m >= f.M || gcol >= f.N) continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < f.splits; ++k) {
            const float4 v =
                *reinterpret_cast<const float4*>(f.part + ((int64_t)(t * f.splits + k) * 512 + row) * f.bn + c4 * 4);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        *reinterpret_cast<uint2*>(f.out + m * f.ld_out + gcol) =
            make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
}

cudaError_t launch_tail_fin(const TailFin& f, cudaStream_t st) {
    const int64_t total = (int64_t)f.ntail * 512 * (f.bn / 4);
    if (total == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, 4096);
    return launch_pdl(tail_fin_kernel, dim3((unsigned)blocks), dim3(256), 0, st, nullptr, 0, f);
}

// ------------------------------------------------------------------ block-diagonal rank-r operand
// [Bg | 0 ; 0 | Bu] (2n x 2rp bf16): one thread per 8 consecutive columns of a row (one 16-byte
// store); 2rp is a multiple of 32.
// Rows [first, ...) step `stride` of the flattened (row, 8-column group) index of [B_g 0; 0 B_u]
__device__ void blockdiag_rows(const uint16_t* __restrict__ Bg, const uint16_t* __restrict__ Bu, int64_t n, int r,
                               int rp, uint16_t* __restrict__ out, int64_t first, int64_t stride) {
    const int groups = (2 * rp) / 8;
    const int64_t total = 2 * n * groups;
    for (int64_t idx = first; idx < total; idx += stride) {
        const int64_t row = idx / groups;
        const int c0 = (int)(idx - row * groups) * 8;
        const bool upper = row < n;
        const uint16_t* src = upper ? Bg + row * r : Bu + (row - n) * r;
        const int off = upper ? 0 : rp;  // first output column of this row's block
        uint16_t v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + i - off;
            v[i] = (c >= 0 && c < r) ? src[c] : (uint16_t)0;
        }
        *reinterpret_cast<uint4*>(out + row * 2 * rp + c0) =
            make_uint4(v[0] | ((uint32_t)v[1] << 16), v[2] | ((uint32_t)v[3] << 16), v[4] | ((uint32_t)v[5] << 16),
                       v[6] | ((uint32_t)v[7] << 16));
    }
}

// ------------------------------------------------------------------ NF4
static const float* const kNf4Code = kNf4Values;

void nf4_codebook_host(float* out16) {
    for (int i = 0; i < 16; ++i) out16[i] = kNf4Code[i];
}

struct Nf4Tables {
    float code[16];
    // thr[i] = the smallest fp32 strictly above the exact midpoint of code[i] and code[i+1]:
    // for an fp32 v, (v >= thr[i]) <=> (v is strictly closer to code[i+1] than to code[i]),
    // so an exact tie stays with the lower index.
    float thr[15];
};

static Nf4Tables make_tables() {
    Nf4Tables t;
    for (int i = 0; i < 16; ++i) t.code[i] = kNf4Code[i];
    for (int i = 0; i < 15; ++i) {
        const double mid = 0.5 * ((double)kNf4Code[i] + (double)kNf4Code[i + 1]);  // exact
        float f = (float)mid;
        if ((double)f <= mid) f = std::nextafter(f, INFINITY);
        t.thr[i] = f;
    }
    return t;
}

// One CTA per group of 256 blocks (16384 elements); thread t quantises block t.
__global__ void __launch_bounds__(256) nf4_pack_kernel(const uint16_t* __restrict__ W,
                                                       uint8_t* __restrict__ codes,
                                                       int8_t* __restrict__ absmax_q,
                                                       float* __restrict__ scale, Nf4Tables tb) {
    __shared__ float wmax[8];
    const int64_t g = blockIdx.x;
    const int t = threadIdx.x;
    const int64_t b = g * 256 + t;
    const uint4* src = reinterpret_cast<const uint4*>(W + b * 64);
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = __ldg(src + i);
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(w[i])), fabsf(bf16hi(w[i]))));
    float m = amax;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((t & 31) == 0) wmax[t >> 5] = m;
    __syncthreads();
    float gmax = wmax[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) gmax = fmaxf(gmax, wmax[i]);
    const float c = __fdiv_rn(gmax, 127.0f);
    if (t == 0) scale[g] = c;
    int q = 0;
    if (c > 0.0f) {
        q = (int)rintf(__fdiv_rn(amax, c));
        q = min(max(q, 0), 127);
    }
    absmax_q[b] = (int8_t)q;

    uint32_t packed[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) packed[i] = 0;
#pragma unroll
    for (int e = 0; e < 64; ++e) {
        const uint32_t word = w[e >> 1];
        const float x = (e & 1) ? bf16hi(word) : bf16lo(word);
        const float v = amax > 0.0f ? __fdiv_rn(x, amax) : 0.0f;
        uint32_t idx = 0;
#pragma unroll
        for (int k = 0; k < 15; ++k) idx += (v >= tb.thr[k]) ? 1u : 0u;
        // element 2i -> high nibble of byte i; byte i sits at bits 8*(i%4) of word i/4
        const int byte = e >> 1;
        const uint32_t nib = (e & 1) ? idx : (idx << 4);
        packed[byte >> 2] |= nib << (8 * (byte & 3));
    }
    uint4* dst = reinterpret_cast<uint4*>(codes + b * 32);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
}

cudaError_t launch_nf4_pack(const uint16_t* W, int64_t numel, uint8_t* codes, int8_t* absmax_q,
                            float* scale, cudaStream_t st) {
    static const Nf4Tables tb = make_tables();
    const int64_t groups = numel / 16384;
    if (groups == 0) return cudaSuccess;
    nf4_pack_kernel<<<(unsigned)groups, 256, 0, st>>>(W, codes, absmax_q, scale, tb);
    return cudaGetLastError();
}

// Each thread decodes 8 elements (4 code bytes).
__global__ void __launch_bounds__(256) nf4_dequant_kernel(const uint32_t* __restrict__ codes,
                                                          const int8_t* __restrict__ absmax_q,
                                                          const float* __restrict__ scale,
                                                          int64_t n8, int bf16_out, void* out,
                                                          Nf4Tables tb) {
    __shared__ float cb[16];
    if (threadIdx.x < 16) cb[threadIdx.x] = tb.code[threadIdx.x];
    __syncthreads();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t c4 = __ldg(codes + i);
        const int64_t blk = i >> 3;  // 8 elements per thread, 64 per block
        const float amax = __fmul_rn((float)__ldg(absmax_q + blk), __ldg(scale + (blk >> 8)));
        float w[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t byte = (c4 >> (8 * k)) & 0xFFu;
            w[2 * k] = __fmul_rn(cb[byte >> 4], amax);
            w[2 * k + 1] = __fmul_rn(cb[byte & 15u], amax);
        }
        if (bf16_out) {
            uint4 v;
            v.x = pack_bf16x2(w[0], w[1]);
            v.y = pack_bf16x2(w[2], w[3]);
            v.z = pack_bf16x2(w[4], w[5]);
            v.w = pack_bf16x2(w[6], w[7]);
            reinterpret_cast<uint4*>(out)[i] = v;
        } else {
            float4* o = reinterpret_cast<float4*>(out) + 2 * i;
            o[0] = make_float4(w[0], w[1], w[2], w[3]);
            o[1] = make_float4(w[4], w[5], w[6], w[7]);
        }
    }
}

cudaError_t launch_nf4_dequant(const uint8_t* codes, const int8_t* absmax_q, const float* scale,
                               int64_t numel, bool bf16_out, void* out, cudaStream_t st) {
    static const Nf4Tables tb = make_tables();
    const int64_t n8 = numel / 8;
    if (n8 == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, (int64_t)sms * 8);
    nf4_dequant_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const uint32_t*>(codes), absmax_q,
                                                          scale, n8, bf16_out ? 1 : 0, out, tb);
    return cudaGetLastError();
}

// Block-scale table of an NF4 weight (rows x cols): table[kb * rows + row] = fp32(absmax_q[b] *
// group_scale[b / 256]) with b = row * (cols / 64) + kb, the scale of 64-element block kb of row
// `row` (QLoRA, "Double Quantization").  Laid out K-block-major so that one TMA box brings a
// stage's scales next to its codes: 128 rows of one K block (weight read K-major), or 64 rows of
// two 64-wide column blocks (weight read MN-major).
// One CTA per 64-row x 64-K-block tile of one job: the int8 block scales are read along K (64
// consecutive bytes of a row) and the table is written along rows (64 consecutive floats of a K
// block), transposed through shared memory, so both sides are coalesced.
__device__ void nf4_scale_tile(const Nf4ScaleJobs& jobs, int njobs, int t, float (*tile)[65]) {
    int j = 0;
    for (; j < njobs; ++j) {
        const int tiles = (int)(((jobs.j[j].rows + 63) / 64) * ((jobs.j[j].kblocks + 63) / 64));
        if (t < tiles) break;
        t -= tiles;
    }
    if (j == njobs) return;
    const Nf4ScaleJob& J = jobs.j[j];
    const int64_t tk = (J.kblocks + 63) / 64;
    const int64_t r0 = (t / tk) * 64, k0 = (t % tk) * 64;
    // read: rows of 64 consecutive K blocks, four per thread: one 32-bit load of the four codes when
    // they are inside the row and 4-byte aligned (then one group scale serves all four: 256 is a
    // multiple of 4), else byte by byte.  The loads of all four iterations are issued first.
    uint32_t q4[4];
    float g4[4];
    bool whole[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int i = threadIdx.x + 256 * it;
        const int rr = i >> 4, kk = (i & 15) * 4;
        const int64_t row = r0 + rr, kb = k0 + kk;
        const int64_t b = row * J.kblocks + kb;
        whole[it] = row < J.rows && kb + 4 <= J.kblocks && (b & 3) == 0;
        q4[it] = whole[it] ? __ldg(reinterpret_cast<const uint32_t*>(J.absmax_q + b)) : 0u;
        g4[it] = whole[it] ? __ldg(J.scale + (b >> 8)) : 0.0f;
    }
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int i = threadIdx.x + 256 * it;
        const int rr = i >> 4, kk = (i & 15) * 4;
        const int64_t row = r0 + rr, kb = k0 + kk;
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (whole[it]) {
#pragma unroll
            for (int c = 0; c < 4; ++c) v[c] = __fmul_rn((float)(int8_t)(q4[it] >> (8 * c)), g4[it]);
        } else if (row < J.rows) {
            const int64_t b = row * J.kblocks + kb;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (kb + c < J.kblocks)
                    v[c] = __fmul_rn((float)__ldg(J.absmax_q + b + c), __ldg(J.scale + ((b + c) >> 8)));
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) tile[kk + c][rr] = v[c];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 64 * 64; i += 256) {  // write: K blocks of 64 consecutive rows
        const int kk = i >> 6, rr = i & 63;
        const int64_t row = r0 + rr, kb = k0 + kk;
        if (row < J.rows && kb < J.kblocks) J.table[kb * J.rows + row] = tile[kk][rr];
    }
}


// ------------------------------------------------------------------ int4 groupwise base
// "loralei" README, QLoRA section (int4 base, groups of 32 to 256 elements of a row): asymmetric
// min/max quantisation with a bf16 scale s and a bf16 zero z (the value of the middle code 8):
//   s = bf16(fp32((mx - mn) / 15)), z = bf16(fp32(mn + 8 s)),
//   q = clamp(rint(fp32(fp32(x - z) / s)) + 8, 0, 15)   (q = 8 when s == 0),
// codes packed as for NF4, (s, z) stored as one 32-bit word (s low, z high) at sz[g * rows + row].

__device__ __forceinline__ uint32_t bf16_bits_rn(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// one thread per group; two passes over the group's bf16 values (range, then codes)
__global__ void __launch_bounds__(256) int4_pack_kernel(const uint16_t* __restrict__ W, int64_t rows,
                                                        int64_t cols, int group, uint8_t* __restrict__ codes,
                                                        uint32_t* __restrict__ sz) {
    const int64_t ng = cols / group;
    const int64_t n = rows * ng;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / ng, g = i - row * ng;
        const int64_t e0 = row * cols + g * group;
        const uint4* src = reinterpret_cast<const uint4*>(W + e0);
        float mn = INFINITY, mx = -INFINITY;
        for (int c = 0; c < group / 8; ++c) {
            const uint4 v = __ldg(src + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mn = fminf(mn, fminf(bf16lo(w[k]), bf16hi(w[k])));
                mx = fmaxf(mx, fmaxf(bf16lo(w[k]), bf16hi(w[k])));
            }
        }
        const uint32_t sb = bf16_bits_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
        const float s = __uint_as_float(sb << 16);
        const uint32_t zb = bf16_bits_rn(__fadd_rn(mn, __fmul_rn(8.0f, s)));
        const float z = __uint_as_float(zb << 16);
        sz[g * rows + row] = sb | (zb << 16);
        uint32_t* dst = reinterpret_cast<uint32_t*>(codes + e0 / 2);
        for (int c = 0; c < group / 8; ++c) {
            const uint4 v = __ldg(src + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t packed = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float x = (e & 1) ? bf16hi(w[e >> 1]) : bf16lo(w[e >> 1]);
                uint32_t q = 8;
                if (s > 0.0f) {
                    const float r = rintf(__fdiv_rn(__fsub_rn(x, z), s)) + 8.0f;
                    q = (uint32_t)fminf(fmaxf(r, 0.0f), 15.0f);
                }
                // element 2i -> high nibble of byte i; byte i at bits 8 * i of the word
                packed |= ((e & 1) ? q : (q << 4)) << (8 * (e >> 1));
            }
            dst[c] = packed;
        }
    }
}

cudaError_t launch_int4_pack(const uint16_t* W, int64_t rows, int64_t cols, int group, uint8_t* codes,
                             uint32_t* sz, cudaStream_t st) {
    const int64_t n = rows * (cols / group);
    if (n == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)sms * 8);
    int4_pack_kernel<<<(unsigned)blocks, 256, 0, st>>>(W, rows, cols, group, codes, sz);
    return cudaGetLastError();
}

// Each thread decodes 8 elements (4 code bytes) of one group: w = fp32((q - 8) s + z), one
// rounding ((q - 8) s is exact).
__global__ void __launch_bounds__(256) int4_dequant_kernel(const uint32_t* __restrict__ codes,
                                                           const uint32_t* __restrict__ sz, int64_t rows,
                                                           int64_t cols, int group, int bf16_out, void* out) {
    const int64_t n8 = rows * cols / 8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e0 = i * 8, row = e0 / cols, g = (e0 - row * cols) / group;
        const uint32_t word = __ldg(sz + g * rows + row);
        const float s = __uint_as_float(word << 16), z = __uint_as_float(word & 0xFFFF0000u);
        const uint32_t c4 = __ldg(codes + i);
        float w[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t byte = (c4 >> (8 * k)) & 0xFFu;
            w[2 * k] = __fmaf_rn((float)((int)(byte >> 4) - 8), s, z);
            w[2 * k + 1] = __fmaf_rn((float)((int)(byte & 15u) - 8), s, z);
        }
        if (bf16_out) {
            uint4 v;
            v.x = pack_bf16x2(w[0], w[1]);
            v.y = pack_bf16x2(w[2], w[3]);
            v.z = pack_bf16x2(w[4], w[5]);
            v.w = pack_bf16x2(w[6], w[7]);
            reinterpret_cast<uint4*>(out)[i] = v;
        } else {
            float4* o = reinterpret_cast<float4*>(out) + 2 * i;
            o[0] = make_float4(w[0], w[1], w[2], w[3]);
            o[1] = make_float4(w[4], w[5], w[6], w[7]);
        }
    }
}

cudaError_t launch_int4_dequant(const uint8_t* codes, const uint32_t* sz, int64_t rows, int64_t cols, int group,
                                bool bf16_out, void* out, cudaStream_t st) {
    const int64_t n8 = rows * cols / 8;
    if (n8 == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, (int64_t)sms * 8);
    int4_dequant_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const uint32_t*>(codes), sz, rows, cols,
                                                           group, bf16_out ? 1 : 0, out);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ NVFP4 weight-only base
// E2M1 codes (element 2i in the low nibble of byte i), one E4M3 scale per 16 elements of a row
// stored as sf[((col / 64) * rows + row) * 4 + (col % 64) / 16], and one fp32 tensor scale
// S_g = amax / (6 * 448) (1 when that is 0).  Per block: s_b = E4M3(fp32(fp32(bmax / 6) / S_g)),
// nearest, ties to even, saturated at 448; per element: code = E2M1(fp32(x / fp32(s_b * S_g))),
// nearest, ties to even, saturated at 6, sign of x (all codes 0 when s_b * S_g == 0).

// value of an E4M3 byte (finite encodings; exact)
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    const float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
    return (b & 0x80u) ? -mag : mag;
}

// nearest E4M3 byte of d >= 0, ties to even, saturated at 448 (byte 126)
__device__ __forceinline__ uint32_t f32_to_e4m3_sat(float d) {
    if (!(d < 448.0f)) return 126u;
    if (d < 0.015625f) return (uint32_t)rintf(d * 512.0f);  // subnormal steps of 2^-9 (8 -> 2^-6)
    uint32_t u = __float_as_uint(d);
    u += 0x7FFFFu + ((u >> 20) & 1u);                        // round the mantissa to 3 bits, even
    return min((u >> 20) - 960u, 126u);                      // rebias the exponent from 127 to 7
}

// nearest E2M1 code of y, ties to even, saturated at 6, sign bit of y
__device__ __forceinline__ uint32_t f32_to_e2m1_sat(float y) {
    const float a = fabsf(y);
    const uint32_t i = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
    return i | (signbit(y) ? 8u : 0u);
}

__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    const float mag = e ? __uint_as_float(((e + 126u) << 23) | (m << 22)) : (m ? 0.5f : 0.0f);
    return (c & 8u) ? -mag : mag;
}

__device__ __forceinline__ float nvfp4_tensor_scale(float amax) {
    const float sg = __fdiv_rn(amax, 2688.0f);
    return sg > 0.0f ? sg : 1.0f;
}

__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const uint4* __restrict__ W, int64_t n8,
                                                         uint32_t* __restrict__ amax_bits) {
    float m = 0.0f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldg(W + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) m = fmaxf(m, fmaxf(fabsf(bf16lo(w[k])), fabsf(bf16hi(w[k]))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));  // non-negative: bits order as values
}

// one thread per 16-element block
__global__ void __launch_bounds__(256) nvfp4_pack_kernel(const uint16_t* __restrict__ W, int64_t rows, int64_t cols,
                                                         const uint32_t* __restrict__ amax_bits,
                                                         uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
    const float sg = nvfp4_tensor_scale(__uint_as_float(__ldg(amax_bits)));
    const int64_t nbr = cols / 16, n = rows * nbr;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / nbr, b = i - row * nbr;
        const uint4* src = reinterpret_cast<const uint4*>(W + row * cols + b * 16);
        const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float bmax = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) bmax = fmaxf(bmax, fmaxf(fabsf(bf16lo(w[k])), fabsf(bf16hi(w[k]))));
        const uint32_t sb = f32_to_e4m3_sat(__fdiv_rn(__fdiv_rn(bmax, 6.0f), sg));
        const float S = __fmul_rn(e4m3_to_f32(sb), sg);
        uint32_t packed[2] = {0u, 0u};
        if (S > 0.0f) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float x = (e & 1) ? bf16hi(w[e >> 1]) : bf16lo(w[e >> 1]);
                const uint32_t c = f32_to_e2m1_sat(__fdiv_rn(x, S));
                packed[e >> 3] |= c << (4 * (e & 7));  // element 2i low nibble of byte i
            }
        }
        *reinterpret_cast<uint2*>(codes + (row * cols + b * 16) / 2) = make_uint2(packed[0], packed[1]);
        sf[((b >> 2) * rows + row) * 4 + (b & 3)] = (uint8_t)sb;
    }
}

__global__ void nvfp4_scale_kernel(float* gs) {
    *gs = nvfp4_tensor_scale(__uint_as_float(*reinterpret_cast<const uint32_t*>(gs)));
}

cudaError_t launch_nvfp4_pack(const uint16_t* W, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* sf, float* gs,
                              cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(gs, 0, sizeof(float), st);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t n8 = rows * cols / 8, nb = rows * cols / 16;
    uint32_t* amax_bits = reinterpret_cast<uint32_t*>(gs);  // holds the tensor amax until the last launch
    nvfp4_amax_kernel<<<(unsigned)std::min<int64_t>((n8 + 255) / 256, (int64_t)sms * 8), 256, 0, st>>>(
        reinterpret_cast<const uint4*>(W), n8, amax_bits);
    nvfp4_pack_kernel<<<(unsigned)std::min<int64_t>((nb + 255) / 256, (int64_t)sms * 8), 256, 0, st>>>(
        W, rows, cols, amax_bits, codes, sf);
    nvfp4_scale_kernel<<<1, 1, 0, st>>>(gs);
    return cudaGetLastError();
}

// Each thread decodes 8 elements (4 code bytes): w = fp32(e2m1 * fp32(s_b * S_g)).
__global__ void __launch_bounds__(256) nvfp4_dequant_kernel(const uint32_t* __restrict__ codes,
                                                            const uint8_t* __restrict__ sf,
                                                            const float* __restrict__ gs, int64_t rows,
                                                            int64_t cols, int bf16_out, void* out) {
    const float sg = __ldg(gs);
    const int64_t n8 = rows * cols / 8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e0 = i * 8, row = e0 / cols, col = e0 - row * cols;
        const float S = __fmul_rn(e4m3_to_f32(__ldg(sf + ((col >> 6) * rows + row) * 4 + ((col & 63) >> 4))), sg);
        const uint32_t c8 = __ldg(codes + i);
        float w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = __fmul_rn(e2m1_to_f32((c8 >> (4 * k)) & 15u), S);
        if (bf16_out) {
            uint4 v;
            v.x = pack_bf16x2(w[0], w[1]);
            v.y = pack_bf16x2(w[2], w[3]);
            v.z = pack_bf16x2(w[4], w[5]);
            v.w = pack_bf16x2(w[6], w[7]);
            reinterpret_cast<uint4*>(out)[i] = v;
        } else {
            float4* o = reinterpret_cast<float4*>(out) + 2 * i;
            o[0] = make_float4(w[0], w[1], w[2], w[3]);
            o[1] = make_float4(w[4], w[5], w[6], w[7]);
        }
    }
}

cudaError_t launch_nvfp4_dequant(const uint8_t* codes, const uint8_t* sf, const float* gs, int64_t rows, int64_t cols,
                                 bool bf16_out, void* out, cudaStream_t st) {
    const int64_t n8 = rows * cols / 8;
    if (n8 == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, (int64_t)sms * 8);
    nvfp4_dequant_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const uint32_t*>(codes), sf, gs, rows,
                                                            cols, bf16_out ? 1 : 0, out);
    return cudaGetLastError();
}

}  // namespace lm
