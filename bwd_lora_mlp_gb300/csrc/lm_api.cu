// C ABI of liblora_mlp.so: argument validation, workspace planning, TMA descriptor set-up
// and the kernel sequence of each entry point.  See include/lora_mlp.h for the contract.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <string>
#include <vector>

#include "lm_internal.h"
#include "lora_mlp.h"

using namespace lm;

namespace {

thread_local char g_err[768] = "";
// test hook (lm_debug_inject): kernel families whose producers issue no loads (bits 0-3), the dual
// rank-r reductions wherever feasible (bit 4), and the wait limit
constexpr int32_t kForceDual = 16;
thread_local int32_t g_inject_mask = 0;
thread_local uint64_t g_wait_ns = 0;

lm_status fail(lm_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

#define LM_TRY(expr)                      \
    do {                                  \
        const lm_status _s = (expr);      \
        if (_s != LM_OK) return _s;       \
    } while (0)

lm_status cuda_fail(cudaError_t e, const char* what) {
    return fail(LM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define LM_CUDA(expr, what)                                \
    do {                                                   \
        const cudaError_t _e = (expr);                     \
        if (_e != cudaSuccess) return cuda_fail(_e, what); \
    } while (0)

// ------------------------------------------------------------------ tracing
struct ProfRec {
    const char* tag;
    cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
    if (!g_prof_pool.empty()) {
        cudaEvent_t e = g_prof_pool.back();
        g_prof_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Records an event pair around the kernel launched inside its lifetime (when tracing is on).
struct ProfScope {
    ProfRec rec{};
    bool on = false;
    cudaStream_t st;
    ProfScope(const char* tag, cudaStream_t s) : st(s) {
        std::lock_guard<std::mutex> g(g_prof_mu);
        if (!g_prof_on) return;
        rec.tag = tag;
        rec.a = prof_event();
        rec.b = prof_event();
        on = rec.a && rec.b && cudaEventRecord(rec.a, st) == cudaSuccess;
    }
    ~ProfScope() {
        if (!on) return;
        cudaEventRecord(rec.b, st);
        std::lock_guard<std::mutex> g(g_prof_mu);
        g_prof.push_back(rec);
    }
};

// ------------------------------------------------------------------ device / driver entry
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

lm_status get_encode() {
    if (g_encode) return LM_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return fail(LM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return LM_OK;
}

lm_status device_sms(int* sms) {
    static int cached[64] = {0};  // 0 unknown, > 0 SM count, -1 unsupported
    int dev = 0;
    LM_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(LM_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    if (cached[dev] == 0) {
        int major = 0, minor = 0, n = 0;
        LM_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "cudaDeviceGetAttribute");
        LM_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "cudaDeviceGetAttribute");
        LM_CUDA(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
        cached[dev] = (major == 10 && minor == 3) ? n : -1;
    }
    if (cached[dev] < 0)
        return fail(LM_ERR_UNSUPPORTED, "device %d is not compute capability 10.3; the kernels are built for sm_103a", dev);
    *sms = cached[dev];
    return LM_OK;
}

lm_status ready(int* sms) {
    LM_TRY(device_sms(sms));
    return get_encode();
}

// ------------------------------------------------------------------ validation
// 32 bytes: TMA wants 16, the epilogues read and write 32-byte chunks of rows
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

lm_status need_ptr(const void* p, const char* name) {
    if (!p) return fail(LM_ERR_NULL, "%s is NULL", name);
    if (!aligned32(p)) return fail(LM_ERR_ALIGN, "%s is not 32-byte aligned", name);
    return LM_OK;
}

// a scalar the kernels read with a plain load (no TMA): 4-byte alignment
lm_status need_ptr4(const void* p, const char* name) {
    if (!p) return fail(LM_ERR_NULL, "%s is NULL", name);
    if (reinterpret_cast<uintptr_t>(p) % 4 != 0) return fail(LM_ERR_ALIGN, "%s is not 4-byte aligned", name);
    return LM_OK;
}

lm_status check_dim(int64_t v, const char* name) {
    if (v <= 0 || v % 32 != 0 || v > (int64_t(1) << 20))
        return fail(LM_ERR_SHAPE, "%s = %lld must be a positive multiple of 32 (at most 2^20)", name, (long long)v);
    return LM_OK;
}

lm_status check_T(int64_t T) {
    if (T < 0 || T > (int64_t(1) << 30)) return fail(LM_ERR_SHAPE, "T = %lld out of range", (long long)T);
    return LM_OK;
}

lm_status check_r(int32_t r) {
    if (r < 8 || r > 64 || r % 8 != 0) return fail(LM_ERR_SHAPE, "r = %d must be a multiple of 8 in [8, 64]", r);
    return LM_OK;
}

lm_status check_lora(const lm_lora* L, const char* name, int64_t in, int64_t out, int32_t r) {
    if (!L) return fail(LM_ERR_NULL, "%s is NULL", name);
    if (L->r != r) return fail(LM_ERR_SHAPE, "%s.r = %d differs from r = %d", name, L->r, r);
    if (L->W.rows != out || L->W.cols != in)
        return fail(LM_ERR_SHAPE, "%s.W is %lld x %lld, expected %lld x %lld (out x in)", name, (long long)L->W.rows,
                    (long long)L->W.cols, (long long)out, (long long)in);
    if (!std::isfinite(L->s)) return fail(LM_ERR_SHAPE, "%s.s is not finite", name);
    char buf[64];
    if (L->W.kind == LM_WEIGHT_BF16) {
        snprintf(buf, sizeof buf, "%s.W.w", name);
        LM_TRY(need_ptr(L->W.w, buf));
    } else if (L->W.kind == LM_WEIGHT_NF4) {
        if ((L->W.rows * L->W.cols) % 16384 != 0 || L->W.cols % 64 != 0)
            return fail(LM_ERR_SHAPE, "%s: an NF4 weight needs rows*cols %% 16384 == 0 and cols %% 64 == 0", name);
        snprintf(buf, sizeof buf, "%s.W.codes", name);
        LM_TRY(need_ptr(L->W.codes, buf));
        snprintf(buf, sizeof buf, "%s.W.absmax_q", name);
        LM_TRY(need_ptr(L->W.absmax_q, buf));
        snprintf(buf, sizeof buf, "%s.W.group_scale", name);
        LM_TRY(need_ptr(L->W.group_scale, buf));
    } else if (L->W.kind == LM_WEIGHT_INT4) {
        const int32_t G = L->W.group;
        if (G != 32 && G != 64 && G != 128 && G != 256)
            return fail(LM_ERR_SHAPE, "%s.W.group = %d: an int4 group holds 32, 64, 128 or 256 elements", name, G);
        if (L->W.cols % 64 != 0 || L->W.cols % G != 0)
            return fail(LM_ERR_SHAPE, "%s: an int4 weight needs cols %% 64 == 0 and cols %% group == 0", name);
        snprintf(buf, sizeof buf, "%s.W.codes", name);
        LM_TRY(need_ptr(L->W.codes, buf));
        snprintf(buf, sizeof buf, "%s.W.scale_zero", name);
        LM_TRY(need_ptr(L->W.scale_zero, buf));
    } else if (L->W.kind == LM_WEIGHT_NVFP4) {
        if (L->W.cols % 64 != 0) return fail(LM_ERR_SHAPE, "%s: an NVFP4 weight needs cols %% 64 == 0", name);
        snprintf(buf, sizeof buf, "%s.W.codes", name);
        LM_TRY(need_ptr(L->W.codes, buf));
        snprintf(buf, sizeof buf, "%s.W.block_scale", name);
        LM_TRY(need_ptr(L->W.block_scale, buf));
        snprintf(buf, sizeof buf, "%s.W.global_scale", name);
        LM_TRY(need_ptr4(L->W.global_scale, buf));
    } else {
        return fail(LM_ERR_DTYPE, "%s.W.kind = %d is not a known weight kind", name, L->W.kind);
    }
    if (L->ab_dtype != LM_AB_BF16 && L->ab_dtype != LM_AB_F32)
        return fail(LM_ERR_DTYPE, "%s.ab_dtype = %d is not a known A/B dtype", name, L->ab_dtype);
    snprintf(buf, sizeof buf, "%s.A", name);
    LM_TRY(need_ptr(L->A, buf));
    snprintf(buf, sizeof buf, "%s.B", name);
    LM_TRY(need_ptr(L->B, buf));
    return LM_OK;
}

// bytes of `elems` elements of a LoRA A or B matrix
size_t ab_bytes(const lm_lora* L, int64_t elems) { return (size_t)elems * (L->ab_dtype == LM_AB_F32 ? 4 : 2); }
inline const uint16_t* bf(const void* p) { return static_cast<const uint16_t*>(p); }

struct Span {
    const void* p;
    size_t bytes;
    const char* name;
};

bool overlap(const Span& a, const Span& b) {
    if (!a.p || !b.p || !a.bytes || !b.bytes) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// every output against every input and every other output
lm_status check_alias(std::initializer_list<Span> outs, std::initializer_list<Span> ins) {
    const Span* o = outs.begin();
    for (size_t i = 0; i < outs.size(); ++i) {
        for (const Span& in : ins)
            if (overlap(o[i], in)) return fail(LM_ERR_ALIAS, "%s overlaps %s", o[i].name, in.name);
        for (size_t j = i + 1; j < outs.size(); ++j)
            if (overlap(o[i], o[j])) return fail(LM_ERR_ALIAS, "%s overlaps %s", o[i].name, o[j].name);
    }
    return LM_OK;
}

Span wspan(const lm_lora* L, const char* name) {
    if (L->W.kind != LM_WEIGHT_BF16) return Span{L->W.codes, (size_t)(L->W.rows * L->W.cols / 2), name};
    return Span{L->W.w, (size_t)(L->W.rows * L->W.cols * 2), name};
}

// every projection of one call must use the same kind of base weight
// (*q4: a packed 4-bit base, NF4, int4 or NVFP4, decoded inside the GEMM mainloop)
lm_status same_kind(std::initializer_list<const lm_lora*> Ls, bool* q4) {
    const lm_lora* first = *Ls.begin();
    for (const lm_lora* L : Ls)
        if (L->W.kind != first->W.kind)
            return fail(LM_ERR_UNSUPPORTED, "the projections of one call mix base weight kinds (%d and %d)",
                        first->W.kind, L->W.kind);
    *q4 = first->W.kind != LM_WEIGHT_BF16;
    return LM_OK;
}

// ------------------------------------------------------------------ workspace planning
int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
// bf16 elements of the converted A and B of one projection (fp32 LoRA parameters)
int64_t ab_elems(int64_t r, int64_t in, int64_t out) { return round_up(r * in, 128) + round_up(out * r, 128); }

struct Bump {
    size_t off = 0;
    size_t take(size_t bytes) {
        off = (off + 255) & ~size_t(255);
        const size_t o = off;
        off += bytes;
        return o;
    }
};

constexpr int kMaxSplits = 16;
// Row or column ranges of a dual rank-r reduction (lm_dual.cuh).  Its G partials (ranges x T x rp
// per job, at most three jobs) then fit the split-K partial region, which is free until the
// gradient reductions; its dB partials have their own regions.
constexpr int kDualMaxSplits = 16;
// Split tail tiles of a plain-store NF4 pair GEMM: at most this many fp32 partial tiles
// (512 x 256 each) per launch, in a workspace slot of kTailParts * 512 KiB.
constexpr int kTailParts = 80;
constexpr size_t kTailBytes = (size_t)kTailParts * 512 * 256 * 4;

struct Dims {
    int64_t T, ldT;
    int32_t r, rp;
};

Dims make_dims(int64_t T, int32_t r) {
    Dims D;
    D.T = T;
    D.ldT = round_up(std::max<int64_t>(T, 1), 64);
    D.r = r;
    D.rp = (int32_t)round_up(r, 16);
    return D;
}

// rank-r product buffer: (T x cols) bf16 and its transpose (cols x ldT)
struct RankBuf {
    size_t rows_off, t_off;
};

RankBuf take_rank(Bump& b, const Dims& D, int cols) {
    RankBuf r;
    r.rows_off = b.take((size_t)D.T * cols * 2);
    r.t_off = b.take((size_t)cols * D.ldT * 2);
    return r;
}

// rank-r buffers whose transposes are stacked: buffer i's transpose starts i * cols rows after
// buffer 0's, so one tensor map over the first covers all of them
void take_rank_stack(Bump& b, const Dims& D, int cols, std::initializer_list<RankBuf*> bufs) {
    for (RankBuf* r : bufs) r->rows_off = b.take((size_t)D.T * cols * 2);
    const size_t block = (size_t)cols * D.ldT * 2;
    const size_t t0 = b.take(bufs.size() * block);
    size_t i = 0;
    for (RankBuf* r : bufs) r->t_off = t0 + (i++) * block;
}

struct MlpPlan {
    Dims D;
    RankBuf xa, ha;         // saved: s*[X Ag^T | X Au^T] (T x 2rp), s*h Ad^T (T x rp)
    size_t saved_total;
    size_t part;            // workspace
    RankBuf gd, gg, gu;     // s*dY Bd, s*de Bg, s*du Bu
    size_t de, du;
    size_t bdiag;           // [Bg | 0 ; 0 | Bu] (2n x 2rp) for the CTA-pair gate/up GEMM
    size_t sc[3];           // NF4 base: fp32 block-scale tables of W_gate, W_up, W_down
    size_t tail;            // NF4 base: split tail tiles of the down and dX GEMMs
    size_t abc;             // bf16 copies of fp32 LoRA A and B
    size_t dpart[3];        // dual reductions: dB partials of dBd ([ranges][d][rp]), dBg, dBu ([ranges][n][rp])
    size_t ws_total;
};

MlpPlan plan_mlp(int64_t T, int64_t d, int64_t n, int32_t r) {
    MlpPlan P;
    P.D = make_dims(T, r);
    const int64_t rp = P.D.rp;
    Bump s;
    P.xa = take_rank(s, P.D, 2 * rp);
    P.ha = take_rank(s, P.D, rp);
    P.saved_total = s.off;
    Bump w;
    w.take(256);  // error word
    const int64_t part_elems = std::max<int64_t>(T * 2 * rp, 3 * (n + d) * rp);
    P.part = w.take((size_t)kMaxSplits * part_elems * 4);
    P.gd = take_rank(w, P.D, rp);
    take_rank_stack(w, P.D, rp, {&P.gg, &P.gu});
    P.de = w.take((size_t)T * n * 2);
    P.du = w.take((size_t)T * n * 2);
    P.bdiag = w.take((size_t)2 * n * 2 * rp * 2);
    for (int i = 0; i < 3; ++i) P.sc[i] = w.take((size_t)n * d / 64 * 4);
    P.tail = w.take(kTailBytes);
    P.abc = w.take((size_t)(2 * ab_elems(r, d, n) + ab_elems(r, n, d)) * 2);
    const int64_t cols[3] = {d, n, n};
    for (int i = 0; i < 3; ++i) {
        P.dpart[i] = w.take((size_t)kDualMaxSplits * cols[i] * rp * 4);
    }
    P.ws_total = w.off;
    return P;
}

struct QkvPlan {
    Dims D;
    RankBuf xa;             // saved: s*[X Aq^T | X Ak^T | X Av^T] (T x 3rp)
    size_t saved_total;
    size_t part;
    RankBuf g[3];
    size_t sc[3];           // NF4 base: fp32 block-scale tables of W_q, W_k, W_v
    size_t tail;            // NF4 base: split tail tiles of the dX GEMM
    size_t abc;             // bf16 copies of fp32 LoRA A and B
    size_t dpart[3];        // dual reduction: dB partials ([ranges][out][rp] fp32)
    size_t ws_total;
};

QkvPlan plan_qkv(int64_t T, int64_t d, int64_t nq, int64_t nk, int64_t nv, int32_t r) {
    QkvPlan P;
    P.D = make_dims(T, r);
    const int64_t rp = P.D.rp;
    Bump s;
    P.xa = take_rank(s, P.D, 3 * rp);
    P.saved_total = s.off;
    Bump w;
    w.take(256);
    const int64_t part_elems = std::max<int64_t>(T * 3 * rp, (3 * d + nq + nk + nv) * rp);
    P.part = w.take((size_t)kMaxSplits * part_elems * 4);
    take_rank_stack(w, P.D, rp, {&P.g[0], &P.g[1], &P.g[2]});
    const int64_t nout[3] = {nq, nk, nv};
    for (int i = 0; i < 3; ++i) P.sc[i] = w.take((size_t)nout[i] * d / 64 * 4);
    P.tail = w.take(kTailBytes);
    P.abc = w.take((size_t)(ab_elems(r, d, nq) + ab_elems(r, d, nk) + ab_elems(r, d, nv)) * 2);
    for (int i = 0; i < 3; ++i) {
        P.dpart[i] = w.take((size_t)kDualMaxSplits * nout[i] * rp * 4);
    }
    P.ws_total = w.off;
    return P;
}

struct OPlan {
    Dims D;
    RankBuf xa;
    size_t saved_total;
    size_t part;
    RankBuf g;
    size_t sc;              // NF4 base: fp32 block-scale table of W_o
    size_t tail;            // NF4 base: split tail tiles of the O and dX GEMMs
    size_t abc;             // bf16 copies of fp32 LoRA A and B
    size_t dpart;           // dual reduction: dB partials
    size_t ws_total;
};

OPlan plan_o(int64_t T, int64_t d_in, int64_t d_out, int32_t r) {
    OPlan P;
    P.D = make_dims(T, r);
    const int64_t rp = P.D.rp;
    Bump s;
    P.xa = take_rank(s, P.D, rp);
    P.saved_total = s.off;
    Bump w;
    w.take(256);
    const int64_t part_elems = std::max<int64_t>(T * rp, (d_in + d_out) * rp);
    P.part = w.take((size_t)kMaxSplits * part_elems * 4);
    P.g = take_rank(w, P.D, rp);
    P.sc = w.take((size_t)d_out * d_in / 64 * 4);
    P.tail = w.take(kTailBytes);
    P.abc = w.take((size_t)ab_elems(r, d_in, d_out) * 2);
    P.dpart = w.take((size_t)kDualMaxSplits * d_out * rp * 4);
    P.ws_total = w.off;
    return P;
}

// fp32 block-scale tables of the NF4 weights among `ws` for the NF4 GEMMs, built as side work of
// a finalisation launch (FinSide) that runs before the first GEMM reading them; int4 and NVFP4
// weights need none: their scales are read where they are
struct ScaleTable {
    const lm_weight* W;
    float* table;
};
void side_scale_tables(FinSide& side, std::initializer_list<ScaleTable> ws) {
    constexpr int kMax = (int)(sizeof(side.nf4.j) / sizeof(side.nf4.j[0]));  // every block has at most 3 weights
    for (const ScaleTable& t : ws)
        if (t.W->kind == LM_WEIGHT_NF4 && side.nf4_jobs < kMax)
            side.nf4.j[side.nf4_jobs++] = Nf4ScaleJob{t.W->absmax_q, t.W->group_scale, t.W->rows, t.W->cols / 64, t.table};
}

// fp32 LoRA parameters ([LO] "FP32 LoRA gradients"): A (r x in) and B (out x r) of every fp32
// projection rounded to bf16 (RNE) into `dst`, one launch; each copy then points at its bf16
// matrices.  bf16 parameters are used as they are.
struct AbProj {
    lm_lora* L;
    int64_t in, out;
};
lm_status ab_to_bf16(const char* tag, std::initializer_list<AbProj> projs, uint16_t* dst, cudaStream_t st) {
    CvtJobs jobs{};
    int nj = 0;
    for (const AbProj& a : projs) {
        if (a.L->ab_dtype != LM_AB_F32) continue;
        const int64_t na = (int64_t)a.L->r * a.in, nb = a.out * (int64_t)a.L->r;
        jobs.j[nj++] = CvtJob{static_cast<const float*>(a.L->A), dst, na};
        a.L->A = dst;
        dst += round_up(na, 128);
        jobs.j[nj++] = CvtJob{static_cast<const float*>(a.L->B), dst, nb};
        a.L->B = dst;
        dst += round_up(nb, 128);
        a.L->ab_dtype = LM_AB_BF16;
    }
    if (nj == 0) return LM_OK;
    ProfScope prof(tag, st);
    const cudaError_t e = launch_f32_to_bf16(jobs, nj, st);
    return e == cudaSuccess ? LM_OK : cuda_fail(e, "fp32 -> bf16 launch");
}

// 2D bf16 tensor map (rows x cols, row stride ld elements), box 64 columns x box_rows rows,
// 128-byte swizzle
lm_status encode_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1u, 1u};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(LM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %lld x %lld tensor, box rows %d", (int)r,
                    (long long)rows, (long long)cols, box_rows);
    return LM_OK;
}

// A LoRA B matrix (C rows x r columns bf16, row-major) as the MN-major B operand of the dual
// reduction's row reduction: box 16 columns x 128 rows with 32-byte swizzle (columns beyond r read 0)
lm_status encode_b_sw32(CUtensorMap* m, const void* base, int64_t C, int r) {
    cuuint64_t dims[2] = {(cuuint64_t)r, (cuuint64_t)C};
    cuuint64_t strides[1] = {(cuuint64_t)r * 2};
    cuuint32_t box[2] = {16u, 128u};
    cuuint32_t es[2] = {1u, 1u};
    const CUresult res = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS)
        return fail(LM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %lld x %d LoRA B", (int)res, (long long)C, r);
    return LM_OK;
}

// ------------------------------------------------------------------ GEMM launch builder
struct Builder {
    Params p;
    float* tail_buf = nullptr;  // workspace slot for split tail tiles (NF4 plain-store GEMMs)
    int nmaps = 0;
    int tile_m = kBM;
    lm_status st = LM_OK;
    GemmKind kind;

    explicit Builder(GemmKind k) : kind(k) {
        memset(&p, 0, sizeof p);
        if (gemm_is_pair(k)) tile_m = 256;
        if (gemm_is_pair_nf4(k)) {
            tile_m = 512;
            nf4_codebook_host(p.nf4_code);
        }
    }

    // 2D uint8 tensor (NF4 codes: rows x cols bytes), box = box_w bytes x box_rows rows, no swizzle
    int map_u8(const void* base, int64_t rows, int64_t cols, int64_t ld, int box_w, int box_rows) {
        if (st != LM_OK) return 0;
        if (nmaps >= kMaxMaps) {
            st = fail(LM_ERR_UNSUPPORTED, "too many tensor maps in one launch");
            return 0;
        }
        cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)ld};
        cuuint32_t box[2] = {(cuuint32_t)box_w, (cuuint32_t)box_rows};
        cuuint32_t es[2] = {1u, 1u};
        const CUresult r = g_encode(&p.maps[nmaps], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                                    strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            st = fail(LM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for NF4 codes %lld x %lld bytes", (int)r,
                      (long long)rows, (long long)cols);
            return 0;
        }
        p.map_bytes[nmaps] = (uint32_t)(box_w * box_rows);
        p.map_w[nmaps] = (int32_t)cols;
        return nmaps++;
    }

    // codes map of an NF4 weight read K-major (forward: box 32 bytes = 64 elements x rows)
    int codes_k(const lm_weight& W, int box_rows) { return map_u8(W.codes, W.rows, W.cols / 2, W.cols / 2, 32, box_rows); }
    // codes map of an NF4 weight read MN-major (input gradient: box 64 bytes = 128 elements x 64 rows)
    int codes_mn(const lm_weight& W) { return map_u8(W.codes, W.rows, W.cols / 2, W.cols / 2, 64, 64); }

    // fp32 block-scale table of an NF4 weight ([cols / 64][rows], see nf4_scale_tile):
    // box 128 rows x 1 K block (weight read K-major) or 64 rows x 2 column blocks (MN-major);
    // rows outside the weight read 0
    // An NVFP4 weight maps its E4M3 block scales the same way (four per 32-bit word); an int4
    // weight instead maps its (scale, zero) words ([cols / G][rows] 32-bit words): box
    // 128 rows x (G == 32 ? 2 : 1) groups (K-major: the groups of one 64-wide K block) or 64 rows x
    // max(1, 128 / G) groups (MN-major: the groups of 128 columns).
    int scales(const float* table, const lm_weight& W, bool mn) {
        if (st != LM_OK) return 0;
        if (nmaps >= kMaxMaps) {
            st = fail(LM_ERR_UNSUPPORTED, "too many tensor maps in one launch");
            return 0;
        }
        if (W.kind == LM_WEIGHT_NVFP4) {  // E4M3 scales, four per word: [cols / 64][rows] words
            cuuint64_t dims[2] = {(cuuint64_t)W.rows, (cuuint64_t)(W.cols / 64)};
            cuuint64_t strides[1] = {(cuuint64_t)W.rows * 4};
            cuuint32_t box[2] = {mn ? 64u : 128u, mn ? 2u : 1u};
            cuuint32_t es[2] = {1u, 1u};
            const CUresult r = g_encode(&p.maps[nmaps], CU_TENSOR_MAP_DATA_TYPE_UINT32, 2,
                                        const_cast<uint8_t*>(W.block_scale), dims, strides, box, es,
                                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) {
                st = fail(LM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for NVFP4 scales %lld x %lld", (int)r,
                          (long long)W.rows, (long long)(W.cols / 64));
                return 0;
            }
            p.map_bytes[nmaps] = 512u;
            p.map_w[nmaps] = (int32_t)W.rows;
            p.map_group[nmaps] = -1;
            p.map_gscale[nmaps] = W.global_scale;
            return nmaps++;
        }
        if (W.kind == LM_WEIGHT_INT4) {
            const int G = W.group;
            cuuint64_t dims[2] = {(cuuint64_t)W.rows, (cuuint64_t)(W.cols / G)};
            cuuint64_t strides[1] = {(cuuint64_t)W.rows * 4};
            cuuint32_t box[2] = {mn ? 64u : 128u, mn ? (cuuint32_t)std::max(1, 128 / G) : (G == 32 ? 2u : 1u)};
            cuuint32_t es[2] = {1u, 1u};
            const CUresult r = g_encode(&p.maps[nmaps], CU_TENSOR_MAP_DATA_TYPE_UINT32, 2,
                                        const_cast<uint16_t*>(W.scale_zero), dims, strides, box, es,
                                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) {
                st = fail(LM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for int4 scales %lld x %lld", (int)r,
                          (long long)W.rows, (long long)(W.cols / G));
                return 0;
            }
            p.map_bytes[nmaps] = 4u * box[0] * box[1];
            p.map_w[nmaps] = (int32_t)W.rows;
            p.map_group[nmaps] = G;
            return nmaps++;
        }
        cuuint64_t dims[2] = {(cuuint64_t)W.rows, (cuuint64_t)(W.cols / 64)};
        cuuint64_t strides[1] = {(cuuint64_t)W.rows * 4};
        cuuint32_t box[2] = {mn ? 64u : 128u, mn ? 2u : 1u};
        cuuint32_t es[2] = {1u, 1u};
        const CUresult r = g_encode(&p.maps[nmaps], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(table), dims,
                                    strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            st = fail(LM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for an NF4 scale table %lld x %lld", (int)r,
                      (long long)W.rows, (long long)(W.cols / 64));
            return 0;
        }
        p.map_bytes[nmaps] = 512u;
        p.map_w[nmaps] = (int32_t)W.rows;
        return nmaps++;
    }

    // The base-weight operand of a segment of the 512 x 256 pair GEMM: a bf16 W loaded as it is
    // (K-major box 64 x 128 rows, MN-major 64 x 64), a packed W as its codes plus scales (`table`:
    // the per-call NF4 block-scale table; unused for the other formats).
    // (`slot`: which of the segment's B operands; the gate/up GEMM has W_g in 0 and W_u in 1)
    void base_k(Seg& S, const lm_weight& W, const float* table, int slot = 0) {
        if (W.kind == LM_WEIGHT_BF16) {
            S.b_map[slot] = map(W.w, W.rows, W.cols, W.cols, 128);
        } else {
            S.b_map[slot] = codes_k(W, 128);
            S.b_scale[slot] = scales(table, W, false);
        }
    }
    void base_mn(Seg& S, const lm_weight& W, const float* table) {
        if (W.kind == LM_WEIGHT_BF16) {
            S.b_map[0] = map(W.w, W.rows, W.cols, W.cols, 64);
        } else {
            S.b_map[0] = codes_mn(W);
            S.b_scale[0] = scales(table, W, true);
        }
    }

    // 2D bf16 tensor (rows x cols, row stride ld elements) read by the staged GLU backward
    // epilogue of the packed pair kernel: box 16 columns x 128 rows, 32-byte swizzle
    int map_epi(const void* base, int64_t rows, int64_t cols, int64_t ld) {
        if (st != LM_OK) return 0;
        if (nmaps >= kMaxMaps) {
            st = fail(LM_ERR_UNSUPPORTED, "too many tensor maps in one launch");
            return 0;
        }
        cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
        cuuint32_t box[2] = {16u, 128u};
        cuuint32_t es[2] = {1u, 1u};
        const CUresult r = g_encode(&p.maps[nmaps], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                                    strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            st = fail(LM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %lld x %lld epilogue input", (int)r,
                      (long long)rows, (long long)cols);
            return 0;
        }
        p.map_bytes[nmaps] = 16u * 128u * 2u;
        p.map_w[nmaps] = (int32_t)cols;
        return nmaps++;
    }

    // 2D bf16 tensor (rows x cols, row stride ld elements), box = 64 columns x box_rows rows
    int map(const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
        if (st != LM_OK) return 0;
        if (nmaps >= kMaxMaps) {
            st = fail(LM_ERR_UNSUPPORTED, "too many tensor maps in one launch");
            return 0;
        }
        st = encode_bf16(&p.maps[nmaps], base, rows, cols, ld, box_rows);
        if (st != LM_OK) return 0;
        p.map_bytes[nmaps] = 128u * (uint32_t)box_rows;
        p.map_w[nmaps] = (int32_t)cols;
        return nmaps++;
    }

    Prob& prob() {
        Prob& P = p.prob[p.nprob++];
        memset(&P, 0, sizeof P);
        P.splits = 1;
        P.in_map[0] = P.in_map[1] = -1;
        for (int s = 0; s < kMaxSegs; ++s) {
            for (int i = 0; i < 3; ++i) P.seg[s].b_map[i] = -1;
            P.seg[s].b_scale[0] = P.seg[s].b_scale[1] = -1;
        }
        return P;
    }

    // tiles, split-K and work-unit numbering; returns the grid size
    int finish(int sms, int32_t* err) {
        p.err = err;
        p.kernel_id = gemm_is_pair(kind) ? 2 : gemm_is_pair_nf4(kind) ? 3 : 1;
        p.wait_ns = g_wait_ns ? g_wait_ns : kDefaultWaitNs;
        p.inject = (g_inject_mask >> (p.kernel_id - 1)) & 1;  // (ids 1-3: bits 0-2)
        if (kind == G_PART_KK) {  // the narrower stage layout keeps twice the bytes in flight
            bool narrow = true;
            for (int i = 0; i < p.nprob; ++i) narrow = narrow && p.prob[i].bn <= 64;
            if (narrow) kind = G_PART_KK64;
        }
        const bool partial = (kind == G_PART_KK || kind == G_PART_KK64 || kind == G_PART_KMN || kind == G_PART_MNK);
        // resident CTAs of the one-CTA kernel: two per SM for the 64-wide variants
        const int slots = (kind == G_PART_KK64 || kind == G_PART_KMN || kind == G_PART_MNK) ? 2 * sms : sms;
        int64_t tiles = 0;
        for (int i = 0; i < p.nprob; ++i) {
            Prob& P = p.prob[i];
            P.tiles_m = (int32_t)((P.M + tile_m - 1) / tile_m);
            tiles += (int64_t)P.tiles_m * P.tiles_n;
            P.group_m = 16;
            if (gemm_is_pair_nf4(kind)) {
                // about 16 MiB of A rows (bf16, all K segments) per raster group: the NF4 stage
                // ring is bound by load latency, and with 16 M tiles of 512 rows per group every
                // N column re-reads all of A from DRAM once the output stream has evicted it
                // (measured: 4-6 % per NF4 GEMM; the bf16 pair kernels are indifferent)
                int64_t k = 0;
                for (int si = 0; si < P.nseg; ++si) k += P.seg[si].kext;
                const int64_t per_tile = std::max<int64_t>(1, (int64_t)tile_m * k * 2);
                P.group_m = (int32_t)std::max<int64_t>(1, std::min<int64_t>(P.tiles_m, (16ll << 20) / per_tile));
            }
        }
        int S = 1;
        if (partial) {
            // split count with the least modelled time, counted in A-tile loads (128 x 64 bf16) of
            // one CTA: waves x (K blocks per unit + the unit's fp32 partial write, bn / 32 of them)
            // + the finalisation's read of every partial spread over as many CTAs.  (Without the
            // partial terms six column reductions over 4096 tokens at r = 64 took eight splits,
            // one wave fewer, and 226 MB of partials to write and read back.)
            double best = 1e300;
            for (int cand = 1; cand <= kMaxSplits; ++cand) {
                int64_t units_c = 0, kbps_max = 0;
                double ep_max = 0.0, part = 0.0;
                for (int i = 0; i < p.nprob; ++i) {
                    const Prob& P = p.prob[i];
                    const int64_t nkb = (P.seg[0].kext + kBK - 1) / kBK;
                    const int64_t kbps = (nkb + cand - 1) / cand;
                    const int64_t u = (int64_t)P.tiles_m * P.tiles_n * ((nkb + kbps - 1) / kbps);
                    units_c += u;
                    kbps_max = std::max(kbps_max, kbps);
                    ep_max = std::max(ep_max, P.bn / 32.0);
                    part += (double)u * kBM * P.bn * 4.0;
                }
                const double cost = (double)((units_c + slots - 1) / slots) * ((double)kbps_max + ep_max) +
                                     part / ((double)kBM * kBK * 2.0 * slots);
                if (cost < best * (1.0 - 1e-9)) {
                    best = cost;
                    S = cand;
                }
            }
        }
        int64_t units = 0;
        for (int i = 0; i < p.nprob; ++i) {
            Prob& P = p.prob[i];
            if (partial) {
                const int nkb = (P.seg[0].kext + kBK - 1) / kBK;
                P.kb_per_split = (nkb + S - 1) / S;
                P.splits = (nkb + P.kb_per_split - 1) / P.kb_per_split;
            } else {
                P.splits = 1;
                P.kb_per_split = 0;
            }
            P.unit_begin = (int32_t)units;
            units += (int64_t)P.tiles_m * P.tiles_n * P.splits;
        }
        p.total_units = (int32_t)units;
        // NF4 plain-store GEMM whose last wave is partly idle: split each tile of that wave over
        // its K blocks into the number of parts that finishes the tail soonest
        int ncl = 0;
        if (tail_buf && (kind == G2N_STORE_K || kind == G2N_STORE_MN) &&
            pair_nf4_clusters(kind, &ncl) == cudaSuccess && ncl > 1) {
            // the tail must lie inside the last problem (units run problem by problem)
            Prob& P = p.prob[p.nprob - 1];
            const int all = (int)units, tiles = P.tiles_m * P.tiles_n;
            const int full_all = all / ncl * ncl, tail = all - full_all;
            const int full = tiles - tail;  // the last problem's first tail tile
            int best = 1;
            double best_t = 1.0;  // the tail's makespan in tile times
            for (int S = 2; S <= 4 && full_all > 0 && tail > 0 && full >= 0; ++S) {
                if (tail * S > kTailParts) break;
                const double t = (double)((tail * S + ncl - 1) / ncl) / S;
                if (t < best_t - 1e-9) {
                    best_t = t;
                    best = S;
                }
            }
            if (best > 1 && full >= 0) {
                P.tail_begin = full;
                P.tail_splits = best;
                P.tail_part = tail_buf;
                p.total_units = full_all + tail * best;
            }
        }
        return (int)std::min<int64_t>(p.total_units, partial ? slots : sms);
    }

    lm_status launch(const char* tag, int sms, int32_t* err, cudaStream_t st_) {
        if (st != LM_OK) return st;
        const int grid = finish(sms, err);
        if (grid == 0) return LM_OK;
        {
            ProfScope prof(tag, st_);
            const cudaError_t e = gemm_is_pair(kind)       ? launch_gemm_pair(kind, p, p.total_units, st_)
                                  : gemm_is_pair_nf4(kind) ? launch_gemm_pair_nf4(kind, p, p.total_units, st_)
                                                           : launch_gemm(kind, p, grid, st_);
            if (e != cudaSuccess) return cuda_fail(e, "GEMM kernel launch");
        }
        const Prob& P = p.prob[p.nprob - 1];
        if (P.tail_splits > 1) {
            ProfScope prof("tail.fin", st_);
            TailFin f{};
            f.part = P.tail_part;
            f.out = static_cast<uint16_t*>(P.out0);
            f.M = P.M;
            f.N = P.N;
            f.ld_out = P.ld_out;
            f.out_col_step = P.out_col_step;
            f.ntail = P.tiles_m * P.tiles_n - P.tail_begin;
            f.splits = P.tail_splits;
            f.bn = P.bn;
            f.tail_begin = P.tail_begin;
            f.tiles_m = P.tiles_m;
            f.tiles_n = P.tiles_n;
            f.group_m = P.group_m;
            const cudaError_t e = launch_tail_fin(f, st_);
            if (e != cudaSuccess) return cuda_fail(e, "tail finalisation launch");
        }
        return LM_OK;
    }
};

Seg& seg(Prob& P, int i) {
    P.nseg = std::max(P.nseg, i + 1);
    return P.seg[i];
}

// rank-r input projection, K-major B made of stacked A matrices:
//   part[ks][t][i*rp + j] = sum_k Z[t][k] * A_i[j][k]
void add_rowproj_in(Builder& b, const uint16_t* Z, int64_t T, int64_t K, std::initializer_list<const void*> As,
                    const Dims& D, float* part) {
    Prob& P = b.prob();
    const int cnt = (int)As.size();
    P.M = (int32_t)T;
    P.N = cnt * D.rp;
    P.bn = cnt * D.rp;
    P.tiles_n = 1;
    Seg& S = seg(P, 0);
    S.a_map = b.map(Z, T, K, K, 128);
    int i = 0;
    for (const void* A : As) S.b_map[i++] = b.map(A, D.r, K, K, D.rp);
    S.b_rows = D.rp;
    S.kext = (int32_t)K;
    P.out0 = part;
    P.ld_out = P.bn;
    P.split_stride = T * P.bn;
}

// rank-r output-gradient projection, MN-major B:  part[ks][t][j] = sum_c dO[t][c] * Bm[c][j]
void add_rowproj_out(Builder& b, const uint16_t* dO, int64_t T, int64_t C, const void* Bm, const Dims& D,
                     float* part) {
    Prob& P = b.prob();
    P.M = (int32_t)T;
    P.N = D.rp;
    P.bn = D.rp;
    P.tiles_n = 1;
    Seg& S = seg(P, 0);
    S.a_map = b.map(dO, T, C, C, 128);
    S.b_map[0] = b.map(Bm, C, D.r, D.r, 64);
    S.kext = (int32_t)C;
    P.out0 = part;
    P.ld_out = P.bn;
    P.split_stride = T * P.bn;
}

// column reduction over tokens: part[ks][c][j] = sum_t Z[t][c] * PT[j][t], j < nb * rp (PT holds
// nb stacked blocks of rp rows)
void add_colreduce(Builder& b, const uint16_t* Z, int64_t T, int64_t C, const uint16_t* PT, const Dims& D,
                   float* part, int nb = 1) {
    Prob& P = b.prob();
    P.M = (int32_t)C;
    P.N = nb * D.rp;
    P.bn = P.N;
    P.tiles_n = 1;
    Seg& S = seg(P, 0);
    S.a_map = b.map(Z, T, C, C, 64);
    S.b_map[0] = b.map(PT, P.N, T, D.ldT, P.N);
    S.kext = (int32_t)T;
    P.out0 = part;
    P.ld_out = P.bn;
    P.split_stride = C * P.bn;
}

// The dA / dB column reductions of one backward call: one launch of split-K problems, one
// finalisation launch.  Each problem streams its activation Z once; gradients that reduce the
// same Z (the dA of every projection fed by X) are one problem whose B stacks their rank blocks.
struct ColReduce {
    static constexpr int kMaxJobs = kMaxFinColJobs;
    Builder b{G_PART_MNK};
    const Dims& D;
    float* next;
    FinColJob js[kMaxJobs];
    int prob_of[kMaxJobs];
    int njobs = 0;
    ColReduce(const Dims& D_, float* part) : D(D_), next(part) {}
    // outs[i] = the reduction against rank block i of PT, in dA layout (r x C) if `transposed`,
    // else in dB layout (C x r)
    void add(const uint16_t* Z, int64_t C, const uint16_t* PT, std::initializer_list<float*> outs, int transposed) {
        const int nb = (int)outs.size();
        if (njobs + nb > kMaxJobs || b.p.nprob >= kMaxProbs) {
            if (b.st == LM_OK) b.st = fail(LM_ERR_UNSUPPORTED, "too many gradient reductions in one launch");
            return;
        }
        const int64_t w = (int64_t)nb * D.rp;
        float* q = next;
        next += (size_t)kMaxSplits * C * w;
        add_colreduce(b, Z, D.T, C, PT, D, q, nb);
        int i = 0;
        for (float* o : outs) {
            js[njobs] = FinColJob{q + (size_t)(i++) * D.rp, C * w, C, 0, D.rp, D.r, transposed, o, (int32_t)w};
            prob_of[njobs++] = b.p.nprob - 1;
        }
    }
    // one more finalisation job over partials another launch wrote (its split count set)
    void add_fin(const FinColJob& j) {
        if (njobs >= kMaxJobs) {
            if (b.st == LM_OK) b.st = fail(LM_ERR_UNSUPPORTED, "too many gradient reductions in one launch");
            return;
        }
        js[njobs] = j;
        prob_of[njobs++] = -1;
    }
    lm_status run(const char* tag, const char* fin_tag, int sms, int32_t* err, cudaStream_t st) {
        if (b.p.nprob > 0) LM_TRY(b.launch(tag, sms, err, st));
        else LM_TRY(b.st);
        for (int i = 0; i < njobs; ++i)
            if (prob_of[i] >= 0) js[i].splits = b.p.prob[prob_of[i]].splits;
        ProfScope prof(fin_tag, st);
        const cudaError_t e = launch_fin_colreduce(js, njobs, st);
        if (e != cudaSuccess) return cuda_fail(e, "gradient finalisation launch");
        return LM_OK;
    }
};

lm_status fin_rows(const char* tag, const Builder& b, std::initializer_list<FinRowJob> jobs, int64_t T,
                   cudaStream_t st, const FinSide* side = nullptr) {
    FinRowJob js[3];
    int n = 0;
    for (const FinRowJob& j : jobs) {
        js[n] = j;
        js[n].splits = b.p.prob[n].splits;
        ++n;
    }
    ProfScope prof(tag, st);
    const cudaError_t e = launch_fin_rowproj(js, n, T, st, side);
    if (e != cudaSuccess) return cuda_fail(e, "rank-r finalisation launch");
    return LM_OK;
}

// Explicit split counts (a dual reduction's column ranges)
lm_status fin_rows_split(const char* tag, std::initializer_list<FinRowJob> jobs, int64_t T, cudaStream_t st,
                         const FinSide* side = nullptr) {
    FinRowJob js[3];
    int n = 0;
    for (const FinRowJob& j : jobs) js[n++] = j;
    ProfScope prof(tag, st);
    const cudaError_t e = launch_fin_rowproj(js, n, T, st, side);
    if (e != cudaSuccess) return cuda_fail(e, "rank-r finalisation launch");
    return LM_OK;
}

// ------------------------------------------------------------------ dual rank-r reduction
// One pass over an output gradient Z for both G = Z B (row reduction) and dB = Z^T (s X A^T)
// (column reduction); see lm_dual.cuh.  A unit is RB x CB tiles of 128 x 128; the partials of G
// have one slice per column range, those of dB one per row range.

struct DualShape {
    int RB = 0, CB = 0, nrr = 0;  // the column ranges of a job follow its width (dual_ranges)
    bool use = false;
};

// The unit shape with the shortest estimated time: the busiest CTA's tiles at what one SM draws
// (about 50 GB/s) or all bytes -- Z once, the partials written and read back -- at HBM speed,
// whichever is longer; at most kDualMaxSplits row and column ranges, and two sets of CB dB
// accumulators beside the two G accumulators in TMEM (512 columns).  `use` when that beats the
// separate row- and column-reduction passes, which stream Z twice at HBM speed (or always where
// feasible under the test hook's flag).
constexpr double kSmBytesPerS = 50e9, kHbmBytesPerS = 6.5e12;
// One shape for every job of a launch (jobs of widths Cs, all T rows); ncr of the job of width C
// is dual_ranges(C, CB).
inline int dual_ranges(int64_t C, int CB) { return (int)(((C + 127) / 128 + CB - 1) / CB); }
DualShape plan_dual(int64_t T, std::initializer_list<int64_t> Cs, int rp, int grid) {
    DualShape best;
    const int64_t nrb = (T + 127) / 128;
    const int cbmax = std::min(8, (512 - 2 * rp) / (2 * rp));
    double best_t = 1e300;
    for (int CB = 1; CB <= cbmax; ++CB) {
        bool fits = true;
        for (int64_t C : Cs) fits = fits && dual_ranges(C, CB) <= kDualMaxSplits;
        if (!fits) continue;
        for (int RB = 1; RB <= 16; ++RB) {
            const int64_t nrr = (nrb + RB - 1) / RB;
            if (nrr > kDualMaxSplits) continue;
            int64_t units = 0;
            double total = 0.0;
            for (int64_t C : Cs) {
                const int64_t ncr = dual_ranges(C, CB);
                units += nrr * ncr;
                total += (double)T * C * 2.0 + 2.0 * (double)(ncr * T + nrr * C) * rp * 4.0;
            }
            const int64_t waves = (units + grid - 1) / grid;
            const double busiest = (double)waves * RB * CB * 32768.0;
            const double t = std::max(busiest / kSmBytesPerS, total / kHbmBytesPerS);
            if (t < best_t * 0.999) {
                best_t = t;
                best.RB = RB;
                best.CB = CB;
                best.nrr = (int)nrr;
            }
        }
    }
    double separate = 0.0;
    for (int64_t C : Cs) separate += 2.0 * (double)T * C * 2.0 / kHbmBytesPerS;
    best.use = best.RB > 0 && (best_t < separate || (g_inject_mask & kForceDual));
    return best;
}

struct DualLaunch {
    DualParams p;
    int nmaps = 0;
    lm_status st = LM_OK;
    DualLaunch() { memset(&p, 0, sizeof p); }
    // Z (T x C), B (C x r), rows [p_row0, p_row0 + rp) of P (p_rows x T, row stride ldT)
    void add(const uint16_t* Z, int64_t T, int64_t C, const void* B, int r, const uint16_t* P, int64_t p_rows, int p_row0,
             int64_t ldT, int rp, const DualShape& sh, float* gpart, float* dpart) {
        if (st != LM_OK) return;
        if (p.njobs >= kDualMaxJobs) {
            st = fail(LM_ERR_UNSUPPORTED, "too many jobs in one dual reduction");
            return;
        }
        DualJob& J = p.job[p.njobs++];
        J.z_map = nmaps;
        if ((st = encode_bf16(&p.maps[nmaps++], Z, T, C, C, 128)) != LM_OK) return;
        J.b_map = nmaps;
        if ((st = encode_b_sw32(&p.maps[nmaps++], B, C, r)) != LM_OK) return;
        J.p_map = nmaps;
        if ((st = encode_bf16(&p.maps[nmaps++], P, p_rows, T, ldT, rp)) != LM_OK) return;
        J.p_row0 = p_row0;
        J.T = (int32_t)T;
        J.C = (int32_t)C;
        J.nrb = (int32_t)((T + 127) / 128);
        J.ncb = (int32_t)((C + 127) / 128);
        J.RB = sh.RB;
        J.CB = sh.CB;
        J.nrr = sh.nrr;
        J.ncr = dual_ranges(C, sh.CB);
        J.gpart = gpart;
        J.dpart = dpart;
    }
    lm_status launch(const char* tag, int sms, int rp, int32_t* err, cudaStream_t st_) {
        if (st != LM_OK) return st;
        int64_t units = 0;
        for (int j = 0; j < p.njobs; ++j) {
            p.job[j].unit_begin = (int32_t)units;
            units += (int64_t)p.job[j].nrr * p.job[j].ncr;
        }
        p.total_units = (int32_t)units;
        p.rp = rp;
        p.stage_bytes = 32768 + 512 * rp;
        p.stages = std::min(kDualMaxStages, (kDualSmemBytes - 2048) / p.stage_bytes);
        p.err = err;
        p.kernel_id = 4;
        p.wait_ns = g_wait_ns ? g_wait_ns : kDefaultWaitNs;
        p.inject = (g_inject_mask >> 3) & 1;
        const int grid = (int)std::min<int64_t>(units, sms);
        if (grid == 0) return LM_OK;
        ProfScope prof(tag, st_);
        const cudaError_t e = launch_dual_reduce(p, grid, st_);
        return e == cudaSuccess ? LM_OK : cuda_fail(e, "dual reduction launch");
    }
};

template <typename T_>
T_* at(void* base, size_t off) {
    return reinterpret_cast<T_*>(static_cast<char*>(base) + off);
}
template <typename T_>
const T_* at(const void* base, size_t off) {
    return reinterpret_cast<const T_*>(static_cast<const char*>(base) + off);
}

}  // namespace

// Sets the calling thread's last-error text from another translation unit of the library.
namespace lm {
lm_status report_error(lm_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}
}  // namespace lm

// ====================================================================== utilities
extern "C" const char* lm_last_error(void) { return g_err; }

extern "C" lm_status lm_nf4_codebook(float* out) {
    if (!out) return fail(LM_ERR_NULL, "out is NULL");
    nf4_codebook_host(out);
    return LM_OK;
}

extern "C" lm_status lm_workspace_reset(void* ws, lm_stream stream) {
    LM_TRY(need_ptr(ws, "ws"));
    LM_CUDA(cudaMemsetAsync(ws, 0, 256, (cudaStream_t)stream), "cudaMemsetAsync");
    return LM_OK;
}

extern "C" lm_status lm_debug_inject(int32_t family_mask, uint64_t wait_ns) {
    if (family_mask < 0 || family_mask > 31) return fail(LM_ERR_SHAPE, "family_mask = %d is not in [0, 31]", family_mask);
    g_inject_mask = family_mask;
    g_wait_ns = wait_ns;
    return LM_OK;
}

extern "C" lm_status lm_workspace_check(void* ws, lm_stream stream) {
    LM_TRY(need_ptr(ws, "ws"));
    int32_t h[4] = {0, 0, 0, 0};
    LM_CUDA(cudaMemcpyAsync(h, ws, sizeof h, cudaMemcpyDeviceToHost, (cudaStream_t)stream), "cudaMemcpyAsync");
    LM_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "cudaStreamSynchronize");
    if (h[0] != 0) {
        LM_CUDA(cudaMemsetAsync(ws, 0, 256, (cudaStream_t)stream), "cudaMemsetAsync");
        LM_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "cudaStreamSynchronize");
        return fail((lm_status)h[0], "a kernel gave up on a bounded wait (kernel family %d, role %d, block %d)", h[3],
                    h[1], h[2]);
    }
    return LM_OK;
}

// ====================================================================== tracing
extern "C" lm_status lm_profile_enable(int32_t on) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    g_prof_on = on != 0;
    return LM_OK;
}

extern "C" lm_status lm_profile_reset(void) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    for (const ProfRec& r : g_prof) {
        cudaEventSynchronize(r.b);
        g_prof_pool.push_back(r.a);
        g_prof_pool.push_back(r.b);
    }
    g_prof.clear();
    return LM_OK;
}

extern "C" lm_status lm_profile_summary(char* buf, size_t buf_len) {
    if (!buf || buf_len == 0) return fail(LM_ERR_NULL, "buf is NULL or empty");
    std::lock_guard<std::mutex> g(g_prof_mu);
    struct Agg {
        std::string tag;
        long long n;
        double ms;
    };
    std::vector<Agg> agg;
    for (const ProfRec& r : g_prof) {
        LM_CUDA(cudaEventSynchronize(r.b), "cudaEventSynchronize");
        float ms = 0.f;
        LM_CUDA(cudaEventElapsedTime(&ms, r.a, r.b), "cudaEventElapsedTime");
        size_t i = 0;
        while (i < agg.size() && agg[i].tag != r.tag) ++i;
        if (i == agg.size()) agg.push_back(Agg{r.tag, 0, 0.0});
        agg[i].n += 1;
        agg[i].ms += ms;
    }
    std::string out;
    char line[160];
    for (const Agg& a : agg) {
        snprintf(line, sizeof line, "%s\t%lld\t%.6f\n", a.tag.c_str(), a.n, a.ms);
        out += line;
    }
    const size_t n = std::min(out.size(), buf_len - 1);
    memcpy(buf, out.data(), n);
    buf[n] = 0;
    return LM_OK;
}

// ====================================================================== LoRA MLP
extern "C" lm_status lora_mlp_saved_size(int64_t T, int32_t r, size_t* bytes) {
    if (!bytes) return fail(LM_ERR_NULL, "bytes is NULL");
    LM_TRY(check_T(T));
    LM_TRY(check_r(r));
    *bytes = plan_mlp(T, 32, 32, r).saved_total;
    return LM_OK;
}

extern "C" lm_status lora_mlp_workspace_size(int64_t T, int64_t d, int64_t n, int32_t r, size_t* bytes) {
    if (!bytes) return fail(LM_ERR_NULL, "bytes is NULL");
    LM_TRY(check_T(T));
    LM_TRY(check_dim(d, "d"));
    LM_TRY(check_dim(n, "n"));
    LM_TRY(check_r(r));
    *bytes = plan_mlp(T, d, n, r).ws_total;
    return LM_OK;
}

static lm_status check_mlp_common(int64_t T, int64_t d, int64_t n, int32_t act, const lm_lora* gate,
                                  const lm_lora* up, const lm_lora* down) {
    LM_TRY(check_T(T));
    LM_TRY(check_dim(d, "d"));
    LM_TRY(check_dim(n, "n"));
    if (act != LM_ACT_SWIGLU && act != LM_ACT_GEGLU_ERF) return fail(LM_ERR_DTYPE, "act = %d is not known", act);
    if (!gate) return fail(LM_ERR_NULL, "gate is NULL");
    LM_TRY(check_r(gate->r));
    LM_TRY(check_lora(gate, "gate", d, n, gate->r));
    LM_TRY(check_lora(up, "up", d, n, gate->r));
    LM_TRY(check_lora(down, "down", n, d, gate->r));
    bool q4 = false;
    LM_TRY(same_kind({gate, up, down}, &q4));
    return LM_OK;
}

extern "C" lm_status lora_mlp_fwd(int64_t T, int64_t d, int64_t n, int32_t act, const uint16_t* X,
                                  const lm_lora* gate, const lm_lora* up, const lm_lora* down, uint16_t* y,
                                  uint16_t* e_save, uint16_t* u_save, uint16_t* h_save, void* saved,
                                  size_t saved_bytes, void* ws, size_t ws_bytes, lm_stream stream) {
    LM_TRY(check_mlp_common(T, d, n, act, gate, up, down));
    LM_TRY(need_ptr(X, "X"));
    LM_TRY(need_ptr(y, "y"));
    LM_TRY(need_ptr(e_save, "e_save"));
    LM_TRY(need_ptr(u_save, "u_save"));
    LM_TRY(need_ptr(h_save, "h_save"));
    LM_TRY(need_ptr(saved, "saved"));
    LM_TRY(need_ptr(ws, "ws"));
    const int32_t r = gate->r;
    const bool q4 = gate->W.kind != LM_WEIGHT_BF16;  // packed 4-bit base (NF4, int4 or NVFP4)
    const MlpPlan PL = plan_mlp(T, d, n, r);
    if (saved_bytes < PL.saved_total)
        return fail(LM_ERR_WORKSPACE, "saved buffer has %zu bytes, needs %zu", saved_bytes, PL.saved_total);
    if (ws_bytes < PL.ws_total) return fail(LM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, PL.ws_total);
    const size_t td = (size_t)T * d * 2, tn = (size_t)T * n * 2;
    LM_TRY(check_alias({{y, td, "y"}, {e_save, tn, "e_save"}, {u_save, tn, "u_save"}, {h_save, tn, "h_save"},
                        {saved, PL.saved_total, "saved"}, {ws, PL.ws_total, "ws"}},
                       {{X, td, "X"}, wspan(gate, "gate.W"), wspan(up, "up.W"), wspan(down, "down.W"),
                        {gate->A, ab_bytes(gate, r * d), "gate.A"}, {gate->B, ab_bytes(gate, n * r), "gate.B"},
                        {up->A, ab_bytes(up, r * d), "up.A"}, {up->B, ab_bytes(up, n * r), "up.B"},
                        {down->A, ab_bytes(down, r * n), "down.A"}, {down->B, ab_bytes(down, d * r), "down.B"}}));
    if (T == 0) return LM_OK;
    int sms = 0;
    LM_TRY(ready(&sms));
    cudaStream_t st = (cudaStream_t)stream;
    const Dims& D = PL.D;
    const int rp = D.rp;
    int32_t* err = static_cast<int32_t*>(ws);
    float* part = at<float>(ws, PL.part);
    lm_lora gate_c = *gate, up_c = *up, down_c = *down;
    LM_TRY(ab_to_bf16("mlp.ab", {{&gate_c, d, n}, {&up_c, d, n}, {&down_c, n, d}}, at<uint16_t>(ws, PL.abc), st));
    gate = &gate_c;
    up = &up_c;
    down = &down_c;
    float* sc[3] = {at<float>(ws, PL.sc[0]), at<float>(ws, PL.sc[1]), at<float>(ws, PL.sc[2])};
    // Side work of the X A^T finalisation launch, which nothing before the gate/up GEMM needs: the
    // per-K-block fp32 block scales of the NF4 weights (read by the NF4 GEMMs) and the
    // block-diagonal rank-r operand [Bg | 0 ; 0 | Bu] of the gate/up GEMM
    uint16_t* bdiag = at<uint16_t>(ws, PL.bdiag);
    FinSide side;
    side_scale_tables(side, {{&gate->W, sc[0]}, {&up->W, sc[1]}, {&down->W, sc[2]}});
    side.bd_Bg = bf(gate->B);
    side.bd_Bu = bf(up->B);
    side.bd_n = n;
    side.bd_r = r;
    side.bd_rp = rp;
    side.bd_out = bdiag;
    uint16_t* xa = at<uint16_t>(saved, PL.xa.rows_off);
    uint16_t* xaT = at<uint16_t>(saved, PL.xa.t_off);
    uint16_t* ha = at<uint16_t>(saved, PL.ha.rows_off);
    uint16_t* haT = at<uint16_t>(saved, PL.ha.t_off);

    {  // s*[X Ag^T | X Au^T]
        Builder b(G_PART_KK);
        add_rowproj_in(b, X, T, d, {gate->A, up->A}, D, part);
        LM_TRY(b.launch("mlp.xa", sms, err, st));
        LM_TRY(fin_rows("mlp.xa.fin", b, {FinRowJob{part, T * 2 * rp, 0, 2 * rp, rp, {gate->s, up->s, 0.f}, xa, xaT, D.ldT}}, T,
                        st, &side));
    }
    {  // e, u and h = act(e) * u; the rank-r terms enter the same accumulator
        // CTA pair: CTA 0 holds (or decodes) the 128 W_g rows of a tile, CTA 1 the matching W_u rows;
        // the rank-r segment multiplies [s XAg | s XAu] by the block-diagonal [Bg | 0 ; 0 | Bu]
        Builder b(q4 ? G2N_GLU_FWD : G2_GLU_FWD);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)n;
        P.bn = 256;
        P.tiles_n = (int32_t)((n + 127) / 128);
        P.n_step = 128;
        P.out_col_step = 128;
        P.act = act;
        Seg& S0 = seg(P, 0);
        S0.a_map = b.map(X, T, d, d, 128);
        b.base_k(S0, gate->W, sc[0], 0);
        b.base_k(S0, up->W, sc[1], 1);
        S0.kext = (int32_t)d;
        Seg& S1 = seg(P, 1);
        S1.a_map = b.map(xa, T, 2 * rp, 2 * rp, 128);
        S1.b_map[0] = b.map(bdiag, n, 2 * rp, 2 * rp, 128);
        S1.b_map[1] = b.map(bdiag + (size_t)n * 2 * rp, n, 2 * rp, 2 * rp, 128);
        S1.kext = 2 * rp;
        P.out0 = e_save;
        P.out1 = u_save;
        P.out2 = h_save;
        P.ld_out = n;
        LM_TRY(b.launch("mlp.gateup", sms, err, st));
    }
    {  // s_d * h Ad^T
        Builder b(G_PART_KK);
        add_rowproj_in(b, h_save, T, n, {down->A}, D, part);
        LM_TRY(b.launch("mlp.ha", sms, err, st));
        LM_TRY(fin_rows("mlp.ha.fin", b, {FinRowJob{part, T * rp, 0, rp, rp, {down->s, 0.f, 0.f}, ha, haT, D.ldT}}, T, st));
    }
    {  // y = h Wd^T + (s_d h Ad^T) Bd^T on 512 x 256 tiles for every base (a bf16 W is loaded as
       // is, a packed one decoded); with its light plain-store epilogue the single accumulator
       // costs less than the 256 x 256 kernel's extra operand traffic
        Builder b(G2N_STORE_K);
        b.tail_buf = at<float>(ws, PL.tail);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)d;
        P.bn = 256;
        P.tiles_n = (int32_t)((d + 255) / 256);
        P.n_step = 256;
        P.out_col_step = 256;
        Seg& S0 = seg(P, 0);
        S0.a_map = b.map(h_save, T, n, n, 128);
        b.base_k(S0, down->W, sc[2]);
        S0.b_rank_off = 128;
        S0.kext = (int32_t)n;
        Seg& S1 = seg(P, 1);
        S1.a_map = b.map(ha, T, rp, rp, 128);
        S1.b_map[0] = b.map(down->B, d, r, r, 128);
        S1.b_rank_off = 128;
        S1.kext = rp;
        P.out0 = y;
        P.ld_out = d;
        LM_TRY(b.launch("mlp.down", sms, err, st));
    }
    return LM_OK;
}

extern "C" lm_status lora_mlp_bwd(int64_t T, int64_t d, int64_t n, int32_t act, const uint16_t* X, const uint16_t* dY,
                                  const uint16_t* e_save, const uint16_t* u_save, const uint16_t* h_save,
                                  const void* saved, size_t saved_bytes, const lm_lora* gate, const lm_lora* up,
                                  const lm_lora* down, uint16_t* dX, float* dA_gate, float* dB_gate, float* dA_up,
                                  float* dB_up, float* dA_down, float* dB_down, void* ws, size_t ws_bytes,
                                  lm_stream stream) {
    LM_TRY(check_mlp_common(T, d, n, act, gate, up, down));
    LM_TRY(need_ptr(X, "X"));
    LM_TRY(need_ptr(dY, "dY"));
    LM_TRY(need_ptr(e_save, "e_save"));
    LM_TRY(need_ptr(u_save, "u_save"));
    LM_TRY(need_ptr(h_save, "h_save"));
    LM_TRY(need_ptr(saved, "saved"));
    LM_TRY(need_ptr(dX, "dX"));
    LM_TRY(need_ptr(dA_gate, "dA_gate"));
    LM_TRY(need_ptr(dB_gate, "dB_gate"));
    LM_TRY(need_ptr(dA_up, "dA_up"));
    LM_TRY(need_ptr(dB_up, "dB_up"));
    LM_TRY(need_ptr(dA_down, "dA_down"));
    LM_TRY(need_ptr(dB_down, "dB_down"));
    LM_TRY(need_ptr(ws, "ws"));
    const int32_t r = gate->r;
    const bool q4 = gate->W.kind != LM_WEIGHT_BF16;  // packed 4-bit base (NF4, int4 or NVFP4)
    const MlpPlan PL = plan_mlp(T, d, n, r);
    if (saved_bytes < PL.saved_total)
        return fail(LM_ERR_WORKSPACE, "saved buffer has %zu bytes, needs %zu", saved_bytes, PL.saved_total);
    if (ws_bytes < PL.ws_total) return fail(LM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, PL.ws_total);
    const size_t td = (size_t)T * d * 2, tn = (size_t)T * n * 2;
    const size_t ad = (size_t)r * d * 4, an = (size_t)r * n * 4;
    LM_TRY(check_alias({{dX, td, "dX"}, {dA_gate, ad, "dA_gate"}, {dB_gate, an, "dB_gate"}, {dA_up, ad, "dA_up"},
                        {dB_up, an, "dB_up"}, {dA_down, an, "dA_down"}, {dB_down, ad, "dB_down"},
                        {ws, PL.ws_total, "ws"}},
                       {{X, td, "X"}, {dY, td, "dY"}, {e_save, tn, "e_save"}, {u_save, tn, "u_save"},
                        {h_save, tn, "h_save"}, {saved, PL.saved_total, "saved"}, wspan(gate, "gate.W"),
                        wspan(up, "up.W"), wspan(down, "down.W")}));
    if (T == 0) {
        // no tokens: every LoRA gradient is an empty sum
        cudaStream_t st = (cudaStream_t)stream;
        LM_CUDA(cudaMemsetAsync(dA_gate, 0, ad, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dA_up, 0, ad, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dB_down, 0, ad, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dB_gate, 0, an, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dB_up, 0, an, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dA_down, 0, an, st), "cudaMemsetAsync");
        return LM_OK;
    }
    int sms = 0;
    LM_TRY(ready(&sms));
    cudaStream_t st = (cudaStream_t)stream;
    const Dims& D = PL.D;
    const int rp = D.rp;
    int32_t* err = static_cast<int32_t*>(ws);
    float* part = at<float>(ws, PL.part);
    lm_lora gate_c = *gate, up_c = *up, down_c = *down;
    LM_TRY(ab_to_bf16("mlp.ab", {{&gate_c, d, n}, {&up_c, d, n}, {&down_c, n, d}}, at<uint16_t>(ws, PL.abc), st));
    gate = &gate_c;
    up = &up_c;
    down = &down_c;
    float* sc[3] = {at<float>(ws, PL.sc[0]), at<float>(ws, PL.sc[1]), at<float>(ws, PL.sc[2])};
    // the NF4 weights' fp32 block-scale tables, first read by the dh GEMM: side work of the G_d
    // finalisation launch
    FinSide side;
    side_scale_tables(side, {{&gate->W, sc[0]}, {&up->W, sc[1]}, {&down->W, sc[2]}});
    const uint16_t* xaT = at<uint16_t>(saved, PL.xa.t_off);
    const uint16_t* haT = at<uint16_t>(saved, PL.ha.t_off);
    uint16_t* gd = at<uint16_t>(ws, PL.gd.rows_off);
    uint16_t* gdT = at<uint16_t>(ws, PL.gd.t_off);
    uint16_t* gg = at<uint16_t>(ws, PL.gg.rows_off);
    uint16_t* ggT = at<uint16_t>(ws, PL.gg.t_off);
    uint16_t* gu = at<uint16_t>(ws, PL.gu.rows_off);
    uint16_t* guT = at<uint16_t>(ws, PL.gu.t_off);
    uint16_t* de = at<uint16_t>(ws, PL.de);
    uint16_t* du = at<uint16_t>(ws, PL.du);

    // The dual rank-r reductions (lm_dual.cuh) read each output gradient once for both its G and
    // its dB, where the planner finds that cheaper than the two separate passes.
    const DualShape dsA = plan_dual(T, {d}, rp, sms), dsB = plan_dual(T, {n, n}, rp, sms);
    // G partials in the split-K partial region ([ranges][T][rp] each, at most kDualMaxSplits
    // ranges): Gd's are finalised before the de, du pass writes Gg's and Gu's
    float* gp[3] = {part, part, part + (size_t)kDualMaxSplits * T * rp};
    float* dp[3] = {at<float>(ws, PL.dpart[0]), at<float>(ws, PL.dpart[1]), at<float>(ws, PL.dpart[2])};
    if (dsA.use) {  // Gd = s_d dY Bd, formed once (feeds dh and dA_down), and dB_down's partials
        DualLaunch L;
        L.add(dY, T, d, down->B, r, haT, rp, 0, D.ldT, rp, dsA, gp[0], dp[0]);
        LM_TRY(L.launch("mlp.gd", sms, rp, err, st));
        LM_TRY(fin_rows_split("mlp.gd.fin",
                              {FinRowJob{gp[0], T * rp, dual_ranges(d, dsA.CB), rp, rp, {down->s, 0.f, 0.f}, gd, gdT, D.ldT}},
                              T, st, &side));
    } else {  // Gd = s_d dY Bd, formed once (feeds dh and dA_down)
        Builder b(G_PART_KMN);
        add_rowproj_out(b, dY, T, d, down->B, D, part);
        LM_TRY(b.launch("mlp.gd", sms, err, st));
        LM_TRY(fin_rows("mlp.gd.fin", b, {FinRowJob{part, T * rp, 0, rp, rp, {down->s, 0.f, 0.f}, gd, gdT, D.ldT}}, T, st,
                        &side));
    }
    {  // dh = dY Wd + Gd Ad with the activation backward in the epilogue: de, du
        Builder b(q4 ? G2N_GLU_BWD : G2_GLU_BWD);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)n;
        P.bn = 256;
        P.tiles_n = (int32_t)((n + 255) / 256);
        P.n_step = 256;
        P.out_col_step = 256;
        P.act = act;
        Seg& S0 = seg(P, 0);
        S0.a_map = b.map(dY, T, d, d, 128);
        b.base_mn(S0, down->W, sc[2]);
        S0.b_rank_off = 128;
        S0.kext = (int32_t)d;
        Seg& S1 = seg(P, 1);
        S1.a_map = b.map(gd, T, rp, rp, 128);
        S1.b_map[0] = b.map(down->A, r, n, n, 64);
        S1.b_rank_off = 128;
        S1.kext = rp;
        P.in0 = e_save;
        P.in1 = u_save;
        P.ld_in = n;
        P.out0 = de;
        P.out1 = du;
        P.ld_out = n;
        // packed base: the single-accumulator kernel stages e, u through shared memory when every
        // tile has the four K blocks its slot borrowing needs
        if (q4 && (d + kBK - 1) / kBK + (rp + kBK - 1) / kBK >= 4) {
            P.in_map[0] = b.map_epi(e_save, T, n, n);
            P.in_map[1] = b.map_epi(u_save, T, n, n);
        }
        LM_TRY(b.launch("mlp.dh", sms, err, st));
    }
    if (dsB.use) {  // Gg = s_g de Bg, Gu = s_u du Bu, formed once (feed dA and dX), and dB_gate's, dB_up's partials
        DualLaunch L;
        L.add(de, T, n, gate->B, r, xaT, 2 * rp, 0, D.ldT, rp, dsB, gp[1], dp[1]);
        L.add(du, T, n, up->B, r, xaT, 2 * rp, rp, D.ldT, rp, dsB, gp[2], dp[2]);
        LM_TRY(L.launch("mlp.gg_gu", sms, rp, err, st));
        LM_TRY(fin_rows_split("mlp.gg_gu.fin",
                              {FinRowJob{gp[1], T * rp, dual_ranges(n, dsB.CB), rp, rp, {gate->s, 0.f, 0.f}, gg, ggT, D.ldT},
                               FinRowJob{gp[2], T * rp, dual_ranges(n, dsB.CB), rp, rp, {up->s, 0.f, 0.f}, gu, guT, D.ldT}},
                              T, st));
    } else {  // Gg = s_g de Bg, Gu = s_u du Bu, formed once (feed dA and dX)
        Builder b(G_PART_KMN);
        float* part_u = part + (size_t)kMaxSplits * T * rp;
        add_rowproj_out(b, de, T, n, gate->B, D, part);
        add_rowproj_out(b, du, T, n, up->B, D, part_u);
        LM_TRY(b.launch("mlp.gg_gu", sms, err, st));
        LM_TRY(fin_rows("mlp.gg_gu.fin", b,
                        {FinRowJob{part, T * rp, 0, rp, rp, {gate->s, 0.f, 0.f}, gg, ggT, D.ldT},
                         FinRowJob{part_u, T * rp, 0, rp, rp, {up->s, 0.f, 0.f}, gu, guT, D.ldT}},
                        T, st));
    }
    {  // the six LoRA gradients as column reductions over the tokens (those of B from the dual
       // reductions' partials where they ran), one finalisation launch for all six
        ColReduce cr(D, part);
        cr.add(h_save, n, gdT, {dA_down}, 1);              // dA_down^T = h^T Gd
        if (!dsA.use) cr.add(dY, d, haT, {dB_down}, 0);    // dB_down   = dY^T (s h Ad^T)
        if (2 * rp <= 64) {
            cr.add(X, d, ggT, {dA_gate, dA_up}, 1);        // [dA_gate; dA_up]^T = X^T [Gg | Gu]
        } else {
            cr.add(X, d, ggT, {dA_gate}, 1);
            cr.add(X, d, guT, {dA_up}, 1);
        }
        if (!dsB.use) {
            cr.add(de, n, xaT, {dB_gate}, 0);                  // dB_gate   = de^T (s X Ag^T)
            cr.add(du, n, xaT + (size_t)rp * D.ldT, {dB_up}, 0);  // dB_up  = du^T (s X Au^T)
        }
        if (dsA.use) cr.add_fin(FinColJob{dp[0], d * rp, d, dsA.nrr, rp, r, 0, dB_down, rp});
        if (dsB.use) {
            cr.add_fin(FinColJob{dp[1], n * rp, n, dsB.nrr, rp, r, 0, dB_gate, rp});
            cr.add_fin(FinColJob{dp[2], n * rp, n, dsB.nrr, rp, r, 0, dB_up, rp});
        }
        LM_TRY(cr.run("mlp.dAdB", "mlp.dAdB.fin", sms, err, st));
    }
    {  // dX = de Wg + du Wu + Gg Ag + Gu Au on 512 x 256 tiles for every base
        Builder b(G2N_STORE_MN);
        b.tail_buf = at<float>(ws, PL.tail);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)d;
        P.bn = 256;
        P.tiles_n = (int32_t)((d + 255) / 256);
        P.n_step = 256;
        P.out_col_step = 256;
        const lm_lora* Ls[2] = {gate, up};
        const uint16_t* dOut[2] = {de, du};
        const uint16_t* G[2] = {gg, gu};
        for (int i = 0; i < 2; ++i) {
            Seg& S = seg(P, i);
            S.a_map = b.map(dOut[i], T, n, n, 128);
            b.base_mn(S, Ls[i]->W, sc[i]);
            S.b_rank_off = 128;
            S.kext = (int32_t)n;
            Seg& R = seg(P, 2 + i);
            R.a_map = b.map(G[i], T, rp, rp, 128);
            R.b_map[0] = b.map(Ls[i]->A, r, d, d, 64);
            R.b_rank_off = 128;
            R.kext = rp;
        }
        P.out0 = dX;
        P.ld_out = d;
        LM_TRY(b.launch("mlp.dX", sms, err, st));
    }
    return LM_OK;
}

// ====================================================================== LoRA QKV
// ====================================================================== non-gated ReLU^2 MLP
// [LO] "FP32 LoRA gradients": dense ReLU^2 MLPs with up/down LoRA projections and a fused ReLU^2
// activation derivative.  u = X Wu^T + su (X Au^T) Bu^T, h = max(u, 0)^2, y = h Wd^T + sd (h Ad^T) Bd^T.
struct Relu2Plan {
    Dims D;
    RankBuf xa, ha;         // saved: s_u X Au^T (T x rp), s_d h Ad^T (T x rp)
    size_t saved_total;
    size_t part;            // workspace
    RankBuf gd, gu;         // s_d dY Bd, s_u du Bu
    size_t du;
    size_t sc[2];           // NF4 base: fp32 block-scale tables of W_up, W_down
    size_t tail;            // NF4 base: split tail tiles of the down and dX GEMMs
    size_t abc;             // bf16 copies of fp32 LoRA A and B
    size_t dpart[2];        // dual reductions: dB partials of dBd ([ranges][d][rp]), dBu ([ranges][n][rp])
    size_t ws_total;
};

Relu2Plan plan_relu2(int64_t T, int64_t d, int64_t n, int32_t r) {
    Relu2Plan P;
    P.D = make_dims(T, r);
    const int64_t rp = P.D.rp;
    Bump s;
    P.xa = take_rank(s, P.D, rp);
    P.ha = take_rank(s, P.D, rp);
    P.saved_total = s.off;
    Bump w;
    w.take(256);  // error word
    const int64_t part_elems = std::max<int64_t>(T * rp, 2 * (n + d) * rp);
    P.part = w.take((size_t)kMaxSplits * part_elems * 4);
    P.gd = take_rank(w, P.D, rp);
    P.gu = take_rank(w, P.D, rp);
    P.du = w.take((size_t)T * n * 2);
    P.sc[0] = w.take((size_t)n * d / 64 * 4);
    P.sc[1] = w.take((size_t)d * n / 64 * 4);
    P.tail = w.take(kTailBytes);
    P.abc = w.take((size_t)(ab_elems(r, d, n) + ab_elems(r, n, d)) * 2);
    P.dpart[0] = w.take((size_t)kDualMaxSplits * d * rp * 4);
    P.dpart[1] = w.take((size_t)kDualMaxSplits * n * rp * 4);
    P.ws_total = w.off;
    return P;
}

extern "C" lm_status lora_relu2_mlp_saved_size(int64_t T, int32_t r, size_t* bytes) {
    if (!bytes) return fail(LM_ERR_NULL, "bytes is NULL");
    LM_TRY(check_T(T));
    LM_TRY(check_r(r));
    *bytes = plan_relu2(T, 32, 32, r).saved_total;
    return LM_OK;
}

extern "C" lm_status lora_relu2_mlp_workspace_size(int64_t T, int64_t d, int64_t n, int32_t r, size_t* bytes) {
    if (!bytes) return fail(LM_ERR_NULL, "bytes is NULL");
    LM_TRY(check_T(T));
    LM_TRY(check_dim(d, "d"));
    LM_TRY(check_dim(n, "n"));
    LM_TRY(check_r(r));
    *bytes = plan_relu2(T, d, n, r).ws_total;
    return LM_OK;
}

static lm_status check_relu2_common(int64_t T, int64_t d, int64_t n, const lm_lora* up, const lm_lora* down) {
    LM_TRY(check_T(T));
    LM_TRY(check_dim(d, "d"));
    LM_TRY(check_dim(n, "n"));
    if (!up) return fail(LM_ERR_NULL, "up is NULL");
    LM_TRY(check_r(up->r));
    LM_TRY(check_lora(up, "up", d, n, up->r));
    LM_TRY(check_lora(down, "down", n, d, up->r));
    bool q4 = false;
    LM_TRY(same_kind({up, down}, &q4));
    return LM_OK;
}

extern "C" lm_status lora_relu2_mlp_fwd(int64_t T, int64_t d, int64_t n, const uint16_t* X, const lm_lora* up,
                                        const lm_lora* down, uint16_t* y, uint16_t* u_save, uint16_t* h_save,
                                        void* saved, size_t saved_bytes, void* ws, size_t ws_bytes, lm_stream stream) {
    LM_TRY(check_relu2_common(T, d, n, up, down));
    LM_TRY(need_ptr(X, "X"));
    LM_TRY(need_ptr(y, "y"));
    LM_TRY(need_ptr(u_save, "u_save"));
    LM_TRY(need_ptr(h_save, "h_save"));
    LM_TRY(need_ptr(saved, "saved"));
    LM_TRY(need_ptr(ws, "ws"));
    const int32_t r = up->r;
    const bool q4 = up->W.kind != LM_WEIGHT_BF16;  // packed 4-bit base (NF4, int4 or NVFP4)
    const Relu2Plan PL = plan_relu2(T, d, n, r);
    if (saved_bytes < PL.saved_total)
        return fail(LM_ERR_WORKSPACE, "saved buffer has %zu bytes, needs %zu", saved_bytes, PL.saved_total);
    if (ws_bytes < PL.ws_total) return fail(LM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, PL.ws_total);
    const size_t td = (size_t)T * d * 2, tn = (size_t)T * n * 2;
    LM_TRY(check_alias({{y, td, "y"}, {u_save, tn, "u_save"}, {h_save, tn, "h_save"}, {saved, PL.saved_total, "saved"},
                        {ws, PL.ws_total, "ws"}},
                       {{X, td, "X"}, wspan(up, "up.W"), wspan(down, "down.W"), {up->A, ab_bytes(up, r * d), "up.A"},
                        {up->B, ab_bytes(up, n * r), "up.B"}, {down->A, ab_bytes(down, r * n), "down.A"},
                        {down->B, ab_bytes(down, d * r), "down.B"}}));
    if (T == 0) return LM_OK;
    int sms = 0;
    LM_TRY(ready(&sms));
    cudaStream_t st = (cudaStream_t)stream;
    const Dims& D = PL.D;
    const int rp = D.rp;
    int32_t* err = static_cast<int32_t*>(ws);
    float* part = at<float>(ws, PL.part);
    lm_lora up_c = *up, down_c = *down;
    LM_TRY(ab_to_bf16("relu2.ab", {{&up_c, d, n}, {&down_c, n, d}}, at<uint16_t>(ws, PL.abc), st));
    up = &up_c;
    down = &down_c;
    float* sc[2] = {at<float>(ws, PL.sc[0]), at<float>(ws, PL.sc[1])};
    FinSide side;  // the NF4 tables: side work of the X A^T finalisation, before the up GEMM
    side_scale_tables(side, {{&up->W, sc[0]}, {&down->W, sc[1]}});
    uint16_t* xa = at<uint16_t>(saved, PL.xa.rows_off);
    uint16_t* xaT = at<uint16_t>(saved, PL.xa.t_off);
    uint16_t* ha = at<uint16_t>(saved, PL.ha.rows_off);
    uint16_t* haT = at<uint16_t>(saved, PL.ha.t_off);
    {  // s_u X Au^T
        Builder b(G_PART_KK);
        add_rowproj_in(b, X, T, d, {up->A}, D, part);
        LM_TRY(b.launch("relu2.xa", sms, err, st));
        LM_TRY(fin_rows("relu2.xa.fin", b, {FinRowJob{part, T * rp, 0, rp, rp, {up->s, 0.f, 0.f}, xa, xaT, D.ldT}}, T, st,
                        &side));
    }
    {  // u = X Wu^T + (s_u X Au^T) Bu^T; the epilogue writes u and h = relu(u)^2
        Builder b(q4 ? G2N_ACT_FWD : G2_ACT_FWD);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)n;
        P.bn = 256;
        P.tiles_n = (int32_t)((n + 255) / 256);
        P.n_step = 256;
        P.out_col_step = 256;
        P.act = ACT_RELU2;
        Seg& S0 = seg(P, 0);
        S0.a_map = b.map(X, T, d, d, 128);
        b.base_k(S0, up->W, sc[0]);
        S0.b_rank_off = 128;
        S0.kext = (int32_t)d;
        Seg& S1 = seg(P, 1);
        S1.a_map = b.map(xa, T, rp, rp, 128);
        S1.b_map[0] = b.map(up->B, n, r, r, 128);
        S1.b_rank_off = 128;
        S1.kext = rp;
        P.out0 = u_save;
        P.out1 = h_save;
        P.ld_out = n;
        LM_TRY(b.launch("relu2.up", sms, err, st));
    }
    {  // s_d h Ad^T
        Builder b(G_PART_KK);
        add_rowproj_in(b, h_save, T, n, {down->A}, D, part);
        LM_TRY(b.launch("relu2.ha", sms, err, st));
        LM_TRY(fin_rows("relu2.ha.fin", b, {FinRowJob{part, T * rp, 0, rp, rp, {down->s, 0.f, 0.f}, ha, haT, D.ldT}}, T, st));
    }
    {  // y = h Wd^T + (s_d h Ad^T) Bd^T
        Builder b(G2N_STORE_K);  // 512 x 256 tiles for every base
        b.tail_buf = at<float>(ws, PL.tail);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)d;
        P.bn = 256;
        P.tiles_n = (int32_t)((d + 255) / 256);
        P.n_step = 256;
        P.out_col_step = 256;
        Seg& S0 = seg(P, 0);
        S0.a_map = b.map(h_save, T, n, n, 128);
        b.base_k(S0, down->W, sc[1]);
        S0.b_rank_off = 128;
        S0.kext = (int32_t)n;
        Seg& S1 = seg(P, 1);
        S1.a_map = b.map(ha, T, rp, rp, 128);
        S1.b_map[0] = b.map(down->B, d, r, r, 128);
        S1.b_rank_off = 128;
        S1.kext = rp;
        P.out0 = y;
        P.ld_out = d;
        LM_TRY(b.launch("relu2.down", sms, err, st));
    }
    return LM_OK;
}

extern "C" lm_status lora_relu2_mlp_bwd(int64_t T, int64_t d, int64_t n, const uint16_t* X, const uint16_t* dY,
                                        const uint16_t* u_save, const uint16_t* h_save, const void* saved,
                                        size_t saved_bytes, const lm_lora* up, const lm_lora* down, uint16_t* dX,
                                        float* dA_up, float* dB_up, float* dA_down, float* dB_down, void* ws,
                                        size_t ws_bytes, lm_stream stream) {
    LM_TRY(check_relu2_common(T, d, n, up, down));
    LM_TRY(need_ptr(X, "X"));
    LM_TRY(need_ptr(dY, "dY"));
    LM_TRY(need_ptr(u_save, "u_save"));
    LM_TRY(need_ptr(h_save, "h_save"));
    LM_TRY(need_ptr(saved, "saved"));
    LM_TRY(need_ptr(dX, "dX"));
    LM_TRY(need_ptr(dA_up, "dA_up"));
    LM_TRY(need_ptr(dB_up, "dB_up"));
    LM_TRY(need_ptr(dA_down, "dA_down"));
    LM_TRY(need_ptr(dB_down, "dB_down"));
    LM_TRY(need_ptr(ws, "ws"));
    const int32_t r = up->r;
    const bool q4 = up->W.kind != LM_WEIGHT_BF16;  // packed 4-bit base (NF4, int4 or NVFP4)
    const Relu2Plan PL = plan_relu2(T, d, n, r);
    if (saved_bytes < PL.saved_total)
        return fail(LM_ERR_WORKSPACE, "saved buffer has %zu bytes, needs %zu", saved_bytes, PL.saved_total);
    if (ws_bytes < PL.ws_total) return fail(LM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, PL.ws_total);
    const size_t td = (size_t)T * d * 2, tn = (size_t)T * n * 2;
    const size_t ad = (size_t)r * d * 4, an = (size_t)r * n * 4;
    LM_TRY(check_alias({{dX, td, "dX"}, {dA_up, ad, "dA_up"}, {dB_up, an, "dB_up"}, {dA_down, an, "dA_down"},
                        {dB_down, ad, "dB_down"}, {ws, PL.ws_total, "ws"}},
                       {{X, td, "X"}, {dY, td, "dY"}, {u_save, tn, "u_save"}, {h_save, tn, "h_save"},
                        {saved, PL.saved_total, "saved"}, wspan(up, "up.W"), wspan(down, "down.W")}));
    cudaStream_t st = (cudaStream_t)stream;
    if (T == 0) {
        LM_CUDA(cudaMemsetAsync(dA_up, 0, ad, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dB_up, 0, an, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dA_down, 0, an, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dB_down, 0, ad, st), "cudaMemsetAsync");
        return LM_OK;
    }
    int sms = 0;
    LM_TRY(ready(&sms));
    const Dims& D = PL.D;
    const int rp = D.rp;
    int32_t* err = static_cast<int32_t*>(ws);
    float* part = at<float>(ws, PL.part);
    lm_lora up_c = *up, down_c = *down;
    LM_TRY(ab_to_bf16("relu2.ab", {{&up_c, d, n}, {&down_c, n, d}}, at<uint16_t>(ws, PL.abc), st));
    up = &up_c;
    down = &down_c;
    float* sc[2] = {at<float>(ws, PL.sc[0]), at<float>(ws, PL.sc[1])};
    FinSide side;  // the NF4 tables: side work of the G_d finalisation, before the dh GEMM
    side_scale_tables(side, {{&up->W, sc[0]}, {&down->W, sc[1]}});
    const uint16_t* xaT = at<uint16_t>(saved, PL.xa.t_off);
    const uint16_t* haT = at<uint16_t>(saved, PL.ha.t_off);
    uint16_t* gd = at<uint16_t>(ws, PL.gd.rows_off);
    uint16_t* gdT = at<uint16_t>(ws, PL.gd.t_off);
    uint16_t* gu = at<uint16_t>(ws, PL.gu.rows_off);
    uint16_t* guT = at<uint16_t>(ws, PL.gu.t_off);
    uint16_t* du = at<uint16_t>(ws, PL.du);

    // the dual rank-r reductions (lm_dual.cuh) read dY and du once each for both G and dB, where
    // the planner finds that cheaper than the separate passes
    const DualShape dsA = plan_dual(T, {d}, rp, sms), dsB = plan_dual(T, {n}, rp, sms);
    float* dp[2] = {at<float>(ws, PL.dpart[0]), at<float>(ws, PL.dpart[1])};
    if (dsA.use) {  // Gd = s_d dY Bd (feeds dh and dA_down) and dB_down's partials
        DualLaunch L;
        L.add(dY, T, d, down->B, r, haT, rp, 0, D.ldT, rp, dsA, part, dp[0]);
        LM_TRY(L.launch("relu2.gd", sms, rp, err, st));
        LM_TRY(fin_rows_split("relu2.gd.fin",
                              {FinRowJob{part, T * rp, dual_ranges(d, dsA.CB), rp, rp, {down->s, 0.f, 0.f}, gd, gdT, D.ldT}},
                              T, st, &side));
    } else {  // Gd = s_d dY Bd, formed once (feeds dh and dA_down)
        Builder b(G_PART_KMN);
        add_rowproj_out(b, dY, T, d, down->B, D, part);
        LM_TRY(b.launch("relu2.gd", sms, err, st));
        LM_TRY(fin_rows("relu2.gd.fin", b, {FinRowJob{part, T * rp, 0, rp, rp, {down->s, 0.f, 0.f}, gd, gdT, D.ldT}}, T, st,
                        &side));
    }
    {  // dh = dY Wd + Gd Ad with the ReLU^2 derivative in the epilogue: du = dh * 2 relu(u)
        Builder b(q4 ? G2N_ACT_BWD : G2_ACT_BWD);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)n;
        P.bn = 256;
        P.tiles_n = (int32_t)((n + 255) / 256);
        P.n_step = 256;
        P.out_col_step = 256;
        P.act = ACT_RELU2;
        Seg& S0 = seg(P, 0);
        S0.a_map = b.map(dY, T, d, d, 128);
        b.base_mn(S0, down->W, sc[1]);
        S0.b_rank_off = 128;
        S0.kext = (int32_t)d;
        Seg& S1 = seg(P, 1);
        S1.a_map = b.map(gd, T, rp, rp, 128);
        S1.b_map[0] = b.map(down->A, r, n, n, 64);
        S1.b_rank_off = 128;
        S1.kext = rp;
        P.in0 = u_save;
        P.ld_in = n;
        P.out0 = du;
        P.ld_out = n;
        LM_TRY(b.launch("relu2.dh", sms, err, st));
    }
    if (dsB.use) {  // Gu = s_u du Bu (feeds dA_up and dX) and dB_up's partials
        DualLaunch L;
        L.add(du, T, n, up->B, r, xaT, rp, 0, D.ldT, rp, dsB, part, dp[1]);
        LM_TRY(L.launch("relu2.gu", sms, rp, err, st));
        LM_TRY(fin_rows_split("relu2.gu.fin",
                              {FinRowJob{part, T * rp, dual_ranges(n, dsB.CB), rp, rp, {up->s, 0.f, 0.f}, gu, guT, D.ldT}},
                              T, st));
    } else {  // Gu = s_u du Bu, formed once (feeds dA_up and dX)
        Builder b(G_PART_KMN);
        add_rowproj_out(b, du, T, n, up->B, D, part);
        LM_TRY(b.launch("relu2.gu", sms, err, st));
        LM_TRY(fin_rows("relu2.gu.fin", b, {FinRowJob{part, T * rp, 0, rp, rp, {up->s, 0.f, 0.f}, gu, guT, D.ldT}}, T, st));
    }
    {  // the four LoRA gradients as column reductions over the tokens (those of B from the dual
       // reductions' partials where they ran), one finalisation launch
        ColReduce cr(D, part);
        cr.add(h_save, n, gdT, {dA_down}, 1);                  // dA_down^T = h^T Gd
        if (!dsA.use) cr.add(dY, d, haT, {dB_down}, 0);        // dB_down   = dY^T (s h Ad^T)
        cr.add(X, d, guT, {dA_up}, 1);                         // dA_up^T   = X^T Gu
        if (!dsB.use) cr.add(du, n, xaT, {dB_up}, 0);          // dB_up     = du^T (s X Au^T)
        if (dsA.use) cr.add_fin(FinColJob{dp[0], d * rp, d, dsA.nrr, rp, r, 0, dB_down, rp});
        if (dsB.use) cr.add_fin(FinColJob{dp[1], n * rp, n, dsB.nrr, rp, r, 0, dB_up, rp});
        LM_TRY(cr.run("relu2.dAdB", "relu2.dAdB.fin", sms, err, st));
    }
    {  // dX = du Wu + Gu Au
        Builder b(G2N_STORE_MN);  // 512 x 256 tiles for every base
        b.tail_buf = at<float>(ws, PL.tail);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)d;
        P.bn = 256;
        P.tiles_n = (int32_t)((d + 255) / 256);
        P.n_step = 256;
        P.out_col_step = 256;
        Seg& S0 = seg(P, 0);
        S0.a_map = b.map(du, T, n, n, 128);
        b.base_mn(S0, up->W, sc[0]);
        S0.b_rank_off = 128;
        S0.kext = (int32_t)n;
        Seg& S1 = seg(P, 1);
        S1.a_map = b.map(gu, T, rp, rp, 128);
        S1.b_map[0] = b.map(up->A, r, d, d, 64);
        S1.b_rank_off = 128;
        S1.kext = rp;
        P.out0 = dX;
        P.ld_out = d;
        LM_TRY(b.launch("relu2.dX", sms, err, st));
    }
    return LM_OK;
}

extern "C" lm_status lora_qkv_saved_size(int64_t T, int32_t r, size_t* bytes) {
    if (!bytes) return fail(LM_ERR_NULL, "bytes is NULL");
    LM_TRY(check_T(T));
    LM_TRY(check_r(r));
    *bytes = plan_qkv(T, 32, 32, 32, 32, r).saved_total;
    return LM_OK;
}

extern "C" lm_status lora_qkv_workspace_size(int64_t T, int64_t d, int64_t nq, int64_t nk, int64_t nv, int32_t r,
                                             size_t* bytes) {
    if (!bytes) return fail(LM_ERR_NULL, "bytes is NULL");
    LM_TRY(check_T(T));
    LM_TRY(check_dim(d, "d"));
    LM_TRY(check_dim(nq, "nq"));
    LM_TRY(check_dim(nk, "nk"));
    LM_TRY(check_dim(nv, "nv"));
    LM_TRY(check_r(r));
    *bytes = plan_qkv(T, d, nq, nk, nv, r).ws_total;
    return LM_OK;
}

static lm_status check_qkv_common(int64_t T, int64_t d, int64_t nq, int64_t nk, int64_t nv, const lm_lora* q,
                                  const lm_lora* k, const lm_lora* v) {
    LM_TRY(check_T(T));
    LM_TRY(check_dim(d, "d"));
    LM_TRY(check_dim(nq, "nq"));
    LM_TRY(check_dim(nk, "nk"));
    LM_TRY(check_dim(nv, "nv"));
    if (!q) return fail(LM_ERR_NULL, "q is NULL");
    LM_TRY(check_r(q->r));
    LM_TRY(check_lora(q, "q", d, nq, q->r));
    LM_TRY(check_lora(k, "k", d, nk, q->r));
    LM_TRY(check_lora(v, "v", d, nv, q->r));
    bool q4 = false;
    LM_TRY(same_kind({q, k, v}, &q4));
    return LM_OK;
}

extern "C" lm_status lora_qkv_fwd(int64_t T, int64_t d, int64_t nq, int64_t nk, int64_t nv, const uint16_t* X,
                                  const lm_lora* q, const lm_lora* k, const lm_lora* v, uint16_t* Q, uint16_t* K,
                                  uint16_t* V, void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                                  lm_stream stream) {
    LM_TRY(check_qkv_common(T, d, nq, nk, nv, q, k, v));
    LM_TRY(need_ptr(X, "X"));
    LM_TRY(need_ptr(Q, "Q"));
    LM_TRY(need_ptr(K, "K"));
    LM_TRY(need_ptr(V, "V"));
    LM_TRY(need_ptr(saved, "saved"));
    LM_TRY(need_ptr(ws, "ws"));
    const int32_t r = q->r;
    const bool q4 = q->W.kind != LM_WEIGHT_BF16;  // packed 4-bit base (NF4, int4 or NVFP4)
    const QkvPlan PL = plan_qkv(T, d, nq, nk, nv, r);
    if (saved_bytes < PL.saved_total)
        return fail(LM_ERR_WORKSPACE, "saved buffer has %zu bytes, needs %zu", saved_bytes, PL.saved_total);
    if (ws_bytes < PL.ws_total) return fail(LM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, PL.ws_total);
    LM_TRY(check_alias({{Q, (size_t)T * nq * 2, "Q"}, {K, (size_t)T * nk * 2, "K"}, {V, (size_t)T * nv * 2, "V"},
                        {saved, PL.saved_total, "saved"}, {ws, PL.ws_total, "ws"}},
                       {{X, (size_t)T * d * 2, "X"}, wspan(q, "q.W"), wspan(k, "k.W"), wspan(v, "v.W")}));
    if (T == 0) return LM_OK;
    int sms = 0;
    LM_TRY(ready(&sms));
    cudaStream_t st = (cudaStream_t)stream;
    const Dims& D = PL.D;
    const int rp = D.rp;
    int32_t* err = static_cast<int32_t*>(ws);
    float* part = at<float>(ws, PL.part);
    lm_lora q_c = *q, k_c = *k, v_c = *v;
    LM_TRY(ab_to_bf16("qkv.ab", {{&q_c, d, nq}, {&k_c, d, nk}, {&v_c, d, nv}}, at<uint16_t>(ws, PL.abc), st));
    q = &q_c;
    k = &k_c;
    v = &v_c;
    float* sc[3] = {at<float>(ws, PL.sc[0]), at<float>(ws, PL.sc[1]), at<float>(ws, PL.sc[2])};
    FinSide side;  // the NF4 tables of W_q, W_k, W_v: side work of the X A^T finalisation
    side_scale_tables(side, {{&q->W, sc[0]}, {&k->W, sc[1]}, {&v->W, sc[2]}});
    uint16_t* xa = at<uint16_t>(saved, PL.xa.rows_off);
    uint16_t* xaT = at<uint16_t>(saved, PL.xa.t_off);
    {
        Builder b(G_PART_KK);
        add_rowproj_in(b, X, T, d, {q->A, k->A, v->A}, D, part);
        LM_TRY(b.launch("qkv.xa", sms, err, st));
        LM_TRY(fin_rows("qkv.xa.fin", b, {FinRowJob{part, T * 3 * rp, 0, 3 * rp, rp, {q->s, k->s, v->s}, xa, xaT, D.ldT}}, T,
                        st, &side));
    }
    // A bf16 base keeps the 256 x 256 kernel here: with outputs this narrow (4096 / 1024 columns)
    // the 512-row tiles leave too few units for the machine (measured at the 8B sizes: QKV 0.614
    // against 0.628 ms, O 0.425 against 0.467 ms per fwd+bwd).
    {
        Builder b(q4 ? G2N_STORE_K : G2_STORE_K);
        if (q4) b.tail_buf = at<float>(ws, PL.tail);
        const int xmap = b.map(X, T, d, d, 128);
        const int amap = b.map(xa, T, 3 * rp, 3 * rp, 128);
        const lm_lora* Ls[3] = {q, k, v};
        uint16_t* outs[3] = {Q, K, V};
        const int64_t ns[3] = {nq, nk, nv};
        for (int i = 0; i < 3; ++i) {
            Prob& P = b.prob();
            P.M = (int32_t)T;
            P.N = (int32_t)ns[i];
            P.bn = 256;
            P.tiles_n = (int32_t)((ns[i] + 255) / 256);
            P.n_step = 256;
            P.out_col_step = 256;
            Seg& S0 = seg(P, 0);
            S0.a_map = xmap;
            b.base_k(S0, Ls[i]->W, sc[i]);
            S0.b_rank_off = 128;
            S0.kext = (int32_t)d;
            Seg& S1 = seg(P, 1);
            S1.a_map = amap;
            S1.a_xoff = i * rp;
            S1.b_map[0] = b.map(Ls[i]->B, ns[i], r, r, 128);
            S1.b_rank_off = 128;
            S1.kext = rp;
            P.out0 = outs[i];
            P.ld_out = ns[i];
        }
        LM_TRY(b.launch("qkv.fwd", sms, err, st));
    }
    return LM_OK;
}

extern "C" lm_status lora_qkv_bwd(int64_t T, int64_t d, int64_t nq, int64_t nk, int64_t nv, const uint16_t* X,
                                  const uint16_t* dQ, const uint16_t* dK, const uint16_t* dV, const void* saved,
                                  size_t saved_bytes, const lm_lora* q, const lm_lora* k, const lm_lora* v,
                                  uint16_t* dX, float* dA_q, float* dB_q, float* dA_k, float* dB_k, float* dA_v,
                                  float* dB_v, void* ws, size_t ws_bytes, lm_stream stream) {
    LM_TRY(check_qkv_common(T, d, nq, nk, nv, q, k, v));
    LM_TRY(need_ptr(X, "X"));
    LM_TRY(need_ptr(dQ, "dQ"));
    LM_TRY(need_ptr(dK, "dK"));
    LM_TRY(need_ptr(dV, "dV"));
    LM_TRY(need_ptr(saved, "saved"));
    LM_TRY(need_ptr(dX, "dX"));
    LM_TRY(need_ptr(dA_q, "dA_q"));
    LM_TRY(need_ptr(dB_q, "dB_q"));
    LM_TRY(need_ptr(dA_k, "dA_k"));
    LM_TRY(need_ptr(dB_k, "dB_k"));
    LM_TRY(need_ptr(dA_v, "dA_v"));
    LM_TRY(need_ptr(dB_v, "dB_v"));
    LM_TRY(need_ptr(ws, "ws"));
    const int32_t r = q->r;
    const bool q4 = q->W.kind != LM_WEIGHT_BF16;  // packed 4-bit base (NF4, int4 or NVFP4)
    const QkvPlan PL = plan_qkv(T, d, nq, nk, nv, r);
    if (saved_bytes < PL.saved_total)
        return fail(LM_ERR_WORKSPACE, "saved buffer has %zu bytes, needs %zu", saved_bytes, PL.saved_total);
    if (ws_bytes < PL.ws_total) return fail(LM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, PL.ws_total);
    const size_t ad = (size_t)r * d * 4;
    LM_TRY(check_alias({{dX, (size_t)T * d * 2, "dX"}, {dA_q, ad, "dA_q"}, {dA_k, ad, "dA_k"}, {dA_v, ad, "dA_v"},
                        {dB_q, (size_t)nq * r * 4, "dB_q"}, {dB_k, (size_t)nk * r * 4, "dB_k"},
                        {dB_v, (size_t)nv * r * 4, "dB_v"}, {ws, PL.ws_total, "ws"}},
                       {{X, (size_t)T * d * 2, "X"}, {dQ, (size_t)T * nq * 2, "dQ"}, {dK, (size_t)T * nk * 2, "dK"},
                        {dV, (size_t)T * nv * 2, "dV"}, {saved, PL.saved_total, "saved"}, wspan(q, "q.W"),
                        wspan(k, "k.W"), wspan(v, "v.W")}));
    cudaStream_t st = (cudaStream_t)stream;
    if (T == 0) {
        LM_CUDA(cudaMemsetAsync(dA_q, 0, ad, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dA_k, 0, ad, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dA_v, 0, ad, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dB_q, 0, (size_t)nq * r * 4, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dB_k, 0, (size_t)nk * r * 4, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dB_v, 0, (size_t)nv * r * 4, st), "cudaMemsetAsync");
        return LM_OK;
    }
    int sms = 0;
    LM_TRY(ready(&sms));
    const Dims& D = PL.D;
    const int rp = D.rp;
    int32_t* err = static_cast<int32_t*>(ws);
    float* part = at<float>(ws, PL.part);
    lm_lora q_c = *q, k_c = *k, v_c = *v;
    LM_TRY(ab_to_bf16("qkv.ab", {{&q_c, d, nq}, {&k_c, d, nk}, {&v_c, d, nv}}, at<uint16_t>(ws, PL.abc), st));
    q = &q_c;
    k = &k_c;
    v = &v_c;
    float* sc[3] = {at<float>(ws, PL.sc[0]), at<float>(ws, PL.sc[1]), at<float>(ws, PL.sc[2])};
    FinSide side;  // the NF4 tables: side work of the G finalisation, before the dX GEMM
    side_scale_tables(side, {{&q->W, sc[0]}, {&k->W, sc[1]}, {&v->W, sc[2]}});
    const uint16_t* xaT = at<uint16_t>(saved, PL.xa.t_off);
    const lm_lora* Ls[3] = {q, k, v};
    const uint16_t* dOut[3] = {dQ, dK, dV};
    const int64_t ns[3] = {nq, nk, nv};
    uint16_t* g[3];
    uint16_t* gT[3];
    for (int i = 0; i < 3; ++i) {
        g[i] = at<uint16_t>(ws, PL.g[i].rows_off);
        gT[i] = at<uint16_t>(ws, PL.g[i].t_off);
    }
    // the dual rank-r reduction reads each dOut_x once for both G_x and dB_x, where that pays
    const DualShape ds = plan_dual(T, {nq, nk, nv}, rp, sms);
    float* dps[3] = {at<float>(ws, PL.dpart[0]), at<float>(ws, PL.dpart[1]), at<float>(ws, PL.dpart[2])};
    if (ds.use) {  // G_x = s_x dOut_x B_x once per projection, and dB_x's partials
        float* gps[3];
        for (int i = 0; i < 3; ++i) gps[i] = part + (size_t)i * kDualMaxSplits * T * rp;  // in the split-K partial region
        DualLaunch L;
        for (int i = 0; i < 3; ++i)
            L.add(dOut[i], T, ns[i], Ls[i]->B, r, xaT, 3 * rp, i * rp, D.ldT, rp, ds, gps[i], dps[i]);
        LM_TRY(L.launch("qkv.g", sms, rp, err, st));
        LM_TRY(fin_rows_split(
            "qkv.g.fin",
            {FinRowJob{gps[0], T * rp, dual_ranges(nq, ds.CB), rp, rp, {q->s, 0.f, 0.f}, g[0], gT[0], D.ldT},
             FinRowJob{gps[1], T * rp, dual_ranges(nk, ds.CB), rp, rp, {k->s, 0.f, 0.f}, g[1], gT[1], D.ldT},
             FinRowJob{gps[2], T * rp, dual_ranges(nv, ds.CB), rp, rp, {v->s, 0.f, 0.f}, g[2], gT[2], D.ldT}},
            T, st, &side));
    } else {  // G_x = s_x dOut_x B_x, formed once per projection
        Builder b(G_PART_KMN);
        float* parts[3];
        for (int i = 0; i < 3; ++i) {
            parts[i] = part + (size_t)i * kMaxSplits * T * rp;
            add_rowproj_out(b, dOut[i], T, ns[i], Ls[i]->B, D, parts[i]);
        }
        LM_TRY(b.launch("qkv.g", sms, err, st));
        LM_TRY(fin_rows("qkv.g.fin", b,
                        {FinRowJob{parts[0], T * rp, 0, rp, rp, {q->s, 0.f, 0.f}, g[0], gT[0], D.ldT},
                         FinRowJob{parts[1], T * rp, 0, rp, rp, {k->s, 0.f, 0.f}, g[1], gT[1], D.ldT},
                         FinRowJob{parts[2], T * rp, 0, rp, rp, {v->s, 0.f, 0.f}, g[2], gT[2], D.ldT}},
                        T, st, &side));
    }
    {  // dA_x^T = X^T G_x (one pass over X for q, k, v: G_q, G_k, G_v are stacked), dB_x = dOut_x^T (s X A_x^T)
        ColReduce cr(D, part);
        if (3 * rp <= 64) {
            cr.add(X, d, gT[0], {dA_q, dA_k, dA_v}, 1);
        } else {
            cr.add(X, d, gT[0], {dA_q}, 1);
            cr.add(X, d, gT[1], {dA_k}, 1);
            cr.add(X, d, gT[2], {dA_v}, 1);
        }
        if (ds.use) {
            float* dBs[3] = {dB_q, dB_k, dB_v};
            for (int i = 0; i < 3; ++i) cr.add_fin(FinColJob{dps[i], ns[i] * rp, ns[i], ds.nrr, rp, r, 0, dBs[i], rp});
        } else {
            cr.add(dQ, nq, xaT, {dB_q}, 0);
            cr.add(dK, nk, xaT + (size_t)rp * D.ldT, {dB_k}, 0);
            cr.add(dV, nv, xaT + (size_t)2 * rp * D.ldT, {dB_v}, 0);
        }
        LM_TRY(cr.run("qkv.dAdB", "qkv.dAdB.fin", sms, err, st));
    }
    {  // dX = sum_x dOut_x W_x + G_x A_x
        Builder b(q4 ? G2N_STORE_MN : G2_STORE_MN);
        if (q4) b.tail_buf = at<float>(ws, PL.tail);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)d;
        P.bn = 256;
        P.tiles_n = (int32_t)((d + 255) / 256);
        P.n_step = 256;
        P.out_col_step = 256;
        for (int i = 0; i < 3; ++i) {
            Seg& S = seg(P, i);
            S.a_map = b.map(dOut[i], T, ns[i], ns[i], 128);
            b.base_mn(S, Ls[i]->W, sc[i]);
            S.b_rank_off = 128;
            S.kext = (int32_t)ns[i];
        }
        for (int i = 0; i < 3; ++i) {
            Seg& S = seg(P, 3 + i);
            S.a_map = b.map(g[i], T, rp, rp, 128);
            S.b_map[0] = b.map(Ls[i]->A, r, d, d, 64);
            S.b_rank_off = 128;
            S.kext = rp;
        }
        P.out0 = dX;
        P.ld_out = d;
        LM_TRY(b.launch("qkv.dX", sms, err, st));
    }
    return LM_OK;
}

// ====================================================================== LoRA O
extern "C" lm_status lora_o_saved_size(int64_t T, int32_t r, size_t* bytes) {
    if (!bytes) return fail(LM_ERR_NULL, "bytes is NULL");
    LM_TRY(check_T(T));
    LM_TRY(check_r(r));
    *bytes = plan_o(T, 32, 32, r).saved_total;
    return LM_OK;
}

extern "C" lm_status lora_o_workspace_size(int64_t T, int64_t d_in, int64_t d_out, int32_t r, size_t* bytes) {
    if (!bytes) return fail(LM_ERR_NULL, "bytes is NULL");
    LM_TRY(check_T(T));
    LM_TRY(check_dim(d_in, "d_in"));
    LM_TRY(check_dim(d_out, "d_out"));
    LM_TRY(check_r(r));
    *bytes = plan_o(T, d_in, d_out, r).ws_total;
    return LM_OK;
}

static lm_status check_o_common(int64_t T, int64_t d_in, int64_t d_out, const lm_lora* o) {
    LM_TRY(check_T(T));
    LM_TRY(check_dim(d_in, "d_in"));
    LM_TRY(check_dim(d_out, "d_out"));
    if (!o) return fail(LM_ERR_NULL, "o is NULL");
    LM_TRY(check_r(o->r));
    LM_TRY(check_lora(o, "o", d_in, d_out, o->r));
    return LM_OK;
}

extern "C" lm_status lora_o_fwd(int64_t T, int64_t d_in, int64_t d_out, const uint16_t* X, const lm_lora* o,
                                uint16_t* Y, void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                                lm_stream stream) {
    LM_TRY(check_o_common(T, d_in, d_out, o));
    LM_TRY(need_ptr(X, "X"));
    LM_TRY(need_ptr(Y, "Y"));
    LM_TRY(need_ptr(saved, "saved"));
    LM_TRY(need_ptr(ws, "ws"));
    const int32_t r = o->r;
    const bool q4 = o->W.kind != LM_WEIGHT_BF16;  // packed 4-bit base (NF4, int4 or NVFP4)
    const OPlan PL = plan_o(T, d_in, d_out, r);
    if (saved_bytes < PL.saved_total)
        return fail(LM_ERR_WORKSPACE, "saved buffer has %zu bytes, needs %zu", saved_bytes, PL.saved_total);
    if (ws_bytes < PL.ws_total) return fail(LM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, PL.ws_total);
    LM_TRY(check_alias({{Y, (size_t)T * d_out * 2, "Y"}, {saved, PL.saved_total, "saved"}, {ws, PL.ws_total, "ws"}},
                       {{X, (size_t)T * d_in * 2, "X"}, wspan(o, "o.W")}));
    if (T == 0) return LM_OK;
    int sms = 0;
    LM_TRY(ready(&sms));
    cudaStream_t st = (cudaStream_t)stream;
    const Dims& D = PL.D;
    const int rp = D.rp;
    int32_t* err = static_cast<int32_t*>(ws);
    float* part = at<float>(ws, PL.part);
    lm_lora o_c = *o;
    LM_TRY(ab_to_bf16("o.ab", {{&o_c, d_in, d_out}}, at<uint16_t>(ws, PL.abc), st));
    o = &o_c;
    float* sc = at<float>(ws, PL.sc);
    FinSide side;  // the NF4 table of W_o: side work of the X A^T finalisation
    side_scale_tables(side, {{&o->W, sc}});
    uint16_t* xa = at<uint16_t>(saved, PL.xa.rows_off);
    uint16_t* xaT = at<uint16_t>(saved, PL.xa.t_off);
    {
        Builder b(G_PART_KK);
        add_rowproj_in(b, X, T, d_in, {o->A}, D, part);
        LM_TRY(b.launch("o.xa", sms, err, st));
        LM_TRY(fin_rows("o.xa.fin", b, {FinRowJob{part, T * rp, 0, rp, rp, {o->s, 0.f, 0.f}, xa, xaT, D.ldT}}, T, st, &side));
    }
    // (a bf16 base keeps the 256 x 256 kernel: see the QKV forward)
    {
        Builder b(q4 ? G2N_STORE_K : G2_STORE_K);
        if (q4) b.tail_buf = at<float>(ws, PL.tail);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)d_out;
        P.bn = 256;
        P.tiles_n = (int32_t)((d_out + 255) / 256);
        P.n_step = 256;
        P.out_col_step = 256;
        Seg& S0 = seg(P, 0);
        S0.a_map = b.map(X, T, d_in, d_in, 128);
        b.base_k(S0, o->W, sc);
        S0.b_rank_off = 128;
        S0.kext = (int32_t)d_in;
        Seg& S1 = seg(P, 1);
        S1.a_map = b.map(xa, T, rp, rp, 128);
        S1.b_map[0] = b.map(o->B, d_out, r, r, 128);
        S1.b_rank_off = 128;
        S1.kext = rp;
        P.out0 = Y;
        P.ld_out = d_out;
        LM_TRY(b.launch("o.fwd", sms, err, st));
    }
    return LM_OK;
}

// Every argument check of lora_o_bwd; touches no device state.  With lib_ws the scratch is the
// library's own array (lora_o_bwd_static): ws and ws_bytes are not looked at, the caller has
// checked the scratch size, and no caller buffer can overlap a __device__ array of the library.
namespace lm {
lm_status check_o_bwd_args(int64_t T, int64_t d_in, int64_t d_out, const uint16_t* X, const uint16_t* dY,
                           const void* saved, size_t saved_bytes, const lm_lora* o, uint16_t* dX, float* dA,
                           float* dB, void* ws, size_t ws_bytes, bool lib_ws) {
    LM_TRY(check_o_common(T, d_in, d_out, o));
    LM_TRY(need_ptr(X, "X"));
    LM_TRY(need_ptr(dY, "dY"));
    LM_TRY(need_ptr(saved, "saved"));
    LM_TRY(need_ptr(dX, "dX"));
    LM_TRY(need_ptr(dA, "dA"));
    LM_TRY(need_ptr(dB, "dB"));
    if (!lib_ws) LM_TRY(need_ptr(ws, "ws"));
    const int32_t r = o->r;
    const OPlan PL = plan_o(T, d_in, d_out, r);
    if (saved_bytes < PL.saved_total)
        return fail(LM_ERR_WORKSPACE, "saved buffer has %zu bytes, needs %zu", saved_bytes, PL.saved_total);
    if (!lib_ws && ws_bytes < PL.ws_total)
        return fail(LM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, PL.ws_total);
    const Span ins[] = {{X, (size_t)T * d_in * 2, "X"}, {dY, (size_t)T * d_out * 2, "dY"},
                        {saved, PL.saved_total, "saved"}, wspan(o, "o.W")};
    if (lib_ws)
        LM_TRY(check_alias({{dX, (size_t)T * d_in * 2, "dX"}, {dA, (size_t)r * d_in * 4, "dA"},
                            {dB, (size_t)d_out * r * 4, "dB"}},
                           {ins[0], ins[1], ins[2], ins[3]}));
    else
        LM_TRY(check_alias({{dX, (size_t)T * d_in * 2, "dX"}, {dA, (size_t)r * d_in * 4, "dA"},
                            {dB, (size_t)d_out * r * 4, "dB"}, {ws, PL.ws_total, "ws"}},
                           {ins[0], ins[1], ins[2], ins[3]}));
    return LM_OK;
}
}  // namespace lm

extern "C" lm_status lora_o_bwd(int64_t T, int64_t d_in, int64_t d_out, const uint16_t* X, const uint16_t* dY,
                                const void* saved, size_t saved_bytes, const lm_lora* o, uint16_t* dX, float* dA,
                                float* dB, void* ws, size_t ws_bytes, lm_stream stream) {
    LM_TRY(check_o_bwd_args(T, d_in, d_out, X, dY, saved, saved_bytes, o, dX, dA, dB, ws, ws_bytes, false));
    const int32_t r = o->r;
    const bool q4 = o->W.kind != LM_WEIGHT_BF16;  // packed 4-bit base (NF4, int4 or NVFP4)
    const OPlan PL = plan_o(T, d_in, d_out, r);
    cudaStream_t st = (cudaStream_t)stream;
    if (T == 0) {
        LM_CUDA(cudaMemsetAsync(dA, 0, (size_t)r * d_in * 4, st), "cudaMemsetAsync");
        LM_CUDA(cudaMemsetAsync(dB, 0, (size_t)d_out * r * 4, st), "cudaMemsetAsync");
        return LM_OK;
    }
    int sms = 0;
    LM_TRY(ready(&sms));
    const Dims& D = PL.D;
    const int rp = D.rp;
    int32_t* err = static_cast<int32_t*>(ws);
    float* part = at<float>(ws, PL.part);
    lm_lora o_c = *o;
    LM_TRY(ab_to_bf16("o.ab", {{&o_c, d_in, d_out}}, at<uint16_t>(ws, PL.abc), st));
    o = &o_c;
    float* sc = at<float>(ws, PL.sc);
    FinSide side;  // the NF4 table of W_o: side work of the G finalisation, before the dX GEMM
    side_scale_tables(side, {{&o->W, sc}});
    const uint16_t* xaT = at<uint16_t>(saved, PL.xa.t_off);
    uint16_t* g = at<uint16_t>(ws, PL.g.rows_off);
    uint16_t* gT = at<uint16_t>(ws, PL.g.t_off);
    // the dual rank-r reduction reads dY once for both G and dB, where that pays
    const DualShape ds = plan_dual(T, {d_out}, rp, sms);
    float* dpo = at<float>(ws, PL.dpart);
    if (ds.use) {  // G = s dY B, formed once (feeds dA and dX), and dB's partials
        float* gpo = part;  // in the split-K partial region
        DualLaunch L;
        L.add(dY, T, d_out, o->B, r, xaT, rp, 0, D.ldT, rp, ds, gpo, dpo);
        LM_TRY(L.launch("o.g", sms, rp, err, st));
        LM_TRY(fin_rows_split(
            "o.g.fin", {FinRowJob{gpo, T * rp, dual_ranges(d_out, ds.CB), rp, rp, {o->s, 0.f, 0.f}, g, gT, D.ldT}}, T, st,
            &side));
    } else {  // G = s dY B, formed once (feeds dA and dX)
        Builder b(G_PART_KMN);
        add_rowproj_out(b, dY, T, d_out, o->B, D, part);
        LM_TRY(b.launch("o.g", sms, err, st));
        LM_TRY(fin_rows("o.g.fin", b, {FinRowJob{part, T * rp, 0, rp, rp, {o->s, 0.f, 0.f}, g, gT, D.ldT}}, T, st, &side));
    }
    {  // dA^T = X^T G, dB = dY^T (s X A^T)
        ColReduce cr(D, part);
        cr.add(X, d_in, gT, {dA}, 1);
        if (ds.use) cr.add_fin(FinColJob{dpo, d_out * rp, d_out, ds.nrr, rp, r, 0, dB, rp});
        else cr.add(dY, d_out, xaT, {dB}, 0);
        LM_TRY(cr.run("o.dAdB", "o.dAdB.fin", sms, err, st));
    }
    {  // dX = dY W + G A
        Builder b(q4 ? G2N_STORE_MN : G2_STORE_MN);
        if (q4) b.tail_buf = at<float>(ws, PL.tail);
        Prob& P = b.prob();
        P.M = (int32_t)T;
        P.N = (int32_t)d_in;
        P.bn = 256;
        P.tiles_n = (int32_t)((d_in + 255) / 256);
        P.n_step = 256;
        P.out_col_step = 256;
        Seg& S0 = seg(P, 0);
        S0.a_map = b.map(dY, T, d_out, d_out, 128);
        b.base_mn(S0, o->W, sc);
        S0.b_rank_off = 128;
        S0.kext = (int32_t)d_out;
        Seg& S1 = seg(P, 1);
        S1.a_map = b.map(g, T, rp, rp, 128);
        S1.b_map[0] = b.map(o->A, r, d_in, d_in, 64);
        S1.b_rank_off = 128;
        S1.kext = rp;
        P.out0 = dX;
        P.ld_out = d_in;
        LM_TRY(b.launch("o.dX", sms, err, st));
    }
    return LM_OK;
}

// ====================================================================== NF4
extern "C" lm_status nf4_pack(const uint16_t* W, int64_t numel, uint8_t* codes, int8_t* absmax_q, float* group_scale,
                              lm_stream stream) {
    if (numel < 0 || numel % 16384 != 0)
        return fail(LM_ERR_SHAPE, "numel = %lld must be a non-negative multiple of 64*256", (long long)numel);
    LM_TRY(need_ptr(W, "W"));
    LM_TRY(need_ptr(codes, "codes"));
    LM_TRY(need_ptr(absmax_q, "absmax_q"));
    LM_TRY(need_ptr(group_scale, "group_scale"));
    LM_TRY(check_alias({{codes, (size_t)numel / 2, "codes"}, {absmax_q, (size_t)numel / 64, "absmax_q"},
                        {group_scale, (size_t)numel / 16384 * 4, "group_scale"}},
                       {{W, (size_t)numel * 2, "W"}}));
    if (numel == 0) return LM_OK;
    int sms = 0;
    LM_TRY(device_sms(&sms));
    const cudaError_t e = launch_nf4_pack(W, numel, codes, absmax_q, group_scale, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "nf4_pack launch");
    return LM_OK;
}

extern "C" lm_status nf4_dequant(const uint8_t* codes, const int8_t* absmax_q, const float* group_scale, int64_t numel,
                                 int32_t out_dtype, void* out, lm_stream stream) {
    if (numel < 0 || numel % 16384 != 0)
        return fail(LM_ERR_SHAPE, "numel = %lld must be a non-negative multiple of 64*256", (long long)numel);
    if (out_dtype != LM_OUT_F32 && out_dtype != LM_OUT_BF16)
        return fail(LM_ERR_DTYPE, "out_dtype = %d is not known", out_dtype);
    LM_TRY(need_ptr(codes, "codes"));
    LM_TRY(need_ptr(absmax_q, "absmax_q"));
    LM_TRY(need_ptr(group_scale, "group_scale"));
    LM_TRY(need_ptr(out, "out"));
    const size_t ob = (size_t)numel * (out_dtype == LM_OUT_F32 ? 4 : 2);
    LM_TRY(check_alias({{out, ob, "out"}}, {{codes, (size_t)numel / 2, "codes"},
                                            {absmax_q, (size_t)numel / 64, "absmax_q"},
                                            {group_scale, (size_t)numel / 16384 * 4, "group_scale"}}));
    if (numel == 0) return LM_OK;
    int sms = 0;
    LM_TRY(device_sms(&sms));
    const cudaError_t e =
        launch_nf4_dequant(codes, absmax_q, group_scale, numel, out_dtype == LM_OUT_BF16, out, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "nf4_dequant launch");
    return LM_OK;
}

// ====================================================================== int4
namespace {
lm_status check_int4_shape(int64_t rows, int64_t cols, int32_t group) {
    if (group != 32 && group != 64 && group != 128 && group != 256)
        return fail(LM_ERR_SHAPE, "group = %d: an int4 group holds 32, 64, 128 or 256 elements", group);
    if (rows < 0 || cols < 0 || cols % group != 0 || rows > (int64_t(1) << 24) || cols > (int64_t(1) << 24))
        return fail(LM_ERR_SHAPE, "an int4 weight of %lld x %lld needs cols a multiple of the group (%d)",
                    (long long)rows, (long long)cols, group);
    return LM_OK;
}
}  // namespace

extern "C" lm_status int4_pack(const uint16_t* W, int64_t rows, int64_t cols, int32_t group, uint8_t* codes,
                               uint16_t* scale_zero, lm_stream stream) {
    LM_TRY(check_int4_shape(rows, cols, group));
    LM_TRY(need_ptr(W, "W"));
    LM_TRY(need_ptr(codes, "codes"));
    LM_TRY(need_ptr(scale_zero, "scale_zero"));
    const int64_t numel = rows * cols;
    LM_TRY(check_alias({{codes, (size_t)numel / 2, "codes"}, {scale_zero, (size_t)(numel / group) * 4, "scale_zero"}},
                       {{W, (size_t)numel * 2, "W"}}));
    if (numel == 0) return LM_OK;
    int sms = 0;
    LM_TRY(device_sms(&sms));
    const cudaError_t e = launch_int4_pack(W, rows, cols, group, codes, reinterpret_cast<uint32_t*>(scale_zero),
                                           (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "int4_pack launch");
    return LM_OK;
}

extern "C" lm_status int4_dequant(const uint8_t* codes, const uint16_t* scale_zero, int64_t rows, int64_t cols,
                                  int32_t group, int32_t out_dtype, void* out, lm_stream stream) {
    LM_TRY(check_int4_shape(rows, cols, group));
    if (out_dtype != LM_OUT_F32 && out_dtype != LM_OUT_BF16)
        return fail(LM_ERR_DTYPE, "out_dtype = %d is not known", out_dtype);
    LM_TRY(need_ptr(codes, "codes"));
    LM_TRY(need_ptr(scale_zero, "scale_zero"));
    LM_TRY(need_ptr(out, "out"));
    const int64_t numel = rows * cols;
    const size_t ob = (size_t)numel * (out_dtype == LM_OUT_F32 ? 4 : 2);
    LM_TRY(check_alias({{out, ob, "out"}}, {{codes, (size_t)numel / 2, "codes"},
                                            {scale_zero, (size_t)(numel / group) * 4, "scale_zero"}}));
    if (numel == 0) return LM_OK;
    int sms = 0;
    LM_TRY(device_sms(&sms));
    const cudaError_t e = launch_int4_dequant(codes, reinterpret_cast<const uint32_t*>(scale_zero), rows, cols, group,
                                              out_dtype == LM_OUT_BF16, out, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "int4_dequant launch");
    return LM_OK;
}

// ====================================================================== NVFP4
extern "C" lm_status nvfp4_pack(const uint16_t* W, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* block_scale,
                                float* global_scale, lm_stream stream) {
    if (rows < 0 || cols < 0 || cols % 64 != 0 || rows > (int64_t(1) << 24) || cols > (int64_t(1) << 24))
        return fail(LM_ERR_SHAPE, "an NVFP4 weight of %lld x %lld needs cols a multiple of 64", (long long)rows,
                    (long long)cols);
    LM_TRY(need_ptr(W, "W"));
    LM_TRY(need_ptr(codes, "codes"));
    LM_TRY(need_ptr(block_scale, "block_scale"));
    LM_TRY(need_ptr4(global_scale, "global_scale"));
    const int64_t numel = rows * cols;
    LM_TRY(check_alias({{codes, (size_t)numel / 2, "codes"}, {block_scale, (size_t)numel / 16, "block_scale"},
                        {global_scale, 4, "global_scale"}},
                       {{W, (size_t)numel * 2, "W"}}));
    if (numel == 0) return LM_OK;
    int sms = 0;
    LM_TRY(device_sms(&sms));
    const cudaError_t e = launch_nvfp4_pack(W, rows, cols, codes, block_scale, global_scale, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "nvfp4_pack launch");
    return LM_OK;
}

extern "C" lm_status nvfp4_dequant(const uint8_t* codes, const uint8_t* block_scale, const float* global_scale,
                                   int64_t rows, int64_t cols, int32_t out_dtype, void* out, lm_stream stream) {
    if (rows < 0 || cols < 0 || cols % 64 != 0 || rows > (int64_t(1) << 24) || cols > (int64_t(1) << 24))
        return fail(LM_ERR_SHAPE, "an NVFP4 weight of %lld x %lld needs cols a multiple of 64", (long long)rows,
                    (long long)cols);
    if (out_dtype != LM_OUT_F32 && out_dtype != LM_OUT_BF16)
        return fail(LM_ERR_DTYPE, "out_dtype = %d is not known", out_dtype);
    LM_TRY(need_ptr(codes, "codes"));
    LM_TRY(need_ptr(block_scale, "block_scale"));
    LM_TRY(need_ptr4(global_scale, "global_scale"));
    LM_TRY(need_ptr(out, "out"));
    const int64_t numel = rows * cols;
    const size_t ob = (size_t)numel * (out_dtype == LM_OUT_F32 ? 4 : 2);
    LM_TRY(check_alias({{out, ob, "out"}}, {{codes, (size_t)numel / 2, "codes"},
                                            {block_scale, (size_t)numel / 16, "block_scale"},
                                            {global_scale, 4, "global_scale"}}));
    if (numel == 0) return LM_OK;
    int sms = 0;
    LM_TRY(device_sms(&sms));
    const cudaError_t e = launch_nvfp4_dequant(codes, block_scale, global_scale, rows, cols,
                                               out_dtype == LM_OUT_BF16, out, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "nvfp4_dequant launch");
    return LM_OK;
}
