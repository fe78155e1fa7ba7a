/*
 * lora_mlp.h -- C ABI of the GB300 (sm_103a) fused LoRA MLP / QKV / O library.
 *
 * The library computes the LoRA-adapted MLP block, the LoRA Q/K/V projections and the LoRA
 * output projection, forward and backward, on one GPU, with hand-written tcgen05/TMA kernels.
 *
 * Where the operations are defined (web pages on the subject):
 *   [LO]  "LoRA Optimizations" (docs.axolotl.ai, lora_optims): sections "Custom autograd
 *         functions" (LoRA MLP, QKV and O functions), "Triton kernels" (SwiGLU / GeGLU forward
 *         and backward), "Requirements" (no dropout, no bias on adapted projections) and
 *         "FP32 LoRA gradients" (bf16 GEMM inputs, fp32 parameter-gradient outputs).
 *   [UN]  "Avoid recomputing LoRA B-projected gradient in fused-LoRA backward" (unsloth
 *         fast_lora diff): LoRA_MLP.backward, LoRA_QKV.backward, LoRA_W.backward and
 *         matmul_lora; dY.B^T is formed once per projection and reused for dA and dX.
 *   [LL]  "loralei" README, QLoRA section: NF4 base weights with 64-element blocks and
 *         double-quantised block scales (256 blocks per scale), dimensions divisible by 32,
 *         unpacking and double-scale reconstruction fused into the matmul; the alternative
 *         groupwise int4 base (group sizes 32, 64, 128, 256), input gradients from the packed
 *         weight.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layouts are the PEFT nn.Linear ones ([UN] matmul_lora computes X @ W.t()): a base weight
 *    W is (out, in) row-major; LoRA A is (r, in); LoRA B is (out, r); activations are (T, in)
 *    or (T, out) row-major with T = batch * sequence flattened.  The LoRA term of a projection
 *    is s * (X A^T) B^T with s = alpha / r (or alpha / sqrt(r) for rsLoRA: the caller passes s).
 *  - bf16 tensors are passed as uint16_t bit patterns.  Activations are bf16; A and B are bf16
 *    or fp32 (lm_lora.ab_dtype: fp32 LoRA parameters, [LO] "FP32 LoRA gradients", enter the
 *    GEMMs rounded to bf16, round-to-nearest-even); LoRA gradients are fp32 and are written in
 *    parameter layout (dA: r x in, dB: out x r), overwriting the destination ([UN]: the
 *    weight-gradient GEMMs use beta = 0).
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise.  The caller owns every
 *    buffer, including the workspace; the library allocates no device memory and keeps no state
 *    other than a per-thread last-error string, cached function pointers and per-device launch
 *    attributes.  The one exception is lora_o_bwd_static below, whose scratch is a fixed
 *    64 MiB __device__ array of the library on every GPU that loads it.
 *  - Every compute call is asynchronous on the given stream (a cudaStream_t; NULL is the legacy
 *    default stream) and never synchronises.  Calls that share a workspace or a saved buffer
 *    must be ordered (same stream or explicit events).
 *  - Sizes: T >= 0 (T == 0 is a no-op), feature sizes > 0 and multiples of 32 ([LL]), 8 <= r <= 64
 *    with r a multiple of 8.  Base pointers must be 32-byte aligned (TMA wants 16 bytes; the
 *    epilogues move 32-byte chunks of rows).  Outputs must not
 *    overlap inputs (the in-place dX of [UN] is not offered).
 *  - Errors: every call returns an lm_status; no exception or abort crosses the ABI.  Argument
 *    errors are detected on the host before anything is enqueued.  Kernels never trap: a
 *    pipeline wait that exceeds its time limit records LM_ERR_TIMEOUT in the workspace's error
 *    word and the kernel returns; lm_workspace_check() reads and clears that word.
 *  - Workspace: the first 256 bytes hold the error word.  Zero them once after allocation
 *    (lm_workspace_reset) -- the kernels only ever set them.
 */
#ifndef LORA_MLP_H
#define LORA_MLP_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LM_API __attribute__((visibility("default")))
#else
#define LM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* lm_stream; /* identical to cudaStream_t */

typedef enum lm_status {
    LM_OK = 0,
    LM_ERR_NULL = 1,        /* a required pointer is NULL */
    LM_ERR_SHAPE = 2,       /* a size breaks the rules above */
    LM_ERR_ALIGN = 3,       /* a pointer is not 32-byte aligned */
    LM_ERR_DTYPE = 4,       /* unknown weight kind, activation or output dtype */
    LM_ERR_ALIAS = 5,       /* an output overlaps an input or another output */
    LM_ERR_WORKSPACE = 6,   /* workspace or saved buffer smaller than the size query returns */
    LM_ERR_CUDA = 7,        /* a CUDA runtime / driver call failed (see lm_last_error) */
    LM_ERR_TIMEOUT = 8,     /* a kernel gave up on a bounded wait (lm_workspace_check) */
    LM_ERR_UNSUPPORTED = 9  /* no device of compute capability 10.3, or a combination not built */
} lm_status;

typedef enum lm_weight_kind {
    LM_WEIGHT_BF16 = 0,
    LM_WEIGHT_NF4 = 1,
    LM_WEIGHT_INT4 = 2,
    LM_WEIGHT_NVFP4 = 3
} lm_weight_kind;
typedef enum lm_act { LM_ACT_SWIGLU = 0, LM_ACT_GEGLU_ERF = 1 } lm_act;
typedef enum lm_out_dtype { LM_OUT_F32 = 0, LM_OUT_BF16 = 1 } lm_out_dtype;
typedef enum lm_ab_dtype { LM_AB_BF16 = 0, LM_AB_F32 = 1 } lm_ab_dtype;

/* A frozen base weight W (out x in).  kind == LM_WEIGHT_BF16: `w` holds rows*cols bf16.
 * kind == LM_WEIGHT_NF4 ([LL]): `codes` holds rows*cols/2 bytes (element 2i in the high nibble
 * of byte i), `absmax_q` rows*cols/64 int8 block scales and `group_scale` rows*cols/16384 fp32
 * scales, exactly as nf4_pack writes them; rows*cols must be a multiple of 16384 and cols a
 * multiple of 64.  Element (i, j) decodes to code[idx] * (absmax_q[b] * group_scale[b/256])
 * with b = (i*cols + j)/64, then rounds to bf16 for the matmul.
 * kind == LM_WEIGHT_INT4 ([LL] "int4" groupwise base): `codes` as for NF4 and `scale_zero`
 * 2*rows*cols/group bf16 values, [cols/group][rows][2] (the scale s then the zero z of group g of
 * row i at index 2*(g*rows + i)), exactly as int4_pack writes them; `group` is 32, 64, 128 or 256
 * and cols a multiple of 64 and of group.  Element (i, j) with code q decodes to
 * fp32((q - 8) * s + z) of its group g = j / group, then rounds to bf16 for the matmul.
 * kind == LM_WEIGHT_NVFP4 ([LO] FP32 LoRA gradients: weight-only NVFP4 bases; activations stay
 * bf16): `codes` rows*cols/2 bytes of E2M1 codes (element 2i in the LOW nibble of byte i),
 * `block_scale` rows*cols/16 E4M3 bytes, [cols/64][rows][4] (the scale of elements
 * [16k, 16k+16) of row i at index ((k/4)*rows + i)*4 + k%4), and `global_scale` one fp32 value
 * on the device (4-byte aligned), exactly as nvfp4_pack writes them; cols a multiple of 64.
 * Element (i, j) decodes to fp32(e2m1(code) * fp32(s_b * global_scale)) with s_b the E4M3 scale
 * of its 16-element block, then rounds to bf16 for the matmul.
 * Unused pointers of a kind are ignored; `group` is ignored unless kind == LM_WEIGHT_INT4. */
typedef struct lm_weight {
    int32_t kind;
    int32_t group;             /* LM_WEIGHT_INT4: elements per quantisation group */
    int64_t rows;              /* out_features */
    int64_t cols;              /* in_features  */
    const uint16_t* w;
    const uint8_t* codes;
    const int8_t* absmax_q;
    const float* group_scale;
    const uint16_t* scale_zero;
    const uint8_t* block_scale;
    const float* global_scale;
} lm_weight;

/* One adapted projection: base W, A (r x in), B (out x r), rank r and scale s.  A and B hold
 * bf16 bits (ab_dtype LM_AB_BF16) or fp32 values (LM_AB_F32: [LO] "FP32 LoRA gradients" keeps
 * the trainable parameters in fp32; each call rounds them to bf16 into its workspace, RNE, and
 * every GEMM reads the bf16 copy).  Any other ab_dtype is LM_ERR_DTYPE. */
typedef struct lm_lora {
    lm_weight W;
    const void* A;
    const void* B;
    int32_t r;
    float s;
    int32_t ab_dtype;
    int32_t reserved;
} lm_lora;

/* ---- utilities ------------------------------------------------------------------------- */

/* Text of the last error raised on the calling thread ("" if none).  Host only. */
LM_API const char* lm_last_error(void);

/* The 16 fp32 NF4 code values the kernels use, ascending ([LL]; NormalFloat-4 of the QLoRA
 * paper).  Host only: `out` is a host array of 16 floats.  Never fails for a non-NULL out. */
LM_API lm_status lm_nf4_codebook(float* out);

/* Zero the error word at the start of a workspace (enqueued on `stream`). */
LM_API lm_status lm_workspace_reset(void* ws, lm_stream stream);

/* Synchronise `stream`, read the workspace's error word, clear it, and return LM_ERR_TIMEOUT if
 * a kernel recorded a timeout since the last reset (LM_OK otherwise).  This call synchronises. */
LM_API lm_status lm_workspace_check(void* ws, lm_stream stream);

/* Test hook for the timeout path and the planner ([LO] names no failure handling beyond argument
 * validation; the bounded waits are this library's).  Applies to the kernels launched afterwards
 * by the calling thread.  Bits 0-3 of family_mask select kernel families whose TMA producers issue
 * no loads at all -- bit 0 the split-K rank-r kernel, bit 1 the bf16 CTA-pair kernel, bit 2 the
 * packed-base (and plain-store) CTA-pair kernel, bit 3 the dual rank-r reduction -- so their
 * consumers' waits run out, no copy is in flight when they do, and the call's error word reads
 * LM_ERR_TIMEOUT (lm_workspace_check); the outputs of such a call are undefined.  Bit 4 makes the
 * MLP backward take the dual rank-r reductions wherever they are feasible, not only where they
 * are estimated faster (the results are the same up to the order of fp32 additions).  wait_ns
 * sets the time limit of every pipeline wait, in nanoseconds (0: the default, 2 s).
 * lm_debug_inject(0, 0) restores normal operation.  Host only; never fails for a mask in [0, 31]
 * (else LM_ERR_SHAPE). */
LM_API lm_status lm_debug_inject(int32_t family_mask, uint64_t wait_ns);

/* ---- tracing ---------------------------------------------------------------------------
 * When enabled, the library records a CUDA event pair around every kernel it launches, on the
 * launch stream, tagged with the call site (e.g. "mlp.dX").  lm_profile_summary synchronises on
 * the recorded events and writes one line per tag, "tag<TAB>launches<TAB>total_ms\n", into the
 * host buffer `buf` (truncated to buf_len - 1 characters, always NUL-terminated).  Host only;
 * recording costs two cudaEventRecord calls per launch and nothing when disabled. */
LM_API lm_status lm_profile_enable(int32_t on);
LM_API lm_status lm_profile_reset(void);
LM_API lm_status lm_profile_summary(char* buf, size_t buf_len);

/* ---- LoRA MLP ([LO] LoRA MLP autograd function; [UN] LoRA_MLP) -------------------------
 *   e = X Wg^T + sg (X Ag^T) Bg^T,   u = X Wu^T + su (X Au^T) Bu^T,
 *   h = act(e) * u  (act = SiLU or exact-erf GELU),   y = h Wd^T + sd (h Ad^T) Bd^T.
 * gate, up: in = d, out = n.  down: in = n, out = d.  All three must have the same r.
 * The backward produces dX and fp32 dA / dB for the three projections.  It forms
 * Gd = dY Bd, Gg = de Bg and Gu = du Bu once each and uses them both for dA and for dX ([UN]).
 *
 * Buffers: X (T x d), y (T x d), e_save / u_save / h_save (T x n) bf16 written by the forward
 * and read by the backward; `saved` (lora_mlp_saved_size bytes) holds the rank-r products
 * s * X A^T and s * h Ad^T between the two calls.  dX (T x d) bf16.  dA_gate, dA_up (r x d),
 * dB_gate, dB_up (n x r), dA_down (r x n), dB_down (d x r) fp32. */
LM_API lm_status lora_mlp_saved_size(int64_t T, int32_t r, size_t* bytes);
LM_API lm_status lora_mlp_workspace_size(int64_t T, int64_t d, int64_t n, int32_t r, size_t* bytes);

LM_API lm_status lora_mlp_fwd(int64_t T, int64_t d, int64_t n, int32_t act,
                       const uint16_t* X, const lm_lora* gate, const lm_lora* up,
                       const lm_lora* down,
                       uint16_t* y, uint16_t* e_save, uint16_t* u_save, uint16_t* h_save,
                       void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                       lm_stream stream);

LM_API lm_status lora_mlp_bwd(int64_t T, int64_t d, int64_t n, int32_t act,
                       const uint16_t* X, const uint16_t* dY,
                       const uint16_t* e_save, const uint16_t* u_save, const uint16_t* h_save,
                       const void* saved, size_t saved_bytes,
                       const lm_lora* gate, const lm_lora* up, const lm_lora* down,
                       uint16_t* dX, float* dA_gate, float* dB_gate, float* dA_up,
                       float* dB_up, float* dA_down, float* dB_down,
                       void* ws, size_t ws_bytes, lm_stream stream);

/* ---- non-gated ReLU^2 MLP with LoRA up / down projections ([LO] "FP32 LoRA gradients":
 * dense ReLU^2 MLPs use up/down LoRA projections and a fused ReLU^2 activation derivative) ----
 *   u = X Wu^T + su (X Au^T) Bu^T,   h = max(u, 0)^2,   y = h Wd^T + sd (h Ad^T) Bd^T.
 * The backward hoists Gd = sd dY Bd and Gu = su du Bu and fuses the activation derivative into
 * the dh GEMM's epilogue:  dh = dY Wd + Gd Ad,  du = dh * 2 max(u, 0),  dX = du Wu + Gu Au,
 * dAd = Gd^T h, dBd = sd dY^T (h Ad^T), dAu = Gu^T X, dBu = su du^T (X Au^T).  up is d -> n,
 * down is n -> d, same r; bf16 or NF4 base (both the same kind).  X, y, dX (T x d); u_save,
 * h_save (T x n) are written by the forward (u = pre-activation, h = activation, bf16, h taken
 * from the bf16 u) and read by the backward; saved (lora_relu2_mlp_saved_size bytes) holds the
 * rank-r products.  dA_up (r x d), dB_up (n x r), dA_down (r x n), dB_down (d x r) fp32. */
LM_API lm_status lora_relu2_mlp_saved_size(int64_t T, int32_t r, size_t* bytes);
LM_API lm_status lora_relu2_mlp_workspace_size(int64_t T, int64_t d, int64_t n, int32_t r, size_t* bytes);
LM_API lm_status lora_relu2_mlp_fwd(int64_t T, int64_t d, int64_t n, const uint16_t* X, const lm_lora* up,
                                    const lm_lora* down, uint16_t* y, uint16_t* u_save, uint16_t* h_save,
                                    void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                                    lm_stream stream);
LM_API lm_status lora_relu2_mlp_bwd(int64_t T, int64_t d, int64_t n, const uint16_t* X, const uint16_t* dY,
                                    const uint16_t* u_save, const uint16_t* h_save, const void* saved,
                                    size_t saved_bytes, const lm_lora* up, const lm_lora* down, uint16_t* dX,
                                    float* dA_up, float* dB_up, float* dA_down, float* dB_down, void* ws,
                                    size_t ws_bytes, lm_stream stream);

/* ---- LoRA QKV ([LO] query/key/value function; [UN] LoRA_QKV) ---------------------------
 * Q = X Wq^T + sq (X Aq^T) Bq^T, and likewise K (nk columns) and V (nv columns); one read of
 * X feeds all three.  The backward sums the three input gradients into dX.  q, k, v must have
 * the same r.  X, dX (T x d); Q, dQ (T x nq); K, dK (T x nk); V, dV (T x nv) bf16.
 * dA_q/k/v (r x d), dB_q (nq x r), dB_k (nk x r), dB_v (nv x r) fp32. */
LM_API lm_status lora_qkv_saved_size(int64_t T, int32_t r, size_t* bytes);
LM_API lm_status lora_qkv_workspace_size(int64_t T, int64_t d, int64_t nq, int64_t nk, int64_t nv,
                                  int32_t r, size_t* bytes);
LM_API lm_status lora_qkv_fwd(int64_t T, int64_t d, int64_t nq, int64_t nk, int64_t nv,
                       const uint16_t* X, const lm_lora* q, const lm_lora* k, const lm_lora* v,
                       uint16_t* Q, uint16_t* K, uint16_t* V,
                       void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                       lm_stream stream);
LM_API lm_status lora_qkv_bwd(int64_t T, int64_t d, int64_t nq, int64_t nk, int64_t nv,
                       const uint16_t* X, const uint16_t* dQ, const uint16_t* dK,
                       const uint16_t* dV, const void* saved, size_t saved_bytes,
                       const lm_lora* q, const lm_lora* k, const lm_lora* v,
                       uint16_t* dX, float* dA_q, float* dB_q, float* dA_k, float* dB_k,
                       float* dA_v, float* dB_v, void* ws, size_t ws_bytes, lm_stream stream);

/* ---- LoRA O ([LO] output projection function; [UN] LoRA_W) -----------------------------
 * Y = X W^T + s (X A^T) B^T;  backward G = dY B, dA = s G^T X, dB = s dY^T (X A^T),
 * dX = dY W + s G A.  X, dX (T x d_in); Y, dY (T x d_out); dA (r x d_in), dB (d_out x r). */
LM_API lm_status lora_o_saved_size(int64_t T, int32_t r, size_t* bytes);
LM_API lm_status lora_o_workspace_size(int64_t T, int64_t d_in, int64_t d_out, int32_t r,
                                size_t* bytes);
LM_API lm_status lora_o_fwd(int64_t T, int64_t d_in, int64_t d_out, const uint16_t* X,
                     const lm_lora* o, uint16_t* Y, void* saved, size_t saved_bytes,
                     void* ws, size_t ws_bytes, lm_stream stream);
LM_API lm_status lora_o_bwd(int64_t T, int64_t d_in, int64_t d_out, const uint16_t* X,
                     const uint16_t* dY, const void* saved, size_t saved_bytes,
                     const lm_lora* o, uint16_t* dX, float* dA, float* dB,
                     void* ws, size_t ws_bytes, lm_stream stream);

/* lora_o_bwd_static: lora_o_bwd for callers that must not allocate device memory (for example a
 * plugin whose host framework owns the device memory pool, a process under a hard device-memory
 * cap, or a latency-critical loop that cannot afford cudaFree's device-wide wait).  The web pages
 * have no counterpart: this is a deployment variant, not a step of the method.  The arguments and
 * results are those of lora_o_bwd without ws / ws_bytes: the scratch is a 64 MiB __device__ array
 * inside the library, held by every GPU that loads it until the process exits.  Shapes whose
 * lora_o_workspace_size exceeds 64 MiB are rejected with LM_ERR_WORKSPACE, and every other argument
 * error is reported as lora_o_bwd reports it, all before any CUDA call.  The call allocates
 * nothing.  All calls share the one array and it keeps the last call's contents; each call clears
 * the array's error word on its stream, so calls whose kernels overlap on the GPU race and must be
 * ordered by the caller.  Each call looks up the array's address on the current device; the first
 * call on a device may load the library's device code there, so make it before capturing any
 * stream.  lm_static_scratch_check(stream) synchronises `stream`, reads and clears the array's
 * error word and returns LM_ERR_TIMEOUT if a kernel of a static call gave up on a bounded wait
 * since the last check (LM_OK otherwise), as lm_workspace_check does for a workspace. */
LM_API lm_status lora_o_bwd_static(int64_t T, int64_t d_in, int64_t d_out, const uint16_t* X,
                                   const uint16_t* dY, const void* saved, size_t saved_bytes,
                                   const lm_lora* o, uint16_t* dX, float* dA, float* dB,
                                   lm_stream stream);
LM_API lm_status lm_static_scratch_check(lm_stream stream);

/* ---- NF4 ([LL] QLoRA section) -----------------------------------------------------------
 * nf4_pack: quantise numel bf16 values W (flattened row-major) to NF4.  numel must be a
 * multiple of 16384.  Per 64-element block b: absmax_b = max |x|; per group g of 256 blocks:
 * c_g = fp32(max_b absmax_b / 127) -> group_scale[g]; absmax_q[b] = clamp(round-half-even(
 * fp32(absmax_b / c_g)), 0, 127) (0 when c_g == 0).  Each element x of block b is normalised
 * as v = fp32(x / absmax_b) (0 when absmax_b == 0) and coded as the index of the nearest of the
 * 16 NF4 values (lm_nf4_codebook); an exact tie takes the lower index.  codes (numel/2 bytes),
 * absmax_q (numel/64), group_scale (numel/16384) are written.  Bit-exact and deterministic.
 * nf4_dequant: w = fp32(code[idx] * fp32(absmax_q[b] * group_scale[b/256])), written as fp32
 * (out_dtype LM_OUT_F32) or rounded to nearest-even bf16 (LM_OUT_BF16); numel values. */
LM_API lm_status nf4_pack(const uint16_t* W, int64_t numel, uint8_t* codes, int8_t* absmax_q,
                   float* group_scale, lm_stream stream);
LM_API lm_status nf4_dequant(const uint8_t* codes, const int8_t* absmax_q, const float* group_scale,
                      int64_t numel, int32_t out_dtype, void* out, lm_stream stream);

/* ---- int4 groupwise base ([LL] QLoRA section: "int4", group sizes 32, 64, 128, 256) --------
 * int4_pack: quantise a rows x cols bf16 weight W (row-major) in groups of `group` consecutive
 * elements of a row (group 32, 64, 128 or 256; cols a multiple of group; else LM_ERR_SHAPE).
 * Per group, with mn and mx its minimum and maximum: s = bf16(fp32((mx - mn) / 15)),
 * z = bf16(fp32(mn + 8*s)); each element x gets q = clamp(rint(fp32(fp32(x - z) / s)) + 8, 0, 15)
 * (rint: half to even; q = 8 for every element when s == 0).  Writes codes (rows*cols/2 bytes,
 * element 2i in the high nibble of byte i) and scale_zero (2*rows*cols/group bf16 values,
 * [cols/group][rows][2], s before z).  Bit-exact and deterministic.
 * int4_dequant: w = fp32((q - 8) * s + z) (one rounding: the product is exact), written as fp32
 * (LM_OUT_F32) or rounded to nearest-even bf16 (LM_OUT_BF16); rows*cols values, row-major. */
LM_API lm_status int4_pack(const uint16_t* W, int64_t rows, int64_t cols, int32_t group, uint8_t* codes,
                           uint16_t* scale_zero, lm_stream stream);
LM_API lm_status int4_dequant(const uint8_t* codes, const uint16_t* scale_zero, int64_t rows, int64_t cols,
                              int32_t group, int32_t out_dtype, void* out, lm_stream stream);

/* ---- NVFP4 weight-only base ([LO] FP32 LoRA gradients) --------------------------------------
 * nvfp4_pack: quantise a rows x cols bf16 weight W (row-major; cols a multiple of 64, else
 * LM_ERR_SHAPE) to NVFP4 with two-level scaling.  global_scale (one fp32 on the device, 4-byte
 * aligned) = S_g = fp32(amax / 2688), amax = max |W| (S_g = 1 when that is 0); per 16-element
 * block of a row, with bmax its max |x|: s_b = E4M3(fp32(fp32(bmax / 6) / S_g)) (nearest, ties to
 * even, saturated at 448); each element x gets code = E2M1(fp32(x / fp32(s_b * S_g))) (nearest,
 * ties to even, saturated at 6; the sign bit is the sign of x; every code of the block is 0 when
 * s_b * S_g == 0).  Writes codes, block_scale and global_scale in the layout of lm_weight above.
 * Bit-exact and deterministic; three launches (tensor maximum, blocks, tensor scale).
 * nvfp4_dequant: w = fp32(e2m1(code) * fp32(s_b * S_g)), written as fp32 (LM_OUT_F32) or rounded
 * to nearest-even bf16 (LM_OUT_BF16); rows*cols values, row-major. */
LM_API lm_status nvfp4_pack(const uint16_t* W, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* block_scale,
                            float* global_scale, lm_stream stream);
LM_API lm_status nvfp4_dequant(const uint8_t* codes, const uint8_t* block_scale, const float* global_scale,
                               int64_t rows, int64_t cols, int32_t out_dtype, void* out, lm_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* LORA_MLP_H */
