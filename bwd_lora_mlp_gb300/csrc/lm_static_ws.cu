// lora_o_bwd_static: the LoRA output-projection backward with its scratch memory in a fixed,
// library-owned device array instead of a caller-provided workspace.
//
// Who needs it: callers that must not allocate device memory themselves.  Examples are a plugin
// hosted by a framework whose memory pool owns (almost) all of the device memory, a process
// running under a hard device-memory cap where a late cudaMalloc can fail, or a latency-critical
// loop that cannot afford cudaFree, which waits for the whole device.  Such a caller passes only
// its inputs and outputs; this entry point allocates nothing (no cudaMalloc, cudaFree or
// allocating library routine) and runs the same kernels as lora_o_bwd.
//
// The scratch is kStaticWsBytes (64 MiB) of __device__ memory per GPU that loads the library,
// held until the process exits.  It covers the O-projection shapes whose lora_o_workspace_size
// is at most that (for example T = 8192 tokens, 4096 -> 4096, r = 16 needs about 54 MiB);
// larger shapes are rejected with LM_ERR_WORKSPACE before anything is enqueued.  So is every
// other argument error: all of lora_o_bwd's checks run on the host before the first device call.
//
// Sharing: every call, from any thread or stream, uses the same array, and the array keeps what
// the previous call left in it.  Calls whose kernels overlap on the GPU therefore race on the
// scratch and must be ordered by the caller (one stream, or events between streams).  The first
// 256 bytes (the kernels' error word) are cleared on the call's stream at the start of every
// call; the rest is fully rewritten before it is read.  lm_static_scratch_check reads that error
// word back, as lm_workspace_check does for a caller-provided workspace.
//
// Set-up: each call looks up the array's device address on the current device with
// cudaGetSymbolAddress.  Once the library's device code is loaded on a device this is a host-side
// lookup; the first call on a device may load it, so make that first call before capturing any
// stream.  Looking the address up on every call (rather than caching it per device) keeps it right
// after cudaDeviceReset or under another context, where the array may sit at another address.
#include <cuda_runtime.h>

#include "lora_mlp.h"

namespace lm {
lm_status report_error(lm_status s, const char* fmt, ...);
lm_status check_o_bwd_args(int64_t T, int64_t d_in, int64_t d_out, const uint16_t* X, const uint16_t* dY,
                           const void* saved, size_t saved_bytes, const lm_lora* o, uint16_t* dX, float* dA,
                           float* dB, void* ws, size_t ws_bytes, bool lib_ws);
}

namespace {

constexpr size_t kStaticWsBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// device address of the scratch array on the current device
lm_status scratch_address(const char* who, void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess || !p)
        return lm::report_error(LM_ERR_CUDA, "%s: cudaGetSymbolAddress: %s", who, cudaGetErrorString(e));
    *out = p;
    return LM_OK;
}

}  // namespace

extern "C" lm_status lora_o_bwd_static(int64_t T, int64_t d_in, int64_t d_out, const uint16_t* X,
                                       const uint16_t* dY, const void* saved, size_t saved_bytes,
                                       const lm_lora* o, uint16_t* dX, float* dA, float* dB,
                                       lm_stream stream) {
    if (o) {
        size_t need = 0;
        const lm_status qs = lora_o_workspace_size(T, d_in, d_out, o->r, &need);
        if (qs != LM_OK) return qs;  // the size query has set the error text
        if (need > kStaticWsBytes)
            return lm::report_error(LM_ERR_WORKSPACE,
                                    "lora_o_bwd_static: this shape needs %zu bytes of scratch, more than the %zu-byte "
                                    "static scratch; use lora_o_bwd with a caller-provided workspace",
                                    need, kStaticWsBytes);
    }
    // every other argument error, before any CUDA call
    const lm_status as = lm::check_o_bwd_args(T, d_in, d_out, X, dY, saved, saved_bytes, o, dX, dA, dB, nullptr, 0,
                                              true);
    if (as != LM_OK) return as;
    void* ws = nullptr;
    const lm_status ls = scratch_address("lora_o_bwd_static", &ws);
    if (ls != LM_OK) return ls;
    const cudaError_t e = cudaMemsetAsync(ws, 0, 256, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return lm::report_error(LM_ERR_CUDA, "lora_o_bwd_static: cudaMemsetAsync: %s", cudaGetErrorString(e));
    return lora_o_bwd(T, d_in, d_out, X, dY, saved, saved_bytes, o, dX, dA, dB, ws, kStaticWsBytes, stream);
}

extern "C" lm_status lm_static_scratch_check(lm_stream stream) {
    void* ws = nullptr;
    const lm_status ls = scratch_address("lm_static_scratch_check", &ws);
    if (ls != LM_OK) return ls;
    return lm_workspace_check(ws, stream);
}
