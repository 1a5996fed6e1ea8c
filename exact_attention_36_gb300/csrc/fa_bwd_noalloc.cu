// fa_bwd_noalloc.cu -- a backward entry point for callers that cannot
// allocate device memory.
//
// fa_bwd needs fp32 scratch (the dQ accumulator and Delta) that the caller
// allocates.  Some callers cannot do that: code running where the allocator
// is off limits (inside a host callback or a driver-managed region that must
// not call cudaMalloc), plug-ins that only receive their inputs and outputs
// from a host framework, or tools that must not change the device memory
// footprint between calls.  fa_bwd_noalloc serves them from a fixed scratch
// array compiled into the library instead.
//
// The array lives in device global memory of every GPU that loads this
// library and stays there until the process exits.  Its address is looked up
// on the first call made with a device current, and again on the first call
// after that device's context was replaced (cudaDeviceReset reloads the
// module, which can move the array); make those calls before capturing any
// stream.  All calls on a device share the array, so two calls whose kernels
// overlap on that GPU (for example on two streams) race on it and must be
// serialised by the caller.  The backward's first kernel zeroes the part of
// the accumulator a call uses and rewrites Delta, so nothing is carried over
// from an earlier call.
#include <cuda.h>

#include <mutex>

#include "fa.h"

namespace {

// Capacity of the shared scratch: 72 MiB, which holds the dQ accumulator and
// Delta of e.g. B*H*S = 131072 rows at D = 128 (B=4, H=16, S=2048).
constexpr size_t kScratchBytes = size_t(72) << 20;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
    unsigned long long ctx_id = 0;  // unique id of the context the address belongs to
    void *addr = nullptr;
};
ScratchSlot g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Unique id of the calling thread's current context (0 if none yet).
unsigned long long current_ctx_id() {
    std::call_once(g_ctx_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
    });
    if (!g_ctx_current || !g_ctx_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_bwd_scratch on the current device.  In host code the
// symbol's name is only a stand-in: the address the kernels need comes from
// cudaGetSymbolAddress, looked up once per device and context.
fa_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchSlot &slot = g_scratch[dev];
    const unsigned long long id = current_ctx_id();
    if (!slot.addr || id == 0 || id != slot.ctx_id) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
        slot.addr = p;
        // the lookup made the device's context current if it was not yet
        slot.ctx_id = id ? id : current_ctx_id();
    }
    *out = slot.addr;
    return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv,
                         int B, int H, int S, int D, int causal, float scale, void *stream) {
    const size_t need = fa_bwd_workspace_size(B, H, S, D);
    if (need == 0) return FA_ERR_INVALID_ARG;     // invalid sizes (same rule as fa_bwd)
    if (need > kScratchBytes) return FA_ERR_INVALID_ARG;  // larger than the fixed scratch
    void *base = nullptr;
    fa_status st = scratch_address(&base);
    if (st != FA_OK) return st;
    // same carving as fa_bwd_workspace_size: accumulator, then Delta, each
    // rounded up to 256 bytes
    const size_t rows = static_cast<size_t>(B) * H * S;
    const size_t acc_bytes = (rows * D * sizeof(float) + 255) & ~static_cast<size_t>(255);
    float *dq_acc = static_cast<float *>(base);
    float *delta = reinterpret_cast<float *>(static_cast<unsigned char *>(base) + acc_bytes);
    return fa_bwd(q, k, v, o, dout, lse, dq_acc, delta, dq, dk, dv, B, H, S, D, causal, scale,
                  stream);
}

}  // extern "C"
