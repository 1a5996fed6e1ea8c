// fa_api.cu -- the extern "C" boundary of libfa_gb300.so (declared in
// include/fa.h): argument checks, TMA tensor-map encoding, per-device set-up
// and kernel launches.  The exp2 test kernels live here too.
//
// The library allocates no device memory.  Per-device state is limited to
// cached attributes (SM count, compute capability) and the address of a
// file-scope __device__ error word that bounded device waits write to.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "exp2_poly.cuh"
#include "fa_common.cuh"
#include "sm100_ptx.cuh"

namespace {

constexpr int kMaxDevices = 64;

// Device error word (one per device that loads the library).
__device__ int g_fa_error_word;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    int *err_word = nullptr;  // device address of g_fa_error_word
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;
thread_local int t_last_cuda_error = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

fa_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return FA_ERR_CUDA;
}

// Query (once per device) what the launches need.
fa_status device_info(const DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) !=
            cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) !=
            cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
            cudaSuccess)
            return cuda_fail(e);
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_fa_error_word)) != cudaSuccess) return cuda_fail(e);
        d.err_word = static_cast<int *>(p);
        d.ready = true;
    }
    // the kernels are built for sm_103a only
    if (d.cc_major != 10 || d.cc_minor != 3) return FA_ERR_UNSUPPORTED;
    *out = &d;
    return FA_OK;
}

fa_status get_encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode ? FA_OK : FA_ERR_CUDA;
}

// Tensor map over a bf16 [B,S,H,D] tensor: dims (D, H, S, B), box
// 64 x 1 x 128 x 1 (a 128-row x 128-byte tile), 128-byte swizzle, zero fill
// outside the tensor (ragged sequence tails read as zeros).
fa_status make_map_bshd(CUtensorMap *m, const void *ptr, int B, int S, int H, int D,
                        unsigned box_rows = 128) {
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                                   (cuuint64_t)S * H * D * 2};
    const cuuint32_t box[4] = {64, 1, box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

// Tensor map over the fp32 dQ accumulator viewed as [B*H][S][D]: box
// 32 x 128 x 1 (128 rows x 128 bytes), 128-byte swizzle; rows past S are
// outside the tensor, so reductions into them are dropped.
fa_status make_map_dqacc(CUtensorMap *m, void *ptr, int BH, int S, int D, unsigned box_rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)S * D * 4};
    const cuuint32_t box[3] = {32, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared size/scale checks.  Sizes: B,H,S >= 1; D in the supported set;
// one tensor below 2^31 elements.
fa_status check_shape(int B, int H, int S, int D, float scale) {
    if (B < 1 || H < 1 || S < 1) return FA_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
    const long long n = static_cast<long long>(B) * S * H * D;
    if (D < 1 || n >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

size_t pad256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Deterministic-mode scratch at D = 64 and 128: turn counters
// [B*H][ceil(S/128)][4 drain warps][2 accumulators], the order keys
// [B*H][ceil(S/128)] of the key tiles, then the second fp32 dQ accumulator
// over all query rows; each part padded to 256 bytes.  At D = 256: counters
// [B*H][2 halves][ceil(S/64)][4 drain warps] only.
size_t det_counter_bytes(int B, int H, int S) {
    return pad256(static_cast<size_t>(B) * H * 8 * ((static_cast<size_t>(S) + 127) / 128) * 4);
}
size_t det_key_bytes(int B, int H, int S) {
    return pad256(static_cast<size_t>(B) * H * ((static_cast<size_t>(S) + 127) / 128) * 4);
}
size_t d256_counter_bytes(int B, int H, int S) {
    return pad256(static_cast<size_t>(B) * H * 8 * ((static_cast<size_t>(S) + 63) / 64) * 4);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kDefaultRescaleThreshold = 8.0f;  // log2 units: P <= 2^8 between rescales
// Measured on GB300 (S = 32768, D = 128): 0 of 8 columns on the FMA
// polynomial gives 1419 TFLOPS, 1 gives 1380, 2 gives 1318, 8 gives 970; its
// MUFU keeps up with the tensor core, so the default leaves exp2 on MUFU.
constexpr int kDefaultPolyGroups = 0;
constexpr int kDefaultPolyDegree = 3;  // the cheaper of the two degrees the method allows

}  // namespace

// ----------------------------------------------------------------- exp2 test kernels

namespace {

__device__ __forceinline__ float exp2_variant(float x, int variant) {
    if (variant == 0) return fa::exp2_poly<3>(x);
    if (variant == 1) return fa::exp2_poly_full<3>(x);
    if (variant == 3) return fa::exp2_poly3_x2(make_float2(x, -x)).x;
    if (variant == 4) return fa::exp2_poly_full<5>(x);
    if (variant == 5) return fa::exp2_poly_x2<5>(make_float2(x, -x)).x;
    return fa::ex2_mufu(x);
}

__global__ void exp2_eval_kernel(const float *x, float *y, long long n, int variant) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        y[i] = exp2_variant(x[i], variant);
}

// Order-preserving map float bits <-> unsigned key (-inf < ... < -0 < +0 < ... ).
__host__ __device__ __forceinline__ uint32_t float_key(uint32_t bits) {
    return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}
__device__ __forceinline__ uint32_t key_float(uint32_t key) {
    return (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
}

__global__ void exp2_sweep_init(unsigned long long *acc) { *acc = 0ull; }

// Relative error |y - 2^x| / max(2^x, 2^-126), maximised over all floats
// whose keys lie in [k_lo, k_lo + count).  The running maximum is kept as
// (error as float bits) << 32 | (x bits), which orders by error.
__global__ void exp2_sweep_kernel(uint32_t k_lo, unsigned long long count, int variant,
                                  unsigned long long *acc) {
    unsigned long long best = 0ull;
    for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x;
         i < count; i += (unsigned long long)gridDim.x * blockDim.x) {
        const uint32_t bits = key_float(k_lo + static_cast<uint32_t>(i));
        const float x = __uint_as_float(bits);
        const float y = exp2_variant(x, variant);
        const double ref = exp2(static_cast<double>(x));
        const double den = fmax(ref, 1.1754943508222875e-38);  // 2^-126
        const float err = static_cast<float>(fabs(static_cast<double>(y) - ref) / den);
        const unsigned long long key =
            (static_cast<unsigned long long>(__float_as_uint(err)) << 32) | bits;
        best = key > best ? key : best;
    }
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
    }
    if ((threadIdx.x & 31) == 0) atomicMax(acc, best);
}

__global__ void exp2_sweep_finish(double *out) {
    const unsigned long long v = *reinterpret_cast<unsigned long long *>(out);
    out[0] = static_cast<double>(__uint_as_float(static_cast<uint32_t>(v >> 32)));
    out[1] = static_cast<double>(__uint_as_float(static_cast<uint32_t>(v & 0xffffffffu)));
}

}  // namespace

// ----------------------------------------------------------------- C ABI

extern "C" {

const char *fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    }
    return "FA_ERR_UNKNOWN";
}

fa_status fa_last_cuda_error(int *cuda_err) {
    if (!cuda_err) return FA_ERR_INVALID_ARG;
    *cuda_err = t_last_cuda_error;
    return FA_OK;
}

fa_status fa_device_error(int *code, int clear) {
    if (!code) return FA_ERR_INVALID_ARG;
    const DeviceInfo *d = nullptr;
    fa_status st = device_info(&d);
    if (st != FA_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    int v = 0;
    if ((e = cudaMemcpy(&v, d->err_word, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e);
    if (clear && v != 0) {
        const int zero = 0;
        if ((e = cudaMemcpy(d->err_word, &zero, sizeof(int), cudaMemcpyHostToDevice)) !=
            cudaSuccess)
            return cuda_fail(e);
    }
    *code = v;
    return v ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"

namespace {
// fa_fwd_ex and fa_fwd_varlen.  cu == nullptr: fixed length, [B, S, H, D];
// else packed: B sequences in [T, H, D], S = the longest.
fa_status fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse, const int *cu,
                   int B, int H, int S, int T, int D, int causal, float scale,
                   float rescale_threshold, int poly_exp2_groups, int poly_exp2_degree,
                   void *stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID_ARG;
    fa_status st = cu ? check_shape(1, H, T, D, scale) : check_shape(B, H, S, D, scale);
    if (st != FA_OK) return st;
    if (cu && (B < 1 || S < 1 || S > T || (reinterpret_cast<uintptr_t>(cu) & 3u)))
        return FA_ERR_INVALID_ARG;
    if (rescale_threshold < 0.f) rescale_threshold = kDefaultRescaleThreshold;
    if (!(rescale_threshold <= 16.f)) return FA_ERR_INVALID_ARG;
    if (poly_exp2_groups < 0) poly_exp2_groups = kDefaultPolyGroups;
    if (poly_exp2_groups != 0 && poly_exp2_groups != 1 && poly_exp2_groups != 2 &&
        poly_exp2_groups != 8)
        return FA_ERR_INVALID_ARG;
    if (poly_exp2_degree < 0) poly_exp2_degree = kDefaultPolyDegree;
    if (poly_exp2_degree != 3 && poly_exp2_degree != 5) return FA_ERR_INVALID_ARG;
    const DeviceInfo *d = nullptr;
    if ((st = device_info(&d)) != FA_OK) return st;
    if ((st = get_encoder()) != FA_OK) return st;
    fa::FwdArgs a;
    std::memset(&a, 0, sizeof(a));
    const int mb = cu ? 1 : B, ms = cu ? T : S;  // the tensors' [B, S] as the maps see them
    if ((st = make_map_bshd(&a.tm_q, q, mb, ms, H, D)) != FA_OK) return st;
    if ((st = make_map_bshd(&a.tm_k, k, mb, ms, H, D)) != FA_OK) return st;
    if ((st = make_map_bshd(&a.tm_v, v, mb, ms, H, D)) != FA_OK) return st;
    if ((st = make_map_bshd(&a.tm_o, o, mb, ms, H, D, 32)) != FA_OK) return st;
    if (D == 256 && (st = make_map_bshd(&a.tm_v64, v, mb, ms, H, D, 64)) != FA_OK) return st;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.S = S;
    a.D = D;
    a.causal = causal ? 1 : 0;
    a.scale_log2 = scale * kLog2e;
    a.rescale_threshold = rescale_threshold;
    a.poly_groups = poly_exp2_groups;
    a.poly_degree = poly_exp2_degree;
    a.err_word = d->err_word;
    a.num_sms = d->num_sms;
    a.cu_seqlens = cu;
    a.T = cu ? T : B * S;
    cudaError_t e = fa::launch_fwd(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}
}  // namespace

extern "C" {

fa_status fa_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                    int H, int S, int D, int causal, float scale, float rescale_threshold,
                    int poly_exp2_groups, int poly_exp2_degree, void *stream) {
    return fwd_impl(q, k, v, o, lse, nullptr, B, H, S, 0, D, causal, scale, rescale_threshold,
                    poly_exp2_groups, poly_exp2_degree, stream);
}

fa_status fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                        const int *cu_seqlens, int B, int max_seqlen, int total, int H, int D,
                        int causal, float scale, void *stream) {
    if (!cu_seqlens) return FA_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, lse, cu_seqlens, B, H, max_seqlen, total, D, causal, scale, -1.f,
                    -1, -1, stream);
}

fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                 int S, int D, int causal, float scale, void *stream) {
    return fa_fwd_ex(q, k, v, o, lse, B, H, S, D, causal, scale, -1.f, -1, -1, stream);
}

static size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t fa_bwd_workspace_size(int B, int H, int S, int D) {
    if (check_shape(B, H, S, D, 1.f) != FA_OK) return 0;
    const size_t n = static_cast<size_t>(B) * H * S;
    return round256(n * D * sizeof(float)) + round256(n * sizeof(float));
}

}  // extern "C"

namespace {
// fa_bwd and fa_bwd_deterministic; sem == nullptr selects the atomic-order dQ.
// cu == nullptr: fixed length [B, S, H, D]; else a packed batch of B
// sequences in [T, H, D] with S the longest.
fa_status bwd_impl(const void *q, const void *k, const void *v, const void *o, const void *dout,
                   const float *lse, float *dq_acc, float *delta, int *sem, void *dq, void *dk,
                   void *dv, const int *cu, int B, int H, int S, int T, int D, int causal,
                   float scale, int pair_mode, void *stream) {
    const void *ptrs[11] = {q, k, v, o, dout, lse, dq_acc, delta, dq, dk, dv};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return FA_ERR_INVALID_ARG;
    fa_status st = cu ? check_shape(1, H, T, D, scale) : check_shape(B, H, S, D, scale);
    if (st != FA_OK) return st;
    if (cu && (B < 1 || S < 1 || S > T || (reinterpret_cast<uintptr_t>(cu) & 3u)))
        return FA_ERR_INVALID_ARG;
    if (pair_mode < -1 || pair_mode > 1) return FA_ERR_INVALID_ARG;
    // CTA pairs: fixed-length batches with atomic-order dQ, D = 128 or 256.
    // Not the default: on GB300 the single-CTA kernels are faster.  D = 128:
    // the pair's dQ MMA (M = 128 over two SMs) runs at half the per-SM tensor
    // rate, and the dS exchange adds latency to the block chain.  D = 256: the
    // pair splits the work by role and computes nothing twice, but each block
    // waits for a round trip of P^T and dS^T between the two SMs (measured
    // 498 / 489 TFLOPS against 591 / 548 at S = 16384).
    if (pair_mode == 1 && (cu || sem || D == 64)) return FA_ERR_UNSUPPORTED;
    const bool pair = pair_mode == 1;
    const DeviceInfo *d = nullptr;
    if ((st = device_info(&d)) != FA_OK) return st;
    if ((st = get_encoder()) != FA_OK) return st;
    fa::BwdArgs a;
    std::memset(&a, 0, sizeof(a));
    // D = 256 streams 64-query blocks; dQ is staged as 32 x 32 tiles (each
    // drain warp its own)
    const unsigned qrows = D == 256 ? 64 : 128;
    const unsigned dqrows = 32;
    const int mb = cu ? 1 : B, ms = cu ? T : S;  // the tensors' [B, S] as the maps see them
    if ((st = make_map_bshd(&a.tm_q, q, mb, ms, H, D, qrows)) != FA_OK) return st;
    if ((st = make_map_bshd(&a.tm_k, k, mb, ms, H, D)) != FA_OK) return st;
    if ((st = make_map_bshd(&a.tm_v, v, mb, ms, H, D)) != FA_OK) return st;
    if ((st = make_map_bshd(&a.tm_do, dout, mb, ms, H, D, qrows)) != FA_OK) return st;
    if ((st = make_map_dqacc(&a.tm_dqacc, dq_acc, mb * H, ms, D, dqrows)) != FA_OK) return st;
    if (D != 256) {
        if ((st = make_map_bshd(&a.tm_dk32, dk, mb, ms, H, D, 32)) != FA_OK) return st;
        if ((st = make_map_bshd(&a.tm_dv32, dv, mb, ms, H, D, 32)) != FA_OK) return st;
    }
    if (pair && D == 256) {
        if ((st = make_map_dqacc(&a.tm_dqacc16, dq_acc, mb * H, ms, D, 16)) != FA_OK) return st;
    }
    if (pair && D == 128) {
        if ((st = make_map_bshd(&a.tm_q64, q, B, S, H, D, 64)) != FA_OK) return st;
        if ((st = make_map_bshd(&a.tm_do64, dout, B, S, H, D, 64)) != FA_OK) return st;
    }
    a.pair = pair ? 1 : 0;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq_acc = dq_acc;
    a.delta = delta;
    a.dq_sem = sem;
    if (sem && D != 256) {
        // fixed order at D = 64/128: order keys, then the second accumulator
        char *base = reinterpret_cast<char *>(sem);
        a.dq_key = reinterpret_cast<int *>(base + det_counter_bytes(B, H, S));
        a.dq_acc2 = reinterpret_cast<float *>(base + det_counter_bytes(B, H, S) +
                                              det_key_bytes(B, H, S));
        if ((st = make_map_dqacc(&a.tm_dqacc2, a.dq_acc2, mb * H, ms, D, dqrows)) != FA_OK)
            return st;
    }
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.H = H;
    a.S = S;
    a.D = D;
    a.causal = causal ? 1 : 0;
    a.scale = scale;
    a.scale_log2 = scale * kLog2e;
    a.err_word = d->err_word;
    a.num_sms = d->num_sms;
    a.cu_seqlens = cu;
    a.T = cu ? T : B * S;
    cudaError_t e = fa::launch_bwd(a, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return FA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}
}  // namespace

extern "C" {

fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                 const float *lse, float *dq_acc, float *delta, void *dq, void *dk, void *dv,
                 int B, int H, int S, int D, int causal, float scale, void *stream) {
    return bwd_impl(q, k, v, o, dout, lse, dq_acc, delta, nullptr, dq, dk, dv, nullptr, B, H, S,
                    0, D, causal, scale, -1, stream);
}

fa_status fa_bwd_ex(const void *q, const void *k, const void *v, const void *o, const void *dout,
                    const float *lse, float *dq_acc, float *delta, void *dq, void *dk, void *dv,
                    int B, int H, int S, int D, int causal, float scale, int pair_mode,
                    void *stream) {
    return bwd_impl(q, k, v, o, dout, lse, dq_acc, delta, nullptr, dq, dk, dv, nullptr, B, H, S,
                    0, D, causal, scale, pair_mode, stream);
}

size_t fa_bwd_varlen_workspace_size(int total, int H, int D) {
    return fa_bwd_workspace_size(1, H, total, D);
}

fa_status fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                        const void *dout, const float *lse, float *dq_acc, float *delta, void *dq,
                        void *dk, void *dv, const int *cu_seqlens, int B, int max_seqlen,
                        int total, int H, int D, int causal, float scale, void *stream) {
    if (!cu_seqlens) return FA_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, o, dout, lse, dq_acc, delta, nullptr, dq, dk, dv, cu_seqlens, B, H,
                    max_seqlen, total, D, causal, scale, 0, stream);
}

fa_status fa_bwd_varlen_deterministic(const void *q, const void *k, const void *v, const void *o,
                                      const void *dout, const float *lse, float *dq_acc,
                                      float *delta, int *dq_sem, void *dq, void *dk, void *dv,
                                      const int *cu_seqlens, int B, int max_seqlen, int total,
                                      int H, int D, int causal, float scale, void *stream) {
    if (!cu_seqlens || !dq_sem || !aligned16(dq_sem)) return FA_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, o, dout, lse, dq_acc, delta, dq_sem, dq, dk, dv, cu_seqlens, B, H,
                    max_seqlen, total, D, causal, scale, 0, stream);
}

size_t fa_bwd_semaphore_bytes(int B, int H, int S, int D) {
    if (check_shape(B, H, S, D, 1.f) != FA_OK) return 0;
    if (D == 256) return d256_counter_bytes(B, H, S);  // one counter set per output half
    return det_counter_bytes(B, H, S) + det_key_bytes(B, H, S) +
           pad256(static_cast<size_t>(B) * H * S * D * 4);
}

size_t fa_bwd_varlen_semaphore_bytes(int B, int max_seqlen, int total, int H, int D) {
    if (B < 1 || max_seqlen < 1 || max_seqlen > total) return 0;
    if (check_shape(1, H, total, D, 1.f) != FA_OK) return 0;
    if (D == 256) return d256_counter_bytes(B, H, max_seqlen);
    return det_counter_bytes(B, H, max_seqlen) + det_key_bytes(B, H, max_seqlen) +
           pad256(static_cast<size_t>(H) * total * D * 4);
}

fa_status fa_bwd_deterministic(const void *q, const void *k, const void *v, const void *o,
                               const void *dout, const float *lse, float *dq_acc, float *delta,
                               int *dq_sem, void *dq, void *dk, void *dv, int B, int H, int S,
                               int D, int causal, float scale, void *stream) {
    if (!dq_sem || !aligned16(dq_sem)) return FA_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, o, dout, lse, dq_acc, delta, dq_sem, dq, dk, dv, nullptr, B, H, S,
                    0, D, causal, scale, 0, stream);
}

fa_status fa_exp2_eval(const float *x, float *y, long long n, int variant, void *stream) {
    if (!x || !y || n < 0 || variant < 0 || variant > 5) return FA_ERR_INVALID_ARG;
    if (n == 0) return FA_OK;
    const DeviceInfo *d = nullptr;
    fa_status st = device_info(&d);
    if (st != FA_OK) return st;
    const long long want = (n + 255) / 256;
    const int grid = static_cast<int>(want < 8LL * d->num_sms ? want : 8LL * d->num_sms);
    exp2_eval_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n, variant);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

fa_status fa_exp2_sweep(float lo, float hi, int variant, double *out, void *stream) {
    if (!out || !(std::isfinite(lo) && std::isfinite(hi)) || lo > hi || variant < 0 ||
        variant > 5)
        return FA_ERR_INVALID_ARG;
    const DeviceInfo *d = nullptr;
    fa_status st = device_info(&d);
    if (st != FA_OK) return st;
    uint32_t blo, bhi;
    std::memcpy(&blo, &lo, 4);
    std::memcpy(&bhi, &hi, 4);
    const uint32_t klo = float_key(blo), khi = float_key(bhi);
    const unsigned long long count = static_cast<unsigned long long>(khi - klo) + 1ull;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto *acc = reinterpret_cast<unsigned long long *>(out);
    exp2_sweep_init<<<1, 1, 0, s>>>(acc);
    exp2_sweep_kernel<<<d->num_sms * 8, 256, 0, s>>>(klo, count, variant, acc);
    exp2_sweep_finish<<<1, 1, 0, s>>>(out);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

}  // extern "C"
