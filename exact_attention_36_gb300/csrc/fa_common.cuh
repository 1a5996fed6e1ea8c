// fa_common.cuh -- launch-side declarations shared by the kernels' translation
// units and the C-ABI layer (fa_api.cu).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Error codes written to the device error word by bounded waits that ran out.
// The low byte names the wait site.
enum DeviceError : int {
    kErrNone = 0,
    kErrFwdWait = 0x100,  // + site
    kErrBwdWait = 0x200,  // + site
    kErrSeqlens = 0x300,  // packed batches: cu_seqlens not non-decreasing within
                          // [0, T] or a sequence longer than max_seqlen
};

struct FwdArgs {
    CUtensorMap tm_q, tm_k, tm_v;  // bf16 [B,S,H,D], box 64 x 1 x 128 x 1, 128B swizzle
    CUtensorMap tm_o;              // the output, box 64 x 1 x 32 x 1 (one warp's rows; TMA-store epilogue)
    CUtensorMap tm_v64;            // D = 256: V with 64-row boxes (key halves of a tile)
    void *o;                       // bf16 [B,S,H,D]
    float *lse;                    // fp32 [B,H,S]
    int B, H, S, D;
    int causal;
    float scale_log2;         // softmax scale * log2(e)
    float rescale_threshold;  // log2 units
    int poly_groups;          // columns of every 8 whose exp2 uses the FMA polynomial
    int poly_degree;          // that polynomial's degree: 3 or 5
    int *err_word;            // device error word
    int num_sms;
    const int *cu_seqlens;    // packed variable-length batch: B+1 offsets, else null
    int T;                    // packed: total tokens (S is then the longest sequence)
};

struct BwdArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;  // bf16 [B,S,H,D], same boxes as the forward
    CUtensorMap tm_dqacc;                 // fp32 [B*H, S, D], box 32 x 32 x 1
    CUtensorMap tm_dqacc16;               // D = 256 on CTA pairs: the same, box 32 x 16 x 1
    CUtensorMap tm_q64, tm_do64;          // CTA pairs: Q and dO with 64-row boxes
    CUtensorMap tm_dk32, tm_dv32;         // D = 64/128: dK, dV with 32-row boxes (TMA-store epilogue)
    const void *o, *dout;                 // bf16 [B,S,H,D]
    const float *lse;                     // fp32 [B,H,S]
    float *dq_acc;                        // fp32 [B,H,S,D]
    float *delta;                         // fp32 [B,H,S]
    int *dq_sem;                          // deterministic mode: turn counters, else null
                                          // (D = 64/128: [B*H][ceil(S/128)][4 drain warps]
                                          // [2 accumulators]; D = 256: [B*H][2 halves]
                                          // [ceil(S/64)][4 drain warps])
    int *dq_key;                          // deterministic mode: [B*H][ceil(S/128)] order keys of the key tiles
    CUtensorMap tm_dqacc2;                // deterministic mode, D = 64/128: the second accumulator
    float *dq_acc2;                       // deterministic mode, D = 64/128: second fp32 dQ
                                          // accumulator (the layout of dq_acc), else null
    int grid;                             // main kernel's persistent grid (for the order keys)
    void *dq, *dk, *dv;                   // bf16 [B,S,H,D]
    int B, H, S, D;
    int causal;
    float scale;
    float scale_log2;
    int *err_word;
    int num_sms;
    int pair;                             // 1: main kernel on CTA pairs (D = 128, 256)
    const int *cu_seqlens;                // packed variable-length batch, else null
    int T;                                // packed: total tokens (S = longest sequence)
};

// Rows of batch entry b.  Fixed length: rows [0, S) of entry b, read through
// [B, S, H, D] tensor maps (TMA row coordinate = row, batch coordinate b).
// Packed variable length (cu != null): rows [cu[b], cu[b+1]) of [T, H, D]
// tensors, read through [1, T, H, D] maps; per-query statistics, Delta and the
// dQ accumulator are then [H, T] (and [H, T, D]).  An entry whose offsets are
// out of order, past T or longer than S is marked bad (len 0).
struct SeqSpan {
    int tok0;   // token index of row 0 (b*S for fixed length)
    int len;    // rows
    int trow0;  // TMA row coordinate of row 0
    int tb;     // TMA batch coordinate
    bool ok;
};

__device__ __forceinline__ SeqSpan seq_span(const int *cu, int T, int S, int b) {
    SeqSpan s;
    if (cu) {
        const int a0 = __ldg(cu + b), a1 = __ldg(cu + b + 1);
        s.ok = 0 <= a0 && a0 <= a1 && a1 <= T && a1 - a0 <= S;
        s.tok0 = a0;
        s.len = s.ok ? a1 - a0 : 0;
        s.trow0 = a0;
        s.tb = 0;
    } else {
        s.ok = true;
        s.tok0 = b * S;
        s.len = S;
        s.trow0 = 0;
        s.tb = b;
    }
    return s;
}

// Index of (b, h, row) in the per-query arrays: [B, H, S], or [H, T] packed.
__device__ __forceinline__ size_t stat_index(const int *cu, int T, int S, int H, int b, int h,
                                             const SeqSpan &sp, int row) {
    return cu ? static_cast<size_t>(h) * T + sp.tok0 + row
              : (static_cast<size_t>(b) * H + h) * S + row;
}

// Launchers (defined in fa_fwd.cu / fa_bwd.cu).  Return the CUDA error of the
// launch (cudaSuccess when enqueued).
cudaError_t launch_fwd(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t stream);
// main backward kernel for D = 256 (fa_bwd_d256.cu); Q/dO tensor maps with
// 64-row boxes and a dQ-accumulator map with 32 x 32 boxes
cudaError_t launch_bwd_main_d256(const BwdArgs &a, cudaStream_t stream);
// main backward kernel for D = 128 on CTA pairs (fa_bwd_pair.cu); Q/dO maps
// with 128- and 64-row boxes and a dQ-accumulator map with 32 x 64 boxes
cudaError_t launch_bwd_main_pair(const BwdArgs &a, cudaStream_t stream);
// main backward kernel for D = 256 on CTA pairs split by role
// (fa_bwd_d256_split.cu); fixed-length batches, atomic-order dQ; maps as for
// launch_bwd_main_d256
cudaError_t launch_bwd_main_d256_split(const BwdArgs &a, cudaStream_t stream);

}  // namespace fa
