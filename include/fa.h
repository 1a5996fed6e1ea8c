/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library libfa_gb300.so.
 *
 * Sources cited below:
 *   [hyper] hyper.ai story on FlashAttention-4 (German): exact attention,
 *           faster without changing the mathematical result; 128x128 tiles;
 *           LPT scheduling for causal masks.
 *   [nl]    "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
 *           Asymmetric Hardware Scaling" (gist.science/nl), section
 *           "Technische samenvatting": Methodologie §1 (asynchronous MMA into
 *           Tensor Memory, 128x128 tiles, ping-pong of softmax and MMA),
 *           §2 (exp2 split between the MUFU unit and an FMA polynomial of
 *           degree 3 or 5), §3 (backward pass: intermediates in Tensor Memory,
 *           2-CTA MMA, dQ reduced by atomic additions in global memory).
 *   [de]    "FlashAttention-4: Der neue Rennwagen fuer die kuenstliche
 *           Intelligenz" (gist.science/de), §3: the rescale of the running
 *           output is skipped unless it is really needed.
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, contiguous, row-major.  Q, K, V, O, dO, dQ, dK, dV
 *     are bf16 [B, S, H, D] (element (b,s,h,d) at ((b*S + s)*H + h)*D + d).
 *     LSE and Delta are fp32 [B, H, S]; the dQ accumulator is fp32
 *     [B, H, S, D].
 *   - Every pointer is a device pointer, owned by the caller, 16-byte aligned.
 *     The library allocates no device memory, keeps no state across calls
 *     and never synchronises the device (except fa_device_error).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous: results are ready when the stream reaches them.
 *   - Supported: D in {64, 128, 256}; any S >= 1; B, H >= 1 with B*S*H*D
 *     below 2^31 elements per tensor; scale finite and > 0.  causal != 0
 *     means key j is visible to query i iff j <= i.
 *   - Errors: FA_ERR_INVALID_ARG for a null or misaligned pointer, a
 *     non-positive size, overflow or a bad scale; FA_ERR_UNSUPPORTED for a
 *     head dim outside the supported set or a device other than compute
 *     capability 10.3 (the kernels are built for sm_103a only), and for
 *     option combinations an entry point names; FA_ERR_CUDA when a CUDA call or launch
 *     fails (see fa_last_cuda_error).  Nothing is enqueued when an error is
 *     returned by the argument checks.
 *   - Device-side waits are bounded.  A wait that runs out (which correct
 *     code never reaches) records a code that fa_device_error reports; the
 *     kernel then returns instead of hanging.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,
    FA_ERR_UNSUPPORTED = 2,
    FA_ERR_CUDA = 3,
    FA_ERR_TIMEOUT = 4
} fa_status;

/*
 * Forward: O = softmax(scale * Q K^T [+ causal mask]) V and
 * LSE[b,h,i] = ln sum_{j visible} exp(scale * q_i . k_j)   ([hyper]; [nl]
 * Methodologie §1).  One fused, persistent kernel: TMA loads into a
 * multi-stage shared-memory ring, tcgen05 MMAs into Tensor Memory, two
 * 128-row query tiles per CTA whose softmax ping-pongs with the tensor core,
 * conditional rescale of O ([de] §3), exp2 split between MUFU and a degree-3
 * or degree-5 polynomial ([nl] Methodologie §2; MUFU only by default, see
 * fa_fwd_ex), longest-first tile order for causal
 * masks ([hyper]).
 *   q, k, v : bf16 [B,S,H,D] inputs.      o   : bf16 [B,S,H,D] output.
 *   lse     : fp32 [B,H,S] output (natural log of the scaled, masked scores).
 */
fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                 int B, int H, int S, int D, int causal, float scale, void *stream);

/*
 * Forward with explicit numerics knobs (used to test that they do not change
 * the result beyond rounding, and to measure the exp2 split).
 *   rescale_threshold : the running maximum (log2 units) may grow by this
 *                       much before O and the row sum are rescaled; 0 means
 *                       rescale whenever the maximum grows ([de] §3).
 *                       Range [0, 16]; a negative value selects the default.
 *   poly_exp2_groups  : how many of every 8 consecutive score columns take
 *                       exp2 from the FMA polynomial instead of MUFU ([nl]
 *                       Methodologie §2): one of 0 (MUFU only), 1 (12.5 %),
 *                       2 (25 %), 8 (polynomial only); -1 selects the
 *                       library default (0).
 *   poly_exp2_degree  : degree of that polynomial, 3 or 5 ([nl] Methodologie
 *                       §2: "degree 3 or 5"); -1 selects the default (3).
 *                       Ignored when poly_exp2_groups is 0.
 * Other values of a knob give FA_ERR_INVALID_ARG.
 */
fa_status fa_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                    int B, int H, int S, int D, int causal, float scale,
                    float rescale_threshold, int poly_exp2_groups, int poly_exp2_degree,
                    void *stream);

/*
 * Forward over a packed batch of sequences of different lengths (prefill
 * style, the pages' integration target; [hyper]): sequence b holds the
 * tokens [cu_seqlens[b], cu_seqlens[b+1]) of the packed tensors, and
 * attention (and the causal mask) stays within each sequence.
 *   q, k, v, o : bf16 [total, H, D] (token-major, like [B,S,H,D] with B = 1).
 *   lse        : fp32 [H, total].
 *   cu_seqlens : device int32 [B+1], 4-byte aligned, cu_seqlens[0] = 0,
 *                non-decreasing, cu_seqlens[B] <= total; read on the device.
 *   max_seqlen : >= every sequence's length, <= total (sizes the launch).
 * A sequence whose offsets break these rules is skipped (its rows of o and
 * lse are left as they were) and the device error word records
 * 0x300 (see fa_device_error).  At tile edges the kernel reads rows of the
 * neighbouring sequence and gives them zero weight, so all of k and v must
 * be finite.  Errors otherwise as fa_fwd.
 */
fa_status fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                        const int *cu_seqlens, int B, int max_seqlen, int total, int H, int D,
                        int causal, float scale, void *stream);

/*
 * Bytes of caller-provided scratch the backward pass needs: the fp32 dQ
 * accumulator [B,H,S,D] followed by fp32 Delta [B,H,S], each rounded up to
 * 256 bytes.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int S, int D);

/*
 * Backward ([nl] Methodologie §3): given Q, K, V, the forward output O, its
 * LSE and the upstream gradient dO, computes
 *   Delta_i = dO_i . O_i, dS = P o (dO V^T - Delta), dV = P^T dO,
 *   dK = scale dS^T Q, dQ = scale dS K,   P = exp(scale Q K^T - LSE).
 * Three launches on `stream`: Delta + zeroing of the dQ accumulator; the
 * fused main kernel (K/V-stationary, intermediates in Tensor Memory, dQ by
 * fp32 atomic additions); conversion of the accumulator to bf16 dQ.
 *   dq_acc : fp32 [B,H,S,D] scratch (contents on entry ignored).
 *   delta  : fp32 [B,H,S] scratch (written).
 *   dq, dk, dv : bf16 [B,S,H,D] outputs.
 * dq_acc/delta may be carved from one buffer of fa_bwd_workspace_size bytes.
 */
fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o,
                 const void *dout, const float *lse, float *dq_acc, float *delta,
                 void *dq, void *dk, void *dv,
                 int B, int H, int S, int D, int causal, float scale, void *stream);

/*
 * Backward over a packed batch (see fa_fwd_varlen): q, k, v, o, dout, dq, dk,
 * dv bf16 [total, H, D]; lse fp32 [H, total] from fa_fwd_varlen; dq_acc fp32
 * [H, total, D] and delta fp32 [H, total] scratch, fa_bwd_varlen_workspace_size
 * bytes in all (carved like fa_bwd's).  cu_seqlens and max_seqlen as for the
 * forward, with the same 0x300 report for bad offsets.  D in {64, 128, 256}.
 * Other arguments, results and errors as fa_bwd.
 */
size_t fa_bwd_varlen_workspace_size(int total, int H, int D);
fa_status fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                        const void *dout, const float *lse, float *dq_acc, float *delta,
                        void *dq, void *dk, void *dv, const int *cu_seqlens, int B,
                        int max_seqlen, int total, int H, int D, int causal, float scale,
                        void *stream);

/*
 * Backward with the choice of main kernel ([nl] Methodologie §3: the 2-CTA
 * MMA mode splits operand B between two CTAs, and the pair exchanges halves
 * of the dQ work through distributed shared memory).
 *   pair_mode : 0  one CTA per 128-key tile (every head dimension; at
 *                  D = 256 a CTA per key tile and half of the head dim, which
 *                  computes S^T and dP^T for both halves);
 *               1  CTA pairs (fixed-length batches, atomic-order dQ):
 *                  D = 128: two neighbouring SMs own two adjacent key tiles
 *                  and issue their MMAs together (tcgen05 .cta_group::2);
 *                  each CTA stages half of every Q/dO operand the MMAs read
 *                  and reduces only half of the dQ rows.
 *                  D = 256: two neighbouring SMs share one key tile and split
 *                  the work by role: one forms P^T, dV and half of dQ, the
 *                  other dP^T, dS^T, dK and the other half of dQ; P^T and dS^T
 *                  cross between them through distributed shared memory.
 *                  D = 64: FA_ERR_UNSUPPORTED;
 *              -1  library default (0: on GB300 both pair kernels measure
 *                  slower than the single-CTA ones, see their sources).
 * Other arguments, results and errors as fa_bwd; the results agree with
 * pair_mode 0 to rounding (fp32 operations in a different order).
 */
fa_status fa_bwd_ex(const void *q, const void *k, const void *v, const void *o,
                    const void *dout, const float *lse, float *dq_acc, float *delta,
                    void *dq, void *dk, void *dv,
                    int B, int H, int S, int D, int causal, float scale, int pair_mode,
                    void *stream);

/*
 * Deterministic backward ([nl] Methodologie §3 and Belangrijkste Resultaten:
 * a deterministic mode ordered by semaphores and scheduling): the same
 * results as fa_bwd to rounding, except that every element of dQ is summed
 * over the key tiles in an order fixed by (B, H, S, causal) and the device's
 * SM count, so repeated calls on the same inputs on the same GPU model give
 * bitwise-identical dQ, dK and dV.  Each 128-query block has a place for
 * every key tile that reaches it; without a causal mask the order puts the
 * tiles that run at the same time one step apart, with one it follows the
 * order in which the tiles reach the block in the persistent schedule (one
 * step per block).  At D = 64 and 128 the places alternate between two fp32
 * accumulators (so consecutive tiles do not wait on each other), each summed
 * in its fixed order under a counter, and the two are added in a fixed order
 * at the end.  The kernel is launched cooperatively, so all its CTAs are
 * resident while they wait on one another.
 *   dq_sem : scratch of fa_bwd_semaphore_bytes(B,H,S,D) bytes, 16-byte
 *            aligned: the counters, the order keys of the key tiles and (D =
 *            64, 128) the second accumulator (contents on entry ignored; the
 *            first launch initialises all three).
 * At D = 256 (a work unit is a key tile and one half of the head dim) the
 * key tiles take their turns in ascending order per half, in one accumulator.
 * Other arguments, results and errors as fa_bwd.
 */
size_t fa_bwd_semaphore_bytes(int B, int H, int S, int D);
fa_status fa_bwd_deterministic(const void *q, const void *k, const void *v, const void *o,
                               const void *dout, const float *lse, float *dq_acc, float *delta,
                               int *dq_sem, void *dq, void *dk, void *dv,
                               int B, int H, int S, int D, int causal, float scale, void *stream);

/*
 * fa_bwd_deterministic over a packed batch (arguments as fa_bwd_varlen, plus
 * dq_sem): every sequence's dQ is summed over its key tiles in a fixed order,
 * so repeated calls give bitwise-identical dQ, dK and dV.
 *   dq_sem : scratch of fa_bwd_varlen_semaphore_bytes(B, max_seqlen, total,
 *            H, D) bytes (B = number of sequences), 16-byte aligned, contents
 *            ignored.  The size function returns 0 for invalid sizes.
 */
size_t fa_bwd_varlen_semaphore_bytes(int B, int max_seqlen, int total, int H, int D);
fa_status fa_bwd_varlen_deterministic(const void *q, const void *k, const void *v, const void *o,
                                      const void *dout, const float *lse, float *dq_acc,
                                      float *delta, int *dq_sem, void *dq, void *dk, void *dv,
                                      const int *cu_seqlens, int B, int max_seqlen, int total,
                                      int H, int D, int causal, float scale, void *stream);

/*
 * Backward for callers that cannot allocate device memory: code that runs
 * where cudaMalloc is not allowed or not wanted (host callbacks, plug-ins
 * that only get their inputs and outputs from a host framework, tools that
 * must keep the device footprint fixed).  It computes what fa_bwd computes
 * (the backward of "FlashAttention-4: Algorithm and Kernel Pipelining
 * Co-Design for Asymmetric Hardware Scaling" (gist.science/nl), Technische
 * samenvatting, Methodologie §3); the pages have no counterpart of this
 * calling convention, which exists for those callers only.
 * Same arguments, results and errors as fa_bwd minus dq_acc and delta
 * (sizes that fa_bwd_workspace_size rejects give FA_ERR_INVALID_ARG); the
 * scratch comes from one fixed array of 72 MiB inside the library, held on
 * every GPU that loads the library until the process exits.  Problems whose
 * scratch (fa_bwd_workspace_size) exceeds 72 MiB are rejected with
 * FA_ERR_INVALID_ARG.  The first call on each device, and the first call
 * after that device's context was replaced (cudaDeviceReset), looks up the
 * array's device address (make those calls before any stream capture).  All
 * calls on a device share the array: calls whose kernels may overlap on the
 * GPU race and must be serialised by the caller.  Each call re-zeroes the
 * part of the scratch it uses, so nothing carries over between calls.
 * Allocates nothing.
 */
fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv,
                         int B, int H, int S, int D, int causal, float scale, void *stream);

/* Human-readable name of a status code (static string). */
const char *fa_status_string(fa_status s);

/* The last cudaError_t seen by any entry point of this thread (0 if none);
 * returns FA_OK. */
fa_status fa_last_cuda_error(int *cuda_err);

/*
 * Synchronises the current device, then reports and (if clear != 0) resets
 * the device-side error word: the first error any kernel recorded.  0x1nn /
 * 0x2nn: a bounded wait of the forward / backward kernel ran out (nn names
 * the wait); 0x300: a packed batch's cu_seqlens broke its rules.  *code = 0
 * means none.  Returns FA_ERR_TIMEOUT when the word is non-zero, FA_ERR_CUDA
 * if the synchronisation fails.
 */
fa_status fa_device_error(int *code, int clear);

/*
 * Test hooks for the exp2 approximation ([nl] Methodologie §2; degree 3,
 * accurate enough because bf16 rounding dominates its error).
 * fa_exp2_eval: y[i] = approximate 2^x[i] for n device floats.
 *   variant 0 = the softmax kernel's polynomial (inputs below -125 are
 *               clamped, giving a value in (0, 2^-124]),
 *   variant 1 = the same polynomial with exact subnormal scaling,
 *   variant 2 = hardware MUFU ex2.approx (flush-to-zero),
 *   variant 3 = the kernel polynomial in its two-lane (f32x2) form, as the
 *               softmax evaluates it (same range and clamp as variant 0),
 *   variant 4 = the degree-5 polynomial ([nl] Methodologie §2: degree 3 or
 *               5) with exact subnormal scaling, like variant 1,
 *   variant 5 = the degree-5 polynomial in the two-lane form the softmax
 *               evaluates (range and clamp of variant 0).
 * fa_exp2_sweep: every fp32 x with lo <= x <= hi (lo, hi finite, lo <= hi)
 *   is evaluated with `variant` and compared to 2^x in double precision;
 *   the largest relative error |y - 2^x| / max(2^x, 2^-126) and its
 *   argument are written to out[0], out[1] (device doubles; out[0] is also
 *   used as an accumulator while the sweep runs).
 */
fa_status fa_exp2_eval(const float *x, float *y, long long n, int variant, void *stream);
fa_status fa_exp2_sweep(float lo, float hi, int variant, double *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
