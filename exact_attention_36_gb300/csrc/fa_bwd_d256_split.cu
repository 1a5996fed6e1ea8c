// fa_bwd_d256_split.cu -- fused attention backward for head dim 256 on CTA
// pairs that split the work by role, sm_103a.
//
// Same mathematics as fa_bwd.cu ("FlashAttention-4: Algorithm and Kernel
// Pipelining Co-Design for Asymmetric Hardware Scaling" (gist.science/nl),
// Technische samenvatting, Methodologie §3: intermediates in Tensor Memory,
// CTA pairs that exchange work through distributed shared memory).  With
// P = exp(scale*S - LSE):
//   dS = P o (dO V^T - Delta),  dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K.
//
// At D = 256 one SM cannot hold the dK and dV accumulators of a 128-key tile
// beside S^T and dP^T (each accumulator is 256 Tensor Memory columns), so the
// single-CTA kernel (fa_bwd_d256.cu) splits the head dim into halves and
// computes S^T and dP^T twice.  Here a cluster of two CTAs works on one key
// tile j (128 keys, all 256 columns) and splits the work by role instead, so
// nothing is computed twice:
//   rank 0  S^T = K Q_i^T - LSE/scale, P^T = 2^(S^T scale log2 e)  (bf16),
//           dV += P^T dO_i (256 columns in TMEM), dQ_i^T[0:128] = K[:,0:128]^T dS^T
//   rank 1  dP^T = V dO_i^T - Delta, dS^T = P^T o dP^T (bf16),
//           dK += dS^T Q_i (256 columns in TMEM), dQ_i^T[128:256] = K[:,128:256]^T dS^T
// P^T goes to rank 1 and dS^T back to rank 0 as bulk copies between the two
// shared memories, one 4 KB copy per softmax warp (its 32 key rows), each
// completing on the receiver's barrier.  Each rank issues 1712 tensor
// cycles of MMA per 64-query block (S^T or dP^T: 16 K-steps of N = 64 plus a
// bias step; dV or dK: 4 K-steps of N = 256; its dQ^T half: 8 K-steps of
// N = 64), where the single-CTA kernel issues 2528 per block and half-unit.
// Queries stream in blocks of 64 rows.  Keys sit on the TMEM lanes.
//
// Per-query terms enter through an extra K step of S^T and dP^T (A = ones,
// B = the value as three bf16 terms), as in fa_bwd.cu.
//
// Shared memory (bytes; 1024-aligned tiles, 128B swizzle unless noted):
//   rank 0  K 64K | Q 2 x 32K | dO 32K | dS^T from rank 1, 2 x 16K |
//           dQ staging 8K | P^T to send 16K | ones 4K | LSE bias 2 x 2K
//   rank 1  V 64K | K[:,128:256] 32K | dO 32K | Q 32K | P^T from rank 0 16K |
//           dS^T 16K | dQ staging 16K | ones 4K | Delta bias 2K
// Tensor Memory (512 columns per CTA):
//   rank 0  S^T/P^T X0 [0,64) X1 [64,128) | dV [128,384) | dQ^T half [384,448)
//   rank 1  dP^T Y0 [0,64) Y1 [64,128) | dK [128,384) | dQ^T half [384,448)
//
// Warp roles (384 threads per CTA): warp 0 TMA producer; warp 1 TMEM
// allocation and MMA issue (one lane); warps 4-7 P^T (rank 0) or dS^T
// (rank 1), lane = key, each warp also copying its rows to the other CTA;
// warps 8-11 dQ drain and the dV (rank 0) / dK (rank 1) epilogue.  Rank 0
// issues each block's dQ^T one block late, so that waiting for its dS^T (a
// round trip between the CTAs) does not hold up the next block's S^T.
//
// Used for fixed-length batches with atomic-order dQ; packed batches and the
// fixed-order mode take the single-CTA kernel.
#include <cuda_bf16.h>

#include "fa_common.cuh"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr int kKeys = 128;    // keys per unit
constexpr int kQB = 64;       // queries per block
constexpr int kD = 256;
constexpr int kBoxK = 16384;  // 128 rows x 64 bf16, 128B swizzle
constexpr int kBoxQ = 8192;   // 64 rows x 64 bf16
constexpr int kRow = 16384;   // one 128 x 64 bf16 P^T / dS^T tile (rows = keys)

struct SplitCfg {
    // rank 0
    static constexpr int kOffK = 0;
    static constexpr int kOffQ0 = kOffK + 4 * kBoxK;       // 2 stages x 4 boxes
    static constexpr int kOffDO0 = kOffQ0 + 8 * kBoxQ;     // 4 boxes
    static constexpr int kOffDSR = kOffDO0 + 4 * kBoxQ;    // 2 stages
    static constexpr int kOffRed0 = kOffDSR + 2 * kRow;    // 4 warps x 2K (16-row boxes)
    static constexpr int kOffPS = kOffRed0 + 8192;         // P^T rows on their way to rank 1
    static constexpr int kOffOnes0 = kOffPS + kRow;
    static constexpr int kOffLb = kOffOnes0 + 4096;       // 2 stages x 2K
    static constexpr int kEnd0 = kOffLb + 4096;
    // rank 1
    static constexpr int kOffV = 0;
    static constexpr int kOffKh = kOffV + 4 * kBoxK;       // 2 boxes
    static constexpr int kOffDO1 = kOffKh + 2 * kBoxK;
    static constexpr int kOffQ1 = kOffDO1 + 4 * kBoxQ;
    static constexpr int kOffPR = kOffQ1 + 4 * kBoxQ;
    static constexpr int kOffDSL = kOffPR + kRow;
    static constexpr int kOffRed1 = kOffDSL + kRow;
    static constexpr int kOffOnes1 = kOffRed1 + 16384;
    static constexpr int kOffDb = kOffOnes1 + 4096;
    static constexpr int kEnd1 = kOffDb + 2048;
    static constexpr int kOffBar = kEnd0 > kEnd1 ? kEnd0 : kEnd1;
    static constexpr int kNumBars = 31;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kSmemBytes = kOffMisc + 16;  // base must be 1024-aligned (checked)
    static constexpr uint32_t kT0 = 0, kT1 = 64, kTAcc = 128, kTdQ = 384;
    static constexpr uint32_t kIdescS = idesc_bf16_f32(128, kQB, false, false);   // S^T, dP^T
    static constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, kD, false, true);   // dV, dK
    static constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, kQB, true, true);    // dQ^T half
};
static_assert(SplitCfg::kSmemBytes <= 232448, "shared memory budget");

// barrier slots (same offsets in both CTAs, so either can address the
// other's; each rank initialises the ones its role uses)
enum SplitBar : int {
    kKvFull, kKvEmpty, kQFull0, kQFull1, kQEmpty0, kQEmpty1, kDoFull, kDoEmpty,
    kXFull0, kXFull1,  // rank 0: S^T of a stage complete; rank 1: dP^T
    kPReady0, kPReady1,  // rank 0: P^T of a stage written to TMEM (128 threads).  One
                         // per stage: S^T(n+1) is issued before P(n) is waited for, so
                         // the softmax can finish block n+1 first; two barriers keep
                         // that from completing a phase twice before it is waited on
    kPrFree0,          // rank 0 [4]: rank 1's warp q has read its P^T rows (remote, 1)
    kDsrFull0 = kPrFree0 + 4, kDsrFull1,  // rank 0: dS^T landed (4 remote expect_tx + bytes)
    kPrFull0,          // rank 1 [4]: P^T rows of warp q landed (remote expect_tx + bytes)
    kDsStaged = kPrFull0 + 4,  // rank 1: dS^T in shared memory (4 warps)
    kDsFree,           // rank 1: the dK and dQ^T MMAs have read dS^T (drain, 1)
    kDsrFree0, kDsrFree1,  // rank 1: rank 0's dS^T stage free (remote, 1)
    kDqFull, kDqEmpty, kAccFull, kAccEmpty, kDrain, kNumSplitBars
};
static_assert(kNumSplitBars == SplitCfg::kNumBars, "barrier slots");

struct SUnit {
    int bh, j;  // j = -1: no unit for this pair this round
};

// Unit u -> (head, key tile).  Causal: tile-major (every head's tile 0, then
// tile 1, ...), i.e. longest first across heads; otherwise head by head (the
// concurrent pairs share a head's Q, dO and dQ accumulator in L2).  Pairs take
// units in a serpentine round robin.
__device__ __forceinline__ bool sunit_at(int it, int U, int BH, int nT, bool causal, SUnit &out) {
    const int G = gridDim.x >> 1;
    const int pid = blockIdx.x >> 1;
    const int base = it * G;
    if (base >= U) return false;
    const int c = (it & 1) ? (G - 1 - pid) : pid;
    const int u = base + c;
    if (u >= U) {
        out.j = -1;
        return true;
    }
    if (causal) {
        out.j = u / BH;
        out.bh = u % BH;
    } else {
        out.bh = u / nT;
        out.j = u % nT;
    }
    return true;
}

// Byte offset of element (row r, k) of a no-swizzle K-major rows x 16 bf16 tile.
__host__ __device__ constexpr uint32_t bias_off(int r, int k) {
    return (r / 8) * 256 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2;
}

// First 16 bytes of a bias row: v as three bf16 terms hi + mid + lo in k = 0..2
// (exact for normal fp32 v); an infinite v goes whole into hi.
__device__ __forceinline__ uint4 bias_row(float v) {
    const float hi = __bfloat162float(__float2bfloat16_rn(v));
    if (!isfinite(v)) return make_uint4(pack_bf16x2(hi, 0.f), 0u, 0u, 0u);
    const float r1 = v - hi;
    const float mid = __bfloat162float(__float2bfloat16_rn(r1));
    const float lo = r1 - mid;
    return make_uint4(pack_bf16x2(hi, mid), pack_bf16x2(lo, 0.f), 0u, 0u);
}

// S^T = K Q^T or dP^T = V dO^T (128 x 64, K = 256), plus the bias K step
__device__ __forceinline__ void issue_rowcol(uint32_t tD, uint32_t a_saddr, uint32_t b_saddr,
                                             uint32_t ones_saddr, uint32_t bias_saddr) {
    const uint64_t ad = sdesc_sw128(a_saddr, 16, 1024), bd = sdesc_sw128(b_saddr, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk)
        mma_ss(tD, ad + (((kk / 4) * kBoxK + (kk % 4) * 32) >> 4),
               bd + (((kk / 4) * kBoxQ + (kk % 4) * 32) >> 4), SplitCfg::kIdescS,
               kk > 0 ? 1u : 0u);
    mma_ss(tD, sdesc_none(ones_saddr, 128, 256), sdesc_none(bias_saddr, 128, 256),
           SplitCfg::kIdescS, 1u);
}

// dQ^T half = Kx^T dS^T: A = 128 keys x 128 d (two MN-major boxes), B = dS^T
// (keys x 64 queries, MN-major)
__device__ __forceinline__ void issue_dqt(uint32_t tD, uint32_t k_saddr, uint32_t ds_saddr) {
    const uint64_t ad = sdesc_sw128(k_saddr, kBoxK, 1024), bd = sdesc_sw128(ds_saddr, kBoxK, 1024);
#pragma unroll
    for (int kk = 0; kk < kKeys / 16; ++kk)
        mma_ss(tD, ad + ((kk * 2048) >> 4), bd + ((kk * 2048) >> 4), SplitCfg::kIdescDQ,
               kk > 0 ? 1u : 0u);
}

// One drain warp's 32 columns of dQ^T (lane = column d0 + lane) for the 64
// queries of a block, in pieces of ROWS queries: each piece is staged as
// [query][32 columns] fp32 (128B swizzle) and added into the accumulator by
// one TMA bulk reduction (box 32 x ROWS).
template <int ROWS>
__device__ __forceinline__ void stage_reduce(const uint32_t (&col)[2][32], uint8_t *stage,
                                             const CUtensorMap *map, int d0, int row0, int z,
                                             int lane, volatile int *abort_flag) {
#pragma unroll
    for (int q0 = 0; q0 < kQB; q0 += ROWS) {
        if (lane == 0) bulk_wait_read<0>();  // the previous reduction has read `stage`
        __syncwarp();
#pragma unroll
        for (int q = 0; q < ROWS; ++q)
            *reinterpret_cast<float *>(stage + q * 128 + ((((lane >> 2) ^ (q & 7))) << 4) +
                                       (lane & 3) * 4) =
                __uint_as_float(col[(q0 + q) >> 5][(q0 + q) & 31]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && !*abort_flag) {
            tma_reduce_add_3d(map, stage, d0, row0 + q0, z);
            bulk_commit();
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_d256_split_kernel(const __grid_constant__ BwdArgs args) {
    using Cfg = SplitCfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    const bool bad_base = (smem_u32(smem) & 1023u) != 0;  // the same in both CTAs
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);

    const uint32_t rank = cluster_rank();
    const uint32_t peer = rank ^ 1u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = args.H, S = args.S;
    const int BH = args.B * H;
    const int nT = (S + kKeys - 1) / kKeys;
    const int nQ = (S + kQB - 1) / kQB;
    const int U = BH * nT;
    const bool causal = args.causal != 0;
    if (bad_base) {
        if (threadIdx.x == 0) atomicCAS(args.err_word, 0, kErrBwdWait + 0xfd);
        return;
    }

    if (threadIdx.x == 0) {
        uint32_t counts[Cfg::kNumBars];
        for (int i = 0; i < Cfg::kNumBars; ++i) counts[i] = 1;
        counts[kPReady0] = counts[kPReady1] = 128;
        counts[kDsrFull0] = counts[kDsrFull1] = 4;
        counts[kDsStaged] = 4;
        counts[kDqEmpty] = 4;
        counts[kAccEmpty] = 4;
        counts[kQFull0] = counts[kQFull1] = (rank == 0) ? 2 : 1;  // rank 0: TMA + LSE bias rows
        counts[kDoFull] = (rank == 0) ? 1 : 2;                    // rank 1: TMA + Delta bias rows
        for (int i = 0; i < Cfg::kNumBars; ++i) mbar_init(&bars[i], counts[i]);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    // bias tiles: zero everywhere (the MMA reads all 16 K columns), ones in
    // k = 0, 1, 2 of the A tile
    const int ones_off = rank == 0 ? Cfg::kOffOnes0 : Cfg::kOffOnes1;
    const int bias_bytes = rank == 0 ? 4096 + 4096 : 4096 + 2048;
    for (int t = threadIdx.x; t < bias_bytes / 16; t += kThreads)
        reinterpret_cast<uint4 *>(smem + ones_off)[t] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (threadIdx.x < 128)
        *reinterpret_cast<uint4 *>(smem + ones_off + bias_off(threadIdx.x, 0)) =
            make_uint4(pack_bf16x2(1.f, 1.f), pack_bf16x2(1.f, 0.f), 0u, 0u);
    fence_proxy_async_smem();
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&args.tm_q);
        tma_prefetch_desc(&args.tm_k);
        tma_prefetch_desc(&args.tm_v);
        tma_prefetch_desc(&args.tm_do);
        tma_prefetch_desc(&args.tm_dqacc);
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t sbase = smem_u32(smem);
    auto peer_bar = [&](int slot) { return mapa_shared(smem_u32(&bars[slot]), peer); };
    auto first_block = [&](int j) { return causal ? (j * kKeys) / kQB : 0; };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0xa0};
        const float inv_scale = 1.f / args.scale;
        uint32_t nunit = 0, nq = 0, ndo = 0;  // units, Q loads, dO loads issued
        uint32_t nkv = 0;                    // K/V loads issued
        bool ok = true;
        // rank 0: Q with its LSE bias rows into stage nq & 1; rank 1: Q alone
        auto load_q = [&](int b, int h, int i) -> bool {
            const uint32_t st = (rank == 0) ? (nq & 1) : 0;
            const uint32_t use = (rank == 0) ? (nq >> 1) : nq;
            float lv[2];
            if (rank == 0) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int q = i * kQB + r * 32 + lane;
                    lv[r] = q < S ? -args.lse[(static_cast<size_t>(b) * H + h) * S + q] * inv_scale
                                  : -INFINITY;
                }
            }
            w.code = kErrBwdWait + 0xa1;
            bool good = mbar_wait(&bars[kQEmpty0 + st], (use & 1) ^ 1, w);
            good = __all_sync(0xffffffffu, good ? 1 : 0) != 0;
            if (!good) return false;
            uint64_t *full = &bars[kQFull0 + st];
            uint8_t *dst = smem + (rank == 0 ? Cfg::kOffQ0 + st * 4 * kBoxQ : Cfg::kOffQ1);
            if (lane == 0) {
                mbar_arrive_expect_tx(full, 4 * kBoxQ);
                for (int c = 0; c < 4; ++c)
                    tma_load_4d(dst + c * kBoxQ, &args.tm_q, full, 64 * c, h, i * kQB, b);
            }
            if (rank == 0) {
                uint8_t *lb = smem + Cfg::kOffLb + st * 2048;
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    *reinterpret_cast<uint4 *>(lb + bias_off(r * 32 + lane, 0)) = bias_row(lv[r]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full);
            }
            ++nq;
            return true;
        };
        // dO (single stage); rank 1 writes its Delta bias rows
        auto load_do = [&](int b, int h, int i) -> bool {
            float dv[2];
            if (rank == 1) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int q = i * kQB + r * 32 + lane;
                    dv[r] = q < S ? -args.delta[(static_cast<size_t>(b) * H + h) * S + q] : 0.f;
                }
            }
            w.code = kErrBwdWait + 0xa2;
            bool good = mbar_wait(&bars[kDoEmpty], (ndo & 1) ^ 1, w);
            good = __all_sync(0xffffffffu, good ? 1 : 0) != 0;
            if (!good) return false;
            uint8_t *dst = smem + (rank == 0 ? Cfg::kOffDO0 : Cfg::kOffDO1);
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[kDoFull], 4 * kBoxQ);
                for (int c = 0; c < 4; ++c)
                    tma_load_4d(dst + c * kBoxQ, &args.tm_do, &bars[kDoFull], 64 * c, h, i * kQB, b);
            }
            if (rank == 1) {
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    *reinterpret_cast<uint4 *>(smem + Cfg::kOffDb + bias_off(r * 32 + lane, 0)) =
                        bias_row(dv[r]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kDoFull]);
            }
            ++ndo;
            return true;
        };
        for (int it = 0; ok; ++it) {
            SUnit un;
            if (!sunit_at(it, U, BH, nT, causal, un)) break;
            if (un.j < 0) continue;
            const int b = un.bh / H, h = un.bh % H;
            if (lane == 0) {
                w.code = kErrBwdWait + 0xa0;
                ok = mbar_wait(&bars[kKvEmpty], (nunit & 1) ^ 1, w);
                if (ok) {
                    if (rank == 0) {
                        mbar_arrive_expect_tx(&bars[kKvFull], 4 * kBoxK);
                        for (int c = 0; c < 4; ++c)
                            tma_load_4d(smem + Cfg::kOffK + c * kBoxK, &args.tm_k, &bars[kKvFull],
                                        64 * c, h, un.j * kKeys, b);
                    } else {
                        mbar_arrive_expect_tx(&bars[kKvFull], 6 * kBoxK);
                        for (int c = 0; c < 4; ++c)
                            tma_load_4d(smem + Cfg::kOffV + c * kBoxK, &args.tm_v, &bars[kKvFull],
                                        64 * c, h, un.j * kKeys, b);
                        for (int c = 0; c < 2; ++c)
                            tma_load_4d(smem + Cfg::kOffKh + c * kBoxK, &args.tm_k, &bars[kKvFull],
                                        128 + 64 * c, h, un.j * kKeys, b);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (ok) ++nkv;
            ++nunit;
            const int i0 = first_block(un.j);
            if (rank == 0) {
                // Q one block ahead of dO (Q is read by S^T, issued a block early)
                if (ok) ok = load_q(b, h, i0);
                for (int i = i0; i < nQ && ok; ++i) {
                    if (i + 1 < nQ) ok = load_q(b, h, i + 1);
                    if (ok) ok = load_do(b, h, i);
                }
            } else {
                // dO one block ahead of Q (dO is read by dP^T, issued a block early)
                if (ok) ok = load_do(b, h, i0);
                for (int i = i0; i < nQ && ok; ++i) {
                    if (i + 1 < nQ) ok = load_do(b, h, i + 1);
                    if (ok) ok = load_q(b, h, i);
                }
            }
        }
        if (!ok && lane == 0) {
            // let issued copies land before the CTA exits
            // (only those issued; rank 0 has two Q stages, both possibly in flight)
            if (nkv > 0) mbar_wait_drain(&bars[kKvFull], (nkv - 1) & 1);
            const uint32_t nst = (rank == 0) ? 2u : 1u;
            for (uint32_t m = nq > nst ? nq - nst : 0; m < nq; ++m) {
                const uint32_t st = (rank == 0) ? (m & 1) : 0;
                const uint32_t use = (rank == 0) ? (m >> 1) : m;
                mbar_wait_drain(&bars[kQFull0 + st], use & 1);
            }
            if (ndo > 0) mbar_wait_drain(&bars[kDoFull], (ndo - 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0xb0};
            uint32_t nunit = 0, n = 0;
            bool ok = true;
            const uint32_t tAcc = tmem + Cfg::kTAcc, tdQ = tmem + Cfg::kTdQ;
#define SW(bar, par, site)                                       \
    do {                                                         \
        w.code = kErrBwdWait + (site);                           \
        if (!mbar_wait((bar), (par), w)) { ok = false; break; } \
    } while (0)
            for (int it = 0; ok; ++it) {
                SUnit un;
                if (!sunit_at(it, U, BH, nT, causal, un)) break;
                if (un.j < 0) continue;
                const int i0 = first_block(un.j);
                SW(&bars[kKvFull], nunit & 1, 0xb0);
                if (!ok) break;
                if (rank == 0) {
                    const uint32_t aK = sbase + Cfg::kOffK, aOnes = sbase + Cfg::kOffOnes0;
                    // S^T of block n into X[n & 1] (Q stage n & 1, use n >> 1)
                    auto issue_s = [&](uint32_t nb) -> bool {
                        const uint32_t st = nb & 1;
                        w.code = kErrBwdWait + 0xb1;
                        if (!mbar_wait(&bars[kQFull0 + st], (nb >> 1) & 1, w)) return false;
                        tc_fence_after();
                        issue_rowcol(tmem + (st ? Cfg::kT1 : Cfg::kT0), aK,
                                     sbase + Cfg::kOffQ0 + st * 4 * kBoxQ, aOnes,
                                     sbase + Cfg::kOffLb + st * 2048);
                        mma_commit(&bars[kXFull0 + st]);
                        mma_commit(&bars[kQEmpty0 + st]);
                        return true;
                    };
                    // dQ^T[0:128] = K[:, 0:128]^T dS^T of block nb (dS^T from rank 1)
                    auto issue_dq0 = [&](uint32_t nb) -> bool {
                        const uint32_t st = nb & 1;
                        w.code = kErrBwdWait + 0xb5;
                        if (!mbar_wait(&bars[kDsrFull0 + st], (nb >> 1) & 1, w)) return false;
                        w.code = kErrBwdWait + 0xb6;
                        if (nb > 0 && !mbar_wait(&bars[kDqEmpty], (nb - 1) & 1, w)) return false;
                        tc_fence_after();
                        issue_dqt(tdQ, aK, sbase + Cfg::kOffDSR + st * kRow);
                        mma_commit(&bars[kDqFull]);
                        return true;
                    };
                    if (!issue_s(n)) { ok = false; break; }
                    // per block: S^T of the next block, dV, then dQ^T of the
                    // previous block, so that waiting for a block's dS^T (two
                    // trips between the CTAs) does not hold up the next S^T
                    for (int i = i0; i < nQ; ++i, ++n) {
                        const uint32_t st = n & 1;
                        const bool first = (i == i0);
                        // the next block's S^T first: its X stage last held P^T of
                        // block n - 1, read by dV(n - 1), which was issued before
                        if (i + 1 < nQ && !issue_s(n + 1)) { ok = false; break; }
                        SW(&bars[kPReady0 + st], (n >> 1) & 1, 0xb2);
                        if (first && nunit > 0) SW(&bars[kAccEmpty], (nunit - 1) & 1, 0xb3);
                        SW(&bars[kDoFull], n & 1, 0xb4);
                        if (!ok) break;
                        tc_fence_after();
                        // dV (+)= P^T dO: A = P^T in X (bf16), B = dO MN-major, N = 256
                        {
                            const uint32_t tX = tmem + (st ? Cfg::kT1 : Cfg::kT0);
                            const uint64_t bd = sdesc_sw128(sbase + Cfg::kOffDO0, kBoxQ, 1024);
#pragma unroll
                            for (int kk = 0; kk < kQB / 16; ++kk)
                                mma_ts(tAcc, tX + kk * 8, bd + ((kk * 2048) >> 4), Cfg::kIdescAcc,
                                       (!first || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&bars[kDoEmpty]);
                        if (!first && !issue_dq0(n - 1)) { ok = false; break; }
                    }
                    if (!ok) break;
                    if (!issue_dq0(n - 1)) { ok = false; break; }  // the unit's last block
                } else {
                    const uint32_t aV = sbase + Cfg::kOffV, aOnes = sbase + Cfg::kOffOnes1;
                    // dP^T of block n into Y[n & 1]
                    auto issue_dp = [&](uint32_t nb) -> bool {
                        w.code = kErrBwdWait + 0xb8;
                        if (!mbar_wait(&bars[kDoFull], nb & 1, w)) return false;
                        tc_fence_after();
                        issue_rowcol(tmem + ((nb & 1) ? Cfg::kT1 : Cfg::kT0), aV,
                                     sbase + Cfg::kOffDO1, aOnes, sbase + Cfg::kOffDb);
                        mma_commit(&bars[kXFull0 + (nb & 1)]);
                        mma_commit(&bars[kDoEmpty]);
                        return true;
                    };
                    if (!issue_dp(n)) { ok = false; break; }
                    for (int i = i0; i < nQ; ++i, ++n) {
                        const bool first = (i == i0);
                        // the next block's dP^T: its Y stage was last read by the
                        // dS^T phase of block n - 1, whose staging was waited for
                        if (i + 1 < nQ && !issue_dp(n + 1)) { ok = false; break; }
                        SW(&bars[kDsStaged], n & 1, 0xb9);
                        if (first && nunit > 0) SW(&bars[kAccEmpty], (nunit - 1) & 1, 0xba);
                        SW(&bars[kQFull0], n & 1, 0xbb);
                        if (!ok) break;
                        tc_fence_after();
                        // dK (+)= dS^T Q: A = dS^T K-major (rows = keys), B = Q MN-major, N = 256
                        {
                            const uint64_t ad = sdesc_sw128(sbase + Cfg::kOffDSL, 16, 1024);
                            const uint64_t bd = sdesc_sw128(sbase + Cfg::kOffQ1, kBoxQ, 1024);
#pragma unroll
                            for (int kk = 0; kk < kQB / 16; ++kk)
                                mma_ss(tAcc, ad + ((kk * 32) >> 4), bd + ((kk * 2048) >> 4),
                                       Cfg::kIdescAcc, (!first || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&bars[kQEmpty0]);
                        if (n > 0) SW(&bars[kDqEmpty], (n - 1) & 1, 0xbc);
                        if (!ok) break;
                        tc_fence_after();
                        issue_dqt(tdQ, sbase + Cfg::kOffKh, sbase + Cfg::kOffDSL);
                        mma_commit(&bars[kDqFull]);
                    }
                }
                if (!ok) break;
                mma_commit(&bars[kAccFull]);
                mma_commit(&bars[kKvEmpty]);
                ++nunit;
            }
#undef SW
            // every MMA issued must have finished before Tensor Memory is released
            mma_commit(&bars[kDrain]);
            mbar_wait_drain(&bars[kDrain], 0);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ P^T (rank 0) / dS^T (rank 1)
        const int quarter = warp & 3;
        const int kr = quarter * 32 + lane;  // key row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float c2 = args.scale_log2;
        const int sw = kr & 7;  // 128B swizzle phase of this row
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0xd0};
        uint32_t n = 0;
        bool ok = true;
        for (int it = 0; ok; ++it) {
            SUnit un;
            if (!sunit_at(it, U, BH, nT, causal, un)) break;
            if (un.j < 0) continue;
            const int key = un.j * kKeys + kr;
            for (int i = first_block(un.j); i < nQ; ++i, ++n) {
                const uint32_t st = n & 1;
                const uint32_t tX = tmem + (st ? Cfg::kT1 : Cfg::kT0) + lane_off;
                w.code = kErrBwdWait + 0xd0;
                if (!mbar_wait(&bars[kXFull0 + st], (n >> 1) & 1, w)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[2][32];
                tmem_ld32(tX, sr[0]);
                tmem_ld32(tX + 32, sr[1]);
                tmem_ld_wait(sr[0]);
                tmem_ld_wait(sr[1]);
                uint32_t pk[32];
                if (rank == 0) {
                    // X = S^T - LSE/scale: P = 2^(X c2); invisible pairs (keys past
                    // S; under a causal mask, queries before the key) get P = 0;
                    // queries past S carry a bias of -inf
                    const int lim = key - i * kQB;  // query columns < lim are hidden
                    if ((causal && lim > 0) || (un.j + 1) * kKeys > S) {
                        const bool key_ok = key < S;
                        const int l = causal ? lim : -1;
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (!key_ok || c * 32 + e < l) sr[c][e] = __float_as_uint(-INFINITY);
                    }
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 x = mul2(make_float2(__uint_as_float(sr[c][e]),
                                                              __uint_as_float(sr[c][e + 1])),
                                                  make_float2(c2, c2));
                            pk[(c * 32 + e) / 2] = pack_bf16x2(ex2_mufu(x.x), ex2_mufu(x.y));
                        }
                    // P^T into X for the dV MMA
                    tmem_st16(tX, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
                    tmem_st16(tX + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&bars[kPReady0 + st]);
                    // this warp's 32 rows of P^T (128 bytes each, 128B-swizzled)
                    // staged locally, then one bulk copy to rank 1's buffer once
                    // rank 1's warp with the same rows has read the last block's
                    if (lane == 0) bulk_wait_read<0>();  // the previous copy has read the slice
                    __syncwarp();
                    uint8_t *prow = smem + Cfg::kOffPS + kr * 128;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        *reinterpret_cast<uint4 *>(prow + ((ch ^ sw) << 4)) =
                            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        w.code = kErrBwdWait + 0xd1;
                        if (mbar_wait(&bars[kPrFree0 + quarter], (n & 1) ^ 1, w)) {
                            const uint32_t full = peer_bar(kPrFull0 + quarter);
                            mbar_arrive_expect_tx_cluster(full, 4096);
                            bulk_copy_to_cluster(
                                mapa_shared(sbase + Cfg::kOffPR + quarter * 4096, peer),
                                smem + Cfg::kOffPS + quarter * 4096, 4096, full);
                            bulk_commit();
                        }
                    }
                    if (*abort_flag) { ok = false; break; }
                } else {
                    // Y = dP^T - Delta; dS^T = P^T o Y with this warp's 32 rows of
                    // P^T from rank 0
                    w.code = kErrBwdWait + 0xd2;
                    if (!mbar_wait(&bars[kPrFull0 + quarter], n & 1, w)) { ok = false; break; }
                    const uint8_t *prow = smem + Cfg::kOffPR + kr * 128;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(prow + ((ch ^ sw) << 4));
                        pk[4 * ch] = v.x;
                        pk[4 * ch + 1] = v.y;
                        pk[4 * ch + 2] = v.z;
                        pk[4 * ch + 3] = v.w;
                    }
                    // the dS^T buffer: the previous block's dK and dQ^T MMAs have
                    // read it, and this warp's copy of its rows has
                    w.code = kErrBwdWait + 0xd3;
                    if (!mbar_wait(&bars[kDsFree], (n & 1) ^ 1, w)) { ok = false; break; }
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
                    uint8_t *drow = smem + Cfg::kOffDSL + kr * 128;
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            uint32_t d4[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int e = t * 8 + u * 2;
                                // the fp32 difference rounded to bf16, times the bf16 P
                                d4[u] = mul_bf16x2(pk[(c * 32 + e) >> 1],
                                                   pack_bf16x2(__uint_as_float(sr[c][e]),
                                                               __uint_as_float(sr[c][e + 1])));
                            }
                            const int ch = c * 4 + t;
                            *reinterpret_cast<uint4 *>(drow + ((ch ^ sw) << 4)) =
                                make_uint4(d4[0], d4[1], d4[2], d4[3]);
                        }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        // every lane has used its P^T row (the loads are complete),
                        // so rank 0 may overwrite this warp's rows with the next block's
                        mbar_arrive_cluster(peer_bar(kPrFree0 + quarter));
                        mbar_arrive(&bars[kDsStaged]);
                        // this warp's rows to rank 0's stage n % 2, once rank 0's
                        // dQ^T MMA has finished with that stage's previous block
                        w.code = kErrBwdWait + 0xd4;
                        if (mbar_wait(&bars[kDsrFree0 + st], ((n >> 1) & 1) ^ 1, w)) {
                            const uint32_t full = peer_bar(kDsrFull0 + st);
                            mbar_arrive_expect_tx_cluster(full, 4096);
                            bulk_copy_to_cluster(
                                mapa_shared(sbase + Cfg::kOffDSR + st * kRow + quarter * 4096, peer),
                                smem + Cfg::kOffDSL + quarter * 4096, 4096, full);
                            bulk_commit();
                        }
                    }
                    if (*abort_flag) { ok = false; break; }
                }
            }
        }
        if (lane == 0) bulk_wait<0>();  // this warp's copies have completed
    } else if (warp >= 8) {
        // ------------------------------------------------------------ dQ drain + dV / dK epilogue
        // dQ^T of this rank's half of d (lane = d column, 64 query columns) is
        // staged per warp as 32 queries x 32 columns (4 KB, 128B swizzle) and
        // added into the accumulator by TMA bulk reductions.
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        // rank 0 has 2 KB per warp (16-row boxes), rank 1 4 KB (32-row boxes)
        const CUtensorMap *red_map = rank == 0 ? &args.tm_dqacc16 : &args.tm_dqacc;
        uint8_t *stage = smem + (rank == 0 ? Cfg::kOffRed0 + quarter * 2048 : Cfg::kOffRed1 + quarter * 4096);
        const bool signaller = (threadIdx.x == 256);
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0xe0};
        uint32_t n = 0, nunit = 0;
        bool ok = true;
        for (int it = 0; ok; ++it) {
            SUnit un;
            if (!sunit_at(it, U, BH, nT, causal, un)) break;
            if (un.j < 0) continue;
            const int b = un.bh / H, h = un.bh % H;
            for (int i = first_block(un.j); i < nQ; ++i, ++n) {
                w.code = kErrBwdWait + 0xe0;
                if (!mbar_wait(&bars[kDqFull], n & 1, w)) { ok = false; break; }
                tc_fence_after();
                uint32_t col[2][32];
                tmem_ld32(tmem + Cfg::kTdQ + lane_off, col[0]);
                tmem_ld32(tmem + Cfg::kTdQ + lane_off + 32, col[1]);
                tmem_ld_wait(col[0]);
                tmem_ld_wait(col[1]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kDqEmpty]);
                if (signaller) {
                    // the dQ^T MMA (and, on rank 1, the dK MMA before it) has
                    // finished reading this block's dS^T
                    if (rank == 0)
                        mbar_arrive_cluster(peer_bar(kDsrFree0 + (n & 1)));
                    else
                        mbar_arrive(&bars[kDsFree]);
                }
                const int d0 = static_cast<int>(rank) * 128 + quarter * 32;
                if (rank == 0)
                    stage_reduce<16>(col, stage, red_map, d0, i * kQB, un.bh, lane, abort_flag);
                else
                    stage_reduce<32>(col, stage, red_map, d0, i * kQB, un.bh, lane, abort_flag);
            }
            if (!ok) break;
            w.code = kErrBwdWait + 0xe1;
            if (!mbar_wait(&bars[kAccFull], nunit & 1, w)) { ok = false; break; }
            ++nunit;
            tc_fence_after();
            // rank 0: dV; rank 1: dK (x scale), all 256 columns of this key row
            const int key = un.j * kKeys + r;
            const float mul = rank ? args.scale : 1.f;
            uint16_t *out = reinterpret_cast<uint16_t *>(rank ? args.dk : args.dv) +
                            ((static_cast<size_t>(b) * S + key) * H + h) * kD;
#pragma unroll 1
            for (int c = 0; c < kD / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + Cfg::kTAcc + lane_off + c * 32, v);
                tmem_ld_wait(v);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul,
                                        __uint_as_float(v[2 * e + 1]) * mul);
                if (key < S) {
                    uint4 *dst = reinterpret_cast<uint4 *>(out + c * 32);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2],
                                             pk[4 * v4 + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kAccEmpty]);
        }
        if (lane == 0) bulk_wait<0>();  // this warp's reductions have read shared memory
    }

    // neither CTA leaves (or releases Tensor Memory) while the other may still
    // write its shared memory or arrive on its barriers
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_bwd_main_d256_split(const BwdArgs &a, cudaStream_t stream) {
    if (a.D != kD || a.cu_seqlens || a.dq_sem) return cudaErrorNotSupported;
    auto kern = fa_bwd_d256_split_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SplitCfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long U = static_cast<long long>(a.B) * a.H * ((a.S + kKeys - 1) / kKeys);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SplitCfg::kSmemBytes;
    cfg.stream = stream;
    cfg.gridDim = dim3(2 * (a.num_sms / 2));
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int max_pairs = 0;
    e = cudaOccupancyMaxActiveClusters(&max_pairs, reinterpret_cast<const void *>(kern), &cfg);
    if (e != cudaSuccess) return e;
    if (max_pairs < 1) return cudaErrorNotSupported;
    const long long pairs = U < max_pairs ? U : max_pairs;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace fa
