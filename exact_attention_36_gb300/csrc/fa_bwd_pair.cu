// fa_bwd_pair.cu -- fused attention backward for D = 128 on CTA pairs
// (tcgen05 .cta_group::2), sm_103a.
//
// Same mathematics as fa_bwd.cu (P = exp(scale*S - LSE), dS = P o (dP - Delta),
// dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K), laid out for a cluster of
// two CTAs on neighbouring SMs as the pages describe for the backward
// ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
// Hardware Scaling" (gist.science/nl), Methodologie §3): in the 2-CTA MMA mode
// operand B is split between the two CTAs, so each loads only half of it from
// shared memory, and the two CTAs exchange halves of the dQ work through
// distributed shared memory, which halves the global dQ reductions.
//
// A work unit is (b, h, key-tile pair p): CTA r of the pair owns key tile
// j = 2p + r (its K_j and V_j stay in its shared memory) and both stream the
// same 128-query blocks Q_i, dO_i.  Keys sit on the TMEM lanes as in the
// single-CTA kernel; the pair's MMAs (issued by one thread of CTA 0) are
//   S^T  = K Q_i^T   M=256 keys, N=128 queries   B: Q_i rows, 64 per CTA
//   dP^T = V dO_i^T  M=256, N=128                B: dO_i rows, 64 per CTA
//   dV  += P^T dO_i  M=256, N=128 (d), A in TMEM B: dO_i columns, 64 per CTA
//   dK  += dS^T Q_i  M=256, N=128 (d), A in TMEM B: Q_i columns, 64 per CTA
//   dQ_i = dS K      M=128 queries, N=128, K=256 keys of the pair
// For dQ, CTA r supplies the dS rows of queries [64r, 64r+64) over all 256
// keys (its own half is written locally, the other CTA writes its keys' half
// remotely) and the d-columns [64r, 64r+64) of K for both key tiles; each CTA
// receives its 64 queries' dQ, summed over both key tiles, and reduces only
// that into the fp32 accumulator.  In Tensor Memory an M = 128 pair result
// holds a CTA's 64 rows on lanes 0-63 (columns 0-63 of N) and again on lanes
// 64-127 (columns 64-127 of N), so dQ takes 64 columns.
//
// Tensor Memory (per CTA): X [0,128) S^T -> P^T | Y [128,256) dP^T -> dS^T in
// Y[0,64), dQ in Y[64,128) | dV [256,384) | dK [384,512).
//
// Warp roles (384 threads per CTA):
//   warp 0      TMA producer of this CTA's operands (+ LSE/Delta of the block)
//   warp 1      CTA 0: TMEM allocation and MMA issue for the pair; CTA 1:
//               TMEM allocation and relay (forwards "operands landed" of CTA
//               1's copies to CTA 0's issuer)
//   warps 4-7   P^T and dS^T of this CTA's 128 keys (lane = key)
//   warps 8-11  dQ drain of this CTA's 64 queries, dK/dV epilogue
#include <cuda_bf16.h>

#include "fa_common.cuh"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr int kBlk = 128;       // keys per tile, queries per block
constexpr int kD = 128;         // head dimension of this kernel
constexpr int kBox = 16384;     // 128 rows x 64 bf16, 128B swizzle
constexpr int kHalfBox = 8192;  // 64 rows x 64 bf16

struct PairCfg {
    // shared memory map (offsets from a 1024-byte aligned base)
    static constexpr int kOffK = 0;                 // K_j: 128 keys x 128 d, K-major (2 boxes)
    static constexpr int kOffV = kOffK + 2 * kBox;  // V_j
    static constexpr int kOffKd = kOffV + 2 * kBox;  // dQ's B: 256 keys x 64 d (2 boxes)
    static constexpr int kOffQs = kOffKd + 2 * kBox;   // S^T's B: 64 query rows x 128 d
    static constexpr int kOffQd = kOffQs + 2 * kHalfBox;  // dK's B: 128 queries x 64 d
    static constexpr int kOffDOs = kOffQd + kBox;         // dP^T's B: 64 rows x 128 d
    static constexpr int kOffDOd = kOffDOs + 2 * kHalfBox;  // dV's B: 128 x 64 d
    static constexpr int kOffDS = kOffDOd + kBox;  // dQ's A: 256 keys x 64 queries bf16
    static constexpr int kOffDSx = kOffDS + 2 * kBox;  // the other CTA's dS half, outgoing
    static constexpr int kOffRed = kOffDSx + kBox;     // dQ staging: 4 warps x 32 x 32 fp32
    static constexpr int kOffStat = kOffRed + kBox;    // 2 x (128 lse2 + 128 delta) fp32
    static constexpr int kOffBar = kOffStat + 2 * 1024;
    static constexpr int kNumBars = 27;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kSmemBytes = kOffMisc + 16;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTX = 0, kTY = 128, kTdQ = 192, kTdV = 256, kTdK = 384;
    static constexpr uint32_t kIdescS = idesc_bf16_f32(256, 128, false, false);   // S^T, dP^T
    static constexpr uint32_t kIdescAcc = idesc_bf16_f32(256, kD, false, true);   // dV, dK
    static constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, kD, true, true);     // dQ
};
static_assert(PairCfg::kSmemBytes <= 232448, "shared memory");

// barrier slots
enum PairBar : int {
    kKvFull, kKvEmpty, kQsFull, kQsEmpty, kQdFull, kQdEmpty, kDosFull, kDosEmpty, kDodFull,
    kDodEmpty, kSFull, kDpFull, kPReady, kDsReady, kDqFull, kDqEmpty, kDkdvFull, kDkdvEmpty,
    kDrain, kPkKv, kPkQs, kPkQd, kPkDos, kPkDod, kDsIn, kPkDs, kStaged
};

struct PUnit {
    int bh;  // b * H + h
    int p;   // key-tile pair; -1 = no unit for this pair this round
};

// Units of one head are consecutive (concurrent pairs share that head's Q, dO
// and dQ accumulator in L2); within a head pair 0 comes first, which under a
// causal mask sees the most query blocks.  Serpentine over the pairs.
__device__ __forceinline__ bool punit_at(int it, int U, int nP, PUnit &out) {
    const int G = gridDim.x >> 1;
    const int pid = blockIdx.x >> 1;
    const int base = it * G;
    if (base >= U) return false;
    const int c = (it & 1) ? (G - 1 - pid) : pid;
    const int u = base + c;
    if (u >= U) {
        out.p = -1;
        return true;
    }
    out.bh = u / nP;
    out.p = u % nP;
    return true;
}

// ---------------------------------------------------------------- pair MMAs

// S^T / dP^T: A = own 128 rows x 128 d (K-major), B = 64 query rows x 128 d
// (descriptors built once per call; a K step adds its byte offset / 16)
__device__ __forceinline__ void issue_s(uint32_t tD, uint32_t a_saddr, uint32_t b_saddr) {
    const uint64_t ad = sdesc_sw128(a_saddr, 16, 1024), bd = sdesc_sw128(b_saddr, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk)
        mma_ss_pair(tD, ad + (((kk / 4) * kBox + (kk % 4) * 32) >> 4),
                    bd + (((kk / 4) * kHalfBox + (kk % 4) * 32) >> 4), PairCfg::kIdescS,
                    kk > 0 ? 1u : 0u);
}

// dV / dK: A = 128 keys x 128 queries bf16 in TMEM, B = 128 queries x 64 d (MN-major)
__device__ __forceinline__ void issue_acc(uint32_t tAcc, uint32_t tA, uint32_t b_saddr, bool acc) {
    const uint64_t bd = sdesc_sw128(b_saddr, kBox, 1024);
#pragma unroll
    for (int kk = 0; kk < kBlk / 16; ++kk)
        mma_ts_pair(tAcc, tA + kk * 8, bd + ((kk * 2048) >> 4), PairCfg::kIdescAcc,
                    (acc || kk > 0) ? 1u : 0u);
}

// dQ: A = 64 queries x 256 keys (MN-major, rows = keys), B = 256 keys x 64 d (MN-major)
__device__ __forceinline__ void issue_dq(uint32_t tD, uint32_t ds_saddr, uint32_t kd_saddr) {
    const uint64_t ad = sdesc_sw128(ds_saddr, kBox, 1024), bd = sdesc_sw128(kd_saddr, kBox, 1024);
#pragma unroll
    for (int kk = 0; kk < 2 * kBlk / 16; ++kk)
        mma_ss_pair(tD, ad + ((kk * 2048) >> 4), bd + ((kk * 2048) >> 4), PairCfg::kIdescDQ,
                    kk > 0 ? 1u : 0u);
}

// ---------------------------------------------------------------- main kernel

__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_pair_kernel(const __grid_constant__ BwdArgs args) {
    using Cfg = PairCfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    // both CTAs take the same path out: a bad base alignment is the same in both
    const bool bad_base = (smem_u32(smem) & 1023u) != 0;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);
    float *stat = reinterpret_cast<float *>(smem + Cfg::kOffStat);  // [stage][lse2 128 | delta 128]

    const uint32_t rank = cluster_rank();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = args.H, S = args.S;
    const int BH = args.B * H;
    const int nT = (S + kBlk - 1) / kBlk;  // key tiles = query blocks
    const int nP = (nT + 1) / 2;           // key-tile pairs
    const int U = BH * nP;
    if (bad_base) {
        if (threadIdx.x == 0) atomicCAS(args.err_word, 0, kErrBwdWait + 0xfe);
        return;
    }

    if (threadIdx.x == 0) {
        // barriers arrived on from both CTAs (CTA 0's copies are the ones used):
        // one elected lane per warp of the four-warp roles
        const uint32_t counts[Cfg::kNumBars] = {
            1, 1, 2, 1, 1, 1, 1, 1, 1, 1,  // kv .. dod_empty
            1, 1, 8, 8, 1, 8, 1, 8,        // s_full .. dkdv_empty
            1, 1, 1, 1, 1, 1,              // drain, pk_*
            1, 1,                          // ds_in (+ the other CTA's copy), pk_ds
            4};                            // staged: the four softmax warps' dS rows
        for (int i = 0; i < Cfg::kNumBars; ++i) mbar_init(&bars[i], counts[i]);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, Cfg::kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&args.tm_q);
        tma_prefetch_desc(&args.tm_q64);
        tma_prefetch_desc(&args.tm_k);
        tma_prefetch_desc(&args.tm_v);
        tma_prefetch_desc(&args.tm_do);
        tma_prefetch_desc(&args.tm_do64);
        tma_prefetch_desc(&args.tm_dqacc);
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t sbase = smem_u32(smem);
    // CTA 0's copy of a barrier, as a cluster address
    auto lead = [&](int slot) { return mapa_shared(smem_u32(&bars[slot]), 0); };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0x81};
        uint32_t nunit = 0, nblk = 0;
        // copies issued per barrier, counted by lane 0 (for the unwinding)
        uint32_t nkv = 0, nqs = 0, ndos = 0, ndod = 0, nqd = 0;
        bool ok = true;
        const float log2e = 1.4426950408889634f;
        const int dcol = 64 * static_cast<int>(rank);  // this CTA's half of d
        for (int it = 0; ok; ++it) {
            PUnit un;
            if (!punit_at(it, U, nP, un)) break;
            if (un.p < 0) continue;
            const int b = un.bh / H, h = un.bh % H;
            const int j = 2 * un.p + static_cast<int>(rank);
            const int i0 = args.causal ? 2 * un.p : 0;
            if (lane == 0) {
                w.code = kErrBwdWait + 0x81;
                ok = mbar_wait(&bars[kKvEmpty], (nunit & 1) ^ 1, w);
                if (ok) {
                    mbar_arrive_expect_tx(&bars[kKvFull], 6 * kBox);
                    for (int c = 0; c < 2; ++c) {
                        tma_load_4d(smem + Cfg::kOffK + c * kBox, &args.tm_k, &bars[kKvFull],
                                    64 * c, h, j * kBlk, b);
                        tma_load_4d(smem + Cfg::kOffV + c * kBox, &args.tm_v, &bars[kKvFull],
                                    64 * c, h, j * kBlk, b);
                        tma_load_4d(smem + Cfg::kOffKd + c * kBox, &args.tm_k, &bars[kKvFull],
                                    dcol, h, (2 * un.p + c) * kBlk, b);
                    }
                    ++nkv;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            ++nunit;
            for (int i = i0; i < nT && ok; ++i, ++nblk) {
                const int qrow = i * kBlk + 64 * static_cast<int>(rank);
                // Q rows of this CTA's half for S^T, then LSE / Delta of the block
                w.code = kErrBwdWait + 0x82;
                ok = mbar_wait(&bars[kQsEmpty], (nblk & 1) ^ 1, w);
                ok = __all_sync(0xffffffffu, ok ? 1 : 0) != 0;
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[kQsFull], 2 * kHalfBox);
                    for (int c = 0; c < 2; ++c)
                        tma_load_4d(smem + Cfg::kOffQs + c * kHalfBox, &args.tm_q64,
                                    &bars[kQsFull], 64 * c, h, qrow, b);
                    ++nqs;
                }
                // the stage written here was last read by the dS phase of block
                // nblk - 2, which finished before dK(nblk - 2): the producer
                // waited for that MMA before loading Qd(nblk - 1)
                float *sl = stat + (nblk & 1) * 256;
                const size_t rbase = static_cast<size_t>(un.bh) * S;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int qr = r * 32 + lane;
                    const int q = i * kBlk + qr;
                    const bool in = q < S;
                    sl[qr] = in ? args.lse[rbase + q] * log2e : INFINITY;
                    sl[128 + qr] = in ? args.delta[rbase + q] : 0.f;
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars[kQsFull]);
                    // dO rows for dP^T
                    w.code = kErrBwdWait + 0x83;
                    ok = mbar_wait(&bars[kDosEmpty], (nblk & 1) ^ 1, w);
                    if (ok) {
                        mbar_arrive_expect_tx(&bars[kDosFull], 2 * kHalfBox);
                        for (int c = 0; c < 2; ++c)
                            tma_load_4d(smem + Cfg::kOffDOs + c * kHalfBox, &args.tm_do64,
                                        &bars[kDosFull], 64 * c, h, qrow, b);
                        ++ndos;
                    }
                    // dO columns for dV
                    w.code = kErrBwdWait + 0x84;
                    if (ok) ok = mbar_wait(&bars[kDodEmpty], (nblk & 1) ^ 1, w);
                    if (ok) {
                        mbar_arrive_expect_tx(&bars[kDodFull], kBox);
                        tma_load_4d(smem + Cfg::kOffDOd, &args.tm_do, &bars[kDodFull], dcol, h,
                                    i * kBlk, b);
                        ++ndod;
                    }
                    // Q columns for dK
                    w.code = kErrBwdWait + 0x85;
                    if (ok) ok = mbar_wait(&bars[kQdEmpty], (nblk & 1) ^ 1, w);
                    if (ok) {
                        mbar_arrive_expect_tx(&bars[kQdFull], kBox);
                        tma_load_4d(smem + Cfg::kOffQd, &args.tm_q, &bars[kQdFull], dcol, h,
                                    i * kBlk, b);
                        ++nqd;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            }
        }
        if (!ok && lane == 0) {
            // let issued copies land before the CTA exits
            // (only the copies issued: the loop may stop part-way through a block)
            if (nkv > 0) mbar_wait_drain(&bars[kKvFull], (nkv - 1) & 1);
            if (nqs > 0) mbar_wait_drain(&bars[kQsFull], (nqs - 1) & 1);
            if (ndos > 0) mbar_wait_drain(&bars[kDosFull], (ndos - 1) & 1);
            if (ndod > 0) mbar_wait_drain(&bars[kDodFull], (ndod - 1) & 1);
            if (nqd > 0) mbar_wait_drain(&bars[kQdFull], (nqd - 1) & 1);
        }
    }
    else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // -------------------------------------------------------- MMA issuer of the pair
            WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0x90};
            const uint32_t tX = tmem + Cfg::kTX, tY = tmem + Cfg::kTY, tdQ = tmem + Cfg::kTdQ;
            const uint32_t tdV = tmem + Cfg::kTdV, tdK = tmem + Cfg::kTdK;
            const uint32_t aK = sbase + Cfg::kOffK, aV = sbase + Cfg::kOffV;
            const uint32_t aKd = sbase + Cfg::kOffKd, aQs = sbase + Cfg::kOffQs;
            const uint32_t aQd = sbase + Cfg::kOffQd, aDOs = sbase + Cfg::kOffDOs;
            const uint32_t aDOd = sbase + Cfg::kOffDOd, aDS = sbase + Cfg::kOffDS;
            uint32_t nunit = 0, nblk = 0;
            uint32_t ph_p = 0, ph_ds = 0, ph_dqe = 0;
            bool ok = true;
            // own copy landed (local barrier) and the other CTA's (relayed)
#define PW(slot, par, site)                                              \
    do {                                                                 \
        w.code = kErrBwdWait + (site);                                   \
        if (!mbar_wait(&bars[slot], (par), w)) { ok = false; break; }    \
    } while (0)
#define PWC(slot, par, site) PW(slot, par, site)
            for (int it = 0; ok; ++it) {
                PUnit un;
                if (!punit_at(it, U, nP, un)) break;
                if (un.p < 0) continue;
                const int i0 = args.causal ? 2 * un.p : 0;
                PW(kKvFull, nunit & 1, 0x90);
                if (!ok) break;
                PWC(kPkKv, nunit & 1, 0x91);
                if (!ok) break;
                {
                    // first block of the unit: S^T and dP^T
                    PW(kQsFull, nblk & 1, 0x92);
                    if (!ok) break;
                    PWC(kPkQs, nblk & 1, 0x93);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(tX, aK, aQs);
                    mma_commit_pair(&bars[kSFull]);
                    mma_commit_pair(&bars[kQsEmpty]);
                    if (nblk > 0) {
                        // the previous block's dQ has left Y
                        PWC(kDqEmpty, ph_dqe, 0x94);
                        if (!ok) break;
                        ph_dqe ^= 1;
                    }
                    PW(kDosFull, nblk & 1, 0x95);
                    if (!ok) break;
                    PWC(kPkDos, nblk & 1, 0x96);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(tY, aV, aDOs);
                    mma_commit_pair(&bars[kDpFull]);
                    mma_commit_pair(&bars[kDosEmpty]);
                }
                for (int i = i0; i < nT; ++i, ++nblk) {
                    const bool first = (i == i0), has_next = (i + 1 < nT);
                    PWC(kPReady, ph_p, 0x97);
                    if (!ok) break;
                    ph_p ^= 1;
                    if (first && nunit > 0) {
                        // the previous unit's dK/dV epilogue has read the accumulators
                        PWC(kDkdvEmpty, (nunit - 1) & 1, 0x98);
                        if (!ok) break;
                    }
                    PW(kDodFull, nblk & 1, 0x99);
                    if (!ok) break;
                    PWC(kPkDod, nblk & 1, 0x9a);
                    if (!ok) break;
                    tc_fence_after();
                    issue_acc(tdV, tX, aDOd, !first);
                    mma_commit_pair(&bars[kDodEmpty]);
                    if (has_next) {
                        PW(kQsFull, (nblk + 1) & 1, 0x9b);
                        if (!ok) break;
                        PWC(kPkQs, (nblk + 1) & 1, 0x9c);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(tX, aK, aQs);
                        mma_commit_pair(&bars[kSFull]);
                        mma_commit_pair(&bars[kQsEmpty]);
                    }
                    PWC(kDsReady, ph_ds, 0x9d);
                    if (!ok) break;
                    ph_ds ^= 1;
                    PW(kQdFull, nblk & 1, 0x9e);
                    if (!ok) break;
                    PWC(kPkQd, nblk & 1, 0x9f);
                    if (!ok) break;
                    tc_fence_after();
                    issue_acc(tdK, tY, aQd, !first);
                    mma_commit_pair(&bars[kQdEmpty]);
                    // both CTAs' dS operands complete: the other CTA's half
                    // copied into this one, and this CTA's half into the other
                    PW(kDsIn, nblk & 1, 0xa3);
                    if (!ok) break;
                    PWC(kPkDs, nblk & 1, 0xa4);
                    if (!ok) break;
                    tc_fence_after();
                    issue_dq(tdQ, aDS, aKd);
                    mma_commit_pair(&bars[kDqFull]);
                    if (has_next) {
                        PWC(kDqEmpty, ph_dqe, 0xa0);
                        if (!ok) break;
                        ph_dqe ^= 1;
                        PW(kDosFull, (nblk + 1) & 1, 0xa1);
                        if (!ok) break;
                        PWC(kPkDos, (nblk + 1) & 1, 0xa2);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(tY, aV, aDOs);
                        mma_commit_pair(&bars[kDpFull]);
                        mma_commit_pair(&bars[kDosEmpty]);
                    } else {
                        mma_commit_pair(&bars[kDkdvFull]);
                        mma_commit_pair(&bars[kKvEmpty]);
                    }
                }
                ++nunit;
            }
#undef PW
#undef PWC
            // every MMA issued must have finished before Tensor Memory is released
            mma_commit_pair(&bars[kDrain]);
            mbar_wait_drain(&bars[kDrain], 0);
        } else if (lane == 0) {
            // -------------------------------------------------------- relay (CTA 1)
            // CTA 0's issuer cannot wait on this CTA's barriers; forward each
            // completed copy to its pair barrier in CTA 0, in load order
            WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0xb0};
            uint32_t nunit = 0, nblk = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                PUnit un;
                if (!punit_at(it, U, nP, un)) break;
                if (un.p < 0) continue;
                const int i0 = args.causal ? 2 * un.p : 0;
                w.code = kErrBwdWait + 0xb0;
                if (!(ok = mbar_wait(&bars[kKvFull], nunit & 1, w))) break;
                mbar_arrive_cluster(lead(kPkKv));
                ++nunit;
                for (int i = i0; i < nT && ok; ++i, ++nblk) {
                    const int slots[4] = {kQsFull, kDosFull, kDodFull, kQdFull};
                    const int pk[4] = {kPkQs, kPkDos, kPkDod, kPkQd};
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) {
                        w.code = kErrBwdWait + 0xb1 + s2;
                        if (!(ok = mbar_wait(&bars[slots[s2]], nblk & 1, w))) break;
                        mbar_arrive_cluster(lead(pk[s2]));
                    }
                }
            }
        }
    }
    else if (warp == 2) {
        if (lane == 0 && rank == 1) {
            // -------------------------------------------------------- relay of dS copies (CTA 1)
            WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0xb8};
            uint32_t nblk = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                PUnit un;
                if (!punit_at(it, U, nP, un)) break;
                if (un.p < 0) continue;
                const int i0 = args.causal ? 2 * un.p : 0;
                for (int i = i0; i < nT && ok; ++i, ++nblk) {
                    if (!(ok = mbar_wait(&bars[kDsIn], nblk & 1, w))) break;
                    mbar_arrive_cluster(lead(kPkDs));
                }
            }
        }
    }
    else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ P^T and dS^T
        const int quarter = warp & 3;
        const int kr = quarter * 32 + lane;  // key row of this CTA's tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tX = tmem + Cfg::kTX + lane_off, tY = tmem + Cfg::kTY + lane_off;
        const float c2 = args.scale_log2;
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0xc0};
        uint32_t n = 0;
        bool ok = true;
        // this key's row of the dQ operand in both CTAs: queries [0,64) go to
        // CTA 0, [64,128) to CTA 1, row = 128 * rank + kr, 128B-swizzled.  The
        // other CTA's half is staged here (row kr, same swizzle) and sent as one
        // bulk copy.
        uint8_t *ds_own = smem + Cfg::kOffDS + (rank * 128 + kr) * 128;
        uint8_t *ds_out = smem + Cfg::kOffDSx + kr * 128;
        const uint32_t peer = rank ^ 1;
        const uint32_t ds_peer_rows = mapa_shared(sbase + Cfg::kOffDS + rank * 128 * 128, peer);
        const uint32_t ds_peer_bar = mapa_shared(smem_u32(&bars[kDsIn]), peer);
        const bool copier = (threadIdx.x == 128);
        const int sw = kr & 7;
        const uint32_t bar_p = lead(kPReady), bar_ds = lead(kDsReady);
        for (int it = 0; ok; ++it) {
            PUnit un;
            if (!punit_at(it, U, nP, un)) break;
            if (un.p < 0) continue;
            const int j = 2 * un.p + static_cast<int>(rank);
            const int i0 = args.causal ? 2 * un.p : 0;
            const int key = j * kBlk + kr;
            for (int i = i0; i < nT; ++i, ++n) {
                w.code = kErrBwdWait + 0xc0;
                if (!mbar_wait(&bars[kQsFull], n & 1, w)) { ok = false; break; }
                w.code = kErrBwdWait + 0xc1;
                if (!mbar_wait(&bars[kSFull], n & 1, w)) { ok = false; break; }
                tc_fence_after();
                const float *lse2 = stat + (n & 1) * 256;
                const float *dlt = lse2 + 128;
                uint32_t pk[64];
                {
                    uint32_t sr[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(tX + c * 32, sr[c]);
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
                    // invisible pairs: keys past S, and under a causal mask
                    // queries before the key (query column c < lim); queries
                    // past S carry lse2 = +inf, which gives P = 0
                    const bool diag = args.causal && i <= j;
                    if (diag || (j + 1) * kBlk > S) {
                        const int lim = diag ? (j - i) * kBlk + kr : -1;
                        const bool key_ok = key < S;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (!key_ok || c * 32 + e < lim)
                                    sr[c][e] = __float_as_uint(-INFINITY);
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            const float4 l4 = *reinterpret_cast<const float4 *>(lse2 + c * 32 + e);
                            const float p0 = ex2_mufu(fmaf(__uint_as_float(sr[c][e]), c2, -l4.x));
                            const float p1 = ex2_mufu(fmaf(__uint_as_float(sr[c][e + 1]), c2, -l4.y));
                            const float p2 = ex2_mufu(fmaf(__uint_as_float(sr[c][e + 2]), c2, -l4.z));
                            const float p3 = ex2_mufu(fmaf(__uint_as_float(sr[c][e + 3]), c2, -l4.w));
                            pk[(c * 32 + e) / 2] = pack_bf16x2(p0, p1);
                            pk[(c * 32 + e) / 2 + 1] = pack_bf16x2(p2, p3);
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tmem_st16(tX + c * 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[c * 16]));
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(bar_p);
                // ---- dS^T = P^T o (dP^T - Delta)
                w.code = kErrBwdWait + 0xc2;
                if (!mbar_wait(&bars[kDpFull], n & 1, w)) { ok = false; break; }
                if (n > 0) {
                    // the previous dQ MMA has finished reading both CTAs' dS
                    w.code = kErrBwdWait + 0xc3;
                    if (!mbar_wait(&bars[kDqFull], (n - 1) & 1, w)) { ok = false; break; }
                }
                tc_fence_after();
#pragma unroll
                for (int c2i = 0; c2i < 4; c2i += 2) {
                    uint32_t drr[2][32];
                    tmem_ld32(tY + c2i * 32, drr[0]);
                    tmem_ld32(tY + c2i * 32 + 32, drr[1]);
                    tmem_ld_wait(drr[0]);
                    tmem_ld_wait(drr[1]);
#pragma unroll
                    for (int c = c2i; c < c2i + 2; ++c) {
                        const uint32_t(&dr)[32] = drr[c - c2i];
                        uint32_t dsw[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            // dS = P o (dP - Delta): the difference in fp32, rounded
                            // to bf16 and multiplied by the bf16 P, two columns per
                            // instruction
                            const float4 d4 = *reinterpret_cast<const float4 *>(dlt + c * 32 + e);
                            const float2 t0 = sub2(make_float2(__uint_as_float(dr[e]),
                                                               __uint_as_float(dr[e + 1])),
                                                   make_float2(d4.x, d4.y));
                            const float2 t1 = sub2(make_float2(__uint_as_float(dr[e + 2]),
                                                               __uint_as_float(dr[e + 3])),
                                                   make_float2(d4.z, d4.w));
                            dsw[e / 2] = mul_bf16x2(pk[(c * 32 + e) >> 1], pack_bf16x2(t0.x, t0.y));
                            dsw[e / 2 + 1] =
                                mul_bf16x2(pk[(c * 32 + e + 2) >> 1], pack_bf16x2(t1.x, t1.y));
                        }
                        tmem_st16(tY + c * 16, dsw);
                        // queries [32c, 32c+32) of this key: CTA c/2's dQ operand,
                        // 16-byte units 4(c&1) .. 4(c&1)+3 of the row
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int unit = (c & 1) * 4 + t;
                            const uint4 v4 = make_uint4(dsw[4 * t], dsw[4 * t + 1],
                                                        dsw[4 * t + 2], dsw[4 * t + 3]);
                            uint8_t *row = (c >> 1) == static_cast<int>(rank) ? ds_own : ds_out;
                            *reinterpret_cast<uint4 *>(row + ((unit ^ sw) << 4)) = v4;
                        }
                    }
                }
                fence_proxy_async_smem();
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kStaged]);  // this warp's 32 rows staged
                if (copier) {
                    // all 128 rows staged (bounded wait; the other warps do not
                    // wait here); the other CTA's half arrives in this phase
                    w.code = kErrBwdWait + 0xc4;
                    if (!mbar_wait(&bars[kStaged], n & 1, w)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bars[kDsIn], kBox);
                    bulk_copy_to_cluster(ds_peer_rows, smem + Cfg::kOffDSx, kBox, ds_peer_bar);
                }
                if (lane == 0) mbar_arrive_cluster(bar_ds);
            }
        }
        // the copy into this CTA must have landed before either CTA exits
        if (copier && n > 0) mbar_wait_drain(&bars[kDsIn], (n - 1) & 1);
    }
    else if (warp >= 8) {
        // ------------------------------------------------------------ dQ drain + dK/dV epilogue
        // This CTA's 64 queries of dQ_i: warps 8-9 hold d [0,64), warps 10-11
        // d [64,128) (lanes 0-63 and 64-127 of the M = 128 pair result), each
        // warp 32 query rows.  Each warp stages its rows as two 32 x 32 fp32
        // tiles (128B-swizzled, 4 KB of its own) and adds them into the
        // accumulator by TMA bulk reductions.
        const int quarter = warp & 3;
        const int half = quarter >> 1;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0xd0};
        uint32_t n = 0, nunit = 0;
        bool ok = true;
        const uint32_t bar_dqe = lead(kDqEmpty), bar_dkdve = lead(kDkdvEmpty);
        for (int it = 0; ok; ++it) {
            PUnit un;
            if (!punit_at(it, U, nP, un)) break;
            if (un.p < 0) continue;
            const int b = un.bh / H, h = un.bh % H;
            const int j = 2 * un.p + static_cast<int>(rank);
            const int i0 = args.causal ? 2 * un.p : 0;
            for (int i = i0; i < nT; ++i, ++n) {
                w.code = kErrBwdWait + 0xd0;
                if (!mbar_wait(&bars[kDqFull], n & 1, w)) { ok = false; break; }
                tc_fence_after();
                uint32_t acc[64];
                tmem_ld32(tmem + Cfg::kTdQ + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&acc[0]));
                tmem_ld32(tmem + Cfg::kTdQ + lane_off + 32,
                          *reinterpret_cast<uint32_t(*)[32]>(&acc[32]));
                tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&acc[0]));
                tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&acc[32]));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(bar_dqe);
                // this warp's 32 query rows, its 64 columns in two 32 x 32
                // tiles, staged in its own 4 KB and reduced on its own
                const int q0 = i * kBlk + 64 * static_cast<int>(rank) + (quarter & 1) * 32;
                uint8_t *buf = smem + Cfg::kOffRed + quarter * 4096;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (lane == 0) bulk_wait_read<0>();  // the previous reduction has read buf
                    __syncwarp();
                    uint8_t *row = buf + lane * 128;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<uint4 *>(row + ((k ^ (lane & 7)) << 4)) =
                            make_uint4(acc[t * 32 + 4 * k], acc[t * 32 + 4 * k + 1],
                                       acc[t * 32 + 4 * k + 2], acc[t * 32 + 4 * k + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && !*abort_flag) {
                        tma_reduce_add_3d(&args.tm_dqacc, buf, half * 64 + 32 * t, q0, un.bh);
                        bulk_commit();
                    }
                }
            }
            if (!ok) break;
            w.code = kErrBwdWait + 0xd1;
            if (!mbar_wait(&bars[kDkdvFull], nunit & 1, w)) { ok = false; break; }
            ++nunit;
            tc_fence_after();
            const int r = quarter * 32 + lane;  // key row (TMEM lane)
            const int key = j * kBlk + r;
            const size_t orow = ((static_cast<size_t>(b) * S + key) * H + h) * kD;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t tsrc = tmem + lane_off + (which ? Cfg::kTdK : Cfg::kTdV);
                const float mul = which ? args.scale : 1.f;
                uint16_t *out = reinterpret_cast<uint16_t *>(which ? args.dk : args.dv) + orow;
#pragma unroll 1
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tsrc + c * 32, v);
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
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(bar_dkdve);
        }
        if (lane == 0) bulk_wait<0>();  // every drain warp's reductions have read shared memory
    }

    // neither CTA leaves (or releases Tensor Memory) while the other may still
    // touch its shared memory, barriers or Tensor Memory
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, Cfg::kTmemCols);
}

}  // namespace

cudaError_t launch_bwd_main_pair(const BwdArgs &a, cudaStream_t stream) {
    if (a.D != kD) return cudaErrorNotSupported;
    auto kern = fa_bwd_pair_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairCfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long nT = (a.S + kBlk - 1) / kBlk;
    const long long U = static_cast<long long>(a.B) * a.H * ((nT + 1) / 2);
    // pairs that can be resident at once (two SMs of a TPC each)
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
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
