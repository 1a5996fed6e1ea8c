// fa_fwd.cu -- fused attention forward for sm_103a (tcgen05 + TMA).
//
// Computes O = softmax(scale * Q K^T [+ causal mask]) V and the per-row
// log-sum-exp, exactly (hyper.ai story on FlashAttention-4: faster without
// changing the mathematical result).
//
// Design, after "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design
// for Asymmetric Hardware Scaling" (gist.science/nl), Technische samenvatting:
//   Methodologie §1  S = Q K^T and O += P V are asynchronous tcgen05 MMAs
//                    whose accumulators live in Tensor Memory; 128x128 tiles;
//                    the softmax of one query tile runs while the tensor core
//                    works on the other ("ping-pong").
//   Methodologie §2  2^x is split between MUFU.EX2 and an FMA polynomial.
// and "FlashAttention-4: Der neue Rennwagen ..." (gist.science/de) §3: the
// rescale of O is skipped unless the running maximum grew past a threshold.
// Causal work is visited longest-first (hyper.ai story: LPT scheduling).
//
// CTA layout (384 threads = 3 warpgroups, one CTA per SM, persistent over
// work units):
//   warp 0       TMA producer: Q tile pair, then K_j / V_j into a ring of
//                shared-memory slots guarded by full/empty mbarriers (at
//                D = 128 one barrier pair per group of slots {V_j, K_j+1}).
//   warp 1       TMEM allocator and MMA issuer (one elected lane).
//   warps 2-3    idle (they complete warpgroup 0).
//   warps 4-7    softmax + epilogue of query tile 0.
//   warps 8-11   softmax + epilogue of query tile 1.
// A warp may only touch TMEM lanes 32*(warp%4) .. +31, so each warpgroup
// covers the 128 lanes (= query rows) of its tile.  Each SM sub-partition
// holds three warps (one of each warpgroup), so a thread gets 168 registers.
// A work unit is (batch b, head h, 256 query rows = two 128-row tiles).
//
// Tensor Memory (512 columns x 128 lanes x 32 bit):
//   [0,128)      S of tile 0; P (bf16 pairs) overwrites its first 64 columns
//   [128,256)    S / P of tile 1
//   [256,256+D)  O of tile 0;  [256+D, 256+2D) O of tile 1
// The MMA warp issues, per key tile j:  PV0(j), S0(j+1), PV1(j), S1(j+1).
// tcgen05.mma instructions from one thread execute in issue order, so S(j+1)
// overwrites the P(j) it aliases only after PV(j) has read it, and the
// commit that signals S(j+1) also covers PV(j) (so the softmax may rescale O).
//
// D = 256 (one query tile; O takes columns 256-511): S alternates between two
// buffers, [0,128) and [128,256), and the MMA warp issues S(j+1) as soon as
// K(j+1) is in, before it waits for P(j); then PV(j).  The tensor core works
// on S(j+1) while the softmax of tile j runs.  K (in head-dim halves) and V
// (in key halves) stream through one ring of five 32 KB half-slots in the
// order the MMAs read them, S(j+1)'s two halves then PV(j)'s two halves, so
// every load can start about a key tile before it is read.  A rescale of O
// waits for PV(j-1), which the commit of S(j+1) no longer covers.
#include "fa_common.cuh"
#include "sm100_ptx.cuh"
#include "exp2_poly.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // keys per tile
constexpr int kBox = 16384;   // one TMA box: 128 rows x 64 bf16 (128 B), 128B swizzle
constexpr int kWarpStage = 4096;  // one warp's O staging: 32 rows x 64 bf16, 128B swizzle

template <int D>
struct FwdCfg {
    static constexpr int kBoxes = D / 64;                // TMA boxes per 128-row tile
    static constexpr int kTileBytes = kBox * kBoxes;     // 128 x D bf16
    // query tiles per CTA: two ping-pong tiles, except at D = 256 where two O
    // accumulators (2 x 256 columns) and two S tiles exceed Tensor Memory
    static constexpr int kNQ = (D == 256) ? 1 : 2;
    static constexpr int kRows = kBlockM * kNQ;          // query rows per work unit
    static constexpr int kStages = (D == 64) ? 8 : (D == 128 ? 4 : 2);  // ring slots
    // At D = 128 the slots are used in groups of two, {V_j, K_j+1}, each group
    // with one full and one empty barrier (kv_full/kv_empty[g]): fewer waits
    // and commits for the MMA thread.  At D = 64 the softmax, not the MMA
    // issue, sets the pace, and single slots measured faster.
    static constexpr bool kGrouped = (D == 128);
    static constexpr int kGroups = kStages / 2;
    static constexpr int kQBytes = kNQ * kTileBytes;
    static constexpr int kRingOff = kQBytes;
    // D = 256: five 32 KB half-slots at kRingOff, each holding half of a K
    // tile's head dim (S's K steps 0-7 read the first half, 8-15 the second)
    // or half of a V tile's keys (PV's K steps 0-3 / 4-7).  Other head dims:
    // kStages whole-tile slots.
    static constexpr int kHalfSlots = 5;
    static constexpr int kRingBytes = (D == 256) ? kHalfSlots * (kTileBytes / 2) : kStages * kTileBytes;
    // Epilogue staging: 4 KB per softmax warp (its 32 rows x 64 columns of O
    // in bf16, the TMA box layout), from which O leaves by TMA stores.
    // D = 256: none (no room beside Q and the ring; direct stores).
    static constexpr bool kTmaEpilogue = (D != 256);
    static constexpr int kStageOff = kRingOff + kRingBytes;
    static constexpr int kBarOff = kStageOff + (kTmaEpilogue ? 8 * kWarpStage : 0);
    // q_full, q_empty, full[S], empty[S], s_full[2], p_full[2], o_full[2], drain,
    // pv_done, hs_full[5], hs_empty[5]
    static constexpr int kNumBars = 2 + 2 * kStages + 18;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
};

struct Unit {
    int bh;  // b * H + h
    int p;   // query rows [256p, 256p + 256); -1: no unit for this CTA this round
};

// Work-unit order; CTAs take units in a serpentine round-robin.  Without a
// mask every unit has the same work and units are numbered head by head, so
// the CTAs running at once share a few heads' K and V in L2 (with the head
// index fastest and more heads than CTAs, every CTA streamed its own K/V
// from DRAM: 718 against 1135 TFLOPS at D = 256, B = 16, H = 16, S = 1024).
// Under a causal mask units are numbered longest-first (p descending, the
// order of decreasing work) with the head index fastest, which balances the
// triangular work like an LPT list schedule; with many heads, within groups
// of gs heads (gs = BH: one group).  Returns false when the CTA has no
// further rounds.
__device__ __forceinline__ bool unit_at(int it, int U, int BH, int P, bool head_major, int gs, Unit &out) {
    const int G = gridDim.x;
    const int base = it * G;
    if (base >= U) return false;
    const int c = (it & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    const int u = base + c;
    if (u >= U) {
        out.p = -1;
        return true;
    }
    if (head_major) {  // without a mask every unit has the same work
        out.bh = u / P;
        out.p = u % P;
    } else {
        // longest-first within groups of gs heads (gs = BH: over all heads)
        const int grp = u / (gs * P), r = u - grp * gs * P;
        const int ge = min(gs, BH - grp * gs);  // heads in this (possibly last) group
        out.bh = grp * gs + r % ge;
        out.p = P - 1 - r / ge;
    }
    return true;
}

// S = Q K^T for one 128x128 tile: both operands K-major (head dim contiguous).
template <int D>
// The descriptors are built once per call; a K step only adds its byte offset
// / 16 to the start-address field (one add per operand), which keeps the single
// issuing thread ahead of the tensor core.
__device__ __forceinline__ void issue_qk(uint32_t tS, uint32_t q_saddr, uint32_t k_saddr) {
    const uint64_t qd = sdesc_sw128(q_saddr, 16, 1024), kd = sdesc_sw128(k_saddr, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off16 = ((kk / 4) * kBox + (kk % 4) * 32) >> 4;
        mma_ss(tS, qd + off16, kd + off16, FwdCfg<D>::kIdescS, kk > 0 ? 1u : 0u);
    }
}

// Half of S = Q K^T at D = 256: K steps [8 half, 8 half + 8), i.e. head-dim
// columns [128 half, 128 half + 128), with that half of K in its own 32 KB
// half-slot (two TMA boxes).
__device__ __forceinline__ void issue_qk_half(uint32_t tS, uint32_t q_saddr, uint32_t kh_saddr, int half) {
    const uint64_t qd = sdesc_sw128(q_saddr + half * 2 * kBox, 16, 1024), kd = sdesc_sw128(kh_saddr, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off16 = ((kk / 4) * kBox + (kk % 4) * 32) >> 4;
        mma_ss(tS, qd + off16, kd + off16, FwdCfg<256>::kIdescS, (half > 0 || kk > 0) ? 1u : 0u);
    }
}

// Half of O += P V at D = 256: keys [64 half, 64 half + 64) (K steps 4 half ..
// 4 half + 3), that half of V in a 32 KB half-slot as four 64-row boxes, one
// per 64 head-dim columns (MN-major, 8 KB apart).
__device__ __forceinline__ void issue_pv_half(uint32_t tO, uint32_t tP, uint32_t vh_saddr, int half, bool acc) {
    const uint64_t vd = sdesc_sw128(vh_saddr, kBox / 2, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ts(tO, tP + (4 * half + kk) * 8, vd + ((kk * 2048) >> 4), FwdCfg<256>::kIdescPV,
               (acc || kk > 0) ? 1u : 0u);
}

// O (+)= P V: P from TMEM, V MN-major (head dim contiguous, keys along K).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint32_t v_saddr, bool acc) {
    const uint64_t vd = sdesc_sw128(v_saddr, kBox, 1024);
#pragma unroll
    for (int kk = 0; kk < kBlockN / 16; ++kk)
        mma_ts(tO, tP + kk * 8, vd + ((kk * 2048) >> 4), FwdCfg<D>::kIdescPV,
               (acc || kk > 0) ? 1u : 0u);
}

// POLY_PER8: columns of every 8 whose exp2 takes the FMA polynomial;
// POLY_DEG: that polynomial's degree (3 or 5)
template <int D, int POLY_PER8, int POLY_DEG>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_kernel(const __grid_constant__ FwdArgs args) {
    using Cfg = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kBarOff);
    uint64_t *q_full = bars + 0;
    uint64_t *q_empty = bars + 1;
    uint64_t *kv_full = bars + 2;
    uint64_t *kv_empty = bars + 2 + Cfg::kStages;
    uint64_t *s_full = bars + 2 + 2 * Cfg::kStages;
    uint64_t *p_full = s_full + 2;
    uint64_t *o_full = s_full + 4;
    uint64_t *drain = s_full + 6;
    uint64_t *pv_done = s_full + 7;     // D = 256: a PV MMA completed
    uint64_t *hs_full = s_full + 8;     // D = 256: [5] K/V half-slots
    uint64_t *hs_empty = s_full + 13;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + Cfg::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = args.H, S = args.S;
    const int BH = args.B * H;
    const int P = (S + Cfg::kRows - 1) / Cfg::kRows;  // S: the longest sequence if packed
    const int U = BH * P;
    // causal order: longest-first over all heads, unless more heads than half
    // the grid would run at once with their K/V above the L2 size (128 MB);
    // then longest-first within groups of half a grid of heads (D = 256, B = 16,
    // H = 16, S = 1024: 568 -> 670 TFLOPS)
    const long long kv_bytes = static_cast<long long>(min(BH, static_cast<int>(gridDim.x))) * S * D * 4;
    const int gs = (2 * BH > static_cast<int>(gridDim.x) && kv_bytes > (128ll << 20))
                       ? max(1, static_cast<int>(gridDim.x) / 2) : BH;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < Cfg::kStages; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 128);
            mbar_init(&o_full[t], 1);
        }
        mbar_init(drain, 1);
        mbar_init(pv_done, 1);
        for (int i = 0; i < 5; ++i) {
            mbar_init(&hs_full[i], 1);
            mbar_init(&hs_empty[i], 1);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, Cfg::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&args.tm_q);
        tma_prefetch_desc(&args.tm_k);
        tma_prefetch_desc(&args.tm_v);
        if constexpr (D == 256) tma_prefetch_desc(&args.tm_v64);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t smem_base = smem_u32(smem);

    // key tiles visited by query tile 0 / 1 of unit p of a sequence of len rows
    // (with a single query tile, n1 = n0)
    auto tiles_for = [&](int p, int len, int &n0, int &n1) {
        if (args.causal) {
            n0 = min(p * Cfg::kRows + kBlockM - 1, len - 1) / kBlockN + 1;
            n1 = min(p * Cfg::kRows + Cfg::kNQ * kBlockM - 1, len - 1) / kBlockN + 1;
        } else {
            n0 = n1 = (len + kBlockN - 1) / kBlockN;
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            WaitCtx w{abort_flag, args.err_word, kErrFwdWait + 1};
            uint32_t ring = 0, qi = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                Unit un;
                if (!unit_at(it, U, BH, P, !args.causal, gs, un)) break;
                if (un.p < 0) continue;
                const int b = un.bh / H, h = un.bh % H;
                const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, b);
                if (!sp.ok && un.p == 0 && h == 0) atomicCAS(args.err_word, 0, kErrSeqlens);
                if (un.p * Cfg::kRows >= sp.len) continue;  // past this sequence's end
                int n0, n1;
                tiles_for(un.p, sp.len, n0, n1);
                w.code = kErrFwdWait + 1;
                if (!mbar_wait(q_empty, (qi & 1) ^ 1, w)) { ok = false; break; }
                ++qi;
                mbar_arrive_expect_tx(q_full, Cfg::kQBytes);
                for (int t = 0; t < Cfg::kNQ; ++t)
                    for (int c = 0; c < Cfg::kBoxes; ++c)
                        tma_load_4d(smem + t * Cfg::kTileBytes + c * kBox, &args.tm_q, q_full,
                                    64 * c, h, sp.trow0 + un.p * Cfg::kRows + t * kBlockM, sp.tb);
                if constexpr (Cfg::kGrouped) {
                    // groups {K_0}, then {V_j, K_j+1} for j = 0 .. n1-1: one
                    // full and one empty barrier per group of two slots
                    for (int j = -1; j < n1 && ok; ++j) {
                        const uint32_t g = ring % Cfg::kGroups;
                        w.code = kErrFwdWait + 3;
                        if (!mbar_wait(&kv_empty[g], ((ring / Cfg::kGroups) & 1) ^ 1, w)) {
                            ok = false;
                            break;
                        }
                        const bool has_v = j >= 0, has_k = j + 1 < n1;
                        mbar_arrive_expect_tx(&kv_full[g], Cfg::kTileBytes * ((has_v ? 1 : 0) + (has_k ? 1 : 0)));
                        uint8_t *dst = smem + Cfg::kRingOff + 2 * g * Cfg::kTileBytes;
                        for (int c = 0; c < Cfg::kBoxes; ++c) {
                            if (has_v)
                                tma_load_4d(dst + c * kBox, &args.tm_v, &kv_full[g], 64 * c, h,
                                            sp.trow0 + j * kBlockN, sp.tb);
                            if (has_k)
                                tma_load_4d(dst + Cfg::kTileBytes + c * kBox, &args.tm_k, &kv_full[g],
                                            64 * c, h, sp.trow0 + (j + 1) * kBlockN, sp.tb);
                        }
                        ++ring;
                    }
                } else if constexpr (Cfg::kNQ == 1) {
                    // K in head-dim halves and V in key halves, one ring of
                    // half-slots, in the order the MMAs read them: K_0, then
                    // per key tile j: K_j+1 (if any), V_j; load r goes to
                    // half-slot r % 5
                    constexpr uint32_t kHalf = Cfg::kTileBytes / 2;
                    auto load_half = [&](bool is_v, int j, int half) -> bool {
                        const uint32_t hs = ring % Cfg::kHalfSlots;
                        w.code = kErrFwdWait + 2;
                        if (!mbar_wait(&hs_empty[hs], ((ring / Cfg::kHalfSlots) & 1) ^ 1, w)) return false;
                        mbar_arrive_expect_tx(&hs_full[hs], kHalf);
                        uint8_t *dst = smem + Cfg::kRingOff + hs * kHalf;
                        if (is_v) {
                            for (int c = 0; c < 4; ++c)
                                tma_load_4d(dst + c * (kBox / 2), &args.tm_v64, &hs_full[hs], 64 * c, h,
                                            sp.trow0 + j * kBlockN + 64 * half, sp.tb);
                        } else {
                            for (int c = 0; c < 2; ++c)
                                tma_load_4d(dst + c * kBox, &args.tm_k, &hs_full[hs], 64 * (2 * half + c), h,
                                            sp.trow0 + j * kBlockN, sp.tb);
                        }
                        ++ring;
                        return true;
                    };
                    ok = load_half(false, 0, 0) && load_half(false, 0, 1);
                    for (int j = 0; j < n1 && ok; ++j) {
                        if (j + 1 < n1) ok = load_half(false, j + 1, 0) && load_half(false, j + 1, 1);
                        if (ok) ok = load_half(true, j, 0) && load_half(true, j, 1);

                    }
                } else {
                    for (int j = 0; j < n1 && ok; ++j) {
                        for (int which = 0; which < 2; ++which) {
                            const uint32_t slot = ring % Cfg::kStages;
                            w.code = kErrFwdWait + 2;
                            if (!mbar_wait(&kv_empty[slot], ((ring / Cfg::kStages) & 1) ^ 1, w)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&kv_full[slot], Cfg::kTileBytes);
                            uint8_t *dst = smem + Cfg::kRingOff + slot * Cfg::kTileBytes;
                            const CUtensorMap *map = which ? &args.tm_v : &args.tm_k;
                            for (int c = 0; c < Cfg::kBoxes; ++c)
                                tma_load_4d(dst + c * kBox, map, &kv_full[slot], 64 * c, h,
                                            sp.trow0 + j * kBlockN, sp.tb);
                            ++ring;
                        }
                    }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                if constexpr (Cfg::kNQ == 1) {
                    constexpr uint32_t kH = Cfg::kHalfSlots;
                    for (uint32_t r = ring > kH ? ring - kH : 0; r < ring; ++r)
                        mbar_wait_drain(&hs_full[r % kH], (r / kH) & 1);
                } else {
                    constexpr uint32_t kBufs = Cfg::kGrouped ? Cfg::kGroups : Cfg::kStages;
                    const uint32_t lo = ring > kBufs ? ring - kBufs : 0;
                    for (uint32_t r = lo; r < ring; ++r)
                        mbar_wait_drain(&kv_full[r % kBufs], (r / kBufs) & 1);
                }
                if (qi > 0) mbar_wait_drain(q_full, (qi - 1) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            WaitCtx w{abort_flag, args.err_word, kErrFwdWait + 10};
            uint32_t ring = 0, qi = 0;
            uint32_t pph0 = 0, pph1 = 0;
            uint32_t g = 0, kc = 0;  // D = 256: tiles, half-slot loads consumed
            const uint32_t tS0 = tmem, tS1 = tmem + 128;
            const uint32_t tO0 = tmem + 256, tO1 = tmem + 256 + D;
            const uint32_t q0 = smem_base, q1 = smem_base + Cfg::kTileBytes;
            const uint32_t ring_base = smem_base + Cfg::kRingOff;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                Unit un;
                if (!unit_at(it, U, BH, P, !args.causal, gs, un)) break;
                if (un.p < 0) continue;
                const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, un.bh / H);
                if (un.p * Cfg::kRows >= sp.len) continue;
                int n0, n1;
                tiles_for(un.p, sp.len, n0, n1);
                w.code = kErrFwdWait + 10;
                if (!mbar_wait(q_full, qi & 1, w)) { ok = false; break; }
                ++qi;
                if constexpr (Cfg::kGrouped) {
                    // tcgen05.mma issue returns only when the pipe takes the
                    // MMA, so the pipe has next to nothing queued when the
                    // thread stops issuing: every wait or commit between two
                    // MMA groups idles it for its whole length (measured: a
                    // 64-cycle gap costs about 56).  Per key tile this issues
                    // [wait group, wait P0] PV0 S0 [commit, wait P1] PV1 S1
                    // [commit].  Groups are released by the softmax of tile 1
                    // (S1(j+1), or S1(0) for {K_0}, done: the group's last reader).
                    uint32_t g = ring % Cfg::kGroups;
                    w.code = kErrFwdWait + 11;
                    if (!mbar_wait(&kv_full[g], (ring / Cfg::kGroups) & 1, w)) { ok = false; break; }
                    ++ring;
                    tc_fence_after();
                    uint32_t kaddr = ring_base + (2 * g + 1) * Cfg::kTileBytes;
                    issue_qk<D>(tS0, q0, kaddr);
                    mma_commit(&s_full[0]);
                    issue_qk<D>(tS1, q1, kaddr);
                    mma_commit(&s_full[1]);
                    // Q is read only by the S MMAs: once the unit's last one is
                    // issued, the next unit's Q may load (its latency then
                    // overlaps this unit's last key tile and epilogue)
                    if (n1 == 1) mma_commit(q_empty);
                    for (int j = 0; j < n1; ++j) {
                        g = ring % Cfg::kGroups;
                        w.code = kErrFwdWait + 12;
                        if (!mbar_wait(&kv_full[g], (ring / Cfg::kGroups) & 1, w)) { ok = false; break; }
                        ++ring;
                        const uint32_t vaddr = ring_base + 2 * g * Cfg::kTileBytes;
                        kaddr = vaddr + Cfg::kTileBytes;
                        if (j < n0) {
                            w.code = kErrFwdWait + 13;
                            if (!mbar_wait(&p_full[0], pph0, w)) { ok = false; break; }
                            pph0 ^= 1;
                            tc_fence_after();
                            issue_pv<D>(tO0, tS0, vaddr, j > 0);
                            if (j + 1 < n0) {
                                issue_qk<D>(tS0, q0, kaddr);
                                mma_commit(&s_full[0]);
                            } else {
                                mma_commit(&o_full[0]);
                            }
                        }
                        w.code = kErrFwdWait + 15;
                        if (!mbar_wait(&p_full[1], pph1, w)) { ok = false; break; }
                        pph1 ^= 1;
                        tc_fence_after();
                        issue_pv<D>(tO1, tS1, vaddr, j > 0);
                        if (j + 1 < n1) {
                            issue_qk<D>(tS1, q1, kaddr);
                            mma_commit(&s_full[1]);
                            if (j + 2 == n1) mma_commit(q_empty);  // the last S MMA
                        } else {
                            mma_commit(&o_full[1]);
                        }
                    }
                } else if constexpr (Cfg::kNQ == 1) {
                    // S(j+1) into the other S buffer as soon as K(j+1) is in,
                    // then [wait V(j), P(j)] PV(j).  Buffer and phase of tile
                    // g (counted over the CTA's units): g & 1, (g >> 1) & 1.
                    // S of tile buffer b: two halves of K steps, then PV(j):
                    // two halves of keys, each behind its own half-slot's
                    // barrier and released by the commit after its MMAs
                    constexpr uint32_t kHalf = Cfg::kTileBytes / 2;
                    auto next_half = [&](uint32_t &addr) -> bool {
                        const uint32_t hs = kc % Cfg::kHalfSlots;
                        w.code = kErrFwdWait + 14;
                        if (!mbar_wait(&hs_full[hs], (kc / Cfg::kHalfSlots) & 1, w)) return false;
                        ++kc;
                        tc_fence_after();
                        addr = ring_base + hs * kHalf;
                        return true;
                    };
                    auto release_half = [&](uint32_t addr) {
                        mma_commit(&hs_empty[(addr - ring_base) / kHalf]);
                    };
                    auto issue_s = [&](uint32_t b) -> bool {
                        for (int half = 0; half < 2; ++half) {
                            uint32_t ka;
                            if (!next_half(ka)) return false;
                            issue_qk_half(tmem + b * 128, q0, ka, half);
                            release_half(ka);
                        }
                        mma_commit(&s_full[b]);
                        return true;
                    };
                    if (!issue_s(g & 1)) { ok = false; break; }
                    if (n0 == 1) mma_commit(q_empty);
                    for (int j = 0; j < n0; ++j, ++g) {
                        if (j + 1 < n0) {
                            if (!issue_s((g + 1) & 1)) { ok = false; break; }
                            if (j + 2 == n0) mma_commit(q_empty);  // the last S MMA
                        }
                        w.code = kErrFwdWait + 13;
                        if (!mbar_wait(&p_full[g & 1], (g >> 1) & 1, w)) { ok = false; break; }
                        for (int half = 0; half < 2 && ok; ++half) {
                            uint32_t va;
                            if (!next_half(va)) { ok = false; break; }
                            issue_pv_half(tO0, tmem + (g & 1) * 128, va, half, j > 0 || half > 0);
                            release_half(va);
                        }
                        if (!ok) break;
                        mma_commit(pv_done);
                        if (j + 1 == n0) mma_commit(&o_full[0]);
                    }
                } else {
                    // K_j and V_j in single slots, each with its own barriers
                    const uint32_t kslot = ring % Cfg::kStages;
                    w.code = kErrFwdWait + 11;
                    if (!mbar_wait(&kv_full[kslot], (ring / Cfg::kStages) & 1, w)) { ok = false; break; }
                    ++ring;
                    tc_fence_after();
                    issue_qk<D>(tS0, q0, ring_base + kslot * Cfg::kTileBytes);
                    mma_commit(&s_full[0]);
                    issue_qk<D>(tS1, q1, ring_base + kslot * Cfg::kTileBytes);
                    mma_commit(&s_full[1]);
                    mma_commit(&kv_empty[kslot]);
                    // Q is read only by the S MMAs (see the grouped path)
                    if (n1 == 1) mma_commit(q_empty);
                    for (int j = 0; j < n1; ++j) {
                        const uint32_t vslot = ring % Cfg::kStages;
                        w.code = kErrFwdWait + 12;
                        if (!mbar_wait(&kv_full[vslot], (ring / Cfg::kStages) & 1, w)) { ok = false; break; }
                        ++ring;
                        const bool has_next = (j + 1 < n1);
                        uint32_t nslot = 0, nphase = 0;
                        if (has_next) {
                            nslot = ring % Cfg::kStages;
                            nphase = (ring / Cfg::kStages) & 1;
                            ++ring;
                        }
                        const uint32_t vaddr = ring_base + vslot * Cfg::kTileBytes;
                        const uint32_t naddr = ring_base + nslot * Cfg::kTileBytes;
                        bool next_ready = false;
                        if (j < n0) {
                            w.code = kErrFwdWait + 13;
                            if (!mbar_wait(&p_full[0], pph0, w)) { ok = false; break; }
                            pph0 ^= 1;
                            tc_fence_after();
                            issue_pv<D>(tO0, tS0, vaddr, j > 0);
                            if (j + 1 < n0) {
                                w.code = kErrFwdWait + 14;
                                if (!mbar_wait(&kv_full[nslot], nphase, w)) { ok = false; break; }
                                next_ready = true;
                                tc_fence_after();
                                issue_qk<D>(tS0, q0, naddr);
                                mma_commit(&s_full[0]);
                            } else {
                                mma_commit(&o_full[0]);
                            }
                        }
                        w.code = kErrFwdWait + 15;
                        if (!mbar_wait(&p_full[1], pph1, w)) { ok = false; break; }
                        pph1 ^= 1;
                        tc_fence_after();
                        issue_pv<D>(tO1, tS1, vaddr, j > 0);
                        mma_commit(&kv_empty[vslot]);
                        if (has_next) {
                            if (!next_ready) {
                                w.code = kErrFwdWait + 16;
                                if (!mbar_wait(&kv_full[nslot], nphase, w)) { ok = false; break; }
                                tc_fence_after();
                            }
                            issue_qk<D>(tS1, q1, naddr);
                            mma_commit(&s_full[1]);
                            mma_commit(&kv_empty[nslot]);
                            if (j + 2 == n1) mma_commit(q_empty);  // the last S MMA
                        } else {
                            mma_commit(&o_full[1]);
                        }
                    }
                }
            }
            // every MMA issued must have finished before TMEM is released
            mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax + epilogue
        const int t = (warp - 4) >> 2;  // query tile of this warpgroup (idle if t >= kNQ)
        const int quarter = warp & 3;   // TMEM lane quarter this warp may access
        const int r_in_tile = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tO = tmem + 256 + t * D + lane_off;
        const float c2 = args.scale_log2;
        const float tau = args.rescale_threshold;
        WaitCtx w{abort_flag, args.err_word, kErrFwdWait + 20 + t};
        uint32_t sph = 0, oph = 0;
        uint32_t g = 0;  // D = 256: tiles processed; tile g uses S buffer g & 1
        bool ok = (t < Cfg::kNQ);
        // With grouped K/V slots one thread of tile 1 frees each group: S1(j)
        // complete means the MMAs of key tile j-1 (PV0, S0(j), PV1) are done
        // too, since one thread issues them in order; O1 complete frees the
        // unit's last group.
        const bool releaser = Cfg::kGrouped && t == 1 && r_in_tile == 0;
        uint32_t grp = 0;
        for (int it = 0; ok; ++it) {
            Unit un;
            if (!unit_at(it, U, BH, P, !args.causal, gs, un)) break;
            if (un.p < 0) continue;
            const int b = un.bh / H, h = un.bh % H;
            const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, b);
            if (un.p * Cfg::kRows >= sp.len) continue;
            const int len = sp.len;
            int n0, n1;
            tiles_for(un.p, len, n0, n1);
            const int n = t ? n1 : n0;
            const int row = un.p * Cfg::kRows + t * kBlockM + r_in_tile;
            float m_used = -INFINITY;  // reference maximum, log2 units of scaled scores
            float l = 0.f;             // running row sum relative to m_used
            for (int j = 0; j < n; ++j, ++g) {
                // this tile's S buffer and the phase of its barriers
                const int buf = (Cfg::kNQ == 1) ? static_cast<int>(g & 1) : t;
                const uint32_t spar = (Cfg::kNQ == 1) ? ((g >> 1) & 1) : sph;
                const uint32_t tS = tmem + buf * 128 + lane_off;
                if (!mbar_wait(&s_full[buf], spar, w)) { ok = false; break; }
                if (releaser) mbar_arrive(&kv_empty[grp++ % Cfg::kGroups]);
                sph ^= 1;
                tc_fence_after();
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
                if (j == n - 1) {
                    // last tile of the row: keys past S and, if causal, past the row
                    const int lim = (args.causal ? min(row, len - 1) : len - 1) - j * kBlockN;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (c * 32 + e > lim) sr[c][e] = __float_as_uint(-INFINITY);
                }
                // row maximum: four independent chains of 3-input max
                float mx[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    mx[c] = fmax3(__uint_as_float(sr[c][0]), __uint_as_float(sr[c][1]),
                                  __uint_as_float(sr[c][2]));
#pragma unroll
                    for (int e = 3; e < 31; e += 2)
                        mx[c] = fmax3(mx[c], __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
                    mx[c] = fmaxf(mx[c], __uint_as_float(sr[c][31]));
                }
                const float m_tile = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * c2;
                const float m_new = fmaxf(m_used, m_tile);
                if (__any_sync(0xffffffffu, m_new > m_used + tau)) {
                    // conditional rescale: move the reference maximum to m_new
                    const float alpha = ex2_mufu(m_used - m_new);
                    l *= alpha;
                    if (j > 0) {
                        if constexpr (Cfg::kNQ == 1) {
                            // S(j) was issued before PV(j-1): wait for that PV
                            if (!mbar_wait(pv_done, (g - 1) & 1, w)) { ok = false; break; }
                            tc_fence_after();
                        }
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t orr[32];
                            tmem_ld32(tO + c * 32, orr);
                            tmem_ld_wait(orr);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                            tmem_st32(tO + c * 32, orr);
                        }
                    }
                    m_used = m_new;
                }
                // p = 2^(s*c2 - m_used): in every group of 8 columns the last
                // POLY_PER8 go to the FMA polynomial (degree POLY_DEG), the rest
                // to MUFU, so both units work at once; arguments and row sums
                // use two-lane fp32
                const float2 c2v = make_float2(c2, c2);
                const float2 nmv = make_float2(-m_used, -m_used);
                float2 lsum[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 xv = fma2(make_float2(__uint_as_float(sr[c][e]),
                                                           __uint_as_float(sr[c][e + 1])),
                                               c2v, nmv);
                        // columns e, e+1 of their group of 8 (both lanes, the
                        // odd one only, or neither take the polynomial)
                        constexpr int kFirstPoly = 8 - POLY_PER8;
                        float2 pv;
                        if ((e & 7) >= kFirstPoly) {
                            pv = exp2_poly_x2<POLY_DEG>(xv);
                        } else if (((e + 1) & 7) >= kFirstPoly) {
                            pv.x = ex2_mufu(xv.x);
                            pv.y = exp2_poly<POLY_DEG>(xv.y);
                        } else {
                            pv.x = ex2_mufu(xv.x);
                            pv.y = ex2_mufu(xv.y);
                        }
                        acc = add2(acc, pv);
                        pk[e >> 1] = pack_bf16x2(pv.x, pv.y);
                    }
                    lsum[c] = acc;
                    // P columns [16c, 16c+16) hold keys [32c, 32c+32); they
                    // overwrite S columns whose values are already in registers
                    tmem_st16(tS + c * 16, pk);
                }
                const float2 ls = add2(add2(lsum[0], lsum[1]), add2(lsum[2], lsum[3]));
                l += ls.x + ls.y;
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&p_full[buf]);
            }
            if (!ok) break;
            // ---- epilogue: O / l -> bf16, LSE
            if (!mbar_wait(&o_full[t], oph, w)) { ok = false; break; }
            if (releaser) mbar_arrive(&kv_empty[grp++ % Cfg::kGroups]);
            oph ^= 1;
            tc_fence_after();
            const float inv_l = 1.f / l;
            const int tile_row0 = un.p * Cfg::kRows + t * kBlockM;
            uint16_t *orow = reinterpret_cast<uint16_t *>(args.o) +
                             ((static_cast<size_t>(sp.tok0) + row) * H + h) * D;
            if constexpr (Cfg::kTmaEpilogue) {
                // Each warp writes its own 32 rows of O: 64 columns at a time
                // into its 4 KB of the staging area (the TMA box layout, 128B
                // swizzle), then one TMA store per 64 columns issued by its lane
                // 0.  No warp waits for another, and the last store's read of
                // shared memory is waited for only before the region is written
                // again (the next 64 columns, or the next unit).  A warp whose
                // rows run past a packed sequence's end would overwrite the next
                // sequence's rows: it keeps direct stores.
                const int wrow0 = tile_row0 + quarter * 32;  // this warp's first row
                const bool use_tma = !args.cu_seqlens || wrow0 + 32 <= len;
                uint8_t *stg = smem + Cfg::kStageOff + (t * 4 + quarter) * kWarpStage;
                uint8_t *srow = stg + lane * 128;
#pragma unroll 1
                for (int hc = 0; hc < D / 64; ++hc) {
                    uint32_t orr[2][32];
                    tmem_ld32(tO + hc * 64, orr[0]);
                    tmem_ld32(tO + hc * 64 + 32, orr[1]);
                    tmem_ld_wait(orr[0]);
                    tmem_ld_wait(orr[1]);
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(orr[e >> 4][2 * (e & 15)]) * inv_l,
                                            __uint_as_float(orr[e >> 4][2 * (e & 15) + 1]) * inv_l);
                    if (use_tma) {
                        if (lane == 0) bulk_wait_read<0>();  // this region's last store has read it
                        __syncwarp();
                        // row `lane` of the box: 16-byte chunk k at (k ^ (lane % 8)) * 16
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            *reinterpret_cast<uint4 *>(srow + ((k ^ (lane & 7)) << 4)) =
                                make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_4d(&args.tm_o, stg, 64 * hc, h, sp.trow0 + wrow0, sp.tb);
                            bulk_commit();
                        }
                    } else if (row < len) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + hc * 64);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(tO + c * 32, orr);
                    tmem_ld_wait(orr);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(orr[2 * e]) * inv_l,
                                            __uint_as_float(orr[2 * e + 1]) * inv_l);
                    if (row < len) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2],
                                                 pk[4 * v4 + 3]);
                    }
                }
            }
            if (row < len)
                args.lse[stat_index(args.cu_seqlens, args.T, S, H, b, h, sp, row)] =
                    (m_used + log2f(l)) * 0.69314718055994531f;
        }
        if (Cfg::kTmaEpilogue && lane == 0) bulk_wait<0>();  // its O stores are complete
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
}

template <int D, int PG, int DEG>
cudaError_t launch_fwd_inst(const FwdArgs &a, cudaStream_t stream) {
    using Cfg = FwdCfg<D>;
    static_assert(Cfg::kSmemBytes <= 232448, "shared memory budget");
    auto kern = fa_fwd_kernel<D, PG, DEG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long P = (a.S + Cfg::kRows - 1) / Cfg::kRows;
    const long long U = static_cast<long long>(a.B) * a.H * P;
    const int grid = static_cast<int>(U < a.num_sms ? U : a.num_sms);
    kern<<<grid, kThreads, Cfg::kSmemBytes, stream>>>(a);
    return cudaGetLastError();
}

template <int D, int DEG>
cudaError_t launch_fwd_deg(const FwdArgs &a, cudaStream_t stream) {
    switch (a.poly_groups) {
        case 1: return launch_fwd_inst<D, 1, DEG>(a, stream);
        case 2: return launch_fwd_inst<D, 2, DEG>(a, stream);
        case 8: return launch_fwd_inst<D, 8, DEG>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t launch_fwd_d(const FwdArgs &a, cudaStream_t stream) {
    if (a.poly_groups == 0) return launch_fwd_inst<D, 0, 3>(a, stream);  // MUFU only
    switch (a.poly_degree) {
        case 3: return launch_fwd_deg<D, 3>(a, stream);
        case 5: return launch_fwd_deg<D, 5>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs &a, cudaStream_t stream) {
    switch (a.D) {
        case 64: return launch_fwd_d<64>(a, stream);
        case 128: return launch_fwd_d<128>(a, stream);
        case 256: return launch_fwd_d<256>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
