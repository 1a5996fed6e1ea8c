// fa_bwd.cu -- fused attention backward for sm_103a (tcgen05 + TMA).
//
// Given Q, K, V, O, dO and LSE, computes dQ, dK, dV of exact softmax
// attention ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling" (gist.science/nl), Technische samenvatting,
// Methodologie §3: the backward pass keeps its intermediates in Tensor Memory
// because shared-memory bandwidth is its bottleneck; dQ is reduced with
// atomic additions in global memory).  With P = exp(scale*S - LSE):
//   Delta_i = dO_i . O_i,   dS = P o (dO V^T - Delta),
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
//
// Three launches:
//   fa_bwd_prep     Delta = rowsum(dO o O) (fp32) and dQ accumulator = 0
//   fa_bwd_kernel   the fused main kernel (below)
//   fa_bwd_dq_cvt   dQ = bf16(scale * accumulator)
//
// Main kernel: persistent, one CTA per SM, a work unit is (b, h, key tile j
// of 128 keys).  K_j and V_j stay in shared memory; 128-query blocks Q_i,
// dO_i stream through.  Everything is computed transposed (keys on the 128
// TMEM lanes), so P^T lands in Tensor Memory exactly where the dV MMA wants
// its A operand, and dS^T in shared memory in the K-major layout of dK's A:
//   S^T  = K_j Q_i^T - LSE/scale   -> X (fp32, 128 cols)  A=K smem, B=Q smem
//   dP^T = V_j dO_i^T - Delta      -> Y (fp32, 128 cols)  A=V smem, B=dO smem
//   P^T = 2^(X scale log2 e) (bf16) over X;  dS^T = P^T o Y (bf16) into
//   shared memory
// The per-query terms -LSE/scale and -Delta enter through one extra K step
// of those two MMAs: A = ones, B = the value as three bf16 terms (exact sum),
// written by the producer next to Q_i and dO_i.  The softmax warps then read
// no per-query statistics from shared memory, whose bandwidth the MMAs need.
//   dV  += P^T dO_i       (TMEM acc, D cols)         A=X tmem,  B=dO smem
//   dQ_i = dS K_j  -> Y   (fp32, queries on lanes)   A=dS smem, B=K smem
//   dK  += dS^T Q_i       (TMEM acc, D cols)         A=dS smem, B=Q smem
// dQ is issued before dK so that the drain of dQ_i out of Y runs while the
// tensor core does dK_i; dP^T(i+1) needs Y back.  (With dS^T in TMEM, dK
// would have to read it from Y before dQ could overwrite it.)
// Tensor Memory: X [0,128) | Y [128,256) | dV [256,256+D) | dK [256+D,256+2D).
// tcgen05.mma from one thread executes in issue order: S(i+1) may overwrite
// X once dV(i) was issued, dQ(i) may overwrite Y once dS(i) was formed.
//
// Warp roles (384 threads):
//   warp 0      TMA producer (K_j/V_j per unit; Q_i + LSE bias rows, dO_i +
//               Delta bias rows per block)
//   warp 1      TMEM allocation + MMA issue (one lane)
//   warps 2-3   idle
//   warps 4-7   "softmax": P^T and dS^T for one 128x128 block (lane = key)
//   warps 8-11  dQ drain (lane = query; TMA bulk reduce-add into the fp32
//               accumulator)
//               and the dK / dV epilogue of each unit
// Causal units are visited longest first (key tile 0 sees every query
// block) in a serpentine order over the CTAs, as in the forward.
#include <cuda_bf16.h>

#include "fa_common.cuh"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr int kBlk = 128;    // keys per unit and queries per block
constexpr int kBox = 16384;  // one TMA box: 128 rows x 64 bf16, 128B swizzle

template <int D>
struct BwdCfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTile = kBox * kBoxes;  // 128 x D bf16
    // shared memory map
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTile;
    static constexpr int kOffQ = kOffV + kTile;      // 2 stages
    static constexpr int kOffDO = kOffQ + 2 * kTile;  // 1 stage
    static constexpr int kOffDS = kOffDO + kTile;     // dS: 128 keys x 128 queries bf16
    static constexpr int kOffRed = kOffDS + 32768;    // dQ staging: 4 warps x 32 x 32 fp32
    // bias K step of S^T and dP^T (no-swizzle K-major, 128 rows x 16 bf16):
    // A = (1, 1, 1, 0, ...) on every row; B = three bf16 terms of -LSE/scale
    // (2 stages, with Q) or of -Delta (1 stage, with dO) per query
    static constexpr int kBias = 4096;
    static constexpr int kOffOnes = kOffRed + 16384;
    static constexpr int kOffLb = kOffOnes + kBias;
    static constexpr int kOffDb = kOffLb + 2 * kBias;
    static constexpr int kOffBar = kOffDb + kBias;
    // kv_full, kv_empty, q_full[2], q_empty[2], do_full, do_empty, s_full, dp_full,
    // p_ready, ds_ready, dq_full, dq_empty, dkdv_full, dv_empty, drain, dk_empty
    static constexpr int kNumBars = 18;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    // no alignment slack: the dynamic shared memory base must be 1024-byte
    // aligned (checked at kernel entry)
    static constexpr int kSmemBytes = kOffMisc + 16;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTX = 0, kTY = 128, kTdV = 256, kTdK = 256 + D;
    static constexpr uint32_t kIdescSS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
    static constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, false, true);    // dV, dK
    static constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, D, true, true);      // dQ
};

__device__ __forceinline__ int nT_of(int U, int BH) { return U / BH; }

struct BUnit {
    int bh;  // b * H + h
    int j;   // key tile; -1 = no unit for this CTA this round
};

// Unit u -> (bh, key tile).  Without a mask the key tiles of one head are
// consecutive (concurrent CTAs share that head's Q, dO and dQ accumulator in
// L2), key tile 0 first.  Under a causal mask tile j has nT - j query blocks,
// and the units are numbered tile-major instead (every head's tile 0, then
// tile 1, ...): with the serpentine rounds that is a longest-first order
// across heads, which balances the CTAs (head by head, the busiest CTA runs
// about 10 % more blocks than the average at S = 32768, H = 16; the
// fixed-order mode went from 572 to 659 TFLOPS).  With more heads than half
// the grid, whose Q, dO and dQ accumulators exceed L2, the atomic-order
// kernel numbers them tile-major within groups of half a grid of heads
// (B = 16, H = 16, S = 2048, D = 128: 541 -> 726 TFLOPS).
__device__ __forceinline__ void unit_coords(int u, int nT, int BH, bool causal, int &bh, int &j) {
    if (causal) {
        j = u / BH;
        bh = u % BH;
    } else {
        bh = u / nT;
        j = u % nT;
    }
}

__device__ __forceinline__ bool bunit_at(int it, int U, int BH, bool causal, BUnit &out, int gs = 0) {
    const int G = gridDim.x;
    const int base = it * G;
    if (base >= U) return false;
    const int c = (it & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    const int u = base + c;
    if (u >= U) {
        out.j = -1;
        return true;
    }
    const int nT = nT_of(U, BH);
    if (causal && gs > 0 && gs < BH) {
        // tile-major within groups of gs heads
        const int grp = u / (gs * nT), r = u - grp * gs * nT;
        const int ge = min(gs, BH - grp * gs);
        out.j = r / ge;
        out.bh = grp * gs + r % ge;
        return true;
    }
    unit_coords(u, nT, BH, causal, out.bh, out.j);
    return true;
}

// first query block a key tile sees (causal: queries >= first key)
__device__ __forceinline__ int first_block(int j, int causal) { return causal ? j : 0; }

// Query block a key tile visits at its step s.  Ascending from the first
// visible block, except in the fixed-order mode without a causal mask, where
// tile j starts at block j (rotated): the tiles that run together then reach
// each block one step apart, which is the order their contributions to it
// are fixed in (dq_position).
__device__ __forceinline__ int block_at(int j, int s, int i0, int nb, bool rotate) {
    return rotate ? (j + s) % nb : i0 + s;
}

// Fixed-order mode without a causal mask: the place of key tile j's
// contribution in the sum of dQ block i (0 = first).  Units are numbered head
// by head (unit u = bh nT + j) and taken in rounds of G by the persistent
// grid; [j0, j1) are the head's tiles in j's round.  Contributions of earlier
// rounds come first; within a round they are ordered by the step at which
// each tile reaches block i, so every wait points to a unit of the same round
// or an earlier one (no cycle), and in the same round to the tile one step
// ahead.
// In a packed batch unit numbers still run over nT (the longest sequence's
// tiles); a sequence has nb <= nT tiles, and its units past them are skipped.
__device__ __forceinline__ int dq_position(int bh, int j, int i, int nT, int nb, int G) {
    const int r = (bh * nT + j) / G;
    const int j0 = min(max(r * G - bh * nT, 0), nb), j1 = min((r + 1) * G - bh * nT, nb);
    // every tile sees every block, reached at step (i - j') mod nb: earlier
    // steps are the tiles in the circular range (j, i]
    auto in_round = [&](int lo, int hi) { return max(0, min(j1, hi) - max(j0, lo)); };
    const int ahead = j < i ? in_round(j + 1, i + 1)
                            : (j > i ? in_round(j + 1, nb) + in_round(0, i + 1) : 0);
    return j0 + ahead;
}

// Fixed-order mode under a causal mask.  Tile lengths differ (tile j visits
// blocks j .. nT-1), so a CTA starts its next unit whenever its current one
// ends, and a fixed order by rounds would make the CTAs that move on early
// wait for the longest tiles.  Instead the order follows the schedule itself:
// counting one step per block, tile j of unit u starts at step start(u) (the
// lengths of the units its CTA ran before, in the persistent grid's
// serpentine order) and reaches block i at step start(u) + i - j.  The
// contributions to block i are summed in the order of that arrival step
// (ties: lower j first), i.e. by key(u) = start(u) - j.  Along one CTA's
// sequence of blocks the arrival step strictly increases, and every wait
// points to a strictly earlier (step, tile), so the waits form no cycle.
// Tiles of sequence bh / H: nT, or fewer in a packed batch (0 for a sequence
// whose offsets are invalid).
__device__ __forceinline__ int seq_tiles(const BwdArgs &args, int bh, int nT) {
    if (!args.cu_seqlens) return nT;
    const SeqSpan sp = seq_span(args.cu_seqlens, args.T, args.S, bh / args.H);
    return (sp.len + kBlk - 1) / kBlk;
}

// Order key of unit u (causal numbering, unit_coords): its start step minus
// its key tile.
__device__ __forceinline__ int causal_order_key(const BwdArgs &args, int u, int U, int nT, int G) {
    const int BH = U / nT;
    const int r = u / G, p = u % G;
    const int c = (r & 1) ? G - 1 - p : p;  // the CTA that runs unit u
    long long start = 0;
    for (int rr = 0; rr < r; ++rr) {
        const int uu = rr * G + ((rr & 1) ? G - 1 - c : c);
        if (uu < U) {
            int bh2, j2;
            unit_coords(uu, nT, BH, true, bh2, j2);
            start += max(seq_tiles(args, bh2, nT) - j2, 0);  // skipped units take no steps
        }
    }
    int bh, j;
    unit_coords(u, nT, BH, true, bh, j);
    return static_cast<int>(start - j);
}

// Rank of tile j among the tiles j' <= i of its head by (key, j'): its place
// in the sum of dQ block i.  All lanes of the warp take part.
__device__ __forceinline__ int causal_rank(const int *keys, int j, int i, int lane) {
    const int kj = keys[j];
    int cnt = 0;
    for (int base = 0; base <= i; base += 32) {
        const int jp = base + lane;
        bool before = false;
        if (jp <= i) {
            const int kp = keys[jp];
            before = kp < kj || (kp == kj && jp < j);
        }
        cnt += __popc(__ballot_sync(0xffffffffu, before));
    }
    return cnt;
}

// ---------------------------------------------------------------- MMA helpers

// Byte offset of element (row r, k) of a no-swizzle K-major 128 x 16 bf16 tile
// (core matrices of 8 rows x 16 bytes, K-direction stride 128, row-group 256).
__host__ __device__ constexpr uint32_t bias_off(int r, int k) {
    return (r / 8) * 256 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2;
}

// First 16 bytes of a bias row: v as three bf16 terms hi + mid + lo (each the
// bf16 rounding of what the previous terms leave; the sum equals v for normal
// fp32 v) in k = 0, 1, 2; an infinite v goes whole into hi.
__device__ __forceinline__ uint4 bias_row(float v) {
    const float hi = __bfloat162float(__float2bfloat16_rn(v));
    if (!isfinite(v)) return make_uint4(pack_bf16x2(hi, 0.f), 0u, 0u, 0u);
    const float r1 = v - hi;
    const float mid = __bfloat162float(__float2bfloat16_rn(r1));
    const float lo = r1 - mid;
    return make_uint4(pack_bf16x2(hi, mid), pack_bf16x2(lo, 0.f), 0u, 0u);
}

// 128x128 (x D) with both operands K-major: S^T = K Q^T, dP^T = V dO^T, plus
// one bias K step that adds B's per-query value (A's ones times its three
// terms) to every key row: S^T - LSE/scale, dP^T - Delta.
// (descriptors built once per call; a K step adds its byte offset / 16)
template <int D>
__device__ __forceinline__ void issue_kmajor(uint32_t tD, uint32_t a_saddr, uint32_t b_saddr,
                                             uint32_t ones_saddr, uint32_t bias_saddr) {
    const uint64_t ad = sdesc_sw128(a_saddr, 16, 1024), bd = sdesc_sw128(b_saddr, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off16 = ((kk / 4) * kBox + (kk % 4) * 32) >> 4;
        mma_ss(tD, ad + off16, bd + off16, BwdCfg<D>::kIdescSS, kk > 0 ? 1u : 0u);
    }
    mma_ss(tD, sdesc_none(ones_saddr, 128, 256), sdesc_none(bias_saddr, 128, 256),
           BwdCfg<D>::kIdescSS, 1u);
}

// acc (+)= A[tmem: 128 keys x 128 queries] * B[smem: 128 queries x D, MN-major]
template <int D>
__device__ __forceinline__ void issue_acc(uint32_t tAcc, uint32_t tA, uint32_t b_saddr, bool acc) {
    const uint64_t bd = sdesc_sw128(b_saddr, kBox, 1024);
#pragma unroll
    for (int kk = 0; kk < kBlk / 16; ++kk)
        mma_ts(tAcc, tA + kk * 8, bd + ((kk * 2048) >> 4), BwdCfg<D>::kIdescAcc,
               (acc || kk > 0) ? 1u : 0u);
}

// dQ = dS K: A = dS (queries x keys, MN-major: rows = keys), B = K (keys x D, MN-major)
template <int D>
__device__ __forceinline__ void issue_dq(uint32_t tD, uint32_t ds_saddr, uint32_t k_saddr) {
    const uint64_t ad = sdesc_sw128(ds_saddr, kBox, 1024), bd = sdesc_sw128(k_saddr, kBox, 1024);
#pragma unroll
    for (int kk = 0; kk < kBlk / 16; ++kk)
        mma_ss(tD, ad + ((kk * 2048) >> 4), bd + ((kk * 2048) >> 4), BwdCfg<D>::kIdescDQ,
               kk > 0 ? 1u : 0u);
}

// dK (+)= dS^T Q with dS^T read from the shared copy the dQ MMA uses: rows =
// keys, queries contiguous in two 64-query boxes, i.e. K-major A (like K in
// S^T); B = Q (queries x D, MN-major)
template <int D>
__device__ __forceinline__ void issue_dk(uint32_t tAcc, uint32_t ds_saddr, uint32_t q_saddr, bool acc) {
    const uint64_t ad = sdesc_sw128(ds_saddr, 16, 1024), bd = sdesc_sw128(q_saddr, kBox, 1024);
#pragma unroll
    for (int kk = 0; kk < kBlk / 16; ++kk) {
        const uint32_t aoff16 = ((kk / 4) * kBox + (kk % 4) * 32) >> 4;
        mma_ss(tAcc, ad + aoff16, bd + ((kk * 2048) >> 4), BwdCfg<D>::kIdescAcc,
               (acc || kk > 0) ? 1u : 0u);
    }
}

// ---------------------------------------------------------------- main kernel

// kDet: the fixed-order dQ mode (args.dq_sem set), a separate instance so
// that the atomic-order kernel carries none of its logic.  kTileMajor: units
// numbered tile-major (unit_coords), the order for causal masks, also a
// separate instance so that the order without a mask keeps its code
template <int D, bool kDet, bool kTileMajor>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_kernel(const __grid_constant__ BwdArgs args) {
    using Cfg = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    if (smem_u32(smem) & 1023u) {  // swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicCAS(args.err_word, 0, kErrBwdWait + 0xff);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint64_t *kv_full = bars + 0, *kv_empty = bars + 1;
    uint64_t *q_full = bars + 2, *q_empty = bars + 4;  // [2] each
    uint64_t *do_full = bars + 6, *do_empty = bars + 7;
    uint64_t *s_full = bars + 8, *dp_full = bars + 9;
    uint64_t *p_ready = bars + 10, *ds_ready = bars + 11;
    uint64_t *dq_full = bars + 12, *dq_empty = bars + 13;
    // dkdv_full: a unit's dV and dK are complete; dv_empty / dk_empty: the drain
    // warps have read the dV / dK accumulator (the next unit may overwrite it)
    uint64_t *dkdv_full = bars + 14, *dv_empty = bars + 15;
    uint64_t *drain = bars + 16, *dk_empty = bars + 17;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = args.H, S = args.S;
    const int BH = args.B * H;
    const int nT = (S + kBlk - 1) / kBlk;  // key tiles = query blocks
    const int U = BH * nT;
    // atomic order under a causal mask with many heads whose Q, dO and dQ
    // accumulator exceed L2: tile-major within groups of half a grid of heads
    // (the fixed-order schedule keeps its own numbering)
    const long long head_bytes = static_cast<long long>(S) * D * 8;
    const int ugs = (!kDet && 2 * BH > static_cast<int>(gridDim.x) &&
                     static_cast<long long>(min(BH, static_cast<int>(gridDim.x))) * head_bytes > (128ll << 20))
                        ? max(1, static_cast<int>(gridDim.x) / 2) : 0;
    const int nSem = 8 * nT;               // deterministic-mode counters per head
    const bool rotate = kDet && !args.causal;  // see block_at

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s2 = 0; s2 < 2; ++s2) {
            mbar_init(&q_full[s2], 2);  // TMA (expect_tx) + LSE bias rows written
            mbar_init(&q_empty[s2], 1);
        }
        mbar_init(do_full, 2);  // TMA (expect_tx) + Delta bias rows written
        mbar_init(do_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(dp_full, 1);
        mbar_init(p_ready, 128);
        mbar_init(ds_ready, 128);
        mbar_init(dq_full, 1);
        mbar_init(dq_empty, 128);
        mbar_init(dkdv_full, 1);
        mbar_init(dv_empty, 128);
        mbar_init(dk_empty, 128);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, Cfg::kTmemCols);
        tmem_relinquish();
    }
    // bias tiles: zero everywhere (the MMA reads all 16 K columns), ones in
    // k = 0, 1, 2 of the A tile
    for (int t = threadIdx.x; t < 4 * Cfg::kBias / 16; t += kThreads)
        reinterpret_cast<uint4 *>(smem + Cfg::kOffOnes)[t] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (threadIdx.x < 128)
        *reinterpret_cast<uint4 *>(smem + Cfg::kOffOnes + bias_off(threadIdx.x, 0)) =
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
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t sbase = smem_u32(smem);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 1};
        uint32_t nunit = 0, nblk = 0;  // units / blocks issued so far
        uint32_t nkv = 0, nq = 0, ndo = 0;  // K/V, Q and dO copies issued (for the unwinding)
        bool ok = true;
        const float inv_scale = 1.f / args.scale;
        for (int it = 0; ok; ++it) {
            BUnit un;
            if (!bunit_at(it, U, BH, kTileMajor, un, ugs)) break;
            if (un.j < 0) continue;
            const int b = un.bh / H, h = un.bh % H;
            const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, b);
            if (!sp.ok && un.j == 0 && h == 0 && lane == 0)
                atomicCAS(args.err_word, 0, kErrSeqlens);
            if (un.j * kBlk >= sp.len) continue;  // past this sequence's end
            const int nb = (sp.len + kBlk - 1) / kBlk;
            const int i0 = first_block(un.j, args.causal);
            // K and V of this unit load after its first block's Q and dO: the
            // previous unit frees their buffers earlier (its second-to-last dK,
            // its last dV) than K and V (its last dK), so the first block's
            // copies and -LSE / -Delta rows are in place when K and V arrive
            const uint32_t kv_par = (nunit & 1) ^ 1;
            ++nunit;
            auto load_kv = [&]() {
                if (lane == 0) {
                    w.code = kErrBwdWait + 1;
                    ok = mbar_wait(kv_empty, kv_par, w);
                    if (ok) {
                        mbar_arrive_expect_tx(kv_full, 2 * Cfg::kTile);
                        for (int c = 0; c < Cfg::kBoxes; ++c) {
                            tma_load_4d(smem + Cfg::kOffK + c * kBox, &args.tm_k, kv_full, 64 * c, h,
                                        sp.trow0 + un.j * kBlk, sp.tb);
                            tma_load_4d(smem + Cfg::kOffV + c * kBox, &args.tm_v, kv_full, 64 * c, h,
                                        sp.trow0 + un.j * kBlk, sp.tb);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (ok) ++nkv;
            };
            // (fixed order: K and V first; the later K/V copy measured 2-3 % slower there)
            if constexpr (kDet) load_kv();
            for (int i_ = i0; i_ < nb && ok; ++i_, ++nblk) {
                const int i = kDet ? block_at(un.j, i_ - i0, i0, nb, rotate) : i_;
                const int st = nblk & 1;
                // this block's -LSE/scale and -Delta per query, loaded before the
                // waits so their latency overlaps them (-inf / 0 past S: P = 0)
                float lv[4], dv[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int q = i * kBlk + r * 32 + lane;
                    const size_t x = stat_index(args.cu_seqlens, args.T, S, H, b, h, sp, q);
                    lv[r] = q < sp.len ? -args.lse[x] * inv_scale : -INFINITY;
                    dv[r] = q < sp.len ? -args.delta[x] : 0.f;
                }
                // Q_i into stage st with the bias rows of S^T, then dO_i (single
                // stage: the previous block's dV MMA, and so its dP^T, has
                // finished) with the bias rows of dP^T.  A unit's first block
                // issues both copies, then the unit's K and V, and writes its
                // rows last: the rows wait for the -LSE / -Delta loads, which
                // must not hold up the K/V copy
                const bool first_blk = !kDet && i_ == i0;
                w.code = kErrBwdWait + 2;
                ok = mbar_wait(&q_empty[st], ((nblk >> 1) & 1) ^ 1, w);
                ok = __all_sync(0xffffffffu, ok ? 1 : 0) != 0;
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&q_full[st], Cfg::kTile);
                    for (int c = 0; c < Cfg::kBoxes; ++c)
                        tma_load_4d(smem + Cfg::kOffQ + st * Cfg::kTile + c * kBox, &args.tm_q,
                                    &q_full[st], 64 * c, h, sp.trow0 + i * kBlk, sp.tb);
                }
                ++nq;
                auto q_rows = [&]() {
                    uint8_t *lb = smem + Cfg::kOffLb + st * Cfg::kBias;
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        *reinterpret_cast<uint4 *>(lb + bias_off(r * 32 + lane, 0)) = bias_row(lv[r]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&q_full[st]);
                };
                if (!first_blk) q_rows();
                w.code = kErrBwdWait + 3;
                ok = mbar_wait(do_empty, (nblk & 1) ^ 1, w);
                ok = __all_sync(0xffffffffu, ok ? 1 : 0) != 0;
                if (!ok) {
                    if (first_blk) q_rows();  // Q's barrier phase completes for the unwinding
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(do_full, Cfg::kTile);
                    for (int c = 0; c < Cfg::kBoxes; ++c)
                        tma_load_4d(smem + Cfg::kOffDO + c * kBox, &args.tm_do, do_full,
                                    64 * c, h, sp.trow0 + i * kBlk, sp.tb);
                }
                ++ndo;
                if (first_blk) {
                    load_kv();  // on failure the rows below still complete Q's and dO's phases
                    q_rows();
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    *reinterpret_cast<uint4 *>(smem + Cfg::kOffDb + bias_off(r * 32 + lane, 0)) =
                        bias_row(dv[r]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(do_full);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            }
        }
        if (!ok && lane == 0) {
            // let issued copies land before the CTA exits: the last K/V pair,
            // the last Q copy of each stage (the loop may stop between a
            // block's Q and its dO) and the last dO
            if (nkv > 0) mbar_wait_drain(kv_full, (nkv - 1) & 1);
            for (uint32_t m = nq > 2 ? nq - 2 : 0; m < nq; ++m)
                mbar_wait_drain(&q_full[m & 1], (m >> 1) & 1);
            if (ndo > 0) mbar_wait_drain(do_full, (ndo - 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 10};
            const uint32_t tX = tmem + Cfg::kTX, tY = tmem + Cfg::kTY;
            const uint32_t tdV = tmem + Cfg::kTdV, tdK = tmem + Cfg::kTdK;
            const uint32_t aK = sbase + Cfg::kOffK, aV = sbase + Cfg::kOffV;
            const uint32_t aDO = sbase + Cfg::kOffDO, aDS = sbase + Cfg::kOffDS;
            const uint32_t aOnes = sbase + Cfg::kOffOnes, aLb = sbase + Cfg::kOffLb;
            const uint32_t aDb = sbase + Cfg::kOffDb;
            uint32_t nunit = 0, nblk = 0;
            uint32_t ph_p = 0, ph_ds = 0, ph_dqe = 0;
            bool ok = true;
#define FA_WAIT(bar, par, site)                                  \
    do {                                                         \
        w.code = kErrBwdWait + (site);                           \
        if (!mbar_wait((bar), (par), w)) { ok = false; break; } \
    } while (0)
            for (int it = 0; ok; ++it) {
                BUnit un;
                if (!bunit_at(it, U, BH, kTileMajor, un, ugs)) break;
                if (un.j < 0) continue;
                const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, un.bh / H);
                if (un.j * kBlk >= sp.len) continue;
                const int nb = (sp.len + kBlk - 1) / kBlk;
                const int i0 = first_block(un.j, args.causal);
                FA_WAIT(kv_full, nunit & 1, 10);
                if (!ok) break;
                // first block: S^T and dP^T (the previous unit's last dQ was
                // drained before its dP would have been issued; wait for it here)
                {
                    const int st = nblk & 1;
                    FA_WAIT(&q_full[st], (nblk >> 1) & 1, 11);
                    if (!ok) break;
                    tc_fence_after();
                    issue_kmajor<D>(tX, aK, sbase + Cfg::kOffQ + st * Cfg::kTile, aOnes,
                                    aLb + st * Cfg::kBias);
                    mma_commit(s_full);
                    if (nblk > 0) {
                        FA_WAIT(dq_empty, ph_dqe, 12);
                        if (!ok) break;
                        ph_dqe ^= 1;
                    }
                    FA_WAIT(do_full, nblk & 1, 13);
                    if (!ok) break;
                    tc_fence_after();
                    issue_kmajor<D>(tY, aV, aDO, aOnes, aDb);
                    mma_commit(dp_full);
                }
                for (int i = i0; i < nb; ++i, ++nblk) {
                    const int st = nblk & 1;
                    const bool first = (i == i0), has_next = (i + 1 < nb);
                    FA_WAIT(p_ready, ph_p, 14);
                    if (!ok) break;
                    ph_p ^= 1;
                    if (first && nunit > 0) {
                        // the previous unit's epilogue has read the dV accumulator
                        FA_WAIT(dv_empty, (nunit - 1) & 1, 15);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    issue_acc<D>(tdV, tX, aDO, !first);
                    mma_commit(do_empty);
                    if (has_next) {
                        const int st2 = (nblk + 1) & 1;
                        FA_WAIT(&q_full[st2], ((nblk + 1) >> 1) & 1, 16);
                        if (!ok) break;
                        tc_fence_after();
                        issue_kmajor<D>(tX, aK, sbase + Cfg::kOffQ + st2 * Cfg::kTile, aOnes,
                                        aLb + st2 * Cfg::kBias);
                        mma_commit(s_full);
                    }
                    FA_WAIT(ds_ready, ph_ds, 17);
                    if (!ok) break;
                    ph_ds ^= 1;
                    tc_fence_after();
                    // dQ first, so that its drain overlaps the dK MMAs; dK reads
                    // dS from shared memory, which leaves Y to dQ
                    issue_dq<D>(tY, aDS, aK);
                    mma_commit(dq_full);
                    if (first && nunit > 0) {
                        // the previous unit's epilogue has read the dK accumulator
                        FA_WAIT(dk_empty, (nunit - 1) & 1, 20);
                        if (!ok) break;
                    }
                    issue_dk<D>(tdK, aDS, sbase + Cfg::kOffQ + st * Cfg::kTile, !first);
                    mma_commit(&q_empty[st]);
                    if (has_next) {
                        FA_WAIT(dq_empty, ph_dqe, 18);
                        if (!ok) break;
                        ph_dqe ^= 1;
                        FA_WAIT(do_full, (nblk + 1) & 1, 19);
                        if (!ok) break;
                        tc_fence_after();
                        issue_kmajor<D>(tY, aV, aDO, aOnes, aDb);
                        mma_commit(dp_full);
                    } else {
                        mma_commit(dkdv_full);
                        mma_commit(kv_empty);
                    }
                }
                ++nunit;
            }
#undef FA_WAIT
            mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
    }
    else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ P^T and dS^T
        const int quarter = warp & 3;
        const int kr = quarter * 32 + lane;  // key row of the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tX = tmem + Cfg::kTX + lane_off, tY = tmem + Cfg::kTY + lane_off;
        const float c2 = args.scale_log2;
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 30};
        uint32_t n = 0;
        bool ok = true;
        uint8_t *ds_row = smem + Cfg::kOffDS + kr * 128;
        const int sw = kr & 7;  // 128B swizzle phase of this row
        for (int it = 0; ok; ++it) {
            BUnit un;
            if (!bunit_at(it, U, BH, kTileMajor, un, ugs)) break;
            if (un.j < 0) continue;
            const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, un.bh / H);
            if (un.j * kBlk >= sp.len) continue;
            const int nb = (sp.len + kBlk - 1) / kBlk;
            const int i0 = first_block(un.j, args.causal);
            const int key = un.j * kBlk + kr;  // row within the sequence
            for (int i_ = i0; i_ < nb; ++i_, ++n) {
                const int i = kDet ? block_at(un.j, i_ - i0, i0, nb, rotate) : i_;
                w.code = kErrBwdWait + 31;
                if (!mbar_wait(s_full, n & 1, w)) { ok = false; break; }
                tc_fence_after();
                uint32_t pk[64];
                {
                    uint32_t sr[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(tX + c * 32, sr[c]);
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
                    // X holds S^T - LSE/scale (the bias K step), so P = 2^(X c2).
                    // Visible: key < S and (non-causal or query >= key); masking
                    // only where a block can hold invisible pairs: the causal
                    // diagonal block and a key tile reaching past S (queries past
                    // S carry a bias of -inf, which gives P = 0)
                    if ((args.causal && i == un.j) || (un.j + 1) * kBlk > sp.len) {
                        const int lim = (args.causal && i == un.j) ? kr : -1;  // col < lim hidden
                        const bool key_ok = key < sp.len;
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
                        for (int e = 0; e < 32; e += 2) {
                            const float2 x = mul2(make_float2(__uint_as_float(sr[c][e]),
                                                              __uint_as_float(sr[c][e + 1])),
                                                  make_float2(c2, c2));
                            pk[(c * 32 + e) / 2] = pack_bf16x2(ex2_mufu(x.x), ex2_mufu(x.y));
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tmem_st16(tX + c * 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[c * 16]));
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(p_ready);
                // ---- dS^T = P^T o (dP^T - Delta); Y holds dP^T - Delta (bias K step)
                w.code = kErrBwdWait + 32;
                if (!mbar_wait(dp_full, n & 1, w)) { ok = false; break; }
                if (n > 0) {
                    // the dQ and dK MMAs of the previous block have finished
                    // reading dS (dK, the later one, is committed with Q's stage)
                    w.code = kErrBwdWait + 33;
                    if (!mbar_wait(&q_empty[(n - 1) & 1], ((n - 1) >> 1) & 1, w)) { ok = false; break; }
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
                    const uint32_t (&dr)[32] = drr[c - c2i];
                    uint32_t dsw[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        // dS = P o (dP - Delta): the fp32 difference rounded to bf16,
                        // times the bf16 P, two columns per instruction
                        dsw[e / 2] = mul_bf16x2(pk[(c * 32 + e) >> 1],
                                                pack_bf16x2(__uint_as_float(dr[e]),
                                                            __uint_as_float(dr[e + 1])));
                    // shared copy for the dQ MMA: queries [32c, 32c+32) of this key row,
                    // 128B-swizzled, two 64-query blocks of 16 KB
                    uint8_t *blk = ds_row + (c >> 1) * kBox;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int chunk = (c & 1) * 4 + t;
                        *reinterpret_cast<uint4 *>(blk + ((chunk ^ sw) << 4)) =
                            make_uint4(dsw[4 * t], dsw[4 * t + 1], dsw[4 * t + 2], dsw[4 * t + 3]);
                    }
                  }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(ds_ready);
            }
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ dQ drain + dK/dV epilogue
        // dQ_i is staged 32 x 32 at a time in 128B-swizzled shared memory (one
        // 4 KB tile per warp) and added into the fp32 accumulator by TMA bulk
        // reductions, which keeps the atomics off the load/store pipe the
        // softmax warps use.
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // TMEM lane: query (dQ) or key (dK, dV)
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        uint8_t *stage = smem + Cfg::kOffRed + quarter * 4096;
        uint8_t *stage_row = stage + lane * 128;
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 40};
        // each warp stages its 32 query rows of dQ_i, 32 columns at a time, and
        // reduces them on its own (no wait on the other drain warps)
        auto stage_and_reduce = [&](const uint32_t (&acc)[D], int row0, int z, bool go,
                                    const CUtensorMap *map) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                if (lane == 0) bulk_wait_read<0>();  // the previous reduction has read buf
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    *reinterpret_cast<uint4 *>(stage_row + ((k ^ (lane & 7)) << 4)) =
                        make_uint4(acc[c * 32 + 4 * k], acc[c * 32 + 4 * k + 1],
                                   acc[c * 32 + 4 * k + 2], acc[c * 32 + 4 * k + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && go && !*abort_flag) {
                    tma_reduce_add_3d(map, stage, 32 * c, row0, z);
                    bulk_commit();
                }
            }
        };
        // Fixed-order mode: each drain warp has its own turn counters (its 32
        // query rows of a block), so the four warps never wait on one another
        // here.  A turn is passed on once this warp's reductions of the block
        // are complete: wait for its bulk groups, order their (async-proxy)
        // writes before the release, then a release add on the counter.
        int *sem_prev = nullptr;
        auto release_block = [&](int *sem_done) {
            if (lane == 0) {
                bulk_wait<0>();
                fence_proxy_async_global();
                red_release_gpu_add(sem_done, 1);
            }
        };
        uint32_t n = 0, nunit = 0;
        bool ok = true;
        for (int it = 0; ok; ++it) {
            BUnit un;
            if (!bunit_at(it, U, BH, kTileMajor, un, ugs)) break;
            if (un.j < 0) continue;
            const int b = un.bh / H, h = un.bh % H;
            const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, b);
            if (un.j * kBlk >= sp.len) continue;
            const int nb = (sp.len + kBlk - 1) / kBlk;
            // accumulator rows: [B*H, S] fixed, [H, T] packed
            const int acc_row0 = args.cu_seqlens ? sp.tok0 : 0;
            const int acc_z = args.cu_seqlens ? h : un.bh;
            const int i0 = first_block(un.j, args.causal);
            for (int i_ = i0; i_ < nb; ++i_, ++n) {
                const int i = kDet ? block_at(un.j, i_ - i0, i0, nb, rotate) : i_;
                w.code = kErrBwdWait + 40;
                if (!mbar_wait(dq_full, n & 1, w)) { ok = false; break; }
                tc_fence_after();
                uint32_t acc[D];
#pragma unroll
                for (int c = 0; c < D / 32; ++c)
                    tmem_ld32(tmem + Cfg::kTY + lane_off + c * 32,
                              *reinterpret_cast<uint32_t(*)[32]>(&acc[c * 32]));
#pragma unroll
                for (int c = 0; c < D / 32; ++c)
                    tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&acc[c * 32]));
                tc_fence_before();
                mbar_arrive(dq_empty);
                if constexpr (kDet) {
                    // Fixed order: key tile j's share of dQ block i has a place
                    // p in the block's sum (dq_position / causal_rank).  Places
                    // alternate between two accumulators: p goes into
                    // accumulator p % 2 as its (p / 2)-th term, so consecutive
                    // contributions do not wait on each other, and each
                    // accumulator's order is still fixed (the convert kernel
                    // adds the two in a fixed order).  This warp waits until
                    // the counter of (block, its 32 rows, accumulator) reaches
                    // p / 2.  Its counter of the previous block is released
                    // first, a block period after its reductions were issued
                    // (so they are complete) and independently of this block's
                    // wait: a release needs only this CTA's own progress (its
                    // warps' earlier turns), which keeps the waits between
                    // tiles acyclic.
                    if (sem_prev) {
                        release_block(sem_prev);
                        sem_prev = nullptr;
                    }
                    const int place =
                        args.causal ? causal_rank(args.dq_key + static_cast<size_t>(un.bh) * nT, un.j, i, lane)
                                    : dq_position(un.bh, un.j, i, nT, nb, gridDim.x);
                    int *sem = args.dq_sem + static_cast<size_t>(un.bh) * nSem + 8 * i + 2 * quarter +
                               (place & 1);
                    bool go = true;
                    if (lane == 0) {
                        w.code = kErrBwdWait + 42;
                        go = counter_wait_geq(sem, place >> 1, w);
                        fence_proxy_async_global();
                    }
                    go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
                    stage_and_reduce(acc, acc_row0 + i * kBlk + quarter * 32, acc_z, go,
                                     (place & 1) ? &args.tm_dqacc2 : &args.tm_dqacc);
                    sem_prev = sem;
                } else {
                    stage_and_reduce(acc, acc_row0 + i * kBlk + quarter * 32, acc_z, true,
                                     &args.tm_dqacc);
                }
            }
            if (kDet && sem_prev) {  // the unit's last block
                release_block(sem_prev);
                sem_prev = nullptr;
            }
            if (!ok) break;
            w.code = kErrBwdWait + 41;
            if (!mbar_wait(dkdv_full, nunit & 1, w)) { ok = false; break; }
            ++nunit;
            tc_fence_after();
            const int key = un.j * kBlk + r;
            const size_t orow = ((static_cast<size_t>(sp.tok0) + key) * H + h) * D;
            // dV, then dK.  Atomic order: each accumulator's columns are read
            // into registers and packed to bf16 first, and released (dv_empty /
            // dk_empty) before they are written out, so the next unit's first dV
            // and dK MMAs wait only for the reads.  Fixed order: 64 columns at a
            // time, released after the last (holding a whole accumulator costs
            // that instance register spills).  They leave by TMA stores from this
            // warp's staging buffer (its 32 key rows x 64 columns, the TMA box,
            // 128B swizzle), unless the tile runs past its sequence in a packed
            // batch (a store would write the next sequence's rows): then by
            // direct stores.
            const bool use_tma = !args.cu_seqlens || (un.j + 1) * kBlk <= sp.len;
            constexpr int kHeld = kDet ? 64 : D;  // columns held in registers at once
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t tsrc = tmem + lane_off + (which ? Cfg::kTdK : Cfg::kTdV);
                const float mul = which ? args.scale : 1.f;
                const CUtensorMap *map = which ? &args.tm_dk32 : &args.tm_dv32;
                uint16_t *out = reinterpret_cast<uint16_t *>(which ? args.dk : args.dv) + orow;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += kHeld) {
                    uint32_t pk[kHeld / 2];  // columns c0 + 2e, c0 + 2e + 1 in pk[e]
#pragma unroll
                    for (int c = 0; c < kHeld / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tsrc + c0 + c * 32, v);
                        tmem_ld_wait(v);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[16 * c + e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul,
                                                         __uint_as_float(v[2 * e + 1]) * mul);
                    }
                    if (c0 + kHeld == D) {  // the accumulator has been read
                        tc_fence_before();
                        mbar_arrive(which ? dk_empty : dv_empty);
                    }
                    if (use_tma) {
#pragma unroll
                        for (int c = 0; c < kHeld / 64; ++c) {
                            if (lane == 0) bulk_wait_read<0>();  // the staging buffer has been read
                            __syncwarp();
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                *reinterpret_cast<uint4 *>(stage_row + ((k ^ (lane & 7)) << 4)) =
                                    make_uint4(pk[32 * c + 4 * k], pk[32 * c + 4 * k + 1],
                                               pk[32 * c + 4 * k + 2], pk[32 * c + 4 * k + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_4d(map, stage, c0 + 64 * c, h,
                                             sp.trow0 + un.j * kBlk + quarter * 32, sp.tb);
                                bulk_commit();
                            }
                        }
                    } else if (key < sp.len) {
                        uint4 *dst = reinterpret_cast<uint4 *>(out + c0);
#pragma unroll
                        for (int k = 0; k < kHeld / 8; ++k)
                            dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                    }
                }
            }
        }
        if (lane == 0) bulk_wait<0>();  // every drain warp's reductions have read shared memory
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
}

// ---------------------------------------------------------------- prep / convert

// One warp per (b, h, query row): Delta = sum_d dO * O (fp32), and the row of
// the dQ accumulator set to zero.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep(const __grid_constant__ BwdArgs args) {
    const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(args.B) * args.H * args.S;
    if (row >= rows) return;
    const int S = args.S, H = args.H;
    const int q = static_cast<int>(row % S);
    const long long bh = row / S;
    const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
    const size_t off = ((static_cast<size_t>(b) * S + q) * H + h) * D;
    constexpr int kPer = D / 32;  // bf16 per lane
    const __nv_bfloat16 *po = reinterpret_cast<const __nv_bfloat16 *>(args.o) + off + lane * kPer;
    const __nv_bfloat16 *pd = reinterpret_cast<const __nv_bfloat16 *>(args.dout) + off + lane * kPer;
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
        const float2 o2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(po + e));
        const float2 d2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(pd + e));
        acc = fmaf(o2.x, d2.x, acc);
        acc = fmaf(o2.y, d2.y, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
        args.delta[row] = acc;
    }
    float4 *z = reinterpret_cast<float4 *>(args.dq_acc + static_cast<size_t>(row) * D);
#pragma unroll
    for (int e = lane; e < D / 4; e += 32) z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (args.dq_acc2) {  // fixed-order mode: the second accumulator too
        float4 *z2 = reinterpret_cast<float4 *>(args.dq_acc2 + static_cast<size_t>(row) * D);
#pragma unroll
        for (int e = lane; e < D / 4; e += 32) z2[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Fixed-order mode: zero the counters (one per (sequence, head, 64 rows) of
// the longest sequence; at D = 256 one per output half as well) and, under a
// causal mask at D = 64 and 128, write each unit's order key.  Launched with
// the batch as given (not the per-token view of a packed batch).
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_det_setup(const __grid_constant__ BwdArgs args) {
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    // D = 64/128: eight per 128-query block (drain warp x accumulator); D =
    // 256: four per 64-query block and output half (one per drain warp)
    const long long nctr = static_cast<long long>(args.B) * args.H *
                           (D == 256 ? 8 * ((args.S + 63) / 64) : 8 * ((args.S + kBlk - 1) / kBlk));
    if (t < nctr) args.dq_sem[t] = 0;
    if constexpr (D != 256) {
        if (args.dq_key && args.causal) {
            const int nT = (args.S + kBlk - 1) / kBlk;
            const long long U = static_cast<long long>(args.B) * args.H * nT;
            if (t < U) {
                int bh, j;
                unit_coords(static_cast<int>(t), nT, args.B * args.H, true, bh, j);
                args.dq_key[static_cast<size_t>(bh) * nT + j] =
                    causal_order_key(args, static_cast<int>(t), static_cast<int>(U), nT, args.grid);
            }
        }
    }
}

// One warp per (b, h, query row): dQ[b, q, h, :] = bf16(scale * accumulator)
// (fixed-order mode: bf16(scale * (accumulator + second accumulator))).
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_dq_cvt(const __grid_constant__ BwdArgs args) {
    const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(args.B) * args.H * args.S;
    if (row >= rows) return;
    const int S = args.S, H = args.H;
    const int q = static_cast<int>(row % S);
    const long long bh = row / S;
    const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
    const float *src = args.dq_acc + static_cast<size_t>(row) * D;
    uint32_t *dst = reinterpret_cast<uint32_t *>(reinterpret_cast<uint16_t *>(args.dq) +
                                                 ((static_cast<size_t>(b) * S + q) * H + h) * D);
    if (args.dq_acc2) {
        const float *src2 = args.dq_acc2 + static_cast<size_t>(row) * D;
#pragma unroll
        for (int e = lane; e < D / 2; e += 32) {
            const float2 a = reinterpret_cast<const float2 *>(src)[e];
            const float2 a2 = reinterpret_cast<const float2 *>(src2)[e];
            dst[e] = pack_bf16x2((a.x + a2.x) * args.scale, (a.y + a2.y) * args.scale);
        }
        return;
    }
#pragma unroll
    for (int e = lane; e < D / 2; e += 32) {
        const float2 a = reinterpret_cast<const float2 *>(src)[e];
        dst[e] = pack_bf16x2(a.x * args.scale, a.y * args.scale);
    }
}

template <int D>
cudaError_t launch_det_setup(const BwdArgs &a, int grid, cudaStream_t stream) {
    BwdArgs sa = a;
    sa.grid = grid;
    const long long nctr = static_cast<long long>(a.B) * a.H *
                           (D == 256 ? 8 * ((a.S + 63) / 64) : 8 * ((a.S + kBlk - 1) / kBlk));
    const long long U = static_cast<long long>(a.B) * a.H * ((a.S + kBlk - 1) / kBlk);
    const long long n = nctr > U ? nctr : U;
    fa_bwd_det_setup<D><<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(sa);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs &a, cudaStream_t stream) {
    using Cfg = BwdCfg<D>;
    // Delta, the accumulator and dQ are per token: the prep and convert
    // kernels see a packed batch as one sequence of T tokens
    const long long U = static_cast<long long>(a.B) * a.H * ((a.S + kBlk - 1) / kBlk);
    const int grid = static_cast<int>(U < a.num_sms ? U : a.num_sms);
    BwdArgs rows_view = a;
    if (a.cu_seqlens) {
        rows_view.B = 1;
        rows_view.S = a.T;
    }
    const long long rows = static_cast<long long>(rows_view.B) * a.H * rows_view.S;
    const long long blocks = (rows * 32 + 255) / 256;
    cudaError_t e;
    if (a.dq_sem && (e = launch_det_setup<D>(a, grid, stream)) != cudaSuccess) return e;
    fa_bwd_prep<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(rows_view);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.pair) {
        if ((e = launch_bwd_main_pair(a, stream)) != cudaSuccess) return e;
        fa_bwd_dq_cvt<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(rows_view);
        return cudaGetLastError();
    }
    // causal masks: units tile-major, i.e. longest first across heads (head
    // by head, the serpentine rounds leave the busiest CTA about 10 % more
    // blocks than the average at S = 32768, H = 16)
    auto kern = a.dq_sem ? (a.causal ? fa_bwd_kernel<D, true, true> : fa_bwd_kernel<D, true, false>)
                         : (a.causal ? fa_bwd_kernel<D, false, true> : fa_bwd_kernel<D, false, false>);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (a.dq_sem) {
        // CTAs wait on one another's dQ counters: a cooperative launch
        // guarantees they are all resident at once
        void *params[] = {const_cast<BwdArgs *>(&a)};
        e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(grid),
                                        dim3(kThreads), params, Cfg::kSmemBytes, stream);
        if (e != cudaSuccess) return e;
    } else {
        kern<<<grid, kThreads, Cfg::kSmemBytes, stream>>>(a);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fa_bwd_dq_cvt<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(rows_view);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t stream) {
    switch (a.D) {
        case 64: return launch_bwd_d<64>(a, stream);
        case 128: return launch_bwd_d<128>(a, stream);
        case 256: {
            BwdArgs rows_view = a;  // per-token view for prep and convert, as above
            if (a.cu_seqlens) {
                rows_view.B = 1;
                rows_view.S = a.T;
            }
            const long long rows = static_cast<long long>(rows_view.B) * a.H * rows_view.S;
            const unsigned blocks = static_cast<unsigned>((rows * 32 + 255) / 256);
            cudaError_t e;
            if (a.dq_sem && (e = launch_det_setup<256>(a, 0, stream)) != cudaSuccess) return e;
            fa_bwd_prep<256><<<blocks, 256, 0, stream>>>(rows_view);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
            if ((e = a.pair ? launch_bwd_main_d256_split(a, stream) : launch_bwd_main_d256(a, stream)) !=
                cudaSuccess)
                return e;
            fa_bwd_dq_cvt<256><<<blocks, 256, 0, stream>>>(rows_view);
            return cudaGetLastError();
        }
        default: return cudaErrorNotSupported;
    }
}

}  // namespace fa
