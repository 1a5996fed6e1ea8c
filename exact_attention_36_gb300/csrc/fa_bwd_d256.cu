// fa_bwd_d256.cu -- fused attention backward main kernel for head dim 256.
//
// Same mathematics as fa_bwd.cu ("FlashAttention-4: Algorithm and Kernel
// Pipelining Co-Design for Asymmetric Hardware Scaling" (gist.science/nl),
// Technische samenvatting, Methodologie §3), reorganised so that it fits the
// Tensor Memory and shared memory of one SM at D = 256:
//   * dK and dV for all 256 columns would fill the 512 TMEM columns by
//     themselves, so a work unit is (b, h, key tile j of 128 keys, output
//     half oh): it accumulates dK[:, 128oh : 128oh+128] and the same half of
//     dV, and adds the same half of dQ.  S^T and dP^T (contractions over all
//     256 columns) are recomputed by both halves.
//   * K_j and V_j (64 KB each) stay resident; queries stream in blocks of 64
//     rows (Q_i and dO_i 32 KB each, one stage each).  Q_i is loaded as two
//     head-dim halves with their own barriers: dK of output half oh reads only
//     half oh, so the other half is released when S^T is done and the next
//     block's copy of it loads while dP, dV and dK run; S^T takes its K steps
//     over that half first.  LSE and Delta are double-buffered by block parity.
//   * dQ^T = K_j[:, half]^T dS^T is formed with the head dim on the TMEM
//     lanes (M = 128), so the drain warps hold one dQ column each.
// Tensor Memory: X = S^T / P^T (64 cols) | Y = dP^T / dS^T / dQ^T (64 cols) |
// dV half (128) | dK half (128).  The MMAs of a block run in order
// S, dP, dV, dK, dQ; this variant does not overlap blocks.
#include <cuda_bf16.h>

#include "fa_common.cuh"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr int kKeys = 128;     // keys per unit
constexpr int kQB = 64;        // queries per block
constexpr int kD = 256;
constexpr int kBoxK = 16384;   // K/V box: 128 rows x 64 bf16
constexpr int kBoxQ = 8192;    // Q/dO box: 64 rows x 64 bf16

struct Cfg {
    static constexpr int kOffK = 0;                   // 4 boxes
    static constexpr int kOffV = kOffK + 4 * kBoxK;   // 4 boxes
    static constexpr int kOffQ = kOffV + 4 * kBoxK;   // 4 boxes (64 rows)
    static constexpr int kOffDO = kOffQ + 4 * kBoxQ;  // 4 boxes
    static constexpr int kOffDS = kOffDO + 4 * kBoxQ; // 128 keys x 64 queries bf16 (16 KB)
    static constexpr int kOffRed = kOffDS + 16384;    // 2 x (64 rows x 32 fp32) dQ staging
    static constexpr int kOffStat = kOffRed + 16384;  // [2] x (64 lse2 + 64 delta), by block parity
    static constexpr int kOffBar = kOffStat + 1024;
    static constexpr int kNumBars = 19;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kSmemBytes = kOffMisc + 16;  // base must be 1024-aligned (checked)
    static constexpr uint32_t kTX = 0, kTY = 64, kTdV = 128, kTdK = 256;
    static constexpr uint32_t kIdescSS = idesc_bf16_f32(128, kQB, false, false);   // S^T, dP^T
    static constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, 128, false, true);   // dV, dK half
    static constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, kQB, true, true);     // dQ^T half
};
static_assert(Cfg::kSmemBytes <= 232448, "shared memory budget");

struct Unit256 {
    int bh, j, oh;  // j = -1: no unit for this CTA this round
};

__device__ __forceinline__ bool unit256_at(int it, int U, int nT, Unit256 &out) {
    const int G = gridDim.x;
    const int base = it * G;
    if (base >= U) return false;
    const int c = (it & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    const int u = base + c;
    if (u >= U) {
        out.j = -1;
        return true;
    }
    // the two halves of a key tile, then the key tiles of a head, are adjacent
    out.oh = u & 1;
    out.j = (u >> 1) % nT;
    out.bh = (u >> 1) / nT;
    return true;
}

// kDet: the fixed-order dQ mode (args.dq_sem set), a separate instance so that
// the atomic-order kernel carries none of its logic
template <bool kDet>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_kernel_d256(const __grid_constant__ BwdArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) atomicCAS(args.err_word, 0, kErrBwdWait + 0xfe);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint64_t *kv_full = bars + 0, *kv_empty = bars + 1;
    // Q in two head-dim halves (boxes 0-1 and 2-3), each with its own barriers:
    // dK of output half oh reads only half oh of Q, so the other half is
    // released as soon as S is done and the next block's copy of it loads
    // while dP, dV and dK run
    uint64_t *qh_full = bars + 15, *qh_empty = bars + 17;  // [2] each
    uint64_t *st_full = bars + 2;                          // [2]: LSE/Delta of the block written
    uint64_t *do_full = bars + 4, *do_empty = bars + 5;
    uint64_t *s_full = bars + 6, *dp_full = bars + 7;
    uint64_t *p_ready = bars + 8, *ds_ready = bars + 9;
    uint64_t *dq_full = bars + 10, *dq_empty = bars + 11;
    uint64_t *dkdv_full = bars + 12, *dkdv_empty = bars + 13;
    uint64_t *drain = bars + 14;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);
    float *stat_base = reinterpret_cast<float *>(smem + Cfg::kOffStat);  // [2] x (lse2[64] | delta[64])

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = args.H, S = args.S;
    const int BH = args.B * H;
    const int nT = (S + kKeys - 1) / kKeys;  // key tiles (S: the longest sequence if packed)
    const int U = BH * nT * 2;

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qh_full[i], 1);
            mbar_init(&qh_empty[i], 1);
            mbar_init(&st_full[i], 1);
        }
        mbar_init(do_full, 1);
        mbar_init(do_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(dp_full, 1);
        mbar_init(p_ready, 128);
        mbar_init(ds_ready, 128);
        mbar_init(dq_full, 1);
        mbar_init(dq_empty, 128);
        mbar_init(dkdv_full, 1);
        mbar_init(dkdv_empty, 128);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t sbase = smem_u32(smem);
    // first query block a key tile sees (causal: queries >= first key)
    auto first_qblock = [&](int j) { return args.causal ? (j * kKeys) / kQB : 0; };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0x51};
        const float log2e = 1.4426950408889634f;
        uint32_t nunit = 0, n = 0;
        uint32_t nkv = 0, ndo = 0;  // copies issued (for the unwinding)
        uint32_t nqh[2] = {0, 0};   // Q half copies issued
        bool ok = true;
        for (int it = 0; ok; ++it) {
            Unit256 un;
            if (!unit256_at(it, U, nT, un)) break;
            if (un.j < 0) continue;
            const int b = un.bh / H, h = un.bh % H;
            const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, b);
            if (!sp.ok && un.j == 0 && h == 0 && un.oh == 0 && lane == 0)
                atomicCAS(args.err_word, 0, kErrSeqlens);
            if (un.j * kKeys >= sp.len) continue;  // past this sequence's end
            const int nQ = (sp.len + kQB - 1) / kQB;
            if (lane == 0) {
                w.code = kErrBwdWait + 0x51;
                ok = mbar_wait(kv_empty, (nunit & 1) ^ 1, w);
                if (ok) {
                    mbar_arrive_expect_tx(kv_full, 8 * kBoxK);
                    for (int c = 0; c < 4; ++c) {
                        tma_load_4d(smem + Cfg::kOffK + c * kBoxK, &args.tm_k, kv_full, 64 * c, h,
                                    sp.trow0 + un.j * kKeys, sp.tb);
                        tma_load_4d(smem + Cfg::kOffV + c * kBoxK, &args.tm_v, kv_full, 64 * c, h,
                                    sp.trow0 + un.j * kKeys, sp.tb);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (ok) ++nkv;
            ++nunit;
            // per block: the early Q half (not read by dK), LSE/Delta, dO, then
            // the late Q half (read by dK of the previous block)
            const int eh = 1 - un.oh, lh = un.oh;
            for (int i = first_qblock(un.j); i < nQ && ok; ++i, ++n) {
                // LSE / Delta into registers first: their latency overlaps the waits
                float lv[2], dv[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int q = i * kQB + r * 32 + lane;
                    const size_t x = stat_index(args.cu_seqlens, args.T, S, H, b, h, sp, q);
                    lv[r] = q < sp.len ? args.lse[x] * log2e : INFINITY;
                    dv[r] = q < sp.len ? args.delta[x] : 0.f;
                }
                auto load_q_half = [&](int hs) -> bool {
                    w.code = kErrBwdWait + 0x52;
                    bool good = mbar_wait(&qh_empty[hs], (n & 1) ^ 1, w);
                    good = __all_sync(0xffffffffu, good ? 1 : 0) != 0;
                    if (!good) return false;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&qh_full[hs], 2 * kBoxQ);
                        for (int c = 2 * hs; c < 2 * hs + 2; ++c)
                            tma_load_4d(smem + Cfg::kOffQ + c * kBoxQ, &args.tm_q, &qh_full[hs], 64 * c, h,
                                        sp.trow0 + i * kQB, sp.tb);
                    }
                    ++nqh[hs];
                    return true;
                };
                if (!load_q_half(eh)) { ok = false; break; }
                // stats buffer n & 1 was last read by the softmax of block n - 2,
                // whose dS preceded dQ(n - 2) and so S(n - 1), whose completion
                // (or a later one) released the early half just waited for
                float *st = stat_base + (n & 1) * 128;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    st[r * 32 + lane] = lv[r];
                    st[64 + r * 32 + lane] = dv[r];
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&st_full[n & 1]);
                    w.code = kErrBwdWait + 0x53;
                    ok = mbar_wait(do_empty, (n & 1) ^ 1, w);
                    if (ok) {
                        mbar_arrive_expect_tx(do_full, 4 * kBoxQ);
                        for (int c = 0; c < 4; ++c)
                            tma_load_4d(smem + Cfg::kOffDO + c * kBoxQ, &args.tm_do, do_full,
                                        64 * c, h, sp.trow0 + i * kQB, sp.tb);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                ++ndo;
                if (!load_q_half(lh)) { ok = false; break; }
            }
        }
        if (!ok && lane == 0) {
            // let issued copies land before the CTA exits (only those issued:
            // the loop may stop between a block's Q and its dO)
            if (nkv > 0) mbar_wait_drain(kv_full, (nkv - 1) & 1);
            for (int hs = 0; hs < 2; ++hs)
                if (nqh[hs] > 0) mbar_wait_drain(&qh_full[hs], (nqh[hs] - 1) & 1);
            if (ndo > 0) mbar_wait_drain(do_full, (ndo - 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0x60};
            const uint32_t tX = tmem + Cfg::kTX, tY = tmem + Cfg::kTY;
            const uint32_t tdV = tmem + Cfg::kTdV, tdK = tmem + Cfg::kTdK;
            const uint32_t aK = sbase + Cfg::kOffK, aV = sbase + Cfg::kOffV;
            const uint32_t aQ = sbase + Cfg::kOffQ, aDO = sbase + Cfg::kOffDO;
            const uint32_t aDS = sbase + Cfg::kOffDS;
            uint32_t nunit = 0, n = 0;
            bool ok = true;
#define FA_WAIT(bar, par, site)                                  \
    do {                                                         \
        w.code = kErrBwdWait + (site);                           \
        if (!mbar_wait((bar), (par), w)) { ok = false; break; } \
    } while (0)
            for (int it = 0; ok; ++it) {
                Unit256 un;
                if (!unit256_at(it, U, nT, un)) break;
                if (un.j < 0) continue;
                const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, un.bh / H);
                if (un.j * kKeys >= sp.len) continue;
                const int nQ = (sp.len + kQB - 1) / kQB;
                FA_WAIT(kv_full, nunit & 1, 0x60);
                if (!ok) break;
                const int i0 = first_qblock(un.j);
                const int eh = 1 - un.oh, lh = un.oh;
                for (int i = i0; i < nQ; ++i, ++n) {
                    // S^T over the early head-dim half first (its Q copy came in
                    // while the previous block's dK ran), which is then released
                    for (int g2 = 0; g2 < 2 && ok; ++g2) {
                        const int hs = g2 ? lh : eh;
                        FA_WAIT(&qh_full[hs], n & 1, 0x61);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int k8 = 0; k8 < 8; ++k8) {
                            const int kk = 8 * hs + k8;
                            mma_ss(tX, sdesc_sw128(aK + (kk / 4) * kBoxK + (kk % 4) * 32, 16, 1024),
                                   sdesc_sw128(aQ + (kk / 4) * kBoxQ + (kk % 4) * 32, 16, 1024),
                                   Cfg::kIdescSS, (g2 > 0 || k8 > 0) ? 1u : 0u);
                        }
                        if (g2 == 0) mma_commit(&qh_empty[eh]);  // dK reads only half lh
                    }
                    if (!ok) break;
                    mma_commit(s_full);
                    if (n > 0) {
                        FA_WAIT(dq_empty, (n - 1) & 1, 0x62);  // the drain has read dQ(n-1)
                        if (!ok) break;
                    }
                    FA_WAIT(do_full, n & 1, 0x63);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)
                        mma_ss(tY, sdesc_sw128(aV + (kk / 4) * kBoxK + (kk % 4) * 32, 16, 1024),
                               sdesc_sw128(aDO + (kk / 4) * kBoxQ + (kk % 4) * 32, 16, 1024),
                               Cfg::kIdescSS, kk > 0 ? 1u : 0u);
                    mma_commit(dp_full);
                    FA_WAIT(p_ready, n & 1, 0x64);
                    if (!ok) break;
                    if (i == i0 && nunit > 0) {
                        FA_WAIT(dkdv_empty, (nunit - 1) & 1, 0x65);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const bool acc = (i > i0);
                    // dV[:, half] += P^T dO_i[:, half]   (B MN-major, 2 boxes of 64 columns)
#pragma unroll
                    for (int kk = 0; kk < kQB / 16; ++kk)
                        mma_ts(tdV, tX + kk * 8,
                               sdesc_sw128(aDO + 2 * un.oh * kBoxQ + kk * 2048, kBoxQ, 1024),
                               Cfg::kIdescAcc, (acc || kk > 0) ? 1u : 0u);
                    mma_commit(do_empty);
                    FA_WAIT(ds_ready, n & 1, 0x66);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kQB / 16; ++kk)
                        mma_ts(tdK, tY + kk * 8,
                               sdesc_sw128(aQ + 2 * un.oh * kBoxQ + kk * 2048, kBoxQ, 1024),
                               Cfg::kIdescAcc, (acc || kk > 0) ? 1u : 0u);
                    mma_commit(&qh_empty[lh]);
                    // dQ^T[half] = K_j[:, half]^T dS^T -> Y (head dim on the lanes)
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk)
                        mma_ss(tY, sdesc_sw128(aK + 2 * un.oh * kBoxK + kk * 2048, kBoxK, 1024),
                               sdesc_sw128(aDS + kk * 2048, kBoxK, 1024), Cfg::kIdescDQ,
                               kk > 0 ? 1u : 0u);
                    mma_commit(dq_full);
                    if (i + 1 == nQ) {
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
        // ------------------------------------------------------------ P^T and dS^T (lane = key)
        const int quarter = warp & 3;
        const int kr = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tX = tmem + Cfg::kTX + lane_off, tY = tmem + Cfg::kTY + lane_off;
        const float c2 = args.scale_log2;
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0x70};
        uint32_t n = 0;
        bool ok = true;
        uint8_t *ds_row = smem + Cfg::kOffDS + kr * 128;
        for (int it = 0; ok; ++it) {
            Unit256 un;
            if (!unit256_at(it, U, nT, un)) break;
            if (un.j < 0) continue;
            const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, un.bh / H);
            if (un.j * kKeys >= sp.len) continue;
            const int nQ = (sp.len + kQB - 1) / kQB;
            const int key = un.j * kKeys + kr;
            for (int i = first_qblock(un.j); i < nQ; ++i, ++n) {
                w.code = kErrBwdWait + 0x70;
                if (!mbar_wait(&st_full[n & 1], (n >> 1) & 1, w)) { ok = false; break; }
                const float *stat = stat_base + (n & 1) * 128;
                w.code = kErrBwdWait + 0x71;
                if (!mbar_wait(s_full, n & 1, w)) { ok = false; break; }
                tc_fence_after();
                uint32_t pk[32];
                {
                    uint32_t sr[2][32];
                    tmem_ld32(tX, sr[0]);
                    tmem_ld32(tX + 32, sr[1]);
                    tmem_ld_wait(sr[0]);
                    tmem_ld_wait(sr[1]);
                    const bool diag = args.causal && (i * kQB < (un.j + 1) * kKeys);
                    if (diag || (un.j + 1) * kKeys > sp.len) {
                        const bool key_ok = key < sp.len;
                        const int q0 = i * kQB;
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (!key_ok || (diag && q0 + c * 32 + e < key))
                                    sr[c][e] = __float_as_uint(-INFINITY);
                    }
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float p0 = ex2_mufu(fmaf(__uint_as_float(sr[c][e]), c2, -stat[c * 32 + e]));
                            const float p1 =
                                ex2_mufu(fmaf(__uint_as_float(sr[c][e + 1]), c2, -stat[c * 32 + e + 1]));
                            pk[(c * 32 + e) / 2] = pack_bf16x2(p0, p1);
                        }
                }
                tmem_st16(tX, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
                tmem_st16(tX + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(p_ready);
                w.code = kErrBwdWait + 0x72;
                if (!mbar_wait(dp_full, n & 1, w)) { ok = false; break; }
                if (n > 0) {
                    w.code = kErrBwdWait + 0x73;  // dQ MMA of the previous block has read dS
                    if (!mbar_wait(dq_full, (n - 1) & 1, w)) { ok = false; break; }
                }
                tc_fence_after();
                uint32_t dr[2][32];
                tmem_ld32(tY, dr[0]);
                tmem_ld32(tY + 32, dr[1]);
                tmem_ld_wait(dr[0]);
                tmem_ld_wait(dr[1]);
                uint32_t dsw[32];
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const int col = c * 32 + e;
                        const uint32_t pw = pk[col >> 1];
                        const float d0 = __uint_as_float(pw << 16) *
                                         (__uint_as_float(dr[c][e]) - stat[64 + col]);
                        const float d1 = __uint_as_float(pw & 0xffff0000u) *
                                         (__uint_as_float(dr[c][e + 1]) - stat[64 + col + 1]);
                        dsw[col >> 1] = pack_bf16x2(d0, d1);
                    }
                tmem_st16(tY, *reinterpret_cast<uint32_t(*)[16]>(&dsw[0]));
                tmem_st16(tY + 16, *reinterpret_cast<uint32_t(*)[16]>(&dsw[16]));
                // shared copy (MN-major B of the dQ MMA): this key's 64 queries,
                // 128-byte row, 128B swizzle
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4 *>(ds_row + ((ch ^ (kr & 7)) << 4)) =
                        make_uint4(dsw[4 * ch], dsw[4 * ch + 1], dsw[4 * ch + 2], dsw[4 * ch + 3]);
                fence_proxy_async_smem();
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(ds_ready);
            }
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ dQ drain + dK/dV epilogue
        // dQ^T rows (lane = head-dim column d of the half) are staged per warp
        // as 32 queries x 32 columns (4 KB, 128B swizzle) and added into the
        // accumulator with TMA bulk reductions issued by the warp's lane 0.
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        uint8_t *stage = smem + Cfg::kOffRed + quarter * 4096;
        WaitCtx w{abort_flag, args.err_word, kErrBwdWait + 0x80};
        uint32_t n = 0, nunit = 0;
        const int nQs = (S + kQB - 1) / kQB;  // fixed-order counters per head and half
        bool ok = true;
        for (int it = 0; ok; ++it) {
            Unit256 un;
            if (!unit256_at(it, U, nT, un)) break;
            if (un.j < 0) continue;
            const int b = un.bh / H, h = un.bh % H;
            const SeqSpan sp = seq_span(args.cu_seqlens, args.T, S, b);
            if (un.j * kKeys >= sp.len) continue;
            const int nQ = (sp.len + kQB - 1) / kQB;
            // accumulator rows: [B*H, S] fixed, [H, T] packed
            const int acc_row0 = args.cu_seqlens ? sp.tok0 : 0;
            const int acc_z = args.cu_seqlens ? h : un.bh;
            for (int i = first_qblock(un.j); i < nQ; ++i, ++n) {
                w.code = kErrBwdWait + 0x80;
                if (!mbar_wait(dq_full, n & 1, w)) { ok = false; break; }
                tc_fence_after();
                uint32_t col[2][32];  // dQ^T[d][query] for 64 queries
                tmem_ld32(tmem + Cfg::kTY + lane_off, col[0]);
                tmem_ld32(tmem + Cfg::kTY + lane_off + 32, col[1]);
                tmem_ld_wait(col[0]);
                tmem_ld_wait(col[1]);
                tc_fence_before();
                mbar_arrive(dq_empty);
                // Fixed-order mode: the key tiles add their shares of this
                // (head, half, 64-query block) in ascending order, each drain
                // warp (32 columns of the half) under its own counter.  Units are
                // numbered with ascending key tiles within a head and half and
                // taken in rounds by the persistent grid, so a tile waits only
                // for units of its own round or of earlier ones (no cycle).
                int *sem = nullptr;
                bool go = true;
                if constexpr (kDet) {
                    // this warp's counter: its 32 columns of the (head, half,
                    // 64-query block)
                    sem = args.dq_sem + ((static_cast<size_t>(un.bh) * 2 + un.oh) * nQs + i) * 4 +
                          quarter;
                    if (lane == 0) {
                        w.code = kErrBwdWait + 0x82;
                        go = counter_wait_geq(sem, un.j, w);
                        fence_proxy_async_global();
                    }
                    go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (lane == 0) bulk_wait_read<0>();  // previous reduction has read `stage`
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 32; ++q)
                        *reinterpret_cast<float *>(stage + q * 128 + ((((lane >> 2) ^ (q & 7))) << 4) +
                                                   (lane & 3) * 4) = __uint_as_float(col[half][q]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && go) {
                        tma_reduce_add_3d(&args.tm_dqacc, stage, un.oh * 128 + quarter * 32,
                                          acc_row0 + i * kQB + half * 32, acc_z);
                        bulk_commit();
                    }
                }
                if (kDet && sem) {
                    // this warp's share of the block is complete in L2: its
                    // (async-proxy) reductions are ordered before the release
                    // that passes the turn on
                    if (lane == 0) {
                        bulk_wait<0>();
                        fence_proxy_async_global();
                        red_release_gpu_add(sem, 1);
                    }
                }
            }
            if (!ok) break;
            w.code = kErrBwdWait + 0x81;
            if (!mbar_wait(dkdv_full, nunit & 1, w)) { ok = false; break; }
            ++nunit;
            tc_fence_after();
            const int key = un.j * kKeys + r;  // dK / dV lanes are keys
            const size_t orow = ((static_cast<size_t>(sp.tok0) + key) * H + h) * kD + un.oh * 128;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t tsrc = tmem + lane_off + (which ? Cfg::kTdK : Cfg::kTdV);
                const float mul = which ? args.scale : 1.f;
                uint16_t *out = reinterpret_cast<uint16_t *>(which ? args.dk : args.dv) + orow;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tsrc + c * 32, v);
                    tmem_ld_wait(v);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul,
                                            __uint_as_float(v[2 * e + 1]) * mul);
                    if (key < sp.len) {
                        uint4 *dst = reinterpret_cast<uint4 *>(out + c * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2],
                                                 pk[4 * v4 + 3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(dkdv_empty);
        }
        if (lane == 0) bulk_wait<0>();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_bwd_main_d256(const BwdArgs &a, cudaStream_t stream) {
    auto kern = a.dq_sem ? fa_bwd_kernel_d256<true> : fa_bwd_kernel_d256<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long U = static_cast<long long>(a.B) * a.H * ((a.S + kKeys - 1) / kKeys) * 2;
    const int grid = static_cast<int>(U < a.num_sms ? U : a.num_sms);
    if (a.dq_sem) {
        // CTAs wait on one another's counters: all must be resident at once
        void *params[] = {const_cast<BwdArgs *>(&a)};
        e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(grid),
                                        dim3(kThreads), params, Cfg::kSmemBytes, stream);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    kern<<<grid, kThreads, Cfg::kSmemBytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace fa
