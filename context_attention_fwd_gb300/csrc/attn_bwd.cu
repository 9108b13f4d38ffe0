// attn_bwd.cu -- ring-chunked attention backward for sm_103a.
//
// One CTA owns one 128-row KV tile of ring chunk c for one (batch, kv head).
// It keeps K_c and V_c resident in shared memory and visits the query
// chunks in ring order r = (c + i) mod P, i = 0..P-1 (at iteration i query
// chunk r met KV chunk (r - i) mod P = c in the forward), for every query
// head of its GQA group.  For every (query tile, this KV tile) pair the
// probabilities are recomputed against this chunk's own K_c with the merged
// log-sum-exp of the forward -- the per-iteration K/V the backward must see
// (diffusers issue #14265, "Expected behavior"; recompute instead of saving
// per-iteration tensors) -- so the stale iteration-0 K/V defect of
// "Root cause" cannot occur: the only K/V in the CTA is K_c, V_c.
//
// Per query tile (all matrices are per (b, h), fp32 accumulation):
//   S^T  = K_c Q^T                      TMEM[S]     (M = kv, N = q, K = D)
//   P^T  = exp2(S^T * scale*log2e - lse*log2e)      -> bf16 into TMEM[S]
//   dP^T = V_c dO^T                     TMEM[dP]
//   dS^T = P^T o (dP^T - delta)         -> bf16 into shared memory
//   dV  += P^T dO                       TMEM[dV]    (A from TMEM)
//   dK  += dS^T Q                       TMEM[dK]    (A = dS^T, K-major)
//   dQ   = dS K_c                       TMEM[dP]    (A = dS, MN-major view of dS^T)
// dQ tiles are added into an fp32 accumulator in global memory (vector
// reductions); dK, dV stay in TMEM for the whole CTA and are written once.
//
// Warp roles (512 threads):
//   warps 0..7   P / dS math: one KV row per thread (TMEM lane quarter =
//                warp mod 4), warps 0..3 take query columns 0..63 and warps
//                4..7 columns 64..127; dV epilogue (half the columns each)
//   warps 8..11  dQ drain (one query row per thread); dK epilogue
//   warp 12      TMA producer (K, V once; Q, dO, lse, delta per query tile, 2 stages)
//   warp 13      TMEM owner; issues S (the product that feeds the softmax)
//   warp 15      issues dP (the product that feeds dS)
//   warp 14      issues dV, dK and dQ (the products that consume the math)
// Three MMA issuers keep the tensor core fed: while one waits on a barrier,
// the products the others have queued keep running, and S_{i+1} never waits
// behind dP_i.  Their TMEM hazards are ordered explicitly: S_{i+1} waits
// until dV_i (which reads P^T_i from the S columns) is done, dP_{i+1} until
// dQ_i (written over dP_i) has been drained.
// P^T is written back into the S^T columns it was computed from (bf16
// pairs): columns 0..31 for query columns 0..63, columns 96..127 for query
// columns 64..127, so the two math warps of a lane quarter never overwrite
// scores the other still has to read.
#include "internal.h"
#include "ptx.cuh"
#include "walk.cuh"

namespace ctxattn {
namespace {

template <int D>
struct BwdLayout {
    static constexpr int NBOX = D / 64;
    static constexpr uint32_t BOX = kTile * 128;     // 128 rows x 128 bytes
    static constexpr uint32_t TILE = kTile * D * 2;  // 128 x D bf16
    static constexpr uint32_t DS_TILE = kTile * 128 * 2;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + TILE;
    static constexpr uint32_t OFF_Q = OFF_V + TILE;          // 2 stages
    static constexpr uint32_t OFF_DO = OFF_Q + 2 * TILE;     // 2 stages
    static constexpr uint32_t OFF_DS = OFF_DO + 2 * TILE;
    static constexpr uint32_t OFF_STAT = OFF_DS + DS_TILE;   // 2 stages x (-lse2[128], delta[128])
    static constexpr uint32_t OFF_BARS = OFF_STAT + 2 * 1024;
    static constexpr uint32_t SMEM = OFF_BARS + 256;
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 384, TM_COLS = 512;
};

struct BwdBars {
    uint64_t kv_full;
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full, dp_full, p_ready, ds_ready, ds_free, dv_done;
    uint64_t dq_full, dq_drained;
    uint64_t final_mma;
    uint64_t drain, drain2, drain3;
    uint32_t tmem_slot;
    int abort_flag;
};

constexpr int kMathWarps = 8;
constexpr int kMathThreads = 32 * kMathWarps;
constexpr int kDrainThreads = 128;
constexpr int kThreads = 512;
constexpr int kProducerWarp = 12, kMmaWarp = 13, kMma2Warp = 14, kMmaDpWarp = 15;

__device__ __forceinline__ int pick3(int o, int s, int h, int b) {
    return o == 0 ? s : (o == 1 ? h : b);
}
__device__ __forceinline__ void tma_tile(const TmaMap& m, uint32_t dst, uint32_t bar, int d0, int s,
                                         int h, int b) {
    tma_load_4d(dst, &m.map, bar, d0, pick3(m.ord[0], s, h, b), pick3(m.ord[1], s, h, b),
                pick3(m.ord[2], s, h, b));
}
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) break;
}
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

template <int D, bool kHeadMajor>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
    griddep_wait();  // the previous kernel in the stream is complete (launch_kernel)
    griddep_launch_dependents();
    using L = BwdLayout<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    BwdBars& bars = *reinterpret_cast<BwdBars*>(smem + L::OFF_BARS);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sK = sbase + L::OFF_K, sV = sbase + L::OFF_V, sQ = sbase + L::OFF_Q,
                   sDO = sbase + L::OFF_DO, sDS = sbase + L::OFF_DS;
    const float* stat_base = reinterpret_cast<const float*>(smem + L::OFF_STAT);
    const int warp = warp_id(), lane = lane_id();
    const GridPos gp = grid_pos<kHeadMajor>();
    const int kt = gp.tile, hk = gp.head, b = gp.z;
    const ChunkTable& ct = p.ct;
    const int c = chunk_of_tile(ct, kt);
    const int kv_start = ct.off[c] + (kt - ct.tile_off[c]) * kTile;
    const int kv_len = min(kTile, ct.off[c + 1] - kv_start);
    const int G = p.group;
    const QWalk qw{&ct, c, p.causal, kv_start, hk * G + G};
    const int n_q = qw.count(G);  // query tiles this CTA visits (all heads of the group)
    const WaitCtx wc{&bars.abort_flag, p.status, p.timeout_ns};

    if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicExch(p.status, 2);
        return;
    }
    if (threadIdx.x == 0) {
        bars.abort_flag = 0;
        mbar_init(smem_u32(&bars.kv_full), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars.q_full[i]), 1);
            mbar_init(smem_u32(&bars.q_empty[i]), 1 + kMathWarps);  // MMA commit + one per math warp
        }
        mbar_init(smem_u32(&bars.s_full), 1);
        mbar_init(smem_u32(&bars.dp_full), 1);
        mbar_init(smem_u32(&bars.p_ready), kMathThreads);
        mbar_init(smem_u32(&bars.ds_ready), kMathThreads);
        mbar_init(smem_u32(&bars.ds_free), 1);
        mbar_init(smem_u32(&bars.dv_done), 1);
        mbar_init(smem_u32(&bars.drain2), 1);
        mbar_init(smem_u32(&bars.dq_full), 1);
        mbar_init(smem_u32(&bars.dq_drained), kDrainThreads);
        mbar_init(smem_u32(&bars.final_mma), 1);
        mbar_init(smem_u32(&bars.drain), 1);
        mbar_init(smem_u32(&bars.drain3), 1);
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&bars.tmem_slot), L::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_slot;

    // query-tile walk: ring order from chunk c (causal: tiles entirely
    // above the diagonal are skipped)
    const QTileIter q0 = qw.first(hk * G);
    auto next = [&](QTileIter& q) { qw.next(q); };
    auto q_first_row = [&](const QTileIter& q) { return qw.first_row(q); };

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tq.map);
            tma_prefetch_desc(&p.tk.map);
            tma_prefetch_desc(&p.tv.map);
            tma_prefetch_desc(&p.tdo.map);
            const uint32_t kvf = smem_u32(&bars.kv_full);
            mbar_arrive_expect_tx(kvf, 2 * L::TILE);
            for (int bx = 0; bx < L::NBOX; ++bx) {
                tma_tile(p.tk, sK + bx * L::BOX, kvf, bx * 64, kv_start, hk, b);
                tma_tile(p.tv, sV + bx * L::BOX, kvf, bx * 64, kv_start, hk, b);
            }
            QTileIter q = q0;
            int last_ph[2] = {-1, -1};
            bool ok = true;
            const int skip = debug_skip_step(p.debug, n_q);  // -1 in normal use
            for (int i = 0; i < n_q; ++i, next(q)) {
                if (i == skip) {  // failure injection: no Q, dO from query tile i on
                    ok = false;
                    break;
                }
                const int st = i & 1, ph = (i >> 1) & 1;
                if (!(ok = mbar_wait(smem_u32(&bars.q_empty[st]), ph ^ 1, wc))) break;
                const uint32_t qf = smem_u32(&bars.q_full[st]);
                mbar_arrive_expect_tx(qf, 2 * L::TILE + 1024);
                const int q_start = ct.off[q.r] + (q.t - ct.tile_off[q.r]) * kTile;
                for (int bx = 0; bx < L::NBOX; ++bx) {
                    tma_tile(p.tq, sQ + st * L::TILE + bx * L::BOX, qf, bx * 64, q_start, q.h, b);
                    tma_tile(p.tdo, sDO + st * L::TILE + bx * L::BOX, qf, bx * 64, q_start, q.h, b);
                }
                const size_t slot = ((size_t)(b * p.Hq + q.h) * ct.ntiles + q.t) * kTile;
                const uint32_t sst = sbase + L::OFF_STAT + st * 1024;
                bulk_load(sst, p.nlse2 + slot, 512, qf);
                bulk_load(sst + 512, p.delta + slot, 512, qf);
                last_ph[st] = ph;
            }
            if (!ok) {
                drain_wait(kvf, 0, p.timeout_ns);
                for (int st = 0; st < 2; ++st)
                    if (last_ph[st] >= 0) drain_wait(smem_u32(&bars.q_full[st]), last_ph[st], p.timeout_ns);
            }
        }
    } else if (warp == kMmaWarp || warp == kMma2Warp || warp == kMmaDpWarp) {
        // ---------------------------------------------------------- MMA issuers
        if (lane == 0) {
            constexpr uint32_t id_st = idesc_bf16_f32(128, 128, false, false);  // K-major A and B
            constexpr uint32_t id_dv = idesc_bf16_f32(128, D, false, true);     // A TMEM, B MN-major
            constexpr uint32_t id_dk = idesc_bf16_f32(128, D, false, true);     // A K-major smem, B MN-major
            constexpr uint32_t id_dq = idesc_bf16_f32(128, D, true, true);      // A MN-major, B MN-major
            // Loop-invariant descriptors; a k-step only advances the 14-bit
            // start-address field (address / 16), which never carries.
            const uint64_t dK_k = sdesc_sw128(sK, 16, 1024), dV_k = sdesc_sw128(sV, 16, 1024);
            const uint64_t dQ_k = sdesc_sw128(sQ, 16, 1024), dO_k = sdesc_sw128(sDO, 16, 1024);
            const uint64_t dQ_mn = sdesc_sw128(sQ, L::BOX, 1024), dO_mn = sdesc_sw128(sDO, L::BOX, 1024);
            const uint64_t dS_k = sdesc_sw128(sDS, 16, 1024), dS_mn = sdesc_sw128(sDS, L::BOX, 1024);
            const uint64_t dK_mn = sdesc_sw128(sK, L::BOX, 1024);
            constexpr uint32_t kStage = L::TILE >> 4, kMnStep = 2048 >> 4;
            auto koff = [](int kk) -> uint32_t { return ((kk >> 2) * L::BOX + (kk & 3) * 32) >> 4; };
            bool ok = mbar_wait(smem_u32(&bars.kv_full), 0, wc);
            if (warp == kMmaWarp) {
                // S_i = K Q_i^T, per query tile
                auto issue_s = [&](int st) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + L::TM_S, dK_k + koff(kk), dQ_k + st * kStage + koff(kk), id_st,
                               kk > 0 ? 1u : 0u);
                    mma_commit(smem_u32(&bars.s_full));
                };
                if (ok && (ok = mbar_wait(smem_u32(&bars.q_full[0]), 0, wc))) issue_s(0);
                for (int i = 0; i + 1 < n_q && ok; ++i) {
                    // S^T_{i+1} overwrites P^T_i: wait until dV_i has read it
                    if (!(ok = mbar_wait(smem_u32(&bars.dv_done), i & 1, wc))) break;
                    if (!(ok = mbar_wait(smem_u32(&bars.q_full[(i + 1) & 1]), ((i + 1) >> 1) & 1, wc))) break;
                    tc_fence_after();
                    issue_s((i + 1) & 1);
                }
                mma_commit(smem_u32(&bars.drain));
                drain_wait(smem_u32(&bars.drain), 0, p.timeout_ns);
            } else if (warp == kMmaDpWarp) {
                // dP_i = V dO_i^T, per query tile, from its own thread: S_{i+1}
                // does not wait behind dP_i, which waits for the drain of dQ_{i-1}
                for (int i = 0; i < n_q && ok; ++i) {
                    const int st = i & 1;
                    if (!(ok = mbar_wait(smem_u32(&bars.q_full[st]), (i >> 1) & 1, wc))) break;
                    // into the columns dQ_{i-1} occupied once it is drained
                    if (i > 0 && !(ok = mbar_wait(smem_u32(&bars.dq_drained), (i - 1) & 1, wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + L::TM_DP, dV_k + koff(kk), dO_k + st * kStage + koff(kk), id_st,
                               kk > 0 ? 1u : 0u);
                    mma_commit(smem_u32(&bars.dp_full));
                }
                mma_commit(smem_u32(&bars.drain3));
                drain_wait(smem_u32(&bars.drain3), 0, p.timeout_ns);
            } else {
                // dV_i += P^T dO, dK_i += dS^T Q, dQ_i = dS K, per query tile
                for (int i = 0; i < n_q && ok; ++i) {
                    const int st = i & 1;
                    if (!(ok = mbar_wait(smem_u32(&bars.p_ready), i & 1, wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        mma_ts(tmem + L::TM_DV, tmem + L::TM_S + (kk < 4 ? kk * 8 : 96 + (kk - 4) * 8),
                               dO_mn + st * kStage + kk * kMnStep, id_dv, (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&bars.dv_done));
                    if (!(ok = mbar_wait(smem_u32(&bars.ds_ready), i & 1, wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        mma_ss(tmem + L::TM_DK, dS_k + koff(kk), dQ_mn + st * kStage + kk * kMnStep, id_dk,
                               (i > 0 || kk > 0) ? 1u : 0u);
                    // dK_i is the last reader of Q_i and dO_i: release the stage now,
                    // half a tile before dQ_i completes, so the next load starts earlier
                    mma_commit(smem_u32(&bars.q_empty[st]));
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        mma_ss(tmem + L::TM_DP, dS_mn + kk * kMnStep, dK_mn + kk * kMnStep, id_dq,
                               kk > 0 ? 1u : 0u);
                    mma_commit(smem_u32(&bars.dq_full));
                    mma_commit(smem_u32(&bars.ds_free));
                }
                mma_commit(smem_u32(&bars.final_mma));
                mma_commit(smem_u32(&bars.drain2));
                drain_wait(smem_u32(&bars.drain2), 0, p.timeout_ns);
            }
        }
    } else if (warp < kMathWarps) {
        // ---------------------------------------------------------- P / dS math
        const int quarter = warp & 3;
        const int half = warp >> 2;            // query columns [64*half, 64*half + 64)
        const int row = quarter * 32 + lane;   // KV row of this thread
        const uint32_t taddr = tmem + (uint32_t(quarter * 32) << 16);
        const uint32_t s_cols = L::TM_S + half * 64, p_cols = L::TM_S + half * 96;
        const float sc = p.scale_log2;
        const bool row_valid = row < kv_len;
        bool ok = true;
        QTileIter q = q0;
        for (int i = 0; i < n_q; ++i, next(q)) {
            const int st = i & 1, ph = (i >> 1) & 1;
            // causal diagonal tile: query columns before this thread's key are masked
            const int q_start = q_first_row(q);
            const bool diag = p.causal && q.r == c && kv_start + kv_len - 1 > q_start;
            const int lo = diag ? kv_start + row - q_start - half * 64 : 0;  // mask columns k < lo
            const float4* nlse2 = reinterpret_cast<const float4*>(stat_base + st * 256 + half * 64);
            const float4* delta = reinterpret_cast<const float4*>(stat_base + st * 256 + 128 + half * 64);
            if (!(ok = mbar_wait(smem_u32(&bars.q_full[st]), ph, wc))) break;
            if (!(ok = mbar_wait(smem_u32(&bars.s_full), i & 1, wc))) break;
            tc_fence_after();
            uint32_t pr[64];
            tmem_ld64_sync(taddr + s_cols, pr);
            // P^T (fp32 kept in pr); padded query columns have -lse2 = -inf -> 0
            const float2 sc2 = make_float2(sc, sc);
#pragma unroll
            for (int k4 = 0; k4 < 16; ++k4) {  // query columns in pairs: two-lane fp32 instructions
                const float4 l4 = nlse2[k4];
                const float2 x0 = ffma2(make_float2(__uint_as_float(pr[4 * k4]), __uint_as_float(pr[4 * k4 + 1])), sc2,
                                        make_float2(l4.x, l4.y));
                const float2 x1 = ffma2(make_float2(__uint_as_float(pr[4 * k4 + 2]), __uint_as_float(pr[4 * k4 + 3])),
                                        sc2, make_float2(l4.z, l4.w));
                pr[4 * k4 + 0] = __float_as_uint(ex2(x0.x));
                pr[4 * k4 + 1] = __float_as_uint(ex2(x0.y));
                pr[4 * k4 + 2] = __float_as_uint(ex2(x1.x));
                pr[4 * k4 + 3] = __float_as_uint(ex2(x1.y));
            }
            if (diag || kv_len < kTile) {  // tile-uniform: only edge tiles pay for masking
                const int lo_eff = row_valid ? lo : 64;  // zero columns k < lo_eff
#pragma unroll
                for (int k = 0; k < 64; ++k)
                    if (k < lo_eff) pr[k] = 0u;
            }
            {
                uint32_t pk[32];
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    pk[k] = pack_bf16x2(__uint_as_float(pr[2 * k]), __uint_as_float(pr[2 * k + 1]));
                tmem_st32(taddr + p_cols, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars.p_ready));
            // dS^T = P^T o (dP^T - delta), to shared memory as bf16
            if (!(ok = mbar_wait(smem_u32(&bars.dp_full), i & 1, wc))) break;
            if (i > 0 && !(ok = mbar_wait(smem_u32(&bars.ds_free), (i - 1) & 1, wc))) break;
            tc_fence_after();
            const uint32_t box = sDS + half * L::BOX;  // this half's 64 query columns
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t dp[32];
                tmem_ld32_sync(taddr + L::TM_DP + half * 64 + cc * 32, dp);
                uint32_t w[16];
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) {
                    const float4 d4 = delta[cc * 8 + k4];
                    const int q0 = cc * 32 + 4 * k4;
                    const float2 a01 = fmul2(make_float2(__uint_as_float(pr[q0]), __uint_as_float(pr[q0 + 1])),
                                             fsub2(make_float2(__uint_as_float(dp[4 * k4]), __uint_as_float(dp[4 * k4 + 1])),
                                                   make_float2(d4.x, d4.y)));
                    const float2 a23 = fmul2(make_float2(__uint_as_float(pr[q0 + 2]), __uint_as_float(pr[q0 + 3])),
                                             fsub2(make_float2(__uint_as_float(dp[4 * k4 + 2]), __uint_as_float(dp[4 * k4 + 3])),
                                                   make_float2(d4.z, d4.w)));
                    w[2 * k4] = pack_bf16x2(a01.x, a01.y);
                    w[2 * k4 + 1] = pack_bf16x2(a23.x, a23.y);
                }
                // 32 query columns = four 16-byte chunks of the 128-byte swizzled row
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t addr = box + sw128_offset(row, cc * 4 + m);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[4 * m]),
                                 "r"(w[4 * m + 1]), "r"(w[4 * m + 2]), "r"(w[4 * m + 3])
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars.ds_ready));
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.q_empty[st]));
        }
        // ---------------------------------------------------------- dV epilogue
        if (ok && mbar_wait(smem_u32(&bars.final_mma), 0, wc)) {
            tc_fence_after();
            constexpr int kHalfCols = D / 2;
            __nv_bfloat16* dst = p.dv + (int64_t)b * p.k_sb + (int64_t)(kv_start + row) * p.k_ss +
                                 (int64_t)hk * p.k_sh + half * kHalfCols;
#pragma unroll
            for (int cc = 0; cc < kHalfCols / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32_sync(taddr + L::TM_DV + half * kHalfCols + cc * 32, o);
                if (row_valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        d4[k] = make_uint4(
                            pack_bf16x2(__uint_as_float(o[8 * k + 0]), __uint_as_float(o[8 * k + 1])),
                            pack_bf16x2(__uint_as_float(o[8 * k + 2]), __uint_as_float(o[8 * k + 3])),
                            pack_bf16x2(__uint_as_float(o[8 * k + 4]), __uint_as_float(o[8 * k + 5])),
                            pack_bf16x2(__uint_as_float(o[8 * k + 6]), __uint_as_float(o[8 * k + 7])));
                }
            }
        }
    } else if (warp < kMathWarps + 4) {
        // ---------------------------------------------------------- dQ drain
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // query row of the current tile
        const uint32_t taddr = tmem + (uint32_t(quarter * 32) << 16);
        QTileIter q = q0;
        bool ok = true;
        for (int i = 0; i < n_q; ++i, next(q)) {
            if (!(ok = mbar_wait(smem_u32(&bars.dq_full), i & 1, wc))) break;
            tc_fence_after();
            // tile-major accumulator: [(b,h,t)][D/4][128 rows][4]
            float* tile = p.dq_acc + ((size_t)(b * p.Hq + q.h) * ct.ntiles + q.t) * (size_t)(kTile * D);
            // 64 columns at a time; the TMEM columns are released after the last load
#pragma unroll
            for (int hc = 0; hc < D / 64; ++hc) {
                uint32_t v[64];
                tmem_ld64_sync(taddr + L::TM_DP + hc * 64, v);
                if (hc == D / 64 - 1) {
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bars.dq_drained));
                }
#pragma unroll
                for (int g = 0; g < 16; ++g)
                    red_add_v4(tile + ((size_t)(hc * 16 + g) * kTile + row) * 4, __uint_as_float(v[4 * g]),
                               __uint_as_float(v[4 * g + 1]), __uint_as_float(v[4 * g + 2]),
                               __uint_as_float(v[4 * g + 3]));
            }
        }
        // ---------------------------------------------------------- dK epilogue
        if (ok && mbar_wait(smem_u32(&bars.final_mma), 0, wc)) {
            tc_fence_after();
            const bool row_valid = row < kv_len;
            __nv_bfloat16* dst =
                p.dk + (int64_t)b * p.k_sb + (int64_t)(kv_start + row) * p.k_ss + (int64_t)hk * p.k_sh;
            const float scale = p.scale;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32_sync(taddr + L::TM_DK + cc * 32, o);
                if (row_valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        d4[k] = make_uint4(
                            pack_bf16x2(__uint_as_float(o[8 * k + 0]) * scale, __uint_as_float(o[8 * k + 1]) * scale),
                            pack_bf16x2(__uint_as_float(o[8 * k + 2]) * scale, __uint_as_float(o[8 * k + 3]) * scale),
                            pack_bf16x2(__uint_as_float(o[8 * k + 4]) * scale, __uint_as_float(o[8 * k + 5]) * scale),
                            pack_bf16x2(__uint_as_float(o[8 * k + 6]) * scale, __uint_as_float(o[8 * k + 7]) * scale));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, L::TM_COLS);
}

template <int D, bool kHeadMajor>
int launch_bwd_do(const BwdParams& p, cudaStream_t s) {
    using L = BwdLayout<D>;
    static OncePerDevice attr;
    if (!attr.run([] {
            return cudaFuncSetAttribute(attn_bwd_kernel<D, kHeadMajor>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        L::SMEM) == cudaSuccess;
        }))
        return 4;
    const cudaError_t e = launch_kernel(p.pdl != 0, attn_bwd_kernel<D, kHeadMajor>,
                                        grid_dims(kHeadMajor, p.ct.ntiles, p.Hkv, p.B), dim3(kThreads), L::SMEM, s, p);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? 0 : 4;
}

template <int D>
int launch_bwd_d(const BwdParams& p, cudaStream_t s) {
    return p.head_major ? launch_bwd_do<D, true>(p, s) : launch_bwd_do<D, false>(p, s);
}

}  // namespace

int launch_attn_bwd(const BwdParams& p, int D, cudaStream_t s) {
    if (D == 64) return launch_bwd_d<64>(p, s);
    if (D == 128) return launch_bwd_d<128>(p, s);
    if (D == 256) return launch_attn_bwd256(p, s);
    return 2;
}

}  // namespace ctxattn
