// attn_d256.cu -- ring-chunked attention forward and backward for head
// dimension 256 on sm_103a.
//
// Same method and walks as the D = 64 / 128 kernels (attn_fwd.cu,
// attn_bwd.cu); what changes is the budget.  A 128 x 256 bf16 tile is 64 KB
// and a 128 x 256 fp32 accumulator fills half of TMEM, so:
//   * forward: one 128-row query tile per CTA; TMEM holds two score buffers
//     (S_0, S_1: 128 columns each) and O (256 columns), so S(j+1) is computed
//     while the softmax of tile j runs; two threads issue the products (S
//     from one, PV from the other) so that both reach the tensor core at
//     once.  K and V stream through a ring of 32 KB slots, loaded by two
//     threads: K(j) as two column halves (the two halves of the QK^T
//     contraction), V(j) as two 64-row halves (the two halves of the PV
//     contraction, N = 256 each).
//   * backward: dK and dV of one KV tile do not fit in TMEM together with
//     S^T and dP^T (4 x 256 columns), so each KV tile is split over two CTAs
//     by column half h of dK, dV and dQ.  Both recompute S^T and dP^T over
//     the full 256-column contraction; TMEM is then S^T, dP^T (later dQ_h),
//     dV_h, dK_h = 4 x 128 columns as in the D = 128 kernel.  K stays
//     resident; Q, V and dO stream through a ring of 32 KB column-half slots
//     loaded by two threads.  Warps 0..7 do the P / dS math, 8..11 drain dQ_h,
//     12 and 15 load, 13 issues S^T and dP^T, 14 dV_h, dK_h and dQ_h.
//     Short sequences give few KV tiles, so the query heads of a GQA group
//     may further be split over hsplit CTAs, which then write fp32 partial
//     dK/dV rows for a separate summing kernel.
#include "internal.h"
#include "ptx.cuh"
#include "walk.cuh"

namespace ctxattn {
namespace {

constexpr int kD = 256;
constexpr uint32_t kBox = kTile * 128;  // 128 rows x 128 bytes (64 columns), 128-byte swizzle
constexpr uint32_t kSlot = 32768;       // one ring slot: half of a 128 x 256 bf16 tile

__device__ __forceinline__ int pick3(int o, int s, int h, int b) {
    return o == 0 ? s : (o == 1 ? h : b);
}
__device__ __forceinline__ void tma_tile(const TmaMap& m, uint32_t dst, uint32_t bar, int d0, int s, int h,
                                         int b) {
    tma_load_4d(dst, &m.map, bar, d0, pick3(m.ord[0], s, h, b), pick3(m.ord[1], s, h, b),
                pick3(m.ord[2], s, h, b));
}
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) break;
}
// k-step kk (16 columns) of a K-major operand made of 64-column boxes
__device__ __forceinline__ uint32_t kmajor_koff(int kk) {
    return ((kk >> 2) * kBox + (kk & 3) * 32) >> 4;
}

// =================================================================== forward
struct F256 {
    static constexpr int SLOTS = 5;
    static constexpr uint32_t OFF_Q = 0;                         // 4 boxes (columns 64e..64e+63)
    static constexpr uint32_t OFF_RING = 4 * kBox;               // 64 KB
    static constexpr uint32_t END = OFF_RING + SLOTS * kSlot;    // 224 KB
    static constexpr uint32_t SMEM = END + 1024;                 // + alignment slack
    static constexpr uint32_t TM_S = 0, TM_O = 256, TM_COLS = 512;
    static constexpr int LOADS = 4;                              // ring loads per KV tile
};
struct F256Bars {
    uint64_t q_full;
    uint64_t full[F256::SLOTS], empty[F256::SLOTS];
    uint64_t s_full[2];  // S buffer b holds S(j) for j = b mod 2
    // P(j) (and any O rescale) written by the softmax threads, one barrier per
    // score buffer: with S(j+1) already computed, the softmax may finish tile
    // j+1 before the issuer has waited for tile j, so a single barrier could
    // complete two phases and its parity would no longer identify tile j
    uint64_t p_full[2];
    uint64_t pv_done;    // one completion per PV product
    uint64_t pv_buf[2];  // PV(j) done, per score buffer j mod 2 (S(j+2) may overwrite P(j))
    uint64_t o_done;     // the last PV of a chunk (partials) or of the walk
    uint64_t drain, drain_s;
};
// warps 0 and 3 load, warp 1 TMEM + PV products, warp 2 S products, warps 4..7 softmax
constexpr int kF256Threads = 256;
constexpr float kRescaleThreshold = 8.0f;

template <bool kPartials, bool kHeadMajor>
__global__ void __launch_bounds__(kF256Threads, 1) attn_fwd256_kernel(const __grid_constant__ FwdParams p) {
    griddep_wait();  // the previous kernel in the stream is complete (launch_kernel)
    griddep_launch_dependents();
    using L = F256;
    extern __shared__ uint8_t smem_raw[];
    __shared__ F256Bars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = sbase + L::OFF_Q, sRing = sbase + L::OFF_RING;
    const int warp = warp_id(), lane = lane_id();
    const ChunkTable& ct = p.ct;
    // the last tiles carry the most work under causal masking: launch them first
    const GridPos gp = grid_pos<kHeadMajor>();
    const int tq = ct.ntiles - 1 - gp.tile, h = gp.head, b = gp.z;
    const int r = chunk_of_tile(ct, tq);
    const int q_start = ct.off[r] + (tq - ct.tile_off[r]) * kTile;
    const int q_rows = min(kTile, ct.off[r + 1] - q_start);
    const int hk = h / p.group;
    const WalkCfg g{r, ct.P, p.causal, p.allgather, q_start + q_rows - 1};
    const int n_kv = kv_count(ct, g);
    const WaitCtx wc{&abort_flag, p.status, p.timeout_ns};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bars.q_full), 1);
        for (int i = 0; i < L::SLOTS; ++i) {
            mbar_init(smem_u32(&bars.full[i]), 1);
            mbar_init(smem_u32(&bars.empty[i]), 1);
        }
        mbar_init(smem_u32(&bars.s_full[0]), 1);
        mbar_init(smem_u32(&bars.s_full[1]), 1);
        mbar_init(smem_u32(&bars.p_full[0]), 128);  // every softmax thread
        mbar_init(smem_u32(&bars.p_full[1]), 128);
        mbar_init(smem_u32(&bars.pv_done), 1);
        mbar_init(smem_u32(&bars.pv_buf[0]), 1);
        mbar_init(smem_u32(&bars.pv_buf[1]), 1);
        mbar_init(smem_u32(&bars.o_done), 1);
        mbar_init(smem_u32(&bars.drain), 1);
        mbar_init(smem_u32(&bars.drain_s), 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), L::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0 || warp == 3) {
        // ---------------------------------------------------------- producers
        // Two loading threads: one thread's bulk copies stream at about 35 B per
        // clock into its CTA, two at twice that.  Each ring slot belongs to one
        // of them (warp 0: even slots, warp 3: odd slots), so the loads of a
        // slot are issued in order and a slot's empty barrier is never waited
        // on more than one phase ahead.
        if (lane == 0) {
            const int me = warp == 0 ? 0 : 1;
            tma_prefetch_desc(&p.tk.map);
            tma_prefetch_desc(&p.tv.map);
            const uint32_t qf = smem_u32(&bars.q_full);
            if (me == 0) {
                tma_prefetch_desc(&p.tq.map);
                mbar_arrive_expect_tx(qf, 4 * kBox);
                for (int e = 0; e < 4; ++e) tma_tile(p.tq, sQ + e * kBox, qf, e * 64, q_start, h, b);
            }
            int last[L::SLOTS];
            for (int i = 0; i < L::SLOTS; ++i) last[i] = -1;
            bool ok = true;
            const int skip = debug_skip_step(p.debug, n_kv);  // -1 in normal use
            KvWalk w;
            kv_first(ct, g, w);
            for (int j = 0; j < n_kv && ok; ++j, kv_next(ct, g, w)) {
                if (j == skip) {  // failure injection: no K, V from step j on
                    ok = false;
                    break;
                }
                const int kv_start = ct.off[w.c] + (w.t - w.t0) * kTile;
                for (int k = 0; k < L::LOADS; ++k) {
                    const int n = j * L::LOADS + k, slot = n % L::SLOTS, ph = (n / L::SLOTS) & 1;
                    if ((slot & 1) != me) continue;
                    if (!(ok = mbar_wait(smem_u32(&bars.empty[slot]), ph ^ 1, wc))) break;
                    const uint32_t f = smem_u32(&bars.full[slot]), dst = sRing + slot * kSlot;
                    mbar_arrive_expect_tx(f, kSlot);
                    if (k < 2) {  // K columns [128k, 128k + 128): two 64-column boxes of 128 rows
                        for (int e = 0; e < 2; ++e)
                            tma_tile(p.tk, dst + e * kBox, f, (2 * k + e) * 64, kv_start, hk, b);
                    } else {      // V rows [64(k-2), +64), all 256 columns: four boxes of 64 rows
                        for (int e = 0; e < 4; ++e)
                            tma_tile(p.tv, dst + e * (kBox / 2), f, e * 64, kv_start + (k - 2) * 64, hk, b);
                    }
                    last[slot] = ph;
                }
            }
            if (!ok) {
                if (me == 0) drain_wait(qf, 0, p.timeout_ns);
                for (int i = 0; i < L::SLOTS; ++i)
                    if (last[i] >= 0) drain_wait(smem_u32(&bars.full[i]), last[i], p.timeout_ns);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------------------------------------------------- MMA issuers
        // Two issuing threads.  Warp 2 issues S(j) = Q K(j)^T into score buffer
        // j mod 2 as soon as that buffer is free (PV(j-2) has read P(j-2));
        // warp 1 issues PV(j) once the softmax has written P(j).  S(j+1) and
        // PV(j) thus reach the tensor core from two threads at once, which it
        // runs at its full rate; one thread issuing both in turn left it idle
        // between products.
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t id_pv = idesc_bf16_f32(128, kD, false, true);
            const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
            const uint64_t dk0 = sdesc_sw128(sRing, 16, 1024);
            const uint64_t dv0 = sdesc_sw128(sRing, kBox / 2, 1024);  // 64-column blocks of 64 rows
            auto wait_full = [&](int n) {
                return mbar_wait(smem_u32(&bars.full[n % L::SLOTS]), (n / L::SLOTS) & 1, wc);
            };
            bool ok = true;
            if (warp == 2) {
                auto issue_s = [&](int j) -> bool {  // S(j) = Q K(j)^T into buffer j mod 2
                    const int n0 = j * L::LOADS;
                    const uint32_t d = tmem + L::TM_S + (j & 1) * 128;
                    for (int e = 0; e < 2; ++e) {
                        if (!wait_full(n0 + e)) return false;
                        tc_fence_after();
                        const uint64_t bk = dk0 + ((((n0 + e) % L::SLOTS) * kSlot) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(d, dq0 + kmajor_koff(8 * e + kk), bk + kmajor_koff(kk), id_s,
                                   (e > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&bars.s_full[j & 1]));
                    mma_commit(smem_u32(&bars.empty[n0 % L::SLOTS]));
                    mma_commit(smem_u32(&bars.empty[(n0 + 1) % L::SLOTS]));
                    return true;
                };
                ok = mbar_wait(smem_u32(&bars.q_full), 0, wc);
                for (int j = 0; j < n_kv && ok; ++j) {
                    // buffer j mod 2 holds P(j-2) until PV(j-2) has read it
                    if (j >= 2 && !(ok = mbar_wait(smem_u32(&bars.pv_buf[j & 1]), ((j - 2) >> 1) & 1, wc))) break;
                    ok = issue_s(j);
                }
                if (!ok) abort_flag = 1;
                mma_commit(smem_u32(&bars.drain_s));
                drain_wait(smem_u32(&bars.drain_s), 0, p.timeout_ns);
            } else {
                KvWalk w;
                kv_first(ct, g, w);
                for (int j = 0; j < n_kv && ok; ++j, kv_next(ct, g, w)) {
                    const bool first_c = w.t == w.t0, last_c = kv_chunk_last(ct, g, w);
                    const bool acc0 = kPartials ? !first_c : j > 0;
                    if (!(ok = mbar_wait(smem_u32(&bars.p_full[j & 1]), (j >> 1) & 1, wc))) break;
                    tc_fence_after();
                    const int n0 = j * L::LOADS + 2;
                    const uint32_t pa = tmem + L::TM_S + (j & 1) * 128;  // P(j), bf16 pairs
                    for (int e = 0; e < 2; ++e) {  // O += P[:, 64e:64e+64] V[64e:64e+64, :]
                        if (!(ok = wait_full(n0 + e))) break;
                        tc_fence_after();
                        const uint64_t bv = dv0 + ((((n0 + e) % L::SLOTS) * kSlot) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ts(tmem + L::TM_O, pa + 32 * e + 8 * kk, bv + kk * (2048 >> 4), id_pv,
                                   (acc0 || e > 0 || kk > 0) ? 1u : 0u);
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&bars.empty[n0 % L::SLOTS]));
                    mma_commit(smem_u32(&bars.empty[(n0 + 1) % L::SLOTS]));
                    mma_commit(smem_u32(&bars.pv_done));
                    mma_commit(smem_u32(&bars.pv_buf[j & 1]));
                    if (kPartials ? last_c : j == n_kv - 1) mma_commit(smem_u32(&bars.o_done));
                }
                if (!ok) abort_flag = 1;
                mma_commit(smem_u32(&bars.drain));
                drain_wait(smem_u32(&bars.drain), 0, p.timeout_ns);
            }
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------- softmax
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t taddr = tmem + (uint32_t(quarter * 32) << 16);
        const float sc = p.scale_log2;
        const bool valid = row < q_rows;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        KvWalk w;
        kv_first(ct, g, w);
        for (int j = 0; j < n_kv; ++j, kv_next(ct, g, w)) {
            const int kv_start = ct.off[w.c] + (w.t - w.t0) * kTile;
            const int kv_len = min(kTile, ct.off[w.c + 1] - kv_start);
            const bool first = kPartials ? (w.t == w.t0) : (j == 0);
            const bool diag = g.causal && kv_start + kv_len - 1 > q_start;
            const int lim = diag ? max(0, min(kv_len, q_start + row - kv_start + 1)) : kv_len;
            const uint32_t s_cols = L::TM_S + (j & 1) * 128;
            if (!(ok = mbar_wait(smem_u32(&bars.s_full[j & 1]), (j >> 1) & 1, wc))) break;
            tc_fence_after();
            uint32_t s[128];
            tmem_ld128_sync(taddr + s_cols, s);
            if (kv_len < kTile || diag) {
#pragma unroll
                for (int k = 0; k < 128; ++k)
                    if (k >= lim) s[k] = __float_as_uint(-INFINITY);
            }
            float mx8[8];  // eight running maxima, three-input max
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(__uint_as_float(s[e]), __uint_as_float(s[120 + e]));
#pragma unroll
            for (int k = 8; k < 120; k += 16)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    mx8[e] = fmax3(mx8[e], __uint_as_float(s[k + e]), __uint_as_float(s[k + 8 + e]));
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            if (first) {
                m_ref = -INFINITY;
                l = 0.f;
            }
            float alpha = 1.f;
            bool rescale = false;
            if (mx > m_ref) {
                if (m_ref == -INFINITY) {
                    m_ref = mx;
                } else if ((mx - m_ref) * sc > kRescaleThreshold) {
                    alpha = ex2((m_ref - mx) * sc);
                    m_ref = mx;
                    rescale = true;
                }
            }
            const float neg = m_ref == -INFINITY ? 0.f : -m_ref * sc;
            // columns in pairs (two-lane fp32 instructions); four running pair sums
            const float2 sc2 = make_float2(sc, sc), neg2 = make_float2(neg, neg);
            float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                              make_float2(0.f, 0.f)};
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                const float2 x = ffma2(make_float2(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1])), sc2, neg2);
                const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                sum4[k & 3] = fadd2(sum4[k & 3], pp);
                s[k] = pack_bf16x2(pp.x, pp.y);
            }
            tmem_st32(taddr + s_cols + 0, s);
            tmem_st32(taddr + s_cols + 32, s + 32);
            const float sum = ((sum4[0].x + sum4[0].y) + (sum4[1].x + sum4[1].y)) +
                              ((sum4[2].x + sum4[2].y) + (sum4[3].x + sum4[3].y));
            l = l * alpha + sum;
            if (__any_sync(0xffffffffu, rescale)) {
                // O must hold PV(j-1) before it is rescaled.  At this point
                // PV(j-2) has completed (S(j) was issued after it), so the
                // parity of completion j-1 is unambiguous.
                if (!(ok = mbar_wait(smem_u32(&bars.pv_done), (j - 1) & 1, wc))) break;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < kD / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32_sync(taddr + L::TM_O + cc * 32, o);
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    tmem_st32(taddr + L::TM_O + cc * 32, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars.p_full[j & 1]));
            if (kPartials && kv_chunk_last(ct, g, w)) {
                const int it = w.it;
                if (!(ok = mbar_wait(smem_u32(&bars.o_done), it & 1, wc))) break;
                tc_fence_after();
                const float inv_l = 1.f / l;
                const size_t prow = ((size_t)(it * p.B + b) * p.Hq + h) * p.S + q_start + row;
#pragma unroll
                for (int cc = 0; cc < kD / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32_sync(taddr + L::TM_O + cc * 32, o);
                    if (valid) {
                        float4* dst = reinterpret_cast<float4*>(p.part_o + prow * kD + cc * 32);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv_l, __uint_as_float(o[4 * k + 1]) * inv_l,
                                                 __uint_as_float(o[4 * k + 2]) * inv_l,
                                                 __uint_as_float(o[4 * k + 3]) * inv_l);
                    }
                }
                if (valid) p.part_lse[prow] = m_ref * p.scale + logf(l);
                tc_fence_before();
            }
        }
        if (ok && !kPartials) {
            ok = mbar_wait(smem_u32(&bars.o_done), 0, wc);
            tc_fence_after();
            if (ok) {
                const float inv_l = 1.f / l;
                __nv_bfloat16* dst_row =
                    p.out + (int64_t)b * p.o_sb + (int64_t)(q_start + row) * p.o_ss + (int64_t)h * p.o_sh;
#pragma unroll
                for (int cc = 0; cc < kD / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32_sync(taddr + L::TM_O + cc * 32, o);
                    if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(dst_row + cc * 32);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            dst[k] = make_uint4(
                                pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l),
                                pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l),
                                pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l),
                                pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l));
                    }
                }
                if (valid) p.lse[((int64_t)b * p.Hq + h) * p.S + q_start + row] = m_ref * p.scale + logf(l);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::TM_COLS);
}


// ================================================================== backward
struct B256 {
    static constexpr int SLOTS = 4;
    static constexpr int LOADS = 6;  // ring loads per query tile (see the producer)
    static constexpr uint32_t DS_TILE = kTile * 128 * 2;
    static constexpr uint32_t OFF_K = 0;                          // resident K: 4 boxes
    static constexpr uint32_t OFF_RING = OFF_K + 4 * kBox;        // 64 KB
    static constexpr uint32_t OFF_DS = OFF_RING + SLOTS * kSlot;  // 192 KB
    static constexpr uint32_t OFF_STAT = OFF_DS + DS_TILE;        // 2 stages x (-lse2[128], delta[128])
    static constexpr uint32_t OFF_BARS = OFF_STAT + 2 * 1024;
    static constexpr uint32_t SMEM = OFF_BARS + 256;
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 384, TM_COLS = 512;
};
struct B256Bars {
    uint64_t k_full;
    uint64_t full[B256::SLOTS], empty[B256::SLOTS];
    uint64_t s_full, dp_full, p_ready, ds_ready, ds_free, dv_done;
    uint64_t dq_full, dq_drained;
    uint64_t final_mma;
    uint64_t drain, drain2;
    uint32_t tmem_slot;
    int abort_flag;
};
static_assert(sizeof(B256Bars) <= 256, "barrier block");
constexpr int kB256MathWarps = 8, kB256MathThreads = 256, kB256DrainThreads = 128;
constexpr int kB256Threads = 512;
constexpr int kB256Producer = 12, kB256MmaX = 13, kB256MmaY = 14, kB256Producer2 = 15;

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Ring loads of query tile i (column half h of this CTA), in this order:
//   0: Q[:, other half]   1: V[:, other half]   2: dO[:, other half]
//   3: Q[:, half h] (+ -lse2, delta)   4: V[:, half h]   5: dO[:, half h]
// Load n goes to slot n mod 4 and waits for the release of load n - 4; the
// releases happen in the order S part A (0), dP part A (1, 2), dK (3),
// dP part B (4), dV (5), so no load waits on a product that needs it.  Two
// threads issue the loads (one thread's bulk copies stream at about 35 B per
// clock into its CTA, two at twice that): warp 12 those of slots 0 and 2,
// warp 15 those of slots 1 and 3, each in load order, so the loads of a slot
// stay in order and its empty barrier is never waited on a phase ahead.
// Q_h is read by S part B and dK, dO_h by dP part B and dV: a slot is free
// once each product that reads it has completed (two releases per load, one
// per reader), whichever thread then refills it.
template <bool kHeadMajor>
__global__ void __launch_bounds__(kB256Threads, 1) attn_bwd256_kernel(const __grid_constant__ BwdParams p) {
    griddep_wait();  // the previous kernel in the stream is complete (launch_kernel)
    griddep_launch_dependents();
    using L = B256;
    extern __shared__ __align__(1024) uint8_t smem[];
    B256Bars& bars = *reinterpret_cast<B256Bars*>(smem + L::OFF_BARS);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sK = sbase + L::OFF_K, sRing = sbase + L::OFF_RING, sDS = sbase + L::OFF_DS;
    const float* stat_base = reinterpret_cast<const float*>(smem + L::OFF_STAT);
    const int warp = warp_id(), lane = lane_id();
    // Head-major grid (kv heads, 2 (b * hsplit + split) + column half, tiles);
    // tile-major grid (2 tile + column half, kv heads, b * hsplit + split):
    // there the two column halves of a KV tile are launched side by side and
    // stream the same Q, dO and V tiles at the same time, so the second read
    // of each tile hits in L2.
    const int kt = kHeadMajor ? (int)blockIdx.z : (int)(blockIdx.x >> 1);
    const int hk = kHeadMajor ? (int)blockIdx.x : (int)blockIdx.y;
    const int hh = kHeadMajor ? (int)(blockIdx.y & 1) : (int)(blockIdx.x & 1);
    const int zs = kHeadMajor ? (int)(blockIdx.y >> 1) : (int)blockIdx.z;  // b * hsplit + split
    const int b = zs / p.hsplit, split = zs % p.hsplit;
    const ChunkTable& ct = p.ct;
    const int c = chunk_of_tile(ct, kt);
    const int kv_start = ct.off[c] + (kt - ct.tile_off[c]) * kTile;
    const int kv_len = min(kTile, ct.off[c + 1] - kv_start);
    const int Gs = p.group / p.hsplit;       // query heads of this CTA
    const int h0 = hk * p.group + split * Gs;
    const QWalk qw{&ct, c, p.causal, kv_start, h0 + Gs};
    const int n_q = qw.count(Gs);
    const WaitCtx wc{&bars.abort_flag, p.status, p.timeout_ns};

    if (sbase & 1023u) {
        if (threadIdx.x == 0) atomicExch(p.status, 2);
        return;
    }
    if (threadIdx.x == 0) {
        bars.abort_flag = 0;
        mbar_init(smem_u32(&bars.k_full), 1);
        for (int i = 0; i < L::SLOTS; ++i) {
            mbar_init(smem_u32(&bars.full[i]), 1);
            mbar_init(smem_u32(&bars.empty[i]), 2);  // two releases per load (see the producers)
        }
        mbar_init(smem_u32(&bars.s_full), 1);
        mbar_init(smem_u32(&bars.dp_full), 1);
        mbar_init(smem_u32(&bars.p_ready), kB256MathThreads);
        mbar_init(smem_u32(&bars.ds_ready), kB256MathThreads);
        mbar_init(smem_u32(&bars.ds_free), 1);
        mbar_init(smem_u32(&bars.dv_done), 1);
        mbar_init(smem_u32(&bars.dq_full), 1);
        mbar_init(smem_u32(&bars.dq_drained), kB256DrainThreads);
        mbar_init(smem_u32(&bars.final_mma), 1);
        mbar_init(smem_u32(&bars.drain), 1);
        mbar_init(smem_u32(&bars.drain2), 1);
        mbar_fence_init();
    }
    if (warp == kB256MmaX) {
        tmem_alloc(smem_u32(&bars.tmem_slot), L::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_slot;
    const QTileIter q0 = qw.first(h0);
    // fp32 partial rows of this CTA's (split, b, hk) when the group is split
    float* const part_row = p.dkv_part
        ? p.dkv_part + ((((size_t)(split * p.B + b) * p.Hkv + hk) * p.S + kv_start) * 2) * kD + hh * 128
        : nullptr;
    auto slot_of = [](int n) { return n % L::SLOTS; };
    auto phase_of = [](int n) { return (n / L::SLOTS) & 1; };
    auto full_bar = [&](int n) { return smem_u32(&bars.full[n % L::SLOTS]); };
    auto empty_bar = [&](int n) { return smem_u32(&bars.empty[n % L::SLOTS]); };

    if (warp == kB256Producer || warp == kB256Producer2) {
        // ---------------------------------------------------------- producers
        if (lane == 0) {
            const int me = warp == kB256Producer ? 0 : 1;
            tma_prefetch_desc(&p.tq.map);
            tma_prefetch_desc(&p.tv.map);
            tma_prefetch_desc(&p.tdo.map);
            const uint32_t kf = smem_u32(&bars.k_full);
            if (me == 0) {
                tma_prefetch_desc(&p.tk.map);
                mbar_arrive_expect_tx(kf, 4 * kBox);
                for (int e = 0; e < 4; ++e) tma_tile(p.tk, sK + e * kBox, kf, e * 64, kv_start, hk, b);
            }
            QTileIter q = q0;
            int last[L::SLOTS] = {-1, -1, -1, -1};
            bool ok = true;
            const int skip = debug_skip_step(p.debug, n_q);  // -1 in normal use
            for (int i = 0; i < n_q && ok; ++i, qw.next(q)) {
                if (i == skip) {  // failure injection: no loads from query tile i on
                    ok = false;
                    break;
                }
                const int q_start = qw.first_row(q);
                for (int k = 0; k < L::LOADS; ++k) {
                    const int n = i * L::LOADS + k;
                    if ((slot_of(n) & 1) != me) continue;
                    if (!(ok = mbar_wait(empty_bar(n), phase_of(n) ^ 1, wc))) break;
                    const uint32_t f = full_bar(n), dst = sRing + slot_of(n) * kSlot;
                    const int half = k < 3 ? 1 - hh : hh;
                    const TmaMap& m = (k % 3 == 0) ? p.tq : (k % 3 == 1) ? p.tv : p.tdo;
                    const int row0 = (k % 3 == 1) ? kv_start : q_start;  // V rows are this CTA's keys
                    const int hsel = (k % 3 == 1) ? hk : q.h;
                    mbar_arrive_expect_tx(f, kSlot + (k == 3 ? 1024 : 0));
                    for (int e = 0; e < 2; ++e) tma_tile(m, dst + e * kBox, f, (2 * half + e) * 64, row0, hsel, b);
                    if (k == 3) {
                        const size_t slot = ((size_t)(b * p.Hq + q.h) * ct.ntiles + q.t) * kTile;
                        const uint32_t sst = sbase + L::OFF_STAT + (i & 1) * 1024;
                        bulk_load(sst, p.nlse2 + slot, 512, f);
                        bulk_load(sst + 512, p.delta + slot, 512, f);
                    }
                    last[slot_of(n)] = phase_of(n);
                }
            }
            if (!ok) {
                if (me == 0) drain_wait(kf, 0, p.timeout_ns);
                for (int s = 0; s < L::SLOTS; ++s)
                    if (last[s] >= 0) drain_wait(smem_u32(&bars.full[s]), last[s], p.timeout_ns);
            }
        }
    } else if (warp == kB256MmaX || warp == kB256MmaY) {
        // ---------------------------------------------------------- MMA issuers
        if (lane == 0) {
            constexpr uint32_t id_st = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t id_dv = idesc_bf16_f32(128, 128, false, true);
            constexpr uint32_t id_dk = idesc_bf16_f32(128, 128, false, true);
            constexpr uint32_t id_dq = idesc_bf16_f32(128, 128, true, true);
            const uint64_t dK_k = sdesc_sw128(sK, 16, 1024);
            const uint64_t dR_k = sdesc_sw128(sRing, 16, 1024), dR_mn = sdesc_sw128(sRing, kBox, 1024);
            const uint64_t dS_k = sdesc_sw128(sDS, 16, 1024), dS_mn = sdesc_sw128(sDS, kBox, 1024);
            const uint64_t dK_mn = sdesc_sw128(sK + 2 * hh * kBox, kBox, 1024);  // K[:, half h]
            constexpr uint32_t kMnStep = 2048 >> 4;
            auto ring_off = [&](int n) -> uint32_t { return (uint32_t)(slot_of(n) * kSlot) >> 4; };
            // a slot's empty barrier completes after two releases: each product that
            // reads the load gives one (a sole reader gives both), so a slot is
            // refilled only after every product reading it has completed
            auto release = [&](int n, int times) {
                for (int t = 0; t < times; ++t) mma_commit(empty_bar(n));
            };
            bool ok = mbar_wait(smem_u32(&bars.k_full), 0, wc);
            if (warp == kB256MmaX) {
                // S^T = K Q^T and dP^T = V dO^T, each as two column-half contractions
                for (int i = 0; i < n_q && ok; ++i) {
                    const int n0 = i * L::LOADS;
                    // S^T_i overwrites P^T_{i-1}: wait until dV_{i-1} has read it
                    if (i > 0 && !(ok = mbar_wait(smem_u32(&bars.dv_done), (i - 1) & 1, wc))) break;
                    if (!(ok = mbar_wait(full_bar(n0), phase_of(n0), wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + L::TM_S, dK_k + kmajor_koff(8 * (1 - hh) + kk), dR_k + ring_off(n0) + kmajor_koff(kk),
                               id_st, kk > 0 ? 1u : 0u);
                    release(n0, 2);
                    // dP^T_i overwrites dQ_{i-1}: wait until it has been drained
                    if (i > 0 && !(ok = mbar_wait(smem_u32(&bars.dq_drained), (i - 1) & 1, wc))) break;
                    if (!(ok = mbar_wait(full_bar(n0 + 1), phase_of(n0 + 1), wc))) break;
                    if (!(ok = mbar_wait(full_bar(n0 + 2), phase_of(n0 + 2), wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + L::TM_DP, dR_k + ring_off(n0 + 1) + kmajor_koff(kk),
                               dR_k + ring_off(n0 + 2) + kmajor_koff(kk), id_st, kk > 0 ? 1u : 0u);
                    release(n0 + 1, 2);
                    release(n0 + 2, 2);
                    if (!(ok = mbar_wait(full_bar(n0 + 3), phase_of(n0 + 3), wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + L::TM_S, dK_k + kmajor_koff(8 * hh + kk), dR_k + ring_off(n0 + 3) + kmajor_koff(kk),
                               id_st, 1u);
                    mma_commit(smem_u32(&bars.s_full));
                    release(n0 + 3, 1);  // Q_h: dK gives the other release
                    if (!(ok = mbar_wait(full_bar(n0 + 4), phase_of(n0 + 4), wc))) break;
                    if (!(ok = mbar_wait(full_bar(n0 + 5), phase_of(n0 + 5), wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + L::TM_DP, dR_k + ring_off(n0 + 4) + kmajor_koff(kk),
                               dR_k + ring_off(n0 + 5) + kmajor_koff(kk), id_st, 1u);
                    release(n0 + 4, 2);
                    release(n0 + 5, 1);  // dO_h: dV gives the other release
                    mma_commit(smem_u32(&bars.dp_full));
                }
                mma_commit(smem_u32(&bars.drain));
                drain_wait(smem_u32(&bars.drain), 0, p.timeout_ns);
            } else {
                // dV_h += P^T dO_h, dK_h += dS^T Q_h, dQ_h = dS K_h
                for (int i = 0; i < n_q && ok; ++i) {
                    const int n0 = i * L::LOADS;
                    if (!(ok = mbar_wait(smem_u32(&bars.p_ready), i & 1, wc))) break;
                    if (!(ok = mbar_wait(full_bar(n0 + 5), phase_of(n0 + 5), wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        mma_ts(tmem + L::TM_DV, tmem + L::TM_S + (kk < 4 ? kk * 8 : 96 + (kk - 4) * 8),
                               dR_mn + ring_off(n0 + 5) + kk * kMnStep, id_dv, (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&bars.dv_done));
                    release(n0 + 5, 1);
                    if (!(ok = mbar_wait(smem_u32(&bars.ds_ready), i & 1, wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        mma_ss(tmem + L::TM_DK, dS_k + kmajor_koff(kk), dR_mn + ring_off(n0 + 3) + kk * kMnStep, id_dk,
                               (i > 0 || kk > 0) ? 1u : 0u);
                    release(n0 + 3, 1);
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        mma_ss(tmem + L::TM_DP, dS_mn + kk * kMnStep, dK_mn + kk * kMnStep, id_dq, kk > 0 ? 1u : 0u);
                    mma_commit(smem_u32(&bars.dq_full));
                    mma_commit(smem_u32(&bars.ds_free));
                }
                mma_commit(smem_u32(&bars.final_mma));
                mma_commit(smem_u32(&bars.drain2));
                drain_wait(smem_u32(&bars.drain2), 0, p.timeout_ns);
            }
        }
    } else if (warp < kB256MathWarps) {
        // ---------------------------------------------------------- P / dS math
        const int quarter = warp & 3;
        const int half = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t taddr = tmem + (uint32_t(quarter * 32) << 16);
        const uint32_t s_cols = L::TM_S + half * 64, p_cols = L::TM_S + half * 96;
        const float sc = p.scale_log2;
        const bool row_valid = row < kv_len;
        bool ok = true;
        QTileIter q = q0;
        for (int i = 0; i < n_q; ++i, qw.next(q)) {
            const int n3 = i * L::LOADS + 3;  // carries this tile's row statistics
            const int q_start = qw.first_row(q);
            const bool diag = p.causal && q.r == c && kv_start + kv_len - 1 > q_start;
            const int lo = diag ? kv_start + row - q_start - half * 64 : 0;
            const float4* nlse2 = reinterpret_cast<const float4*>(stat_base + (i & 1) * 256 + half * 64);
            const float4* delta = reinterpret_cast<const float4*>(stat_base + (i & 1) * 256 + 128 + half * 64);
            if (!(ok = mbar_wait(full_bar(n3), phase_of(n3), wc))) break;
            if (!(ok = mbar_wait(smem_u32(&bars.s_full), i & 1, wc))) break;
            tc_fence_after();
            uint32_t pr[64];
            tmem_ld64_sync(taddr + s_cols, pr);
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
            if (diag || kv_len < kTile) {
                const int lo_eff = row_valid ? lo : 64;
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
            if (!(ok = mbar_wait(smem_u32(&bars.dp_full), i & 1, wc))) break;
            if (i > 0 && !(ok = mbar_wait(smem_u32(&bars.ds_free), (i - 1) & 1, wc))) break;
            tc_fence_after();
            const uint32_t box = sDS + half * kBox;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t dp[32];
                tmem_ld32_sync(taddr + L::TM_DP + half * 64 + cc * 32, dp);
                uint32_t wv[16];
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) {
                    const float4 d4 = delta[cc * 8 + k4];
                    const int qc = cc * 32 + 4 * k4;
                    const float2 a01 = fmul2(make_float2(__uint_as_float(pr[qc]), __uint_as_float(pr[qc + 1])),
                                             fsub2(make_float2(__uint_as_float(dp[4 * k4]), __uint_as_float(dp[4 * k4 + 1])),
                                                   make_float2(d4.x, d4.y)));
                    const float2 a23 = fmul2(make_float2(__uint_as_float(pr[qc + 2]), __uint_as_float(pr[qc + 3])),
                                             fsub2(make_float2(__uint_as_float(dp[4 * k4 + 2]), __uint_as_float(dp[4 * k4 + 3])),
                                                   make_float2(d4.z, d4.w)));
                    wv[2 * k4] = pack_bf16x2(a01.x, a01.y);
                    wv[2 * k4 + 1] = pack_bf16x2(a23.x, a23.y);
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t addr = box + sw128_offset(row, cc * 4 + m);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(wv[4 * m]),
                                 "r"(wv[4 * m + 1]), "r"(wv[4 * m + 2]), "r"(wv[4 * m + 3])
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars.ds_ready));
        }
        // ---------------------------------------------------------- dV_h epilogue
        if (ok && mbar_wait(smem_u32(&bars.final_mma), 0, wc)) {
            tc_fence_after();
            __nv_bfloat16* dst = p.dv + (int64_t)b * p.k_sb + (int64_t)(kv_start + row) * p.k_ss +
                                 (int64_t)hk * p.k_sh + hh * 128 + half * 64;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t o[32];
                tmem_ld32_sync(taddr + L::TM_DV + half * 64 + cc * 32, o);
                if (row_valid && part_row) {  // fp32 partial, summed by dkv_reduce_kernel
                    float4* d4 = reinterpret_cast<float4*>(part_row + ((size_t)row * 2 + 1) * kD + half * 64 + cc * 32);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        d4[k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                            __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
                } else if (row_valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        d4[k] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * k + 0]), __uint_as_float(o[8 * k + 1])),
                                           pack_bf16x2(__uint_as_float(o[8 * k + 2]), __uint_as_float(o[8 * k + 3])),
                                           pack_bf16x2(__uint_as_float(o[8 * k + 4]), __uint_as_float(o[8 * k + 5])),
                                           pack_bf16x2(__uint_as_float(o[8 * k + 6]), __uint_as_float(o[8 * k + 7])));
                }
            }
        }
    } else if (warp < kB256MathWarps + 4) {
        // ---------------------------------------------------------- dQ_h drain
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t taddr = tmem + (uint32_t(quarter * 32) << 16);
        QTileIter q = q0;
        bool ok = true;
        for (int i = 0; i < n_q; ++i, qw.next(q)) {
            if (!(ok = mbar_wait(smem_u32(&bars.dq_full), i & 1, wc))) break;
            tc_fence_after();
            // tile-major accumulator [(b,h,t)][D/4][128 rows][4]; this CTA's columns start at 128 hh
            float* tile = p.dq_acc + ((size_t)(b * p.Hq + q.h) * ct.ntiles + q.t) * (size_t)(kTile * kD) +
                          (size_t)hh * 32 * kTile * 4;
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                uint32_t v[64];
                tmem_ld64_sync(taddr + L::TM_DP + hc * 64, v);
                if (hc == 1) {
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bars.dq_drained));
                }
#pragma unroll
                for (int gq = 0; gq < 16; ++gq)
                    red_add_v4(tile + ((size_t)(hc * 16 + gq) * kTile + row) * 4, __uint_as_float(v[4 * gq]),
                               __uint_as_float(v[4 * gq + 1]), __uint_as_float(v[4 * gq + 2]),
                               __uint_as_float(v[4 * gq + 3]));
            }
        }
        // ---------------------------------------------------------- dK_h epilogue
        if (ok && mbar_wait(smem_u32(&bars.final_mma), 0, wc)) {
            tc_fence_after();
            const bool row_valid = row < kv_len;
            __nv_bfloat16* dst =
                p.dk + (int64_t)b * p.k_sb + (int64_t)(kv_start + row) * p.k_ss + (int64_t)hk * p.k_sh + hh * 128;
            const float scale = p.scale;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
                tmem_ld32_sync(taddr + L::TM_DK + cc * 32, o);
                if (row_valid && part_row) {  // unscaled fp32 partial
                    float4* d4 = reinterpret_cast<float4*>(part_row + (size_t)row * 2 * kD + cc * 32);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        d4[k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                            __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
                } else if (row_valid) {
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
    if (warp == kB256MmaX) tmem_dealloc(tmem, L::TM_COLS);
}

}  // namespace

int launch_attn_fwd256(const FwdParams& p, cudaStream_t s) {
    const bool partials = p.part_o != nullptr;
    auto kern = partials ? (p.head_major ? attn_fwd256_kernel<true, true> : attn_fwd256_kernel<true, false>)
                         : (p.head_major ? attn_fwd256_kernel<false, true> : attn_fwd256_kernel<false, false>);
    static OncePerDevice attr[4];
    if (!attr[(partials ? 2 : 0) + (p.head_major ? 1 : 0)].run([&] {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F256::SMEM) == cudaSuccess;
        }))
        return 4;
    const cudaError_t e = launch_kernel(p.pdl != 0, kern, grid_dims(p.head_major, p.ct.ntiles, p.Hq, p.B),
                                        dim3(kF256Threads), F256::SMEM, s, p);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int launch_attn_bwd256(const BwdParams& p, cudaStream_t s) {
    auto kern = p.head_major ? attn_bwd256_kernel<true> : attn_bwd256_kernel<false>;
    static OncePerDevice attr[2];
    if (!attr[p.head_major ? 1 : 0].run([&] {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, B256::SMEM) == cudaSuccess;
        }))
        return 4;
    // grid decode at the top of attn_bwd256_kernel
    const dim3 grid = p.head_major ? dim3(p.Hkv, p.B * 2 * p.hsplit, p.ct.ntiles)
                                   : dim3(2 * p.ct.ntiles, p.Hkv, p.B * p.hsplit);
    const cudaError_t e = launch_kernel(p.pdl != 0, kern, grid, dim3(kB256Threads), B256::SMEM, s, p);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? 0 : 4;
}

}  // namespace ctxattn
