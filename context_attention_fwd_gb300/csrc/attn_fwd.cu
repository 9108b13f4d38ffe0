// attn_fwd.cu -- ring-chunked attention forward for sm_103a.
//
// One CTA owns two 128-row query tiles (A and B, consecutive tiles of the
// same ring chunk r) of one (batch, query head).  It walks the ring
// iterations i = 0..P-1, meeting KV chunk c = (r - i) mod P at iteration i
// (diffusers issue #14265, "Root cause": the query stays put while the K/V
// chunks rotate), and within an iteration the 128-row KV tiles of chunk c.
// Keys past the chunk's end are masked, so every iteration sees exactly its
// own chunk.  Both query tiles share every K/V tile the CTA loads.
//
// Merging.  Each iteration's partial (O_i, LSE_i) is merged by LSE
// weighting (same issue, "How it surfaces": the ring needs the LSE to merge
// partial results).  By default the merge is done online: the running
// (max, sum, O) state absorbs each KV tile, which is the pairwise LSE merge
// of partials applied tile by tile.  With materialised partials the state is
// reset at every chunk boundary and (O_i / l_i, m_i + log l_i) is written out
// for a separate merge kernel.
//
// Warp roles (384 threads):
//   warp 0       TMA producer: Q_A, Q_B once, K/V tiles through a 2-stage ring
//   warp 1       TMEM owner
//   warps 2, 3   idle (keep the softmax warpgroups warpgroup-aligned)
//   warps 4..7   tile A, warps 8..11 tile B: one query row per thread; S from
//                TMEM, mask, max, exp2, sum, P back to TMEM as bf16 (the A
//                operand of the PV product), lazy O rescale, epilogue.  Lane 0
//                of the first warp of each group issues that tile's own
//                tcgen05.mma: PV_x(j) then S_x(j+1), so each tile is an
//                independent pipeline and the tensor core is fed by two
//                issuers: while one waits on a barrier, the other's queued
//                products keep it busy.
// TMEM (512 columns): S_A 0, S_B 128, O_A 256, O_B 256 + D.
// S_x = Q_x K^T: A = Q (smem, K-major), B = K (smem, K-major), M=N=128.
// O_x += P_x V:  A = P (TMEM), B = V (smem, MN-major: V rows are the K index).
#include "internal.h"
#include "ptx.cuh"
#include "walk.cuh"

namespace ctxattn {
namespace {

template <int D>
struct FwdLayout {
    static constexpr int NBOX = D / 64;              // 128-byte swizzle boxes per row
    static constexpr uint32_t BOX = kTile * 128;     // one box: 128 rows x 128 bytes
    static constexpr uint32_t TILE = kTile * D * 2;  // a 128 x D bf16 tile
    static constexpr int STAGES = 2;
    static constexpr uint32_t OFF_Q = 0;              // Q_A, Q_B
    static constexpr uint32_t OFF_K = OFF_Q + 2 * TILE;
    static constexpr uint32_t OFF_V = OFF_K + STAGES * TILE;
    static constexpr uint32_t END = OFF_V + STAGES * TILE;
    // Request enough shared memory that only one CTA fits per SM: each CTA
    // holds all 512 TMEM columns.
    static constexpr uint32_t SMEM = (END + 1024) < 120u * 1024 ? 120u * 1024 : (END + 1024);
    static constexpr uint32_t TM_S = 0, TM_O = 256, TM_COLS = 512;
};

struct FwdBars {
    uint64_t q_full;
    uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];  // empties: one commit per tile issuer
    uint64_t s_done[2];   // per tile: S_x(j) computed
    uint64_t o_done[2];   // per tile: the last PV of a chunk (partials) or of the walk computed
    uint64_t drain[2];    // per tile issuer, teardown: all its MMAs retired
};

constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 128;
constexpr int kSoftmaxWarp0 = 4;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: move the reference max lazily

// Barrier among the 128 threads of one softmax warpgroup (ids 1 and 2).
__device__ __forceinline__ void group_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kSoftmaxThreads) : "memory");
}

__device__ __forceinline__ int pick3(int o, int s, int h, int b) {
    return o == 0 ? s : (o == 1 ? h : b);
}
__device__ __forceinline__ void tma_tile(const TmaMap& m, uint32_t dst, uint32_t bar, int d0, int s,
                                         int h, int b) {
    tma_load_4d(dst, &m.map, bar, d0, pick3(m.ord[0], s, h, b), pick3(m.ord[1], s, h, b),
                pick3(m.ord[2], s, h, b));
}

// Bounded wait that ignores the abort flag: used at teardown for work that
// completes on its own (TMA copies, issued MMAs).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) break;
}

template <int D, bool kPartials, bool kHeadMajor>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
    griddep_wait();  // the previous kernel in the stream is complete (launch_kernel)
    griddep_launch_dependents();
    using L = FwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ FwdBars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = sbase + L::OFF_Q, sK = sbase + L::OFF_K, sV = sbase + L::OFF_V;
    const int warp = warp_id(), lane = lane_id();
    // the last pairs carry the most work under causal masking: launch them first
    const GridPos gp = grid_pos<kHeadMajor>();
    const int pair = p.ct.npairs - 1 - gp.tile, h = gp.head, b = gp.z;
    const ChunkTable& ct = p.ct;
    const int P = ct.P;
    int r = 0;
    while (r + 1 < P && ct.pair_off[r + 1] <= pair) ++r;
    const int tA = ct.tile_off[r] + 2 * (pair - ct.pair_off[r]);
    const bool hasB = tA + 1 < ct.tile_off[r + 1];
    const int ntile = hasB ? 2 : 1;
    const int qs0 = ct.off[r] + (tA - ct.tile_off[r]) * kTile;
    const int hk = h / p.group;
    const WalkCfg g{r, P, p.causal, p.allgather,
                    qs0 + (hasB ? kTile : 0) + min(kTile, ct.off[r + 1] - (qs0 + (hasB ? kTile : 0))) - 1};
    const int n_kv = kv_count(ct, g);
    constexpr bool partials = kPartials;
    const WaitCtx wc{&abort_flag, p.status, p.timeout_ns};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bars.q_full), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars.k_full[i]), 1);
            mbar_init(smem_u32(&bars.k_empty[i]), ntile);
            mbar_init(smem_u32(&bars.v_full[i]), 1);
            mbar_init(smem_u32(&bars.v_empty[i]), ntile);
            mbar_init(smem_u32(&bars.s_done[i]), 1);
            mbar_init(smem_u32(&bars.o_done[i]), 1);
            mbar_init(smem_u32(&bars.drain[i]), 1);
        }
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
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tq.map);
            tma_prefetch_desc(&p.tk.map);
            tma_prefetch_desc(&p.tv.map);
            const uint32_t qf = smem_u32(&bars.q_full);
            mbar_arrive_expect_tx(qf, ntile * L::TILE);
            for (int x = 0; x < ntile; ++x)
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_tile(p.tq, sQ + x * L::TILE + bx * L::BOX, qf, bx * 64, qs0 + x * kTile, h, b);
            int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
            bool ok = true;
            const int skip = debug_skip_step(p.debug, n_kv);  // -1 in normal use
            KvWalk w;
            kv_first(ct, g, w);
            for (int j = 0; j < n_kv; ++j, kv_next(ct, g, w)) {
                if (j == skip) {  // failure injection: no K, V from step j on
                    ok = false;
                    break;
                }
                const int st = j & 1, ph = (j >> 1) & 1;
                const int kv_start = ct.off[w.c] + (w.t - w.t0) * kTile;
                if (!(ok = mbar_wait(smem_u32(&bars.k_empty[st]), ph ^ 1, wc))) break;
                const uint32_t kf = smem_u32(&bars.k_full[st]);
                mbar_arrive_expect_tx(kf, L::TILE);
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_tile(p.tk, sK + st * L::TILE + bx * L::BOX, kf, bx * 64, kv_start, hk, b);
                last_k[st] = ph;
                if (!(ok = mbar_wait(smem_u32(&bars.v_empty[st]), ph ^ 1, wc))) break;
                const uint32_t vf = smem_u32(&bars.v_full[st]);
                mbar_arrive_expect_tx(vf, L::TILE);
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_tile(p.tv, sV + st * L::TILE + bx * L::BOX, vf, bx * 64, kv_start, hk, b);
                last_v[st] = ph;
            }
            if (!ok) {
                // wait for our own copies in flight before the CTA retires
                drain_wait(qf, 0, p.timeout_ns);
                for (int st = 0; st < 2; ++st) {
                    if (last_k[st] >= 0) drain_wait(smem_u32(&bars.k_full[st]), last_k[st], p.timeout_ns);
                    if (last_v[st] >= 0) drain_wait(smem_u32(&bars.v_full[st]), last_v[st], p.timeout_ns);
                }
            }
        }
    } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4 * ntile) {
        // ------------------------------------------------------ softmax + MMA issue of tile x
        const int x = (warp - kSoftmaxWarp0) >> 2;  // query tile A (0) or B (1)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const bool issuer = (warp & 3) == 0 && lane == 0;
        const uint32_t taddr = tmem + (uint32_t(quarter * 32) << 16);
        const uint32_t s_cols = L::TM_S + x * 128, o_cols = L::TM_O + x * D;
        const int q_start = qs0 + x * kTile;
        const float sc = p.scale_log2;
        const bool valid = row < ct.off[r + 1] - q_start;
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
        // Loop-invariant descriptors; a k-step only advances the 14-bit
        // start-address field (address / 16), which never carries.
        const uint64_t dq0 = sdesc_sw128(sQ + x * L::TILE, 16, 1024), dk0 = sdesc_sw128(sK, 16, 1024);
        const uint64_t dv0 = sdesc_sw128(sV, L::BOX, 1024);
        const uint32_t s_done = smem_u32(&bars.s_done[x]), o_done = smem_u32(&bars.o_done[x]);
        auto issue_s = [&](int st) {  // S_x = Q_x K^T, K tile in stage st
            const uint64_t bk = dk0 + ((st * L::TILE) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t koff = ((kk >> 2) * L::BOX + (kk & 3) * 32) >> 4;
                mma_ss(tmem + s_cols, dq0 + koff, bk + koff, idesc_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit(s_done);
            mma_commit(smem_u32(&bars.k_empty[st]));
        };
        bool ok = true;
        if (issuer) {
            ok = mbar_wait(smem_u32(&bars.q_full), 0, wc) && mbar_wait(smem_u32(&bars.k_full[0]), 0, wc);
            if (ok) issue_s(0);
        }
        __syncwarp();  // park the issuer's warp-mates instead of letting them spin
        float m_ref = -INFINITY, l = 0.f;
        KvWalk w;
        kv_first(ct, g, w);
        for (int j = 0; j < n_kv && ok; ++j, kv_next(ct, g, w)) {
            const int kv_start = ct.off[w.c] + (w.t - w.t0) * kTile;
            const int kv_len = min(kTile, ct.off[w.c + 1] - kv_start);
            const bool first = partials ? (w.t == w.t0) : (j == 0);
            // keys this row may see in the tile: [0, lim)
            const bool diag = g.causal && kv_start + kv_len - 1 > q_start;
            const int lim = diag ? max(0, min(kv_len, q_start + row - kv_start + 1)) : kv_len;
            if (!(ok = mbar_wait(s_done, j & 1, wc))) break;
            tc_fence_after();
            uint32_t s[128];
            tmem_ld128_sync(taddr + s_cols, s);
            if (kv_len < kTile || diag) {
#pragma unroll
                for (int k = 0; k < 128; ++k)
                    if (k >= lim) s[k] = __float_as_uint(-INFINITY);
            }
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = __uint_as_float(s[e]);
#pragma unroll
            for (int k = 8; k < 128; k += 8)
#pragma unroll
                for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(mx8[e], __uint_as_float(s[k + e]));
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
                    m_ref = mx;  // nothing accumulated yet for this row
                } else if ((mx - m_ref) * sc > kRescaleThreshold) {
                    alpha = ex2((m_ref - mx) * sc);
                    m_ref = mx;
                    rescale = true;
                }
            }
            const float neg = m_ref == -INFINITY ? 0.f : -m_ref * sc;  // a row with no key yet
            float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                float x0, x1;
                if constexpr (D == 64) {
                    // columns in pairs (one two-lane fp32 instruction): faster at
                    // D = 64, slower at D = 128, where the kernel is at its
                    // register limit and the pairs need aligned register pairs
                    const float2 x = ffma2(make_float2(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1])),
                                           make_float2(sc, sc), make_float2(neg, neg));
                    x0 = x.x;
                    x1 = x.y;
                } else {
                    x0 = fmaf(__uint_as_float(s[2 * k]), sc, neg);
                    x1 = fmaf(__uint_as_float(s[2 * k + 1]), sc, neg);
                }
                const float p0 = ex2(x0), p1 = ex2(x1);
                sum8[(2 * k) & 7] += p0;
                sum8[(2 * k + 1) & 7] += p1;
                s[k] = pack_bf16x2(p0, p1);  // packed P overwrites scores already consumed
            }
            tmem_st32(taddr + s_cols + 0, s);
            tmem_st32(taddr + s_cols + 32, s + 32);
            const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
                              ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
            l = l * alpha + sum;
            if (__any_sync(0xffffffffu, rescale)) {
                // PV of the previous KV tile was issued before this S (same
                // issuer) and has completed with it: rescale O in place.
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32_sync(taddr + o_cols + cc * 32, o);
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    tmem_st32(taddr + o_cols + cc * 32, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            group_sync(1 + x);  // every P (and O rescale) of this tile is in TMEM
            const bool first_c = w.t == w.t0, last_c = kv_chunk_last(ct, g, w);
            if (issuer) {
                tc_fence_after();
                const int st = j & 1, st1 = (j + 1) & 1;
                // O_x += P_x V: V tile of stage st
                if (!(ok = mbar_wait(smem_u32(&bars.v_full[st]), (j >> 1) & 1, wc))) {
                    *wc.abort_flag = 1;
                } else {
                    const bool acc0 = partials ? !first_c : j > 0;
                    const uint64_t bv = dv0 + ((st * L::TILE) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        mma_ts(tmem + o_cols, tmem + s_cols + kk * 8, bv + kk * (2048 >> 4), idesc_pv,
                               (acc0 || kk > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&bars.v_empty[st]));
                    if (partials ? last_c : j == n_kv - 1) mma_commit(o_done);
                    // S_x(j+1) overwrites P_x(j): issued after the PV that reads it (in order)
                    if (j + 1 < n_kv) {
                        if (mbar_wait(smem_u32(&bars.k_full[st1]), ((j + 1) >> 1) & 1, wc))
                            issue_s(st1);
                        else
                            *wc.abort_flag = 1;
                    }
                }
            }
            __syncwarp();
            if (partials && last_c) {
                // this chunk's partial is complete: O_it / l, LSE_it
                const int it = w.it;
                if (!(ok = mbar_wait(o_done, it & 1, wc))) break;
                tc_fence_after();
                const float inv_l = 1.f / l;
                const size_t prow = ((size_t)(it * p.B + b) * p.Hq + h) * p.S + q_start + row;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32_sync(taddr + o_cols + cc * 32, o);
                    if (valid) {
                        float4* dst = reinterpret_cast<float4*>(p.part_o + prow * D + cc * 32);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv_l,
                                                 __uint_as_float(o[4 * k + 1]) * inv_l,
                                                 __uint_as_float(o[4 * k + 2]) * inv_l,
                                                 __uint_as_float(o[4 * k + 3]) * inv_l);
                    }
                }
                if (valid) p.part_lse[prow] = m_ref * p.scale + logf(l);
                tc_fence_before();  // the next chunk's first PV overwrites O after the next group_sync
            }
        }
        if (ok && !partials) {
            // --------------------------------------------------- epilogue
            ok = mbar_wait(o_done, 0, wc);
            tc_fence_after();
            if (ok) {
                const float inv_l = 1.f / l;
                __nv_bfloat16* dst_row =
                    p.out + (int64_t)b * p.o_sb + (int64_t)(q_start + row) * p.o_ss + (int64_t)h * p.o_sh;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32_sync(taddr + o_cols + cc * 32, o);
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
                if (valid)
                    p.lse[((int64_t)b * p.Hq + h) * p.S + q_start + row] = m_ref * p.scale + logf(l);
            }
        }
    }

    if (warp >= kSoftmaxWarp0 && (warp & 3) == 0 && lane == 0 && warp < kSoftmaxWarp0 + 4 * ntile) {
        const int x = (warp - kSoftmaxWarp0) >> 2;  // this tile's issued MMAs must retire first
        mma_commit(smem_u32(&bars.drain[x]));
        drain_wait(smem_u32(&bars.drain[x]), 0, p.timeout_ns);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::TM_COLS);
}

template <int D, bool kPartials, bool kHeadMajor>
int launch_fwd_dpo(const FwdParams& p, cudaStream_t s) {
    using L = FwdLayout<D>;
    static OncePerDevice attr;
    if (!attr.run([] {
            return cudaFuncSetAttribute(attn_fwd_kernel<D, kPartials, kHeadMajor>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM) == cudaSuccess;
        }))
        return 4;
    const cudaError_t e = launch_kernel(p.pdl != 0, attn_fwd_kernel<D, kPartials, kHeadMajor>,
                                        grid_dims(kHeadMajor, p.ct.npairs, p.Hq, p.B), dim3(kThreads), L::SMEM, s, p);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? 0 : 4;
}

template <int D, bool kPartials>
int launch_fwd_dp(const FwdParams& p, cudaStream_t s) {
    return p.head_major ? launch_fwd_dpo<D, kPartials, true>(p, s) : launch_fwd_dpo<D, kPartials, false>(p, s);
}

// The materialised-partials code path is a separate instantiation so that
// the default online kernel carries none of its registers.
template <int D>
int launch_fwd_d(const FwdParams& p, cudaStream_t s) {
    return p.part_o ? launch_fwd_dp<D, true>(p, s) : launch_fwd_dp<D, false>(p, s);
}

}  // namespace

int attn_fwd_binary_version() {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, attn_fwd_kernel<128, false, false>) != cudaSuccess) return -1;
    return a.binaryVersion;
}

int launch_attn_fwd(const FwdParams& p, int D, cudaStream_t s) {
    if (D == 64) return launch_fwd_d<64>(p, s);
    if (D == 128) return launch_fwd_d<128>(p, s);
    if (D == 256) return launch_attn_fwd256(p, s);
    return 2;
}

}  // namespace ctxattn
