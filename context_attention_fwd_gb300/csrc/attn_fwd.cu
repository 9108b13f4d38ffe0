// attn_fwd.cu -- ring-chunked attention forward for sm_103a.
//
// One CTA owns one 128-row query tile of one (batch, query head).  The tile
// belongs to ring chunk r; the CTA walks the ring iterations i = 0..P-1,
// meeting KV chunk c = (r - i) mod P at iteration i (diffusers issue #14265,
// "Root cause": the query stays put while the K/V chunks rotate), and within
// an iteration the 128-row KV tiles of chunk c.  Keys past the chunk's end
// are masked, so every iteration sees exactly its own chunk.
//
// Merging.  Each iteration's partial (O_i, LSE_i) is merged by LSE
// weighting (same issue, "How it surfaces": the ring needs the LSE to merge
// partial results).  By default the merge is done online: the running
// (max, sum, O) state absorbs each KV tile, which is the pairwise LSE merge
// of partials applied tile by tile.  With materialised partials the state is
// reset at every chunk boundary and (O_i / l_i, m_i + log l_i) is written out
// for a separate merge kernel.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q once, K/V tiles through a 2-stage ring
//   warp 1      TMEM owner and tcgen05.mma issuer (one elected lane)
//   warps 2..5  softmax: one query row per thread, S from TMEM, P back to
//               TMEM as bf16 (A operand of the PV product), O rescale,
//               epilogue
// TMEM (512 columns): S/P double buffer at columns 0 and 128, O at 256.
// S = Q K^T: A = Q (smem, K-major), B = K (smem, K-major), M=N=128.
// O += P V:  A = P (TMEM), B = V (smem, MN-major: V rows are the K index).
#include "internal.h"
#include "ptx.cuh"

namespace ctxattn {
namespace {

template <int D>
struct FwdLayout {
    static constexpr int NBOX = D / 64;                 // 128-byte swizzle boxes per row
    static constexpr uint32_t BOX = kTile * 128;        // one box: 128 rows x 128 bytes
    static constexpr uint32_t TILE = kTile * D * 2;     // a 128 x D bf16 tile
    static constexpr int STAGES = 2;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + TILE;
    static constexpr uint32_t OFF_V = OFF_K + STAGES * TILE;
    static constexpr uint32_t END = OFF_V + STAGES * TILE;
    // Request enough shared memory that only one CTA fits per SM: each CTA
    // holds all 512 TMEM columns.
    static constexpr uint32_t SMEM = (END + 1024) < 120u * 1024 ? 120u * 1024 : (END + 1024);
    static constexpr uint32_t TM_S = 0, TM_O = 256, TM_COLS = 512;
};

struct FwdBars {
    uint64_t q_full;
    uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
    uint64_t s_full[2], p_full[2];
    uint64_t o_done;   // one arrival per PV product
    uint64_t o_chunk;  // after the last PV of a chunk (every chunk with partials, else once)
    uint64_t o_free;   // partials: O drained, the next chunk may overwrite it
    uint64_t drain;    // teardown: all MMAs retired
};

constexpr int kSoftmaxThreads = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: move the reference max lazily

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

template <int D>
__global__ void __launch_bounds__(192, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
    using L = FwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ FwdBars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = sbase + L::OFF_Q, sK = sbase + L::OFF_K, sV = sbase + L::OFF_V;
    const int warp = warp_id(), lane = lane_id();
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const ChunkTable& ct = p.ct;
    const int P = ct.P;
    const int r = chunk_of_tile(ct, qt);
    const int q_start = ct.off[r] + (qt - ct.tile_off[r]) * kTile;
    const int q_len = min(kTile, ct.off[r + 1] - q_start);
    const int hk = h / p.group;
    const int n_kv = ct.ntiles;
    const bool partials = p.part_o != nullptr;
    const WaitCtx wc{&abort_flag, p.status, p.timeout_ns};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bars.q_full), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars.k_full[i]), 1);
            mbar_init(smem_u32(&bars.k_empty[i]), 1);
            mbar_init(smem_u32(&bars.v_full[i]), 1);
            mbar_init(smem_u32(&bars.v_empty[i]), 1);
            mbar_init(smem_u32(&bars.s_full[i]), 1);
            mbar_init(smem_u32(&bars.p_full[i]), kSoftmaxThreads);
        }
        mbar_init(smem_u32(&bars.o_done), 1);
        mbar_init(smem_u32(&bars.o_chunk), 1);
        mbar_init(smem_u32(&bars.o_free), kSoftmaxThreads);
        mbar_init(smem_u32(&bars.drain), 1);
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
            mbar_arrive_expect_tx(qf, L::TILE);
            for (int bx = 0; bx < L::NBOX; ++bx)
                tma_tile(p.tq, sQ + bx * L::BOX, qf, bx * 64, q_start, h, b);
            int j = 0, last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
            bool ok = true;
            for (int it = 0; it < P && ok; ++it) {
                const int c = (r - it + P) % P;
                for (int t = ct.tile_off[c]; t < ct.tile_off[c + 1]; ++t, ++j) {
                    const int st = j & 1, ph = (j >> 1) & 1;
                    const int kv_start = ct.off[c] + (t - ct.tile_off[c]) * kTile;
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
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
            bool ok = mbar_wait(smem_u32(&bars.q_full), 0, wc);
            tc_fence_after();
            // PV of the previous tile is issued after QK of the current one, so
            // the tensor core computes S_{j+1} while the softmax works on S_j.
            int j = 0, prev_it = 0;
            bool prev_first = false, prev_last = false;
            auto issue_pv = [&](int jp, bool first, bool last, int itp) -> bool {
                const int stp = jp & 1, php = (jp >> 1) & 1;
                if (!mbar_wait(smem_u32(&bars.p_full[stp]), php, wc)) return false;
                if (!mbar_wait(smem_u32(&bars.v_full[stp]), php, wc)) return false;
                if (partials && first && itp > 0 &&
                    !mbar_wait(smem_u32(&bars.o_free), (itp - 1) & 1, wc))
                    return false;
                tc_fence_after();
                const bool acc0 = partials ? !first : jp > 0;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint64_t bdesc = sdesc_sw128(sV + stp * L::TILE + kk * 2048, L::BOX, 1024);
                    mma_ts(tmem + L::TM_O, tmem + L::TM_S + stp * 128 + kk * 8, bdesc, idesc_pv,
                           (acc0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars.o_done));
                mma_commit(smem_u32(&bars.v_empty[stp]));
                if (last && (partials || itp == P - 1)) mma_commit(smem_u32(&bars.o_chunk));
                return true;
            };
            for (int it = 0; it < P && ok; ++it) {
                const int c = (r - it + P) % P;
                const int t0 = ct.tile_off[c], t1 = ct.tile_off[c + 1];
                for (int t = t0; t < t1; ++t, ++j) {
                    const int st = j & 1, ph = (j >> 1) & 1;
                    if (!(ok = mbar_wait(smem_u32(&bars.k_full[st]), ph, wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = (kk >> 2) * L::BOX + (kk & 3) * 32;
                        mma_ss(tmem + L::TM_S + st * 128, sdesc_sw128(sQ + koff, 16, 1024),
                               sdesc_sw128(sK + st * L::TILE + koff, 16, 1024), idesc_qk,
                               kk > 0 ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&bars.s_full[st]));
                    mma_commit(smem_u32(&bars.k_empty[st]));
                    if (j > 0 && !(ok = issue_pv(j - 1, prev_first, prev_last, prev_it))) break;
                    prev_first = (t == t0);
                    prev_last = (t == t1 - 1);
                    prev_it = it;
                }
            }
            if (ok && n_kv > 0) issue_pv(n_kv - 1, prev_first, prev_last, prev_it);
            mma_commit(smem_u32(&bars.drain));
            drain_wait(smem_u32(&bars.drain), 0, p.timeout_ns);
        }
    } else {
        // ------------------------------------------------------ softmax
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t taddr = tmem + (uint32_t(quarter * 32) << 16);
        const float sc = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        int j = 0;
        bool ok = true;
        for (int it = 0; it < P && ok; ++it) {
            const int c = (r - it + P) % P;
            const int t0 = ct.tile_off[c], t1 = ct.tile_off[c + 1];
            for (int t = t0; t < t1; ++t, ++j) {
                const int st = j & 1, ph = (j >> 1) & 1;
                const int kv_len = min(kTile, ct.off[c + 1] - (ct.off[c] + (t - t0) * kTile));
                const bool first = partials ? (t == t0) : (j == 0);
                if (!(ok = mbar_wait(smem_u32(&bars.s_full[st]), ph, wc))) break;
                tc_fence_after();
                uint32_t s[128];
                tmem_ld32(taddr + L::TM_S + st * 128 + 0, s);
                tmem_ld32(taddr + L::TM_S + st * 128 + 32, s + 32);
                tmem_ld32(taddr + L::TM_S + st * 128 + 64, s + 64);
                tmem_ld32(taddr + L::TM_S + st * 128 + 96, s + 96);
                tmem_ld_wait();
                reg_fence32(s);
                reg_fence32(s + 32);
                reg_fence32(s + 64);
                reg_fence32(s + 96);
                if (kv_len < kTile) {
#pragma unroll
                    for (int k = 0; k < 128; ++k)
                        if (k >= kv_len) s[k] = __float_as_uint(-INFINITY);
                }
                float mx = -INFINITY;
#pragma unroll
                for (int k = 0; k < 128; ++k) mx = fmaxf(mx, __uint_as_float(s[k]));
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
                const float neg = -m_ref * sc;
                float sum = 0.f;
                uint32_t pk[64];
#pragma unroll
                for (int k = 0; k < 64; ++k) {
                    const float p0 = ex2(fmaf(__uint_as_float(s[2 * k]), sc, neg));
                    const float p1 = ex2(fmaf(__uint_as_float(s[2 * k + 1]), sc, neg));
                    sum += p0 + p1;
                    pk[k] = pack_bf16x2(p0, p1);
                }
                tmem_st32(taddr + L::TM_S + st * 128 + 0, pk);
                tmem_st32(taddr + L::TM_S + st * 128 + 32, pk + 32);
                l = l * alpha + sum;
                if (__any_sync(0xffffffffu, rescale)) {
                    // O holds the product of the tiles before j: wait for the
                    // last of them (PV_{j-1}) and rescale in place.
                    if (!(ok = mbar_wait(smem_u32(&bars.o_done), (j - 1) & 1, wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(taddr + L::TM_O + cc * 32, o);
                        tmem_ld_wait();
                        reg_fence32(o);
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tmem_st32(taddr + L::TM_O + cc * 32, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars.p_full[st]));
                if (partials && t == t1 - 1) {
                    // this chunk's partial is complete: O_it / l, LSE_it
                    if (!(ok = mbar_wait(smem_u32(&bars.o_chunk), it & 1, wc))) break;
                    tc_fence_after();
                    const float inv_l = 1.f / l;
                    const bool valid = row < q_len;
                    const size_t prow = ((size_t)(it * p.B + b) * p.Hq + h) * p.S + q_start + row;
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(taddr + L::TM_O + cc * 32, o);
                        tmem_ld_wait();
                        reg_fence32(o);
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
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bars.o_free));
                }
            }
        }
        if (ok && !partials) {
            // --------------------------------------------------- epilogue
            ok = mbar_wait(smem_u32(&bars.o_chunk), 0, wc);
            tc_fence_after();
            if (ok) {
                const float inv_l = 1.f / l;
                const bool valid = row < q_len;
                __nv_bfloat16* dst_row =
                    p.out + (int64_t)b * p.o_sb + (int64_t)(q_start + row) * p.o_ss + (int64_t)h * p.o_sh;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(taddr + L::TM_O + cc * 32, o);
                    tmem_ld_wait();
                    reg_fence32(o);
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

template <int D>
int launch_fwd_d(const FwdParams& p, cudaStream_t s) {
    using L = FwdLayout<D>;
    if (cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::SMEM) != cudaSuccess)
        return 4;
    dim3 grid(p.ct.ntiles, p.Hq, p.B);
    attn_fwd_kernel<D><<<grid, 192, L::SMEM, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

}  // namespace

int launch_attn_fwd(const FwdParams& p, int D, cudaStream_t s) {
    if (D == 64) return launch_fwd_d<64>(p, s);
    if (D == 128) return launch_fwd_d<128>(p, s);
    return 2;
}

}  // namespace ctxattn
