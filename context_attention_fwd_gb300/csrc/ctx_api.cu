// ctx_api.cu -- the C ABI (include/ctx_attn.h): argument validation, the
// ring chunk schedule, TMA descriptors, workspace carving, launches; plus the
// bandwidth-bound kernels of the path: the Ulysses exchange, the backward's
// row statistics (delta = rowsum(dO o O)), the dQ fp32 -> bf16 conversion and
// the LSE merge of materialised partials.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <functional>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/ctx_attn.h"
#include "internal.h"
#include "ptx.cuh"

using namespace ctxattn;

namespace {

// Device status word: kernels record a wait that ran out here.
__device__ int g_device_status;

int* status_ptr() {
    static std::mutex mu;
    static int* ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int*>(p);
    }
    return ptrs[dev];
}

// Test-only switches set by ctx_debug_set (0 in normal use).
std::atomic<unsigned> g_debug_flags{0};
std::atomic<unsigned> g_wait_limit_ms{0};  // 0: the environment's or the default limit

uint64_t timeout_ns() {
    const unsigned over = g_wait_limit_ms.load(std::memory_order_relaxed);
    if (over) return (uint64_t)over * 1000000ull;
    static uint64_t ns = 0;
    if (!ns) {
        const char* e = getenv("CTX_ATTN_WAIT_LIMIT_MS");
        long ms = e ? atol(e) : 0;
        ns = (ms > 0 ? (uint64_t)ms : 2000ull) * 1000000ull;
    }
    return ns;
}

int kernel_debug_bits() {
    return (g_debug_flags.load(std::memory_order_relaxed) & CTX_DEBUG_SKIP_ARRIVAL) ? kDebugSkipArrival : 0;
}

// CTX_ATTN_LOG=1: one line per attention call on stderr (schedule, tiles,
// kernel variant).
bool log_enabled() {
    static const bool on = [] {
        const char* e = getenv("CTX_ATTN_LOG");
        return e && *e && *e != '0';
    }();
    return on;
}

// An NVTX range around an entry point (visible in a profiler's timeline;
// nearly free when no tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

int num_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

// Launch order of the attention kernels.  Under causal masking the work of
// a CTA falls off along the tile index, and the kernels launch the heaviest
// tile of a head first.  On grids of a few waves the order across heads
// decides the makespan too: in the head-major order (grid (heads, z, tiles))
// the heaviest tile of every head starts before any lighter one (longest
// job first).  Larger grids keep the tile-major order (grid (tiles, heads,
// z)): the CTAs in flight share one head's K/V, which stays hot in L2.
int pick_head_major(int causal, int64_t ctas) {
    return causal && ctas <= 4LL * num_sms() ? 1 : 0;
}

// Programmatic dependent launch (launch_kernel) lets each kernel of a call
// be scheduled while the previous one drains.  It pays where the gaps
// between kernels are a visible share of a call, i.e. where the kernels are
// short: at most 16 tile steps per SM if every CTA visited every tile (at
// 1024 tokens a forward + backward step went from 79.6 to 70.8 us at
// D = 128, from 138.6 to 136.6 us at D = 256).  Longer calls were slower
// with it (up to 7% at 2048 tokens, 0.5-1% on long sequences), and so was
// the D = 256 backward call (3-4% at 1536 tokens), which keeps plain
// launches.  Replaying a CUDA graph already removes the gaps (and was slower
// with it), so a stream that is being captured gets plain launches too.
int use_pdl(int64_t ctas, int ntiles, cudaStream_t s) {
    if (ctas * ntiles > 16LL * num_sms()) return 0;
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return st == cudaStreamCaptureStatusNone ? 1 : 0;
}

struct Dense {
    void* data;
    int64_t sb, ss, sh;
};

// Validates a logical [B,S,H,D] tensor and resolves its strides.
int resolve(const ctx_tensor_t* t, int64_t B, int64_t S, int64_t H, int64_t D, ctx_layout_t layout,
            Dense* out) {
    if (!t || !t->data) return CTX_ERR_INVALID_ARG;
    if (t->B != B || t->S != S || t->H != H || t->D != D) return CTX_ERR_INVALID_ARG;
    int64_t sb = t->stride_b, ss = t->stride_s, sh = t->stride_h;
    if (sb == 0 && ss == 0 && sh == 0) {
        if (layout == CTX_LAYOUT_BSHD) {
            sh = D; ss = H * D; sb = S * H * D;
        } else if (layout == CTX_LAYOUT_SBHD) {
            sh = D; sb = H * D; ss = B * H * D;
        } else {
            return CTX_ERR_INVALID_ARG;
        }
    }
    if (sb < 0 || ss < 0 || sh < 0) return CTX_ERR_INVALID_ARG;
    if ((B > 1 && sb == 0) || (S > 1 && ss == 0) || (H > 1 && sh == 0)) return CTX_ERR_INVALID_ARG;
    if (sh < D && H > 1) return CTX_ERR_INVALID_ARG;  // heads would overlap
    // TMA and 16-byte vector access: 16-byte aligned base and strides
    if ((reinterpret_cast<uintptr_t>(t->data) & 15) || (sb & 7) || (ss & 7) || (sh & 7))
        return CTX_ERR_UNSUPPORTED;
    out->data = t->data;
    out->sb = sb;
    out->ss = ss;
    out->sh = sh;
    return CTX_OK;
}

int build_chunks(int S, int P, const int* offsets, ChunkTable* ct) {
    if (P < 1 || P > kMaxChunks || P > S) return CTX_ERR_INVALID_ARG;
    ct->P = P;
    if (offsets) {
        if (offsets[0] != 0 || offsets[P] != S) return CTX_ERR_INVALID_ARG;
        for (int c = 0; c <= P; ++c) ct->off[c] = offsets[c];
        for (int c = 0; c < P; ++c)
            if (ct->off[c + 1] <= ct->off[c]) return CTX_ERR_INVALID_ARG;
    } else {
        ctx_chunk_offsets(S, P, ct->off);
    }
    ct->tile_off[0] = 0;
    for (int c = 0; c < P; ++c) {
        const int len = ct->off[c + 1] - ct->off[c];
        ct->tile_off[c + 1] = ct->tile_off[c] + (len + kTile - 1) / kTile;
    }
    ct->ntiles = ct->tile_off[P];
    ct->pair_off[0] = 0;
    for (int c = 0; c < P; ++c)
        ct->pair_off[c + 1] = ct->pair_off[c] + (ct->tile_off[c + 1] - ct->tile_off[c] + 1) / 2;
    ct->npairs = ct->pair_off[P];
    for (int c = P + 1; c <= kMaxChunks; ++c) ct->off[c] = ct->tile_off[c] = ct->pair_off[c] = 0;
    return CTX_OK;
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int64_t ntiles_upper(int S, int P) {  // tiles of any chunking of S into P chunks
    return (S + kTile - 1) / kTile + P;
}

// ---------------------------------------------------------------- kernels

// Ulysses exchange: y rows (u, b, s) of Hu*D elements, 16-byte vectors
// inside a row.  Each block takes kExRows rows per iteration of a
// block-stride loop and issues all their loads before any store, so that
// enough bytes are in flight to cover HBM latency.
constexpr int kExRows = 4;

__device__ __forceinline__ void exchange_row_index(int64_t ri, int B, int64_t Sp, int layout, int64_t& u,
                                                   int64_t& bb, int64_t& s) {
    u = ri / ((int64_t)B * Sp);
    const int64_t rem = ri - u * B * Sp;
    if (layout == 0) {  // [U][B][Sp]
        bb = rem / Sp;
        s = rem - bb * Sp;
    } else {  // [U][Sp][B]
        s = rem / B;
        bb = rem - s * B;
    }
}

__global__ void exchange_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ y, int B,
                                int S, int Hu, int D, int64_t xsb, int64_t xss, int64_t xsh,
                                int64_t Sp, int layout, int dir, int64_t nrows) {
    const int vec_per_head = D / 8;
    const int vec_per_row = Hu * vec_per_head;
    for (int64_t r0 = (int64_t)blockIdx.x * kExRows; r0 < nrows; r0 += (int64_t)gridDim.x * kExRows) {
        int64_t xrow[kExRows];
        bool real[kExRows], live[kExRows];
#pragma unroll
        for (int k = 0; k < kExRows; ++k) {
            int64_t u, bb, s;
            live[k] = r0 + k < nrows;
            exchange_row_index(live[k] ? r0 + k : 0, B, Sp, layout, u, bb, s);
            real[k] = live[k] && s < S;
            xrow[k] = bb * xsb + s * xss + u * Hu * xsh;
        }
        for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
            const int hh = v / vec_per_head, d8 = v - hh * vec_per_head;
            const int64_t off = hh * xsh + d8 * 8;
            uint4 val[kExRows];
            if (dir == 0) {
#pragma unroll
                for (int k = 0; k < kExRows; ++k)
                    val[k] = real[k] ? *reinterpret_cast<const uint4*>(x + xrow[k] + off) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int k = 0; k < kExRows; ++k)
                    if (live[k]) reinterpret_cast<uint4*>(y + (r0 + k) * Hu * D)[v] = val[k];
            } else {
#pragma unroll
                for (int k = 0; k < kExRows; ++k)
                    if (real[k]) val[k] = reinterpret_cast<const uint4*>(y + (r0 + k) * Hu * D)[v];
#pragma unroll
                for (int k = 0; k < kExRows; ++k)
                    if (real[k]) *reinterpret_cast<uint4*>(const_cast<uint16_t*>(x) + xrow[k] + off) = val[k];
            }
        }
    }
}

// Row statistics for the backward, written in tile-major order
// [B][Hq][ntiles][128]: delta = sum_d dO o O (fp32) and -lse * log2(e)
// (negated, so the backward adds it in one fused multiply-add).  Slots past
// a chunk's end get delta 0 and -inf, which makes their probabilities
// exactly 0 in the backward kernel.  Each thread also zeroes
// its 8 columns of the row's fp32 dQ accumulator (tile-major
// [B][Hq][ntiles][D/4][128][4]), which the backward kernel adds into.
__global__ void bwd_stats_kernel(const __nv_bfloat16* __restrict__ out, int64_t osb, int64_t oss,
                                 int64_t osh, const __nv_bfloat16* __restrict__ dout, int64_t dsb,
                                 int64_t dss, int64_t dsh, const float* __restrict__ lse,
                                 float* __restrict__ nlse2_t, float* __restrict__ delta_t,
                                 float* __restrict__ dq_acc, const ChunkTable ct, int Hq, int S, int D,
                                 int64_t nslots) {
    griddep_wait();  // the previous kernel in the stream is complete (launch_kernel)
    griddep_launch_dependents();
    const int tpr = D / 8;  // threads per row, 8 elements each
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t slot = gt / tpr;
    const int part = (int)(gt - slot * tpr);
    const bool in_range = slot < nslots;
    const int64_t sl = in_range ? slot : 0;
    const int rr = (int)(sl % kTile);
    const int64_t bht = sl / kTile;
    if (in_range) {
        float* tile = dq_acc + bht * kTile * D;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(tile + ((int64_t)(2 * part) * kTile + rr) * 4) = z;
        *reinterpret_cast<float4*>(tile + ((int64_t)(2 * part + 1) * kTile + rr) * 4) = z;
    }
    const int t = (int)(bht % ct.ntiles);
    const int64_t bh = bht / ct.ntiles;
    const int h = (int)(bh % Hq), b = (int)(bh / Hq);
    const int c = chunk_of_tile(ct, t);
    const int s = ct.off[c] + (t - ct.tile_off[c]) * kTile + rr;
    const bool valid = in_range && s < ct.off[c + 1];
    float acc = 0.f;
    if (valid) {
        const uint4 o = *reinterpret_cast<const uint4*>(out + b * osb + (int64_t)s * oss + h * osh + part * 8);
        const uint4 g = *reinterpret_cast<const uint4*>(dout + b * dsb + (int64_t)s * dss + h * dsh + part * 8);
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 a = __bfloat1622float2(o2[k]), d = __bfloat1622float2(g2[k]);
            acc = fmaf(a.x, d.x, acc);
            acc = fmaf(a.y, d.y, acc);
        }
    }
    for (int w = tpr / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w, tpr);
    if (in_range && part == 0) {
        delta_t[slot] = valid ? acc : 0.f;
        nlse2_t[slot] = valid ? -(lse[((int64_t)b * Hq + h) * S + s] * 1.4426950408889634f) : -INFINITY;
    }
}

// dq = scale * dq_acc, from tile-major fp32 [B][Hq][ntiles][D/4][128][4] to
// bf16 rows of the caller's layout.  One thread per 8 columns of a row.
__global__ void dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                  int64_t sb, int64_t ss, int64_t sh, const ChunkTable ct, int Hq,
                                  int D, float scale, int64_t nslots) {
    griddep_wait();  // the previous kernel in the stream is complete (launch_kernel)
    griddep_launch_dependents();
    const int g8 = D / 8;
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gt >= nslots * g8) return;
    const int64_t slot = gt / g8;
    const int k8 = (int)(gt - slot * g8);
    const int rr = (int)(slot % kTile);
    const int64_t bht = slot / kTile;
    const int t = (int)(bht % ct.ntiles);
    const int64_t bh = bht / ct.ntiles;
    const int h = (int)(bh % Hq), b = (int)(bh / Hq);
    const int c = chunk_of_tile(ct, t);
    const int s = ct.off[c] + (t - ct.tile_off[c]) * kTile + rr;
    if (s >= ct.off[c + 1]) return;
    const float* tile = acc + bht * kTile * D;
    const float4 lo = *reinterpret_cast<const float4*>(tile + ((int64_t)(2 * k8) * kTile + rr) * 4);
    const float4 hi = *reinterpret_cast<const float4*>(tile + ((int64_t)(2 * k8 + 1) * kTile + rr) * 4);
    uint4 v = make_uint4(pack_bf16x2(lo.x * scale, lo.y * scale), pack_bf16x2(lo.z * scale, lo.w * scale),
                         pack_bf16x2(hi.x * scale, hi.y * scale), pack_bf16x2(hi.z * scale, hi.w * scale));
    *reinterpret_cast<uint4*>(dq + b * sb + (int64_t)s * ss + h * sh + k8 * 8) = v;
}

// Sum of the head-split partial dK / dV of the D = 256 backward:
// part [hs][B][Hkv][S][2][D] fp32 (dK unscaled, dV) -> dk = scale * sum,
// dv = sum, bf16 rows of the caller's layout.  One thread per 8 columns.
__global__ void dkv_reduce_kernel(const float* __restrict__ part, int hs, int B, int Hkv, int S, int D,
                                  __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                                  int64_t sb, int64_t ss, int64_t sh, float scale) {
    griddep_wait();  // the previous kernel in the stream is complete (launch_kernel)
    griddep_launch_dependents();
    const int g8 = D / 8;
    const int64_t n = (int64_t)B * Hkv * S * 2;  // (b, hk, s, which) rows
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gt >= n * g8) return;
    const int64_t r = gt / g8;
    const int k8 = (int)(gt - r * g8);
    const int which = (int)(r & 1);
    const int64_t bhs = r >> 1;
    const int s = (int)(bhs % S);
    const int64_t bh = bhs / S;
    const int hk = (int)(bh % Hkv), b = (int)(bh / Hkv);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < hs; ++i) {
        const float4* src = reinterpret_cast<const float4*>(part + ((int64_t)i * n + r) * D + k8 * 8);
        const float4 lo = src[0], hi = src[1];
        acc[0] += lo.x; acc[1] += lo.y; acc[2] += lo.z; acc[3] += lo.w;
        acc[4] += hi.x; acc[5] += hi.y; acc[6] += hi.z; acc[7] += hi.w;
    }
    const float f = which == 0 ? scale : 1.f;
    uint4 v = make_uint4(pack_bf16x2(acc[0] * f, acc[1] * f), pack_bf16x2(acc[2] * f, acc[3] * f),
                         pack_bf16x2(acc[4] * f, acc[5] * f), pack_bf16x2(acc[6] * f, acc[7] * f));
    __nv_bfloat16* dst = (which == 0 ? dk : dv) + b * sb + (int64_t)s * ss + hk * sh + k8 * 8;
    *reinterpret_cast<uint4*>(dst) = v;
}

// LSE merge of materialised partials: L = log sum_i exp(LSE_i),
// O = sum_i exp(LSE_i - L) O_i.  part_o [P][B][H][S][D], part_lse [P][B][H][S].
// With causal masking a row of chunk r has partials for iterations 0..r only
// (ring order: chunks r, r-1, .., 0; all-gather order: chunks 0..r); the
// later iterations meet chunks after r, whose weight is zero (LSE = -inf),
// and are never written.  One thread per 4 columns of a row.
__global__ void lse_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                                 int P, int B, int H, int S, int D, __nv_bfloat16* __restrict__ out,
                                 int64_t osb, int64_t oss, int64_t osh, float* __restrict__ lse,
                                 const ChunkTable ct, int causal) {
    griddep_wait();  // the previous kernel in the stream is complete (launch_kernel)
    griddep_launch_dependents();
    const int g4 = D / 4;
    const int64_t nrows = (int64_t)B * H * S;
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gt >= nrows * g4) return;
    const int64_t row = gt / g4;
    const int k4 = (int)(gt - row * g4);
    const int s = (int)(row % S);
    const int64_t bh = row / S;
    const int h = (int)(bh % H), b = (int)(bh / H);
    int n_it = P;
    if (causal) {
        int r = 0;
        while (r + 1 < ct.P && ct.off[r + 1] <= s) ++r;
        n_it = r + 1;
    }
    float m = -INFINITY;
    for (int i = 0; i < n_it; ++i) m = fmaxf(m, part_lse[i * nrows + row]);
    float sum = 0.f;
    for (int i = 0; i < n_it; ++i) sum += __expf(part_lse[i * nrows + row] - m);
    const float L = m + __logf(sum);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < n_it; ++i) {
        const float w = __expf(part_lse[i * nrows + row] - L);
        const float4 pi = *reinterpret_cast<const float4*>(part_o + (i * nrows + row) * D + k4 * 4);
        o.x = fmaf(w, pi.x, o.x);
        o.y = fmaf(w, pi.y, o.y);
        o.z = fmaf(w, pi.z, o.z);
        o.w = fmaf(w, pi.w, o.w);
    }
    uint2 v = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
    *reinterpret_cast<uint2*>(out + b * osb + (int64_t)s * oss + h * osh + k4 * 4) = v;
    if (k4 == 0) lse[row] = L;
}

// Self test of the two exponentials the attention kernels use.
__global__ void exp2_selftest_kernel(const float* __restrict__ x, float* __restrict__ y_poly,
                                     float* __restrict__ y_sfu, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        y_poly[i] = ex2_poly(x[i]);
        y_sfu[i] = ex2(x[i]);
    }
}

// Failure-detection self test: wait on an mbarrier nothing arrives on.
__global__ void wait_timeout_kernel(int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    mbar_fence_init();
    WaitCtx wc{&abort_flag, status, limit_ns};
    mbar_wait(smem_u32(&bar), 0, wc);  // gives up after limit_ns and records the timeout
}

// ---------------------------------------------------------------- profiling
struct KernelTimes {
    static constexpr int kCap = 4096;
    cudaEvent_t ev[2][kCap][2];
    int n[2];
    bool created[2][kCap];
    bool on;
};
KernelTimes g_prof;

void prof_record(int kernel, int which, cudaStream_t s) {
    if (!g_prof.on) return;
    const int i = g_prof.n[kernel];
    if (i >= KernelTimes::kCap) return;
    if (!g_prof.created[kernel][i]) {
        if (cudaEventCreate(&g_prof.ev[kernel][i][0]) != cudaSuccess ||
            cudaEventCreate(&g_prof.ev[kernel][i][1]) != cudaSuccess)
            return;
        g_prof.created[kernel][i] = true;
    }
    cudaEventRecord(g_prof.ev[kernel][i][which], s);
    if (which == 1) g_prof.n[kernel] = i + 1;
}

inline int launch_status(cudaError_t launch = cudaSuccess) {
    return launch == cudaSuccess && cudaGetLastError() == cudaSuccess ? CTX_OK : CTX_ERR_CUDA;
}

size_t fwd_ws_bytes(int B, int S, int Hq, int D, int P, int flags) {
    if (!(flags & CTX_FLAG_MATERIALIZE_PARTIALS)) return 0;
    const size_t rows = (size_t)P * B * Hq * S;
    return align256(rows * D * 4) + align256(rows * 4);
}

// D = 256 backward on short sequences: the query heads of one GQA group may
// be split over d CTAs per (KV tile, column half), each writing fp32 partial
// dK/dV rows that dkv_reduce_kernel sums.  The workspace holds the partial
// rows of the largest split a call may use: the smallest divisor d of the
// group size that brings the grid to at least one CTA per SM of the current
// device at the fewest tiles any chunking of S has (ceil(S / 128)).
int bwd_hsplit_cap(int S, int B, int Hq, int Hkv, int D) {
    if (D != 256) return 1;
    const int G = Hq / Hkv;
    const int nsm = num_sms();
    const int64_t base = (int64_t)((S + kTile - 1) / kTile) * Hkv * 2 * B;
    for (int d = 1; d < G; ++d)
        if (G % d == 0 && base * d >= nsm) return d;
    return G;
}

// Estimated time of the D = 256 backward, in query-tile iterations of one
// CTA, for a split d: the CTAs of KV tile kt each run (query tiles they see)
// x (G / d) iterations plus about one for their prologue, heaviest first,
// each on the first SM that is free (list scheduling); summing d partials
// adds about 0.15 d B Hkv S / 1024.  On the GB300 (24/4 heads, S = 512 ..
// 2048, causal or not) the split with the smallest estimate was the fastest
// measured one in every case.
double bwd_split_time(int64_t nt, int B, int Hkv, int G, int d, int S, int causal, int nsm) {
    std::vector<double> sm((size_t)nsm, 0.0);  // min-heap of SM finish times
    const int64_t per_tile = (int64_t)Hkv * 2 * B * d;
    for (int64_t kt = 0; kt < nt; ++kt) {
        const double w = (double)((causal ? nt - kt : nt) * (G / d)) + 1.0;
        for (int64_t j = 0; j < per_tile; ++j) {
            std::pop_heap(sm.begin(), sm.end(), std::greater<double>());
            sm.back() += w;
            std::push_heap(sm.begin(), sm.end(), std::greater<double>());
        }
    }
    const double span = *std::max_element(sm.begin(), sm.end());
    return span + (d > 1 ? 0.15 * d * B * Hkv * S / 1024.0 : 0.0);
}

// The split a call uses: the one of smallest estimated time up to the cap
// (ties to the smaller split).  Memoised: the estimate runs on the host.
int bwd_hsplit(int64_t ntiles, int S, int B, int Hq, int Hkv, int D, int causal) {
    const int cap = bwd_hsplit_cap(S, B, Hq, Hkv, D);
    if (cap == 1) return 1;
    const int G = Hq / Hkv, nsm = num_sms();
    struct Entry {
        int64_t nt;
        int S, B, Hkv, G, causal, nsm, cap, d;
    };
    static std::mutex mu;
    static Entry memo[32];
    static int n_memo = 0, next_slot = 0;
    const Entry key{ntiles, S, B, Hkv, G, causal ? 1 : 0, nsm, cap, 0};
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_memo; ++i) {
        const Entry& e = memo[i];
        if (e.nt == key.nt && e.S == key.S && e.B == key.B && e.Hkv == key.Hkv && e.G == key.G &&
            e.causal == key.causal && e.nsm == key.nsm && e.cap == key.cap)
            return e.d;
    }
    int best = 1;
    double best_t = 0.0;
    for (int d = 1; d <= cap; ++d) {
        if (G % d) continue;
        const double t = bwd_split_time(ntiles, B, Hkv, G, d, S, causal, nsm);
        if (d == 1 || t < best_t) best = d, best_t = t;
    }
    Entry e = key;
    e.d = best;
    memo[next_slot] = e;
    next_slot = (next_slot + 1) % 32;
    if (n_memo < 32) ++n_memo;
    return best;
}

// Launch decisions of one call, shared by the attention entry points and
// ctx_attn_launch_plan.
int64_t fwd_ctas(const ChunkTable& ct, int B, int Hq, int D) {
    return (int64_t)(D == 256 ? ct.ntiles : ct.npairs) * Hq * B;
}
void bwd_plan(const ChunkTable& ct, int S, int B, int Hq, int Hkv, int D, int causal, int* hsplit,
              int* head_major, int64_t* ctas) {
    int hs = bwd_hsplit(ct.ntiles, S, B, Hq, Hkv, D, causal);
    if ((int64_t)B * 2 * hs > 65535) hs = 1;  // grid limit (the backward takes B <= 32767 for D = 256)
    const int64_t n = (int64_t)ct.ntiles * Hkv * B * (D == 256 ? 2 * hs : 1);
    *hsplit = hs;
    *head_major = pick_head_major(causal, n);
    if (ctas) *ctas = n;
}

size_t bwd_ws_bytes(int B, int S, int Hq, int Hkv, int D, int P) {
    const size_t slots = (size_t)B * Hq * ntiles_upper(S, P) * kTile;
    const int hs = bwd_hsplit_cap(S, B, Hq, Hkv, D);
    const size_t part = hs > 1 ? align256((size_t)hs * B * Hkv * S * 2 * D * 4) : 0;
    return align256(slots * 4) * 2 + align256(slots * D * 4) + part;
}

bool sizes_ok(int B, int S, int Hq, int Hkv, int D) {
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1) return false;
    if (Hq % Hkv) return false;
    if (D < 1) return false;
    if ((int64_t)B * Hq * S > ((int64_t)1 << 40)) return false;
    return true;
}

}  // namespace

extern "C" {

const char* ctx_status_string(int s) {
    switch (s) {
        case CTX_OK: return "ok";
        case CTX_ERR_INVALID_ARG: return "invalid argument";
        case CTX_ERR_UNSUPPORTED: return "unsupported configuration";
        case CTX_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case CTX_ERR_CUDA: return "CUDA error";
        case CTX_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

int ctx_chunk_offsets(int S, int P, int* off) {
    if (!off || P < 1 || P > S) return CTX_ERR_INVALID_ARG;
    const int base = S / P, extra = S % P;
    off[0] = 0;
    for (int c = 0; c < P; ++c) off[c + 1] = off[c] + base + (c < extra ? 1 : 0);
    return CTX_OK;
}

size_t ctx_attn_workspace_size(int B, int S, int Hq, int Hkv, int D, int P, int flags) {
    if (!sizes_ok(B, S, Hq, Hkv, D) || P < 1 || P > S || P > kMaxChunks) return 0;
    const size_t f = fwd_ws_bytes(B, S, Hq, D, P, flags);
    const size_t b = bwd_ws_bytes(B, S, Hq, Hkv, D, P);
    return f > b ? f : b;
}

int ctx_attn_launch_plan(int B, int S, int Hq, int Hkv, int D, int P, const int* chunk_offsets, int causal,
                         ctx_launch_plan_t* plan) {
    if (!plan || !sizes_ok(B, S, Hq, Hkv, D)) return CTX_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256) return CTX_ERR_UNSUPPORTED;
    ChunkTable ct;
    memset(&ct, 0, sizeof(ct));
    const int rc = build_chunks(S, P, chunk_offsets, &ct);
    if (rc) return rc;
    const int c = causal ? 1 : 0;
    plan->fwd_ctas = fwd_ctas(ct, B, Hq, D);
    plan->fwd_head_major = pick_head_major(c, plan->fwd_ctas);
    bwd_plan(ct, S, B, Hq, Hkv, D, c, &plan->bwd_group_split, &plan->bwd_head_major, &plan->bwd_ctas);
    return CTX_OK;
}

int64_t ctx_exchange_padded_len(int64_t S, int ring, int ulysses) {
    if (S < 1 || ring < 1 || ulysses < 1) return -1;
    const int64_t W = (int64_t)ring * ulysses;
    return (S + W - 1) / W * W;
}

int ctx_attn_fwd(const ctx_tensor_t* q, const ctx_tensor_t* k, const ctx_tensor_t* v, int P,
                 const int* chunk_offsets, ctx_layout_t layout, int causal, float scale,
                 const ctx_tensor_t* out, float* lse, void* workspace, size_t workspace_bytes,
                 int flags, ctx_stream_t stream) {
    NvtxRange range("ctx_attn_fwd");
    if (!q || !k || !v || !out || !lse) return CTX_ERR_INVALID_ARG;
    if (layout != CTX_LAYOUT_BSHD && layout != CTX_LAYOUT_SBHD) return CTX_ERR_INVALID_ARG;
    if (flags & ~(CTX_FLAG_MATERIALIZE_PARTIALS | CTX_FLAG_KV_ALLGATHER)) return CTX_ERR_INVALID_ARG;
    const int64_t B = q->B, S = q->S, Hq = q->H, D = q->D, Hkv = k->H;
    if (B > INT32_MAX || S > INT32_MAX || Hq > 65535 || Hkv > 65535 || B > 65535)
        return CTX_ERR_INVALID_ARG;
    if (!sizes_ok((int)B, (int)S, (int)Hq, (int)Hkv, (int)D)) return CTX_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256) return CTX_ERR_UNSUPPORTED;
    Dense dq_, dk_, dv_, do_;
    int rc;
    if ((rc = resolve(q, B, S, Hq, D, layout, &dq_))) return rc;
    if ((rc = resolve(k, B, S, Hkv, D, layout, &dk_))) return rc;
    if ((rc = resolve(v, B, S, Hkv, D, layout, &dv_))) return rc;
    if ((rc = resolve(out, B, S, Hq, D, layout, &do_))) return rc;
    if (reinterpret_cast<uintptr_t>(lse) & 3) return CTX_ERR_INVALID_ARG;
    FwdParams p;
    memset(&p, 0, sizeof(p));
    if ((rc = build_chunks((int)S, P, chunk_offsets, &p.ct))) return rc;
    const bool partials = flags & CTX_FLAG_MATERIALIZE_PARTIALS;
    if (partials) {
        const size_t need = fwd_ws_bytes((int)B, (int)S, (int)Hq, (int)D, P, flags);
        if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
            return CTX_ERR_WORKSPACE;
        const size_t rows = (size_t)P * B * Hq * S;
        p.part_o = static_cast<float*>(workspace);
        p.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * D * 4));
    }
    if (!make_tmap_bshd(&p.tq, dq_.data, B, S, Hq, D, dq_.sb, dq_.ss, dq_.sh, 64, kTile) ||
        !make_tmap_bshd(&p.tk, dk_.data, B, S, Hkv, D, dk_.sb, dk_.ss, dk_.sh, 64, kTile) ||
        // D = 256 streams V in 64-row halves (each half is one PV k-range)
        !make_tmap_bshd(&p.tv, dv_.data, B, S, Hkv, D, dv_.sb, dv_.ss, dv_.sh, 64, D == 256 ? 64 : kTile))
        return CTX_ERR_CUDA;
    p.B = (int)B; p.S = (int)S; p.Hq = (int)Hq; p.Hkv = (int)Hkv;
    p.group = (int)(Hq / Hkv);
    p.causal = causal ? 1 : 0;
    p.allgather = (flags & CTX_FLAG_KV_ALLGATHER) ? 1 : 0;
    p.head_major = pick_head_major(p.causal, fwd_ctas(p.ct, (int)B, (int)Hq, (int)D));
    p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16*>(do_.data);
    p.o_sb = do_.sb; p.o_ss = do_.ss; p.o_sh = do_.sh;
    p.lse = lse;
    p.status = status_ptr();
    p.timeout_ns = timeout_ns();
    p.debug = kernel_debug_bits();
    if (!p.status) return CTX_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    p.pdl = use_pdl(fwd_ctas(p.ct, (int)B, (int)Hq, (int)D), p.ct.ntiles, s);
    if (log_enabled())
        fprintf(stderr,
                "ctx_attn_fwd: B=%d S=%d Hq=%d Hkv=%d D=%d P=%d causal=%d order=%s partials=%d | %d query "
                "tiles, %lld CTAs (%s), grid order %s\n",
                p.B, p.S, p.Hq, p.Hkv, (int)D, P, p.causal, p.allgather ? "all-gather" : "ring", partials ? 1 : 0,
                p.ct.ntiles, (long long)fwd_ctas(p.ct, p.B, p.Hq, (int)D),
                D == 256 ? "attn_fwd256_kernel, one tile per CTA" : "attn_fwd_kernel, two tiles per CTA",
                p.head_major ? "head-major" : "tile-major");
    prof_record(0, 0, s);
    rc = launch_attn_fwd(p, (int)D, s);
    prof_record(0, 1, s);
    if (rc) return rc;
    if (partials) {
        const int64_t threads = B * Hq * S * (D / 4);
        const int blk = 256;
        rc = launch_status(launch_kernel(p.pdl != 0, lse_merge_kernel, dim3((unsigned)((threads + blk - 1) / blk)),
                                         dim3(blk), 0, s,
            p.part_o, p.part_lse, P, (int)B, (int)Hq, (int)S, (int)D, p.out, p.o_sb, p.o_ss, p.o_sh,
            lse, p.ct, p.causal));
        if (rc) return rc;
    }
    return CTX_OK;
}

int ctx_attn_bwd(const ctx_tensor_t* q, const ctx_tensor_t* k, const ctx_tensor_t* v,
                 const ctx_tensor_t* out, const float* lse, const ctx_tensor_t* dout, int P,
                 const int* chunk_offsets, ctx_layout_t layout, int causal, float scale,
                 const ctx_tensor_t* dq, const ctx_tensor_t* dk, const ctx_tensor_t* dv,
                 void* workspace, size_t workspace_bytes, ctx_stream_t stream) {
    NvtxRange range("ctx_attn_bwd");
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return CTX_ERR_INVALID_ARG;
    if (layout != CTX_LAYOUT_BSHD && layout != CTX_LAYOUT_SBHD) return CTX_ERR_INVALID_ARG;
    const int64_t B = q->B, S = q->S, Hq = q->H, D = q->D, Hkv = k->H;
    if (B > INT32_MAX || S > INT32_MAX || Hq > 65535 || Hkv > 65535 || B > 65535)
        return CTX_ERR_INVALID_ARG;
    if (!sizes_ok((int)B, (int)S, (int)Hq, (int)Hkv, (int)D)) return CTX_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256) return CTX_ERR_UNSUPPORTED;
    if (D == 256 && B > 32767) return CTX_ERR_INVALID_ARG;  // grid z = 2 B (column halves)
    Dense tq, tk, tv, to, tdo, tdq, tdk, tdv;
    int rc;
    if ((rc = resolve(q, B, S, Hq, D, layout, &tq))) return rc;
    if ((rc = resolve(k, B, S, Hkv, D, layout, &tk))) return rc;
    if ((rc = resolve(v, B, S, Hkv, D, layout, &tv))) return rc;
    if ((rc = resolve(out, B, S, Hq, D, layout, &to))) return rc;
    if ((rc = resolve(dout, B, S, Hq, D, layout, &tdo))) return rc;
    if ((rc = resolve(dq, B, S, Hq, D, layout, &tdq))) return rc;
    if ((rc = resolve(dk, B, S, Hkv, D, layout, &tdk))) return rc;
    if ((rc = resolve(dv, B, S, Hkv, D, layout, &tdv))) return rc;
    if (tdk.sb != tdv.sb || tdk.ss != tdv.ss || tdk.sh != tdv.sh) return CTX_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(lse) & 3) return CTX_ERR_INVALID_ARG;
    BwdParams p;
    memset(&p, 0, sizeof(p));
    if ((rc = build_chunks((int)S, P, chunk_offsets, &p.ct))) return rc;
    const size_t need = bwd_ws_bytes((int)B, (int)S, (int)Hq, (int)Hkv, (int)D, P);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return CTX_ERR_WORKSPACE;
    const size_t slots = (size_t)B * Hq * p.ct.ntiles * kTile;
    char* ws = static_cast<char*>(workspace);
    float* nlse2_t = reinterpret_cast<float*>(ws);
    float* delta_t = reinterpret_cast<float*>(ws + align256(slots * 4));
    float* dq_acc = reinterpret_cast<float*>(ws + 2 * align256(slots * 4));
    int64_t bwd_ctas = 0;
    bwd_plan(p.ct, (int)S, (int)B, (int)Hq, (int)Hkv, (int)D, causal ? 1 : 0, &p.hsplit, &p.head_major,
             &bwd_ctas);
    p.dkv_part = p.hsplit > 1 ? reinterpret_cast<float*>(ws + 2 * align256(slots * 4) + align256(slots * D * 4))
                              : nullptr;
    if (!make_tmap_bshd(&p.tq, tq.data, B, S, Hq, D, tq.sb, tq.ss, tq.sh, 64, kTile) ||
        !make_tmap_bshd(&p.tk, tk.data, B, S, Hkv, D, tk.sb, tk.ss, tk.sh, 64, kTile) ||
        !make_tmap_bshd(&p.tv, tv.data, B, S, Hkv, D, tv.sb, tv.ss, tv.sh, 64, kTile) ||
        !make_tmap_bshd(&p.tdo, tdo.data, B, S, Hq, D, tdo.sb, tdo.ss, tdo.sh, 64, kTile))
        return CTX_ERR_CUDA;
    p.B = (int)B; p.S = (int)S; p.Hq = (int)Hq; p.Hkv = (int)Hkv;
    p.group = (int)(Hq / Hkv);
    p.causal = causal ? 1 : 0;
    p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.nlse2 = nlse2_t;
    p.delta = delta_t;
    p.dq_acc = dq_acc;
    p.dk = static_cast<__nv_bfloat16*>(tdk.data);
    p.dv = static_cast<__nv_bfloat16*>(tdv.data);
    p.k_sb = tdk.sb; p.k_ss = tdk.ss; p.k_sh = tdk.sh;
    p.status = status_ptr();
    p.timeout_ns = timeout_ns();
    p.debug = kernel_debug_bits();
    if (!p.status) return CTX_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    p.pdl = D == 256 ? 0 : use_pdl(bwd_ctas, p.ct.ntiles, s);
    if (log_enabled())
        fprintf(stderr,
                "ctx_attn_bwd: B=%d S=%d Hq=%d Hkv=%d D=%d P=%d causal=%d | %d KV tiles, %lld CTAs (%s), "
                "GQA group split %d, grid order %s\n",
                p.B, p.S, p.Hq, p.Hkv, (int)D, P, p.causal, p.ct.ntiles, (long long)bwd_ctas,
                D == 256 ? "attn_bwd256_kernel, column halves" : "attn_bwd_kernel, one KV tile per CTA",
                p.hsplit, p.head_major ? "head-major" : "tile-major");
    {
        // row statistics, and the fp32 dQ accumulator zeroed
        const int64_t threads = (int64_t)slots * (D / 8);
        const int blk = 256;
        rc = launch_status(launch_kernel(p.pdl != 0, bwd_stats_kernel, dim3((unsigned)((threads + blk - 1) / blk)),
                                         dim3(blk), 0, s,
            static_cast<const __nv_bfloat16*>(to.data), to.sb, to.ss, to.sh,
            static_cast<const __nv_bfloat16*>(tdo.data), tdo.sb, tdo.ss, tdo.sh, lse, nlse2_t,
            delta_t, dq_acc, p.ct, (int)Hq, (int)S, (int)D, (int64_t)slots));
        if (rc) return rc;
    }
    prof_record(1, 0, s);
    rc = launch_attn_bwd(p, (int)D, s);
    prof_record(1, 1, s);
    if (rc) return rc;
    if (p.dkv_part) {
        const int64_t threads = B * Hkv * S * 2 * (D / 8);
        const int blk = 256;
        rc = launch_status(launch_kernel(p.pdl != 0, dkv_reduce_kernel, dim3((unsigned)((threads + blk - 1) / blk)),
                                         dim3(blk), 0, s,
            p.dkv_part, p.hsplit, (int)B, (int)Hkv, (int)S, (int)D, p.dk, p.dv, p.k_sb, p.k_ss, p.k_sh,
            p.scale));
        if (rc) return rc;
    }
    {
        const int64_t threads = (int64_t)slots * (D / 8);
        const int blk = 256;
        rc = launch_status(launch_kernel(p.pdl != 0, dq_convert_kernel, dim3((unsigned)((threads + blk - 1) / blk)),
                                         dim3(blk), 0, s,
            dq_acc, static_cast<__nv_bfloat16*>(tdq.data), tdq.sb, tdq.ss, tdq.sh, p.ct, (int)Hq,
            (int)D, p.scale, (int64_t)slots));
        if (rc) return rc;
    }
    return CTX_OK;
}

}  // extern "C"

namespace {

// Scratch of ctx_attn_bwd_noalloc: a file-scope device array, so the entry
// point needs no allocation.  Host code only sees a stand-in symbol; the
// device address is looked up once per device with that device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CTX_NOALLOC_SCRATCH_BYTES];

void* noalloc_scratch_ptr() {
    static std::mutex mu;
    static void* ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        ptrs[dev] = p;
    }
    return ptrs[dev];
}

}  // namespace

extern "C" {

int ctx_attn_bwd_noalloc(const ctx_tensor_t* q, const ctx_tensor_t* k, const ctx_tensor_t* v,
                         const ctx_tensor_t* out, const float* lse, const ctx_tensor_t* dout, int P,
                         const int* chunk_offsets, ctx_layout_t layout, int causal, float scale,
                         const ctx_tensor_t* dq, const ctx_tensor_t* dk, const ctx_tensor_t* dv,
                         ctx_stream_t stream) {
    if (!q || !k) return CTX_ERR_INVALID_ARG;
    if (q->B > INT32_MAX || q->S > INT32_MAX || q->H > INT32_MAX || k->H > INT32_MAX || q->D > INT32_MAX)
        return CTX_ERR_INVALID_ARG;
    const size_t need = ctx_attn_workspace_size((int)q->B, (int)q->S, (int)q->H, (int)k->H, (int)q->D, P, 0);
    if (need == 0) return CTX_ERR_INVALID_ARG;
    if (need > (size_t)CTX_NOALLOC_SCRATCH_BYTES) return CTX_ERR_WORKSPACE;
    void* scratch = noalloc_scratch_ptr();
    if (!scratch) return CTX_ERR_CUDA;
    return ctx_attn_bwd(q, k, v, out, lse, dout, P, chunk_offsets, layout, causal, scale, dq, dk, dv,
                        scratch, (size_t)CTX_NOALLOC_SCRATCH_BYTES, stream);
}

int ctx_seq_head_exchange(const ctx_tensor_t* x, void* y, int ring, int ulysses, int dir,
                          ctx_layout_t layout, ctx_stream_t stream) {
    NvtxRange range("ctx_seq_head_exchange");
    if (!x || !x->data || !y || ring < 1 || ulysses < 1 || (dir != 0 && dir != 1))
        return CTX_ERR_INVALID_ARG;
    if (layout != CTX_LAYOUT_BSHD && layout != CTX_LAYOUT_SBHD) return CTX_ERR_INVALID_ARG;
    const int64_t B = x->B, S = x->S, H = x->H, D = x->D;
    if (B < 1 || S < 1 || H < 1 || D < 1 || H % ulysses) return CTX_ERR_INVALID_ARG;
    if (B > INT32_MAX || S > INT32_MAX || H > INT32_MAX) return CTX_ERR_INVALID_ARG;
    if (D % 8 || (reinterpret_cast<uintptr_t>(y) & 15)) return CTX_ERR_UNSUPPORTED;
    Dense tx;
    int rc;
    if ((rc = resolve(x, B, S, H, D, layout, &tx))) return rc;
    const int64_t Sp = ctx_exchange_padded_len(S, ring, ulysses);
    const int Hu = (int)(H / ulysses);
    const int64_t nrows = (int64_t)ulysses * B * Sp;
    const int vec_per_row = Hu * (int)(D / 8);
    int blk = 32;
    while (blk < vec_per_row && blk < 512) blk *= 2;
    const int64_t nblk = (nrows + kExRows - 1) / kExRows;
    const int64_t grid = nblk < (int64_t)num_sms() * 16 ? nblk : (int64_t)num_sms() * 16;
    exchange_kernel<<<(unsigned)grid, blk, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(tx.data), static_cast<uint16_t*>(y), (int)B, (int)S, Hu, (int)D,
        tx.sb, tx.ss, tx.sh, Sp, layout == CTX_LAYOUT_BSHD ? 0 : 1, dir, nrows);
    return launch_status();
}

int ctx_get_device_status(ctx_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CTX_ERR_CUDA;
    int* p = status_ptr();
    if (!p) return CTX_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CTX_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return CTX_ERR_CUDA;
    return v;
}

int ctx_profile_enable(int enable) {
    g_prof.on = enable != 0;
    if (g_prof.on) g_prof.n[0] = g_prof.n[1] = 0;
    return CTX_OK;
}

int ctx_profile_read(int kernel, double* total_ms, int* launches) {
    if ((kernel != 0 && kernel != 1) || !total_ms || !launches) return CTX_ERR_INVALID_ARG;
    double sum = 0.0;
    for (int i = 0; i < g_prof.n[kernel]; ++i) {
        float ms = 0.f;
        if (cudaEventSynchronize(g_prof.ev[kernel][i][1]) != cudaSuccess ||
            cudaEventElapsedTime(&ms, g_prof.ev[kernel][i][0], g_prof.ev[kernel][i][1]) != cudaSuccess)
            return CTX_ERR_CUDA;
        sum += ms;
    }
    *total_ms = sum;
    *launches = g_prof.n[kernel];
    return CTX_OK;
}

int ctx_selftest_exp2(const float* x, float* y_poly, float* y_sfu, int64_t n, ctx_stream_t stream) {
    if (!x || !y_poly || !y_sfu || n < 1 || n > ((int64_t)1 << 31)) return CTX_ERR_INVALID_ARG;
    exp2_selftest_kernel<<<(unsigned)((n + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        x, y_poly, y_sfu, n);
    return launch_status();
}

int ctx_debug_set(unsigned flags, unsigned wait_limit_ms) {
    if (flags & ~(unsigned)CTX_DEBUG_SKIP_ARRIVAL) return CTX_ERR_INVALID_ARG;
    if (wait_limit_ms > 60u * 1000u) return CTX_ERR_INVALID_ARG;
    g_wait_limit_ms.store(wait_limit_ms, std::memory_order_relaxed);
    g_debug_flags.store(flags, std::memory_order_relaxed);
    return CTX_OK;
}

int ctx_kernel_binary_version(int* version) {
    if (!version) return CTX_ERR_INVALID_ARG;
    const int v = attn_fwd_binary_version();
    if (v < 0) return CTX_ERR_CUDA;
    *version = v;
    return CTX_OK;
}

int ctx_selftest_wait_timeout(unsigned timeout_us, ctx_stream_t stream) {
    if (timeout_us == 0 || timeout_us > 10u * 1000u * 1000u) return CTX_ERR_INVALID_ARG;
    int* p = status_ptr();
    if (!p) return CTX_ERR_CUDA;
    wait_timeout_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        p, (uint64_t)timeout_us * 1000ull);
    return launch_status();
}

}  // extern "C"
