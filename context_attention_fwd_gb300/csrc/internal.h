// internal.h -- parameter blocks and launchers shared by the translation
// units of the library (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "tmap.h"

namespace ctxattn {

constexpr int kMaxChunks = 64;
constexpr int kTile = 128;  // rows of a query or key/value tile

// Test-only switches carried by the parameter blocks (values of the
// CTX_DEBUG_* bits of the C ABI).  kDebugSkipArrival: the TMA producers of
// the attention kernel issue no loads (and so no mbarrier arrivals) from
// their second load step on, so a consumer's bounded wait runs out and the
// kernel takes its abort path.  The producers stop rather than leave out a
// single step: with one step missing, the later loads into a ring slot
// would wait on an empty barrier that lags one phase behind, which a parity
// wait cannot tell from a completed release, and would overrun the slot.
constexpr int kDebugSkipArrival = 1;

// Index of the load step at which a producer stops under kDebugSkipArrival,
// or -1: the second of n steps (the first when there is only one).
__host__ __device__ inline int debug_skip_step(int debug, int n) {
    return (debug & kDebugSkipArrival) ? (n > 1 ? 1 : 0) : -1;
}

// A set-up that is done once per device (a kernel's shared-memory limit is
// an attribute of the function on each device; setting it on every launch
// costs host time).  f() returns true on success.
// Launches a kernel of the attention calls.  With pdl set it uses
// programmatic stream serialization: the kernel may be scheduled while the
// previous kernel in the stream finishes, and waits for it (griddep_wait in
// ptx.cuh) before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct OncePerDevice {
    std::atomic<uint64_t> done{0};
    template <typename F>
    bool run(F&& f) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return false;
        const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
        if (bit && (done.load(std::memory_order_acquire) & bit)) return true;
        if (!f()) return false;
        if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
        return true;
    }
};

// Ring chunk table: chunk c holds rows [off[c], off[c+1]) and 128-row tiles
// [tile_off[c], tile_off[c+1]) of the tile numbering (tiles never straddle
// a chunk boundary; a chunk's last tile may be partial).
struct ChunkTable {
    int P;
    int ntiles;  // tile_off[P]
    int npairs;  // pair_off[P]
    int off[kMaxChunks + 1];
    int tile_off[kMaxChunks + 1];
    int pair_off[kMaxChunks + 1];  // forward CTAs: pairs of consecutive tiles of one chunk
};

__host__ __device__ inline int chunk_of_tile(const ChunkTable& ct, int t) {
    int c = 0;
    while (c + 1 < ct.P && ct.tile_off[c + 1] <= t) ++c;
    return c;
}

struct FwdParams {
    TmaMap tq, tk, tv;
    ChunkTable ct;
    int B, S, Hq, Hkv, group;
    int causal;        // key j visible to query i iff j <= i (global row indices)
    int allgather;     // visit KV chunks in order 0..P-1 instead of the ring order
    float scale;       // softmax scale
    float scale_log2;  // scale * log2(e)
    __nv_bfloat16* out;
    int64_t o_sb, o_ss, o_sh;
    float* lse;  // [B,Hq,S]
    // materialised partials (nullptr unless requested):
    // part_o [P][B][Hq][S][D] fp32 normalised, part_lse [P][B][Hq][S] natural log
    float* part_o;
    float* part_lse;
    int* status;
    uint64_t timeout_ns;
    int head_major;  // launch order of the attention kernel (grid_pos in walk.cuh)
    int debug;       // kDebug* bits (0 in normal use)
    int pdl;         // launch with programmatic stream serialization (launch_kernel)
};

struct BwdParams {
    TmaMap tq, tk, tv, tdo;
    ChunkTable ct;
    int B, S, Hq, Hkv, group;
    int causal;
    float scale, scale_log2;
    // per-row statistics in tile-major order [B][Hq][ntiles][128]:
    const float* nlse2;  // -lse * log2(e)
    const float* delta;  // rowsum(dO o O)
    // fp32 dQ accumulator, tile-major [B][Hq][ntiles][D/4][128][4], zeroed
    float* dq_acc;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int64_t k_sb, k_ss, k_sh;  // strides of dk/dv
    // D = 256 only: the query heads of a GQA group are split over hsplit
    // CTAs per (KV tile, column half); with hsplit > 1 each writes fp32
    // partial dK (unscaled) / dV to dkv_part [hsplit][B][Hkv][S][2][D] and
    // dkv_reduce_kernel sums them
    int hsplit;
    float* dkv_part;
    int* status;
    uint64_t timeout_ns;
    int head_major;  // launch order of the attention kernel (grid_pos in walk.cuh)
    int debug;       // kDebug* bits (0 in normal use)
    int pdl;         // launch with programmatic stream serialization (launch_kernel)
};

int launch_attn_fwd(const FwdParams& p, int D, cudaStream_t s);
int launch_attn_bwd(const BwdParams& p, int D, cudaStream_t s);
// head dimension 256 (attn_d256.cu); the forward's V map uses 64-row boxes
int launch_attn_fwd256(const FwdParams& p, cudaStream_t s);
int launch_attn_bwd256(const BwdParams& p, cudaStream_t s);
// cudaFuncAttributes::binaryVersion of the D = 128 forward kernel (the
// architecture its machine code was built for, e.g. 103), or -1
int attn_fwd_binary_version();

}  // namespace ctxattn
