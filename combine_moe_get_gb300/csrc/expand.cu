// expand.cu -- receive rows of expand mode: one row per valid top-k entry,
// grouped by expert.
//
// Follows the copy epilogue of the DeepEP V2 deep-dive page ("DeepEP V2
// 深度深潜", section 3.3 stage 3) in expand mode: a received token's
// destination comes from a counter per expert that starts at the exclusive
// prefix of the per-expert counts (psum_num_recv_tokens_per_expert) and
// advances by one per placed token. The page advances the counter with
// atomicAdd (arrival order); here the entries of each expert are placed in
// source order -- token ascending, then choice index ascending -- so
//   row(t, j) = expert_prefix[e] + #{(t', j') < (t, j) : topk_idx[t', j'] == e},
// a column-wise exclusive scan over tokens of the one-hot expert matrix.
//
// One CTA of 256 threads per tile of 256 tokens, tiles claimed by an atomic
// ticket (so every predecessor of a tile has started and never waits on it):
//   load    the tile's top-k entries into shared memory as 16-bit expert ids.
//   count   each warp walks its 32 tokens in order; __match_any_sync groups
//           the lanes naming one expert, and a per-warp counter per expert
//           gives each entry its rank among the warp's entries of that expert.
//   scan    per expert, the warp counters become exclusive offsets and their
//           sum, the tile aggregate, is published for every expert first;
//           then a decoupled lookback (Merrill & Garland, 2016) over E-wide
//           vectors gives the tile's exclusive prefix. Each thread reads a
//           window of 8 predecessor statuses per step (independent loads in
//           flight together). A status is one 64-bit word {flag | value}, so
//           value and flag change together; waits are bounded
//           (MOE_ERR_TIMEOUT).
//   rows    expert_prefix[e] + tile prefix + warp offset + rank in the warp.
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kXTile = 256;                       // tokens per tile
constexpr int kXThreads = 256;
constexpr int kXWarps = kXThreads / 32;
constexpr int kXWarpTokens = kXTile / kXWarps;    // tokens walked by one warp
constexpr int kWindow = 8;                        // predecessors read per lookback step
constexpr uint64_t kFlagAggregate = 1ull << 32;
constexpr uint64_t kFlagInclusive = 2ull << 32;
constexpr uint64_t kFlagMask = 0xffffffff00000000ull;
constexpr size_t kHeaderBytes = 128;              // ticket counter, one 128-byte line

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Shared memory: warp counters u16 [kXWarps][E] | tile base i32 [E] |
// expert ids i16 [kXTile * k] | rank in warp u16 [kXTile * k]
struct XSmem {
    size_t base, eid, rank, total;
};

__host__ __device__ inline XSmem xsmem(int E, int k) {
    XSmem s;
    s.base = align_up((size_t)kXWarps * E * 2, 16);
    s.eid = s.base + align_up((size_t)E * 4, 16);
    s.rank = s.eid + align_up((size_t)kXTile * k * 2, 16);
    s.total = s.rank + align_up((size_t)kXTile * k * 2, 16);
    return s;
}

struct ExpandArgs {
    const int64_t *topk;
    int T, k, E, num_tiles;
    const int32_t *expert_prefix;
    int32_t *token_expert_row;
    uint8_t *ws;
    int32_t *status;
    uint64_t timeout_ns;
    int unpublished_tile;  // test hook: this tile never publishes its status (-1 = none)
    TraceArgs trace;       // MOE_PROFILE builds: where the warps' records go
};

__global__ void __launch_bounds__(kXThreads) layout_expand_kernel(const ExpandArgs a) {
    WarpTrace wt(a.trace, MOE_TRACE_EXPAND_LAYOUT);
    extern __shared__ __align__(16) uint8_t smem[];
    const int E = a.E, k = a.k;
    const XSmem sl = xsmem(E, k);
    uint16_t *cnt = reinterpret_cast<uint16_t *>(smem);
    int32_t *base = reinterpret_cast<int32_t *>(smem + sl.base);
    int16_t *eid = reinterpret_cast<int16_t *>(smem + sl.eid);
    uint16_t *rank = reinterpret_cast<uint16_t *>(smem + sl.rank);
    __shared__ int s_tile;

    uint32_t *ticket = reinterpret_cast<uint32_t *>(a.ws);
    uint64_t *tile_status = reinterpret_cast<uint64_t *>(a.ws + kHeaderBytes);

    grid_dependency_wait();
    if (threadIdx.x == 0) s_tile = (int)atomicAdd(ticket, 1u);
    for (int i = threadIdx.x; i < kXWarps * E / 2; i += kXThreads) reinterpret_cast<uint32_t *>(cnt)[i] = 0u;
    __syncthreads();
    const int tile = s_tile;
    const int t0 = tile * kXTile;
    const int tcount = min(kXTile, a.T - t0);
    const int n_ent = tcount * k;

    // ---- the tile's entries as expert ids (-1: masked or invalid)
    for (int i = threadIdx.x; i < n_ent; i += kXThreads) {
        const int64_t v = ld_nc_i64(a.topk + (int64_t)t0 * k + i);
        int16_t e = -1;
        if (v >= 0 && v < E) e = (int16_t)v;
        else if (v != -1) report(a.status, MOE_ERR_BAD_TOPK);
        eid[i] = e;
    }
    __syncthreads();

    // ---- each warp ranks its tokens' entries per expert, in (token, choice) order
    {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const int tpp = 32 / k;                 // tokens per pass
        const int sub = lane / k, j = lane - sub * k;
        const bool lane_used = sub < tpp;
        const unsigned lt = (1u << lane) - 1u;
        uint16_t *my_cnt = cnt + (size_t)warp * E;
        const int wt0 = warp * kXWarpTokens;
        for (int b = 0; b < kXWarpTokens && wt0 + b < tcount; b += tpp) {
            const int tw = b + sub;
            const int tl = wt0 + tw;
            const bool act = lane_used && tw < kXWarpTokens && tl < tcount;
            const int e = act ? (int)eid[tl * k + j] : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, e >= 0 ? e : -(lane + 1));
            const int r = (e >= 0) ? (int)my_cnt[e] + __popc(peers & lt) : 0;
            __syncwarp();
            if (e >= 0 && (peers & lt) == 0) my_cnt[e] = (uint16_t)(my_cnt[e] + __popc(peers));
            __syncwarp();
            if (act) rank[tl * k + j] = (e >= 0) ? (uint16_t)r : (uint16_t)0xffffu;
        }
    }
    __syncthreads();

    // ---- warp offsets and tile aggregates, published for every expert before any lookback
    uint64_t *my_status = tile_status + (size_t)tile * E;
    const bool publish = tile != a.unpublished_tile;
    for (int e = threadIdx.x; e < E; e += kXThreads) {
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < kXWarps; ++w) {
            const uint32_t c = cnt[(size_t)w * E + e];
            cnt[(size_t)w * E + e] = (uint16_t)run;
            run += c;
        }
        base[e] = (int32_t)run;    // the aggregate until the lookback below
        if (publish) st_relaxed_gpu_u64(my_status + e, (tile == 0 ? kFlagInclusive : kFlagAggregate) | run);
    }

    // ---- decoupled lookback, one thread per expert, kWindow predecessors per step
    for (int e = threadIdx.x; e < E; e += kXThreads) {
        const uint32_t agg = (uint32_t)base[e];
        uint32_t ex = 0;
        if (tile > 0) {
            int p_hi = tile - 1;
            uint64_t deadline = 0;
            while (true) {
                uint64_t w[kWindow];
#pragma unroll
                for (int i = 0; i < kWindow; ++i) {
                    const int p = p_hi - i;
                    w[i] = (p >= 0) ? ld_relaxed_gpu_u64(tile_status + (size_t)p * E + e) : kFlagInclusive;
                }
                bool ready = true, found = false;
                uint32_t sum = 0;
#pragma unroll
                for (int i = 0; i < kWindow; ++i) {
                    if (ready && !found) {
                        const uint64_t f = w[i] & kFlagMask;
                        if (f == 0) {
                            ready = false;
                        } else {
                            sum += (uint32_t)w[i];
                            found = f == kFlagInclusive;
                        }
                    }
                }
                if (!ready) {                    // a needed predecessor has not published yet
                    const uint64_t now = globaltimer_ns();
                    if (deadline == 0) {
                        deadline = now + a.timeout_ns;
                    } else if (now > deadline) {
                        report(a.status, MOE_ERR_TIMEOUT);
                        break;
                    }
                    continue;
                }
                ex += sum;
                if (found) break;
                p_hi -= kWindow;
            }
            if (publish) st_relaxed_gpu_u64(my_status + e, kFlagInclusive | (ex + agg));
        }
        base[e] = a.expert_prefix[e] + (int32_t)ex;
    }
    __syncthreads();

    // ---- rows
    for (int i = threadIdx.x; i < n_ent; i += kXThreads) {
        const int e = eid[i];
        int32_t row = -1;
        if (e >= 0) {
            const int w = (i / k) / kXWarpTokens;
            row = base[e] + (int32_t)cnt[(size_t)w * E + e] + (int32_t)rank[i];
        }
        a.token_expert_row[(int64_t)t0 * k + i] = row;
    }
}


// ------------------------------------------------------------------ cluster mode
//
// For T <= 16 * 256: one thread-block cluster of 16 CTAs (1024 threads), each a
// contiguous tile of up to 256 tokens. The per-warp ranks and warp offsets are
// those of the tiled kernel above; the tiles' per-expert aggregates are
// exchanged through distributed shared memory between two cluster barriers,
// so there is no workspace, no clear and no wait that could expire.

constexpr int kXCThreads = 1024;
constexpr int kXCWarps = kXCThreads / 32;
constexpr int kXCMax = 16;             // CTAs per cluster
constexpr int kXCMaxTile = 256;        // tokens per CTA
constexpr int kXCMaxExperts = 1024;    // per-warp counters: kXCWarps * E * 2 bytes

// Shared memory: warp counters u16 [kXCWarps][E] | tile aggregate i32 [E] |
// row base i32 [E] | expert ids i16 [tile * k] | rank in warp u16 [tile * k]
struct XCSmem {
    size_t agg, base, eid, rank, total;
};

__host__ __device__ inline XCSmem xcsmem(int tile, int E, int k) {
    XCSmem s;
    s.agg = align_up((size_t)kXCWarps * E * 2, 16);
    s.base = s.agg + align_up((size_t)E * 4, 16);
    s.eid = s.base + align_up((size_t)E * 4, 16);
    s.rank = s.eid + align_up((size_t)tile * k * 2, 16);
    s.total = s.rank + align_up((size_t)tile * k * 2, 16);
    return s;
}

__device__ __forceinline__ uint32_t x_cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void x_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ int32_t x_ld_cluster(const void *local, uint32_t rank) {
    uint32_t remote;
    int32_t v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

struct ExpandClusterArgs {
    const int64_t *topk;
    int T, k, E, tile;
    const int32_t *expert_prefix;
    int32_t *token_expert_row;
    int32_t *status;
    TraceArgs trace;
};

__global__ void __launch_bounds__(kXCThreads) layout_expand_cluster_kernel(const ExpandClusterArgs a) {
    WarpTrace wt(a.trace, MOE_TRACE_EXPAND_LAYOUT_CLUSTER);
    extern __shared__ __align__(16) uint8_t smem[];
    const int E = a.E, k = a.k, tile = a.tile;
    const XCSmem sl = xcsmem(tile, E, k);
    uint16_t *cnt = reinterpret_cast<uint16_t *>(smem);
    int32_t *agg = reinterpret_cast<int32_t *>(smem + sl.agg);
    int32_t *base = reinterpret_cast<int32_t *>(smem + sl.base);
    int16_t *eid = reinterpret_cast<int16_t *>(smem + sl.eid);
    uint16_t *rank = reinterpret_cast<uint16_t *>(smem + sl.rank);

    const int C = (int)gridDim.x;
    const int c = (int)x_cluster_ctarank();
    const int t0 = c * tile;
    const int tcount = max(0, min(tile, a.T - t0));
    const int n_ent = tcount * k;
    const int wtok = tile / kXCWarps;   // tokens walked by one warp (tile is a multiple of kXCWarps)
    grid_dependency_wait();
    grid_launch_dependents();

    for (int i = threadIdx.x; i < kXCWarps * E / 2; i += kXCThreads) reinterpret_cast<uint32_t *>(cnt)[i] = 0u;
    // ---- the tile's entries as expert ids (-1: masked or invalid), 8 loads in flight per thread
    for (int b0 = threadIdx.x; b0 < n_ent; b0 += 8 * kXCThreads) {
        int64_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b0 + u * kXCThreads;
            v[u] = i < n_ent ? ld_nc_i64(a.topk + (int64_t)t0 * k + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b0 + u * kXCThreads;
            if (i < n_ent) {
                int16_t e = -1;
                if (v[u] >= 0 && v[u] < E) e = (int16_t)v[u];
                else if (v[u] != -1) report(a.status, MOE_ERR_BAD_TOPK);
                eid[i] = e;
            }
        }
    }
    __syncthreads();

    // ---- each warp ranks its tokens' entries per expert, in (token, choice) order
    {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const int tpp = 32 / k;                 // tokens per pass
        const int sub = lane / k, j = lane - sub * k;
        const bool lane_used = sub < tpp;
        const unsigned lt = (1u << lane) - 1u;
        uint16_t *my_cnt = cnt + (size_t)warp * E;
        const int wt0 = warp * wtok;
        for (int b = 0; b < wtok && wt0 + b < tcount; b += tpp) {
            const int tw = b + sub;
            const int tl = wt0 + tw;
            const bool act = lane_used && tw < wtok && tl < tcount;
            const int e = act ? (int)eid[tl * k + j] : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, e >= 0 ? e : -(lane + 1));
            const int r = (e >= 0) ? (int)my_cnt[e] + __popc(peers & lt) : 0;
            __syncwarp();
            if (e >= 0 && (peers & lt) == 0) my_cnt[e] = (uint16_t)(my_cnt[e] + __popc(peers));
            __syncwarp();
            if (act) rank[tl * k + j] = (e >= 0) ? (uint16_t)r : (uint16_t)0xffffu;
        }
    }
    __syncthreads();

    // ---- warp offsets and the tile's aggregate per expert
    for (int e = threadIdx.x; e < E; e += kXCThreads) {
        uint32_t run = 0;
        for (int w = 0; w < kXCWarps; ++w) {
            const uint32_t cw = cnt[(size_t)w * E + e];
            cnt[(size_t)w * E + e] = (uint16_t)run;
            run += cw;
        }
        agg[e] = (int32_t)run;
    }

    // ---- exclusive prefix over the lower tiles, through distributed shared memory
    x_cluster_sync();
    for (int e = threadIdx.x; e < E; e += kXCThreads) {
        int32_t v[kXCMax];
#pragma unroll
        for (int cc = 0; cc < kXCMax; ++cc) v[cc] = cc < c ? x_ld_cluster(agg + e, (uint32_t)cc) : 0;
        int32_t ex = 0;
#pragma unroll
        for (int cc = 0; cc < kXCMax; ++cc) ex += v[cc];
        base[e] = a.expert_prefix[e] + ex;
    }
    x_cluster_sync();   // no tile reads another's shared memory after this
    (void)C;

    // ---- rows
    for (int i = threadIdx.x; i < n_ent; i += kXCThreads) {
        const int e = eid[i];
        int32_t row = -1;
        if (e >= 0) {
            const int w = (i / k) / wtok;
            row = base[e] + (int32_t)cnt[(size_t)w * E + e] + (int32_t)rank[i];
        }
        a.token_expert_row[(int64_t)t0 * k + i] = row;
    }
}

}  // namespace

size_t expand_workspace_bytes(int T, int E) {
    const size_t tiles = (size_t)((T + kXTile - 1) / kXTile);
    return align_up(kHeaderBytes + tiles * (size_t)E * 8, 128);
}

namespace {

// Cluster mode for this batch (16 CTAs of up to 256 tokens), or false.
bool expand_cluster_config(int T, int E, int k, int &tile, size_t &smem) {
    if (T > kXCMax * kXCMaxTile || E > kXCMaxExperts || tuning().layout_cluster != kXCMax) return false;
    tile = (int)align_up((size_t)((T + kXCMax - 1) / kXCMax), kXCWarps);
    smem = xcsmem(tile, E, k).total;
    if (smem > device_smem_optin()) return false;
    struct Entry { int dev; size_t smem; bool ok; };
    static std::mutex mu;
    static Entry cache[16];
    static int n_cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < std::min(n_cached, 16); ++i)
        if (cache[i].dev == dev && cache[i].smem == smem) return cache[i].ok;
    const void *fn = (const void *)layout_expand_cluster_kernel;
    bool ok = ensure_dynamic_smem(fn, smem) == MOE_OK &&
              cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kXCMax);
        cfg.blockDim = dim3(kXCThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kXCMax;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        ok = cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) == cudaSuccess && clusters >= 1;
    }
    cudaGetLastError();   // a refused attribute or query only means: no cluster mode
    cache[n_cached % 16] = Entry{dev, smem, ok};
    ++n_cached;
    return ok;
}

}  // namespace

int launch_expand_layout(const ExpandLaunch &L) {
    const int T = L.num_tokens, k = L.num_topk, E = L.num_experts;
    if (T == 0) return MOE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(L.stream);
    int tile = 0;
    size_t csmem = 0;
    if (L.unpublished_tile < 0 && !L.no_cluster && expand_cluster_config(T, E, k, tile, csmem)) {
        ExpandClusterArgs c;
        c.trace = trace_args();
        c.topk = L.topk_idx;
        c.T = T; c.k = k; c.E = E; c.tile = tile;
        c.expert_prefix = L.expert_prefix;
        c.token_expert_row = L.token_expert_row;
        c.status = L.status;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kXCMax);
        cfg.blockDim = dim3(kXCThreads);
        cfg.dynamicSmemBytes = csmem;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kXCMax;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = tuning().overlap != 0 ? 2 : 1;
        return cudaLaunchKernelEx(&cfg, layout_expand_cluster_kernel, c) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    const size_t ws = expand_workspace_bytes(T, E);
    if (cudaMemsetAsync(L.workspace, 0, ws, s) != cudaSuccess) return MOE_ERR_CUDA;
    ExpandArgs a;
    a.trace = trace_args();
    a.topk = L.topk_idx;
    a.T = T; a.k = k; a.E = E;
    a.num_tiles = (T + kXTile - 1) / kXTile;
    a.expert_prefix = L.expert_prefix;
    a.token_expert_row = L.token_expert_row;
    a.ws = static_cast<uint8_t *>(L.workspace);
    a.status = L.status;
    a.timeout_ns = L.timeout_ns > 0 ? (uint64_t)L.timeout_ns : kDefaultWaitNs;
    a.unpublished_tile = L.unpublished_tile;
    const size_t smem = xsmem(E, k).total;
    if (smem > device_smem_optin()) return MOE_ERR_INVALID_ARG;
    if (ensure_dynamic_smem((const void *)layout_expand_kernel, smem) != MOE_OK) return MOE_ERR_CUDA;
    return launch_kernel(layout_expand_kernel, dim3(a.num_tiles), dim3(kXThreads), smem, s, tuning().overlap != 0, a) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

}  // namespace moe
