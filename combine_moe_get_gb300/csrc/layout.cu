// layout.cu -- routing counts, rank membership and receive rows.
//
// Follows the notify stage of the dispatch kernel on the DeepEP V2 deep-dive
// page ("DeepEP V2 深度深潜", section 3.3 stage 1 and section 3.5): a count per
// expert for every valid top-k entry, a count per rank once per token after
// de-duplicating the token's entries by rank (rank = expert / m, section
// 2.2), then prefix sums. The page hands out receive slots with atomicAdd
// (arrival order); here each rank's rows are ordered by source token, so the
// in-rank position of (t, r) is a column-wise exclusive scan of
// is_token_in_rank over tokens.
//
// Kernel 1 (one CTA per tile of kTile tokens, tiles claimed by an atomic
// ticket so that every predecessor of a tile is already resident):
//   pass 1  lanes hold one top-k entry each; __match_any_sync de-duplicates the
//           (token, rank) pairs, the lowest lane owning each; a shared bitmap
//           [rank][token-word] records membership; a shared histogram counts
//           experts.
//   scan    per rank, popcounts give the tile aggregate; a decoupled lookback
//           (Merrill & Garland, "Single-pass Parallel Prefix Scan with
//           Decoupled Look-back", 2016) over R-wide vectors gives the tile's
//           exclusive prefix. Each (tile, rank) status is one 64-bit word
//           {flag:32 | value:32}, written in one store, so no fence is needed
//           between value and flag. Waits are bounded (MOE_ERR_TIMEOUT).
//   pass 2  the owning lane writes its in-rank position; is_token_in_rank rows
//           are expanded from the bitmap.
//   last    the last CTA to finish (done counter) writes per-rank and
//           per-expert counts and their exclusive prefixes.
// Kernel 2 adds rank_prefix[r] to each owned in-rank position.
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kTile = 128;                 // tokens per tile
constexpr int kWords = kTile / 32;         // bitmap words per rank
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr uint64_t kFlagAggregate = 1ull << 32;
constexpr uint64_t kFlagInclusive = 2ull << 32;

struct WsHeader {
    uint32_t ticket;
    uint32_t done;
    uint32_t pad[30];
};
static_assert(sizeof(WsHeader) == 128, "header is one 128-byte line");

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct WsLayout {
    size_t expert_off, status_off, total;
};

inline WsLayout ws_layout(int T, int E, int R) {
    WsLayout w;
    size_t tiles = (size_t)((T + kTile - 1) / kTile);
    w.expert_off = sizeof(WsHeader);
    w.status_off = align_up(w.expert_off + (size_t)E * 4, 128);
    w.total = align_up(w.status_off + tiles * (size_t)R * 8, 128);
    return w;
}

inline size_t smem_bytes(int E, int R) {
    // bitmap u32 [R][kWords] | word prefix u16 [R][kWords] | exclusive prefix i32 [R] | expert hist i32 [E]
    return align_up((size_t)R * kWords * 4, 16) + align_up((size_t)R * kWords * 2, 16) +
           align_up((size_t)R * 4, 16) + align_up((size_t)E * 4, 16);
}

// Exclusive scan of n int32 counts (read from `in`, copied to `copy_out` when
// non-null) into prefix[0..n]; one CTA of kThreads threads.
__device__ void block_exclusive_scan(const int32_t *in, int n, int32_t *copy_out, int32_t *prefix, bool in_volatile) {
    __shared__ int32_t warp_sums[kWarps];
    __shared__ int32_t carry_total;
    const int per = (n + kThreads - 1) / kThreads;
    const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
    int32_t local = 0;
    for (int i = lo; i < hi; ++i) {
        int32_t v = in_volatile ? *reinterpret_cast<const volatile int32_t *>(in + i) : in[i];
        local += v;
    }
    // inclusive warp scan of the per-thread sums
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t run = 0;
        for (int w = 0; w < kWarps; ++w) {
            int32_t s = warp_sums[w];
            warp_sums[w] = run;
            run += s;
        }
        carry_total = run;
    }
    __syncthreads();
    int32_t run = warp_sums[warp] + incl - local;
    for (int i = lo; i < hi; ++i) {
        int32_t v = in_volatile ? *reinterpret_cast<const volatile int32_t *>(in + i) : in[i];
        if (copy_out) copy_out[i] = v;
        prefix[i] = run;
        run += v;
    }
    if (threadIdx.x == 0) prefix[n] = carry_total;
    __syncthreads();
}

struct TileArgs {
    const int64_t *topk;
    int T, k, E, R, m, num_tiles;
    uint8_t *is_token_in_rank;
    int32_t *token_dst_row;
    int32_t *num_tokens_per_rank, *num_tokens_per_expert, *rank_prefix, *expert_prefix;
    uint8_t *ws;
    size_t expert_off, status_off;
    int32_t *status;
    uint64_t timeout_ns;
    int unpublished_tile;  // test hook: this tile never publishes its status (-1 = none)
};

// Route of one lane: expert e (or -1) and its rank (or -1); flags bad entries.
__device__ __forceinline__ int lane_route(const TileArgs &a, int64_t e, int32_t *status, bool report_bad) {
    if (e == -1) return -1;
    if (e < 0 || e >= a.E) {
        if (report_bad) report(status, MOE_ERR_BAD_TOPK);
        return -1;
    }
    return (int)(e / a.m);
}

__global__ void __launch_bounds__(kThreads) layout_tiles_kernel(TileArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int R = a.R, E = a.E, k = a.k;
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem);
    uint16_t *wprefix = reinterpret_cast<uint16_t *>(smem + align_up((size_t)R * kWords * 4, 16));
    int32_t *excl = reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(wprefix) + align_up((size_t)R * kWords * 2, 16));
    int32_t *hist = reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(excl) + align_up((size_t)R * 4, 16));
    __shared__ int s_tile;
    __shared__ int s_last;

    WsHeader *hdr = reinterpret_cast<WsHeader *>(a.ws);
    int32_t *ws_expert = reinterpret_cast<int32_t *>(a.ws + a.expert_off);
    uint64_t *tile_status = reinterpret_cast<uint64_t *>(a.ws + a.status_off);

    if (threadIdx.x == 0) s_tile = (int)atomicAdd(&hdr->ticket, 1u);
    for (int i = threadIdx.x; i < R * kWords; i += kThreads) bitmap[i] = 0u;
    for (int i = threadIdx.x; i < E; i += kThreads) hist[i] = 0;
    __syncthreads();

    const int tile = s_tile;
    const int t0 = tile * kTile;
    const int tcount = min(kTile, a.T - t0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tpp = 32 / k;                   // tokens per warp pass
    const int sub = lane / k, j = lane - sub * k;
    const bool lane_used = sub < tpp;

    // ---- pass 1: membership bitmap and expert histogram
    for (int base = warp * tpp; base < tcount; base += kWarps * tpp) {
        const int tl = base + sub;
        const bool act = lane_used && tl < tcount;
        int r = -1;
        if (act) {
            int64_t e = ld_nc_i64(a.topk + (int64_t)(t0 + tl) * k + j);
            r = lane_route(a, e, a.status, true);
            if (r >= 0) atomicAdd(&hist[(int)e], 1);
        }
        const int key = (r >= 0) ? (sub * R + r) : -(lane + 1);
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (r >= 0 && (__ffs(peers) - 1) == lane) atomicOr(&bitmap[r * kWords + (tl >> 5)], 1u << (tl & 31));
    }
    __syncthreads();

    // ---- tile aggregates, published for every rank before any lookback
    uint64_t *my_status = tile_status + (size_t)tile * R;
    const bool publish = tile != a.unpublished_tile;
    for (int r = threadIdx.x; r < R; r += kThreads) {
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < kWords; ++w) {
            wprefix[r * kWords + w] = (uint16_t)run;
            run += __popc(bitmap[r * kWords + w]);
        }
        excl[r] = (int32_t)run;   // holds the aggregate until the lookback below
        if (publish) st_relaxed_gpu_u64(my_status + r, (tile == 0 ? kFlagInclusive : kFlagAggregate) | run);
    }
    // ---- decoupled lookback: exclusive prefix of this tile, then its inclusive prefix
    for (int r = threadIdx.x; r < R; r += kThreads) {
        const uint32_t agg = (uint32_t)excl[r];
        uint32_t ex = 0;
        if (tile > 0) {
            int p = tile - 1;
            uint64_t deadline = 0;
            while (p >= 0) {
                const uint64_t w = ld_relaxed_gpu_u64(tile_status + (size_t)p * R + r);
                const uint64_t flag = w & 0xffffffff00000000ull;
                if (flag == 0) {
                    const uint64_t now = globaltimer_ns();
                    if (deadline == 0) {
                        deadline = now + a.timeout_ns;
                    } else if (now > deadline) {
                        report(a.status, MOE_ERR_TIMEOUT);
                        break;
                    }
                    continue;
                }
                ex += (uint32_t)w;
                if (flag == kFlagInclusive) break;
                --p;
            }
            if (publish) st_relaxed_gpu_u64(my_status + r, kFlagInclusive | (ex + agg));
        }
        excl[r] = (int32_t)ex;
    }
    __syncthreads();

    // ---- expert histogram into the global accumulator
    for (int e = threadIdx.x; e < E; e += kThreads) {
        const int h = hist[e];
        if (h) atomicAdd(ws_expert + e, h);
    }

    // ---- pass 2: in-rank positions of the owning lanes
    for (int base = warp * tpp; base < tcount; base += kWarps * tpp) {
        const int tl = base + sub;
        const bool act = lane_used && tl < tcount;
        int r = -1;
        if (act) r = lane_route(a, ld_nc_i64(a.topk + (int64_t)(t0 + tl) * k + j), nullptr, false);
        const int key = (r >= 0) ? (sub * R + r) : -(lane + 1);
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (act) {
            int32_t v = -1;
            if (r >= 0 && (__ffs(peers) - 1) == lane) {
                const uint32_t word = bitmap[r * kWords + (tl >> 5)];
                v = excl[r] + wprefix[r * kWords + (tl >> 5)] + __popc(word & ((1u << (tl & 31)) - 1u));
            }
            a.token_dst_row[(int64_t)(t0 + tl) * k + j] = v;
        }
    }

    // ---- is_token_in_rank rows of this tile, expanded from the bitmap
    uint8_t *dst = a.is_token_in_rank + (int64_t)t0 * R;
    const int nbytes = tcount * R;
    if ((R & 3) == 0) {
        uint32_t *dst4 = reinterpret_cast<uint32_t *>(dst);
        for (int i = threadIdx.x; i < nbytes / 4; i += kThreads) {
            const int tl = (i * 4) / R, r0 = (i * 4) - tl * R;
            uint32_t v = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b)
                v |= ((bitmap[(r0 + b) * kWords + (tl >> 5)] >> (tl & 31)) & 1u) << (8 * b);
            dst4[i] = v;
        }
    } else {
        for (int i = threadIdx.x; i < nbytes; i += kThreads) {
            const int tl = i / R, r = i - tl * R;
            dst[i] = (uint8_t)((bitmap[r * kWords + (tl >> 5)] >> (tl & 31)) & 1u);
        }
    }

    // ---- the last CTA to finish writes counts and prefixes
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(&hdr->done, 1u) == (unsigned)(a.num_tiles - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const uint64_t *last_status = tile_status + (size_t)(a.num_tiles - 1) * R;
    for (int r = threadIdx.x; r < R; r += kThreads) {
        const uint64_t w = ld_relaxed_gpu_u64(last_status + r);
        if ((w & 0xffffffff00000000ull) != kFlagInclusive) report(a.status, MOE_ERR_TIMEOUT);
        a.num_tokens_per_rank[r] = (int32_t)(uint32_t)w;
    }
    __syncthreads();
    __threadfence_block();
    block_exclusive_scan(a.num_tokens_per_rank, R, nullptr, a.rank_prefix, true);
    block_exclusive_scan(ws_expert, E, a.num_tokens_per_expert, a.expert_prefix, true);
}

__global__ void layout_rows_kernel(const int64_t *__restrict__ topk, int64_t n, int m,
                                   const int32_t *__restrict__ rank_prefix, int32_t *__restrict__ token_dst_row) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = token_dst_row[i];
        if (v >= 0) token_dst_row[i] = v + rank_prefix[(int)(topk[i] / m)];
    }
}

}  // namespace

size_t layout_workspace_bytes(int T, int E, int R) { return ws_layout(T, E, R).total; }

int launch_layout(const LayoutLaunch &L) {
    const int T = L.num_tokens, k = L.num_topk, E = L.num_experts, R = L.num_ranks;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(L.stream);
    const moe_layout_t &o = L.out;
    if (T == 0) {
        if (cudaMemsetAsync(o.num_tokens_per_rank, 0, (size_t)R * 4, s) != cudaSuccess ||
            cudaMemsetAsync(o.num_tokens_per_expert, 0, (size_t)E * 4, s) != cudaSuccess ||
            cudaMemsetAsync(o.rank_prefix, 0, (size_t)(R + 1) * 4, s) != cudaSuccess ||
            cudaMemsetAsync(o.expert_prefix, 0, (size_t)(E + 1) * 4, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    const WsLayout w = ws_layout(T, E, R);
    if (cudaMemsetAsync(L.workspace, 0, w.total, s) != cudaSuccess) return MOE_ERR_CUDA;

    TileArgs a;
    a.topk = L.topk_idx;
    a.T = T; a.k = k; a.E = E; a.R = R; a.m = E / R;
    a.num_tiles = (T + kTile - 1) / kTile;
    a.is_token_in_rank = o.is_token_in_rank;
    a.token_dst_row = o.token_dst_row;
    a.num_tokens_per_rank = o.num_tokens_per_rank;
    a.num_tokens_per_expert = o.num_tokens_per_expert;
    a.rank_prefix = o.rank_prefix;
    a.expert_prefix = o.expert_prefix;
    a.ws = static_cast<uint8_t *>(L.workspace);
    a.expert_off = w.expert_off;
    a.status_off = w.status_off;
    a.status = L.status;
    a.timeout_ns = L.timeout_ns > 0 ? (uint64_t)L.timeout_ns : kDefaultWaitNs;
    a.unpublished_tile = L.unpublished_tile;

    const size_t smem = smem_bytes(E, R);
    if (ensure_dynamic_smem((const void *)layout_tiles_kernel, smem) != MOE_OK) return MOE_ERR_CUDA;
    layout_tiles_kernel<<<a.num_tiles, kThreads, smem, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;

    const int64_t n = (int64_t)T * k;
    const int threads = 256;
    int blocks = (int)std::min<int64_t>((n + threads - 1) / threads, (int64_t)device_sm_count() * 8);
    layout_rows_kernel<<<blocks, threads, 0, s>>>(L.topk_idx, n, a.m, o.rank_prefix, o.token_dst_row);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace moe

// ------------------------------------------------------------------ layout without caller workspace
//
// moe_get_layout_noalloc serves callers that cannot allocate device memory
// themselves -- for example a plugin inside a host framework that owns every
// device allocation and hands out no workspace, or a latency-critical loop in
// which a cudaMalloc (which may synchronise the device) is not acceptable.
// Its lookback scratch is this file-scope device array, which every GPU that
// loads the library holds until the process exits. Host code cannot use the
// array's name as a device address (on the host it names a stand-in object),
// so the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device; that first call should therefore come before any stream
// capture. All calls share the array and it keeps the previous call's
// contents: each call clears the part it uses (cudaMemsetAsync on its
// stream), and calls whose executions overlap on the GPU race on it.
namespace moe {
namespace {

static __device__ __align__(256) uint8_t g_layout_scratch[MOE_NOALLOC_SCRATCH_BYTES];

void *noalloc_scratch_address(int *err) {
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *err = MOE_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess || p == nullptr) {
            *err = MOE_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    return addr[dev];
}

bool is_aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace moe

extern "C" MOE_API int moe_get_layout_noalloc(const int64_t *topk_idx, int num_tokens, int num_topk,
                                              int num_experts, int num_ranks, moe_layout_t layout,
                                              int32_t *status, void *stream) {
    const int T = num_tokens, k = num_topk, E = num_experts, R = num_ranks;
    if (T < 0 || k < 1 || k > MOE_MAX_TOPK || R < 1 || R > MOE_MAX_RANKS || E < 1 || E > MOE_MAX_EXPERTS ||
        E % R != 0 || (int64_t)T * k >= ((int64_t)1 << 31) || (int64_t)T * R >= ((int64_t)1 << 40))
        return MOE_ERR_INVALID_ARG;
    if (!status || !layout.num_tokens_per_rank || !layout.num_tokens_per_expert || !layout.rank_prefix ||
        !layout.expert_prefix)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !layout.is_token_in_rank || !layout.token_dst_row)) return MOE_ERR_INVALID_ARG;
    if (!moe::is_aligned(status, 4) || !moe::is_aligned(layout.num_tokens_per_rank, 4) ||
        !moe::is_aligned(layout.num_tokens_per_expert, 4) || !moe::is_aligned(layout.rank_prefix, 4) ||
        !moe::is_aligned(layout.expert_prefix, 4))
        return MOE_ERR_MISALIGNED;
    if (T > 0 && (!moe::is_aligned(topk_idx, 8) || !moe::is_aligned(layout.token_dst_row, 4) ||
                  !moe::is_aligned(layout.is_token_in_rank, 4)))
        return MOE_ERR_MISALIGNED;
    if (moe::layout_workspace_bytes(T, E, R) > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
    int err = MOE_OK;
    void *scratch = moe::noalloc_scratch_address(&err);
    if (scratch == nullptr) return err;
    moe::LayoutLaunch L;
    L.topk_idx = topk_idx;
    L.num_tokens = T;
    L.num_topk = k;
    L.num_experts = E;
    L.num_ranks = R;
    L.out = layout;
    L.workspace = scratch;
    L.status = status;
    L.stream = stream;
    L.timeout_ns = 0;
    L.unpublished_tile = -1;
    return moe::launch_layout(L);
}
