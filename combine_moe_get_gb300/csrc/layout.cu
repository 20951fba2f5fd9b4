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
// One CTA per tile of kTile tokens:
//   pass 1  lanes hold one top-k entry each; __match_any_sync de-duplicates the
//           (token, rank) pairs, the lowest lane owning each; a shared bitmap
//           [token-word][rank] records membership, a shared histogram counts
//           experts, and each entry's owned rank (or -1) is kept in shared
//           memory for pass 2.
//   scan    per rank, popcounts give the tile aggregate, published for all
//           ranks first; then a decoupled lookback (Merrill & Garland,
//           "Single-pass Parallel Prefix Scan with Decoupled Look-back", 2016)
//           over R-wide vectors gives the tile's exclusive prefix. A group of
//           G lanes serves one rank and reads G predecessor tiles per step.
//           Each (tile, rank) status is one 64-bit word {flag:32 | value:32},
//           written in one store, so value and flag change together. Waits
//           are bounded (MOE_ERR_TIMEOUT).
//   pass 2  the owning entries get their receive rows.
//   last    the last CTA to finish (done counter) writes the per-expert counts
//           and their exclusive prefix.
// When every tile fits on the GPU at once, the kernel is launched
// cooperatively (all CTAs co-resident, tile = blockIdx): the last tile's
// inclusive prefix is the vector of rank totals, so every tile waits
// (bounded) for it, scans it in shared memory into rank_prefix and writes
// final global rows -- one launch. Otherwise tiles are claimed by an atomic
// ticket (so every predecessor of a tile is already resident), pass 2 writes
// in-rank positions, the last CTA also writes the rank counts and prefix, and
// a second small kernel adds rank_prefix[r].
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

// Direct mode (few tiles, all co-resident): every tile publishes its rank
// counts as flagged words and reads all tiles' words itself. A batch of at
// most kTile tokens is one tile of kTile (nothing to exchange); larger ones
// use tiles of kDirectTile tokens, which halves each CTA's serial work for
// the price of more (cheap) exchange words.
constexpr int kDirectTile = 64;
constexpr int kDirectMaxTiles = 128;
constexpr int64_t kDirectMaxRankWords = 16384;     // tiles * R

// Tokens per tile of the direct mode for this batch, or 0 when the batch
// takes a lookback mode.
inline int direct_tile(int T, int R) {
    if (T <= 0) return 0;
    if (T <= kTile) return kTile;
    const int64_t tiles = (T + kDirectTile - 1) / kDirectTile;
    return tiles <= kDirectMaxTiles && tiles * R <= kDirectMaxRankWords ? kDirectTile : 0;
}

struct WsLayout {
    size_t expert_off, status_off, total;
};

inline WsLayout ws_layout(int T, int E, int R) {
    WsLayout w;
    const int dt = direct_tile(T, R);
    size_t tiles = (size_t)((T + (dt ? dt : kTile) - 1) / (dt ? dt : kTile));
    w.expert_off = sizeof(WsHeader);
    w.status_off = align_up(w.expert_off + (size_t)E * 4, 128);
    w.total = align_up(w.status_off + tiles * (size_t)R * 8, 128);
    return w;
}

// Shared memory: bitmap u32 [kWords][R] | word prefix u16 [R][kWords] |
// exclusive prefix i32 [R] | tile aggregate i32 [R] | rank totals i32 [R] |
// expert histogram i32 [E] | owned rank i16 [kTile * k]
struct SmemLayout {
    size_t wprefix, excl, agg, tot, hist, own, total;
};

__host__ __device__ inline SmemLayout smem_layout(int E, int R, int k) {
    SmemLayout s;
    s.wprefix = align_up((size_t)R * kWords * 4, 16);
    s.excl = s.wprefix + align_up((size_t)R * kWords * 2, 16);
    s.agg = s.excl + align_up((size_t)R * 4, 16);
    s.tot = s.agg + align_up((size_t)R * 4, 16);
    s.hist = s.tot + align_up((size_t)R * 4, 16);
    s.own = s.hist + align_up((size_t)E * 4, 16);
    s.total = s.own + align_up((size_t)kTile * k * 2, 16);
    return s;
}

// In-place exclusive scan of n int32 values in shared memory; returns the total.
__device__ int32_t smem_exclusive_scan(int32_t *v, int n) {
    __shared__ int32_t warp_sums[kWarps];
    __shared__ int32_t total;
    const int per = (n + kThreads - 1) / kThreads;
    const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
    int32_t local = 0;
    for (int i = lo; i < hi; ++i) local += v[i];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int32_t t = warp_sums[w];
            warp_sums[w] = run;
            run += t;
        }
        total = run;
    }
    __syncthreads();
    int32_t run = warp_sums[warp] + incl - local;
    for (int i = lo; i < hi; ++i) {
        const int32_t x = v[i];
        v[i] = run;
        run += x;
    }
    __syncthreads();
    return total;
}

// Exclusive scan of n int32 counts (read from `in`, copied to `copy_out` when
// non-null) into prefix[0..n]; one CTA of kThreads threads.
__device__ void block_exclusive_scan(const int32_t *in, int n, int32_t *copy_out, int32_t *prefix) {
    __shared__ int32_t warp_sums[kWarps];
    __shared__ int32_t carry_total;
    const int per = (n + kThreads - 1) / kThreads;
    const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
    int32_t local = 0;
    for (int i = lo; i < hi; ++i) local += __ldcg(in + i);
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
        const int32_t v = __ldcg(in + i);
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
    int group;             // lanes per rank in the lookback (power of two, <= 32)
    uint8_t *is_token_in_rank;
    int32_t *token_dst_row;
    int32_t *num_tokens_per_rank, *num_tokens_per_expert, *rank_prefix, *expert_prefix;
    uint8_t *ws;
    size_t expert_off, status_off;
    int32_t *status;
    uint64_t timeout_ns;
    int unpublished_tile;  // test hook: this tile never publishes its status (-1 = none)
    int early_dependents;  // trigger the next grid's launch right after the dependency wait
    int cl_tile;           // cluster mode: tokens per CTA (a multiple of 32)
    unsigned int *spare;   // cluster mode: two workspace words to zero for the next launch (the others clear them)
    TraceArgs trace;       // MOE_PROFILE builds: where the warps' records go
};

template <bool kCooperative>
__global__ void __launch_bounds__(kThreads) layout_tiles_kernel(TileArgs a) {
    WarpTrace wt(a.trace, MOE_TRACE_LAYOUT_TILES);
    extern __shared__ __align__(16) uint8_t smem[];
    const int R = a.R, E = a.E, k = a.k;
    const SmemLayout sl = smem_layout(E, R, k);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem);
    uint16_t *wprefix = reinterpret_cast<uint16_t *>(smem + sl.wprefix);
    int32_t *excl = reinterpret_cast<int32_t *>(smem + sl.excl);
    int32_t *aggs = reinterpret_cast<int32_t *>(smem + sl.agg);
    int32_t *tot = reinterpret_cast<int32_t *>(smem + sl.tot);
    int32_t *hist = reinterpret_cast<int32_t *>(smem + sl.hist);
    int16_t *own = reinterpret_cast<int16_t *>(smem + sl.own);
    __shared__ int s_tile;
    __shared__ int s_last;

    WsHeader *hdr = reinterpret_cast<WsHeader *>(a.ws);
    int32_t *ws_expert = reinterpret_cast<int32_t *>(a.ws + a.expert_off);
    uint64_t *tile_status = reinterpret_cast<uint64_t *>(a.ws + a.status_off);
    grid_dependency_wait();
    if (a.early_dependents) grid_launch_dependents();

    if (threadIdx.x == 0) s_tile = kCooperative ? (int)blockIdx.x : (int)atomicAdd(&hdr->ticket, 1u);
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

    // ---- pass 1: membership bitmap, expert histogram, owned ranks
    for (int base = warp * tpp; base < tcount; base += kWarps * tpp) {
        const int tl = base + sub;
        const bool act = lane_used && tl < tcount;
        int r = -1;
        if (act) {
            const int64_t e = ld_nc_i64(a.topk + (int64_t)(t0 + tl) * k + j);
            if (e >= 0 && e < E) {
                r = (int)e / a.m;
                atomicAdd(&hist[(int)e], 1);
            } else if (e != -1) {
                report(a.status, MOE_ERR_BAD_TOPK);
            }
        }
        const int key = (r >= 0) ? (sub * R + r) : -(lane + 1);
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const bool owner = r >= 0 && (__ffs(peers) - 1) == lane;
        if (owner) atomicOr(&bitmap[(tl >> 5) * R + r], 1u << (tl & 31));
        if (act) own[tl * k + j] = (int16_t)(owner ? r : -1);
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
            run += __popc(bitmap[w * R + r]);
        }
        excl[r] = (int32_t)run;   // holds the aggregate until the lookback below
        aggs[r] = (int32_t)run;
        if (publish) st_relaxed_gpu_u64(my_status + r, (tile == 0 ? kFlagInclusive : kFlagAggregate) | run);
    }
    __syncthreads();

    // ---- decoupled lookback, G lanes per rank, G predecessors per step
    {
        const int G = a.group;
        const int ngroups = kThreads / G;
        const int gi = threadIdx.x / G, gl = threadIdx.x % G;
        const int gbase = lane & ~(G - 1);
        const unsigned low = (G == 32) ? 0xffffffffu : ((1u << G) - 1u);
        const unsigned gmask = low << gbase;
        for (int r = gi; r < R; r += ngroups) {
            const uint32_t agg = (uint32_t)excl[r];
            uint32_t ex = 0;
            if (tile > 0) {
                int p_hi = tile - 1;
                uint64_t deadline = 0;
                while (true) {
                    const int p = p_hi - gl;
                    const uint64_t w = (p >= 0) ? ld_relaxed_gpu_u64(tile_status + (size_t)p * R + r) : kFlagInclusive;
                    const uint64_t flag = w & 0xffffffff00000000ull;
                    const unsigned pm = (__ballot_sync(gmask, flag == kFlagInclusive) >> gbase) & low;
                    const unsigned zm = (__ballot_sync(gmask, flag == 0) >> gbase) & low;
                    const int fp = pm ? __ffs(pm) - 1 : G;                 // nearest inclusive in the window
                    const unsigned need = (fp >= 31) ? low : ((2u << fp) - 1u) & low;
                    if (zm & need) {                                      // a needed predecessor is not ready
                        const uint64_t now = globaltimer_ns();
                        if (deadline == 0) {
                            deadline = now + a.timeout_ns;
                        } else if (now > deadline) {
                            if (gl == 0) report(a.status, MOE_ERR_TIMEOUT);
                            break;
                        }
                        continue;
                    }
                    uint32_t v = (gl <= fp) ? (uint32_t)w : 0u;
                    for (int o = G >> 1; o >= 1; o >>= 1) v += __shfl_xor_sync(gmask, v, o);
                    ex += v;
                    if (fp < G) break;
                    p_hi -= G;
                }
                if (publish && gl == 0) st_relaxed_gpu_u64(my_status + r, kFlagInclusive | (ex + agg));
            }
            if (gl == 0) excl[r] = (int32_t)ex;
        }
    }
    __syncthreads();

    // ---- expert histogram into the global accumulator
    for (int e = threadIdx.x; e < E; e += kThreads) {
        const int h = hist[e];
        if (h) atomicAdd(ws_expert + e, h);
    }

    // ---- the last CTA to finish its histogram writes the expert counts and prefix
    //      (and, when not cooperative, the rank counts and prefix); the other
    //      tiles go on meanwhile
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(&hdr->done, 1u) == (unsigned)(a.num_tiles - 1));
    __syncthreads();
    if (s_last) {
        __threadfence();
        if (!kCooperative) {
            const uint64_t *last_status = tile_status + (size_t)(a.num_tiles - 1) * R;
            for (int r = threadIdx.x; r < R; r += kThreads) {
                const uint64_t w = ld_relaxed_gpu_u64(last_status + r);
                if ((w & 0xffffffff00000000ull) != kFlagInclusive) report(a.status, MOE_ERR_TIMEOUT);
                a.num_tokens_per_rank[r] = (int32_t)(uint32_t)w;
            }
            __threadfence();
            __syncthreads();
            block_exclusive_scan(a.num_tokens_per_rank, R, nullptr, a.rank_prefix);
        } else if (a.unpublished_tile == a.num_tiles - 1) {
            report(a.status, MOE_ERR_TIMEOUT);   // test hook: the last tile never published its totals
        }
        block_exclusive_scan(ws_expert, E, a.num_tokens_per_expert, a.expert_prefix);
    }

    if (kCooperative) {
        // ---- rank totals = inclusive prefix of the last tile (read as it is published)
        const uint64_t *last_status = tile_status + (size_t)(a.num_tiles - 1) * R;
        for (int r = threadIdx.x; r < R; r += kThreads) {
            int32_t v = excl[r] + aggs[r];
            if (tile != a.num_tiles - 1) {
                uint64_t w = ld_relaxed_gpu_u64(last_status + r), deadline = 0;
                while ((w & 0xffffffff00000000ull) != kFlagInclusive) {
                    const uint64_t now = globaltimer_ns();
                    if (deadline == 0) {
                        deadline = now + a.timeout_ns;
                    } else if (now > deadline) {
                        report(a.status, MOE_ERR_TIMEOUT);
                        break;
                    }
                    w = ld_relaxed_gpu_u64(last_status + r);
                }
                v = (int32_t)(uint32_t)w;
            }
            tot[r] = v;
        }
        __syncthreads();
        if (tile == a.num_tiles - 1)
            for (int r = threadIdx.x; r < R; r += kThreads) a.num_tokens_per_rank[r] = tot[r];
        const int32_t n_recv = smem_exclusive_scan(tot, R);   // tot -> rank_prefix
        for (int r = threadIdx.x; r < R; r += kThreads) {
            excl[r] += tot[r];
            if (tile == a.num_tiles - 1) a.rank_prefix[r] = tot[r];
        }
        if (tile == a.num_tiles - 1 && threadIdx.x == 0) a.rank_prefix[R] = n_recv;
        __syncthreads();
    }

    // ---- pass 2: receive rows of the owning entries (global rows when cooperative,
    //      in-rank positions otherwise)
    for (int i = threadIdx.x; i < tcount * k; i += kThreads) {
        const int r = own[i];
        int32_t v = -1;
        if (r >= 0) {
            const int tl = i / k;
            const uint32_t word = bitmap[(tl >> 5) * R + r];
            v = excl[r] + wprefix[r * kWords + (tl >> 5)] + __popc(word & ((1u << (tl & 31)) - 1u));
        }
        a.token_dst_row[(int64_t)t0 * k + i] = v;
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
                v |= ((bitmap[(tl >> 5) * R + r0 + b] >> (tl & 31)) & 1u) << (8 * b);
            dst4[i] = v;
        }
    } else {
        for (int i = threadIdx.x; i < nbytes; i += kThreads) {
            const int tl = i / R, r = i - tl * R;
            dst[i] = (uint8_t)((bitmap[(tl >> 5) * R + r] >> (tl & 31)) & 1u);
        }
    }

}

// Waits (bounded) for the flagged words words[p], p in [0, n) strided over the
// CTA, 8 loads in flight per thread, and hands each value to consume(p, v).
template <typename F>
__device__ void gather_flagged(const uint64_t *words, int n, uint64_t timeout_ns, int32_t *status, F consume) {
    for (int p0 = threadIdx.x; p0 < n; p0 += 8 * kThreads) {
        uint64_t w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int p = p0 + u * kThreads;
            w[u] = p < n ? ld_relaxed_gpu_u64(words + p) : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int p = p0 + u * kThreads;
            if (p >= n) continue;
            uint64_t x = w[u], deadline = 0;
            while ((x & 0xffffffff00000000ull) == 0) {
                const uint64_t now = globaltimer_ns();
                if (deadline == 0) {
                    deadline = now + timeout_ns;
                } else if (now > deadline) {
                    report(status, MOE_ERR_TIMEOUT);
                    break;
                }
                x = ld_relaxed_gpu_u64(words + p);
            }
            consume(p, (int32_t)(uint32_t)x);
        }
    }
}

// Shared memory of the direct kernel: bitmap u32 [kWords][R] | word prefix
// u16 [R][kWords] | exclusive prefix i32 [R] | rank totals i32 [R+1] |
// expert histogram i32 [E+1] | entry expert i16 [kTile*k] | entry rank i16 [kTile*k]
struct DirectSmem {
    size_t wprefix, excl, tot, hist, ent, rk, total;
};

template <int TILE>
__host__ __device__ inline DirectSmem direct_smem(int E, int R, int k) {
    constexpr int kWords = TILE / 32;
    DirectSmem d;
    d.wprefix = align_up((size_t)R * kWords * 4, 16);
    d.excl = d.wprefix + align_up((size_t)R * kWords * 2, 16);
    d.tot = d.excl + align_up((size_t)R * 4, 16);
    d.hist = d.tot + align_up((size_t)(R + 1) * 4, 16);
    d.ent = d.hist + align_up((size_t)(E + 1) * 4, 16);
    d.rk = d.ent + align_up((size_t)TILE * k * 2, 16);
    d.total = d.rk + align_up((size_t)TILE * k * 2, 16);
    return d;
}

// Direct mode, launched cooperatively with one CTA per tile (few tiles): each
// tile adds its expert histogram into the global accumulator, then publishes
// its per-rank counts, then reads every tile's rank words -- the sum over
// lower tiles is its exclusive prefix, the sum over all tiles the rank totals
// -- so no tile waits on a chain of predecessors. A tile's rank words are
// published after a fence that follows its histogram atomics, so once tile 0
// has seen every tile's words the expert totals are complete; it then writes
// the expert counts and prefix. A batch of one tile exchanges nothing.
template <int TILE>
__global__ void __launch_bounds__(kThreads) layout_direct_kernel(TileArgs a) {
    WarpTrace wt(a.trace, MOE_TRACE_LAYOUT_DIRECT);
    constexpr int kTile = TILE;            // tokens per tile of this instance
    constexpr int kWords = TILE / 32;
    extern __shared__ __align__(16) uint8_t smem[];
    const int R = a.R, E = a.E, k = a.k;
    const DirectSmem sl = direct_smem<TILE>(E, R, k);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem);
    uint16_t *wprefix = reinterpret_cast<uint16_t *>(smem + sl.wprefix);
    int32_t *excl = reinterpret_cast<int32_t *>(smem + sl.excl);
    int32_t *tot = reinterpret_cast<int32_t *>(smem + sl.tot);
    int32_t *hist = reinterpret_cast<int32_t *>(smem + sl.hist);
    int16_t *ent = reinterpret_cast<int16_t *>(smem + sl.ent);   // expert of each entry, then its owned rank
    int16_t *rk = reinterpret_cast<int16_t *>(smem + sl.rk);     // rank of each entry
    uint64_t *rank_words = reinterpret_cast<uint64_t *>(a.ws + a.status_off);
    int32_t *ws_expert = reinterpret_cast<int32_t *>(a.ws + a.expert_off);

    const int tile = blockIdx.x;
    const bool multi = a.num_tiles > 1;
    const int t0 = tile * kTile;
    const int tcount = min(kTile, a.T - t0);
    const int n_ent = tcount * k;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool publish = tile != a.unpublished_tile;
    grid_dependency_wait();
    if (a.early_dependents) grid_launch_dependents();

    for (int i = threadIdx.x; i < R * kWords; i += kThreads) bitmap[i] = 0u;
    for (int i = threadIdx.x; i < E; i += kThreads) hist[i] = 0;
    for (int r = threadIdx.x; r < R; r += kThreads) excl[r] = 0;
    // the tile's entries: expert and rank ids (-1: masked or invalid), 8 loads in flight per thread
    for (int base = threadIdx.x; base < n_ent; base += 8 * kThreads) {
        int64_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * kThreads;
            v[u] = i < n_ent ? ld_nc_i64(a.topk + (int64_t)t0 * k + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * kThreads;
            if (i < n_ent) {
                const bool ok = v[u] >= 0 && v[u] < E;
                if (!ok && v[u] != -1) report(a.status, MOE_ERR_BAD_TOPK);
                ent[i] = ok ? (int16_t)v[u] : (int16_t)-1;
                rk[i] = ok ? (int16_t)((int)v[u] / a.m) : (int16_t)-1;
            }
        }
    }
    __syncthreads();

    // ---- pass 1, lanes over (token, entry): expert histogram, each rank of a token
    //      once (__match_any_sync; the lowest entry owns it), membership bits;
    //      ent[] becomes the owned rank (or -1)
    {
        const int tpp = 32 / k;
        const int sub = lane / k, j = lane - sub * k;
        const bool lane_used = sub < tpp;
        for (int base = warp * tpp; base < tcount; base += kWarps * tpp) {
            const int tl = base + sub;
            const bool act = lane_used && tl < tcount;
            const int r = act ? (int)rk[tl * k + j] : -1;
            if (r >= 0) atomicAdd(&hist[ent[tl * k + j]], 1);
            const unsigned peers = __match_any_sync(0xffffffffu, r >= 0 ? sub * R + r : -(lane + 1));
            const bool owner = r >= 0 && (__ffs(peers) - 1) == lane;
            if (owner) atomicOr(&bitmap[(tl >> 5) * R + r], 1u << (tl & 31));
            if (act) ent[tl * k + j] = (int16_t)(owner ? r : -1);
        }
    }
    __syncthreads();

    // ---- this tile's rank counts (and, with several tiles, the exchange)
    if (multi) {
        for (int e = threadIdx.x; e < E; e += kThreads) {
            const int h = hist[e];
            if (h) atomicAdd(ws_expert + e, h);
        }
        __threadfence();
    }
    for (int r = threadIdx.x; r < R; r += kThreads) {
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < kWords; ++w) {
            wprefix[r * kWords + w] = (uint16_t)run;
            run += __popc(bitmap[w * R + r]);
        }
        tot[r] = multi ? 0 : (int32_t)run;
        if (multi && publish) st_relaxed_gpu_u64(rank_words + (size_t)tile * R + r, kFlagAggregate | run);
    }
    __syncthreads();
    if (multi) {
        gather_flagged(rank_words, a.num_tiles * R, a.timeout_ns, a.status, [&](int p, int32_t v) {
            const int b = p / R, r = p - b * R;
            if (b < tile) atomicAdd(&excl[r], v);
            atomicAdd(&tot[r], v);
        });
        __syncthreads();
        if (tile == 0) {
            __threadfence();
            for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = __ldcg(ws_expert + e);
        }
        __syncthreads();
    }

    // ---- rank regions (warp 0); on tile 0 the expert counts and prefix, by the
    //      whole CTA (one warp walking 2048 experts took ~10 us)
    if (warp == 0) {
        if (tile == 0)
            for (int r = lane; r < R; r += 32) a.num_tokens_per_rank[r] = tot[r];
        __syncwarp();
        warp_exclusive_scan(tot, R, lane);
    }
    if (tile == 0) {
        for (int e = threadIdx.x; e < E; e += kThreads) a.num_tokens_per_expert[e] = hist[e];
        const int32_t n_entries = smem_exclusive_scan(hist, E);
        for (int e = threadIdx.x; e < E; e += kThreads) a.expert_prefix[e] = hist[e];
        if (threadIdx.x == 0) a.expert_prefix[E] = n_entries;
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += kThreads) {
        excl[r] += tot[r];
        if (tile == 0) a.rank_prefix[r] = tot[r];
    }
    if (tile == 0 && threadIdx.x == 0) a.rank_prefix[R] = tot[R];
    __syncthreads();

    // ---- pass 2: global receive rows of the owning entries
    for (int i = threadIdx.x; i < n_ent; i += kThreads) {
        const int r = ent[i];
        int32_t v = -1;
        if (r >= 0) {
            const int tl = i / k;
            const uint32_t word = bitmap[(tl >> 5) * R + r];
            v = excl[r] + wprefix[r * kWords + (tl >> 5)] + __popc(word & ((1u << (tl & 31)) - 1u));
        }
        a.token_dst_row[(int64_t)t0 * k + i] = v;
    }

    // ---- is_token_in_rank rows: one warp per token row when rows are long, flat otherwise
    uint8_t *dst = a.is_token_in_rank + (int64_t)t0 * R;
    if ((R & 3) == 0 && R >= 128) {
        for (int tl = warp; tl < tcount; tl += kWarps) {
            const uint32_t *wrow = bitmap + (tl >> 5) * R;
            const int b = tl & 31;
            for (int r0 = 4 * lane; r0 < R; r0 += 128) {
                const uint4 q = *reinterpret_cast<const uint4 *>(wrow + r0);
                const uint32_t v = ((q.x >> b) & 1u) | (((q.y >> b) & 1u) << 8) | (((q.z >> b) & 1u) << 16) |
                                   (((q.w >> b) & 1u) << 24);
                *reinterpret_cast<uint32_t *>(dst + (int64_t)tl * R + r0) = v;
            }
        }
    } else if ((R & 3) == 0) {
        uint32_t *dst4 = reinterpret_cast<uint32_t *>(dst);
        for (int i = threadIdx.x; i < tcount * R / 4; i += kThreads) {
            const int tl = (i * 4) / R, r0 = (i * 4) - tl * R;
            uint32_t v = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) v |= ((bitmap[(tl >> 5) * R + r0 + b] >> (tl & 31)) & 1u) << (8 * b);
            dst4[i] = v;
        }
    } else {
        for (int i = threadIdx.x; i < tcount * R; i += kThreads) {
            const int tl = i / R, r = i - tl * R;
            dst[i] = (uint8_t)((bitmap[(tl >> 5) * R + r] >> (tl & 31)) & 1u);
        }
    }
}


// ------------------------------------------------------------------ cluster mode
//
// One thread-block cluster of C CTAs (1024 threads each) covers the whole
// batch, each CTA a contiguous tile of cl_tile tokens. The tiles exchange their
// per-rank counts and expert histograms through distributed shared memory
// between two cluster barriers, so there is no global exchange state: no
// workspace clear, no flags, no waits that could expire. Everything else is
// the direct mode's: pass 1 over (token, entry) lanes, word prefixes of the
// membership bitmap, receive rows from the ranks' exclusive prefixes.

constexpr int kCThreads = 1024;
constexpr int kCWarps = kCThreads / 32;
constexpr int kClusterMaxTile = 512;     // tokens per CTA
constexpr int kClusterMax = 16;          // CTAs per cluster

// Shared memory: bitmap u32 [W][R] | word prefix u16 [R][W] | exclusive prefix
// i32 [R] | rank totals i32 [R+1] | own rank counts i32 [R] | expert
// histogram i32 [E+1] | expert totals i32 [E+1] | entry expert i16 [tile*k] |
// entry rank i16 [tile*k]
struct ClusterSmem {
    size_t wprefix, excl, tot, cnt, hist, htot, ent, rk, total;
};

__host__ __device__ inline ClusterSmem cluster_smem(int tile, int E, int R, int k) {
    const size_t W = (size_t)tile / 32;
    ClusterSmem c;
    c.wprefix = align_up(W * R * 4, 16);
    c.excl = c.wprefix + align_up(W * R * 2, 16);
    c.tot = c.excl + align_up((size_t)R * 4, 16);
    c.cnt = c.tot + align_up((size_t)(R + 1) * 4, 16);
    c.hist = c.cnt + align_up((size_t)R * 4, 16);
    c.htot = c.hist + align_up((size_t)(E + 1) * 4, 16);
    c.ent = c.htot + align_up((size_t)(E + 1) * 4, 16);
    c.rk = c.ent + align_up((size_t)tile * k * 2, 16);
    c.total = c.rk + align_up((size_t)tile * k * 2, 16);
    return c;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 32-bit load from the shared memory of CTA `rank` of this cluster, at the
// offset of `local` in this CTA's shared memory
__device__ __forceinline__ int32_t ld_cluster_i32(const void *local, uint32_t rank) {
    uint32_t remote;
    int32_t v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

__global__ void __launch_bounds__(kCThreads) layout_cluster_kernel(TileArgs a) {
    WarpTrace wt(a.trace, MOE_TRACE_LAYOUT_CLUSTER);
    MOE_PHASES(MOE_TRACE_LAYOUT_CLUSTER, 8);
    extern __shared__ __align__(16) uint8_t smem[];
    const int R = a.R, E = a.E, k = a.k, tile = a.cl_tile, W = tile / 32;
    const ClusterSmem sl = cluster_smem(tile, E, R, k);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem);
    uint16_t *wprefix = reinterpret_cast<uint16_t *>(smem + sl.wprefix);
    int32_t *excl = reinterpret_cast<int32_t *>(smem + sl.excl);
    int32_t *tot = reinterpret_cast<int32_t *>(smem + sl.tot);
    int32_t *cnt = reinterpret_cast<int32_t *>(smem + sl.cnt);
    int32_t *hist = reinterpret_cast<int32_t *>(smem + sl.hist);
    int32_t *htot = reinterpret_cast<int32_t *>(smem + sl.htot);
    int16_t *ent = reinterpret_cast<int16_t *>(smem + sl.ent);   // expert of each entry, then its owned rank
    int16_t *rk = reinterpret_cast<int16_t *>(smem + sl.rk);     // rank of each entry

    const int C = (int)gridDim.x;              // one cluster spans the grid
    const int c = (int)cluster_ctarank();
    const int t0 = c * tile;
    const int tcount = max(0, min(tile, a.T - t0));
    const int n_ent = tcount * k;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    grid_dependency_wait();
    MOE_PHASE(1);
    if (a.early_dependents) grid_launch_dependents();
    if (c == 0 && threadIdx.x == 0 && a.spare != nullptr) {   // the workspace is not cleared in this mode
        a.spare[0] = 0u;
        a.spare[1] = 0u;
    }

    for (int i = threadIdx.x; i < R * W; i += kCThreads) bitmap[i] = 0u;
    for (int i = threadIdx.x; i <= E; i += kCThreads) hist[i] = 0;
    for (int r = threadIdx.x; r <= R; r += kCThreads) tot[r] = 0;
    for (int r = threadIdx.x; r < R; r += kCThreads) excl[r] = 0;
    // the tile's entries: expert and rank ids (-1: masked or invalid), 8 loads in flight per thread
    for (int base = threadIdx.x; base < n_ent; base += 8 * kCThreads) {
        int64_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * kCThreads;
            v[u] = i < n_ent ? ld_nc_i64(a.topk + (int64_t)t0 * k + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * kCThreads;
            if (i < n_ent) {
                const bool ok = v[u] >= 0 && v[u] < E;
                if (!ok && v[u] != -1) report(a.status, MOE_ERR_BAD_TOPK);
                ent[i] = ok ? (int16_t)v[u] : (int16_t)-1;
                rk[i] = ok ? (int16_t)((int)v[u] / a.m) : (int16_t)-1;
            }
        }
    }
    __syncthreads();
    MOE_PHASE(2);

    // ---- pass 1: expert histogram, each rank of a token once (the lowest entry
    //      owns it), membership bits; ent[] becomes the owned rank (or -1)
    if (R <= 32) {
        // a lane per token: its ranks as a 32-bit mask, then one ballot per rank
        // gives a whole bitmap word (32 tokens) without shared-memory atomics
        const int tpad = (tcount + 31) & ~31;
        for (int tl = threadIdx.x; tl < tpad; tl += kCThreads) {
            uint32_t mask = 0u;
            if (tl < tcount) {
                for (int j = 0; j < k; ++j) {
                    const int r = rk[tl * k + j];
                    int own = -1;
                    if (r >= 0) {
                        atomicAdd(&hist[ent[tl * k + j]], 1);
                        if (!((mask >> r) & 1u)) {
                            mask |= 1u << r;
                            own = r;
                        }
                    }
                    ent[tl * k + j] = (int16_t)own;
                }
            }
            for (int r = 0; r < R; ++r) {
                const unsigned word = __ballot_sync(0xffffffffu, (mask >> r) & 1u);
                if (lane == 0) bitmap[(tl >> 5) * R + r] = word;
            }
        }
    } else {
        const int tpp = 32 / k;
        const int sub = lane / k, j = lane - sub * k;
        const bool lane_used = sub < tpp;
        for (int base = warp * tpp; base < tcount; base += kCWarps * tpp) {
            const int tl = base + sub;
            const bool act = lane_used && tl < tcount;
            const int r = act ? (int)rk[tl * k + j] : -1;
            if (r >= 0) atomicAdd(&hist[ent[tl * k + j]], 1);
            const unsigned peers = __match_any_sync(0xffffffffu, r >= 0 ? sub * R + r : -(lane + 1));
            const bool owner = r >= 0 && (__ffs(peers) - 1) == lane;
            if (owner) atomicOr(&bitmap[(tl >> 5) * R + r], 1u << (tl & 31));
            if (act) ent[tl * k + j] = (int16_t)(owner ? r : -1);
        }
    }
    __syncthreads();
    MOE_PHASE(3);

    // ---- this tile's rank counts and word prefixes
    for (int r = threadIdx.x; r < R; r += kCThreads) {
        uint32_t run = 0;
        for (int w = 0; w < W; ++w) {
            wprefix[r * W + w] = (uint16_t)run;
            run += __popc(bitmap[w * R + r]);
        }
        cnt[r] = (int32_t)run;
    }

    // ---- exchange through distributed shared memory: every tile's counts are
    //      complete after the first barrier and read before the second
    cluster_sync_all();
    MOE_PHASE(4);
    for (int idx = threadIdx.x; idx < C * R; idx += kCThreads) {
        const int cc = idx / R, r = idx - cc * R;
        const int32_t v = ld_cluster_i32(cnt + r, (uint32_t)cc);
        if (cc < c) atomicAdd(&excl[r], v);
        atomicAdd(&tot[r], v);
    }
    if (c == 0) {   // expert totals: all C tiles' counts of an expert in flight at once
        for (int e = threadIdx.x; e < E; e += kCThreads) {
            int32_t v[kClusterMax];
#pragma unroll
            for (int cc = 0; cc < kClusterMax; ++cc) v[cc] = cc < C ? ld_cluster_i32(hist + e, (uint32_t)cc) : 0;
            int32_t s = 0;
#pragma unroll
            for (int cc = 0; cc < kClusterMax; ++cc) s += v[cc];
            htot[e] = s;
        }
    }
    cluster_sync_all();   // no tile reads another's shared memory after this
    MOE_PHASE(5);

    // ---- rank regions (warp 0) and, on tile 0, expert counts and prefix (warp 1)
    if (warp == 0) {
        if (c == 0)
            for (int r = lane; r < R; r += 32) a.num_tokens_per_rank[r] = tot[r];
        __syncwarp();
        warp_exclusive_scan(tot, R, lane);
    } else if (warp == 1 && c == 0) {
        for (int e = lane; e < E; e += 32) a.num_tokens_per_expert[e] = htot[e];
        __syncwarp();
        warp_exclusive_scan(htot, E, lane);
        __syncwarp();
        for (int e = lane; e <= E; e += 32) a.expert_prefix[e] = htot[e];
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += kCThreads) {
        excl[r] += tot[r];
        if (c == 0) a.rank_prefix[r] = tot[r];
    }
    if (c == 0 && threadIdx.x == 0) a.rank_prefix[R] = tot[R];
    __syncthreads();

    MOE_PHASE(6);
    // ---- pass 2: global receive rows of the owning entries
    for (int i = threadIdx.x; i < n_ent; i += kCThreads) {
        const int r = ent[i];
        int32_t v = -1;
        if (r >= 0) {
            const int tl = i / k;
            const uint32_t word = bitmap[(tl >> 5) * R + r];
            v = excl[r] + wprefix[r * W + (tl >> 5)] + __popc(word & ((1u << (tl & 31)) - 1u));
        }
        a.token_dst_row[(int64_t)t0 * k + i] = v;
    }

    MOE_PHASE(7);
    // ---- is_token_in_rank rows: one warp per token row when rows are long, flat otherwise
    uint8_t *dst = a.is_token_in_rank + (int64_t)t0 * R;
    if ((R & 3) == 0 && R >= 128) {
        for (int tl = warp; tl < tcount; tl += kCWarps) {
            const uint32_t *wrow = bitmap + (tl >> 5) * R;
            const int b = tl & 31;
            for (int r0 = 4 * lane; r0 < R; r0 += 128) {
                const uint4 q = *reinterpret_cast<const uint4 *>(wrow + r0);
                const uint32_t v = ((q.x >> b) & 1u) | (((q.y >> b) & 1u) << 8) | (((q.z >> b) & 1u) << 16) |
                                   (((q.w >> b) & 1u) << 24);
                *reinterpret_cast<uint32_t *>(dst + (int64_t)tl * R + r0) = v;
            }
        }
    } else if ((R & 3) == 0) {
        uint32_t *dst4 = reinterpret_cast<uint32_t *>(dst);
        for (int i = threadIdx.x; i < tcount * R / 4; i += kCThreads) {
            const int tl = (i * 4) / R, r0 = (i * 4) - tl * R;
            uint32_t v = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) v |= ((bitmap[(tl >> 5) * R + r0 + b] >> (tl & 31)) & 1u) << (8 * b);
            dst4[i] = v;
        }
    } else {
        for (int i = threadIdx.x; i < tcount * R; i += kCThreads) {
            const int tl = i / R, r = i - tl * R;
            dst[i] = (uint8_t)((bitmap[(tl >> 5) * R + r] >> (tl & 31)) & 1u);
        }
    }
}

__global__ void layout_rows_kernel(const int64_t *__restrict__ topk, int64_t n, int m,
                                   const int32_t *__restrict__ rank_prefix, int32_t *__restrict__ token_dst_row,
                                   TraceArgs trace) {
    WarpTrace wt(trace, MOE_TRACE_LAYOUT_ROWS);
    grid_dependency_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = token_dst_row[i];
        if (v >= 0) token_dst_row[i] = v + rank_prefix[(int)topk[i] / m];
    }
}

// ------------------------------------------------------------------ scan mode (large batches)
//
// For more tiles than fit on the GPU at once, the decoupled lookback becomes a
// chain through every tile in turn (2^20 tokens over 256 ranks: 8192 tiles,
// 1.6 ms). The scan mode has no waits at all: three launches, each fully
// parallel.
//   count: one CTA per tile of kTile tokens -- the tile's membership rows, each
//          owning entry's position inside the tile's share of its rank, the
//          tile's per-rank counts into the workspace (rank-major, [R][tiles+1]),
//          its expert histogram added into the global accumulator;
//   scan:  one CTA per rank -- the exclusive scan of that rank's tile counts
//          (its total lands in slot [tiles]); the last CTA to finish (a done
//          counter) writes the rank counts and prefix and the expert counts
//          and prefix;
//   rows:  every owning entry's position plus its rank's region start plus
//          its tile's prefix.

__global__ void __launch_bounds__(kThreads) layout_count_kernel(TileArgs a) {
    WarpTrace wt(a.trace, MOE_TRACE_LAYOUT_COUNT);
    extern __shared__ __align__(16) uint8_t smem[];
    const int R = a.R, E = a.E, k = a.k;
    const SmemLayout sl = smem_layout(E, R, k);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem);
    uint16_t *wprefix = reinterpret_cast<uint16_t *>(smem + sl.wprefix);
    int32_t *hist = reinterpret_cast<int32_t *>(smem + sl.hist);
    int16_t *own = reinterpret_cast<int16_t *>(smem + sl.own);
    int32_t *ws_expert = reinterpret_cast<int32_t *>(a.ws + a.expert_off);
    int32_t *counts = reinterpret_cast<int32_t *>(a.ws + a.status_off);   // [R][num_tiles + 1]
    grid_dependency_wait();
    for (int i = threadIdx.x; i < R * kWords; i += kThreads) bitmap[i] = 0u;
    for (int i = threadIdx.x; i < E; i += kThreads) hist[i] = 0;
    __syncthreads();
    const int tile = (int)blockIdx.x;
    const int t0 = tile * kTile;
    const int tcount = min(kTile, a.T - t0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tpp = 32 / k;
    const int sub = lane / k, j = lane - sub * k;
    const bool lane_used = sub < tpp;
    // ---- membership bitmap, expert histogram, owned ranks (the lowest entry of a rank owns it)
    for (int base = warp * tpp; base < tcount; base += kWarps * tpp) {
        const int tl = base + sub;
        const bool act = lane_used && tl < tcount;
        int r = -1;
        if (act) {
            const int64_t e = ld_nc_i64(a.topk + (int64_t)(t0 + tl) * k + j);
            if (e >= 0 && e < E) {
                r = (int)e / a.m;
                atomicAdd(&hist[(int)e], 1);
            } else if (e != -1) {
                report(a.status, MOE_ERR_BAD_TOPK);
            }
        }
        const int key = (r >= 0) ? (sub * R + r) : -(lane + 1);
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const bool owner = r >= 0 && (__ffs(peers) - 1) == lane;
        if (owner) atomicOr(&bitmap[(tl >> 5) * R + r], 1u << (tl & 31));
        if (act) own[tl * k + j] = (int16_t)(owner ? r : -1);
    }
    __syncthreads();
    // ---- the tile's word prefixes and per-rank counts
    const size_t stride = (size_t)a.num_tiles + 1;
    for (int r = threadIdx.x; r < R; r += kThreads) {
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < kWords; ++w) {
            wprefix[r * kWords + w] = (uint16_t)run;
            run += __popc(bitmap[w * R + r]);
        }
        counts[(size_t)r * stride + tile] = (int32_t)run;
    }
    for (int e = threadIdx.x; e < E; e += kThreads) {
        const int h = hist[e];
        if (h) atomicAdd(ws_expert + e, h);
    }
    __syncthreads();
    // ---- positions inside the tile's share of each rank
    for (int i = threadIdx.x; i < tcount * k; i += kThreads) {
        const int r = own[i];
        int32_t v = -1;
        if (r >= 0) {
            const int tl = i / k;
            v = wprefix[r * kWords + (tl >> 5)] + __popc(bitmap[(tl >> 5) * R + r] & ((1u << (tl & 31)) - 1u));
        }
        a.token_dst_row[(int64_t)t0 * k + i] = v;
    }
    // ---- is_token_in_rank rows of the tile, expanded from the bitmap
    uint8_t *dst = a.is_token_in_rank + (int64_t)t0 * R;
    const int nbytes = tcount * R;
    if ((R & 3) == 0) {
        uint32_t *dst4 = reinterpret_cast<uint32_t *>(dst);
        for (int i = threadIdx.x; i < nbytes / 4; i += kThreads) {
            const int tl = (i * 4) / R, r0 = (i * 4) - tl * R;
            uint32_t v = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) v |= ((bitmap[(tl >> 5) * R + r0 + b] >> (tl & 31)) & 1u) << (8 * b);
            dst4[i] = v;
        }
    } else {
        for (int i = threadIdx.x; i < nbytes; i += kThreads) {
            const int tl = i / R, r = i - tl * R;
            dst[i] = (uint8_t)((bitmap[(tl >> 5) * R + r] >> (tl & 31)) & 1u);
        }
    }
}

__global__ void __launch_bounds__(kThreads) layout_scan_kernel(TileArgs a) {
    WarpTrace wt(a.trace, MOE_TRACE_LAYOUT_SCAN);
    __shared__ int s_last;
    WsHeader *hdr = reinterpret_cast<WsHeader *>(a.ws);
    int32_t *ws_expert = reinterpret_cast<int32_t *>(a.ws + a.expert_off);
    int32_t *counts = reinterpret_cast<int32_t *>(a.ws + a.status_off);
    grid_dependency_wait();
    const int r = (int)blockIdx.x;
    int32_t *row = counts + (size_t)r * ((size_t)a.num_tiles + 1);
    block_exclusive_scan(row, a.num_tiles, nullptr, row);   // in place; the total lands in row[num_tiles]
    if (threadIdx.x == 0) a.num_tokens_per_rank[r] = row[a.num_tiles];
    // the last CTA: rank regions and the expert counts and prefix
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(&hdr->done, 1u) == (unsigned)(gridDim.x - 1));
    __syncthreads();
    if (s_last) {
        __threadfence();
        block_exclusive_scan(a.num_tokens_per_rank, a.R, nullptr, a.rank_prefix);
        block_exclusive_scan(ws_expert, a.E, a.num_tokens_per_expert, a.expert_prefix);
    }
}

__global__ void layout_rows_scan_kernel(TileArgs a) {
    WarpTrace wt(a.trace, MOE_TRACE_LAYOUT_ROWS_SCAN);
    grid_dependency_wait();
    const int64_t n = (int64_t)a.T * a.k;   // < 2^31 (checked on the host)
    const int32_t *counts = reinterpret_cast<const int32_t *>(a.ws + a.status_off);
    const size_t stride = (size_t)a.num_tiles + 1;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = a.token_dst_row[i];
        if (v < 0) continue;
        const int r = (int)a.topk[i] / a.m;   // an owning entry is valid
        const int tile = (int)(i / a.k) / kTile;
        a.token_dst_row[i] = v + a.rank_prefix[r] + counts[(size_t)r * stride + tile];
    }
}

// Largest power of two <= min(32, kThreads / R), at least 1.
int lookback_group(int R) {
    int g = 1;
    while (g * 2 <= 32 && g * 2 * R <= kThreads) g *= 2;
    return g;
}

// How many CTAs of `kernel` can be co-resident (cooperative launch bound),
// cached per (device, kernel, shared memory).
int cooperative_capacity(const void *kernel, size_t smem) {
    struct Entry { int dev; const void *fn; size_t smem; int cap; };
    static std::mutex mu;
    static Entry cache[16];
    static int n_cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < std::min(n_cached, 16); ++i)
        if (cache[i].dev == dev && cache[i].fn == kernel && cache[i].smem == smem) return cache[i].cap;
    int coop = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) != cudaSuccess) return 0;
    const int cap = per_sm * device_sm_count();
    cache[n_cached % 16] = Entry{dev, kernel, smem, cap};
    ++n_cached;
    return cap;
}

int launch_cooperative(const void *kernel, int grid, size_t smem, cudaStream_t s, TileArgs &a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&a};
    return cudaLaunchKernelExC(&cfg, kernel, args) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

size_t layout_workspace_bytes(int T, int E, int R) { return ws_layout(T, E, R).total; }

namespace {

// Cluster mode for this batch: CTAs and tokens per CTA, or false (the batch is
// one tile, too large, or clusters of that size cannot be scheduled).
bool cluster_config(int T, int E, int R, int k, int &C, int &tile, size_t &smem) {
    const int want = tuning().layout_cluster;
    if ((want != 8 && want != 16) || T <= kTile || T > want * kClusterMaxTile) return false;
    C = want;
    tile = (int)align_up((size_t)((T + C - 1) / C), 32);
    smem = cluster_smem(tile, E, R, k).total;
    if (smem > device_smem_optin()) return false;
    // whether a cluster of C such CTAs fits on this device (cached per device, size and shared memory)
    struct Entry { int dev, C; size_t smem; bool ok; };
    static std::mutex mu;
    static Entry cache[16];
    static int n_cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < std::min(n_cached, 16); ++i)
        if (cache[i].dev == dev && cache[i].C == C && cache[i].smem == smem) return cache[i].ok;
    bool ok = ensure_dynamic_smem((const void *)layout_cluster_kernel, smem) == MOE_OK;
    if (ok && C > 8)
        ok = cudaFuncSetAttribute((const void *)layout_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                  1) == cudaSuccess;
    if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)C);
        cfg.blockDim = dim3(kCThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        ok = cudaOccupancyMaxActiveClusters(&clusters, (const void *)layout_cluster_kernel, &cfg) == cudaSuccess &&
             clusters >= 1;
    }
    cudaGetLastError();   // a refused attribute or query only means: no cluster mode
    cache[n_cached % 16] = Entry{dev, C, smem, ok};
    ++n_cached;
    return ok;
}

int launch_cluster(int C, size_t smem, cudaStream_t s, bool overlap, TileArgs &a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C);
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, layout_cluster_kernel, a) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

unsigned int *layout_spare_counter(const LayoutLaunch &L) {
    if (L.num_tokens <= kTile || L.workspace == nullptr) return nullptr;   // one tile (or none): no clear
    return &static_cast<WsHeader *>(L.workspace)->pad[0];                  // pad[0], pad[1]
}

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
    int cl_C = 0, cl_tile = 0;
    size_t cl_smem = 0;
    const bool cluster = !L.no_cluster && cluster_config(T, E, R, k, cl_C, cl_tile, cl_smem);
    const size_t smem = smem_layout(E, R, k).total;
    // direct mode: tile size, kernel instance and whether all its tiles fit on the GPU at once
    int dt = direct_tile(T, R);
    const void *direct = dt == kDirectTile ? (const void *)layout_direct_kernel<kDirectTile>
                                           : (const void *)layout_direct_kernel<kTile>;
    const size_t dsmem = dt == kDirectTile ? direct_smem<kDirectTile>(E, R, k).total : direct_smem<kTile>(E, R, k).total;
    const void *coop = (const void *)layout_tiles_kernel<true>;
    if (ensure_dynamic_smem(direct, dsmem) != MOE_OK || ensure_dynamic_smem(coop, smem) != MOE_OK ||
        ensure_dynamic_smem((const void *)layout_tiles_kernel<false>, smem) != MOE_OK ||
        ensure_dynamic_smem((const void *)layout_count_kernel, smem) != MOE_OK)
        return MOE_ERR_CUDA;
    if (dt && (T + dt - 1) / dt > cooperative_capacity(direct, dsmem)) dt = 0;
    if (cluster || L.lookback_only) dt = 0;
    const int tile_tokens = dt ? dt : kTile;
    const int num_tiles = (T + tile_tokens - 1) / tile_tokens;
    // a single-tile direct launch and the cluster mode use no workspace
    if (!cluster && !(dt && num_tiles == 1) && cudaMemsetAsync(L.workspace, 0, w.total, s) != cudaSuccess)
        return MOE_ERR_CUDA;

    TileArgs a;
    a.trace = trace_args();
    a.topk = L.topk_idx;
    a.T = T; a.k = k; a.E = E; a.R = R; a.m = E / R;
    a.num_tiles = num_tiles;
    a.group = lookback_group(R);
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
    a.early_dependents = L.early_dependents ? 1 : 0;
    a.cl_tile = cl_tile;
    a.spare = layout_spare_counter(L);
    if (cluster) return launch_cluster(cl_C, cl_smem, s, tuning().overlap != 0, a);

    if (dt) {
        if (a.num_tiles == 1) {     // nothing to exchange: an ordinary launch (dt == kTile)
            return launch_kernel(layout_direct_kernel<kTile>, dim3(1), dim3(kThreads), dsmem, s, tuning().overlap != 0,
                                 a) == cudaSuccess
                       ? MOE_OK
                       : MOE_ERR_CUDA;
        }
        return launch_cooperative(direct, a.num_tiles, dsmem, s, a);
    }
    if (a.num_tiles <= cooperative_capacity(coop, smem)) return launch_cooperative(coop, a.num_tiles, smem, s, a);
    // more tiles than fit at once: the scan mode (three launches, no waits), unless
    // the lookback is asked for (layout_mode 2, or the unpublished-tile test hook)
    if (!L.lookback_only && L.unpublished_tile < 0 && tuning().layout_scan) {
        const bool ov = tuning().overlap != 0;
        if (launch_kernel(layout_count_kernel, dim3(a.num_tiles), dim3(kThreads), smem, s, ov, a) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (launch_kernel(layout_scan_kernel, dim3(R), dim3(kThreads), 0, s, ov, a) != cudaSuccess)
            return MOE_ERR_CUDA;
        const int64_t n = (int64_t)T * k;
        const int blocks = (int)std::min<int64_t>((n + 255) / 256, (int64_t)device_sm_count() * 8);
        return launch_kernel(layout_rows_scan_kernel, dim3(blocks), dim3(256), 0, s, ov, a) == cudaSuccess
                   ? MOE_OK
                   : MOE_ERR_CUDA;
    }

    if (launch_kernel(layout_tiles_kernel<false>, dim3(a.num_tiles), dim3(kThreads), smem, s, tuning().overlap != 0, a) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    const int64_t n = (int64_t)T * k;
    const int threads = 256;
    const int blocks = (int)std::min<int64_t>((n + threads - 1) / threads, (int64_t)device_sm_count() * 8);
    if (launch_kernel(layout_rows_kernel, dim3(blocks), dim3(threads), 0, s, tuning().overlap != 0, L.topk_idx, n, a.m,
                      (const int32_t *)o.rank_prefix, o.token_dst_row, a.trace) != cudaSuccess)
        return MOE_ERR_CUDA;
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

}  // namespace
}  // namespace moe

extern "C" MOE_API int moe_get_layout_noalloc(const int64_t *topk_idx, int num_tokens, int num_topk,
                                              int num_experts, int num_ranks, moe_layout_t layout,
                                              int32_t *status, void *stream) {
    const int T = num_tokens;
    // the same checks as moe_get_layout, first without the workspace (no CUDA call
    // for a bad argument), then with the scratch standing in for it, so that a size
    // beyond the scratch returns MOE_ERR_WORKSPACE before anything is launched
    int rc = moe::layout_check_args(topk_idx, T, num_topk, num_experts, num_ranks, layout, status);
    if (rc != MOE_OK) return rc;
    if (T > 0 && moe::layout_workspace_bytes(T, num_experts, num_ranks) > (size_t)MOE_NOALLOC_SCRATCH_BYTES)
        return MOE_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (T > 0) {
        scratch = moe::noalloc_scratch_address(&rc);
        if (scratch == nullptr) return rc;
    }
    moe::LayoutLaunch L;
    rc = moe::layout_prepare(topk_idx, T, num_topk, num_experts, num_ranks, layout, scratch,
                             (size_t)MOE_NOALLOC_SCRATCH_BYTES, status, stream, 0, -1, L, false);
    return rc != MOE_OK ? rc : moe::launch_layout(L);
}
