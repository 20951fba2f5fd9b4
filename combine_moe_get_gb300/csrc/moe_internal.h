// moe_internal.h -- host-side interfaces between the C ABI entry points
// (moe_api.cu) and the kernel launchers (layout.cu, expand.cu, dispatch.cu,
// combine.cu).
// Arguments reaching a launcher have already been validated.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/moe_get.h"

namespace moe {

// Per-device facts, queried once per device (thread-safe).
int device_sm_count();             // SMs of the current device
size_t device_smem_per_sm();       // shared memory per SM (bytes)
size_t device_smem_optin();        // max dynamic shared memory per block (bytes)
size_t device_l2_bytes();          // L2 cache size (bytes)

// Raise a kernel's dynamic shared-memory limit to at least `bytes` (cached).
int ensure_dynamic_smem(const void *kernel, size_t bytes);

// Where kernels built with MOE_PROFILE append their warps' records (all null /
// zero: not tracing); every launcher copies it into its kernel's arguments.
struct TraceArgs {
    moe_trace_record_t *rec;
    uint32_t *count;
    int cap;
    int what;   // MOE_TRACE_WARPS | MOE_TRACE_PHASES
};
TraceArgs trace_args();

// Tuning knobs. They are fixed when the library is compiled (the defaults
// below are the measured best on this GPU and the configuration every parity
// test runs); a variant build may override one with -DMOE_TUNE_<NAME>=<value>.
// Nothing is read from the environment at run time.
#ifndef MOE_TUNE_DISPATCH_WARPS
#define MOE_TUNE_DISPATCH_WARPS 8
#endif
#ifndef MOE_TUNE_DISPATCH_STAGES
#define MOE_TUNE_DISPATCH_STAGES 4
#endif
#ifndef MOE_TUNE_DISPATCH_CHUNK
#define MOE_TUNE_DISPATCH_CHUNK 16384
#endif
#ifndef MOE_TUNE_DISPATCH_SMEM
#define MOE_TUNE_DISPATCH_SMEM (200 << 10)
#endif
#ifndef MOE_TUNE_COMBINE_WARPS
#define MOE_TUNE_COMBINE_WARPS 8
#endif
#ifndef MOE_TUNE_COMBINE_CHUNK
#define MOE_TUNE_COMBINE_CHUNK 8192
#endif
#ifndef MOE_TUNE_COMBINE_RING_BYTES
#define MOE_TUNE_COMBINE_RING_BYTES (224 << 10)
#endif
#ifndef MOE_TUNE_COMBINE_FP8_POOL
#define MOE_TUNE_COMBINE_FP8_POOL 15
#endif
#ifndef MOE_TUNE_COMBINE_FP8_POOL_MIN_TOKENS
#define MOE_TUNE_COMBINE_FP8_POOL_MIN_TOKENS 40
#endif
#ifndef MOE_TUNE_COMBINE_FP8_WARPS
#define MOE_TUNE_COMBINE_FP8_WARPS 10
#endif
#ifndef MOE_TUNE_OVERLAP
#define MOE_TUNE_OVERLAP 1
#endif
#ifndef MOE_TUNE_DISPATCH_POOL
#define MOE_TUNE_DISPATCH_POOL 50
#endif
#ifndef MOE_TUNE_COMBINE_PREFETCH
#define MOE_TUNE_COMBINE_PREFETCH (96 << 10)
#endif
#ifndef MOE_TUNE_COMBINE_POOL
#define MOE_TUNE_COMBINE_POOL 30
#endif
#ifndef MOE_TUNE_LAYOUT_CLUSTER
#define MOE_TUNE_LAYOUT_CLUSTER 16
#endif
#ifndef MOE_TUNE_FP8_ROWS
#define MOE_TUNE_FP8_ROWS 1
#endif
#ifndef MOE_TUNE_FP8_IN_SLOTS
#define MOE_TUNE_FP8_IN_SLOTS 12
#endif
#ifndef MOE_TUNE_FP8_ROWS_POOL
#define MOE_TUNE_FP8_ROWS_POOL 50
#endif
#ifndef MOE_TUNE_FP8_ROWS_POOL_MIN_ROWS
#define MOE_TUNE_FP8_ROWS_POOL_MIN_ROWS 40
#endif
#ifndef MOE_TUNE_FP8_QUANT_WARPS
#define MOE_TUNE_FP8_QUANT_WARPS 24
#endif
#ifndef MOE_TUNE_CTAS_PER_SM
#define MOE_TUNE_CTAS_PER_SM 0
#endif
#ifndef MOE_TUNE_L2_HINTS
#define MOE_TUNE_L2_HINTS 1
#endif
#ifndef MOE_TUNE_SPREAD_SMALL
#define MOE_TUNE_SPREAD_SMALL 1
#endif
#ifndef MOE_TUNE_FUSED_SMALL
#define MOE_TUNE_FUSED_SMALL 1
#endif
#ifndef MOE_TUNE_FUSED_MIN_WARPS
#define MOE_TUNE_FUSED_MIN_WARPS 4
#endif
#ifndef MOE_TUNE_LAYOUT_SCAN
#define MOE_TUNE_LAYOUT_SCAN 1
#endif
#ifndef MOE_TUNE_DISPATCH_PREFETCH
#define MOE_TUNE_DISPATCH_PREFETCH (1 << 20)
#endif
#ifndef MOE_TUNE_DISPATCH_PREFETCH_ALWAYS
#define MOE_TUNE_DISPATCH_PREFETCH_ALWAYS 1
#endif
#ifndef MOE_TUNE_DISPATCH_PREFETCH_L2_PCT
#define MOE_TUNE_DISPATCH_PREFETCH_L2_PCT 25
#endif
#ifndef MOE_TUNE_DISPATCH_PREFETCH_L2_PCT_ALONE   // a dispatch not launched behind the layout
#define MOE_TUNE_DISPATCH_PREFETCH_L2_PCT_ALONE 15
#endif
// the dispatch launched behind this library's layout (moe_layout_dispatch, two
// launches): 2 warps x 4 stages, two CTAs per SM, measured faster there
#ifndef MOE_TUNE_LD_DISPATCH_WARPS
#define MOE_TUNE_LD_DISPATCH_WARPS 2
#endif
#ifndef MOE_TUNE_LD_DISPATCH_STAGES
#define MOE_TUNE_LD_DISPATCH_STAGES 4
#endif
#ifndef MOE_TUNE_DISPATCH_PREFETCH_NOSYNC
#define MOE_TUNE_DISPATCH_PREFETCH_NOSYNC 1
#endif
#ifndef MOE_TUNE_DISPATCH_PREFETCH_KEEP
#define MOE_TUNE_DISPATCH_PREFETCH_KEEP 1
#endif
struct Tuning {
    int dispatch_warps, dispatch_stages, dispatch_chunk;
    int ld_dispatch_warps, ld_dispatch_stages;              // ... launched behind this library's layout
    int dispatch_smem;                                       // shared-memory budget of a chunked dispatch CTA
    int combine_warps, combine_chunk, combine_ring_bytes;   // consumer warps, max chunk, ring budget
    int combine_fp8_warps;                                   // consumer warps for E4M3 partial rows
    int combine_fp8_pool, combine_fp8_pool_min_tokens;       // E4M3 rows: pool % and the tokens per CTA it needs
    int fp8_rows, fp8_in_slots, fp8_quant_warps;   // FP8 row pipeline: on/off, input ring slots, worker warps
    int fp8_rows_pool;  // % of the FP8 row pipeline's tokens left to a pool when a cleared counter is at hand
    int fp8_rows_pool_min_rows;  // ... only with at least this many rows per CTA
    int ctas_per_sm;
    int l2_hints;  // bit 0: evict-first on single-use loads; bit 1: evict-first on stores
    int spread_small;   // small batches: fewer dispatch warps per CTA, more CTAs
    int fused_small;    // moe_layout_dispatch: one fused launch for small batches
    int fused_min_warps;  // ... only when each CTA gets at least this many warps
    int overlap;        // programmatic dependent launch of every non-cooperative kernel
    int dispatch_pool;  // % of dispatch units left to a shared pool when a cleared counter is at hand (>= 100: off)
    int combine_pool;   // % of combine tokens left to a shared pool when the caller gives a counter (>= 100: off)
    int combine_prefetch;   // bytes of its first rows each combine CTA prefetches into L2 before the dependency wait
    int layout_cluster; // CTAs of the cluster-mode layout (8 or 16; other values: off)
    int layout_scan;    // the scan mode instead of the ticket lookback for more tiles than fit at once
    int dispatch_prefetch;       // input units per CTA prefetched into L2 (moe_layout_dispatch: during the layout)
    int dispatch_prefetch_keep;  // ... with an evict-last policy (else evict-normal)
    int dispatch_prefetch_always;  // ... in every chunked dispatch, not only behind the layout
    int dispatch_prefetch_l2_pct;  // ... holding at most this share of L2 evict-last
    int dispatch_prefetch_l2_pct_alone;  // ... the same for a dispatch not launched behind the layout
};
const Tuning &tuning();

struct LayoutLaunch {
    const int64_t *topk_idx;
    int num_tokens, num_topk, num_experts, num_ranks;
    moe_layout_t out;
    void *workspace;
    int32_t *status;
    void *stream;
    int64_t timeout_ns;     // <= 0: default
    int unpublished_tile;   // test hook, -1 = off
    // let the next grid on the stream launch as soon as every CTA has passed its
    // dependency wait (the next launch is this library's dispatch)
    bool early_dependents = false;
    bool no_cluster = false;      // never the cluster mode
    bool lookback_only = false;   // only the lookback modes (not cluster, direct or scan)
};

size_t layout_workspace_bytes(int num_tokens, int num_experts, int num_ranks);
int launch_layout(const LayoutLaunch &L);

// Host-side checks of a layout call (moe_api.cu), shared by every layout entry
// point. layout_check_args: shape, pointers and alignment, but not the
// workspace. layout_prepare: those checks, then the workspace (present,
// 16-byte aligned, at least layout_workspace_bytes: else MOE_ERR_WORKSPACE),
// then the launch description. MOE_OK or the error code; nothing is launched.
int layout_check_args(const int64_t *topk_idx, int T, int k, int E, int R, const moe_layout_t &o,
                      const int32_t *status);
int layout_prepare(const int64_t *topk_idx, int T, int k, int E, int R, moe_layout_t o, void *workspace,
                   size_t workspace_bytes, int32_t *status, void *stream, int64_t timeout_ns, int unpublished_tile,
                   LayoutLaunch &L, bool no_cluster);
// Two 32-bit words of the layout workspace that launch_layout(L) zeroes (with
// the workspace clear, or from the cluster-mode kernel) and then leaves alone,
// free for the next launch of the same call -- which may rely on them only
// after its dependency wait; nullptr for a batch of one tile.
unsigned int *layout_spare_counter(const LayoutLaunch &L);

struct ExpandLaunch {
    const int64_t *topk_idx;
    int num_tokens, num_topk, num_experts;
    const int32_t *expert_prefix;
    int32_t *token_expert_row;
    void *workspace;
    int32_t *status;
    void *stream;
    int64_t timeout_ns;     // <= 0: default
    int unpublished_tile;   // test hook, -1 = off
    bool no_cluster = false;   // never the cluster mode
};

size_t expand_workspace_bytes(int num_tokens, int num_experts);
int launch_expand_layout(const ExpandLaunch &L);

struct DispatchLaunch {
    const void *x;
    int num_tokens, hidden;
    const int64_t *topk_idx;
    const float *topk_weights;
    int num_topk, num_experts, num_ranks;
    const int32_t *token_dst_row;
    int recv_capacity;
    int mode;                 // moe_dispatch_mode_t, without MOE_DISPATCH_EXPAND
    bool expand;              // token_dst_row holds expand-mode rows
    void *recv_x;
    float *recv_x_scales;
    int64_t *recv_topk_idx;
    float *recv_topk_weights;
    int32_t *recv_src_idx;
    float *x_scales;
    int32_t *status;
    void *stream;
    // the launch before this one is the layout of the same call, which passed its
    // own dependency wait before letting this grid launch: the input rows are
    // complete, so the first stage loads may be issued before the wait
    bool loads_before_wait = false;
    // optional: two zeroed uint32 for tail balancing (a pool of units shared by all
    // CTAs); the launch leaves them zeroed
    unsigned int *pool = nullptr;
};

int launch_dispatch(const DispatchLaunch &L);
// Layout and dispatch: one fused launch for small batches, else the two launches.
int launch_layout_dispatch(const LayoutLaunch &Ll, const DispatchLaunch &L);

struct CombineLaunch {
    const void *partial;                     // bf16 rows, or E4M3 codes (fp8)
    bool fp8 = false;                        // E4M3 rows with per-128 scales
    const float *partial_scales = nullptr;   // E4M3 rows: fp32 scales [rows, H/128]
    int num_partial_rows, num_tokens, hidden, num_topk;
    const int32_t *token_dst_row;
    const float *row_weights;          // optional
    const float *recv_topk_weights;    // optional, with combined_topk_weights
    float *combined_topk_weights;
    void *out;
    int32_t *status;
    void *stream;
    // optional: two zeroed uint32 of device memory for tail balancing (left zeroed)
    uint32_t *balance = nullptr;
};

int launch_combine(const CombineLaunch &L);

}  // namespace moe
