/*
 * moe_get.h -- C ABI of the single-GPU MoE layout / dispatch / combine library
 * (libmoe_get.so, CUDA kernels for sm_103a).
 *
 * Expert parallelism on one GPU: the R "ranks" are logical destination
 * partitions laid out one after another in one receive buffer in HBM.
 * Nothing crosses GPUs.
 *
 * Notation (DeepEP V2 deep-dive page, "DeepEP V2 深度深潜", sections 2.2-3.5):
 *   T = num_tokens, H = hidden, E = num_experts, R = num_ranks,
 *   m = E / R experts per rank (E % R == 0), k = num_topk (1..32),
 *   rank(e) = e / m for an expert e >= 0; a top-k entry of -1 is masked.
 *   D_t = number of distinct ranks of token t; N = sum_t D_t received rows.
 *
 * Conventions shared by every entry point
 *   - All array arguments are DEVICE pointers, row-major and contiguous,
 *     allocated and owned by the caller. The library never allocates, frees or
 *     synchronises; every call is asynchronous on `stream` (a cudaStream_t
 *     passed as void*; NULL = the legacy default stream).
 *   - The return value reports errors the host can see before launching:
 *     MOE_ERR_INVALID_ARG (null pointer, size out of range), MOE_ERR_MISALIGNED
 *     (a row pointer or row pitch not 16-byte aligned) or MOE_ERR_CUDA (a launch
 *     failed). Nothing is launched when the return value is not MOE_OK.
 *   - Errors that depend on the data are written by the kernels to the device
 *     word `*status` (int32): the first error wins (compare-and-swap from 0),
 *     later ones are dropped. The library never clears `*status`: zero it before
 *     the first call whose errors you want to see, and read it after the stream
 *     has synchronised. Data errors are MOE_ERR_BAD_TOPK (a top-k entry outside
 *     [-1, E); that entry is treated as masked), MOE_ERR_CAPACITY (a receive row
 *     at or beyond the receive capacity; that row is not written / not read) and
 *     MOE_ERR_TIMEOUT (a bounded wait inside a kernel ran out; the outputs of
 *     that call are unspecified).
 *   - T == 0 is a valid no-op that still writes zero counts and prefixes.
 */
#ifndef MOE_GET_H
#define MOE_GET_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_MISALIGNED = 2,
    MOE_ERR_CAPACITY = 3,
    MOE_ERR_BAD_TOPK = 4,
    MOE_ERR_TIMEOUT = 5,
    MOE_ERR_CUDA = 6,
    MOE_ERR_WORKSPACE = 7
} moe_status_t;

/* Limits checked on the host (MOE_ERR_INVALID_ARG beyond them). */
#define MOE_MAX_TOPK 32
#define MOE_MAX_RANKS 1024
#define MOE_MAX_EXPERTS 8192

/* Outputs of moe_get_layout: all DEVICE pointers, caller-owned. */
typedef struct {
    int32_t *num_tokens_per_rank;   /* [R]    tokens received by each rank (each token once per rank) */
    int32_t *num_tokens_per_expert; /* [E]    valid top-k entries naming each expert (one per entry)  */
    uint8_t *is_token_in_rank;      /* [T, R] 1 if token t has at least one expert on rank r, else 0  */
    int32_t *rank_prefix;           /* [R+1]  exclusive prefix of num_tokens_per_rank; [R] = N          */
    int32_t *expert_prefix;         /* [E+1]  exclusive prefix of num_tokens_per_expert                 */
    int32_t *token_dst_row;         /* [T, k] global receive row of (t, rank(topk_idx[t,j])) held by the
                                               lowest entry j naming that rank, -1 for every other entry */
} moe_layout_t;

/* Bytes of device workspace moe_get_layout needs for these sizes (16-byte
 * aligned pointer required). Host-only; never fails (0 for invalid sizes). */
MOE_API size_t moe_get_layout_workspace_size(int num_tokens, int num_experts, int num_ranks);

/*
 * moe_get_layout -- routing counts, membership and receive positions.
 *
 * Page: notify warps of the dispatch kernel (section 3.3 stage 1): per valid
 * top-k entry one count for its expert, and one count per rank after the
 * entries of a token are de-duplicated by rank; then prefix sums giving the
 * receive offsets (section 3.5, "prefix sum -> psum_num_recv_tokens"). The
 * rank of an expert is expert / experts_per_rank (section 2.2).
 *
 * Receive order (the page assigns slots by atomicAdd, i.e. arrival order; this
 * library fixes a deterministic order instead): rank r's rows occupy
 * [rank_prefix[r], rank_prefix[r+1]) in ascending source-token order, so
 *   token_dst_row[t, j] = rank_prefix[r] + #{t' < t : is_token_in_rank[t', r]}.
 * The in-rank position is a column-wise exclusive scan over tokens. For
 * 129..8192 tokens it is computed inside one 16-CTA thread-block cluster,
 * whose tiles exchange their counts through distributed shared memory (no
 * waits, no workspace use). Otherwise it is an all-tile sweep of published
 * counts (up to 128 tiles of 64 tokens), a single-pass decoupled-lookback
 * scan over tiles of 128 tokens while every tile fits on the GPU at once
 * (both wait on other CTAs, bounded, with MOE_ERR_TIMEOUT on expiry), and
 * beyond that the scan mode: per-tile counts, a scan per rank, then the rows
 * (three launches, no waits).
 *
 *   topk_idx   [T, k] int64, device. -1 = masked; other values outside [0, E)
 *              raise MOE_ERR_BAD_TOPK and are treated as masked.
 *   layout     output arrays (all must be non-null when T > 0; rank_prefix and
 *              expert_prefix, num_tokens_per_* are always written).
 *   workspace  device scratch of at least moe_get_layout_workspace_size()
 *              bytes; contents need not be initialised (a mode that uses it
 *              clears it with cudaMemsetAsync on `stream`). Must not be shared
 *              by calls that overlap on the GPU.
 *   status     device int32, see conventions.
 * Limits: 1 <= k <= 32, 1 <= R <= 1024, E <= 8192, E % R == 0,
 * T * k < 2^31, T * R < 2^40.
 */
MOE_API int moe_get_layout(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                           int num_ranks, moe_layout_t layout, void *workspace, size_t workspace_bytes,
                           int32_t *status, void *stream);

/* Options of moe_get_layout_ex. */
typedef struct {
    /* Bound on each wait of the lookback scan, in nanoseconds of the GPU's
     * global timer; <= 0 selects the default (1 s). On expiry the kernel writes
     * MOE_ERR_TIMEOUT to *status and finishes without waiting further. */
    int64_t wait_timeout_ns;
    /* Failure-injection hook for tests: the tile with this index (64 or 128
     * tokens, as the mode sizes it) never publishes its scan status, so that
     * the tiles after it (and the final count step) run out of their bounded
     * waits and report MOE_ERR_TIMEOUT. Naming a tile also keeps the call on
     * the lookback modes (off the cluster and scan modes, which have no
     * waits). -1 = off (the only value for production use). */
    int32_t test_unpublished_tile;
    /* 0: the mode is chosen by size (the cluster mode for 129..8192 tokens
     * where the device can schedule it, the direct mode for few tiles, the
     * cooperative lookback while every tile fits on the GPU at once, and
     * beyond that the scan mode: three launches with no waits); 1: never the
     * cluster mode; 2: only the lookback modes (cooperative, or with tickets
     * beyond what fits at once). All give the same outputs. */
    int32_t layout_mode;
} moe_layout_options_t;

/*
 * moe_get_layout_ex -- moe_get_layout with options (NULL = defaults).
 * Same arguments, outputs and errors as moe_get_layout.
 */
MOE_API int moe_get_layout_ex(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                              int num_ranks, moe_layout_t layout, void *workspace, size_t workspace_bytes,
                              int32_t *status, void *stream, const moe_layout_options_t *options);

/* Bytes of device workspace moe_get_expand_layout needs (16-byte aligned
 * pointer required). Host-only; never fails (0 for invalid sizes). */
MOE_API size_t moe_get_expand_layout_workspace_size(int num_tokens, int num_experts);

/*
 * moe_get_expand_layout -- receive rows of expand mode: one row per valid
 * top-k entry, grouped by expert (the layout a grouped expert GEMM reads).
 *
 * Page: copy epilogue of the dispatch (section 3.3 stage 3), expand mode: the
 * destination of a received token is taken from a counter per expert that
 * starts at the exclusive prefix of the per-expert counts
 * (psum_num_recv_tokens_per_expert) and advances by one per placed token.
 * The page advances it with atomicAdd (arrival order); this library places
 * the entries of each expert in source order instead:
 *   token_expert_row[t, j] = expert_prefix[e] + #{(t', j') < (t, j) in
 *                            (token, choice) order : topk_idx[t', j'] == e}
 * for e = topk_idx[t, j] in [0, E), and -1 for masked or invalid entries.
 * Expert e's rows are [expert_prefix[e], expert_prefix[e+1]); since experts
 * are numbered rank by rank, rank r's rows are [expert_prefix[r*m],
 * expert_prefix[(r+1)*m]). A token naming one expert in two entries gets two
 * rows. The number of rows is expert_prefix[E] (<= T*k). The in-expert
 * position is a column scan over tokens: for T <= 4096 and E <= 1024, inside
 * one 16-CTA thread-block cluster through distributed shared memory (no
 * waits, no workspace use); otherwise a decoupled lookback over tiles of 256
 * tokens (bounded waits, MOE_ERR_TIMEOUT on expiry).
 *
 *   topk_idx          [T, k] int64, device (as for moe_get_layout).
 *   expert_prefix     [E+1] int32, device, input: moe_get_layout's output for
 *                     the same topk_idx (enqueued earlier, e.g. on the same stream).
 *   token_expert_row  [T, k] int32, device, output. Pass it as `token_dst_row`
 *                     to moe_dispatch with MOE_DISPATCH_EXPAND and to
 *                     moe_combine / moe_combine_ex.
 *   workspace         device scratch of at least
 *                     moe_get_expand_layout_workspace_size() bytes, cleared by the
 *                     call on `stream` when the lookback mode uses it; not shared
 *                     by calls that overlap on the GPU.
 *   options           NULL or the options of moe_get_layout_ex; here the test hook
 *                     names a tile of 256 tokens (and keeps the call off the
 *                     cluster mode, as does layout_mode 1).
 * Limits: 1 <= k <= 32, 1 <= E <= 8192, T * k < 2^31.
 */
MOE_API int moe_get_expand_layout(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                                  const int32_t *expert_prefix, int32_t *token_expert_row, void *workspace,
                                  size_t workspace_bytes, int32_t *status, void *stream,
                                  const moe_layout_options_t *options);

/*
 * moe_dispatch -- copy each token once per distinct destination rank.
 *
 * Page: dispatch warps (section 3.3 stage 2) load a token's hidden row once
 * and store it once per de-duplicated destination rank; the HBM model of
 * section 1.3 (factor 2) counts one read per token and one write per rank.
 * Receive rows hold, per row (section 3.4 TokenLayout, section 3.5 outputs):
 *   recv_x[row]            = x[t]                      (bf16 mode), or
 *   recv_x[row]            = e4m3(x[t] / scale) and
 *   recv_x_scales[row, b]  = scale[t, b]               (FP8 mode, see below)
 *   recv_src_idx[row]      = t
 *   recv_topk_idx[row, j]  = topk_idx[t, j] - r*m if rank(topk_idx[t, j]) == r, else -1
 *   recv_topk_weights[row, j] = topk_weights[t, j] if that entry is local, else 0
 * where row = token_dst_row[t, j] >= 0 for the owning entry j and r its rank.
 *
 * Modes (argument `mode`, H % 128 == 0 for the FP8 modes):
 *   MOE_DISPATCH_BF16           x bf16 [T, H]; recv_x bf16.
 *   MOE_DISPATCH_QUANTIZE_FP8   x bf16; recv_x E4M3 codes and recv_x_scales. Per token
 *                               and block of 128 channels: amax = max |x|, scale =
 *                               amax / 448 (fp32, round to nearest), code = E4M3(x /
 *                               scale) (IEEE fp32 division, round to nearest even,
 *                               saturating to +-448); a block with amax == 0 has scale 0
 *                               and codes 0. x_scales, if given, receives the scales.
 *   MOE_DISPATCH_FP8            x already E4M3 [T, H] bytes with its scales x_scales
 *                               [T, H/128] (input, section 3.4's sf next to the hidden
 *                               bytes); codes and scales are copied unchanged.
 * Any of the three may be OR-ed with MOE_DISPATCH_EXPAND (expand mode, section 3.3
 * stage 3): `token_dst_row` is then the token_expert_row of moe_get_expand_layout,
 * the token goes once to the row of every valid entry (t, j), and each row's
 * metadata keeps that entry only:
 *   recv_topk_idx[row, jj] = topk_idx[t, j] - r*m for jj == j, else -1;
 *   recv_topk_weights[row, jj] = topk_weights[t, j] for jj == j, else 0.
 * (In expand mode a token has several rows on one rank, one per local expert, so
 * the rank-wide record would repeat its other local entries.)
 *
 *   x                  [T, H] bf16 (E4M3 bytes in MOE_DISPATCH_FP8), device, 16-byte
 *                      aligned, H % 8 == 0.
 *   topk_idx           [T, k] int64 (the same array given to moe_get_layout).
 *   topk_weights       [T, k] fp32 or NULL (then recv_topk_weights may be NULL).
 *   token_dst_row      [T, k] int32 from moe_get_layout.
 *   recv_capacity      rows available in the receive arrays; rows >= capacity
 *                      raise MOE_ERR_CAPACITY and are skipped. N <= T*min(k, R)
 *                      (expand mode: expert_prefix[E] <= T*k).
 *   recv_x             [capacity, H] bf16, or [capacity, H] uint8 E4M3 in the FP8 modes.
 *   recv_x_scales      [capacity, H/128] fp32 (FP8 modes only, else ignored).
 *   recv_topk_idx      [capacity, k] int64, may be NULL (not written).
 *   recv_topk_weights  [capacity, k] fp32, may be NULL.
 *   recv_src_idx       [capacity] int32, may be NULL.
 *   x_scales           [T, H/128] fp32: output of MOE_DISPATCH_QUANTIZE_FP8 (may be
 *                      NULL), input of MOE_DISPATCH_FP8 (required), else ignored.
 */
typedef enum {
    MOE_DISPATCH_BF16 = 0,
    MOE_DISPATCH_QUANTIZE_FP8 = 1,
    MOE_DISPATCH_FP8 = 2,
    MOE_DISPATCH_EXPAND = 0x100   /* flag, OR-ed with one of the above */
} moe_dispatch_mode_t;

MOE_API int moe_dispatch(const void *x, int num_tokens, int hidden, const int64_t *topk_idx,
                         const float *topk_weights, int num_topk, int num_experts, int num_ranks,
                         const int32_t *token_dst_row, int recv_capacity, int mode,
                         void *recv_x, float *recv_x_scales, int64_t *recv_topk_idx,
                         float *recv_topk_weights, int32_t *recv_src_idx, float *x_scales,
                         int32_t *status, void *stream);

/*
 * moe_dispatch_ex -- moe_dispatch with a balance counter (a library addition,
 * as for moe_combine_ex; results do not depend on it).
 *
 *   balance   NULL, or 2 uint32 of device memory, 8-byte aligned, zero before
 *             the first call that uses them; every call leaves them zero again
 *             (the last CTA to finish clears them, also after a timeout). With
 *             it, half of the (token, chunk) units are dealt round-robin to the
 *             CTAs and the rest are claimed one by one, so that CTAs on SMs with
 *             more bandwidth take more of them (at DSv3 the SMs finished a
 *             statically split dispatch 39-59 us apart). Used by the bf16,
 *             pass-through and expand modes; the quantising FP8 row pipeline and
 *             batches of fewer than 8 units per CTA ignore it. Two calls that use
 *             the same counter must not run at the same time on the GPU.
 *             Misaligned: MOE_ERR_MISALIGNED.
 * Other arguments, errors and limits as for moe_dispatch.
 */
MOE_API int moe_dispatch_ex(const void *x, int num_tokens, int hidden, const int64_t *topk_idx,
                            const float *topk_weights, int num_topk, int num_experts, int num_ranks,
                            const int32_t *token_dst_row, int recv_capacity, int mode, void *recv_x,
                            float *recv_x_scales, int64_t *recv_topk_idx, float *recv_topk_weights,
                            int32_t *recv_src_idx, float *x_scales, uint32_t *balance, int32_t *status,
                            void *stream);

/*
 * moe_layout_dispatch -- moe_get_layout followed by moe_dispatch, in one
 * launch for small batches (decode).
 *
 * Page: the dispatch kernel runs its notify warps (counts, prefix sums) and
 * its dispatch warps in one launch (section 3.5, data-flow figure). Here, for
 * T <= 1024 (and the layout's shared memory fitting
 * beside the copy pipeline), every CTA of the dispatch grid computes the whole
 * layout itself in shared memory -- no CTA waits on another -- while its first
 * row loads are in flight, then stores the rows; the layout outputs are written
 * to `layout` as moe_get_layout writes them. Larger batches take the two
 * launches. On that path
 * the dispatch is launched to overlap the layout: its CTAs load input rows
 * while the layout runs (the layout has passed its own dependency wait, so the
 * rows are complete) and read the layout's outputs only after it ends. It also
 * balances its tail as moe_dispatch_ex does, with two words of the workspace
 * that the layout clears as its counter. Outputs, order,
 * metadata and errors are exactly those of moe_get_layout + moe_dispatch with
 * the same arguments.
 *
 *   layout, workspace, workspace_bytes   as for moe_get_layout (the workspace is
 *                      only used by the two-launch path but is always required).
 *   token_dst_row      not an argument: layout.token_dst_row receives the rows.
 *   other arguments    as for moe_dispatch; `mode` may not include
 *                      MOE_DISPATCH_EXPAND (MOE_ERR_INVALID_ARG).
 */
MOE_API int moe_layout_dispatch(const void *x, int num_tokens, int hidden, const int64_t *topk_idx,
                                const float *topk_weights, int num_topk, int num_experts, int num_ranks,
                                moe_layout_t layout, void *workspace, size_t workspace_bytes, int recv_capacity,
                                int mode, void *recv_x, float *recv_x_scales, int64_t *recv_topk_idx,
                                float *recv_topk_weights, int32_t *recv_src_idx, float *x_scales, int32_t *status,
                                void *stream);

/*
 * moe_combine -- gather the per-rank partial rows of each token back into
 * token order and reduce them.
 *
 * Page: the expert side writes one partial row per (token, rank) into the
 * owner's combine buffer and an epilogue reduces them (Mega-MoE combine push
 * on the DeepEP/DeepGEMM comparison page; "consume ready partial rows in the
 * reduce epilogue" on the Ascend send-ordering page). Reduction order:
 *   out[t] = bf16_rn( sum over the rows of t in ascending rank order of
 *                     float(partial[row]) ), accumulated in fp32 from +0.0f,
 * ascending rank being ascending row because rank regions are in rank order.
 * A token with no rows gets +0. No weights are applied (the expert stage
 * applies them).
 *
 *   partial          [num_partial_rows, H] bf16, device, 16-byte aligned, H % 8 == 0.
 *   token_dst_row    [T, k] int32 from moe_get_layout; rows >= num_partial_rows
 *                    raise MOE_ERR_CAPACITY and are skipped. In expand mode, the
 *                    token_expert_row of moe_get_expand_layout: one partial row per
 *                    valid entry, summed in ascending row (= expert) order.
 *   out              [T, H] bf16, device, 16-byte aligned.
 */
MOE_API int moe_combine(const void *partial, int num_partial_rows, int num_tokens, int hidden,
                        int num_topk, const int32_t *token_dst_row, void *out, int32_t *status,
                        void *stream);

/*
 * moe_combine_fp8 -- moe_combine for partial rows held as E4M3 codes with one
 * fp32 scale per 128 channels (the layout MOE_DISPATCH_QUANTIZE_FP8 writes).
 *
 * Pages: the FP8 path of the intra/inter-node page carries x_scales next to
 * the hidden bytes; the combine reduces the partial rows as moe_combine does.
 * Each element is dequantised on its own, v = RN(value(code) * scale) in fp32
 * (no fused multiply-add), and the token's values are summed as in
 * moe_combine: ascending row, fp32 from +0.0f, one RNE cast to bf16.
 *
 *   partial_codes   [num_partial_rows, H] uint8 E4M3, device, 16-byte aligned.
 *   partial_scales  [num_partial_rows, H/128] fp32, device, 16-byte aligned.
 *   token_dst_row   [T, k] int32 (either row map); rows >= num_partial_rows
 *                   raise MOE_ERR_CAPACITY and are skipped.
 *   out             [T, H] bf16, device, 16-byte aligned.
 * Limits: H % 512 == 0 (so that a row's scales are whole 16-byte pieces),
 * H <= 2^24, 1 <= k <= 32.
 */
MOE_API int moe_combine_fp8(const void *partial_codes, const float *partial_scales, int num_partial_rows,
                            int num_tokens, int hidden, int num_topk, const int32_t *token_dst_row, void *out,
                            int32_t *status, void *stream);

/*
 * moe_combine_fp8_ex -- moe_combine_fp8 with tail balancing, as moe_combine_ex.
 *
 *   balance   two zeroed uint32 of device memory (8-byte aligned) or NULL.
 *             With a counter and a long enough batch (several dozen tokens
 *             per SM), the last tokens are claimed one by one by whichever
 *             SM is free first; the counter is left zeroed. Results are
 *             exactly those of moe_combine_fp8 (each token is reduced by one
 *             CTA in the same order whichever CTA it is). NULL gives exactly
 *             moe_combine_fp8.
 * Other arguments, limits and errors as moe_combine_fp8.
 */
MOE_API int moe_combine_fp8_ex(const void *partial_codes, const float *partial_scales, int num_partial_rows,
                               int num_tokens, int hidden, int num_topk, const int32_t *token_dst_row, void *out,
                               uint32_t *balance, int32_t *status, void *stream);

/*
 * Tracing -- a build option. The pages stamp their kernels' progress with the
 * device's global timer (the GEMM + all-reduce page's command stamps) and count
 * bytes in software counters (the Ascend send-ordering page); this is the
 * equivalent for these kernels. In a library compiled with -DMOE_PROFILE
 * (libmoe_get_trace.so, built beside libmoe_get.so), once moe_trace_enable has
 * been given a buffer, every warp of every kernel launched afterwards appends
 * one moe_trace_record_t when it returns (MOE_TRACE_WARPS): which kernel, CTA
 * and warp, the SM it ran on, and %globaltimer (ns) when the warp began and
 * when it returned. Thread 0 of each CTA of the cluster layout, dispatch and
 * combine kernels appends one record per phase of its own path
 * (MOE_TRACE_PHASES; warp field MOE_TRACE_PHASE + phase number, start and end
 * of the phase), listed below.
 * The default build compiles all of it out (no cost, no argument).
 *
 * Phases (thread 0's view; each ends where the next begins):
 *   MOE_TRACE_LAYOUT_CLUSTER  1 dependency wait, 2 top-k tile loaded, 3 bitmap
 *                             and expert histogram, 4 tile counts and first
 *                             cluster barrier, 5 exchange and second barrier,
 *                             6 prefixes and count writes, 7 receive rows,
 *                             8 is_token_in_rank rows (to thread 0's exit)
 *   MOE_TRACE_DISPATCH        1 set-up (launched behind this library's
 *                             layout: with the first loads and the input
 *                             rows' L2 prefetch), 2 dependency wait, 3 the
 *                             layout of a fused small batch (0 ns when not
 *                             fused), 4 the rest (to thread 0's exit)
 *   MOE_TRACE_DISPATCH_FP8_ROWS, MOE_TRACE_COMBINE
 *                             1 set-up, 2 dependency wait, 3 the rest
 */
enum {
    MOE_TRACE_LAYOUT_TILES = 1,        /* lookback tiles (cooperative or ticket) */
    MOE_TRACE_LAYOUT_DIRECT = 2,
    MOE_TRACE_LAYOUT_CLUSTER = 3,
    MOE_TRACE_LAYOUT_COUNT = 4,        /* scan mode: per-tile counts */
    MOE_TRACE_LAYOUT_SCAN = 5,         /* scan mode: per-rank scans */
    MOE_TRACE_LAYOUT_ROWS_SCAN = 6,    /* scan mode: rows */
    MOE_TRACE_EXPAND_LAYOUT = 7,
    MOE_TRACE_EXPAND_LAYOUT_CLUSTER = 8,
    MOE_TRACE_DISPATCH = 9,            /* relay pipeline (bf16, E4M3 rows, chunked E4M3, fused small batches) */
    MOE_TRACE_DISPATCH_FP8_ROWS = 10,  /* quantising row pipeline */
    MOE_TRACE_COMBINE = 11,
    MOE_TRACE_LAYOUT_ROWS = 12,        /* lookback tiles launched one after another: rows */
    MOE_TRACE_PHASE = 0x10000          /* warp field of a per-CTA phase record: MOE_TRACE_PHASE + phase */
};

/* what moe_trace_enable records (bits) */
enum { MOE_TRACE_WARPS = 1, MOE_TRACE_PHASES = 2 };

typedef struct {
    uint32_t kernel;     /* MOE_TRACE_* */
    uint32_t cta;        /* blockIdx.x */
    uint32_t warp;       /* warp index in the CTA, or MOE_TRACE_PHASE + phase */
    uint32_t sm;         /* SM the CTA ran on */
    uint64_t start_ns;   /* global timer when the warp began */
    uint64_t end_ns;     /* global timer when it returned */
} moe_trace_record_t;

/*
 * moe_trace_enable -- where the warps' records go, for the launches that follow.
 *
 *   records   device array of `capacity` records, or NULL to stop tracing.
 *   what      MOE_TRACE_WARPS (a record per warp), MOE_TRACE_PHASES (the
 *             per-CTA phase records) or both. Each warp record costs its warp
 *             one atomic at its start, which slows the latency-bound layout
 *             noticeably; phases alone cost one atomic per CTA.
 *   count     device uint32, zeroed by the caller: each record claims the slot
 *             *count (atomically incremented; a CTA's phase records claim
 *             consecutive slots at once); records at or beyond `capacity`
 *             are dropped, but still counted, so *count after the stream has
 *             synchronised tells how many there were.
 * Each launch keeps the buffer it was given at launch: a CUDA graph captured
 * while tracing is on writes to it on every replay, so the buffer and counter
 * must outlive such a graph.
 * Process-wide setting (all devices, all streams); not for concurrent use
 * with launches on other host threads. MOE_OK in a -DMOE_PROFILE build;
 * MOE_ERR_INVALID_ARG in the default build (nothing is recorded) or, with
 * non-null records, for a negative capacity, a null or misaligned count, or
 * `what` empty or with other bits.
 */
MOE_API int moe_trace_enable(moe_trace_record_t *records, int capacity, uint32_t *count, int what);

/* Size of the library's own layout scratch (bytes), used by moe_get_layout_noalloc. */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)

/*
 * moe_get_layout_noalloc -- moe_get_layout for callers that cannot allocate
 * device memory (the pages have no counterpart; this is a library addition).
 *
 * Some callers cannot call cudaMalloc: a plugin running inside a host
 * framework that owns every device allocation and hands out no workspace, or
 * a latency-critical loop where an allocation (which may synchronise the
 * device) is not acceptable. This entry point takes the same inputs and
 * outputs as moe_get_layout but no workspace: it uses a scratch array of
 * MOE_NOALLOC_SCRATCH_BYTES that the library keeps in device memory (held by
 * every GPU that loads the library until the process exits). It allocates
 * nothing and calls no allocating routine.
 *
 *   - The first call on a device looks up the scratch's device address with
 *     that device current; make that first call before any stream capture.
 *     The address is kept for the life of the process: after a
 *     cudaDeviceReset (which unloads the library's device code) it is stale,
 *     so do not call this entry point on that device again.
 *   - Sizes whose workspace (moe_get_layout_workspace_size) exceeds
 *     MOE_NOALLOC_SCRATCH_BYTES return MOE_ERR_WORKSPACE and launch nothing.
 *   - Every call shares the one scratch array, which keeps the previous
 *     call's contents; each call clears what it uses on its own stream.
 *     Calls whose executions overlap on the GPU (e.g. on two streams without
 *     ordering between them) race on the scratch and give wrong results.
 * Outputs, status word and errors are as for moe_get_layout.
 */
MOE_API int moe_get_layout_noalloc(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                                   int num_ranks, moe_layout_t layout, int32_t *status, void *stream);

/*
 * moe_combine_ex -- moe_combine with the two combine options of the pages.
 *
 *   row_weights           [num_partial_rows] fp32 or NULL. When given, each term
 *                         is weighted: acc = fma(row_weights[row], float(partial[row]),
 *                         acc) (one rounding per term), same order and start as
 *                         moe_combine; NULL gives exactly moe_combine.
 *   recv_topk_weights     [num_partial_rows, k] fp32 or NULL (e.g. the dispatch's
 *                         recv_topk_weights) and
 *   combined_topk_weights [T, k] fp32 output or NULL: the received top-k weights
 *                         reduced back to the tokens (the combine also returns the
 *                         weights that travelled with the rows, section 3.5 /
 *                         the Ascend page's FP32 weights next to the BF16 hidden):
 *                         combined[t, j] = sum over the rows of t in ascending rank
 *                         order of recv_topk_weights[row, j], fp32 from +0.0f.
 *   balance               NULL, or a combine balance counter: 2 uint32 of device
 *                         memory, 8-byte aligned, zero before the first call that
 *                         uses them; every call leaves them zero again (the last
 *                         CTA to finish clears them, also after a timeout). With it,
 *                         70% of the tokens are split statically over the CTAs and
 *                         the rest are claimed one by one, so that CTAs on SMs with
 *                         more bandwidth take more of them (SMs do not all get the
 *                         same HBM bandwidth; at DSv3 they finished 46-57 us apart
 *                         without it). Batches of fewer than 8 tokens per SM ignore
 *                         it. Results do not depend on it. Two calls
 *                         that use the same counter must not run at the same time on
 *                         the GPU (same stream, or ordered streams).
 *                         Misaligned: MOE_ERR_MISALIGNED. NULL: static split only.
 * Other arguments, errors and limits as for moe_combine.
 */
MOE_API int moe_combine_ex(const void *partial, int num_partial_rows, int num_tokens, int hidden, int num_topk,
                           const int32_t *token_dst_row, const float *row_weights,
                           const float *recv_topk_weights, float *combined_topk_weights, void *out,
                           uint32_t *balance, int32_t *status, void *stream);

/* Human-readable name of a moe_status_t value (static string). */
MOE_API const char *moe_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
MOE_API int moe_get_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GET_H */
