// moe_api.cu -- the extern "C" entry points of libmoe_get.so.
//
// Every entry point validates its arguments on the host before it touches
// CUDA, so argument errors come back as return codes without a launch (and
// can be checked on a machine without a GPU). Then it hands a plain launch
// description to the kernel launcher of its step.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <utility>

#include <cuda_runtime.h>

#include "../../include/moe_get.h"
#include "moe_internal.h"

namespace moe {

// ------------------------------------------------------------------ device facts

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<long long> g_smem_sm[kMaxDevices];
std::atomic<long long> g_smem_optin[kMaxDevices];
std::atomic<long long> g_l2[kMaxDevices];

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return 0;
    return d;
}

int query_attr(cudaDeviceAttr attr, int dev) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess) return 0;
    return v;
}
}  // namespace

int device_sm_count() {
    const int d = current_device();
    int v = g_sm_count[d].load(std::memory_order_relaxed);
    if (v == 0) {
        v = query_attr(cudaDevAttrMultiProcessorCount, d);
        if (v <= 0) v = 1;
        g_sm_count[d].store(v, std::memory_order_relaxed);
    }
    return v;
}

size_t device_smem_per_sm() {
    const int d = current_device();
    long long v = g_smem_sm[d].load(std::memory_order_relaxed);
    if (v == 0) {
        v = query_attr(cudaDevAttrMaxSharedMemoryPerMultiprocessor, d);
        if (v <= 0) v = 48 * 1024;
        g_smem_sm[d].store(v, std::memory_order_relaxed);
    }
    return (size_t)v;
}

size_t device_smem_optin() {
    const int d = current_device();
    long long v = g_smem_optin[d].load(std::memory_order_relaxed);
    if (v == 0) {
        v = query_attr(cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
        if (v <= 0) v = 48 * 1024;
        g_smem_optin[d].store(v, std::memory_order_relaxed);
    }
    return (size_t)v;
}

size_t device_l2_bytes() {
    const int d = current_device();
    long long v = g_l2[d].load(std::memory_order_relaxed);
    if (v == 0) {
        v = query_attr(cudaDevAttrL2CacheSize, d);
        if (v <= 0) v = 1;
        g_l2[d].store(v, std::memory_order_relaxed);
    }
    return (size_t)v;
}

int ensure_dynamic_smem(const void *kernel, size_t bytes) {
    static std::mutex mu;
    static std::unordered_map<const void *, size_t> done[kMaxDevices];
    const int d = current_device();
    std::lock_guard<std::mutex> lock(mu);
    size_t &cur = done[d][kernel];
    if (bytes <= cur) return MOE_OK;
    // set even below 48 KB: the default limit covers dynamic plus static shared
    // memory, so a kernel with static shared memory needs it raised earlier
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return MOE_ERR_CUDA;
    cur = bytes;
    return MOE_OK;
}

namespace {
std::atomic<moe_trace_record_t *> g_trace_rec{nullptr};
std::atomic<uint32_t *> g_trace_count{nullptr};
std::atomic<int> g_trace_cap{0};
std::atomic<int> g_trace_what{0};
}  // namespace

TraceArgs trace_args() {
    TraceArgs t{g_trace_rec.load(std::memory_order_acquire), g_trace_count.load(std::memory_order_acquire),
                g_trace_cap.load(std::memory_order_acquire), g_trace_what.load(std::memory_order_acquire)};
    if (t.rec == nullptr || t.count == nullptr || t.what == 0) t = TraceArgs{nullptr, nullptr, 0, 0};
    return t;
}

const Tuning &tuning() {
    // Compile-time settings (moe_internal.h): nothing read from the environment,
    // so every call takes the configuration the parity tests ran.
    static const Tuning t = [] {
        Tuning x;
        x.dispatch_warps = MOE_TUNE_DISPATCH_WARPS;
        x.dispatch_stages = MOE_TUNE_DISPATCH_STAGES;
        x.ld_dispatch_warps = MOE_TUNE_LD_DISPATCH_WARPS;
        x.ld_dispatch_stages = MOE_TUNE_LD_DISPATCH_STAGES;
        x.dispatch_chunk = MOE_TUNE_DISPATCH_CHUNK;
        x.dispatch_smem = MOE_TUNE_DISPATCH_SMEM;
        x.combine_warps = MOE_TUNE_COMBINE_WARPS;
        x.combine_chunk = MOE_TUNE_COMBINE_CHUNK;
        x.combine_ring_bytes = MOE_TUNE_COMBINE_RING_BYTES;
        x.combine_fp8_warps = MOE_TUNE_COMBINE_FP8_WARPS;
        x.combine_fp8_pool = MOE_TUNE_COMBINE_FP8_POOL;
        x.combine_fp8_pool_min_tokens = MOE_TUNE_COMBINE_FP8_POOL_MIN_TOKENS;
        x.overlap = MOE_TUNE_OVERLAP;
        x.dispatch_pool = MOE_TUNE_DISPATCH_POOL;
        x.combine_pool = MOE_TUNE_COMBINE_POOL;
        x.combine_prefetch = MOE_TUNE_COMBINE_PREFETCH;
        x.layout_cluster = MOE_TUNE_LAYOUT_CLUSTER;
        x.layout_scan = MOE_TUNE_LAYOUT_SCAN;
        x.fp8_rows = MOE_TUNE_FP8_ROWS;
        x.fp8_in_slots = MOE_TUNE_FP8_IN_SLOTS;
        x.fp8_quant_warps = MOE_TUNE_FP8_QUANT_WARPS;
        x.fp8_rows_pool = MOE_TUNE_FP8_ROWS_POOL;
        x.fp8_rows_pool_min_rows = MOE_TUNE_FP8_ROWS_POOL_MIN_ROWS;
        x.ctas_per_sm = MOE_TUNE_CTAS_PER_SM;
        x.l2_hints = MOE_TUNE_L2_HINTS & 3;
        x.spread_small = MOE_TUNE_SPREAD_SMALL;
        x.fused_small = MOE_TUNE_FUSED_SMALL;
        x.fused_min_warps = MOE_TUNE_FUSED_MIN_WARPS;
        x.dispatch_prefetch = MOE_TUNE_DISPATCH_PREFETCH;
        x.dispatch_prefetch_keep = MOE_TUNE_DISPATCH_PREFETCH_KEEP;
        x.dispatch_prefetch_always = MOE_TUNE_DISPATCH_PREFETCH_ALWAYS;
        x.dispatch_prefetch_l2_pct = MOE_TUNE_DISPATCH_PREFETCH_L2_PCT;
        x.dispatch_prefetch_l2_pct_alone = MOE_TUNE_DISPATCH_PREFETCH_L2_PCT_ALONE;
        return x;
    }();
    return t;
}

}  // namespace moe

// ------------------------------------------------------------------ validation helpers

namespace {

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool shape_ok(int T, int k, int E, int R) {
    if (T < 0 || k < 1 || k > MOE_MAX_TOPK) return false;
    if (R < 1 || R > MOE_MAX_RANKS || E < 1 || E > MOE_MAX_EXPERTS || E % R != 0) return false;
    if ((int64_t)T * k >= (int64_t)1 << 31) return false;
    return true;
}

}  // namespace

// ------------------------------------------------------------------ shared layout checks

namespace moe {

int layout_check_args(const int64_t *topk_idx, int T, int k, int E, int R, const moe_layout_t &o,
                      const int32_t *status) {
    if (!shape_ok(T, k, E, R)) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * R >= (int64_t)1 << 40) return MOE_ERR_INVALID_ARG;
    if (!status || !o.num_tokens_per_rank || !o.num_tokens_per_expert || !o.rank_prefix || !o.expert_prefix)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !o.is_token_in_rank || !o.token_dst_row)) return MOE_ERR_INVALID_ARG;
    if (!aligned(status, 4) || !aligned(o.num_tokens_per_rank, 4) || !aligned(o.num_tokens_per_expert, 4) ||
        !aligned(o.rank_prefix, 4) || !aligned(o.expert_prefix, 4))
        return MOE_ERR_MISALIGNED;
    if (T > 0 && (!aligned(topk_idx, 8) || !aligned(o.token_dst_row, 4) || !aligned(o.is_token_in_rank, 4)))
        return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

int layout_prepare(const int64_t *topk_idx, int T, int k, int E, int R, moe_layout_t o, void *workspace,
                   size_t workspace_bytes, int32_t *status, void *stream, int64_t timeout_ns, int unpublished_tile,
                   LayoutLaunch &L, bool no_cluster) {
    const int rc = layout_check_args(topk_idx, T, k, E, R, o, status);
    if (rc != MOE_OK) return rc;
    if (T > 0) {
        if (!workspace) return MOE_ERR_INVALID_ARG;
        if (!aligned(workspace, 16)) return MOE_ERR_MISALIGNED;
        if (workspace_bytes < layout_workspace_bytes(T, E, R)) return MOE_ERR_WORKSPACE;
    }
    L = LayoutLaunch{};
    L.topk_idx = topk_idx;
    L.num_tokens = T;
    L.num_topk = k;
    L.num_experts = E;
    L.num_ranks = R;
    L.out = o;
    L.workspace = workspace;
    L.status = status;
    L.stream = stream;
    L.timeout_ns = timeout_ns;
    L.unpublished_tile = unpublished_tile;
    L.no_cluster = no_cluster || unpublished_tile >= 0;
    return MOE_OK;
}

}  // namespace moe

// ------------------------------------------------------------------ C ABI

extern "C" {

MOE_API int moe_get_version(void) { return 100; }

MOE_API int moe_trace_enable(moe_trace_record_t *records, int capacity, uint32_t *count, int what) {
#ifdef MOE_PROFILE
    if (records != nullptr && (capacity < 0 || count == nullptr || !aligned(records, 8) || !aligned(count, 4) ||
                               what == 0 || (what & ~(MOE_TRACE_WARPS | MOE_TRACE_PHASES)) != 0))
        return MOE_ERR_INVALID_ARG;
    moe::g_trace_what.store(records ? what : 0, std::memory_order_release);
    moe::g_trace_cap.store(records ? capacity : 0, std::memory_order_release);
    moe::g_trace_count.store(records ? count : nullptr, std::memory_order_release);
    moe::g_trace_rec.store(records, std::memory_order_release);
    return MOE_OK;
#else
    (void)records;
    (void)capacity;
    (void)count;
    (void)what;
    return MOE_ERR_INVALID_ARG;   // a build without MOE_PROFILE records nothing
#endif
}

MOE_API const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
        case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY";
        case MOE_ERR_BAD_TOPK: return "MOE_ERR_BAD_TOPK";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        default: return "MOE_ERR_UNKNOWN";
    }
}

MOE_API size_t moe_get_layout_workspace_size(int num_tokens, int num_experts, int num_ranks) {
    if (!shape_ok(num_tokens, 1, num_experts, num_ranks)) return 0;
    return moe::layout_workspace_bytes(num_tokens, num_experts, num_ranks);
}

// mode: 0 by size, 1 never the cluster mode, 2 only the lookback modes
static int layout_common(const int64_t *topk_idx, int T, int k, int E, int R, moe_layout_t o, void *workspace,
                         size_t workspace_bytes, int32_t *status, void *stream, int64_t timeout_ns,
                         int unpublished_tile, int mode = 0) {
    moe::LayoutLaunch L;
    const int rc = moe::layout_prepare(topk_idx, T, k, E, R, o, workspace, workspace_bytes, status, stream,
                                       timeout_ns, unpublished_tile, L, mode != 0);
    L.lookback_only = mode == 2;
    return rc != MOE_OK ? rc : moe::launch_layout(L);
}

MOE_API int moe_get_layout(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts, int num_ranks,
                           moe_layout_t layout, void *workspace, size_t workspace_bytes, int32_t *status,
                           void *stream) {
    return layout_common(topk_idx, num_tokens, num_topk, num_experts, num_ranks, layout, workspace,
                         workspace_bytes, status, stream, 0, -1);
}

MOE_API int moe_get_layout_ex(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                              int num_ranks, moe_layout_t layout, void *workspace, size_t workspace_bytes,
                              int32_t *status, void *stream, const moe_layout_options_t *options) {
    int64_t timeout = 0;
    int unpublished = -1;
    int mode = 0;
    if (options) {
        timeout = options->wait_timeout_ns;
        unpublished = options->test_unpublished_tile;
        if (options->layout_mode < 0 || options->layout_mode > 2) return MOE_ERR_INVALID_ARG;
        mode = options->layout_mode;
    }
    return layout_common(topk_idx, num_tokens, num_topk, num_experts, num_ranks, layout, workspace,
                         workspace_bytes, status, stream, timeout, unpublished, mode);
}

MOE_API size_t moe_get_expand_layout_workspace_size(int num_tokens, int num_experts) {
    if (!shape_ok(num_tokens, 1, num_experts, 1)) return 0;
    return moe::expand_workspace_bytes(num_tokens, num_experts);
}

MOE_API int moe_get_expand_layout(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                                  const int32_t *expert_prefix, int32_t *token_expert_row, void *workspace,
                                  size_t workspace_bytes, int32_t *status, void *stream,
                                  const moe_layout_options_t *options) {
    const int T = num_tokens, k = num_topk, E = num_experts;
    if (!shape_ok(T, k, E, 1)) return MOE_ERR_INVALID_ARG;
    if (!status) return MOE_ERR_INVALID_ARG;
    if (!aligned(status, 4)) return MOE_ERR_MISALIGNED;
    if (T > 0) {
        if (!topk_idx || !expert_prefix || !token_expert_row || !workspace) return MOE_ERR_INVALID_ARG;
        if (!aligned(topk_idx, 8) || !aligned(expert_prefix, 4) || !aligned(token_expert_row, 4) ||
            !aligned(workspace, 16))
            return MOE_ERR_MISALIGNED;
        if (workspace_bytes < moe::expand_workspace_bytes(T, E)) return MOE_ERR_WORKSPACE;
    }
    moe::ExpandLaunch L;
    L.topk_idx = topk_idx;
    L.num_tokens = T;
    L.num_topk = k;
    L.num_experts = E;
    L.expert_prefix = expert_prefix;
    L.token_expert_row = token_expert_row;
    L.workspace = workspace;
    L.status = status;
    L.stream = stream;
    L.timeout_ns = options ? options->wait_timeout_ns : 0;
    L.unpublished_tile = options ? options->test_unpublished_tile : -1;
    if (options && options->layout_mode != 0 && options->layout_mode != 1) return MOE_ERR_INVALID_ARG;
    L.no_cluster = options && options->layout_mode == 1;
    return moe::launch_expand_layout(L);
}

// Validation of a dispatch; `need_rows` is false when the receive rows come from
// the same call (moe_layout_dispatch).
static int dispatch_prepare(const void *x, int num_tokens, int hidden, const int64_t *topk_idx,
                            const float *topk_weights, int num_topk, int num_experts, int num_ranks,
                            const int32_t *token_dst_row, int recv_capacity, int mode, void *recv_x,
                            float *recv_x_scales, int64_t *recv_topk_idx, float *recv_topk_weights,
                            int32_t *recv_src_idx, float *x_scales, int32_t *status, void *stream,
                            moe::DispatchLaunch &L) {
    const int T = num_tokens, H = hidden;
    if (!shape_ok(T, num_topk, num_experts, num_ranks)) return MOE_ERR_INVALID_ARG;
    const bool expand = (mode & MOE_DISPATCH_EXPAND) != 0;
    mode &= ~MOE_DISPATCH_EXPAND;
    if (mode != MOE_DISPATCH_BF16 && mode != MOE_DISPATCH_QUANTIZE_FP8 && mode != MOE_DISPATCH_FP8)
        return MOE_ERR_INVALID_ARG;
    const bool fp8_out = mode != MOE_DISPATCH_BF16;
    if (recv_capacity < 0 || H < 8 || H % 8 != 0 || (fp8_out && H % 128 != 0)) return MOE_ERR_INVALID_ARG;
    if (H > (1 << 24)) return MOE_ERR_INVALID_ARG;
    if (!status) return MOE_ERR_INVALID_ARG;
    if (T > 0) {
        if (!x || !topk_idx || !token_dst_row || (recv_capacity > 0 && !recv_x)) return MOE_ERR_INVALID_ARG;
        if (fp8_out && recv_capacity > 0 && !recv_x_scales) return MOE_ERR_INVALID_ARG;
        if (mode == MOE_DISPATCH_FP8 && !x_scales) return MOE_ERR_INVALID_ARG;
        if (!aligned(x, 16) || (recv_x && !aligned(recv_x, 16)) || !aligned(topk_idx, 8) ||
            !aligned(token_dst_row, 4) || !aligned(status, 4) || (topk_weights && !aligned(topk_weights, 4)) ||
            (recv_x_scales && !aligned(recv_x_scales, 4)) || (recv_topk_idx && !aligned(recv_topk_idx, 8)) ||
            (recv_topk_weights && !aligned(recv_topk_weights, 4)) || (recv_src_idx && !aligned(recv_src_idx, 4)) ||
            (x_scales && !aligned(x_scales, 4)))
            return MOE_ERR_MISALIGNED;
    }
    L.x = x;
    L.num_tokens = T;
    L.hidden = H;
    L.topk_idx = topk_idx;
    L.topk_weights = topk_weights;
    L.num_topk = num_topk;
    L.num_experts = num_experts;
    L.num_ranks = num_ranks;
    L.token_dst_row = token_dst_row;
    L.recv_capacity = recv_capacity;
    L.mode = mode;
    L.expand = expand;
    L.recv_x = recv_x;
    L.recv_x_scales = fp8_out ? recv_x_scales : nullptr;
    L.recv_topk_idx = recv_topk_idx;
    L.recv_topk_weights = recv_topk_weights;
    L.recv_src_idx = recv_src_idx;
    L.x_scales = fp8_out ? x_scales : nullptr;
    L.status = status;
    L.stream = stream;
    return MOE_OK;
}

MOE_API int moe_dispatch(const void *x, int num_tokens, int hidden, const int64_t *topk_idx,
                         const float *topk_weights, int num_topk, int num_experts, int num_ranks,
                         const int32_t *token_dst_row, int recv_capacity, int mode, void *recv_x,
                         float *recv_x_scales, int64_t *recv_topk_idx, float *recv_topk_weights,
                         int32_t *recv_src_idx, float *x_scales, int32_t *status, void *stream) {
    moe::DispatchLaunch L;
    const int rc = dispatch_prepare(x, num_tokens, hidden, topk_idx, topk_weights, num_topk, num_experts, num_ranks,
                                    token_dst_row, recv_capacity, mode, recv_x, recv_x_scales, recv_topk_idx,
                                    recv_topk_weights, recv_src_idx, x_scales, status, stream, L);
    return rc != MOE_OK ? rc : moe::launch_dispatch(L);
}

MOE_API int moe_dispatch_ex(const void *x, int num_tokens, int hidden, const int64_t *topk_idx,
                            const float *topk_weights, int num_topk, int num_experts, int num_ranks,
                            const int32_t *token_dst_row, int recv_capacity, int mode, void *recv_x,
                            float *recv_x_scales, int64_t *recv_topk_idx, float *recv_topk_weights,
                            int32_t *recv_src_idx, float *x_scales, uint32_t *balance, int32_t *status,
                            void *stream) {
    if (!aligned(balance, 8)) return MOE_ERR_MISALIGNED;
    moe::DispatchLaunch L;
    const int rc = dispatch_prepare(x, num_tokens, hidden, topk_idx, topk_weights, num_topk, num_experts, num_ranks,
                                    token_dst_row, recv_capacity, mode, recv_x, recv_x_scales, recv_topk_idx,
                                    recv_topk_weights, recv_src_idx, x_scales, status, stream, L);
    if (rc != MOE_OK) return rc;
    L.pool = balance;
    return moe::launch_dispatch(L);
}

MOE_API int moe_layout_dispatch(const void *x, int num_tokens, int hidden, const int64_t *topk_idx,
                                const float *topk_weights, int num_topk, int num_experts, int num_ranks,
                                moe_layout_t layout, void *workspace, size_t workspace_bytes, int recv_capacity,
                                int mode, void *recv_x, float *recv_x_scales, int64_t *recv_topk_idx,
                                float *recv_topk_weights, int32_t *recv_src_idx, float *x_scales, int32_t *status,
                                void *stream) {
    if (mode & MOE_DISPATCH_EXPAND) return MOE_ERR_INVALID_ARG;
    moe::LayoutLaunch Ll;
    int rc = moe::layout_prepare(topk_idx, num_tokens, num_topk, num_experts, num_ranks, layout, workspace,
                                 workspace_bytes, status, stream, 0, -1, Ll, false);
    if (rc != MOE_OK) return rc;
    moe::DispatchLaunch L;
    rc = dispatch_prepare(x, num_tokens, hidden, topk_idx, topk_weights, num_topk, num_experts, num_ranks,
                          layout.token_dst_row, recv_capacity, mode, recv_x, recv_x_scales, recv_topk_idx,
                          recv_topk_weights, recv_src_idx, x_scales, status, stream, L);
    return rc != MOE_OK ? rc : moe::launch_layout_dispatch(Ll, L);
}

static int combine_common(const void *partial, int num_partial_rows, int num_tokens, int hidden, int num_topk,
                          const int32_t *token_dst_row, const float *row_weights, const float *recv_topk_weights,
                          float *combined_topk_weights, void *out, uint32_t *balance, int32_t *status,
                          void *stream) {
    const int T = num_tokens, H = hidden;
    if (T < 0 || num_topk < 1 || num_topk > MOE_MAX_TOPK || num_partial_rows < 0) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H % 8 != 0 || H > (1 << 24) || (int64_t)T * num_topk >= (int64_t)1 << 31) return MOE_ERR_INVALID_ARG;
    if (!status) return MOE_ERR_INVALID_ARG;
    if ((recv_topk_weights == nullptr) != (combined_topk_weights == nullptr)) return MOE_ERR_INVALID_ARG;
    if (T > 0) {
        if (!token_dst_row || !out || (num_partial_rows > 0 && !partial)) return MOE_ERR_INVALID_ARG;
        if ((partial && !aligned(partial, 16)) || !aligned(out, 16) || !aligned(token_dst_row, 4) ||
            !aligned(status, 4) || !aligned(row_weights, 4) || !aligned(recv_topk_weights, 4) ||
            !aligned(combined_topk_weights, 4))
            return MOE_ERR_MISALIGNED;
    }
    if (!aligned(balance, 8)) return MOE_ERR_MISALIGNED;
    moe::CombineLaunch L;
    L.balance = balance;
    L.partial = partial;
    L.num_partial_rows = num_partial_rows;
    L.num_tokens = T;
    L.hidden = H;
    L.num_topk = num_topk;
    L.token_dst_row = token_dst_row;
    L.row_weights = row_weights;
    L.recv_topk_weights = recv_topk_weights;
    L.combined_topk_weights = combined_topk_weights;
    L.out = out;
    L.status = status;
    L.stream = stream;
    return moe::launch_combine(L);
}

MOE_API int moe_combine(const void *partial, int num_partial_rows, int num_tokens, int hidden, int num_topk,
                        const int32_t *token_dst_row, void *out, int32_t *status, void *stream) {
    return combine_common(partial, num_partial_rows, num_tokens, hidden, num_topk, token_dst_row, nullptr, nullptr,
                          nullptr, out, nullptr, status, stream);
}

MOE_API int moe_combine_ex(const void *partial, int num_partial_rows, int num_tokens, int hidden, int num_topk,
                           const int32_t *token_dst_row, const float *row_weights, const float *recv_topk_weights,
                           float *combined_topk_weights, void *out, uint32_t *balance, int32_t *status,
                           void *stream) {
    return combine_common(partial, num_partial_rows, num_tokens, hidden, num_topk, token_dst_row, row_weights,
                          recv_topk_weights, combined_topk_weights, out, balance, status, stream);
}

static int combine_fp8_common(const void *partial_codes, const float *partial_scales, int num_partial_rows,
                              int num_tokens, int hidden, int num_topk, const int32_t *token_dst_row, void *out,
                              uint32_t *balance, int32_t *status, void *stream) {
    const int T = num_tokens, H = hidden;
    if (T < 0 || num_topk < 1 || num_topk > MOE_MAX_TOPK || num_partial_rows < 0) return MOE_ERR_INVALID_ARG;
    if (H < 512 || H % 512 != 0 || H > (1 << 24) || (int64_t)T * num_topk >= (int64_t)1 << 31) return MOE_ERR_INVALID_ARG;
    if (!status) return MOE_ERR_INVALID_ARG;
    if (T > 0) {
        if (!token_dst_row || !out || (num_partial_rows > 0 && (!partial_codes || !partial_scales)))
            return MOE_ERR_INVALID_ARG;
        if ((partial_codes && !aligned(partial_codes, 16)) || (partial_scales && !aligned(partial_scales, 16)) ||
            !aligned(out, 16) || !aligned(token_dst_row, 4) || !aligned(status, 4))
            return MOE_ERR_MISALIGNED;
    }
    if (!aligned(balance, 8)) return MOE_ERR_MISALIGNED;
    moe::CombineLaunch L;
    L.partial = partial_codes;
    L.fp8 = true;
    L.partial_scales = partial_scales;
    L.num_partial_rows = num_partial_rows;
    L.num_tokens = T;
    L.hidden = H;
    L.num_topk = num_topk;
    L.token_dst_row = token_dst_row;
    L.row_weights = nullptr;
    L.recv_topk_weights = nullptr;
    L.combined_topk_weights = nullptr;
    L.out = out;
    L.status = status;
    L.stream = stream;
    L.balance = balance;
    return moe::launch_combine(L);
}

MOE_API int moe_combine_fp8(const void *partial_codes, const float *partial_scales, int num_partial_rows,
                            int num_tokens, int hidden, int num_topk, const int32_t *token_dst_row, void *out,
                            int32_t *status, void *stream) {
    return combine_fp8_common(partial_codes, partial_scales, num_partial_rows, num_tokens, hidden, num_topk,
                              token_dst_row, out, nullptr, status, stream);
}

MOE_API int moe_combine_fp8_ex(const void *partial_codes, const float *partial_scales, int num_partial_rows,
                               int num_tokens, int hidden, int num_topk, const int32_t *token_dst_row, void *out,
                               uint32_t *balance, int32_t *status, void *stream) {
    return combine_fp8_common(partial_codes, partial_scales, num_partial_rows, num_tokens, hidden, num_topk,
                              token_dst_row, out, balance, status, stream);
}

}  // extern "C"
