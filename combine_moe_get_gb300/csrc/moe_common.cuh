// moe_common.cuh -- device helpers shared by the layout, dispatch and combine
// kernels: status reporting, bounded waits, mbarriers and 1-D bulk copies
// (cp.async.bulk, the non-tensor TMA path of sm_90+/sm_100+), written as
// inline PTX for sm_103a.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "../../include/moe_get.h"
#include "moe_internal.h"

namespace moe {

// Default bound on any spin or barrier wait inside a kernel.
constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // 1 s

// ------------------------------------------------------------------ launch overlap
//
// Programmatic dependent launch (PTX griddepcontrol, sm_90+). A grid launched
// with programmatic stream serialization may be scheduled while the grid
// before it on the stream is still running. Every kernel here calls
// grid_dependency_wait() before its first global memory access, read or
// write: it returns once the previous grid has completed and its writes are
// visible, so reads see the producer's results and writes cannot overtake
// the previous grid's reads. Two exceptions read before it, and neither can
// change a result: L2 prefetches (the combine's first rows, and the address
// lists they come from, read past L1), and the dispatch's first input-row
// loads when it is launched right behind this library's own layout, which
// does not write the input rows (a MOE_PROFILE build's trace counter is
// claimed there too). grid_launch_dependents() then lets the next
// grid's CTAs be placed as this grid's CTAs retire, so that its launch and
// prologue (barrier set-up) overlap this grid's tail. Only the dispatch and
// combine kernels call it: a layout kernel leaves the trigger to its exit,
// because dispatch CTAs placed beside a running layout and waiting there
// slowed the layout down. In a grid launched without the attribute both are
// no-ops.

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kernel`, allowed to overlap the previous grid on the stream when
// `overlap` is set (cudaLaunchAttributeProgrammaticStreamSerialization).
template <typename... Params, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 bool overlap, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------ index arithmetic

// u / n for a non-negative unit counter and n >= 1: no division when n == 1
// and 32-bit division while u fits (a 64-bit division is a long dependent
// instruction sequence, which matters in a single warp's issue loop).
__device__ __forceinline__ int64_t div_count(int64_t u, int n) {
    if (n == 1) return u;
    return u <= 0x7fffffff ? (int64_t)((uint32_t)u / (uint32_t)n) : u / n;
}

// ------------------------------------------------------------------ status

// First data error wins; later ones are dropped.
__device__ __forceinline__ void report(int32_t *status, int code) {
    if (status != nullptr) atomicCAS(reinterpret_cast<int *>(status), 0, code);
}

// In-place exclusive scan of n int32 in shared memory by one warp (all 32
// lanes call it); v[n] receives the total.
__device__ __forceinline__ void warp_exclusive_scan(int32_t *v, int n, int lane) {
    const int per = (n + 31) / 32;
    const int lo = min(n, lane * per), hi = min(n, lo + per);
    int32_t local = 0;
    for (int i = lo; i < hi; ++i) local += v[i];
    int32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int32_t run = incl - local;
    for (int i = lo; i < hi; ++i) {
        const int32_t x = v[i];
        v[i] = run;
        run += x;
    }
    if (lane == 31) v[n] = incl;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ tracing (MOE_PROFILE builds)

// Declared first in a kernel: in a MOE_PROFILE build, lane 0 of each warp stamps
// the global timer here and, when the warp returns (whichever return it takes),
// appends one moe_trace_record_t to the buffer given to moe_trace_enable. In
// the default build it is empty and compiles to nothing.
struct WarpTrace {
#ifdef MOE_PROFILE
    TraceArgs t;
    uint32_t kernel;
    uint32_t i = 0;      // the record's slot, claimed when the warp starts (the
    uint64_t t0 = 0;     // atomic's round trip then overlaps the warp's work)
    __device__ __forceinline__ WarpTrace(const TraceArgs &ta, uint32_t k) : t(ta), kernel(k) {
        if (!(t.what & MOE_TRACE_WARPS)) t.rec = nullptr;
        if (t.rec != nullptr && (threadIdx.x & 31) == 0) {
            t0 = globaltimer_ns();
            i = atomicAdd(t.count, 1u);
        }
    }
    __device__ __forceinline__ ~WarpTrace() {
        if (t.rec == nullptr || (threadIdx.x & 31) != 0) return;
        if (i >= (uint32_t)t.cap) return;
        uint32_t sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        moe_trace_record_t r;
        r.kernel = kernel;
        r.cta = blockIdx.x;
        r.warp = threadIdx.x >> 5;
        r.sm = sm;
        r.start_ns = t0;
        r.end_ns = globaltimer_ns();
        t.rec[i] = r;
    }
#else
    __device__ __forceinline__ WarpTrace(const TraceArgs &, uint32_t) {}
#endif
};

// Per-CTA phase records (MOE_PROFILE builds): MOE_PHASES(kernel, n), declared
// after the WarpTrace of a kernel whose arguments are `a`, makes thread 0 stamp
// the global timer at the kernel's start and claim n record slots at once;
// MOE_PHASE(p) (1 <= p < n) ends phase p; thread 0's exit ends phase n. At
// exit thread 0 writes the n phase intervals. In the default build both
// macros are empty.
#ifdef MOE_PROFILE
constexpr int kMaxPhases = 8;
struct CtaPhases {
    TraceArgs t;
    uint32_t kernel, n, base = 0;
    uint64_t *v;   // v[0]: start; v[p]: end of phase p (0: not reached)
    __device__ __forceinline__ CtaPhases(const TraceArgs &ta, uint32_t k, uint32_t np, uint64_t *sv)
        : t(ta), kernel(k), n(np), v(sv) {
        if (!(t.what & MOE_TRACE_PHASES)) t.rec = nullptr;
        if (t.rec != nullptr && threadIdx.x == 0) {
            v[0] = globaltimer_ns();
            for (uint32_t i = 1; i <= n; ++i) v[i] = 0;
            base = atomicAdd(t.count, n);
        }
    }
    __device__ __forceinline__ void mark(uint32_t p) {
        if (t.rec != nullptr && threadIdx.x == 0 && p < n) v[p] = globaltimer_ns();
    }
    __device__ __forceinline__ ~CtaPhases() {
        if (t.rec == nullptr || threadIdx.x != 0) return;
        v[n] = globaltimer_ns();
        uint32_t sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        uint64_t prev = v[0];
        for (uint32_t p = 1; p <= n; ++p) {
            const uint64_t end = v[p] != 0 ? v[p] : prev;   // a phase not reached lasts 0 ns
            if (base + p - 1 < (uint32_t)t.cap) {
                moe_trace_record_t r;
                r.kernel = kernel;
                r.cta = blockIdx.x;
                r.warp = MOE_TRACE_PHASE + p;
                r.sm = sm;
                r.start_ns = prev;
                r.end_ns = end;
                t.rec[base + p - 1] = r;
            }
            prev = end;
        }
    }
};
#define MOE_PHASES(kernel_id, nphases)                                                          \
    static_assert((nphases) >= 1 && (nphases) <= kMaxPhases, "phase count");                   \
    __shared__ uint64_t moe_phase_stamps_[kMaxPhases + 1];                                       \
    CtaPhases moe_phases_(a.trace, (kernel_id), (nphases), moe_phase_stamps_)
#define MOE_PHASE(p) moe_phases_.mark(p)
#else
#define MOE_PHASES(kernel_id, nphases) static_assert((nphases) >= 1, "phase count")
#define MOE_PHASE(p) ((void)0)
#endif

// ------------------------------------------------------------------ shared-memory addresses

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make initialised barriers visible to the async (TMA) proxy; follow with a CTA barrier.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after `timeout_ns`
// (measured on %globaltimer from the first failed poll). Returns false on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = globaltimer_ns() + timeout_ns;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() > deadline) return false;
    }
}

// ------------------------------------------------------------------ L2 cache policies

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Bring `bytes` (a multiple of 16, 16-byte aligned source) of global memory
// into L2 with a cache policy; nothing is waited for or written.
__device__ __forceinline__ void bulk_prefetch_l2(const void *gmem_src, uint32_t bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;"
                 ::"l"(gmem_src), "r"(bytes), "l"(policy) : "memory");
}

// Give the 128-byte L2 line at `p` (128-byte aligned) normal eviction
// priority again, e.g. after an evict-last prefetch has been consumed.
__device__ __forceinline__ void l2_priority_normal(const void *p) {
    asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------ 1-D bulk copies (TMA, non-tensor)
// Both addresses 16-byte aligned, size a multiple of 16 (checked on the host
// through the row pitch and chunk size).

// global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_addr(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// shared -> global, tracked by this thread's bulk async-groups.
__device__ __forceinline__ void bulk_store(void *gmem_dst, const void *smem_src, uint32_t bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                 ::"l"(gmem_dst), "r"(smem_addr(smem_src)), "r"(bytes), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed (writes done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------------------ plain memory helpers

__device__ __forceinline__ int64_t ld_nc_i64(const int64_t *p) {
    int64_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b64 %0, [%1];" : "=l"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u64(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_release_gpu_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

}  // namespace moe
