// combine.cu -- gather each token's per-rank partial rows and reduce them.
//
// The expert side leaves one partial row per (token, rank) in the receive
// layout; combine brings them back into token order and reduces them, the
// reduce epilogue of the pages (the Mega-MoE combine push on the DeepEP /
// DeepGEMM comparison page; "consume ready partial rows in the reduce
// epilogue" on the Ascend send-ordering page). Reduction order and precision:
// fp32 accumulation from +0.0f over the token's rows in ascending rank order
// (ascending row, since rank regions are laid out in rank order), then one
// round-to-nearest-even cast to bf16.
//
// GB300 design. Combine moves ~85% of its bytes as loads that must sit in
// shared memory until they are summed. Each SM's bulk-copy (TMA) engine keeps
// a bounded number of copies in flight, so the bytes in flight -- and the
// bandwidth -- grow with the size of each copy: whole rows (14 KB at H=7168)
// are copied at once. One CTA per SM owns a ring of chunk-sized slots
// (~220 KB) and a contiguous range of tokens; a unit is one chunk (by default
// a whole row) of one token.
//   producer warp  reads a token's receive rows, ranks them (ascending), takes
//                  D free slots from the ring (D = the token's row count, not
//                  k, so no slot is reserved for an absent row), arms the
//                  unit's mbarrier with D * chunk bytes and issues one
//                  cp.async.bulk per row into the slots. Slots come back in
//                  unit order through per-unit "empty" mbarriers.
//   consumer warps take (unit, slice) items round-robin, a slice being a
//                  <= 4 KB column range of the chunk, wait on the unit's
//                  "full" mbarrier, and sum slot by slot with all of the
//                  lane's vectors in flight at once (up to 8 x 16 B per lane,
//                  packed add.rn.f32x2: 32 independent fp32-pair chains per
//                  lane), store 16-byte bf16 vectors and arrive on the unit's
//                  "empty" mbarrier (one arrival per slice).
// Options (moe_combine_ex): per-row weights turn each add into a single-rounding
// fused multiply-add (packed fma.rn.f32x2), and the received top-k weights can
// be reduced back to [T, k] in the same ascending order.
// E4M3 partial rows (moe_combine_fp8): a slot holds a chunk of codes followed
// by its per-128 scales (two bulk copies per row); each element is
// dequantised on its own -- E4M3 -> f16 -> f32 (both exact), times its
// block's scale (mul.rn) -- and then added in the same ascending order.
// Every wait is bounded (MOE_ERR_TIMEOUT on expiry).
#include <algorithm>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kUnits = 16;       // unit ring entries
constexpr int kVMax = 8;         // 16-byte vectors per lane per slice -> slice <= 32 * 8 * 16 = 4096 B
constexpr int kHeadBytes = 4608; // full[kUnits] + empty[kUnits] mbarriers, unit entries
constexpr unsigned kFull = 0xffffffffu;

struct CombineArgs {
    const uint8_t *partial;
    int64_t row_bytes;   // H * 2 (bf16 rows) or H (E4M3 codes)
    const uint8_t *scales;       // E4M3 rows: fp32 scales [rows, H/128]
    int64_t scale_row_bytes;     // H / 128 * 4
    int64_t out_row_bytes;       // H * 2
    int slot_bytes;              // chunk_bytes, plus chunk_bytes / 32 of scales for E4M3 rows
    int num_rows;
    int T, k;
    const int32_t *dst_row;
    const float *row_weights;        // optional: weight of each receive row
    const float *recv_topk_weights;  // optional, with combined_topk_weights: [rows, k] -> [T, k]
    float *combined_topk_weights;
    uint8_t *out;
    int32_t *status;
    int chunk_bytes, num_chunks;
    int slice_bytes, num_slices;   // consumer column slices of a chunk
    int num_slots;       // ring slots of chunk_bytes
    int l2_hints;
    uint64_t timeout_ns;
    // tail balancing: tokens [0, static_tokens) are split into contiguous CTA
    // ranges; the rest form a pool claimed through balance[0] (balance[1]
    // counts finished CTAs; the last one zeroes both). nullptr: all dealt.
    unsigned int *balance;
    int static_tokens;
    int prefetch_bytes;   // of the CTA's first rows, into L2 before the dependency wait (0: none)
    TraceArgs trace;      // MOE_PROFILE builds: where the warps' records go
};

struct UnitEntry {
    int D;                   // rows of the unit; -1: no more units
    int t;                   // token of the unit
    int start;               // first ring slot (the unit's rows occupy start, start+1, ... mod num_slots)
    float w[MOE_MAX_TOPK];   // weight of the row in slot start + d (weighted combine)
    int row[MOE_MAX_TOPK];   // receive row in slot start + d
};
static_assert(2 * kUnits * 8 + kUnits * sizeof(UnitEntry) <= kHeadBytes, "unit ring header");

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// bf16 pair (lo in bits 0..15, hi in bits 16..31) -> two fp32 {lo, hi}; exact
__device__ __forceinline__ uint64_t widen_bf16x2(uint32_t w) { return pack2(w << 16, w & 0xffff0000u); }

__device__ __forceinline__ uint32_t narrow_bf16x2(uint64_t p) {
    const float lo = __uint_as_float((uint32_t)p), hi = __uint_as_float((uint32_t)(p >> 32));
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// a + b on each half with scalar add.rn.f32: a packed multiply followed by a
// packed add can be contracted into a fused multiply-add by the assembler,
// while a scalar add with an explicit rounding mode is kept separate, so the
// product is rounded before it is added
__device__ __forceinline__ uint64_t add_rn_halves(uint64_t a, uint64_t b) {
    float r0, r1;
    asm("add.rn.f32 %0, %1, %2;" : "=f"(r0) : "f"(__uint_as_float((uint32_t)a)), "f"(__uint_as_float((uint32_t)b)));
    asm("add.rn.f32 %0, %1, %2;"
        : "=f"(r1)
        : "f"(__uint_as_float((uint32_t)(a >> 32))), "f"(__uint_as_float((uint32_t)(b >> 32))));
    return pack2(__float_as_uint(r0), __float_as_uint(r1));
}

// two E4M3 codes (lo byte, hi byte) -> two fp32 {lo, hi}; exact (E4M3 is a subset of f16)
__device__ __forceinline__ uint64_t widen_e4m3x2(uint32_t b16) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)b16, __NV_E4M3);
    const float2 f = __half22float2(__half2(h));
    return pack2(__float_as_uint(f.x), __float_as_uint(f.y));
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// E4M3 rows cost more instructions per byte (dequantisation), so that variant
// runs more consumer warps.
template <bool kWeighted, bool kFP8>
__global__ void __launch_bounds__(kFP8 ? 32 * 13 : 32 * 9, 1) combine_kernel(const CombineArgs a) {
    WarpTrace wt(a.trace, MOE_TRACE_COMBINE);
    MOE_PHASES(MOE_TRACE_COMBINE, 3);
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kUnits;
    UnitEntry *entry = reinterpret_cast<UnitEntry *>(empty + kUnits);
    uint8_t *ring = smem + kHeadBytes;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int consumers = (blockDim.x >> 5) - 1;
    const int NS = a.num_slots, CH = a.chunk_bytes, SB = a.slot_bytes, nch = a.num_chunks;

    // contiguous range of the statically dealt tokens for this CTA
    const int T_st = a.static_tokens;
    const int s_begin = (int)((int64_t)T_st * blockIdx.x / gridDim.x);
    const int s_end = (int)((int64_t)T_st * (blockIdx.x + 1) / gridDim.x);
    const int nsl = a.num_slices;

    if (threadIdx.x == 0) {
        for (int e = 0; e < kUnits; ++e) {
            mbar_init(&full[e], 1);
            mbar_init(&empty[e], (uint32_t)a.num_slices);
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 1 && a.prefetch_bytes > 0) {
        // While the previous grid finishes, the first rows of this CTA's static range
        // go into L2 (evict-normal), in the order the producer will load them. Only
        // prefetch addresses come from these reads, so a row list still being written
        // costs a useless prefetch, never a wrong result: rows out of range are
        // skipped, and the lists are read past L1 (.cg), so no stale line of them is
        // left for the loads after the wait.
        const uint64_t pol = policy_evict_normal();
        const int64_t first = (int64_t)s_begin * a.k, end = (int64_t)s_end * a.k;
        int64_t done = 0;
        for (int64_t i = first; i < end && done < a.prefetch_bytes; i += 32) {
            const int row = i + lane < end ? __ldcg(a.dst_row + i + lane) : -1;
            const bool ok = row >= 0 && row < a.num_rows;
            const unsigned m = __ballot_sync(kFull, ok);
            const int64_t before = done + (int64_t)__popc(m & ((1u << lane) - 1u)) * a.row_bytes;
            if (ok && before < a.prefetch_bytes)
                bulk_prefetch_l2(a.partial + (int64_t)row * a.row_bytes, (uint32_t)a.row_bytes, pol);
            done += (int64_t)__popc(m) * a.row_bytes;
        }
    }
    MOE_PHASE(1);
    grid_dependency_wait();
    MOE_PHASE(2);
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = (a.l2_hints & 1) ? policy_evict_first() : policy_evict_normal();
        int64_t head = 0, tail = 0, oldest = 0;
        int head_slot = 0;   // head % NS, kept without 64-bit division
        float w_cur = 1.0f;
        // tokens in order: the static range, then pool tokens while the pool lasts (warp-uniform; -1: none left)
        int s_next = s_begin;
        bool pool_open = a.balance != nullptr;
        auto next_token = [&]() -> int {
            if (s_next < s_end) return s_next++;
            if (!pool_open) return -1;
            unsigned p = 0;
            if (lane == 0) p = atomicAdd(a.balance, 1u);
            p = __shfl_sync(kFull, p, 0);
            if ((int64_t)T_st + p < a.T) return T_st + (int)p;
            pool_open = false;
            return -1;
        };
        // the next kPre tokens and their receive rows (lanes < k), fetched ahead so that
        // neither a pool claim nor a row list's load stalls the issue of bulk loads
        constexpr int kPre = 8;
        int tq[kPre], rq[kPre];
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
            tq[i] = next_token();
            rq[i] = (tq[i] >= 0 && lane < a.k) ? a.dst_row[(int64_t)tq[i] * a.k + lane] : -1;
        }
        // weighted: the weight of each row of the next token, loaded one token ahead
        float w_next = (kWeighted && rq[0] >= 0 && rq[0] < a.num_rows) ? a.row_weights[rq[0]] : 1.0f;
        int64_t j = 0;       // units issued
        bool ok = true;
        while (ok) {
            const int t = tq[0];
            int row = rq[0];
            if (t < 0) break;
#pragma unroll
            for (int i = 0; i < kPre - 1; ++i) {
                tq[i] = tq[i + 1];
                rq[i] = rq[i + 1];
            }
            tq[kPre - 1] = next_token();
            rq[kPre - 1] = (tq[kPre - 1] >= 0 && lane < a.k) ? a.dst_row[(int64_t)tq[kPre - 1] * a.k + lane] : -1;
            if (row >= a.num_rows) {
                report(a.status, MOE_ERR_CAPACITY);
                row = -1;
            }
            if (kWeighted) {
                w_cur = w_next;
                w_next = (rq[0] >= 0 && rq[0] < a.num_rows) ? a.row_weights[rq[0]] : 1.0f;
            }
            const unsigned vmask = __ballot_sync(kFull, row >= 0);
            const int D = __popc(vmask);
            int pos = 0;
            for (int jj = 0; jj < a.k; ++jj) {
                const int o = __shfl_sync(kFull, row, jj);
                pos += (row >= 0 && ((vmask >> jj) & 1u) && o < row) ? 1 : 0;
            }
          for (int c = 0; c < nch; ++c, ++j) {
            const int64_t off = (int64_t)c * CH;
            const uint32_t nbytes = (uint32_t)min((int64_t)CH, a.row_bytes - off);
            // wait until the unit entry is free (units are released in order)
            auto release_oldest = [&]() {
                const int eo = (int)(oldest % kUnits);
                ok = mbar_wait_bounded(&empty[eo], (uint32_t)((oldest / kUnits) & 1), a.timeout_ns);
                if (ok) {
                    tail += entry[eo].D;
                    ++oldest;
                }
            };
            // E4M3 rows: whole units only (the per-row issue below costs the critical producer
            // more than it gains when a unit's rows are this short)
            while (ok && (j - oldest >= kUnits || (kFP8 && head + D - tail > NS))) release_oldest();
            if (!__all_sync(kFull, ok)) {
                if (lane == 0) report(a.status, MOE_ERR_TIMEOUT);
                ok = false;
                break;
            }
            const int e = (int)(j % kUnits);
            __syncwarp();   // every lane has read entry[eo] before lane 0 rewrites an entry
            if (lane == 0) {
                entry[e].D = D;
                entry[e].t = t;
                entry[e].start = head_slot;
            }
            if (row >= 0) {
                entry[e].row[pos] = row;
                if (kWeighted) entry[e].w[pos] = w_cur;
            }
            __syncwarp();
            const uint32_t sbytes = kFP8 ? nbytes / 32 : 0u;   // the chunk's scales (4 B per 128 codes)
            if (lane == 0) mbar_arrive_expect_tx(&full[e], (uint32_t)D * (nbytes + sbytes));
            // the unit's rows take slots head .. head + D - 1; each row's load is issued as soon as
            // its slot is free, not once all D are (older units release their slots in batches;
            // for E4M3 rows all D are free here)
            int issued = 0;
            while (true) {
                const int can = min(D, NS - (int)(head - tail));   // rows whose slot is free
                if (row >= 0 && pos >= issued && pos < can) {
                    const int slot = head_slot + pos < NS ? head_slot + pos : head_slot + pos - NS;
                    bulk_load(ring + (size_t)slot * SB, a.partial + (int64_t)row * a.row_bytes + off, nbytes,
                              &full[e], pol);
                    if (kFP8)
                        bulk_load(ring + (size_t)slot * SB + CH,
                                  a.scales + (int64_t)row * a.scale_row_bytes + off / 32, sbytes, &full[e], pol);
                }
                issued = max(issued, can);
                if (issued >= D || !ok) break;
                release_oldest();   // an older unit holds the next slot (D <= NS, so one exists)
                if (!__all_sync(kFull, ok)) {
                    if (lane == 0) report(a.status, MOE_ERR_TIMEOUT);
                    ok = false;
                }
            }
            if (!ok) break;
            head += D;
            head_slot += D;
            if (head_slot >= NS) head_slot -= NS;
          }
        }
        // end markers: the next units carry D = -1, so that each consumer's wait for
        // its next item ends (consumer cw's next unit is at most (consumers - 1) / nsl
        // past the last real one)
        const int markers = (consumers + nsl - 1) / nsl + 1;
        for (int i = 0; ok && i < markers; ++i, ++j) {
            while (ok && j - oldest >= kUnits) {
                const int eo = (int)(oldest % kUnits);
                ok = mbar_wait_bounded(&empty[eo], (uint32_t)((oldest / kUnits) & 1), a.timeout_ns);
                if (ok) {
                    tail += entry[eo].D;
                    ++oldest;
                }
            }
            if (!__all_sync(kFull, ok)) {
                if (lane == 0) report(a.status, MOE_ERR_TIMEOUT);
                ok = false;
                break;
            }
            const int e = (int)(j % kUnits);
            __syncwarp();
            if (lane == 0) {
                entry[e].D = -1;
                mbar_arrive(&full[e]);   // completes the phase: no bytes expected
            }
        }
        // every claim of this CTA is made: count it finished; the last CTA re-arms the pool
        if (a.balance != nullptr && lane == 0) {
            __threadfence();
            if (atomicAdd(a.balance + 1, 1u) == gridDim.x - 1) {
                atomicExch(a.balance, 0u);
                atomicExch(a.balance + 1, 0u);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int SL = a.slice_bytes;
    for (int64_t q = cw;; q += consumers) {
        const int64_t j = div_count(q, nsl);
        const int sl = (int)(q - j * nsl);
        const int e = (int)(j % kUnits);
        const bool ok = mbar_wait_bounded(&full[e], (uint32_t)((j / kUnits) & 1), a.timeout_ns);
        if (!__all_sync(kFull, ok)) {
            if (lane == 0) report(a.status, MOE_ERR_TIMEOUT);
            break;
        }
        const int D = entry[e].D;
        if (D < 0) break;                                          // no more units
        const int t = entry[e].t;
        const int c = (int)(j - div_count(j, nch) * nch);          // units are (token, chunk 0..nch-1) in order
        const int64_t off = (int64_t)c * CH;                       // chunk offset in the row
        const int cbytes = (int)min((int64_t)CH, a.row_bytes - off);
        const int soff = sl * SL;                                  // slice offset in the chunk
        const int nvec = max(0, min(SL, cbytes - soff)) / 16;
        int slot = entry[e].start;
        if constexpr (kFP8) {
            constexpr int kV8 = kVMax / 2;   // 16 codes per 16-byte vector
            uint64_t acc[kV8][8];
#pragma unroll
            for (int v = 0; v < kV8; ++v)
#pragma unroll
                for (int p = 0; p < 8; ++p) acc[v][p] = 0ull;   // +0.0f pairs
            for (int d = 0; d < D; ++d) {
                const uint8_t *sbase = ring + (size_t)slot * SB;
                const float *sc = reinterpret_cast<const float *>(sbase + CH);
#pragma unroll
                for (int v = 0; v < kV8; ++v) {
                    if (lane + 32 * v < nvec) {
                        const int pos = soff + lane * 16 + v * 512;   // code index in the chunk
                        const uint4 qv = lds128(sbase + pos);
                        const float sf = sc[pos >> 7];
                        const uint64_t ss = pack2(__float_as_uint(sf), __float_as_uint(sf));
                        const uint32_t wq[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {   // value = RN(code * scale), then acc = RN(acc + value)
                            acc[v][2 * i] = add_rn_halves(acc[v][2 * i], mul_f32x2(widen_e4m3x2(wq[i] & 0xffffu), ss));
                            acc[v][2 * i + 1] = add_rn_halves(acc[v][2 * i + 1], mul_f32x2(widen_e4m3x2(wq[i] >> 16), ss));
                        }
                    }
                }
                if (++slot == NS) slot = 0;
            }
            uint8_t *dst = a.out + (int64_t)t * a.out_row_bytes + (off + soff + lane * 16) * 2;
#pragma unroll
            for (int v = 0; v < kV8; ++v) {
                if (lane + 32 * v < nvec) {
                    uint4 o0, o1;
                    o0.x = narrow_bf16x2(acc[v][0]);
                    o0.y = narrow_bf16x2(acc[v][1]);
                    o0.z = narrow_bf16x2(acc[v][2]);
                    o0.w = narrow_bf16x2(acc[v][3]);
                    o1.x = narrow_bf16x2(acc[v][4]);
                    o1.y = narrow_bf16x2(acc[v][5]);
                    o1.z = narrow_bf16x2(acc[v][6]);
                    o1.w = narrow_bf16x2(acc[v][7]);
                    *reinterpret_cast<uint4 *>(dst + v * 1024) = o0;
                    *reinterpret_cast<uint4 *>(dst + v * 1024 + 16) = o1;
                }
            }
        } else {
            uint64_t acc[kVMax][4];
#pragma unroll
            for (int v = 0; v < kVMax; ++v)
#pragma unroll
                for (int p = 0; p < 4; ++p) acc[v][p] = 0ull;   // +0.0f pairs
            for (int d = 0; d < D; ++d) {
                const uint8_t *base = ring + (size_t)slot * SB + soff + lane * 16;
                uint64_t ww = 0;
                if (kWeighted) {
                    const uint32_t wb = __float_as_uint(entry[e].w[d]);
                    ww = (uint64_t)wb | ((uint64_t)wb << 32);
                }
#pragma unroll
                for (int v = 0; v < kVMax; ++v) {
                    if (lane + 32 * v < nvec) {
                        const uint4 qv = lds128(base + v * 512);
                        if (kWeighted) {   // acc = fma(w, x, acc), one rounding per term
                            acc[v][0] = fma_f32x2(ww, widen_bf16x2(qv.x), acc[v][0]);
                            acc[v][1] = fma_f32x2(ww, widen_bf16x2(qv.y), acc[v][1]);
                            acc[v][2] = fma_f32x2(ww, widen_bf16x2(qv.z), acc[v][2]);
                            acc[v][3] = fma_f32x2(ww, widen_bf16x2(qv.w), acc[v][3]);
                        } else {
                            acc[v][0] = add_f32x2(acc[v][0], widen_bf16x2(qv.x));
                            acc[v][1] = add_f32x2(acc[v][1], widen_bf16x2(qv.y));
                            acc[v][2] = add_f32x2(acc[v][2], widen_bf16x2(qv.z));
                            acc[v][3] = add_f32x2(acc[v][3], widen_bf16x2(qv.w));
                        }
                    }
                }
                if (++slot == NS) slot = 0;
            }
            // received top-k weights back to [T, k]: by the consumer of the first slice of the first chunk
            if (a.combined_topk_weights != nullptr && c == 0 && sl == 0 && lane < a.k) {
                float v[MOE_MAX_TOPK];
#pragma unroll
                for (int d = 0; d < MOE_MAX_TOPK; ++d)
                    if (d < D) v[d] = a.recv_topk_weights[(int64_t)entry[e].row[d] * a.k + lane];
                float cw = 0.0f;
#pragma unroll
                for (int d = 0; d < MOE_MAX_TOPK; ++d)
                    if (d < D) cw += v[d];
                a.combined_topk_weights[(int64_t)t * a.k + lane] = cw;
            }
            uint8_t *dst = a.out + (int64_t)t * a.out_row_bytes + off + soff + lane * 16;
#pragma unroll
            for (int v = 0; v < kVMax; ++v) {
                if (lane + 32 * v < nvec) {
                    uint4 o;
                    o.x = narrow_bf16x2(acc[v][0]);
                    o.y = narrow_bf16x2(acc[v][1]);
                    o.z = narrow_bf16x2(acc[v][2]);
                    o.w = narrow_bf16x2(acc[v][3]);
                    *reinterpret_cast<uint4 *>(dst + v * 512) = o;
                }
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[e]);
    }
}

inline int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

}  // namespace

int launch_combine(const CombineLaunch &L) {
    if (L.num_tokens == 0) return MOE_OK;
    const Tuning &tu = tuning();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(L.stream);

    const bool fp8 = L.fp8;    // E4M3 rows with per-128 scales
    CombineArgs a;
    a.trace = trace_args();
    a.partial = static_cast<const uint8_t *>(L.partial);
    a.row_bytes = fp8 ? (int64_t)L.hidden : (int64_t)L.hidden * 2;
    a.scales = reinterpret_cast<const uint8_t *>(L.partial_scales);
    a.scale_row_bytes = (int64_t)(L.hidden / 128) * 4;
    a.out_row_bytes = (int64_t)L.hidden * 2;
    a.num_rows = L.num_partial_rows;
    a.T = L.num_tokens;
    a.k = L.num_topk;
    a.dst_row = L.token_dst_row;
    a.row_weights = L.row_weights;
    a.recv_topk_weights = L.recv_topk_weights;
    a.combined_topk_weights = L.recv_topk_weights ? L.combined_topk_weights : nullptr;
    a.out = static_cast<uint8_t *>(L.out);
    a.status = L.status;
    a.l2_hints = tu.l2_hints;
    a.timeout_ns = kDefaultWaitNs;
    a.balance = (L.balance != nullptr && tu.combine_pool > 0 && tu.combine_pool < 100) ? L.balance : nullptr;

    // equal chunks no larger than the tuned maximum (E4M3 rows: of 512 codes, so
    // that each chunk's scales are whole 16-byte pieces), small enough that
    // the ring holds a unit of k rows with room to spare (k + 4 slots)
    const int64_t align = fp8 ? 512 : 16;
    const size_t budget = std::min<size_t>(device_smem_optin(), (size_t)std::max(64 << 10, tu.combine_ring_bytes));
    int64_t nch = (a.row_bytes + tu.combine_chunk - 1) / std::max(16, tu.combine_chunk);
    while (true) {
        a.chunk_bytes = (int)round_up((a.row_bytes + nch - 1) / nch, align);
        a.slot_bytes = fp8 ? a.chunk_bytes + a.chunk_bytes / 32 : a.chunk_bytes;
        if ((int64_t)(budget - kHeadBytes) / a.slot_bytes >= (int64_t)a.k + 4 || a.chunk_bytes <= align) break;
        ++nch;
    }
    a.num_chunks = (int)((a.row_bytes + a.chunk_bytes - 1) / a.chunk_bytes);
    a.num_slots = (int)((budget - kHeadBytes) / (size_t)a.slot_bytes);
    if (a.num_slots < a.k) return MOE_ERR_INVALID_ARG;   // a unit of k rows must fit in the ring
    // consumer slices: equal pieces of at most 32 lanes x kVMax x 16 B of bf16
    // (E4M3: 32 lanes x kVMax / 2 x 16 codes), multiples of 16 B
    const int slice_max = fp8 ? 32 * (kVMax / 2) * 16 : 32 * kVMax * 16;
    a.num_slices = (a.chunk_bytes + slice_max - 1) / slice_max;
    a.slice_bytes = (int)round_up((a.chunk_bytes + a.num_slices - 1) / a.num_slices, 16);
    const size_t smem = kHeadBytes + (size_t)a.num_slots * a.slot_bytes;
    const bool weighted = a.row_weights != nullptr;
    const void *fn = fp8 ? (const void *)combine_kernel<false, true>
                         : (weighted ? (const void *)combine_kernel<true, false> : (const void *)combine_kernel<false, false>);
    if (ensure_dynamic_smem(fn, smem) != MOE_OK) return MOE_ERR_CUDA;

    const int consumers = fp8 ? std::max(1, std::min(12, tu.combine_fp8_warps)) : std::max(1, std::min(8, tu.combine_warps));
    const int grid = std::max(1, std::min(L.num_tokens, device_sm_count()));
    // the pool pays off only with several tokens per CTA (its claims and the
    // finishing count cost a few microseconds of latency); for E4M3 rows, whose
    // producer is the critical warp, only with long runs
    if (a.T < (fp8 ? tu.combine_fp8_pool_min_tokens : 8) * grid) a.balance = nullptr;
    const int pool_pct = fp8 ? tu.combine_fp8_pool : tu.combine_pool;
    if (pool_pct <= 0 || pool_pct >= 100) a.balance = nullptr;
    a.static_tokens = a.balance ? (int)((int64_t)a.T * (100 - pool_pct) / 100) : a.T;
    a.prefetch_bytes = (tu.overlap != 0 && !fp8) ? std::max(0, tu.combine_prefetch) : 0;
    void (*kernel)(const CombineArgs) =
        fp8 ? combine_kernel<false, true> : (weighted ? combine_kernel<true, false> : combine_kernel<false, false>);
    return launch_kernel(kernel, dim3(grid), dim3((consumers + 1) * 32), smem, st, tu.overlap != 0, a) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

}  // namespace moe
