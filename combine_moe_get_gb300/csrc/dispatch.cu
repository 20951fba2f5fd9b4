// dispatch.cu -- copy each token's row once per distinct destination rank
// (or, in expand mode, once per valid top-k entry).
//
// DeepEP V2 deep-dive page ("DeepEP V2 深度深潜"), section 3.3 stage 2: a
// dispatch warp loads a token's hidden row into shared memory once and stores
// it once per de-duplicated destination rank; section 1.3 (factor 2) counts
// exactly that HBM traffic (one read per token, one write per rank). The
// DeepEP intra/inter-node page's NVLink receiver shows the relay as a 1-D TMA
// load into shared memory followed by 1-D TMA stores; the same relay is used
// here, but every destination is a region of this GPU's own HBM.
//
// GB300 design: a persistent grid (a multiple of the SM count) of CTAs whose
// warps run independent pipelines. A unit is one chunk of one token's row.
// Lane 0 of each warp keeps S-1 bulk loads (cp.async.bulk global->shared,
// completion on an mbarrier) in flight ahead of the unit being stored, and
// stores each landed chunk with one cp.async.bulk shared->global per
// destination row. The row bytes never pass through registers. The other
// lanes read the receive rows and write the per-row metadata. In FP8 mode the
// warp quantises the landed chunk (per 128 channels: amax, scale = amax/448,
// e4m3 round-to-nearest-even with saturation) into a second shared buffer,
// which the bulk stores then replicate; scales are written with plain stores.
#include <algorithm>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kMaxStages = 8;
constexpr int kBarBytes = 128;
constexpr unsigned kFull = 0xffffffffu;

struct DispatchArgs {
    const uint8_t *x;
    int64_t row_bytes;        // input row pitch (H * 2)
    int k, m, E;
    const int64_t *topk;
    const float *topk_w;
    const int32_t *dst_row;
    int capacity;
    uint8_t *recv_x;
    int64_t recv_row_bytes;   // H * 2 (bf16) or H (FP8)
    float *recv_scales;
    int64_t *recv_topk_idx;
    float *recv_topk_w;
    int32_t *recv_src;
    float *x_scales;
    const float *in_scales;   // E4M3 input: the token's scales, copied to every destination row
    int nb;                   // scale blocks per row (H / 128), FP8
    int expand;               // dst_row holds expand-mode rows: a row's metadata keeps its own entry only
    int32_t *status;
    int chunk_bytes;          // input bytes per unit; multiple of 16 (FP8: of 256)
    int num_chunks;           // units per token
    int64_t num_units;
    int stages;
    int warp_smem;
    int l2_hints;
    uint64_t timeout_ns;
    // fused launch (layout computed by every CTA in shared memory, dst_row unused)
    int T, R;                 // tokens, ranks
    int fl_words;             // bitmap words per rank: ceil(T / 32)
    size_t fl_off;            // byte offset of the layout region in dynamic shared memory
    moe_layout_t fl_out;      // layout outputs, written by CTA 0
    int loads_before_wait;    // first stage loads (input rows only) before the dependency wait
    // input units per CTA to bring into L2 right after the first stage loads
    // (its next dealt units, then pool units blockIdx + i * gridDim), kept with
    // an evict-last policy when prefetch_keep is set; with loads_before_wait
    // this happens while the dependency wait lasts. Bounded on the host so that
    // the grid's evict-last lines take at most a fixed share of L2.
    int64_t prefetch_units;
    int prefetch_keep;
    // tail balancing: units [0, static_units) are dealt round-robin to the CTAs;
    // the rest form a pool claimed through pool[0], so that CTAs on faster SMs
    // take more of them; pool[1] counts the CTAs whose warps will claim no
    // more, and the last of them zeroes both (they are zero at launch).
    // nullptr: every unit is dealt.
    unsigned int *pool;
    int64_t static_units;
    TraceArgs trace;   // MOE_PROFILE builds: where the warps' records go
};

// Whether unit u's input rows were prefetched (evict-last) by the rule of
// dispatch_kernel: CTA b (of G) prefetches its dealt units b + j * G with
// first <= j < first + P (j < its dealt count), then, when every CTA's first
// stage loads took dealt units (dealt >= G * first, so that no pool unit is
// claimed before all prefetches are issued), pool units dealt + b + m * G for
// m < P - (the number of dealt units it prefetched).
__device__ __forceinline__ bool unit_prefetched(int64_t u, int64_t dealt, int64_t G, int64_t first, int64_t P) {
    if (u < dealt) {
        const int64_t j = div_count(u, (int)G);
        return j >= first && j < first + P;
    }
    if (dealt < G * first) return false;
    const int64_t i = u - dealt, m = div_count(i, (int)G), b = i - m * G;
    const int64_t cta_units = dealt > b ? (dealt - 1 - b) / G + 1 : 0;
    const int64_t n_dealt = max((int64_t)0, min(cta_units, first + P) - first);
    return m < P - n_dealt;
}

// Block scale RN(amax / 448) without a division: q0 = RN(amax * C) with
// C = RN(1/448), r = amax - q0 * 448 (exact by FMA), s = RN(r * C + q0).
// amax is a bf16 value, and for every non-negative finite bf16 value this
// equals the IEEE quotient (checked exhaustively with exact arithmetic).
__device__ __forceinline__ float block_scale(float amax) {
    const float C = __uint_as_float(0x3b124925u);   // RN(1 / 448)
    const float q0 = __fmul_rn(amax, C);
    const float r = __fmaf_rn(-q0, 448.0f, amax);
    return __fmaf_rn(r, C, q0);
}

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));   // max error 1 ulp (relative <= 2^-23)
    return r;
}

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// E4M3 codes of y = RN(x / scale) (the IEEE fp32 quotient) without a division.
// r = rcp_approx(scale) is within 1 ulp (relative 2^-23) of 1/scale. With
// r_lo = RN(r * (1 - 2^-20)) and r_hi = RN(r * (1 + 2^-20)), the products
// RN(x * r_lo) and RN(x * r_hi) lie strictly below and above y in magnitude
// (each is off 1/scale by at most 2^-20 + 2^-23 + 2 * 2^-24 < 2^-19 relative
// in one direction and at least 2^-20 - 2^-23 - 2 * 2^-24 > 2^-21 in the
// same direction, while y is within 2^-24 of x / scale). E4M3 rounding
// (RNE, saturating) is monotone in its argument, so when the two products
// give the same code that code is the code of y; otherwise (the quotient is
// within ~2^-19 of a rounding boundary) y itself is computed by the IEEE
// division. A scale below 2^-100 (whose reciprocal may overflow) takes the
// division throughout.
constexpr float kTinyScale = 7.8886090522e-31f;   // 2^-100

__device__ __forceinline__ uint32_t cvt_e4m3x2(uint64_t xy) {   // {x, y} -> (code(y) << 8) | code(x)
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(__uint_as_float((uint32_t)xy),
                                                          __uint_as_float((uint32_t)(xy >> 32))),
                                              __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ uint64_t bf16x2_as_f32x2(uint32_t w) {   // two bf16 in one word -> {lo, hi} as f32x2
    uint64_t xy;
    asm("mov.b64 %0, {%1, %2};" : "=l"(xy) : "r"(w << 16), "r"(w & 0xffff0000u));
    return xy;
}

// Reciprocal bracket of a nonzero block scale (see above).
struct RcpBracket {
    uint64_t lo, hi;   // {r_lo, r_lo} and {r_hi, r_hi} as f32x2 operands
};

__device__ __forceinline__ RcpBracket rcp_bracket(float scale) {
    const float r = rcp_approx(scale);
    const float r_lo = __fmul_rn(r, 0.99999904632568359375f);   // 1 - 2^-20
    const float r_hi = __fmul_rn(r, 1.00000095367431640625f);   // 1 + 2^-20
    RcpBracket b;
    b.lo = (uint64_t)__float_as_uint(r_lo) | ((uint64_t)__float_as_uint(r_lo) << 32);
    b.hi = (uint64_t)__float_as_uint(r_hi) | ((uint64_t)__float_as_uint(r_hi) << 32);
    return b;
}

// Codes of one word's two bf16 values divided by scale, (code1 << 8) | code0.
__device__ __forceinline__ uint32_t e4m3_pair(uint32_t w, float scale, const RcpBracket &b) {
    const uint64_t xy = bf16x2_as_f32x2(w);
    const uint32_t lo = cvt_e4m3x2(mul_f32x2(xy, b.lo));
    const uint32_t hi = cvt_e4m3x2(mul_f32x2(xy, b.hi));
    if (lo == hi && scale >= kTinyScale) return lo;
    // within ~2^-19 of a rounding boundary (rare), or a tiny scale: the IEEE quotient
    const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xffff0000u);
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x0 / scale, x1 / scale), __NV_SATFINITE, __NV_E4M3);
}

// Codes of the 8 values of one uint4 (4 words), packed 4 codes per 32 bits.
__device__ __forceinline__ uint2 e4m3_quad(uint4 v, float scale, const RcpBracket &b) {
    uint2 q;
    q.x = e4m3_pair(v.x, scale, b) | (e4m3_pair(v.y, scale, b) << 16);
    q.y = e4m3_pair(v.z, scale, b) | (e4m3_pair(v.w, scale, b) << 16);
    return q;
}

// Per half: the larger of |a| and |b| (two bf16 in a word), in one instruction;
// the sign bit of each half is the XOR of the inputs' signs and is masked off
// by the caller. A maximum of bf16 magnitudes is exact, so widening the result
// gives the same fp32 value as the maximum of the widened magnitudes.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// max |x| over the bf16 halves of one word, as an fp32
__device__ __forceinline__ float word_absmax(uint32_t m) {
    m = absmax_bf16x2(m, m >> 16);   // low half: the larger of the two halves
    return __uint_as_float((m & 0x7fffu) << 16);
}

// Quantise one 128-channel block held by a half-warp (16 lanes x 8 values).
// Returns the block's scale; writes the 8 codes of this lane to `q8`.
__device__ __forceinline__ float quantize_lane8(const uint4 v, uint2 &q8) {
    float amax = word_absmax(absmax_bf16x2(absmax_bf16x2(v.x, v.y), absmax_bf16x2(v.z, v.w)));
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    const float scale = block_scale(amax);
    if (scale == 0.0f) {
        q8 = make_uint2(0u, 0u);
    } else {
        const RcpBracket b = rcp_bracket(scale);
        q8 = e4m3_quad(v, scale, b);
    }
    return scale;
}

// Quantise one 128-channel block held by a quarter-warp (8 lanes x 16 values;
// `lo`, `hi` are the lane's 32 contiguous bytes). Returns the block's scale;
// writes the 16 codes to `q16`.
__device__ __forceinline__ float quantize_lane16(const uint4 lo, const uint4 hi, uint4 &q16) {
    float amax = word_absmax(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(lo.x, lo.y), absmax_bf16x2(lo.z, lo.w)),
                                           absmax_bf16x2(absmax_bf16x2(hi.x, hi.y), absmax_bf16x2(hi.z, hi.w))));
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    const float scale = block_scale(amax);
    if (scale == 0.0f) {
        q16 = make_uint4(0u, 0u, 0u, 0u);
    } else {
        const RcpBracket b = rcp_bracket(scale);
        const uint2 a0 = e4m3_quad(lo, scale, b), a1 = e4m3_quad(hi, scale, b);
        q16 = make_uint4(a0.x, a0.y, a1.x, a1.y);
    }
    return scale;
}

// ------------------------------------------------------------------ fused layout (small batches)
//
// For a small batch every CTA of the fused launch computes the whole layout
// itself in shared memory, the same definition as layout.cu: per token the
// entries are de-duplicated by rank (__match_any_sync, lowest entry owns
// the rank), a bitmap [word][rank] records membership, per-rank popcounts
// give the counts and word prefixes, and an exclusive scan over ranks gives
// the rank regions. Receive row of (t, r) = rank_prefix[r] + #{t' < t in r}.
// No CTA waits on another. CTA 0 writes the counts and prefixes (and counts
// experts); every CTA writes is_token_in_rank and token_dst_row for its own
// slice of tokens.

// Shared memory of the fused layout: bitmap u32 [W][R] | word prefix u16 [R][W] |
// rank prefix i32 [R+1] | expert histogram i32 [E+1] | expert ids i16 [T*k] |
// rank ids i16 [T*k]
struct FusedSmem {
    size_t wprefix, rprefix, hist, eid, rid, total;
};

__host__ __device__ inline FusedSmem fused_smem(int T, int R, int E, int k) {
    const size_t W = (size_t)((T + 31) / 32);
    FusedSmem f;
    f.wprefix = (W * R * 4 + 15) / 16 * 16;
    f.rprefix = f.wprefix + (W * R * 2 + 15) / 16 * 16;
    f.hist = f.rprefix + ((size_t)(R + 1) * 4 + 15) / 16 * 16;
    f.eid = f.hist + ((size_t)(E + 1) * 4 + 15) / 16 * 16;
    f.rid = f.eid + ((size_t)T * k * 2 + 15) / 16 * 16;
    f.total = f.rid + ((size_t)T * k * 2 + 15) / 16 * 16;
    return f;
}

// The (token, rank) owner of entry j of token t, and its receive row (-1 if not an owner).
__device__ __forceinline__ int fused_row(const DispatchArgs &a, const uint32_t *bitmap, const uint16_t *wprefix,
                                         const int32_t *rprefix, int t, int r, int lane, unsigned peers) {
    if (r < 0 || (__ffs(peers) - 1) != lane) return -1;
    const uint32_t word = bitmap[(t >> 5) * a.R + r];
    return rprefix[r] + wprefix[r * a.fl_words + (t >> 5)] + __popc(word & ((1u << (t & 31)) - 1u));
}

// Every thread of the CTA calls this once.
__device__ void fused_layout(const DispatchArgs &a, uint8_t *region) {
    const FusedSmem fs = fused_smem(a.T, a.R, a.E, a.k);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(region);
    uint16_t *wprefix = reinterpret_cast<uint16_t *>(region + fs.wprefix);
    int32_t *rprefix = reinterpret_cast<int32_t *>(region + fs.rprefix);
    int32_t *hist = reinterpret_cast<int32_t *>(region + fs.hist);
    int16_t *eid = reinterpret_cast<int16_t *>(region + fs.eid);
    int16_t *rid = reinterpret_cast<int16_t *>(region + fs.rid);
    const int R = a.R, W = a.fl_words, k = a.k;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, warps = blockDim.x >> 5;
    const bool cta0 = blockIdx.x == 0;
    for (int i = threadIdx.x; i < W * R; i += blockDim.x) bitmap[i] = 0u;
    if (cta0)
        for (int i = threadIdx.x; i < a.E; i += blockDim.x) hist[i] = 0;
    // the batch's top-k entries as expert ids (-1: masked or invalid), 8 loads in flight per thread
    const int n_ent = a.T * k;
    for (int base = threadIdx.x; base < n_ent; base += 8 * blockDim.x) {
        int64_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * blockDim.x;
            v[u] = i < n_ent ? ld_nc_i64(a.topk + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * blockDim.x;
            if (i < n_ent) {
                const bool ok = v[u] >= 0 && v[u] < a.E;
                if (!ok && v[u] != -1 && cta0) report(a.status, MOE_ERR_BAD_TOPK);
                eid[i] = ok ? (int16_t)v[u] : (int16_t)-1;
                rid[i] = ok ? (int16_t)((int)v[u] / a.m) : (int16_t)-1;
            }
        }
    }
    __syncthreads();
    // a lane per (token, entry), 32 / k tokens per warp: each rank of a token once (its
    // lowest entry, found among the token's lanes by one match), membership bits
    const int tpp = 32 / k, sub = lane / k, j = lane - sub * k;
    const bool lane_used = sub < tpp;
    for (int base = warp * tpp; base < a.T; base += warps * tpp) {
        const int t = base + sub;
        const bool act = lane_used && t < a.T;
        const int r = act ? (int)rid[t * k + j] : -1;
        if (cta0 && r >= 0) atomicAdd(&hist[eid[t * k + j]], 1);
        const unsigned peers = __match_any_sync(kFull, r >= 0 ? sub * R + r : -(lane + 1));
        if (r >= 0 && __ffs(peers) - 1 == lane) atomicOr(&bitmap[(t >> 5) * R + r], 1u << (t & 31));
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        uint32_t run = 0;
        for (int w = 0; w < W; ++w) {
            wprefix[r * W + w] = (uint16_t)run;
            run += __popc(bitmap[w * R + r]);
        }
        rprefix[r] = (int32_t)run;
    }
    __syncthreads();
    if (warp == 0) warp_exclusive_scan(rprefix, R, lane);
    if (cta0 && warp == (warps > 1 ? 1 : 0)) {
        for (int e = lane; e < a.E; e += 32) a.fl_out.num_tokens_per_expert[e] = hist[e];
        __syncwarp();
        warp_exclusive_scan(hist, a.E, lane);
        __syncwarp();
        for (int e = lane; e <= a.E; e += 32) a.fl_out.expert_prefix[e] = hist[e];
    }
    __syncthreads();
    // ---- layout outputs: counts and prefixes by CTA 0, membership and rows by token slice
    if (cta0) {
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            a.fl_out.num_tokens_per_rank[r] = rprefix[r + 1] - rprefix[r];
            a.fl_out.rank_prefix[r] = rprefix[r];
        }
        if (threadIdx.x == 0) a.fl_out.rank_prefix[R] = rprefix[R];
    }
    const int t_lo = (int)((int64_t)a.T * blockIdx.x / gridDim.x);
    const int t_hi = (int)((int64_t)a.T * (blockIdx.x + 1) / gridDim.x);
    uint8_t *in_rank = a.fl_out.is_token_in_rank + (int64_t)t_lo * R;
    const int nbytes = (t_hi - t_lo) * R;
    if ((R & 3) == 0) {
        for (int i = threadIdx.x; i < nbytes / 4; i += blockDim.x) {
            const int tl = (i * 4) / R, r0 = i * 4 - tl * R, t = t_lo + tl;
            uint32_t v = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) v |= ((bitmap[(t >> 5) * R + r0 + b] >> (t & 31)) & 1u) << (8 * b);
            reinterpret_cast<uint32_t *>(in_rank)[i] = v;
        }
    } else {
        for (int i = threadIdx.x; i < nbytes; i += blockDim.x) {
            const int tl = i / R, r = i - tl * R, t = t_lo + tl;
            in_rank[i] = (uint8_t)((bitmap[(t >> 5) * R + r] >> (t & 31)) & 1u);
        }
    }
    for (int base = t_lo + warp * tpp; base < t_hi; base += warps * tpp) {
        const int t = base + sub;
        const bool act = lane_used && t < t_hi;
        const int r = act ? (int)rid[t * k + j] : -1;
        const unsigned peers = __match_any_sync(kFull, r >= 0 ? sub * R + r : -(lane + 1));
        const int row = fused_row(a, bitmap, wprefix, rprefix, t, r, lane, peers);
        if (act) a.fl_out.token_dst_row[(int64_t)t * k + j] = row;
    }
}

template <bool kFP8, bool kFused>
__global__ void __launch_bounds__(512, 1) dispatch_kernel(const DispatchArgs a) {
    WarpTrace wt(a.trace, MOE_TRACE_DISPATCH);
    MOE_PHASES(MOE_TRACE_DISPATCH, 4);
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    const int S = a.stages;
    const int chunk = a.chunk_bytes;
    uint8_t *wbase = smem + (size_t)warp * a.warp_smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(wbase);
    uint8_t *in_stage = wbase + kBarBytes;
    uint8_t *out_stage = in_stage + (size_t)S * chunk;                                  // FP8 codes
    float *sc_stage = reinterpret_cast<float *>(out_stage + (size_t)S * (chunk / 2));  // FP8 scales

    // The CTA owns units blockIdx.x + j * gridDim.x; its warps claim them in
    // order (j) from a shared counter as they refill their stages, so that a
    // warp whose units had fewer destinations takes more of them.
    __shared__ int s_next_unit;
    __shared__ int s_retired;   // warps of this CTA that claim no more
    __shared__ int s_pf_warps;  // warps whose share of the L2 prefetches is issued
    if (threadIdx.x == 0) {
        s_next_unit = 0;
        s_retired = 0;
        s_pf_warps = 0;
    }
    __syncthreads();
    if (!a.loads_before_wait) {
        MOE_PHASE(1);
        grid_dependency_wait();
        MOE_PHASE(2);
    }
    const int64_t G = gridDim.x;
    const int64_t dealt = a.pool ? a.static_units : a.num_units;
    const int64_t cta_units = dealt > (int64_t)blockIdx.x ? (dealt - 1 - blockIdx.x) / G + 1 : 0;
    int64_t *ring = reinterpret_cast<int64_t *>(wbase + 64);   // unit of each stage (after the <= 8 barriers)

    const uint64_t pol_load = (a.l2_hints & 1) ? policy_evict_first() : policy_evict_normal();
    const uint64_t pol_store = (a.l2_hints & 2) ? policy_evict_first() : policy_evict_normal();

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }

    // lane 0: once a claim finds nothing the warp claims no more and counts
    // itself out; the CTA's last warp counts the CTA out of the pool, and the
    // last CTA of the grid re-arms it (no tail barrier: the other warps may
    // still be storing)
    bool exhausted = false;
    auto retire = [&]() {
        exhausted = true;
        if (a.pool != nullptr && atomicAdd(&s_retired, 1) == (int)(blockDim.x >> 5) - 1 &&
            atomicAdd(a.pool + 1, 1u) == gridDim.x - 1) {
            *reinterpret_cast<volatile unsigned int *>(a.pool) = 0u;
            *reinterpret_cast<volatile unsigned int *>(a.pool + 1) = 0u;
        }
    };
    auto claim = [&]() -> int64_t {   // lane 0; -1 once the CTA's units (and the pool) are exhausted
        if (exhausted) return -1;
        const int64_t j = atomicAdd(&s_next_unit, 1);
        if (j < cta_units) return (int64_t)blockIdx.x + j * G;
        if (a.pool != nullptr) {
            const int64_t p = dealt + (int64_t)atomicAdd(a.pool, 1u);
            if (p < a.num_units) return p;
        }
        retire();
        return -1;
    };
    auto issue_load = [&](int64_t u, int s) {   // lane 0
        const int64_t t = div_count(u, a.num_chunks);
        const int64_t off = (u - t * a.num_chunks) * (int64_t)chunk;
        const uint32_t nbytes = (uint32_t)min((int64_t)chunk, a.row_bytes - off);
        mbar_arrive_expect_tx(&bars[s], nbytes);
        bulk_load(in_stage + (size_t)s * chunk, a.x + t * a.row_bytes + off, nbytes, &bars[s], pol_load);
    };
    if (lane == 0) {
        for (int s = 0; s < S; ++s) {
            const int64_t u = claim();
            ring[s] = u;
            if (u >= 0) issue_load(u, s);
        }
    }
    __syncwarp();
    bool pf_pending = false;   // the CTA's L2 prefetches may still be being issued
    // Bring the rows of this CTA's next units into L2 as well, all at once (the
    // input rows are complete here: after the dependency wait, or, launched
    // right behind this library's layout whose outputs are read only after the
    // wait below, before it, so that the reads overlap the layout)
    if (a.prefetch_units > 0) {
        const uint64_t pol_pf = a.prefetch_keep ? policy_evict_last() : policy_evict_normal();
        const int64_t first = (int64_t)warps * S;   // units the stage loads above claimed
        const int64_t n_dealt = max((int64_t)0, min(cta_units, first + a.prefetch_units) - first);
        const int64_t pool_units = (a.pool && dealt >= G * first) ? a.num_units - dealt : 0;
        const int64_t cta_pool = pool_units > (int64_t)blockIdx.x ? (pool_units - 1 - blockIdx.x) / G + 1 : 0;
        const int64_t n_pool = min(cta_pool, max((int64_t)0, (int64_t)a.prefetch_units - n_dealt));
        for (int64_t i = threadIdx.x; i < n_dealt + n_pool; i += blockDim.x) {
            const int64_t u = i < n_dealt ? (int64_t)blockIdx.x + (first + i) * G
                                          : dealt + (int64_t)blockIdx.x + (i - n_dealt) * G;
            const int64_t t = div_count(u, a.num_chunks);
            const int64_t off = (u - t * a.num_chunks) * (int64_t)chunk;
            bulk_prefetch_l2(a.x + t * a.row_bytes + off, (uint32_t)min((int64_t)chunk, a.row_bytes - off), pol_pf);
        }
        // every prefetch of the CTA is issued before any of its warps claims a unit
        // past its stages (a prefetch landing after the unit's own load would keep
        // its lines evict-last): each warp counts itself in, and a warp waits for
        // the count at its first claim instead of at a CTA barrier here, so the
        // warps start on their stage loads while the prefetches are still being
        // accepted by the copy engine (which takes them at the memory's pace)
#if MOE_TUNE_DISPATCH_PREFETCH_NOSYNC
        __syncwarp();
        if (lane == 0) atomicAdd(&s_pf_warps, 1);
        pf_pending = true;
#else
        __syncthreads();
#endif
    }
    if (a.loads_before_wait) {
        MOE_PHASE(1);
        grid_dependency_wait();
        MOE_PHASE(2);
    }
    grid_launch_dependents();

    // fused launch: the layout, computed while the first loads are in flight
    const uint32_t *fl_bitmap = nullptr;
    const uint16_t *fl_wprefix = nullptr;
    const int32_t *fl_rprefix = nullptr;
    const int16_t *fl_eid = nullptr, *fl_rid = nullptr;
    if constexpr (kFused) {
        fused_layout(a, smem + a.fl_off);
        MOE_PHASE(3);
        const FusedSmem fs = fused_smem(a.T, a.R, a.E, a.k);
        fl_bitmap = reinterpret_cast<const uint32_t *>(smem + a.fl_off);
        fl_wprefix = reinterpret_cast<const uint16_t *>(smem + a.fl_off + fs.wprefix);
        fl_rprefix = reinterpret_cast<const int32_t *>(smem + a.fl_off + fs.rprefix);
        fl_eid = reinterpret_cast<const int16_t *>(smem + a.fl_off + fs.eid);
        fl_rid = reinterpret_cast<const int16_t *>(smem + a.fl_off + fs.rid);
    }

    // receive rows (and, for the first chunk, the routing) of the next unit, prefetched one unit ahead
    auto fetch = [&](int64_t u, int &row, int64_t &e, float &w) {
        const int64_t t = div_count(u, a.num_chunks);
        const bool first = (u - t * a.num_chunks) == 0;
        row = -1; e = -1; w = 0.0f;
        if constexpr (kFused) {
            int r = -1;
            if (lane < a.k) {
                e = fl_eid[t * a.k + lane];
                r = fl_rid[t * a.k + lane];
                if (first && a.topk_w) w = a.topk_w[t * a.k + lane];
            }
            const unsigned peers = __match_any_sync(kFull, r >= 0 ? r : -(lane + 1));
            row = fused_row(a, fl_bitmap, fl_wprefix, fl_rprefix, (int)t, r, lane, peers);
            if (!first) e = -1;
        } else {
            if (lane < a.k) {
                row = a.dst_row[t * a.k + lane];
                if (first) {
                    e = a.topk[t * a.k + lane];
                    if (a.topk_w) w = a.topk_w[t * a.k + lane];
                }
            }
        }
    };
    int row_n = -1; int64_t e_n = -1; float w_n = 0.0f;
    if (ring[0] >= 0) fetch(ring[0], row_n, e_n, w_n);

    int s = 0;              // stage of iteration i (i % S)
    uint32_t parity = 0;    // phase parity of that stage ((i / S) & 1)
    for (int64_t i = 0;; ++i, s = (s + 1 == S) ? 0 : s + 1, parity ^= (s == 0) ? 1u : 0u) {
        const int64_t u = ring[s];
        if (u < 0) break;
        const int64_t t = div_count(u, a.num_chunks);
        const int c = (int)(u - t * a.num_chunks);
        const int64_t off = (int64_t)c * chunk;
        const int nbytes = (int)min((int64_t)chunk, a.row_bytes - off);

        int row = row_n;
        const int64_t e = e_n;
        const float wgt = w_n;
        const int64_t u_next = ring[s + 1 == S ? 0 : s + 1];   // claimed at least one iteration ago (S >= 3)
        if (u_next >= 0) fetch(u_next, row_n, e_n, w_n);
        if (row >= a.capacity) {
            if (c == 0) report(a.status, MOE_ERR_CAPACITY);
            row = -1;
        }
        const unsigned dmask = __ballot_sync(kFull, row >= 0);

        bool ok = true;
        if (kFP8 || lane == 0) ok = mbar_wait_bounded(&bars[s], parity, a.timeout_ns);
        if (!__all_sync(kFull, ok)) {
            if (lane == 0) report(a.status, MOE_ERR_TIMEOUT);
            break;
        }
        // input rows brought into L2 with an evict-last policy during the
        // dependency wait return to normal priority once their load has landed
        // (lines aligned down to 128 bytes lie in the same page as the row's own)
        if (a.prefetch_units > 0 && a.prefetch_keep &&
            unit_prefetched(u, dealt, G, (int64_t)warps * S, a.prefetch_units)) {
            const uintptr_t g = reinterpret_cast<uintptr_t>(a.x + t * a.row_bytes + off);
            const uintptr_t lo = g & ~(uintptr_t)127, hi = (g + (uintptr_t)nbytes - 1) & ~(uintptr_t)127;
            for (uintptr_t l = lo + (uintptr_t)lane * 128; l <= hi; l += 32 * 128)
                l2_priority_normal(reinterpret_cast<const void *>(l));
        }

        const uint8_t *src = in_stage + (size_t)s * chunk;
        int out_bytes = nbytes;
        int64_t out_off = off;
        const int cpb = chunk / 256;            // FP8 scale blocks per full chunk
        const int nblk = nbytes / 256;          // FP8 scale blocks in this chunk
        float *sc = sc_stage + (size_t)s * cpb;
        if constexpr (kFP8) {
            uint8_t *q = out_stage + (size_t)s * (chunk / 2);
            const int half = lane >> 4, hl = lane & 15;
            for (int b0 = 0; b0 < nblk; b0 += 2) {
                const int b = b0 + half;
                const bool act = b < nblk;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (act) v = *reinterpret_cast<const uint4 *>(src + (size_t)b * 256 + hl * 16);
                uint2 q8;
                const float scale = quantize_lane8(v, q8);
                if (act) {
                    *reinterpret_cast<uint2 *>(q + (size_t)b * 128 + hl * 8) = q8;
                    if (hl == 0) sc[b] = scale;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            src = q;
            out_bytes = nbytes / 2;
            out_off = off / 2;
        }

        // every bulk store of this chunk first, then the per-row metadata
        for (unsigned mm = dmask; mm; mm &= mm - 1) {
            const int rowd = __shfl_sync(kFull, row, __ffs(mm) - 1);
            if (lane == 0)
                bulk_store(a.recv_x + (int64_t)rowd * a.recv_row_bytes + out_off, src, (uint32_t)out_bytes, pol_store);
        }
        if (lane == 0) bulk_commit();
        // rank of this lane's expert (-1 if masked or invalid) and its index within the rank
        int rl = -1, el = 0;
        if (c == 0 && e >= 0 && e < a.E) {
            rl = (int)e / a.m;
            el = (int)e - rl * a.m;
        }
        // E4M3 input: the token's scales, read once (up to 4 per lane, nb <= 128) for every destination
        constexpr int kInScales = 4;
        float isc[kInScales];
        const bool in_sc = a.in_scales != nullptr && c == 0 && a.nb <= 32 * kInScales;
        if (in_sc) {
#pragma unroll
            for (int i = 0; i < kInScales; ++i) {
                const int b = lane + 32 * i;
                isc[i] = b < a.nb ? a.in_scales[t * a.nb + b] : 0.0f;
            }
        }
        for (unsigned mm = dmask; mm; mm &= mm - 1) {
            const int jd = __ffs(mm) - 1;
            const int rowd = __shfl_sync(kFull, row, jd);
            if constexpr (kFP8) {
                for (int b = lane; b < nblk; b += 32) a.recv_scales[(int64_t)rowd * a.nb + c * cpb + b] = sc[b];
            }
            if (in_sc) {
#pragma unroll
                for (int i = 0; i < kInScales; ++i) {
                    const int b = lane + 32 * i;
                    if (b < a.nb) a.recv_scales[(int64_t)rowd * a.nb + b] = isc[i];
                }
            } else if (a.in_scales != nullptr && c == 0) {
                for (int b = lane; b < a.nb; b += 32) a.recv_scales[(int64_t)rowd * a.nb + b] = a.in_scales[t * a.nb + b];
            }
            if (c == 0) {
                const int rd = __shfl_sync(kFull, rl, jd);
                if (lane < a.k) {
                    const bool local = a.expand ? (lane == jd && rl >= 0) : rl == rd;
                    if (a.recv_topk_idx) a.recv_topk_idx[(int64_t)rowd * a.k + lane] = local ? (int64_t)el : -1;
                    if (a.recv_topk_w) a.recv_topk_w[(int64_t)rowd * a.k + lane] = local ? wgt : 0.0f;
                }
                if (lane == 0 && a.recv_src) a.recv_src[rowd] = (int32_t)t;
            }
        }
        if constexpr (kFP8) {
            if (a.x_scales)
                for (int b = lane; b < nblk; b += 32) a.x_scales[t * a.nb + c * cpb + b] = sc[b];
        }
        if (lane == 0) {
            // the stage stored one unit ago is free once its bulk stores have read it;
            // it takes the next unit claimed by this warp
            if (i >= 1) {
                if (pf_pending) {   // bounded: the other warps only issue their prefetches
                    const uint64_t until = globaltimer_ns() + a.timeout_ns;
                    while (*reinterpret_cast<volatile int *>(&s_pf_warps) < warps && globaltimer_ns() < until)
                        __nanosleep(64);
                    pf_pending = false;
                }
                const int sp = s == 0 ? S - 1 : s - 1;
                const int64_t un = claim();
                ring[sp] = un;
                if (un >= 0) {
                    bulk_wait_read<1>();
                    issue_load(un, sp);
                }
            }
        }
        __syncwarp();
    }
    if (lane == 0) {
        if (!exhausted) retire();   // a warp that stopped early (timeout) still counts itself out
        bulk_wait_all();
    }
}

// ------------------------------------------------------------------ FP8 dispatch, row pipeline
//
// FP8 dispatch does arithmetic per element and writes rows half as wide as
// it reads, so it runs as a CTA-level pipeline over whole rows. One CTA per
// SM owns a contiguous token range:
//   producer warp  one cp.async.bulk per token row (bf16, 14 KB at H=7168)
//                  into an input ring;
//   worker warps   (row, slice) items round-robin, a slice being up to 8
//                  blocks of 128 channels. Each quarter-warp quantises one
//                  block (amax, scale = amax/448, E4M3 codes; 16 values per
//                  lane) and stores its 128 code bytes straight from
//                  registers to every destination row (16 bytes per lane,
//                  one full 128-byte line per quarter-warp store); the
//                  slice's scales go out as one coalesced 32-byte store per
//                  destination. The worker of slice 0 also writes the row
//                  metadata.
// There is no output staging and no single store warp, so the many small
// scattered writes (scales, metadata) spread over all worker warps. Input
// slots are handed back through mbarriers; every wait is bounded.

constexpr int kFp8MaxSlots = 16;
constexpr int kFp8SliceBlocks = 8;

struct Fp8Args {
    const uint8_t *x;
    int64_t row_bytes;           // H * 2
    int H, nb;                   // nb = H / 128
    int T, k, m, E;
    const int64_t *topk;
    const float *topk_w;
    const int32_t *dst_row;
    int capacity;
    uint8_t *recv_x;
    float *recv_scales;
    int64_t *recv_topk_idx;
    float *recv_topk_w;
    int32_t *recv_src;
    float *x_scales;
    int expand;                  // dst_row holds expand-mode rows (metadata: own entry only)
    int32_t *status;
    int n_in;                    // input ring slots
    int num_slices;
    int l2_hints;
    uint64_t timeout_ns;
    int loads_before_wait;       // the producer (input rows only) skips the dependency wait
    // tail balancing: tokens [0, static_tokens) are split into contiguous CTA
    // ranges; the rest are claimed one by one through pool[0] (pool[1] counts
    // CTAs that claim no more; the last of them zeroes both). nullptr: all dealt.
    unsigned int *pool;
    int static_tokens;
    TraceArgs trace;
};

__device__ __forceinline__ void mbar_arrive_plain(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 80 registers (no spills) allow 1 producer + 24 worker warps per SM
template <bool kPool>
__global__ void __maxnreg__(80) dispatch_fp8_rows_kernel(const Fp8Args a) {
    WarpTrace wt(a.trace, MOE_TRACE_DISPATCH_FP8_ROWS);
    MOE_PHASES(MOE_TRACE_DISPATCH_FP8_ROWS, 3);
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *in_full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *in_empty = in_full + kFp8MaxSlots;
    uint8_t *in_ring = smem + 2 * kFp8MaxSlots * 8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int NI = a.n_in, nsl = a.num_slices;

    // this CTA's rows: its contiguous range of the dealt tokens, then (with a
    // pool) tokens claimed one by one
    const int t_begin = (int)((int64_t)a.static_tokens * blockIdx.x / gridDim.x);
    const int t_end = (int)((int64_t)a.static_tokens * (blockIdx.x + 1) / gridDim.x);
    const int n = t_end - t_begin;

    __shared__ int s_next_item;
    __shared__ volatile int s_rows_issued;   // rows whose load the producer has armed
    __shared__ volatile int s_rows_total;    // rows of this CTA once the producer claims no more, else -1
    __shared__ int s_tok[kFp8MaxSlots];      // token of the row in each input slot
    if (threadIdx.x == 0) {
        for (int i = 0; i < NI; ++i) {
            mbar_init(&in_full[i], 1);
            mbar_init(&in_empty[i], (uint32_t)nsl);
        }
        fence_barrier_init();
        s_next_item = 0;
        s_rows_issued = 0;
        s_rows_total = kPool ? -1 : n;
    }
    __syncthreads();
    // launched right behind this library's layout, the input rows were complete
    // before this grid could launch: the producer, which reads nothing else,
    // starts at once; the workers read the layout's outputs and wait
    MOE_PHASE(1);
    if (!(a.loads_before_wait && warp == 0)) grid_dependency_wait();
    MOE_PHASE(2);
    grid_launch_dependents();
    if (!kPool && n <= 0) return;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = (a.l2_hints & 1) ? policy_evict_first() : policy_evict_normal();
            bool waited = !a.loads_before_wait;
            // pool claims are made one row ahead, so that a claim's round trip overlaps
            // the slot wait and arming of the row before it; the pool's counter is
            // zeroed by the launch before this one, so the first claim follows the wait
            int pending = -1;   // pool index claimed for the next row (-1: none)
            auto claim_ahead = [&]() {
                if (!waited) {
                    grid_dependency_wait();
                    waited = true;
                }
                pending = (int)atomicAdd(a.pool, 1u);
            };
            if (kPool && n == 0) claim_ahead();
            int j = 0;
            for (;; ++j) {
                int t = -1;
                if (j < n) t = t_begin + j;
                else if (pending >= 0 && pending < a.T - a.static_tokens) t = a.static_tokens + pending;
                if (t < 0) break;
                pending = -1;
                if (kPool && j + 1 >= n) claim_ahead();
                const int s = j % NI;
                if (j >= NI && !mbar_wait_bounded(&in_empty[s], (uint32_t)(((j / NI) - 1) & 1), a.timeout_ns)) {
                    report(a.status, MOE_ERR_TIMEOUT);
                    break;
                }
                if (kPool) s_tok[s] = t;
                mbar_arrive_expect_tx(&in_full[s], (uint32_t)a.row_bytes);
                bulk_load(in_ring + (size_t)s * a.row_bytes, a.x + (int64_t)t * a.row_bytes,
                          (uint32_t)a.row_bytes, &in_full[s], pol);
                __threadfence_block();
                s_rows_issued = j + 1;
            }
            __threadfence_block();
            s_rows_total = j;   // workers waiting on a later row stop
            // every claim of this CTA is made: count it out; the last CTA re-arms the pool
            if (kPool) {
                __threadfence();
                if (atomicAdd(a.pool + 1, 1u) == gridDim.x - 1) {
                    atomicExch(a.pool, 0u);
                    atomicExch(a.pool + 1, 0u);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- worker warps
    // Items (row j, slice sl) = q = j * nsl + sl are claimed in order from a
    // shared counter, each worker claiming its next item when it starts the
    // current one (so its rows can be prefetched): a worker whose items had
    // fewer destinations takes more of them.
    // (items < 2^31: checked on the host)
    auto claim = [&]() -> int {
        int q = 0;
        if (lane == 0) q = atomicAdd(&s_next_item, 1);
        return __shfl_sync(kFull, q, 0);
    };
    // the token of the CTA's row jq: known in advance for its dealt rows, for a
    // pool row once the producer has armed it (else -1); warp-uniform
    auto row_token = [&](int jq) -> int {
        if (!kPool || jq < n) return jq < n ? t_begin + jq : -1;
        int t = -1;
        if (lane == 0 && s_rows_issued > jq) {
            __threadfence_block();
            t = s_tok[jq % NI];
        }
        return __shfl_sync(kFull, t, 0);
    };
    // destination rows of a token, lanes < k, and, for the item of slice 0, the
    // token's routing (written as the rows' metadata); -1 / none for t < 0
    auto fetch_rows = [&](int t, bool first, int64_t &e, float &w) -> int {
        e = -1;
        w = 0.0f;
        if (t >= 0 && lane < a.k && first) {
            e = a.topk[(int64_t)t * a.k + lane];
            if (a.topk_w) w = a.topk_w[(int64_t)t * a.k + lane];
        }
        return (t >= 0 && lane < a.k) ? a.dst_row[(int64_t)t * a.k + lane] : -1;
    };
    int q = claim();
    int64_t e_next;
    float w_next;
    int t_next = row_token(q / nsl);   // the next item's token when known ahead (its rows prefetched)
    int row_next = fetch_rows(t_next, q % nsl == 0, e_next, w_next);
    while (true) {
        const int q_next = claim();
        const int j = q / nsl;
        const int sl = q - j * nsl;
        const int si = j % NI;
        const int t_pre = t_next;
        int row = row_next;
        int64_t e_cur = e_next;
        float w_cur = w_next;
        t_next = row_token(q_next / nsl);   // prefetched one item ahead (a pool row only once armed)
        row_next = fetch_rows(t_next, q_next % nsl == 0, e_next, w_next);
        // A slot's barrier is waited on by parity, which only names its current or
        // previous phase: wait (bounded) until row j's load has been armed, i.e.
        // the slot has left the phase of row j - NI, before waiting on the barrier
        // -- or until the producer has stopped short of row j (no more rows).
        bool ok = true, done = false;
        if (!kPool && j >= n) break;   // without a pool the CTA's rows are known in advance
        if (s_rows_issued <= j) {
            const uint64_t deadline = globaltimer_ns() + a.timeout_ns;
            while (s_rows_issued <= j) {
                const int total = s_rows_total;
                if (total >= 0 && j >= total) {
                    done = true;
                    break;
                }
                if (globaltimer_ns() > deadline) {
                    ok = false;
                    break;
                }
                if (kPool && j >= n) __nanosleep(128);   // a pool row not yet claimed: leave the issue slots to the workers
            }
        }
        if (kPool && __any_sync(kFull, done)) break;
        __threadfence_block();
        const int t = (!kPool || j < n) ? t_begin + j : s_tok[si];
        if (kPool && t_pre < 0) row = fetch_rows(t, sl == 0, e_cur, w_cur);   // a pool row not armed at prefetch time
        if (row >= a.capacity) {
            if (sl == 0) report(a.status, MOE_ERR_CAPACITY);
            row = -1;
        }
        const unsigned dmask = __ballot_sync(kFull, row >= 0);
        ok = ok && mbar_wait_bounded(&in_full[si], (uint32_t)((j / NI) & 1), a.timeout_ns);
        if (!__all_sync(kFull, ok)) {
            if (lane == 0) report(a.status, MOE_ERR_TIMEOUT);
            break;
        }
        const uint8_t *src = in_ring + (size_t)si * a.row_bytes;
        const int b_begin = sl * kFp8SliceBlocks;
        const int b_end = min(a.nb, b_begin + kFp8SliceBlocks);
        const int quarter = lane >> 3, ql = lane & 7;
        float my_scale = 0.0f;            // lane l < blocks of the slice: scale of block b_begin + l
        for (int b0 = b_begin; b0 < b_end; b0 += 4) {
            const int b = b0 + quarter;
            const bool act = b < b_end;
            uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
            if (act) {
                lo = *reinterpret_cast<const uint4 *>(src + (size_t)b * 256 + ql * 32);
                hi = *reinterpret_cast<const uint4 *>(src + (size_t)b * 256 + ql * 32 + 16);
            }
            uint4 q16;
            const float scale = quantize_lane16(lo, hi, q16);
            // block b0 + i's scale sits in lane 8 i; lane (b0 - b_begin) + i keeps it
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float si_ = __shfl_sync(kFull, scale, 8 * i);
                if (lane == b0 - b_begin + i) my_scale = si_;
            }
            for (unsigned mm = dmask; mm; mm &= mm - 1) {
                const int rowd = __shfl_sync(kFull, row, __ffs(mm) - 1);
                if (act) *reinterpret_cast<uint4 *>(a.recv_x + (int64_t)rowd * a.H + (size_t)b * 128 + ql * 16) = q16;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_plain(&in_empty[si]);   // the row's slice has been read
        // scales of the slice: one coalesced store per destination row (and the source-side copy)
        const int nblk = b_end - b_begin;
        for (unsigned mm = dmask; mm; mm &= mm - 1) {
            const int rowd = __shfl_sync(kFull, row, __ffs(mm) - 1);
            if (lane < nblk) a.recv_scales[(int64_t)rowd * a.nb + b_begin + lane] = my_scale;
        }
        if (a.x_scales && lane < nblk) a.x_scales[(int64_t)t * a.nb + b_begin + lane] = my_scale;
        // row metadata, written by the worker of slice 0
        if (sl == 0) {
            int rl = -1, el = 0;
            const float wgt = w_cur;
            if (lane < a.k && e_cur >= 0 && e_cur < a.E) {
                rl = (int)e_cur / a.m;
                el = (int)e_cur - rl * a.m;
            }
            for (unsigned mm = dmask; mm; mm &= mm - 1) {
                const int jd = __ffs(mm) - 1;
                const int rowd = __shfl_sync(kFull, row, jd);
                const int rd = __shfl_sync(kFull, rl, jd);
                if (lane < a.k) {
                    const bool local = a.expand ? (lane == jd && rl >= 0) : rl == rd;
                    if (a.recv_topk_idx) a.recv_topk_idx[(int64_t)rowd * a.k + lane] = local ? (int64_t)el : -1;
                    if (a.recv_topk_w) a.recv_topk_w[(int64_t)rowd * a.k + lane] = local ? wgt : 0.0f;
                }
                if (lane == 0 && a.recv_src) a.recv_src[rowd] = (int32_t)t;
            }
        }
        q = q_next;
    }
}

inline int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

constexpr int kFusedMaxTokens = 1024;   // largest batch whose layout every CTA of a fused launch computes

// Fields shared by every dispatch launch.
DispatchArgs base_args(const DispatchLaunch &L) {
    const Tuning &tu = tuning();
    const bool fp8 = L.mode == MOE_DISPATCH_QUANTIZE_FP8;      // quantise in the kernel
    const bool fp8_in = L.mode == MOE_DISPATCH_FP8;             // relay E4M3 bytes and their scales
    DispatchArgs a = {};
    a.trace = trace_args();
    a.x = static_cast<const uint8_t *>(L.x);
    a.row_bytes = fp8_in ? (int64_t)L.hidden : (int64_t)L.hidden * 2;
    a.k = L.num_topk;
    a.m = L.num_experts / L.num_ranks;
    a.E = L.num_experts;
    a.topk = L.topk_idx;
    a.topk_w = L.topk_weights;
    a.dst_row = L.token_dst_row;
    a.loads_before_wait = L.loads_before_wait ? 1 : 0;
    a.prefetch_units = (L.loads_before_wait || tu.dispatch_prefetch_always) ? tu.dispatch_prefetch : 0;
    a.prefetch_keep = tu.dispatch_prefetch_keep;
    a.pool = L.pool;
    a.capacity = L.recv_capacity;
    a.recv_x = static_cast<uint8_t *>(L.recv_x);
    a.recv_row_bytes = (fp8 || fp8_in) ? (int64_t)L.hidden : (int64_t)L.hidden * 2;
    a.recv_scales = L.recv_x_scales;
    a.recv_topk_idx = L.recv_topk_idx;
    a.recv_topk_w = L.recv_topk_weights;
    a.recv_src = L.recv_src_idx;
    a.x_scales = fp8 ? L.x_scales : nullptr;
    a.in_scales = fp8_in ? L.x_scales : nullptr;
    a.nb = L.hidden / 128;
    a.expand = L.expand ? 1 : 0;
    a.status = L.status;
    a.l2_hints = tu.l2_hints;
    a.timeout_ns = kDefaultWaitNs;
    a.T = L.num_tokens;
    a.R = L.num_ranks;
    return a;
}

// Chunking, per-warp shared memory, warps per CTA and grid of the chunked
// relay kernel; `extra` bytes of shared memory follow the warps' regions.
int chunked_config(DispatchArgs &a, bool fp8, int num_tokens, size_t extra, int &warps, size_t &smem, int &grid) {
    const Tuning &tu = tuning();
    const int64_t align = fp8 ? 256 : 16;
    const int64_t max_chunk = std::max<int64_t>(align, std::min<int64_t>(65536, tu.dispatch_chunk) / align * align);
    int64_t chunk_cap = max_chunk;
    // a small batch: smaller chunks (down to 2 KB) until there are 4 units per SM
    while (tu.spread_small && chunk_cap > 2048 &&
           (int64_t)num_tokens * ((a.row_bytes + chunk_cap - 1) / chunk_cap) < 4LL * device_sm_count())
        chunk_cap = std::max<int64_t>(2048, chunk_cap / 2 / align * align);
    const int64_t nch = (a.row_bytes + chunk_cap - 1) / chunk_cap;
    a.chunk_bytes = (int)round_up((a.row_bytes + nch - 1) / nch, align);
    a.num_chunks = (int)((a.row_bytes + a.chunk_bytes - 1) / a.chunk_bytes);
    a.num_units = (int64_t)num_tokens * a.num_chunks;
    // behind this library's layout (stage loads issued before the dependency wait) a
    // different shape measured faster: 2 warps x 4 stages, two CTAs per SM
    const int want_warps = a.loads_before_wait ? tu.ld_dispatch_warps : tu.dispatch_warps;
    const int want_stages = a.loads_before_wait ? tu.ld_dispatch_stages : tu.dispatch_stages;
    a.stages = std::min(kMaxStages, std::max(3, want_stages));   // the unit ring needs three
    // stages take at most ~200 KB, so that some L1 cache is left (a full 227 KB of
    // stages measured slower)
    const int64_t room = std::min<int64_t>((int64_t)device_smem_optin(), (int64_t)tu.dispatch_smem) -
                         (int64_t)round_up((int64_t)extra, 128);
    auto warp_bytes = [&](int stages) {
        int64_t b = kBarBytes + (int64_t)stages * a.chunk_bytes;
        if (fp8) b += (int64_t)stages * (a.chunk_bytes / 2) + round_up((int64_t)stages * (a.chunk_bytes / 256) * 4, 128);
        return round_up(b, 128);
    };
    // fewer stages (down to three) before fewer warps than requested
    while (a.stages > 3 && room / warp_bytes(a.stages) < want_warps) --a.stages;
    const int64_t per_warp = warp_bytes(a.stages);
    a.warp_smem = (int)per_warp;
    // as many of the requested warps as fit in one CTA's shared memory
    const int fit = (int)std::min<int64_t>(16, room / per_warp);
    if (fit < 1) return MOE_ERR_INVALID_ARG;
    warps = std::max(1, std::min(fit, want_warps));
    // a small batch: fewer warps per CTA, so that its units spread over every SM
    if (tu.spread_small) {
        const int64_t per_sm = (a.num_units + device_sm_count() - 1) / device_sm_count();
        warps = (int)std::max<int64_t>(1, std::min<int64_t>(warps, per_sm));
    }
    smem = (size_t)per_warp * warps + (extra ? (size_t)round_up((int64_t)extra, 128) : 0);
    a.fl_off = (size_t)per_warp * warps;
    int ctas_per_sm = (int)std::max<size_t>(1, device_smem_per_sm() / (smem + 1024));
    if (tu.ctas_per_sm > 0) ctas_per_sm = std::min(ctas_per_sm, tu.ctas_per_sm);
    const int64_t want = (a.num_units + warps - 1) / warps;
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)device_sm_count() * ctas_per_sm));
    // tail balancing pays off only with several units per CTA
    const int pool_pct = tu.dispatch_pool;
    if (a.pool != nullptr && pool_pct > 0 && pool_pct < 100 && a.num_units >= 8 * (int64_t)grid) {
        a.static_units = a.num_units * (100 - pool_pct) / 100;
        // claims made before the dependency wait (the first stage of every warp) stay in the
        // dealt units: the pool's counter may be zeroed by the launch before this one
        if (a.loads_before_wait)
            a.static_units = std::max(a.static_units, std::min(a.num_units, (int64_t)grid * warps * a.stages));
    } else {
        a.pool = nullptr;
        a.static_units = a.num_units;
    }
    // the L2 prefetch: at most dispatch_prefetch_l2_pct of L2 held evict-last by
    // the grid, and none at all when the first stage loads already take every
    // dealt unit and no pool unit would be prefetched (small batches)
    if (a.prefetch_units > 0) {
        const int pct = a.loads_before_wait ? tu.dispatch_prefetch_l2_pct : tu.dispatch_prefetch_l2_pct_alone;
        const int64_t budget = (int64_t)device_l2_bytes() * pct / 100;
        a.prefetch_units = std::min<int64_t>(a.prefetch_units, budget / ((int64_t)grid * a.chunk_bytes));
        const int64_t first = (int64_t)warps * a.stages;
        const int64_t max_dealt = (a.static_units + grid - 1) / grid;
        const bool pool_prefetch = a.pool != nullptr && a.static_units >= (int64_t)grid * first;
        if (max_dealt <= first && !pool_prefetch) a.prefetch_units = 0;
    }
    return MOE_OK;
}

template <bool kFP8, bool kFused>
int launch_chunked(const DispatchArgs &a, int warps, size_t smem, int grid, cudaStream_t st) {
    const void *fn = (const void *)dispatch_kernel<kFP8, kFused>;
    if (ensure_dynamic_smem(fn, smem) != MOE_OK) return MOE_ERR_CUDA;
    return launch_kernel(dispatch_kernel<kFP8, kFused>, dim3(grid), dim3(warps * 32), smem, st, tuning().overlap != 0,
                         a) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

}  // namespace

int launch_dispatch(const DispatchLaunch &L) {
    if (L.num_tokens == 0) return MOE_OK;
    const Tuning &tu = tuning();
    const bool fp8 = L.mode == MOE_DISPATCH_QUANTIZE_FP8;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(L.stream);
    DispatchArgs a = base_args(L);

    if (fp8 && tu.fp8_rows) {
        Fp8Args f;
        f.trace = a.trace;
        f.x = a.x;
        f.row_bytes = a.row_bytes;
        f.H = L.hidden;
        f.nb = L.hidden / 128;
        f.T = L.num_tokens;
        f.k = a.k; f.m = a.m; f.E = a.E;
        f.topk = a.topk; f.topk_w = a.topk_w; f.dst_row = a.dst_row; f.capacity = a.capacity;
        f.recv_x = a.recv_x; f.recv_scales = a.recv_scales; f.recv_topk_idx = a.recv_topk_idx;
        f.recv_topk_w = a.recv_topk_w; f.recv_src = a.recv_src; f.x_scales = a.x_scales;
        f.expand = a.expand;
        f.status = a.status;
        f.num_slices = (f.nb + kFp8SliceBlocks - 1) / kFp8SliceBlocks;
        f.l2_hints = a.l2_hints;
        f.loads_before_wait = a.loads_before_wait;
        f.timeout_ns = a.timeout_ns;
        const int grid_rows = std::max(1, std::min(L.num_tokens, device_sm_count()));
        // tail balancing (a cleared counter at hand, long runs): the last fp8_rows_pool
        // percent of the tokens are claimed one by one. With fewer rows per CTA the
        // SMs finish close together and the pool's per-row costs are not repaid
        // (4096 tokens over 152 SMs: 42.5 against 41.2 us; 8192: 95.2 against 105.5 us).
        f.pool = (a.pool != nullptr && tu.fp8_rows_pool > 0 && tu.fp8_rows_pool < 100 &&
                  L.num_tokens >= tu.fp8_rows_pool_min_rows * grid_rows) ? a.pool : nullptr;
        f.static_tokens = f.pool ? (int)((int64_t)L.num_tokens * (100 - tu.fp8_rows_pool) / 100) : L.num_tokens;
        const size_t head = 2 * kFp8MaxSlots * 8;
        const size_t optin = device_smem_optin();
        f.n_in = std::max(2, std::min(kFp8MaxSlots, tu.fp8_in_slots));
        while (head + (size_t)f.n_in * f.row_bytes > optin && f.n_in > 2) --f.n_in;
        const size_t smem = head + (size_t)f.n_in * f.row_bytes;
        const int64_t max_cta_items = (f.pool ? (int64_t)L.num_tokens
                                              : ((int64_t)L.num_tokens + device_sm_count() - 1) / device_sm_count()) *
                                          f.num_slices + 64;
        if (smem <= optin && f.row_bytes < (1 << 20) && max_cta_items < ((int64_t)1 << 31)) {
            void (*rows_kernel)(const Fp8Args) = f.pool ? dispatch_fp8_rows_kernel<true> : dispatch_fp8_rows_kernel<false>;
            if (ensure_dynamic_smem((const void *)rows_kernel, smem) != MOE_OK) return MOE_ERR_CUDA;
            // as many of the requested workers as the kernel's register use allows in one CTA
            static int max_threads[64][2] = {};
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
            int &mt = max_threads[dev][f.pool ? 1 : 0];
            if (mt == 0) {
                cudaFuncAttributes fa;
                if (cudaFuncGetAttributes(&fa, (const void *)rows_kernel) != cudaSuccess) return MOE_ERR_CUDA;
                mt = fa.maxThreadsPerBlock;
            }
            const int workers = std::max(1, std::min({24, tu.fp8_quant_warps, mt / 32 - 1}));
            const int grid = grid_rows;
            return launch_kernel(rows_kernel, dim3(grid), dim3((workers + 1) * 32), smem, st,
                                 tu.overlap != 0, f) == cudaSuccess
                       ? MOE_OK
                       : MOE_ERR_CUDA;
        }
        // rows too large for the ring: fall through to the chunked kernel
    }

    int warps = 0, grid = 0;
    size_t smem = 0;
    const int rc = chunked_config(a, fp8, L.num_tokens, 0, warps, smem, grid);
    if (rc != MOE_OK) return rc;
    return fp8 ? launch_chunked<true, false>(a, warps, smem, grid, st)
               : launch_chunked<false, false>(a, warps, smem, grid, st);
}

int launch_layout_dispatch(const LayoutLaunch &Ll, const DispatchLaunch &L) {
    const int T = L.num_tokens;
    const bool fp8 = L.mode == MOE_DISPATCH_QUANTIZE_FP8;
    const Tuning &tu = tuning();
    bool fused = tu.fused_small && T > 0 && T <= kFusedMaxTokens && !L.expand;
    DispatchArgs a = base_args(L);
    int warps = 0, grid = 0;
    size_t smem = 0;
    if (fused) {
        a.fl_words = (T + 31) / 32;
        a.fl_out = Ll.out;
        const size_t extra = fused_smem(T, L.num_ranks, L.num_experts, L.num_topk).total;
        // every CTA computes the whole layout with its own warps: with fewer than
        // fused_min_warps per CTA that costs more than the separate layout launch
        // (128 tokens of 512-byte rows: one warp per CTA, 20.6 against 17.7 us)
        fused = chunked_config(a, fp8, T, extra, warps, smem, grid) == MOE_OK && warps >= tu.fused_min_warps;
    }
    if (!fused) {   // two launches: layout, then dispatch, which loads input rows while the layout runs
        LayoutLaunch l2 = Ll;
        DispatchLaunch d2 = L;
        l2.early_dependents = tu.overlap != 0;
        d2.loads_before_wait = tu.overlap != 0;
        d2.pool = layout_spare_counter(l2);
        const int rc = launch_layout(l2);
        return rc != MOE_OK ? rc : launch_dispatch(d2);
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(L.stream);
    return fp8 ? launch_chunked<true, true>(a, warps, smem, grid, st)
               : launch_chunked<false, true>(a, warps, smem, grid, st);
}

}  // namespace moe
