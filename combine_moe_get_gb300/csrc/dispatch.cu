// dispatch.cu -- copy each token's row once per distinct destination rank.
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
    int nb;                   // scale blocks per row (H / 128), FP8
    int32_t *status;
    int chunk_bytes;          // input bytes per unit; multiple of 16 (FP8: of 256)
    int num_chunks;           // units per token
    int64_t num_units;
    int stages;
    int warp_smem;
    int l2_hints;
    uint64_t timeout_ns;
};

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// x / scale as the IEEE fp32 quotient, as far as its E4M3 code can tell.
// q0 = RN(x * RN(1/scale)) is within 3 fp32 ulps of RN(x / scale) (two
// roundings of relative size <= 2^-24 each against one). E4M3 rounding (3
// mantissa bits, RNE) is a step function of its fp32 argument whose steps sit
// at midpoints, whose fp32 mantissa has low 20 bits == 0x80000 in the normal
// range. So when q0 is more than 4 ulps from a midpoint and |q0| >= 2^-6 (below
// that the E4M3 quantum is fixed), q0 and RN(x / scale) get the same code;
// otherwise the quotient must be taken with the IEEE division.
__device__ __forceinline__ bool e4m3_needs_exact(float q0) {
    const uint32_t b = __float_as_uint(q0) & 0x7fffffffu;
    const uint32_t m = b & 0xfffffu;
    return ((m + 4u - 0x80000u) <= 8u) || (b < 0x3c800000u);   // |m - 0x80000| <= 4, or |q0| < 2^-6
}

// Quantise one 128-channel block held by a half-warp (16 lanes x 8 values).
// Returns the block's scale; writes the 8 codes of this lane to `q8`.
__device__ __forceinline__ float quantize_lane8(const uint4 v, uint2 &q8) {
    float f[8];
    f[0] = bf16_bits_to_float(v.x & 0xffffu); f[1] = bf16_bits_to_float(v.x >> 16);
    f[2] = bf16_bits_to_float(v.y & 0xffffu); f[3] = bf16_bits_to_float(v.y >> 16);
    f[4] = bf16_bits_to_float(v.z & 0xffffu); f[5] = bf16_bits_to_float(v.z >> 16);
    f[6] = bf16_bits_to_float(v.w & 0xffffu); f[7] = bf16_bits_to_float(v.w >> 16);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    const float scale = amax / 448.0f;   // IEEE division (no fast-math)
    uint32_t c[4];
    if (scale == 0.0f) {
        c[0] = c[1] = c[2] = c[3] = 0u;
    } else {
        const float rcp = __frcp_rn(scale);
        float q[8];
        unsigned exact = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            q[i] = f[i] * rcp;
            exact |= e4m3_needs_exact(q[i]) ? (1u << i) : 0u;
        }
        if (exact) {                         // rare: near a rounding midpoint or tiny
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if ((exact >> i) & 1u) q[i] = f[i] / scale;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            c[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(q[2 * i], q[2 * i + 1]), __NV_SATFINITE,
                                                      __NV_E4M3);   // .x -> low byte
    }
    q8.x = c[0] | (c[1] << 16);
    q8.y = c[2] | (c[3] << 16);
    return scale;
}

template <bool kFP8>
__global__ void __launch_bounds__(512) dispatch_kernel(const DispatchArgs a) {
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

    const int64_t gw = (int64_t)blockIdx.x * warps + warp;
    const int64_t GW = (int64_t)gridDim.x * warps;
    if (gw >= a.num_units) return;
    const int64_t n_w = (a.num_units - 1 - gw) / GW + 1;

    const uint64_t pol_load = (a.l2_hints & 1) ? policy_evict_first() : policy_evict_normal();
    const uint64_t pol_store = (a.l2_hints & 2) ? policy_evict_first() : policy_evict_normal();

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();

    auto issue_load = [&](int64_t i) {   // lane 0
        const int64_t u = gw + i * GW;
        const int64_t t = u / a.num_chunks;
        const int64_t off = (u - t * a.num_chunks) * (int64_t)chunk;
        const uint32_t nbytes = (uint32_t)min((int64_t)chunk, a.row_bytes - off);
        const int s = (int)(i % S);
        mbar_arrive_expect_tx(&bars[s], nbytes);
        bulk_load(in_stage + (size_t)s * chunk, a.x + t * a.row_bytes + off, nbytes, &bars[s], pol_load);
    };
    if (lane == 0)
        for (int64_t i = 0; i < min((int64_t)S, n_w); ++i) issue_load(i);

    // receive rows (and, for the first chunk, the routing) of the next unit, prefetched one unit ahead
    auto fetch = [&](int64_t i, int &row, int64_t &e, float &w) {
        const int64_t u = gw + i * GW;
        const int64_t t = u / a.num_chunks;
        const bool first = (u - t * a.num_chunks) == 0;
        row = -1; e = -1; w = 0.0f;
        if (lane < a.k) {
            row = a.dst_row[t * a.k + lane];
            if (first) {
                e = a.topk[t * a.k + lane];
                if (a.topk_w) w = a.topk_w[t * a.k + lane];
            }
        }
    };
    int row_n; int64_t e_n; float w_n;
    fetch(0, row_n, e_n, w_n);

    for (int64_t i = 0; i < n_w; ++i) {
        const int s = (int)(i % S);
        const uint32_t parity = (uint32_t)((i / S) & 1);
        const int64_t u = gw + i * GW;
        const int64_t t = u / a.num_chunks;
        const int c = (int)(u - t * a.num_chunks);
        const int64_t off = (int64_t)c * chunk;
        const int nbytes = (int)min((int64_t)chunk, a.row_bytes - off);

        int row = row_n;
        const int64_t e = e_n;
        const float wgt = w_n;
        if (i + 1 < n_w) fetch(i + 1, row_n, e_n, w_n);
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

        unsigned mm = dmask;
        while (mm) {
            const int jd = __ffs(mm) - 1;
            mm &= mm - 1;
            const int rowd = __shfl_sync(kFull, row, jd);
            if (lane == 0)
                bulk_store(a.recv_x + (int64_t)rowd * a.recv_row_bytes + out_off, src, (uint32_t)out_bytes, pol_store);
            if constexpr (kFP8) {
                for (int b = lane; b < nblk; b += 32) a.recv_scales[(int64_t)rowd * a.nb + c * cpb + b] = sc[b];
            }
            if (c == 0) {
                const int64_t ed = __shfl_sync(kFull, e, jd);
                const int rd = (int)(ed / a.m);
                if (lane < a.k) {
                    const bool local = e >= 0 && e < a.E && (int)(e / a.m) == rd;
                    if (a.recv_topk_idx) a.recv_topk_idx[(int64_t)rowd * a.k + lane] = local ? e - (int64_t)rd * a.m : -1;
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
            bulk_commit();
            // the stage stored one unit ago is free once its bulk stores have read it
            if (i >= 1 && i - 1 + S < n_w) {
                bulk_wait_read<1>();
                issue_load(i - 1 + S);
            }
        }
        __syncwarp();
    }
    if (lane == 0) bulk_wait_all();
}

// ------------------------------------------------------------------ FP8 dispatch, row pipeline
//
// FP8 dispatch does real arithmetic per element, so it runs as a CTA-level
// pipeline over whole rows. One CTA per SM owns a contiguous token range:
//   producer warp    one cp.async.bulk per token row (bf16, 14 KB at H=7168)
//                    into an input ring;
//   quantiser warps  (row, slice) items round-robin, a slice being up to 8
//                    blocks of 128 channels; each half-warp quantises one block
//                    (amax, scale = amax/448, E4M3 codes) into an output ring
//                    slot holding the row's codes followed by its scales;
//   store warp       one cp.async.bulk of the code row (and of the scale row
//                    when its pitch is a multiple of 16 bytes) per destination
//                    rank, plus the per-row metadata.
// Ring slots are handed back through mbarriers; every wait is bounded.

constexpr int kFp8MaxSlots = 16;

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
    int32_t *status;
    int n_in, n_out;             // ring slots
    int slice_blocks, num_slices;
    int out_slot_bytes;          // H + scale bytes, rounded to 16
    int scales_bulk;             // scale rows can be bulk-stored (nb * 4 % 16 == 0)
    int l2_hints;
    uint64_t timeout_ns;
};

__device__ __forceinline__ void mbar_arrive_plain(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__global__ void __launch_bounds__(32 * 18, 1) dispatch_fp8_rows_kernel(const Fp8Args a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *in_full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *in_empty = in_full + kFp8MaxSlots;
    uint64_t *out_full = in_empty + kFp8MaxSlots;
    uint64_t *out_empty = out_full + kFp8MaxSlots;
    uint8_t *in_ring = smem + 4 * kFp8MaxSlots * 8;
    uint8_t *out_ring = in_ring + (size_t)a.n_in * a.row_bytes;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int quantizers = (blockDim.x >> 5) - 2;
    const int NI = a.n_in, NO = a.n_out, nsl = a.num_slices;

    const int t_begin = (int)((int64_t)a.T * blockIdx.x / gridDim.x);
    const int t_end = (int)((int64_t)a.T * (blockIdx.x + 1) / gridDim.x);
    const int n = t_end - t_begin;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NI; ++i) {
            mbar_init(&in_full[i], 1);
            mbar_init(&in_empty[i], (uint32_t)nsl);
        }
        for (int i = 0; i < NO; ++i) {
            mbar_init(&out_full[i], (uint32_t)nsl);
            mbar_init(&out_empty[i], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (n <= 0) return;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = (a.l2_hints & 1) ? policy_evict_first() : policy_evict_normal();
            for (int j = 0; j < n; ++j) {
                const int s = j % NI;
                if (j >= NI && !mbar_wait_bounded(&in_empty[s], (uint32_t)(((j / NI) - 1) & 1), a.timeout_ns)) {
                    report(a.status, MOE_ERR_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&in_full[s], (uint32_t)a.row_bytes);
                bulk_load(in_ring + (size_t)s * a.row_bytes, a.x + (int64_t)(t_begin + j) * a.row_bytes,
                          (uint32_t)a.row_bytes, &in_full[s], pol);
            }
        }
        return;
    }

    if (warp == 1) {
        // ------------------------------------------------------------ store warp
        const uint64_t pol = (a.l2_hints & 2) ? policy_evict_first() : policy_evict_normal();
        const int scale_bytes = a.nb * 4;
        int row_n = -1;
        int64_t e_n = -1;
        float w_n = 0.0f;
        if (lane < a.k) {
            const int64_t base = (int64_t)t_begin * a.k + lane;
            row_n = a.dst_row[base];
            e_n = a.topk[base];
            if (a.topk_w) w_n = a.topk_w[base];
        }
        bool failed = false;
        for (int j = 0; j < n; ++j) {
            const int t = t_begin + j;
            const int o = j % NO;
            int row = row_n;
            const int64_t e = e_n;
            const float wgt = w_n;
            if (j + 1 < n && lane < a.k) {
                const int64_t base = (int64_t)(t + 1) * a.k + lane;
                row_n = a.dst_row[base];
                e_n = a.topk[base];
                if (a.topk_w) w_n = a.topk_w[base];
            }
            if (row >= a.capacity) {
                report(a.status, MOE_ERR_CAPACITY);
                row = -1;
            }
            const unsigned dmask = __ballot_sync(kFull, row >= 0);
            const bool ok = mbar_wait_bounded(&out_full[o], (uint32_t)((j / NO) & 1), a.timeout_ns);
            if (!__all_sync(kFull, ok)) {
                if (lane == 0) report(a.status, MOE_ERR_TIMEOUT);
                failed = true;
                break;
            }
            const uint8_t *codes = out_ring + (size_t)o * a.out_slot_bytes;
            const float *sc = reinterpret_cast<const float *>(codes + a.H);
            unsigned mm = dmask;
            while (mm) {
                const int jd = __ffs(mm) - 1;
                mm &= mm - 1;
                const int rowd = __shfl_sync(kFull, row, jd);
                if (lane == 0) {
                    bulk_store(a.recv_x + (int64_t)rowd * a.H, codes, (uint32_t)a.H, pol);
                    if (a.scales_bulk)
                        bulk_store(a.recv_scales + (int64_t)rowd * a.nb, sc, (uint32_t)scale_bytes, pol);
                }
                if (!a.scales_bulk)
                    for (int b = lane; b < a.nb; b += 32) a.recv_scales[(int64_t)rowd * a.nb + b] = sc[b];
                const int64_t ed = __shfl_sync(kFull, e, jd);
                const int rd = (int)(ed / a.m);
                if (lane < a.k) {
                    const bool local = e >= 0 && e < a.E && (int)(e / a.m) == rd;
                    if (a.recv_topk_idx) a.recv_topk_idx[(int64_t)rowd * a.k + lane] = local ? e - (int64_t)rd * a.m : -1;
                    if (a.recv_topk_w) a.recv_topk_w[(int64_t)rowd * a.k + lane] = local ? wgt : 0.0f;
                }
                if (lane == 0 && a.recv_src) a.recv_src[rowd] = (int32_t)t;
            }
            __syncwarp();
            if (lane == 0) {
                bulk_commit();
                if (j >= 1) {                    // the previous row's stores have read their slot
                    bulk_wait_read<1>();
                    mbar_arrive_plain(&out_empty[(j - 1) % NO]);
                }
            }
            __syncwarp();
        }
        if (lane == 0) {
            bulk_wait_all();
            if (!failed) mbar_arrive_plain(&out_empty[(n - 1) % NO]);
        }
        return;
    }

    // ---------------------------------------------------------------- quantiser warps
    const int qw = warp - 2;
    const int half = lane >> 4, hl = lane & 15;
    const int64_t n_items = (int64_t)n * nsl;
    for (int64_t q = qw; q < n_items; q += quantizers) {
        const int j = (int)(q / nsl);
        const int sl = (int)(q - (int64_t)j * nsl);
        const int t = t_begin + j;
        const int si = j % NI, so = j % NO;
        bool ok = mbar_wait_bounded(&in_full[si], (uint32_t)((j / NI) & 1), a.timeout_ns);
        if (ok && j >= NO) ok = mbar_wait_bounded(&out_empty[so], (uint32_t)(((j / NO) - 1) & 1), a.timeout_ns);
        if (!__all_sync(kFull, ok)) {
            if (lane == 0) report(a.status, MOE_ERR_TIMEOUT);
            break;
        }
        const uint8_t *src = in_ring + (size_t)si * a.row_bytes;
        uint8_t *codes = out_ring + (size_t)so * a.out_slot_bytes;
        float *sc = reinterpret_cast<float *>(codes + a.H);
        const int b_begin = sl * a.slice_blocks;
        const int b_end = min(a.nb, b_begin + a.slice_blocks);
        for (int b0 = b_begin; b0 < b_end; b0 += 2) {
            const int b = b0 + half;
            const bool act = b < b_end;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (act) v = *reinterpret_cast<const uint4 *>(src + (size_t)b * 256 + hl * 16);
            uint2 q8;
            const float scale = quantize_lane8(v, q8);
            if (act) {
                *reinterpret_cast<uint2 *>(codes + (size_t)b * 128 + hl * 8) = q8;
                if (hl == 0) {
                    sc[b] = scale;
                    if (a.x_scales) a.x_scales[(int64_t)t * a.nb + b] = scale;
                }
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_plain(&in_empty[si]);
            mbar_arrive_plain(&out_full[so]);
        }
    }
}

inline int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

}  // namespace

int launch_dispatch(const DispatchLaunch &L) {
    if (L.num_tokens == 0) return MOE_OK;
    const Tuning &tu = tuning();
    const bool fp8 = L.quantize_fp8 != 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(L.stream);

    DispatchArgs a;
    a.x = static_cast<const uint8_t *>(L.x);
    a.row_bytes = (int64_t)L.hidden * 2;
    a.k = L.num_topk;
    a.m = L.num_experts / L.num_ranks;
    a.E = L.num_experts;
    a.topk = L.topk_idx;
    a.topk_w = L.topk_weights;
    a.dst_row = L.token_dst_row;
    a.capacity = L.recv_capacity;
    a.recv_x = static_cast<uint8_t *>(L.recv_x);
    a.recv_row_bytes = fp8 ? (int64_t)L.hidden : (int64_t)L.hidden * 2;
    a.recv_scales = L.recv_x_scales;
    a.recv_topk_idx = L.recv_topk_idx;
    a.recv_topk_w = L.recv_topk_weights;
    a.recv_src = L.recv_src_idx;
    a.x_scales = L.x_scales;
    a.nb = L.hidden / 128;
    a.status = L.status;
    a.l2_hints = tu.l2_hints;
    a.timeout_ns = kDefaultWaitNs;

    if (fp8 && tu.fp8_rows) {
        Fp8Args f;
        f.x = a.x;
        f.row_bytes = a.row_bytes;
        f.H = L.hidden;
        f.nb = L.hidden / 128;
        f.T = L.num_tokens;
        f.k = a.k; f.m = a.m; f.E = a.E;
        f.topk = a.topk; f.topk_w = a.topk_w; f.dst_row = a.dst_row; f.capacity = a.capacity;
        f.recv_x = a.recv_x; f.recv_scales = a.recv_scales; f.recv_topk_idx = a.recv_topk_idx;
        f.recv_topk_w = a.recv_topk_w; f.recv_src = a.recv_src; f.x_scales = a.x_scales;
        f.status = a.status;
        f.slice_blocks = 8;
        f.num_slices = (f.nb + f.slice_blocks - 1) / f.slice_blocks;
        f.out_slot_bytes = (int)round_up((int64_t)f.H + (int64_t)f.nb * 4, 16);
        f.scales_bulk = ((f.nb * 4) % 16 == 0) ? 1 : 0;
        f.l2_hints = a.l2_hints;
        f.timeout_ns = a.timeout_ns;
        const size_t head = 4 * kFp8MaxSlots * 8;
        const size_t optin = device_smem_optin();
        f.n_out = std::max(2, std::min(kFp8MaxSlots, tu.fp8_out_slots));
        f.n_in = std::max(2, std::min(kFp8MaxSlots, tu.fp8_in_slots));
        // shrink the rings until they fit (the input ring first, keeping at least two slots each)
        while (head + (size_t)f.n_in * f.row_bytes + (size_t)f.n_out * f.out_slot_bytes > optin && f.n_in > 2) --f.n_in;
        while (head + (size_t)f.n_in * f.row_bytes + (size_t)f.n_out * f.out_slot_bytes > optin && f.n_out > 2) --f.n_out;
        const size_t smem = head + (size_t)f.n_in * f.row_bytes + (size_t)f.n_out * f.out_slot_bytes;
        if (smem <= optin) {
            if (ensure_dynamic_smem((const void *)dispatch_fp8_rows_kernel, smem) != MOE_OK) return MOE_ERR_CUDA;
            const int qwarps = std::max(1, std::min(16, tu.fp8_quant_warps));
            const int grid = std::max(1, std::min(L.num_tokens, device_sm_count()));
            dispatch_fp8_rows_kernel<<<grid, (qwarps + 2) * 32, smem, st>>>(f);
            return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
        }
        // rows too large for the rings: fall through to the chunked kernel
    }

    // chunking: equal chunks no larger than the tuned maximum
    const int64_t align = fp8 ? 256 : 16;
    const int64_t max_chunk = std::max<int64_t>(align, std::min<int64_t>(65536, tu.dispatch_chunk) / align * align);
    const int64_t nch = (a.row_bytes + max_chunk - 1) / max_chunk;
    a.chunk_bytes = (int)round_up((a.row_bytes + nch - 1) / nch, align);
    a.num_chunks = (int)((a.row_bytes + a.chunk_bytes - 1) / a.chunk_bytes);
    a.num_units = (int64_t)L.num_tokens * a.num_chunks;
    a.stages = std::min(kMaxStages, std::max(2, tu.dispatch_stages));

    int64_t per_warp = kBarBytes + (int64_t)a.stages * a.chunk_bytes;
    if (fp8) per_warp += (int64_t)a.stages * (a.chunk_bytes / 2) + round_up((int64_t)a.stages * (a.chunk_bytes / 256) * 4, 128);
    per_warp = round_up(per_warp, 128);
    a.warp_smem = (int)per_warp;
    // as many of the requested warps as fit in one CTA's shared memory
    const int fit = (int)std::min<int64_t>(16, (int64_t)device_smem_optin() / per_warp);
    if (fit < 1) return MOE_ERR_INVALID_ARG;
    const int warps = std::max(1, std::min(fit, tu.dispatch_warps));
    const size_t smem = (size_t)per_warp * warps;

    const void *fn = fp8 ? (const void *)dispatch_kernel<true> : (const void *)dispatch_kernel<false>;
    if (ensure_dynamic_smem(fn, smem) != MOE_OK) return MOE_ERR_CUDA;
    int ctas_per_sm = (int)std::max<size_t>(1, device_smem_per_sm() / (smem + 1024));
    if (tu.ctas_per_sm > 0) ctas_per_sm = std::min(ctas_per_sm, tu.ctas_per_sm);
    const int64_t want = (a.num_units + warps - 1) / warps;
    const int grid = (int)std::min<int64_t>(want, (int64_t)device_sm_count() * ctas_per_sm);

    if (fp8) dispatch_kernel<true><<<grid, warps * 32, smem, st>>>(a);
    else dispatch_kernel<false><<<grid, warps * 32, smem, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
