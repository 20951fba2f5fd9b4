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
// GB300 design: persistent grid, one independent pipeline per warp. A unit is
// one chunk of one token's output row. For a unit, the lanes holding the
// token's receive rows sort them (rank among valid rows), lane 0 arms the
// stage's mbarrier with D * chunk bytes, and each of those lanes issues one
// cp.async.bulk of its row's chunk into slot `rank` of the stage. S-1 units
// stay in flight while the warp sums the landed stage slot by slot (16-byte
// shared loads, conflict-free) and writes 16-byte bf16 vectors to `out`.
#include <algorithm>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kMaxStages = 8;
constexpr int kHeadBytes = 128;   // mbarriers [kMaxStages] + row counts [kMaxStages]
constexpr unsigned kFull = 0xffffffffu;

struct CombineArgs {
    const uint8_t *partial;
    int64_t row_bytes;   // H * 2
    int num_rows;
    int k;
    const int32_t *dst_row;
    uint8_t *out;
    int32_t *status;
    int chunk_bytes, num_chunks;
    int64_t num_units;
    int stages, slots, warp_smem, l2_hints;
    uint64_t timeout_ns;
};

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 v) {
    acc[0] += __uint_as_float(v.x << 16); acc[1] += __uint_as_float(v.x & 0xffff0000u);
    acc[2] += __uint_as_float(v.y << 16); acc[3] += __uint_as_float(v.y & 0xffff0000u);
    acc[4] += __uint_as_float(v.z << 16); acc[5] += __uint_as_float(v.z & 0xffff0000u);
    acc[6] += __uint_as_float(v.w << 16); acc[7] += __uint_as_float(v.w & 0xffff0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

__global__ void __launch_bounds__(512) combine_kernel(const CombineArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    const int S = a.stages;
    const int chunk = a.chunk_bytes;
    uint8_t *wbase = smem + (size_t)warp * a.warp_smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(wbase);
    int *dcount = reinterpret_cast<int *>(wbase + kMaxStages * 8);
    uint8_t *stages = wbase + kHeadBytes;
    const size_t stage_bytes = (size_t)a.slots * chunk;

    const int64_t gw = (int64_t)blockIdx.x * warps + warp;
    const int64_t GW = (int64_t)gridDim.x * warps;
    if (gw >= a.num_units) return;
    const int64_t n_w = (a.num_units - 1 - gw) / GW + 1;
    const uint64_t pol_load = (a.l2_hints & 1) ? policy_evict_first() : policy_evict_normal();

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();

    auto fetch_row = [&](int64_t i) -> int {
        const int64_t u = gw + i * GW;
        const int64_t t = u / a.num_chunks;
        return lane < a.k ? a.dst_row[t * a.k + lane] : -1;
    };
    // arm stage (i % S) for unit i and issue its row loads; `row` is this lane's receive row
    auto issue = [&](int64_t i, int row) {
        const int64_t u = gw + i * GW;
        const int64_t t = u / a.num_chunks;
        const int64_t off = (u - t * a.num_chunks) * (int64_t)chunk;
        const uint32_t nbytes = (uint32_t)min((int64_t)chunk, a.row_bytes - off);
        const int s = (int)(i % S);
        if (row >= a.num_rows) {
            if (off == 0) report(a.status, MOE_ERR_CAPACITY);
            row = -1;
        }
        const bool valid = row >= 0;
        const unsigned vmask = __ballot_sync(kFull, valid);
        int pos = 0;
        for (int jj = 0; jj < a.k; ++jj) {
            const int o = __shfl_sync(kFull, row, jj);
            pos += (valid && ((vmask >> jj) & 1u) && o < row) ? 1 : 0;
        }
        if (lane == 0) {
            dcount[s] = __popc(vmask);
            mbar_arrive_expect_tx(&bars[s], (uint32_t)__popc(vmask) * nbytes);
        }
        __syncwarp();
        if (valid)
            bulk_load(stages + s * stage_bytes + (size_t)pos * chunk, a.partial + (int64_t)row * a.row_bytes + off,
                      nbytes, &bars[s], pol_load);
    };

    const int64_t pro = min((int64_t)S, n_w);
    for (int64_t i = 0; i < pro; ++i) issue(i, fetch_row(i));

    for (int64_t i = 0; i < n_w; ++i) {
        const int s = (int)(i % S);
        const uint32_t parity = (uint32_t)((i / S) & 1);
        const int row_next = (i + S < n_w) ? fetch_row(i + S) : -1;
        const int64_t u = gw + i * GW;
        const int64_t t = u / a.num_chunks;
        const int64_t off = (u - t * a.num_chunks) * (int64_t)chunk;
        const int nbytes = (int)min((int64_t)chunk, a.row_bytes - off);

        const bool ok = mbar_wait_bounded(&bars[s], parity, a.timeout_ns);
        if (!__all_sync(kFull, ok)) {
            if (lane == 0) report(a.status, MOE_ERR_TIMEOUT);
            break;
        }
        const int D = dcount[s];
        const uint8_t *st = stages + s * stage_bytes;
        uint8_t *dst = a.out + t * a.row_bytes + off;
        for (int v = lane; v < nbytes / 16; v += 32) {
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
            for (int d = 0; d < D; ++d) add_bf16x8(acc, *reinterpret_cast<const uint4 *>(st + (size_t)d * chunk + v * 16));
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            *reinterpret_cast<uint4 *>(dst + v * 16) = o;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (i + S < n_w) issue(i + S, row_next);
    }
}

inline int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

}  // namespace

int launch_combine(const CombineLaunch &L) {
    if (L.num_tokens == 0) return MOE_OK;
    const Tuning &tu = tuning();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(L.stream);

    CombineArgs a;
    a.partial = static_cast<const uint8_t *>(L.partial);
    a.row_bytes = (int64_t)L.hidden * 2;
    a.num_rows = L.num_partial_rows;
    a.k = L.num_topk;
    a.dst_row = L.token_dst_row;
    a.out = static_cast<uint8_t *>(L.out);
    a.status = L.status;
    a.l2_hints = tu.l2_hints;
    a.timeout_ns = kDefaultWaitNs;
    a.slots = L.num_topk;
    a.stages = std::min(kMaxStages, std::max(2, tu.combine_stages));

    const int64_t max_chunk = std::max<int64_t>(16, std::min<int64_t>(65536, tu.combine_stage_bytes) / a.slots / 16 * 16);
    const int64_t nch = (a.row_bytes + max_chunk - 1) / max_chunk;
    a.chunk_bytes = (int)round_up((a.row_bytes + nch - 1) / nch, 16);
    a.num_chunks = (int)((a.row_bytes + a.chunk_bytes - 1) / a.chunk_bytes);
    a.num_units = (int64_t)L.num_tokens * a.num_chunks;

    const int64_t per_warp = round_up(kHeadBytes + (int64_t)a.stages * a.slots * a.chunk_bytes, 128);
    a.warp_smem = (int)per_warp;
    const int fit = (int)std::min<int64_t>(16, (int64_t)device_smem_optin() / per_warp);
    if (fit < 1) return MOE_ERR_INVALID_ARG;
    const int warps = std::max(1, std::min(fit, tu.combine_warps));
    const size_t smem = (size_t)per_warp * warps;
    if (ensure_dynamic_smem((const void *)combine_kernel, smem) != MOE_OK) return MOE_ERR_CUDA;
    int ctas_per_sm = (int)std::max<size_t>(1, device_smem_per_sm() / (smem + 1024));
    if (tu.ctas_per_sm > 0) ctas_per_sm = std::min(ctas_per_sm, tu.ctas_per_sm);
    const int64_t want = (a.num_units + warps - 1) / warps;
    const int grid = (int)std::min<int64_t>(want, (int64_t)device_sm_count() * ctas_per_sm);
    combine_kernel<<<grid, warps * 32, smem, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
