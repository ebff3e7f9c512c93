// phase2.cu -- the per-query log-sum-exp merge of the phase-1 partials, a
// launch of its own after phase 1: over the queries whose path spans more
// than one chunk and those whose path is empty (out = 0, lse = -inf); the
// rows of single-chunk queries were written by phase 1.
//
// DeFT abstract (partial results of a query's KV partitions are combined per
// query) and DeFT Guide, "Deep Dive": the online-softmax identity that makes
// the combination exact.  For query q and query head h with partial slots
// s in S(q), each holding a normalised output o_s and a base-2 log-sum-exp
// L_s of its own chunk:
//     M = max_s L_s,   w_s = 2^(L_s - M),
//     out = sum_s w_s o_s / sum_s w_s,   lse = (M + log2 sum_s w_s) * ln 2.
// A query with no slot (an empty path) gets out = 0 and lse = -inf.
//
// One warp per (query, head); lane i owns head_dim/32 consecutive elements,
// so each slot's partial is read with one coalesced 128-bit (or 64-bit) load
// per lane; the slot ids and weights are loaded one slot per lane and
// broadcast by shuffles.  The kernel is a programmatic dependent of the last
// phase-1 launch: it reads its slot lists while phase 1 finishes, waits for
// the grid dependency, then issues the partials' loads of up to 16 slots
// before the first arithmetic.  The partials were written moments earlier
// and are mostly still in L2.
#include "merge.cuh"

namespace deft {
namespace {

template <int D>
__global__ void __launch_bounds__(256) phase2_merge_kernel(AttnArgs a, const int32_t *__restrict__ q_slot_off,
                                                           const int32_t *__restrict__ q_slot,
                                                           const int32_t *__restrict__ queries, int32_t nq)
{
    constexpr int E = D / 32;  // elements per lane
    constexpr int KP = 16;     // slots whose partial rows are loaded before any arithmetic
    if (threadIdx.x == 0)
        grid_dep_launch();
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    const int num_q_heads = a.num_q_heads;
    if (warp >= nq * num_q_heads)
        return;
    const int i = warp / num_q_heads;
    const int h = warp - i * num_q_heads;
    const int q = queries ? queries[i] : i;
    const float *o_part = a.o_part, *lse_part = a.lse_part;
    // Slot rows come from the plan, so they are read before the partials are
    // ready (lane j: the query's slot j, for the first 32).
    const int s0 = q_slot_off[q], n = q_slot_off[q + 1] - s0;
    size_t row = 0;
    if (lane < n)
        row = (size_t)q_slot[s0 + lane] * num_q_heads + h;
    grid_dep_wait();   // the phase-1 launches have completed

    // Every load of the first KP slots goes out before the first use.
    const float l = lane < n ? lse_part[row] : -INFINITY;
    float ov[KP][E];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
        const size_t rj = __shfl_sync(0xffffffffu, row, j);
#pragma unroll
        for (int e = 0; e < E; ++e)
            ov[j][e] = 0.f;
        if (j < n) {
            const float *src = o_part + rj * D + lane * E;
            if constexpr (E == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(src);
                ov[j][0] = v.x;
                ov[j][1] = v.y;
                ov[j][2] = v.z;
                ov[j][3] = v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(src);
                ov[j][0] = v.x;
                ov[j][1] = v.y;
            }
        }
    }
    float M = l;
    for (int b = 32; b < n; b += 32) {
        const int k = b + lane;
        if (k < n)
            M = fmaxf(M, lse_part[(size_t)q_slot[s0 + k] * num_q_heads + h]);
    }
    M = warp_max(M);

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e)
        acc[e] = 0.f;
    float wsum = 0.f;
    if (M != -INFINITY) {
        auto add_row = [&](size_t rj, float wj) {
            const float *src = o_part + rj * D + lane * E;
            if constexpr (E == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(src);
                acc[0] = fmaf(wj, v.x, acc[0]);
                acc[1] = fmaf(wj, v.y, acc[1]);
                acc[2] = fmaf(wj, v.z, acc[2]);
                acc[3] = fmaf(wj, v.w, acc[3]);
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(src);
                acc[0] = fmaf(wj, v.x, acc[0]);
                acc[1] = fmaf(wj, v.y, acc[1]);
            }
        };
        const float w = lane < n ? exp2f(l - M) : 0.f;   // weights of the first 32 slots
        wsum = w;
#pragma unroll
        for (int j = 0; j < KP; ++j) {
            const float wj = __shfl_sync(0xffffffffu, w, j);
#pragma unroll
            for (int e = 0; e < E; ++e)
                acc[e] = fmaf(wj, ov[j][e], acc[e]);
        }
        const int n32 = n < 32 ? n : 32;
        for (int j = KP; j < n32; ++j)
            add_row(__shfl_sync(0xffffffffu, row, j), __shfl_sync(0xffffffffu, w, j));
        for (int b = 32; b < n; b += 32) {
            const int k = b + lane;
            size_t rb = 0;
            float wb = 0.f;
            if (k < n) {
                rb = (size_t)q_slot[s0 + k] * num_q_heads + h;
                wb = exp2f(lse_part[rb] - M);
            }
            wsum += wb;
            const int nb = n - b < 32 ? n - b : 32;
            for (int j = 0; j < nb; ++j)
                add_row(__shfl_sync(0xffffffffu, rb, j), __shfl_sync(0xffffffffu, wb, j));
        }
        wsum = warp_sum(wsum);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const size_t orow = ((size_t)q * num_q_heads + h) * D + lane * E;
    if (a.out_dtype == DEFT_OUT_F32) {
        float *o = reinterpret_cast<float *>(a.out) + orow;
#pragma unroll
        for (int e = 0; e < E; ++e)
            o[e] = acc[e] * inv;
    } else {
        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(a.out) + orow;
#pragma unroll
        for (int e = 0; e < E; e += 2)
            *reinterpret_cast<__nv_bfloat162 *>(o + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
    }
    if (lane == 0)
        a.lse_out[(size_t)q * num_q_heads + h] = wsum > 0.f ? (M + log2f(wsum)) * kLn2 : -INFINITY;
}

}  // namespace

int launch_phase2(const AttnArgs &a, const DevPartition &p, const int32_t *queries, int32_t nq, void *stream)
{
    const int64_t warps = (int64_t)nq * a.num_q_heads;
    if (warps == 0)
        return 0;
    const int threads = 256;
    const unsigned blocks = (unsigned)((warps * 32 + threads - 1) / threads);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (a.head_dim == 128)
        return (int)launch_dependent(phase2_merge_kernel<128>, dim3(blocks), dim3(threads), 0, st, a, p.q_slot_off,
                                     p.q_slot, queries, nq);
    return (int)launch_dependent(phase2_merge_kernel<64>, dim3(blocks), dim3(threads), 0, st, a, p.q_slot_off,
                                 p.q_slot, queries, nq);
}

}  // namespace deft
