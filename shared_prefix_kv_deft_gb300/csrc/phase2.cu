// phase2.cu -- per-query log-sum-exp merge of the phase-1 partials.
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
// broadcast by shuffles.  The partials were written moments earlier by
// phase 1 and are mostly still in L2.
#include "common.cuh"
#include "deft_internal.h"

namespace deft {
namespace {

template <int D>
__global__ void __launch_bounds__(256) phase2_merge_kernel(
    const float *__restrict__ o_part, const float *__restrict__ lse_part,
    const int32_t *__restrict__ q_slot_off, const int32_t *__restrict__ q_slot, int32_t num_queries,
    int32_t num_q_heads, void *__restrict__ out, int32_t out_dtype, float *__restrict__ lse_out)
{
    constexpr int E = D / 32;  // elements per lane
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= num_queries * num_q_heads)
        return;
    const int q = warp / num_q_heads;
    const int h = warp - q * num_q_heads;
    const int s0 = q_slot_off[q], s1 = q_slot_off[q + 1];

    // Slots are taken 32 at a time: lane j loads slot j's row and lse, so the
    // dependent loads (slot list -> lse) happen once per batch, not per slot;
    // the batch's partial rows are then independent loads.
    float M = -INFINITY;
    for (int b = s0; b < s1; b += 32) {
        const int i = b + lane;
        if (i < s1)
            M = fmaxf(M, lse_part[(size_t)q_slot[i] * num_q_heads + h]);
    }
    M = warp_max(M);

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e)
        acc[e] = 0.f;
    float wsum = 0.f;
    if (M != -INFINITY) {
        for (int b = s0; b < s1; b += 32) {
            const int i = b + lane;
            size_t myrow = 0;
            float myw = 0.f;
            if (i < s1) {
                myrow = (size_t)q_slot[i] * num_q_heads + h;
                myw = exp2f(lse_part[myrow] - M);
            }
            wsum += myw;
            const int nb = min(32, s1 - b);
#pragma unroll 4
            for (int j = 0; j < nb; ++j) {
                const size_t row = __shfl_sync(0xffffffffu, myrow, j);
                const float w = __shfl_sync(0xffffffffu, myw, j);
                const float *src = o_part + row * D + lane * E;
                if constexpr (E == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(src);
                    acc[0] = fmaf(w, v.x, acc[0]);
                    acc[1] = fmaf(w, v.y, acc[1]);
                    acc[2] = fmaf(w, v.z, acc[2]);
                    acc[3] = fmaf(w, v.w, acc[3]);
                } else {
                    const float2 v = *reinterpret_cast<const float2 *>(src);
                    acc[0] = fmaf(w, v.x, acc[0]);
                    acc[1] = fmaf(w, v.y, acc[1]);
                }
            }
        }
        wsum = warp_sum(wsum);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const size_t orow = ((size_t)q * num_q_heads + h) * D + lane * E;
    if (out_dtype == DEFT_OUT_F32) {
        float *o = reinterpret_cast<float *>(out) + orow;
#pragma unroll
        for (int e = 0; e < E; ++e)
            o[e] = acc[e] * inv;
    } else {
        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(out) + orow;
#pragma unroll
        for (int e = 0; e < E; e += 2)
            *reinterpret_cast<__nv_bfloat162 *>(o + e) =
                __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
    }
    if (lane == 0)
        lse_out[(size_t)q * num_q_heads + h] =
            wsum > 0.f ? (M + log2f(wsum)) * kLn2 : -INFINITY;
}

}  // namespace

int launch_phase2(const AttnArgs &a, const DevPartition &p, void *out, int32_t out_dtype,
                  float *lse, void *stream)
{
    const int64_t warps = (int64_t)p.num_queries * a.num_q_heads;
    if (warps == 0)
        return 0;
    const int threads = 256;
    const unsigned blocks = (unsigned)((warps * 32 + threads - 1) / threads);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (a.head_dim == 128)
        phase2_merge_kernel<128><<<blocks, threads, 0, st>>>(
            a.o_part, a.lse_part, p.q_slot_off, p.q_slot, p.num_queries, a.num_q_heads, out,
            out_dtype, lse);
    else
        phase2_merge_kernel<64><<<blocks, threads, 0, st>>>(
            a.o_part, a.lse_part, p.q_slot_off, p.q_slot, p.num_queries, a.num_q_heads, out,
            out_dtype, lse);
    return (int)cudaGetLastError();
}

}  // namespace deft
