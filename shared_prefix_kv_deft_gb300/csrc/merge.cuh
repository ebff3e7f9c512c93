// merge.cuh -- helpers shared by the phase-1 kernels and the merge launch:
// the output store in either dtype, the lse of a row whose query has one
// partial slot (written by phase 1 directly: with a single slot the merge of
// phase2.cu, M = L, w = 1, is the identity), and the failure report.
#pragma once

#include "common.cuh"
#include "deft_internal.h"

namespace deft {

// Stores one output row (fp32 value v of element e) in a.out's dtype.
__device__ __forceinline__ void store_out(const AttnArgs &a, size_t out_row, int e, int D, float v)
{
    if (a.out_dtype == DEFT_OUT_F32)
        reinterpret_cast<float *>(a.out)[out_row * D + e] = v;
    else
        reinterpret_cast<__nv_bfloat16 *>(a.out)[out_row * D + e] = __float2bfloat16_rn(v);
}

// The natural-log lse of a row whose query has this one slot.
__device__ __forceinline__ float direct_lse(float lse2)
{
    return lse2 * kLn2;
}

// Records the first failing wait's code in the partition's status word.
__device__ __forceinline__ void report_failure(uint32_t *status, int code)
{
    if (status && code)
        atomicCAS(status, 0u, (uint32_t)code);
}

}  // namespace deft
