// dispatch.cu -- the launches of one step: phase 1 (tensor-core and
// CUDA-core families) and the phase-2 merge.
//
// Both phase-1 families are persistent, memory-bound kernels over disjoint
// partial slots.  When a step has both, the tensor-core launches run on a
// side stream concurrently with the CUDA-core launches on the caller's
// stream, each family on a share of the SMs proportional to its cost (KV
// tokens plus a per-unit overhead, per KV head, tensor-core tokens weighted
// by kMmaCostNum / kMmaCostDen), so that the two finish together; a fork event orders the side stream after the caller's earlier
// work and a join event orders the merge after both.  The side stream and
// its events are created once per host thread and device and reused.
#include <cuda_runtime.h>

#include "deft_internal.h"

namespace deft {
namespace {

// Relative cost of a tensor-core token against a CUDA-core one when both
// families stream at once: the tensor-core kernel holds its stages longer
// (a V stage through the tile's softmax) and so draws less bandwidth per SM
// (measured about 1.6x slower per byte on the few-shot tree).
constexpr int64_t kMmaCostNum = 8, kMmaCostDen = 5;

struct SideStream {
    int dev = -1;
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

int side_stream(SideStream **out)
{
    thread_local SideStream cache[8];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return (int)cudaErrorInvalidDevice;
    SideStream &c = cache[dev & 7];
    if (c.dev != dev) {
        if (c.s) {   // another device took this slot: make room
            cudaStreamDestroy(c.s);
            cudaEventDestroy(c.fork);
            cudaEventDestroy(c.join);
            c = SideStream{};
        }
        cudaError_t e = cudaStreamCreateWithFlags(&c.s, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&c.fork, cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&c.join, cudaEventDisableTiming);
        if (e != cudaSuccess)
            return (int)e;
        c.dev = dev;
    }
    *out = &c;
    return 0;
}

}  // namespace

int dispatch_step(AttnArgs a, const DevPartition &dp, const Partition &hp, bool use_mma, int32_t family,
                  void *out, int32_t out_dtype, float *lse, void *stream, const LaunchTracer &trace)
{
    const int64_t hkv = a.num_kv_heads;
    const bool mma_on = use_mma && dp.num_mma_items > 0;
    // Cost of each family (the cost prefixes' totals, per KV head).
    const int64_t c_mma = mma_on ? hkv * (hp.mma_cost.back() - hp.mma_cost.front()) * kMmaCostNum / kMmaCostDen : 0;
    const int64_t c_fma = hkv * ((dp.num_fma_items ? hp.fma_cost.back() : 0) +
                                 (!use_mma && dp.num_mma_items ? hp.fallback_cost.back() : 0));
    const int sms = num_sms();
    int cta_mma = sms, cta_fma = sms;
    const bool split = c_mma > 0 && c_fma > 0 && sms >= 2;
    if (split) {
        cta_mma = (int)((c_mma * sms + (c_mma + c_fma) / 2) / (c_mma + c_fma));
        cta_mma = cta_mma < 1 ? 1 : cta_mma > sms - 1 ? sms - 1 : cta_mma;
        cta_fma = sms - cta_mma;
    }
    SideStream *side = nullptr;
    void *mma_stream = stream;
    if (split) {
        int e = side_stream(&side);
        if (e)
            return e;
        cudaStream_t main = reinterpret_cast<cudaStream_t>(stream);
        if ((e = (int)cudaEventRecord(side->fork, main)) || (e = (int)cudaStreamWaitEvent(side->s, side->fork, 0)))
            return e;
        mma_stream = side->s;
    }

    // CUDA-core launches, one per row bucket; each family's first launch
    // waits for the work before it (wait_prior).
    AttnArgs af = a;
    auto fma_launches = [&](const int32_t *items, const uint32_t *rmask, const int32_t *rmask_off,
                            const std::vector<int64_t> &cost, const std::array<int32_t, 6> &off, int fb) {
        for (int b = 0; b < 5; ++b) {
            const int32_t n = off[b + 1] - off[b];
            if (n <= 0)
                continue;
            const int32_t *it = items + 3 * (size_t)off[b];
            const int r = trace({DEFT_K_PHASE1_FMA, family, b, fb, n, 0.f}, stream, [&] {
                const int r2 = launch_phase1_fma(af, dp, it, rmask, rmask_off + off[b], cost.data() + off[b], n, b,
                                                 cta_fma, stream);
                if (r2 == 0)
                    af.wait_prior = 0;
                return r2;
            });
            if (r)
                return r;
        }
        return 0;
    };
    int rc = 0;
    if (mma_on) {
        AttnArgs am = a;
        for (int b = 0; b < 4 && !rc; ++b) {
            const int32_t n = hp.mma_bucket_off[b + 1] - hp.mma_bucket_off[b];
            if (n <= 0)
                continue;
            const int32_t *it = dp.mma_items + 3 * (size_t)hp.mma_bucket_off[b];
            rc = trace({DEFT_K_PHASE1_MMA, family, b, 0, n, 0.f}, mma_stream, [&] {
                const int r2 = launch_phase1_mma(am, dp, it, dp.mma_rmask, dp.mma_rmask_off + hp.mma_bucket_off[b],
                                                 hp.mma_cost.data() + hp.mma_bucket_off[b], n, b, cta_mma,
                                                 mma_stream);
                if (r2 == 0)
                    am.wait_prior = 0;
                return r2;
            });
        }
        if (!split && rc == 0)
            af.wait_prior = 0;   // the CUDA-core launches follow on the same stream
    } else if (dp.num_mma_items > 0) {
        // The tensor-core path covers head_dim 128; other head sizes, or a
        // run with DEFT_DISABLE_MMA set, take the same chunks on CUDA cores
        // in items of at most 16 rows.
        rc = fma_launches(dp.fallback_items, dp.fallback_rmask, dp.fallback_rmask_off, hp.fallback_cost,
                          hp.fallback_bucket_off, 1);
    }
    if (rc == 0 && dp.num_fma_items > 0)
        rc = fma_launches(dp.fma_items, dp.fma_rmask, dp.fma_rmask_off, hp.fma_cost, hp.fma_bucket_off, 0);
    if (split) {
        // Join even after a failed launch, so the caller's stream never runs
        // ahead of work already queued on the side stream.
        const int e1 = (int)cudaEventRecord(side->join, side->s);
        const int e2 = (int)cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream), side->join, 0);
        if (!rc)
            rc = e1 ? e1 : e2;
    }
    if (rc)
        return rc;
    return trace({DEFT_K_PHASE2, family, 0, 0, dp.num_queries, 0.f}, stream,
                 [&] { return launch_phase2(a, dp, out, out_dtype, lse, stream); });
}

}  // namespace deft
