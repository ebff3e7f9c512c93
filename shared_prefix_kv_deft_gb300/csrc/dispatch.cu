// dispatch.cu -- the launches of one step: phase 1 (tensor-core and
// CUDA-core launches, one per bucket) and the phase-2 merge, on the
// caller's stream.
//
// Every launch is a programmatic dependent of the one before and starts its
// CTAs as soon as that one's CTAs are all running, so the phase-1 launches
// run concurrently.  They share the SMs (one persistent CTA per SM): every
// launch but the costliest gets a share of the SMs in proportion to its
// estimated cost, and the costliest, launched first, gets the rest.  Each
// launch has its own work queue (two words in the plan's device memory,
// zero between launches).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "deft_internal.h"

namespace deft {

namespace {

struct Launch {
    int kind;      // 0 tensor core, 1 CUDA core, 2 CUDA core on tensor-core chunks
    int bucket;
    int32_t off;   // first item of the bucket
    int32_t n;     // items
    double cost;   // estimated SM time (KV tokens x KV heads x time per token)
};

}  // namespace

// SM shares of the step's phase-1 launches, the costliest last in `cost`
// and `units` (it is launched first): grid and early CTAs of each.  Every
// CTA of a launch starts with the step (grid = early).
void shape_launches(const double *cost, const int32_t *units, int n, int sms, LaunchShape *out)
{
    if (n <= 0)
        return;
    double total = 0.0;
    for (int i = 0; i < n; ++i)
        total += cost[i];
    int used = 0;
    for (int i = 0; i + 1 < n; ++i) {
        // A quarter over the proportional share: the costliest launch can
        // take no units of the others, so one of them finishing late is the
        // step's tail.
        const double share = total > 0.0 ? 1.25 * sms * cost[i] / total : 1.0;
        int g = (int)std::ceil(share);
        g = std::max(1, std::min({g, (int)units[i], sms}));
        // No more CTAs than the rounds of units need: ceil(units / g)
        // rounds take as long with ceil(units / rounds) CTAs.
        const int rounds = (int)((units[i] + g - 1) / g);
        g = (int)((units[i] + rounds - 1) / rounds);
        out[i] = LaunchShape{g, g, -1};
        used += g;
    }
    // Leave the costliest launch at least a quarter of the SMs.
    const int cap = std::max(n - 1, sms - std::max(1, sms / 4));
    while (used > cap) {
        int j = 0;
        for (int i = 1; i + 1 < n; ++i)
            if (out[i].grid > out[j].grid)
                j = i;
        if (out[j].grid <= 1)
            break;
        --out[j].grid;
        out[j].early = out[j].grid;
        --used;
    }
    const int g = std::max(1, std::min((int)units[n - 1], sms - used));
    out[n - 1] = LaunchShape{g, g, -1};
}

namespace {

// The early CTAs' static blocks when the units' costs differ: the first
// block (items are sorted by cost, largest first) holds no more than 9/10 of
// an even share of the launch's estimated cost; the queue evens out the rest.  Units are item-major,
// `hkv` per item; unit_cost(i) is item i's cost per unit.
template <typename F>
int32_t cost_block(int32_t n_items, int32_t hkv, int32_t early, F unit_cost)
{
    double total = 0.0;
    for (int32_t i = 0; i < n_items; ++i)
        total += unit_cost(i) * hkv;
    const double cap = 0.9 * total / std::max(1, early);
    double acc = 0.0;
    int32_t s = 0;
    for (int32_t i = 0; i < n_items; ++i) {
        const double u = unit_cost(i);
        for (int32_t h = 0; h < hkv; ++h) {
            if (acc + u > cap)
                return s;
            acc += u;
            ++s;
        }
    }
    return s;
}

}  // namespace

int dispatch_step(AttnArgs a, const DevPartition &dp, const Partition &hp, bool use_mma, int32_t family,
                  void *stream, const LaunchTracer &trace)
{
    const int32_t hkv = a.num_kv_heads;
    Launch ls[14];
    int n = 0;
    // One tensor-core launch per column bucket: each is built for its
    // width (stage counts and buffers depend on it).
    if (dp.num_mma_items > 0 && use_mma) {
        for (int b = 0; b < 2; ++b) {
            const int32_t c = hp.mma_bucket_off[b + 1] - hp.mma_bucket_off[b];
            if (c > 0)
                ls[n++] = Launch{0, b, hp.mma_bucket_off[b], c,
                                 (double)hp.mma_bucket_tok[b] * hkv * mma_ns_per_token(b)};
        }
    }
    // CUDA-core items: one launch per row bucket, or one launch at the
    // largest bucket present when that costs little more in all (its smaller
    // items then run at its row count).
    auto add_fma = [&](int kind, const std::array<int32_t, 6> &off, const std::array<int64_t, 5> &tok) {
        int nb = 0, maxb = 0;
        double split = 0.0;
        int64_t all_tok = 0;
        for (int b = 0; b < 5; ++b)
            if (off[b + 1] > off[b]) {
                ++nb;
                maxb = b;
                split += (double)tok[b] * hkv * fma_ns_per_token(b);
                all_tok += tok[b];
            }
        const double one = (double)all_tok * hkv * fma_ns_per_token(maxb);
        if (nb > 1 && one <= kCollapse * split) {
            ls[n++] = Launch{kind, maxb, 0, off[5], one};
            return;
        }
        for (int b = 0; b < 5; ++b) {
            const int32_t c = off[b + 1] - off[b];
            if (c > 0)
                ls[n++] = Launch{kind, b, off[b], c, (double)tok[b] * hkv * fma_ns_per_token(b)};
        }
    };
    // The tensor-core path covers head_dim 128; other head sizes, or a step
    // asked to run on CUDA cores only, take the same chunks on CUDA cores in
    // items of at most 16 rows.
    if (dp.num_mma_items > 0 && !use_mma)
        add_fma(2, hp.fallback_bucket_off, hp.fallback_bucket_tok);
    if (dp.num_fma_items > 0)
        add_fma(1, hp.fma_bucket_off, hp.fma_bucket_tok);
    // Shares are computed with the costliest launch last.
    if (n > 1) {
        int j = 0;
        for (int i = 1; i < n; ++i)
            if (ls[i].cost > ls[j].cost)
                j = i;
        std::rotate(ls + j, ls + j + 1, ls + n);
    }
    double cost[14];
    int32_t units[14];
    LaunchShape shape[14];
    for (int i = 0; i < n; ++i) {
        cost[i] = ls[i].cost;
        units[i] = ls[i].n * hkv;
    }
    shape_launches(cost, units, n, num_sms(), shape);
    // The costliest launch then goes first: each launch ahead of it would
    // hold back its start by the launch latency (~2.5-3.5 us).  (Launched
    // last, with extra CTAs for the SMs the others free, it mostly found its
    // queue drained by the time they started: few-shot tree 50.4 -> 49.2 us.)
    if (n > 1) {
        std::rotate(ls, ls + n - 1, ls + n);
        std::rotate(shape, shape + n - 1, shape + n);
    }
    // Whether a launch's items include row blocks of one chunk (items
    // reading the same KV).
    auto row_blocks = [&](const Launch &l) {
        const std::vector<int32_t> &it = l.kind == 0 ? hp.mma_items : l.kind == 1 ? hp.fma_items : hp.fallback_items;
        for (int32_t k = 0; k < l.n; ++k) {
            const int32_t *t = &it[3 * (size_t)(l.off + k)];
            if (t[1] > 0 || t[2] < hp.chunk_q_off[t[0] + 1] - hp.chunk_q_off[t[0]])
                return true;
        }
        return false;
    };
    // Static blocks by cost (a launch's items differ in size: a block of
    // whole long items would keep its CTA long after the others).
    for (int i = 0; i < n; ++i) {
        const Launch &l = ls[i];
        const std::vector<int32_t> &it = l.kind == 0 ? hp.mma_items : l.kind == 1 ? hp.fma_items : hp.fallback_items;
        shape[i].block = cost_block(l.n, hkv, shape[i].early, [&](int32_t k) {
            const int32_t *t = &it[3 * (size_t)(l.off + k)];
            const double ns = l.kind == 0 ? mma_ns_per_token(l.bucket) : fma_ns_per_token(l.bucket);
            return (double)hp.chunk_tokens[t[0]] * ns;
        });
        // Row blocks of one chunk find its KV in L2 only when they run at
        // about the same time.  The blocks are consecutive items, so their
        // units for head h are Hkv apart; with a static block that divides
        // Hkv they come at the same step of their CTAs' blocks, which start
        // together.  (A block of 3 units at Hkv = 8 had the imbalance shape
        // read its 32768-token prefix from DRAM ~3 times: 1.44x the unique
        // KV instead of 1.03x.)
        if (shape[i].block > 1 && row_blocks(l)) {
            int32_t b = std::min<int32_t>(shape[i].block, hkv);
            while (b > 1 && hkv % b != 0)
                --b;
            shape[i].block = b;
        }
    }

    // Only the step's first launch waits for the stream's earlier work
    // before reading inputs (wait_prior); the rest follow it.
    const int32_t kv_once = a.kv_once;
    for (int i = 0; i < n; ++i) {
        const Launch &l = ls[i];
        int r;
        // A launch whose items include row blocks of one chunk reads that
        // chunk's KV once per block: its copies keep the normal L2 policy so
        // that the later blocks find the KV in L2.
        a.kv_once = kv_once && !row_blocks(l);
        if (l.kind == 0) {
            const int32_t *it = dp.mma_items + 3 * (size_t)l.off;
            uint32_t *queue = dp.queues + 2 * queue_slot(0, l.bucket);
            r = trace({DEFT_K_PHASE1_MMA, family, l.bucket, 0, l.n, 0.f}, stream, [&] {
                return launch_phase1_mma(a, dp, it, dp.mma_rmask, dp.mma_rmask_off + l.off, l.n, l.bucket, queue,
                                         shape[i], stream);
            });
        } else {
            const bool fb = l.kind == 2;
            const int32_t *it = (fb ? dp.fallback_items : dp.fma_items) + 3 * (size_t)l.off;
            const uint32_t *rm = fb ? dp.fallback_rmask : dp.fma_rmask;
            const int32_t *rmo = (fb ? dp.fallback_rmask_off : dp.fma_rmask_off) + l.off;
            const uint32_t *dr = (fb ? dp.fallback_direct : dp.fma_direct) + l.off;
            uint32_t *queue = dp.queues + 2 * queue_slot(fb ? 2 : 1, l.bucket);
            r = trace({DEFT_K_PHASE1_FMA, family, l.bucket, fb ? 1 : 0, l.n, 0.f}, stream, [&] {
                return launch_phase1_fma(a, dp, it, rm, rmo, dr, l.n, l.bucket, queue, shape[i], stream);
            });
        }
        if (r)
            return r;
        a.wait_prior = 0;
    }
    // With direct rows, the merge launch takes the queries with several
    // slots or none, and is left out when there are none.
    const int32_t nq = a.direct ? dp.num_merge_q : dp.num_queries;
    if (nq == 0)
        return 0;
    // Every query merged: no list to read.
    const int32_t *qlist = nq < dp.num_queries ? dp.merge_q : nullptr;
    return trace({DEFT_K_PHASE2, family, 0, 0, nq, 0.f}, stream,
                 [&] { return launch_phase2(a, dp, qlist, nq, stream); });
}

}  // namespace deft
