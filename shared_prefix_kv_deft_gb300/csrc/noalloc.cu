// noalloc.cu -- deft_tree_attn_noalloc: the tree-attention step for callers
// that cannot allocate device memory.
//
// deft_tree_attn needs two pieces of device memory besides its inputs and
// outputs: the plan's device copy (from deft_plan_upload, which calls
// cudaMalloc) and a workspace for the phase-1 partial results.  Some callers
// cannot provide either: code that must not call cudaMalloc while a CUDA
// graph is being captured, runtimes whose memory is owned by a pool or
// allocator they may not bypass, and latency-bound loops where an allocation
// (or its implicit synchronisation) is not acceptable.  This entry point
// serves them from one fixed, file-scope device array instead: the plan's
// tree-partition arrays are copied into it from the plan's host memory on
// the caller's stream, and the partials live after them.  It calls no
// cudaMalloc, cudaFree or other allocating routine.
//
// The array is kNoallocScratchBytes (64 MiB) and exists on every GPU that
// loads the library, until the process exits.  All calls share it and it
// keeps whatever the last call left there.  Nothing in it needs to start at
// zero: every call rewrites the plan arrays, and phase 1 writes every
// partial that phase 2 reads.  Calls that can overlap on the GPU (different
// streams, or different host threads without ordering) race on the array.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>

#include <cuda_runtime.h>

#include "deft_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = DEFT_NOALLOC_SCRATCH_BYTES;
constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {

std::atomic<void *> g_scratch_addr[kMaxDevices];

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Device address of the scratch array on `dev` (the current device).  In host
// code `g_noalloc_scratch` names a host-side stand-in, so the address must come
// from cudaGetSymbolAddress; it is looked up on the first call per device.
int scratch_address(int dev, unsigned char **out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return DEFT_EUNSUPPORTED;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return DEFT_ECUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = static_cast<unsigned char *>(p);
    return DEFT_OK;
}


}  // namespace

extern "C" int deft_tree_attn_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                      const int32_t *node_page_off, const int32_t *page_id,
                                      int32_t num_pages, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                      float scale, const deft_plan_t *plan, void *out,
                                      int32_t out_dtype, float *lse, void *stream)
{
    if (!plan || !q || !k_pages || !v_pages || !node_page_off || !page_id || !out || !lse)
        return DEFT_EINVAL;
    if (out_dtype != DEFT_OUT_BF16 && out_dtype != DEFT_OUT_F32)
        return DEFT_EINVAL;
    if (!(scale > 0.f) || !std::isfinite(scale) || num_pages < 1)
        return DEFT_EINVAL;
    if (num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads != 0)
        return DEFT_EINVAL;
    if (((uintptr_t)q | (uintptr_t)k_pages | (uintptr_t)v_pages) & 15u)
        return DEFT_EINVAL;   // the kernels copy q and KV rows in 16-byte pieces
    if ((head_dim != 64 && head_dim != 128) || page_size != deft::kPageSize)
        return DEFT_EUNSUPPORTED;
    if (num_q_heads / num_kv_heads != plan->gqa_group)
        return DEFT_ESTATE;
    const char *dis = std::getenv("DEFT_DISABLE_MMA");
    const bool use_mma = deft::mma_supported(head_dim) && !(dis && dis[0] && dis[0] != '0');
    if (plan->gqa_group > deft::kFmaMaxRows && !use_mma)
        return DEFT_EUNSUPPORTED;

    // Scratch layout: the tree partition's arrays, then the partials.
    const deft::Partition &p = plan->tree;
    const auto arrays = deft::partition_arrays(p);
    size_t off[deft::kPartArrays];
    size_t cursor = 0;
    for (int i = 0; i < deft::kPartArrays; ++i) {
        off[i] = cursor;
        cursor = align_up(cursor + (arrays[i].bytes ? arrays[i].bytes : 4));
    }
    const size_t slots = (size_t)p.num_slots();
    const size_t o_off = cursor;
    const size_t lse_off = align_up(o_off + slots * num_q_heads * head_dim * sizeof(float));
    const size_t total = align_up(lse_off + slots * num_q_heads * sizeof(float));
    if (total > kNoallocScratchBytes)
        return DEFT_EWORKSPACE;   // this plan and head shape need more than the fixed array
    if (plan->num_queries == 0)
        return DEFT_OK;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DEFT_ECUDA;
    unsigned char *base = nullptr;
    int rc = scratch_address(dev, &base);
    if (rc != DEFT_OK)
        return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    for (int i = 0; i < deft::kPartArrays; ++i)
        if (arrays[i].bytes &&
            cudaMemcpyAsync(base + off[i], arrays[i].ptr, arrays[i].bytes, cudaMemcpyHostToDevice, st) !=
                cudaSuccess)
            return DEFT_ECUDA;

    deft::DevPartition d{};
    deft::bind_partition(p, base, off, cursor, plan->num_nodes, plan->num_queries, plan->mask_words, d);

    deft::AttnArgs a{};
    a.q = q;
    a.k_pages = k_pages;
    a.v_pages = v_pages;
    a.node_page_off = node_page_off;
    a.page_id = page_id;
    a.num_pages = num_pages;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.gqa_group = plan->gqa_group;
    a.scale_log2 = scale * 1.44269504088896340736f;
    a.wait_prior = 1;
    a.kv_once = 1;
    a.o_part = reinterpret_cast<float *>(base + o_off);
    a.lse_part = reinterpret_cast<float *>(base + lse_off);

    const deft::LaunchTracer untraced = [](const deft_trace_record &, void *, const std::function<int()> &launch) {
        return launch();
    };
    return deft::dispatch_step(a, d, p, use_mma, 0, out, out_dtype, lse, stream, untraced) ? DEFT_ECUDA : DEFT_OK;
}
