// noalloc.cu -- deft_tree_attn_noalloc: the tree-attention step for callers
// that cannot allocate device memory.
//
// deft_tree_attn needs two pieces of device memory besides its inputs and
// outputs: the plan's device copy (from deft_plan_upload, which calls
// cudaMalloc) and a workspace for the phase-1 partial results.  Some callers
// cannot provide either: a runtime that has reserved the device memory for
// its own pool and gives kernels no way to take more, a plugin interface
// that hands a plugin its buffers and forbids allocation while it executes,
// a serving loop that cannot afford the device-wide synchronisation a
// cudaMalloc or cudaFree may cause.  This entry point serves them from one
// fixed, file-scope device array instead: the plan's tree-partition arrays
// are copied into it from a host image the plan keeps (one cudaMemcpyAsync
// on the caller's stream), and the partials live after them.  It calls no
// cudaMalloc, cudaFree or other allocating routine.
//
// The array is kNoallocScratchBytes (64 MiB) and exists on every GPU that
// loads the library, until the process exits.  All calls share it and it
// keeps whatever the last call left there.  Each call rewrites the plan
// arrays (the work queues among them start at zero) before its kernels run;
// nothing else in it has to start at zero: phase 1 writes every partial that
// the merge reads.  Calls that can overlap on the GPU (different streams, or
// different host threads without ordering) race on the array.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <new>

#include <cuda_runtime.h>

#include "deft_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = DEFT_NOALLOC_SCRATCH_BYTES;
constexpr size_t kAlign = deft::kWorkAlign;
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

// Offsets of the tree partition's arrays at the start of the scratch array;
// returns the end of the last one.
size_t array_offsets(const deft::Partition &p, size_t *off)
{
    const auto arrays = deft::partition_arrays(p);
    size_t cursor = 0;
    for (int i = 0; i < deft::kPartArrays; ++i) {
        off[i] = cursor;
        cursor = align_up(cursor + (arrays[i].bytes ? arrays[i].bytes : 4));
    }
    return cursor;
}

}  // namespace

extern "C" int deft_tree_attn_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                      const int32_t *node_page_off, const int32_t *page_id,
                                      int32_t num_pages, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                      float scale, const deft_plan_t *plan, void *out,
                                      int32_t out_dtype, float *lse, void *stream)
{
    deft::AttnArgs a;
    bool use_mma = false;
    int rc = deft::prepare_step(q, k_pages, v_pages, node_page_off, page_id, num_pages, num_q_heads, num_kv_heads,
                                head_dim, page_size, scale, plan, out, out_dtype, lse, 0, a, use_mma);
    if (rc != DEFT_OK)
        return rc;

    // Scratch layout: the tree partition's arrays, then the workspace (the
    // partials).
    const deft::Partition &p = plan->tree;
    size_t off[deft::kPartArrays];
    const size_t arrays_end = array_offsets(p, off);
    const int64_t slots = p.num_slots();
    const deft::WorkLayout wl = deft::work_layout(slots > 0 ? slots : 1, num_q_heads, head_dim);
    if (arrays_end + wl.total > kNoallocScratchBytes)
        return DEFT_EWORKSPACE;   // this plan and head shape need more than the fixed array
    if (plan->num_queries == 0)
        return DEFT_OK;

    // The host image of the arrays, packed once per plan build (host memory
    // only; its capacity is kept across rebuilds).
    deft_plan_t *mp = const_cast<deft_plan_t *>(plan);
    if (!mp->noalloc_image_ok) {
        try {
            mp->noalloc_image.assign(arrays_end, 0u);
        } catch (const std::bad_alloc &) {
            return DEFT_ENOMEM;
        }
        const auto arrays = deft::partition_arrays(p);
        for (int i = 0; i < deft::kPartArrays; ++i)
            if (arrays[i].bytes)
                std::memcpy(mp->noalloc_image.data() + off[i], arrays[i].ptr, arrays[i].bytes);
        mp->noalloc_image_ok = true;
    }

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DEFT_ECUDA;
    unsigned char *base = nullptr;
    rc = scratch_address(dev, &base);
    if (rc != DEFT_OK)
        return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *ws = base + arrays_end;
    if (cudaMemcpyAsync(base, mp->noalloc_image.data(), arrays_end, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return DEFT_ECUDA;

    deft::DevPartition d{};
    deft::bind_partition(p, base, off, arrays_end, plan->num_nodes, plan->num_queries, plan->mask_words, d);
    a.o_part = reinterpret_cast<float *>(ws + wl.o_off);
    a.lse_part = reinterpret_cast<float *>(ws + wl.lse_off);

    const deft::LaunchTracer untraced = [](const deft_trace_record &, void *, const std::function<int()> &launch) {
        return launch();
    };
    return deft::dispatch_step(a, d, p, use_mma, 0, stream, untraced) ? DEFT_ECUDA : DEFT_OK;
}
