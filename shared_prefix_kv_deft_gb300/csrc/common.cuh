// common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace deft {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// A persistent CTA is done with its launch's work queue (queue[0]: next
// unit, queue[1]: CTAs done).  The launch's last CTA to get here resets the
// queue to zero for the next launch (every CTA has made its last queue[0]
// access by then) and records that in done[1]; done[0] marks the call.
__device__ __forceinline__ void queue_done(uint32_t *queue, volatile int32_t *done)
{
    done[0] = 1;
    if (atomicAdd(queue + 1, 1u) == gridDim.x - 1) {
        queue[0] = 0u;
        queue[1] = 0u;
        done[1] = 1;
    }
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Packed fp32 pairs: two floats in one 64-bit register (element 0 in the
// low word, as in memory), operated on by the f32x2 instructions, each
// element rounded once as by the scalar instruction.
using f32x2 = unsigned long long;
__device__ __forceinline__ f32x2 f2_pack(float x, float y)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(f32x2 v)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// bf16 pair packed in a 32-bit word -> packed fp32 pair (exact).
__device__ __forceinline__ f32x2 bf16x2_to_f2(uint32_t w)
{
    f32x2 r;
    asm("{\n\t.reg .b32 lo, hi;\n\tshl.b32 lo, %1, 16;\n\tand.b32 hi, %1, 0xffff0000;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "=l"(r)
        : "r"(w));
    return r;
}

// bf16 pair packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w)
{
    float2 r;
    r.x = __uint_as_float(w << 16);
    r.y = __uint_as_float(w & 0xffff0000u);
    return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared asynchronous copy (L2-only caching: the KV is
// streamed once per step).
__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst_smem), "l"(src));
}

// Arrive on the mbarrier at `bar` once this thread's earlier cp.async copies
// have landed; the arrival counts toward the barrier's expected count.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

// Prefetch into L2 this CTA's share (part `part` of `parts`) of the 128-byte
// lines that lie wholly inside [p, p + bytes), spread over `nthr` threads.
__device__ __forceinline__ void prefetch_l2_share(const void *p, size_t bytes, int part, int parts, int tid,
                                                  int nthr)
{
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(p) + 127) & ~(uintptr_t)127;
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(p) + bytes;
    if (a1 < a0 + 128)
        return;
    const size_t lines = (a1 - a0) / 128;
    const size_t l0 = lines * part / parts, l1 = lines * (part + 1) / parts;
    for (size_t l = l0 + tid; l < l1; l += nthr)
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a0 + l * 128));
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their writes are visible / let the next grid launch.
__device__ __forceinline__ void grid_dep_wait()
{
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

__device__ __forceinline__ void grid_dep_launch()
{
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Whether every unit of a launch's work queue has been handed out already
// (queued units: n_units less the early CTAs' blocks, `queued_from`).  Reads
// the counter once without taking a unit; a stale value only sends the CTA
// on to the normal path.  A CTA that starts after the launch's early ones
// checks this before its set-up and, with nothing left, leaves at once.
__device__ __forceinline__ bool queue_drained(const uint32_t *queue, int32_t n_units, int32_t queued_from)
{
    const uint32_t taken = *reinterpret_cast<const volatile uint32_t *>(queue);
    return (int64_t)taken >= (int64_t)n_units - queued_from;
}

// queue_done for a CTA leaving before its set-up: the launch's last CTA to
// count itself resets the queue and waits for the launch before this one.
__device__ __forceinline__ void queue_done_idle(uint32_t *queue)
{
    if (atomicAdd(queue + 1, 1u) == gridDim.x - 1) {
        queue[0] = 0u;
        queue[1] = 0u;
        grid_dep_wait();
    }
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::);
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Host: launch `kernel` as a programmatic dependent of the stream's previous
// kernel (it may be scheduled once that kernel's CTAs have all signalled
// grid_dep_launch or exited; its own grid_dep_wait orders what must wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args &&...args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace deft
