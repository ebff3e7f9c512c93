// capi.cu -- the extern "C" entry points declared in include/deft.h.
//
// Plan calls are host-only; deft_plan_upload copies the plan's arrays into
// one device allocation owned by the plan; deft_tree_attn / deft_naive_attn
// / deft_tree_attn_ex validate their arguments and enqueue phase 1
// (tensor-core and CUDA-core kernels, merging in phase 1) or phase 1 and the
// phase-2 merge on the caller's stream without allocating or synchronising.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <utility>

#include <cuda_runtime.h>

#include "deft_internal.h"

namespace deft {

int num_sms()
{
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            n = v;
        else
            return 1;
    }
    return n;
}

WorkLayout work_layout(int64_t slots, int32_t num_q_heads, int32_t head_dim)
{
    auto up = [](size_t x) { return (x + kWorkAlign - 1) / kWorkAlign * kWorkAlign; };
    WorkLayout w{};
    w.o_off = 0;
    w.lse_off = up((size_t)slots * num_q_heads * head_dim * sizeof(float));
    w.total = w.lse_off + up((size_t)slots * num_q_heads * sizeof(float));
    return w;
}

int prepare_step(const void *q, const void *k_pages, const void *v_pages, const int32_t *node_page_off,
                 const int32_t *page_id, int32_t num_pages, int32_t num_q_heads, int32_t num_kv_heads,
                 int32_t head_dim, int32_t page_size, float scale, const deft_plan_t *plan, void *out,
                 int32_t out_dtype, float *lse, int32_t flags, AttnArgs &a, bool &use_mma)
{
    if (!plan || !q || !k_pages || !v_pages || !node_page_off || !page_id || !out || !lse)
        return DEFT_EINVAL;
    if (flags & ~(int32_t)(DEFT_STEP_NAIVE | DEFT_STEP_CUDA_CORES | DEFT_STEP_SEPARATE_MERGE))
        return DEFT_EINVAL;
    if (out_dtype != DEFT_OUT_BF16 && out_dtype != DEFT_OUT_F32)
        return DEFT_EINVAL;
    if (!(scale > 0.f) || !std::isfinite(scale) || num_pages < 1)
        return DEFT_EINVAL;
    if (num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads != 0)
        return DEFT_EINVAL;
    if (((uintptr_t)q | (uintptr_t)k_pages | (uintptr_t)v_pages) & 15u)
        return DEFT_EINVAL;   // the kernels copy q and KV rows in 16-byte pieces
    if ((head_dim != 64 && head_dim != 128) || page_size != kPageSize)
        return DEFT_EUNSUPPORTED;
    const bool naive = (flags & DEFT_STEP_NAIVE) != 0;
    if (num_q_heads / num_kv_heads != plan->gqa_group || (naive && !plan->has_naive) || plan->broken)
        return DEFT_ESTATE;
    use_mma = mma_supported(head_dim) && !(flags & DEFT_STEP_CUDA_CORES);
    // The CUDA-core kernel holds at most kFmaMaxRows rows per item; one query
    // of a larger GQA group needs the tensor-core path.
    if (plan->gqa_group > kFmaMaxRows && !use_mma)
        return DEFT_EUNSUPPORTED;
    a = AttnArgs{};
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
    a.kv_once = naive ? 0 : 1;
    a.out = out;
    a.out_dtype = out_dtype;
    a.lse_out = lse;
    // Rows of single-chunk queries go to out / lse from phase 1 unless every
    // query is to be merged by the merge launch.
    a.direct = (flags & DEFT_STEP_SEPARATE_MERGE) ? 0 : 1;
    return DEFT_OK;
}

}  // namespace deft

namespace {

constexpr size_t kAlign = deft::kWorkAlign;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

template <typename T>
size_t vbytes(const std::vector<T> &v) { return v.size() * sizeof(T); }

int copy_out(const void *src, size_t n, void *dst, size_t bytes)
{
    if (bytes < n)
        return DEFT_EINVAL;
    if (n)
        std::memcpy(dst, src, n);
    return DEFT_OK;
}

// Layout of one partition inside the device blob.
struct Layout {
    size_t off[deft::kPartArrays];
    size_t end;
};

void plan_partition_layout(const deft::Partition &p, size_t &cursor, Layout &L)
{
    const auto arrays = deft::partition_arrays(p);
    for (int i = 0; i < deft::kPartArrays; ++i) {
        L.off[i] = cursor;
        cursor = align_up(cursor + (arrays[i].bytes ? arrays[i].bytes : 4));
    }
    L.end = cursor;
}

void fill_partition(const deft::Partition &p, const Layout &L, uint8_t *host, uint8_t *dev, int32_t num_nodes,
                    int32_t num_queries, int32_t mask_words, deft::DevPartition &d)
{
    const auto arrays = deft::partition_arrays(p);
    for (int i = 0; i < deft::kPartArrays; ++i)
        if (arrays[i].bytes)
            std::memcpy(host + L.off[i], arrays[i].ptr, arrays[i].bytes);
    deft::bind_partition(p, dev, L.off, L.end, num_nodes, num_queries, mask_words, d);
}

// ---- launch tracing (deft_trace_enable / deft_trace_read) ----
struct TraceEntry {
    deft_trace_record rec;
    cudaEvent_t start, stop;
};
bool g_trace_on = false;
std::vector<TraceEntry> g_trace;          // pending records
std::vector<cudaEvent_t> g_event_pool;    // reusable events

cudaEvent_t take_event()
{
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Runs `launch` (returns a cudaError_t as int), bracketed by events when
// tracing is on.
template <typename F>
int traced(const deft_trace_record &rec, void *stream, F &&launch)
{
    if (!g_trace_on)
        return launch();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    TraceEntry t{rec, take_event(), take_event()};
    if (!t.start || !t.stop)
        return (int)cudaErrorMemoryAllocation;
    cudaEventRecord(t.start, st);
    const int rc = launch();
    cudaEventRecord(t.stop, st);
    g_trace.push_back(t);
    return rc;
}

// A step whose arguments have been checked: what dispatch_step needs.
struct Step {
    deft::AttnArgs a;
    bool use_mma = false;
    bool naive = false;
    bool empty = false;   // no query: nothing to launch
    const deft::Partition *hp = nullptr;
    const deft::DevPartition *dp = nullptr;
};

// Every check of a step, before anything is enqueued.
int check_step(const void *q, const void *k_pages, const void *v_pages, const int32_t *node_page_off,
               const int32_t *page_id, int32_t num_pages, int32_t num_q_heads, int32_t num_kv_heads,
               int32_t head_dim, int32_t page_size, float scale, const deft_plan_t *plan, void *out,
               int32_t out_dtype, float *lse, void *workspace, size_t workspace_bytes, int32_t flags, Step &st)
{
    int rc = deft::prepare_step(q, k_pages, v_pages, node_page_off, page_id, num_pages, num_q_heads, num_kv_heads,
                                head_dim, page_size, scale, plan, out, out_dtype, lse, flags, st.a, st.use_mma);
    if (rc != DEFT_OK)
        return rc;
    if (!plan->uploaded)
        return DEFT_ESTATE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DEFT_ECUDA;
    if (dev != plan->dev_device)
        return DEFT_ESTATE;
    st.naive = (flags & DEFT_STEP_NAIVE) != 0;
    st.hp = st.naive ? &plan->naive : &plan->tree;
    st.dp = st.naive ? &plan->dev_naive : &plan->dev_tree;
    const size_t need = deft_workspace_bytes(plan, num_q_heads, head_dim);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 || workspace_bytes < need)
        return DEFT_EWORKSPACE;
    st.empty = plan->num_queries == 0;
    const int64_t slots = std::max(plan->tree.num_slots(), plan->naive.num_slots());
    const deft::WorkLayout wl = deft::work_layout(slots > 0 ? slots : 1, num_q_heads, head_dim);
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    st.a.o_part = reinterpret_cast<float *>(ws + wl.o_off);
    st.a.lse_part = reinterpret_cast<float *>(ws + wl.lse_off);
    return DEFT_OK;
}

int launch_step(const Step &st, void *stream)
{
    if (st.empty)
        return DEFT_OK;
    const deft::LaunchTracer trace = [](const deft_trace_record &rec, void *s, const std::function<int()> &launch) {
        return traced(rec, s, launch);
    };
    return deft::dispatch_step(st.a, *st.dp, *st.hp, st.use_mma, st.naive ? 1 : 0, stream, trace) ? DEFT_ECUDA
                                                                                                 : DEFT_OK;
}

int run_step(const void *q, const void *k_pages, const void *v_pages, const int32_t *node_page_off,
             const int32_t *page_id, int32_t num_pages, int32_t num_q_heads, int32_t num_kv_heads,
             int32_t head_dim, int32_t page_size, float scale, const deft_plan_t *plan, void *out,
             int32_t out_dtype, float *lse, void *workspace, size_t workspace_bytes, int32_t flags, void *stream)
{
    Step st;
    const int rc = check_step(q, k_pages, v_pages, node_page_off, page_id, num_pages, num_q_heads, num_kv_heads,
                              head_dim, page_size, scale, plan, out, out_dtype, lse, workspace, workspace_bytes,
                              flags, st);
    return rc != DEFT_OK ? rc : launch_step(st, stream);
}

}  // namespace

extern "C" {

namespace {

// Builds the host side of a plan into `p` (its device state untouched).
int build_host(const int32_t *parent, const int32_t *node_len, int32_t num_nodes, const int32_t *query_node,
               const int32_t *query_pos, int32_t num_queries, int32_t chunk_target, int32_t gqa_group,
               int32_t flags, deft_plan_t *p)
{
    if (flags & ~(int32_t)(DEFT_PLAN_TREE_ONLY | DEFT_PLAN_TENSOR_PACK))
        return DEFT_EINVAL;
    // A query's whole GQA group shares one tensor-core item, of at most
    // kMmaMaxRows rows (a larger group once made wider items than the
    // kernel has and overran the planner's per-width tables).
    if (gqa_group > deft::kMmaMaxRows)
        return DEFT_EINVAL;
    int rc;
    try {
        rc = deft::build_plan(parent, node_len, num_nodes, query_node, query_pos, num_queries,
                              chunk_target, gqa_group, (flags & DEFT_PLAN_TREE_ONLY) == 0,
                              (flags & DEFT_PLAN_TENSOR_PACK) != 0, p);
    } catch (const std::bad_alloc &) {
        rc = DEFT_ENOMEM;
    }
    if (rc != DEFT_OK)
        return rc;
    size_t cursor = 0;
    Layout lt, ln;
    plan_partition_layout(p->tree, cursor, lt);
    plan_partition_layout(p->naive, cursor, ln);
    p->stats.device_bytes = (int64_t)cursor;
    return DEFT_OK;
}

}  // namespace

int deft_plan_ex(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
                 const int32_t *query_node, const int32_t *query_pos, int32_t num_queries,
                 int32_t chunk_target, int32_t gqa_group, int32_t flags, deft_plan_t **out)
{
    if (!out)
        return DEFT_EINVAL;
    *out = nullptr;
    deft_plan_t *p = new (std::nothrow) deft_plan_t();
    if (!p)
        return DEFT_ENOMEM;
    const int rc = build_host(parent, node_len, num_nodes, query_node, query_pos, num_queries, chunk_target,
                              gqa_group, flags, p);
    if (rc != DEFT_OK) {
        delete p;
        return rc;
    }
    *out = p;
    return DEFT_OK;
}

int deft_plan_rebuild(deft_plan_t *plan, const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
                      const int32_t *query_node, const int32_t *query_pos, int32_t num_queries,
                      int32_t chunk_target, int32_t gqa_group, int32_t flags)
{
    if (!plan)
        return DEFT_EINVAL;
    // The new host side is built into this thread's spare one and swapped
    // in: the plan is left as it was on an error, and the plan's old arrays
    // become the spare's, so that a loop rebuilding a plan every step
    // reuses their storage instead of allocating it again.
    thread_local deft_plan_t spare;
    const int rc = build_host(parent, node_len, num_nodes, query_node, query_pos, num_queries, chunk_target,
                              gqa_group, flags, &spare);
    if (rc != DEFT_OK)
        return rc;   // the plan is left as it was
    // The host side swaps in; the device copy, staging buffer and event stay.
    plan->num_nodes = spare.num_nodes;
    plan->num_queries = spare.num_queries;
    plan->gqa_group = spare.gqa_group;
    plan->chunk_target = spare.chunk_target;
    plan->mask_words = spare.mask_words;
    std::swap(plan->cover, spare.cover);
    std::swap(plan->order, spare.order);
    std::swap(plan->tree, spare.tree);
    std::swap(plan->naive, spare.naive);
    plan->has_naive = spare.has_naive;
    plan->stats = spare.stats;
    std::swap(plan->in_parent, spare.in_parent);
    std::swap(plan->in_len, spare.in_len);
    std::swap(plan->in_qnode, spare.in_qnode);
    std::swap(plan->in_qpos, spare.in_qpos);
    plan->in_tensor_pack = spare.in_tensor_pack;
    std::swap(plan->own_off, spare.own_off);
    std::swap(plan->own_q, spare.own_q);
    std::swap(plan->order_pos, spare.order_pos);
    std::swap(plan->ckpt, spare.ckpt);
    std::swap(plan->thin, spare.thin);
    std::swap(plan->thin_mask, spare.thin_mask);
    plan->uploaded = false;
    plan->noalloc_image_ok = false;
    plan->broken = false;
    return DEFT_OK;
}

int deft_plan_update(deft_plan_t *plan, const int32_t *node_len, int32_t num_nodes)
{
    if (!plan)
        return DEFT_EINVAL;
    const std::vector<int32_t> before = plan->in_len;
    int rc;
    try {
        rc = deft::update_plan(plan, node_len, num_nodes);   // checks everything before it changes anything
    } catch (const std::bad_alloc &) {
        plan->uploaded = false;
        plan->broken = true;
        return DEFT_ENOMEM;
    }
    if (rc != DEFT_OK || plan->in_len == before)
        return rc;   // an error (the plan as it was), or no length changed (its device copy stands)
    size_t cursor = 0;
    Layout lt, ln;
    plan_partition_layout(plan->tree, cursor, lt);
    plan_partition_layout(plan->naive, cursor, ln);
    plan->stats.device_bytes = (int64_t)cursor;
    plan->uploaded = false;
    plan->noalloc_image_ok = false;
    return DEFT_OK;
}

int deft_plan_at(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
                 const int32_t *query_node, const int32_t *query_pos, int32_t num_queries,
                 int32_t chunk_target, int32_t gqa_group, deft_plan_t **out)
{
    return deft_plan_ex(parent, node_len, num_nodes, query_node, query_pos, num_queries, chunk_target,
                        gqa_group, 0, out);
}

int deft_plan(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
              const int32_t *query_node, int32_t num_queries, int32_t chunk_target,
              int32_t gqa_group, deft_plan_t **out)
{
    return deft_plan_at(parent, node_len, num_nodes, query_node, nullptr, num_queries, chunk_target,
                        gqa_group, out);
}

int deft_plan_stats_get(const deft_plan_t *plan, deft_plan_stats *out)
{
    if (!plan || !out)
        return DEFT_EINVAL;
    *out = plan->stats;
    return DEFT_OK;
}

int deft_plan_get(const deft_plan_t *plan, int32_t which, void *dst, size_t bytes)
{
    if (!plan || (!dst && bytes))
        return DEFT_EINVAL;
    const deft::Partition &t = plan->tree, &n = plan->naive;
    auto cp = [&](const auto &v) { return copy_out(v.data(), vbytes(v), dst, bytes); };
    switch (which) {
    case DEFT_A_CHUNK_SEG_OFF: return cp(t.chunk_seg_off);
    case DEFT_A_CHUNK_Q_OFF: return cp(t.chunk_q_off);
    case DEFT_A_CHUNK_Q: return cp(t.chunk_q);
    case DEFT_A_SEG_NODE: return cp(t.seg_node);
    case DEFT_A_SEG_TOK_BEGIN: return cp(t.seg_tok_begin);
    case DEFT_A_SEG_TOK_LEN: return cp(t.seg_tok_len);
    case DEFT_A_SEG_MASK: return cp(t.seg_mask);
    case DEFT_A_CHUNK_MASK: return cp(t.chunk_mask);
    case DEFT_A_Q_SLOT_OFF: return cp(t.q_slot_off);
    case DEFT_A_Q_SLOT: return cp(t.q_slot);
    case DEFT_A_NODE_COVER: return cp(plan->cover);
    case DEFT_A_NODE_ORDER: return cp(plan->order);
    case DEFT_A_FMA_ITEMS: return cp(t.fma_items);
    case DEFT_A_MMA_ITEMS: return cp(t.mma_items);
    case DEFT_A_FALLBACK_ITEMS: return cp(t.fallback_items);
    case DEFT_A_NAIVE_CHUNK_SEG_OFF: return cp(n.chunk_seg_off);
    case DEFT_A_NAIVE_CHUNK_Q: return cp(n.chunk_q);
    case DEFT_A_NAIVE_SEG_NODE: return cp(n.seg_node);
    case DEFT_A_NAIVE_SEG_TOK_BEGIN: return cp(n.seg_tok_begin);
    case DEFT_A_NAIVE_SEG_TOK_LEN: return cp(n.seg_tok_len);
    case DEFT_A_NAIVE_Q_SLOT_OFF: return cp(n.q_slot_off);
    case DEFT_A_NAIVE_Q_SLOT: return cp(n.q_slot);
    case DEFT_A_FMA_DIRECT: return cp(t.fma_direct);
    case DEFT_A_FALLBACK_DIRECT: return cp(t.fallback_direct);
    case DEFT_A_MERGE_Q: return cp(t.merge_q);
    default: return DEFT_EINVAL;
    }
}

int deft_plan_upload(deft_plan_t *plan, void *stream)
{
    if (!plan)
        return DEFT_EINVAL;
    if (plan->broken)
        return DEFT_ESTATE;
    size_t cursor = 0;
    Layout lt, ln;
    plan_partition_layout(plan->tree, cursor, lt);
    plan_partition_layout(plan->naive, cursor, ln);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DEFT_ECUDA;
    if (plan->dev_blob && (plan->dev_bytes < cursor || plan->dev_device != dev)) {
        cudaFree(plan->dev_blob);
        plan->dev_blob = nullptr;
        plan->uploaded = false;
    }
    if (!plan->dev_blob) {
        if (cudaMalloc(&plan->dev_blob, cursor) != cudaSuccess) {
            plan->dev_blob = nullptr;
            return DEFT_ENOMEM;
        }
        plan->dev_bytes = cursor;
        plan->dev_device = dev;
    }
    // The pinned staging buffer: wait for its previous copy, grow it if
    // needed (the only host allocation, kept across uploads and rebuilds).
    cudaEvent_t done = reinterpret_cast<cudaEvent_t>(plan->stage_done);
    if (done && cudaEventSynchronize(done) != cudaSuccess)
        return DEFT_ECUDA;
    if (done && plan->stage_device != dev) {
        cudaEventDestroy(done);
        done = nullptr;
        plan->stage_done = nullptr;
    }
    if (!done) {
        if (cudaEventCreateWithFlags(&done, cudaEventDisableTiming) != cudaSuccess)
            return DEFT_ECUDA;
        plan->stage_done = done;
        plan->stage_device = dev;
    }
    if (plan->host_stage_bytes < cursor) {
        if (plan->host_stage)
            cudaFreeHost(plan->host_stage);
        plan->host_stage = nullptr;
        plan->host_stage_bytes = 0;
        if (cudaHostAlloc(&plan->host_stage, cursor, cudaHostAllocPortable) != cudaSuccess) {
            plan->host_stage = nullptr;
            return DEFT_ENOMEM;
        }
        plan->host_stage_bytes = cursor;
    }
    // Every array is written in full; the alignment padding between arrays
    // is never read.
    uint8_t *host = reinterpret_cast<uint8_t *>(plan->host_stage);
    uint8_t *dev_base = reinterpret_cast<uint8_t *>(plan->dev_blob);
    fill_partition(plan->tree, lt, host, dev_base, plan->num_nodes, plan->num_queries, plan->mask_words,
                   plan->dev_tree);
    fill_partition(plan->naive, ln, host, dev_base, plan->num_nodes, plan->num_queries, plan->mask_words,
                   plan->dev_naive);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(plan->dev_blob, host, cursor, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaEventRecord(done, st) != cudaSuccess)
        return DEFT_ECUDA;
    plan->uploaded = true;
    return DEFT_OK;
}

size_t deft_workspace_bytes(const deft_plan_t *plan, int32_t num_q_heads, int32_t head_dim)
{
    if (!plan || num_q_heads < 1 || head_dim < 1)
        return 0;
    const int64_t slots = std::max(plan->tree.num_slots(), plan->naive.num_slots());
    return deft::work_layout(slots > 0 ? slots : 1, num_q_heads, head_dim).total;
}

int deft_tree_attn(const void *q, const void *k_pages, const void *v_pages,
                   const int32_t *node_page_off, const int32_t *page_id, int32_t num_pages,
                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                   float scale, const deft_plan_t *plan, void *out, int32_t out_dtype, float *lse,
                   void *workspace, size_t workspace_bytes, void *stream)
{
    return run_step(q, k_pages, v_pages, node_page_off, page_id, num_pages, num_q_heads,
                    num_kv_heads, head_dim, page_size, scale, plan, out, out_dtype, lse, workspace,
                    workspace_bytes, 0, stream);
}

int deft_tree_attn_host(const void *q_host, void *q, const void *k_pages, const void *v_pages,
                        const int32_t *node_page_off, const int32_t *page_id, int32_t num_pages,
                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                        float scale, const deft_plan_t *plan, void *out, int32_t out_dtype, float *lse,
                        void *workspace, size_t workspace_bytes, void *out_host, float *lse_host, void *stream)
{
    if (!q_host || !out_host || !lse_host)
        return DEFT_EINVAL;
    Step st;
    int rc = check_step(q, k_pages, v_pages, node_page_off, page_id, num_pages, num_q_heads, num_kv_heads, head_dim,
                        page_size, scale, plan, out, out_dtype, lse, workspace, workspace_bytes, 0, st);
    if (rc != DEFT_OK)
        return rc;
    const size_t rows = (size_t)plan->num_queries * (size_t)num_q_heads;
    if (rows == 0)
        return DEFT_OK;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const size_t out_elem = out_dtype == DEFT_OUT_F32 ? 4 : 2;
    if (cudaMemcpyAsync(q, q_host, rows * head_dim * 2, cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return DEFT_ECUDA;
    rc = launch_step(st, stream);
    if (rc != DEFT_OK)
        return rc;
    if (cudaMemcpyAsync(out_host, out, rows * head_dim * out_elem, cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
        cudaMemcpyAsync(lse_host, lse, rows * sizeof(float), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return DEFT_ECUDA;
    return DEFT_OK;
}

int deft_naive_attn(const void *q, const void *k_pages, const void *v_pages,
                    const int32_t *node_page_off, const int32_t *page_id, int32_t num_pages,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                    float scale, const deft_plan_t *plan, void *out, int32_t out_dtype, float *lse,
                    void *workspace, size_t workspace_bytes, void *stream)
{
    return run_step(q, k_pages, v_pages, node_page_off, page_id, num_pages, num_q_heads,
                    num_kv_heads, head_dim, page_size, scale, plan, out, out_dtype, lse, workspace,
                    workspace_bytes, DEFT_STEP_NAIVE, stream);
}

int deft_tree_attn_ex(const void *q, const void *k_pages, const void *v_pages,
                      const int32_t *node_page_off, const int32_t *page_id, int32_t num_pages,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                      float scale, const deft_plan_t *plan, void *out, int32_t out_dtype, float *lse,
                      void *workspace, size_t workspace_bytes, int32_t flags, void *stream)
{
    return run_step(q, k_pages, v_pages, node_page_off, page_id, num_pages, num_q_heads,
                    num_kv_heads, head_dim, page_size, scale, plan, out, out_dtype, lse, workspace,
                    workspace_bytes, flags, stream);
}

int deft_step_status(deft_plan_t *plan, void *stream, int32_t *code)
{
    if (!plan || !code)
        return DEFT_EINVAL;
    *code = 0;
    if (!plan->uploaded)
        return DEFT_ESTATE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t words[2] = {0u, 0u};
    if (cudaMemcpyAsync(&words[0], plan->dev_tree.status, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(&words[1], plan->dev_naive.status, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return DEFT_ECUDA;
    if ((words[0] && cudaMemsetAsync(plan->dev_tree.status, 0, 4, st) != cudaSuccess) ||
        (words[1] && cudaMemsetAsync(plan->dev_naive.status, 0, 4, st) != cudaSuccess))
        return DEFT_ECUDA;
    *code = (int32_t)(words[0] ? words[0] : words[1]);
    return *code ? DEFT_EDEVICE : DEFT_OK;
}

int deft_check_pages(const int32_t *node_len, int32_t num_nodes, const int32_t *node_page_off,
                     const int32_t *page_id, int64_t num_page_ids, int32_t num_pages, int32_t page_size)
{
    if (!node_len || !node_page_off || num_nodes < 1 || num_page_ids < 0 || num_pages < 1 || page_size < 1 ||
        (num_page_ids > 0 && !page_id))
        return DEFT_EINVAL;
    for (int32_t n = 0; n < num_nodes; ++n) {
        if (node_len[n] < 0)
            return DEFT_EINVAL;
        if (node_len[n] == 0)
            continue;
        const int64_t first = node_page_off[n];
        const int64_t pages = ((int64_t)node_len[n] + page_size - 1) / page_size;
        if (first < 0 || first + pages > num_page_ids)
            return DEFT_ERANGE;
        for (int64_t i = first; i < first + pages; ++i)
            if (page_id[i] < 0 || page_id[i] >= num_pages)
                return DEFT_ERANGE;
    }
    return DEFT_OK;
}

void deft_plan_free(deft_plan_t *plan)
{
    if (!plan)
        return;
    if (plan->stage_done) {
        cudaEventSynchronize(reinterpret_cast<cudaEvent_t>(plan->stage_done));
        cudaEventDestroy(reinterpret_cast<cudaEvent_t>(plan->stage_done));
    }
    if (plan->host_stage)
        cudaFreeHost(plan->host_stage);
    if (plan->dev_blob)
        cudaFree(plan->dev_blob);
    delete plan;
}

const char *deft_status_str(int status)
{
    switch (status) {
    case DEFT_OK: return "ok";
    case DEFT_EINVAL: return "invalid argument";
    case DEFT_ECYCLE: return "parent array has a cycle";
    case DEFT_ERANGE: return "index out of range";
    case DEFT_ENOMEM: return "out of memory";
    case DEFT_EUNSUPPORTED: return "unsupported head_dim, page_size or GQA shape";
    case DEFT_ECUDA: return "CUDA runtime or launch error";
    case DEFT_EWORKSPACE: return "workspace missing, too small or misaligned";
    case DEFT_ESTATE: return "plan not uploaded on this device, built for another GQA group, or without the naive partition";
    case DEFT_EDEVICE: return "a kernel of an earlier step reported a failed wait (see deft_step_status)";
    default: return "unknown status";
    }
}

int deft_version(void) { return 200; }

int deft_trace_enable(int32_t on)
{
    g_trace_on = on != 0;
    return DEFT_OK;
}

int deft_trace_read(deft_trace_record *out, int32_t cap, int32_t *count)
{
    if (!count || (cap > 0 && !out) || cap < 0)
        return DEFT_EINVAL;
    int rc = DEFT_OK;
    int32_t n = 0;
    for (TraceEntry &t : g_trace) {
        float ms = 0.f;
        if (cudaEventSynchronize(t.stop) != cudaSuccess ||
            cudaEventElapsedTime(&ms, t.start, t.stop) != cudaSuccess)
            rc = DEFT_ECUDA;
        if (n < cap) {
            out[n] = t.rec;
            out[n].ms = ms;
            ++n;
        }
        g_event_pool.push_back(t.start);
        g_event_pool.push_back(t.stop);
    }
    g_trace.clear();
    *count = n;
    return rc;
}

}  // extern "C"
