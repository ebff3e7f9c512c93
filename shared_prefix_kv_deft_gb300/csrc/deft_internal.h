// deft_internal.h -- library-internal plan structures and kernel launchers.
//
// The host plan (built by planner.cpp) is a set of flat arrays describing two
// partitions of the tree's KV:
//   * the DeFT partition: chunks of the DFS-preorder flattened tree (Flattened
//     Tree KV Splitting), each shared by the queries whose paths cover it
//     (KV-Guided Grouping; DeFT abstract, DeFT Guide "The DeFT Architecture");
//   * the naive partition: every query's own path cut into pieces, the
//     per-query flash-decoding baseline (DeFT Guide, "The Tree-Attention
//     Bottleneck").
// Both have the same shape, so one set of kernels runs either.
#pragma once

#include <array>
#include <initializer_list>
#include <cstddef>
#include <cstdint>
#include <functional>
#include <vector>

#include "deft.h"

namespace deft {

constexpr int kPageSize = 16;          // tokens per KV page
constexpr int kMaxChunkTarget = 8192;  // bound on the chunk_target argument
constexpr int kMaxSegsPerChunk = 256;  // packed chunks close at this many segments
constexpr int kFmaMaxRows = 16;        // rows (queries x GQA group) per CUDA-core item
constexpr int kFmaItemRows = 8;        // rows per CUDA-core item of a chunk under kMmaMinRows rows
constexpr int kMmaMaxRows = 64;        // rows per tensor-core item (at most 32 columns per softmax warpgroup)
constexpr int kMmaMinRows = 16;        // a chunk with this many rows goes to the tensor path
constexpr int kSharedTokensPerRow = 16;  // long-chunk rule for shared nodes (see planner.cpp)
// Tensor packing: pieces of at least two 128-token tensor-core tiles, so that
// a tile lies in one segment and its pages go by one box per operand half.
constexpr int kTensorPiece = 256;
// Work-queue slots: tensor-core buckets 0-3, CUDA-core buckets 4-8, the
// CUDA-core fallback for tensor-core chunks 9-13.
constexpr int kQueueSlots = 14;
constexpr int kStatusWord = 2 * kQueueSlots;
constexpr int kQueueWords = 2 * kQueueSlots + 2;
inline int queue_slot(int family, int bucket) { return family == 0 ? bucket : family == 1 ? 4 + bucket : 9 + bucket; }

// One partition, host side.  Items are (chunk, q_begin, q_end) triples where
// [q_begin, q_end) indexes the chunk's query list.
struct Partition {
    std::vector<int32_t> chunk_seg_off;   // [C+1]
    std::vector<int32_t> chunk_q_off;     // [C+1]
    std::vector<int32_t> chunk_tokens;    // [C]
    std::vector<int32_t> chunk_q;         // [slots]
    std::vector<int32_t> seg_node;        // [S]
    std::vector<int32_t> seg_tok_begin;   // [S]
    std::vector<int32_t> seg_tok_len;     // [S]
    std::vector<int32_t> seg_chunk_pos;   // [S] token offset of the segment in its chunk
    std::vector<uint64_t> seg_mask;       // [S * W]
    std::vector<uint64_t> chunk_mask;     // [C * W]
    // Segment s's queries as bits over its chunk's query list (bit k: the
    // chunk's k-th query), ceil(|Q_c| / 32) words at seg_lmask_off[s].
    std::vector<int32_t> seg_lmask_off;   // [S+1]
    std::vector<uint32_t> seg_lmask;
    std::vector<int32_t> q_slot_off;      // [Q+1]
    std::vector<int32_t> q_slot;          // [slots]
    std::vector<int32_t> fma_items;       // [3 * n]
    std::vector<int32_t> mma_items;       // [3 * n]
    std::vector<int32_t> fallback_items;  // [3 * n]
    // fma_items and fallback_items are sorted by row bucket b (rows <= 2^b,
    // b = 0..4); bucket b is items [off[b], off[b+1]).
    std::array<int32_t, 6> fma_bucket_off{};
    std::array<int32_t, 6> fallback_bucket_off{};
    // Row masks of each item over its chunk's segments, so kernels need not
    // expand the segments' query masks: for item i, entries
    // [*_rmask_off[i], *_rmask_off[i + 1]) are its chunk's segments in order.
    // CUDA-core items: bit r = item row r.  Tensor-core items: four words
    // per segment, the first warpgroup's columns (rows 0 .. NPH-1) in bits
    // 0-63, the second's (rows NPH ..) in bits 64-127, NPH =
    // mma_half_cols(rows).
    std::vector<uint32_t> fma_rmask, fallback_rmask, mma_rmask;
    std::vector<int32_t> fma_rmask_off, fallback_rmask_off, mma_rmask_off;   // [n+1]
    // Rows of each CUDA-core item whose query has this one partial slot
    // (its whole path lies in the item's chunk): phase 1 writes them to out /
    // lse directly.  Bit r = item row r.
    std::vector<uint32_t> fma_direct, fallback_direct;
    // Queries the merge launch handles: all but those direct rows belong to
    // (queries with no slot, an empty path, get out = 0 and lse = -inf).
    std::vector<int32_t> merge_q;
    // Work queues of the phase-1 launches (two words each: next unit, CTAs
    // finished), zero between launches: uploaded as zeros, reset by each
    // launch's last CTA.  Slot of a launch: queue_slot().  Then the status
    // word (kStatusWord): 0, or the code of the first bounded wait of a
    // kernel of this partition that ran out (read and cleared by
    // deft_step_status), and one word of padding.
    std::vector<uint32_t> queue_words = std::vector<uint32_t>(kQueueWords, 0u);
    // mma_items are sorted by column bucket b: each of the two softmax
    // warpgroups of an item holds NPH = 16 (b + 1) query rows; bucket b is
    // items [off[b], off[b+1]).
    std::array<int32_t, 3> mma_bucket_off{};
    // KV tokens of each bucket's items (chunk tokens summed over the items).
    std::array<int64_t, 5> fma_bucket_tok{}, fallback_bucket_tok{};
    std::array<int64_t, 2> mma_bucket_tok{};
    int32_t num_chunks() const { return (int32_t)chunk_tokens.size(); }
    int32_t num_segments() const { return (int32_t)seg_node.size(); }
    int32_t num_slots() const { return (int32_t)chunk_q.size(); }
    // Back to a fresh partition, keeping the arrays' storage (a plan rebuilt
    // every decode step then allocates nothing once its arrays have grown).
    void reset()
    {
        for (std::vector<int32_t> *v : {&chunk_seg_off, &chunk_q_off, &chunk_tokens, &chunk_q, &seg_node,
                                        &seg_tok_begin, &seg_tok_len, &seg_chunk_pos, &seg_lmask_off, &q_slot_off,
                                        &q_slot, &fma_items, &mma_items, &fallback_items, &fma_rmask_off,
                                        &fallback_rmask_off, &mma_rmask_off, &merge_q})
            v->clear();
        for (std::vector<uint32_t> *v : {&seg_lmask, &fma_rmask, &fallback_rmask, &mma_rmask, &fma_direct,
                                         &fallback_direct})
            v->clear();
        seg_mask.clear();
        chunk_mask.clear();
        queue_words.assign(kQueueWords, 0u);
        fma_bucket_off.fill(0);
        fallback_bucket_off.fill(0);
        mma_bucket_off.fill(0);
        fma_bucket_tok.fill(0);
        fallback_bucket_tok.fill(0);
        mma_bucket_tok.fill(0);
    }
};

// A segment set aside for tensor packing (tokens [b0, b0 + L) of node n; its
// query mask is entry `mask` of the plan's thin_mask, W words each).
struct ThinSeg {
    int32_t n, b0, L, mask;
};
// The tree partition's emission state before one DFS position: chunks and
// segments closed so far, thin segments set aside, tokens emitted, and
// whether a chunk was open there (only a clean position can be resumed).
struct EmitCkpt {
    int32_t chunks, segs, thin;
    int64_t unique;
    bool clean;
};

// Device view of one partition: plain pointers into the plan's device blob,
// passed to kernels by value.
struct DevPartition {
    const int32_t *chunk_seg_off;
    const int32_t *chunk_q_off;
    const int32_t *chunk_tokens;
    const int32_t *chunk_q;
    const int32_t *seg_node;
    const int32_t *seg_tok_begin;
    const int32_t *seg_tok_len;
    const int32_t *seg_chunk_pos;
    const uint64_t *seg_mask;
    const int32_t *seg_lmask_off;
    const uint32_t *seg_lmask;
    const int32_t *q_slot_off;
    const int32_t *q_slot;
    const int32_t *fma_items;
    const int32_t *mma_items;
    const int32_t *fallback_items;
    const uint32_t *fma_rmask;
    const int32_t *fma_rmask_off;
    const uint32_t *fallback_rmask;
    const int32_t *fallback_rmask_off;
    const uint32_t *mma_rmask;          // uint4 per (item, segment)
    const int32_t *mma_rmask_off;       // in uint4 units
    const uint32_t *fma_direct;         // [num_fma_items]
    const uint32_t *fallback_direct;    // [num_fallback_items]
    const int32_t *merge_q;             // [num_merge_q]
    uint32_t *queues;                   // [kQueueSlots][2]
    uint32_t *status;                   // the partition's status word (queues + kStatusWord)
    int32_t num_fma_items;
    int32_t num_mma_items;
    int32_t num_fallback_items;
    int32_t num_slots;
    int32_t num_queries;
    int32_t num_merge_q;
    int32_t mask_words;
    int32_t num_nodes;
    // All of the partition's arrays lie in [arrays, arrays + array_bytes)
    // (kernels prefetch them into L2 at start-up).
    const uint8_t *arrays;
    uint32_t array_bytes;
};

// The partition's device arrays in blob order, and how a blob placed at
// `base` with offsets `off` binds to a DevPartition (shared by the uploaded
// plan and the allocation-free entry point).
constexpr int kPartArrays = 26;
struct ArrayRef {
    const void *ptr;
    size_t bytes;
};
template <typename T>
inline ArrayRef aref(const std::vector<T> &v) { return ArrayRef{v.data(), v.size() * sizeof(T)}; }
inline std::array<ArrayRef, kPartArrays> partition_arrays(const Partition &p)
{
    return {{aref(p.chunk_seg_off), aref(p.chunk_q_off), aref(p.chunk_tokens), aref(p.chunk_q),
             aref(p.seg_node), aref(p.seg_tok_begin), aref(p.seg_tok_len), aref(p.seg_chunk_pos),
             aref(p.seg_mask), aref(p.q_slot_off), aref(p.q_slot), aref(p.fma_items), aref(p.mma_items),
             aref(p.fallback_items), aref(p.seg_lmask_off), aref(p.seg_lmask), aref(p.fma_rmask),
             aref(p.fma_rmask_off), aref(p.fallback_rmask), aref(p.fallback_rmask_off), aref(p.mma_rmask),
             aref(p.mma_rmask_off), aref(p.queue_words), aref(p.fma_direct), aref(p.fallback_direct),
             aref(p.merge_q)}};
}
inline void bind_partition(const Partition &p, const uint8_t *base, const size_t *off, size_t end,
                           int32_t num_nodes, int32_t num_queries, int32_t mask_words, DevPartition &d)
{
    auto i32 = [&](int i) { return reinterpret_cast<const int32_t *>(base + off[i]); };
    auto u32 = [&](int i) { return reinterpret_cast<const uint32_t *>(base + off[i]); };
    d.chunk_seg_off = i32(0);
    d.chunk_q_off = i32(1);
    d.chunk_tokens = i32(2);
    d.chunk_q = i32(3);
    d.seg_node = i32(4);
    d.seg_tok_begin = i32(5);
    d.seg_tok_len = i32(6);
    d.seg_chunk_pos = i32(7);
    d.seg_mask = reinterpret_cast<const uint64_t *>(base + off[8]);
    d.q_slot_off = i32(9);
    d.q_slot = i32(10);
    d.fma_items = i32(11);
    d.mma_items = i32(12);
    d.fallback_items = i32(13);
    d.seg_lmask_off = i32(14);
    d.seg_lmask = u32(15);
    d.fma_rmask = u32(16);
    d.fma_rmask_off = i32(17);
    d.fallback_rmask = u32(18);
    d.fallback_rmask_off = i32(19);
    d.mma_rmask = u32(20);
    d.mma_rmask_off = i32(21);
    d.queues = reinterpret_cast<uint32_t *>(const_cast<uint8_t *>(base) + off[22]);
    d.status = d.queues + kStatusWord;
    d.fma_direct = u32(23);
    d.fallback_direct = u32(24);
    d.merge_q = i32(25);
    d.num_merge_q = (int32_t)p.merge_q.size();
    d.num_fma_items = (int32_t)(p.fma_items.size() / 3);
    d.num_mma_items = (int32_t)(p.mma_items.size() / 3);
    d.num_fallback_items = (int32_t)(p.fallback_items.size() / 3);
    d.num_slots = p.num_slots();
    d.num_queries = num_queries;
    d.mask_words = mask_words;
    d.num_nodes = num_nodes;
    d.arrays = base + off[0];
    d.array_bytes = (uint32_t)(end - off[0]);
}

}  // namespace deft

struct deft_plan_t {
    int32_t num_nodes = 0;
    int32_t num_queries = 0;
    int32_t gqa_group = 1;
    int32_t chunk_target = 0;
    int32_t mask_words = 0;
    std::vector<uint64_t> cover;   // [N * W]
    std::vector<int32_t> order;    // DFS preorder of all nodes
    deft::Partition tree;
    deft::Partition naive;         // empty unless has_naive
    bool has_naive = true;
    deft_plan_stats stats{};
    // Device copy (deft_plan_upload).
    void *dev_blob = nullptr;
    size_t dev_bytes = 0;
    int dev_device = -1;
    bool uploaded = false;
    deft::DevPartition dev_tree{};
    deft::DevPartition dev_naive{};
    // Pinned host staging buffer of deft_plan_upload, kept across uploads and
    // rebuilds, and the event (a cudaEvent_t, created on device stage_device)
    // recorded after its last copy.
    void *host_stage = nullptr;
    size_t host_stage_bytes = 0;
    void *stage_done = nullptr;
    int stage_device = -1;
    // Host image of the tree partition's device arrays for
    // deft_tree_attn_noalloc (built on its first call after a plan build;
    // the capacity is kept across rebuilds).
    std::vector<uint8_t> noalloc_image;
    bool noalloc_image_ok = false;
    // The tree the plan was built from and the state deft_plan_update
    // resumes from: the inputs, the queries inside each node (CSR), each
    // node's DFS position, the emission checkpoints and the thin segments.
    std::vector<int32_t> in_parent, in_len, in_qnode, in_qpos;   // in_qpos empty: no positions
    bool in_tensor_pack = false;
    std::vector<int32_t> own_off, own_q, order_pos;
    std::vector<deft::EmitCkpt> ckpt;
    std::vector<deft::ThinSeg> thin;
    std::vector<uint64_t> thin_mask;
    bool broken = false;   // an update ran out of memory half way: rebuild before use
};

namespace deft {

// planner.cpp
int build_plan(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
               const int32_t *query_node, const int32_t *query_pos, int32_t num_queries,
               int32_t chunk_target, int32_t gqa_group, bool with_naive, bool tensor_pack,
               deft_plan_t *plan);
// The same plan for new node lengths (same structure, queries and options),
// resuming the emission at the last clean checkpoint before the first
// changed node.
int update_plan(deft_plan_t *plan, const int32_t *node_len, int32_t num_nodes);

// Workspace of a step (caller memory, or the allocation-free entry point's
// static array): fp32 partial outputs [slots][Hq][d], then fp32 partial lse
// [slots][Hq], each piece kWorkAlign-aligned.
constexpr size_t kWorkAlign = 256;
struct WorkLayout {
    size_t o_off, lse_off, total;
};
WorkLayout work_layout(int64_t slots, int32_t num_q_heads, int32_t head_dim);

// Arguments every phase-1 kernel receives.
struct AttnArgs {
    const void *q;            // bf16 [Q][Hq][d]
    const void *k_pages;      // bf16 [pages][Hkv][P][d]
    const void *v_pages;
    const int32_t *node_page_off;
    const int32_t *page_id;
    int32_t num_pages;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t gqa_group;
    float scale_log2;         // scale * log2(e): logits are kept in base 2 on device
    float *o_part;            // fp32 [slots][Hq][d]
    float *lse_part;          // fp32 [slots][Hq], base-2 log-sum-exp of the base-2 logits
    void *out;                // [Q][Hq][d] bf16 or fp32 (out_dtype)
    int32_t out_dtype;
    float *lse_out;           // fp32 [Q][Hq], natural log
    // 1: a CUDA-core row whose query has a single partial slot (the item's
    // direct mask) is written to out / lse by phase 1 and the merge launch
    // handles the partition's merge_q only; 0: every row goes to the
    // partials and the merge launch handles every query.
    int32_t direct;
    // 1 for the step's first launch: it waits for the stream's earlier work
    // before reading anything.  Every launch of a step is a programmatic
    // dependent of the one before (it may start while that one finishes);
    // later phase-1 launches read only what the first one's wait already
    // covered and write disjoint partials, and each waits for its
    // predecessor before it exits, so the merge's single wait covers them all.
    int32_t wait_prior;
    // 1 when the launch reads each KV line once (the tree partition, no
    // chunk cut into row blocks): the KV copies then carry an L2 evict-first
    // policy so that the partials stay in L2; 0 for the naive partition,
    // whose prefix re-reads hit L2, and for launches whose row blocks of a
    // chunk each read its KV.
    int32_t kv_once;
};

// The argument checks shared by every step entry point (flags: DEFT_STEP_*).
// On DEFT_OK, `a` holds everything but the workspace pointers (o_part,
// lse_part) and use_mma says whether >= 16-row items run on the
// tensor cores.  The plan's upload state is the caller's to check.
int prepare_step(const void *q, const void *k_pages, const void *v_pages, const int32_t *node_page_off,
                 const int32_t *page_id, int32_t num_pages, int32_t num_q_heads, int32_t num_kv_heads,
                 int32_t head_dim, int32_t page_size, float scale, const deft_plan_t *plan, void *out,
                 int32_t out_dtype, float *lse, int32_t flags, AttnArgs &a, bool &use_mma);

// Launchers (return a cudaError_t cast to int; 0 = success).
//
// A phase-1 launch is persistent: `grid` CTAs, one per SM, take the launch's
// units (item x KV head).  The step's launches run concurrently, so the
// first `early` CTAs of a launch start at once and the rest only on SMs that
// earlier launches leave; each early CTA first takes a contiguous block of
// units (`block`, sized by the dispatcher from the units' estimated costs,
// and never more than 3/4 of an even share of the units by count:
// static_block), and every CTA then takes single units from the launch's
// work queue.
struct LaunchShape {
    int32_t grid;
    int32_t early;   // 1 <= early <= grid
    int32_t block;   // units of each early CTA's block; -1: 3/4 of an even share by count
};
inline int32_t static_block(int32_t units, int32_t early, int32_t block = -1)
{
    const int32_t even = early > 0 ? (int32_t)((int64_t)units * 3 / (4 * (int64_t)early)) : 0;
    return block >= 0 && block < even ? block : even;
}
// One CUDA-core launch over `n` items (device triples at `items`), all of row
// bucket `bucket` (rows <= 2^bucket).
// `rmask` / `rmask_off`: the items' row masks (device; rmask_off indexed
// like items); `direct`: the items' direct-row masks (indexed like items);
// `queue`: the launch's work queue (two device words, zero).
int launch_phase1_fma(const AttnArgs &a, const DevPartition &p, const int32_t *items, const uint32_t *rmask,
                      const int32_t *rmask_off, const uint32_t *direct, int32_t n, int bucket, uint32_t *queue,
                      LaunchShape shape, void *stream);
// Streaming multiprocessors of the current device.
int num_sms();
// Shares `sms` SMs among n concurrent launches of estimated costs cost[i]
// and units[i] units each, the costliest last in the arrays (dispatch.cu).
void shape_launches(const double *cost, const int32_t *units, int n, int sms, LaunchShape *out);
// One tensor-core launch over `n` items of column bucket `bucket` (its rows
// all go to the partials).
int launch_phase1_mma(const AttnArgs &a, const DevPartition &p, const int32_t *items, const uint32_t *rmask,
                      const int32_t *rmask_off, int32_t n, int bucket, uint32_t *queue, LaunchShape shape,
                      void *stream);
// Runs `launch` (returns a cudaError_t as int) on `stream`, recording it
// under `rec` when tracing is on.
using LaunchTracer = std::function<int(const deft_trace_record &rec, void *stream, const std::function<int()> &launch)>;
// Enqueues one step on `stream`: the phase-1 launches of partition dp and
// the phase-2 merge into a.out / a.lse_out (of every query, or with
// a.direct of the partition's merge_q, skipped when that is empty).  `hp` is
// dp's host copy.  Returns a cudaError_t as int.
int dispatch_step(AttnArgs a, const DevPartition &dp, const Partition &hp, bool use_mma, int32_t family,
                  void *stream, const LaunchTracer &trace);
// Row bucket of an item with `rows` rows: smallest b with rows <= 2^b.
inline int row_bucket(int rows) { return rows <= 1 ? 0 : rows <= 2 ? 1 : rows <= 4 ? 2 : rows <= 8 ? 3 : 4; }
// Rows per softmax warpgroup of a tensor-core item with `rows` rows (two
// warpgroups share the rows; each takes a multiple of 16, at most 64).
inline int mma_half_cols(int rows) { return (((rows + 1) / 2) + 15) & ~15; }
inline int mma_bucket(int rows) { return mma_half_cols(rows) / 16 - 1; }
// Estimated SM time per KV token and KV head (ns, with every SM streaming):
// CUDA-core items by row bucket (up to 2 rows the kernel streams at the
// memory rate; above, the per-row FMA work sets the pace), tensor-core items
// by column bucket (the softmax over the item's columns grows with them).
inline double fma_ns_per_token(int bucket)
{
    static const double ns[5] = {10.0, 12.0, 16.0, 32.0, 56.0};
    return ns[bucket];
}
inline double mma_ns_per_token(int bucket)
{
    static const double ns[2] = {14.0, 18.0};
    return ns[bucket];
}
// Buckets whose launches cost little more as one launch at the widest of
// them (estimated SM time at most kCollapse times that of separate
// launches) run as one: each launch pays its own start on every SM, and
// launches of different widths cannot share their work.
constexpr double kCollapse = 1.3;
// The same for the two tensor-core widths.  A narrower margin: at 32 columns
// a warpgroup the softmax of every tile costs twice that at 16.  Measured:
// reasoning tree (1.20 by the estimate) 53.5 us as one launch, 51.7 us as
// two; imbalance tree (1.12) 554 us as one, 582 us as two (its long prefix
// units keep the 32-column launch busy after the 16-column one ends).
constexpr double kCollapseMma = 1.15;
// The merge launch over `nq` queries: queries[i], or i when queries is null.
int launch_phase2(const AttnArgs &a, const DevPartition &p, const int32_t *queries, int32_t nq, void *stream);
bool mma_supported(int32_t head_dim);

}  // namespace deft
