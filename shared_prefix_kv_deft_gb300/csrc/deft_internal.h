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
#include <cstddef>
#include <cstdint>
#include <vector>

#include "deft.h"

namespace deft {

constexpr int kPageSize = 16;          // tokens per KV page
constexpr int kMaxChunkTarget = 8192;  // bound on the chunk_target argument
constexpr int kMaxSegsPerChunk = 256;  // packed chunks close at this many segments
constexpr int kFmaMaxRows = 16;        // rows (queries x GQA group) per CUDA-core item
constexpr int kMmaMaxRows = 128;       // rows per tensor-core item (one MMA N extent)
constexpr int kMmaMinRows = 16;        // a chunk with this many rows goes to the tensor path
constexpr int kSharedTokensPerRow = 16;  // long-chunk rule for shared nodes (see planner.cpp)
constexpr int kUnitOverheadTokens = 64;  // fixed cost of a CUDA-core unit, in tokens

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
    // Host-only cost prefix sums over fma_items / fallback_items ([n+1]):
    // entry i is the summed cost of items before i, one KV head each, an
    // item costing its chunk's tokens plus kUnitOverheadTokens.  The
    // CUDA-core launch cuts its units into contiguous, equal-cost CTA ranges.
    std::vector<int64_t> fma_cost;
    std::vector<int64_t> fallback_cost;
    std::vector<int64_t> mma_cost;        // the same over mma_items
    // mma_items are sorted by column bucket b: each of the two softmax
    // warpgroups of an item holds NPH = 16 (b + 1) query rows; bucket b is
    // items [off[b], off[b+1]).
    std::array<int32_t, 5> mma_bucket_off{};
    int32_t num_chunks() const { return (int32_t)chunk_tokens.size(); }
    int32_t num_segments() const { return (int32_t)seg_node.size(); }
    int32_t num_slots() const { return (int32_t)chunk_q.size(); }
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
    int32_t num_fma_items;
    int32_t num_mma_items;
    int32_t num_fallback_items;
    int32_t num_slots;
    int32_t num_queries;
    int32_t mask_words;
};

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
    deft::Partition naive;
    deft_plan_stats stats{};
    // Device copy (deft_plan_upload).
    void *dev_blob = nullptr;
    size_t dev_bytes = 0;
    int dev_device = -1;
    bool uploaded = false;
    deft::DevPartition dev_tree{};
    deft::DevPartition dev_naive{};
};

namespace deft {

// planner.cpp
int build_plan(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
               const int32_t *query_node, int32_t num_queries, int32_t chunk_target,
               int32_t gqa_group, deft_plan_t *plan);

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
    unsigned long long *kprof;  // timestamp slots (development builds only; else null)
    // 1 for the step's first launch: it waits for the stream's earlier work
    // before reading anything.  Every launch of a step is a programmatic
    // dependent of the one before (it may start while that one finishes);
    // later phase-1 launches read only what the first one's wait already
    // covered and write disjoint partials, and each waits for its
    // predecessor before it exits, so the merge's single wait covers them all.
    int32_t wait_prior;
};

// Launchers (return a cudaError_t cast to int; 0 = success).
// One CUDA-core launch over `n` items (device triples at `items`), all of row
// bucket `bucket` (rows <= 2^bucket).
// `cost` points at the items' host cost prefix (n + 1 entries).
int launch_phase1_fma(const AttnArgs &a, const DevPartition &p, const int32_t *items, const int64_t *cost,
                      int32_t n, int bucket, void *stream);

// Persistent phase-1 launches split their units (item-major: unit = item *
// num_kv_heads + head) into contiguous per-CTA ranges of about equal cost:
// CTA b takes units [begin[b], begin[b + 1]).
constexpr int kMaxGrid = 256;
struct CtaRanges {
    int32_t begin[kMaxGrid + 1];
};
// Fills r for `grid` CTAs (grid <= kMaxGrid, <= n * hkv) from the items'
// cost prefix; CTA b starts at the first unit whose cost prefix reaches
// b / grid of the total.
void cta_ranges(const int64_t *cost, int32_t n, int32_t hkv, int grid, CtaRanges &r);
// Streaming multiprocessors of the current device.
int num_sms();
// One tensor-core launch over `n` items of column bucket `bucket`.
int launch_phase1_mma(const AttnArgs &a, const DevPartition &p, const int32_t *items, const int64_t *cost,
                      int32_t n,
                      int bucket, void *stream);
// Row bucket of an item with `rows` rows: smallest b with rows <= 2^b.
inline int row_bucket(int rows) { return rows <= 1 ? 0 : rows <= 2 ? 1 : rows <= 4 ? 2 : rows <= 8 ? 3 : 4; }
// Rows per softmax warpgroup of a tensor-core item with `rows` rows (two
// warpgroups share the rows; each takes a multiple of 16, at most 64).
inline int mma_half_cols(int rows) { return (((rows + 1) / 2) + 15) & ~15; }
inline int mma_bucket(int rows) { return mma_half_cols(rows) / 16 - 1; }
int launch_phase2(const AttnArgs &a, const DevPartition &p, void *out, int32_t out_dtype,
                  float *lse, void *stream);
bool mma_supported(int32_t head_dim);

}  // namespace deft
