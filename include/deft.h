/*
 * deft.h -- C ABI of the GB300 DeFT tree-attention decode library.
 *
 * The operation (DeFT: Decoding with Flash Tree-attention, arXiv 2404.00242,
 * abstract; aifetchly "DeFT Guide: Flash Tree-Attention for LLM Serving",
 * sections "The DeFT Architecture" and "Deep Dive: Mathematical Formulation"):
 * queries sitting at nodes of a token tree attend, with one softmax each, to
 * the KV tokens of every node on their root-to-node path (the node itself
 * included).  The library splits the tree's KV into chunks (Flattened Tree KV
 * Splitting), reads each chunk once for all queries whose path covers it
 * (KV-Guided Grouping, recorded as a per-segment query bitmask), computes a
 * partial softmax attention with its log-sum-exp per (chunk, query, head)
 * and merges the partials per query by lse weight (a query whose path lies
 * in one CUDA-core chunk needs no merge: its rows are written by the kernel
 * that reads the chunk, the Guide's "Fused In-SRAM Online Softmax
 * Merging").
 *
 * Conventions shared by every call:
 *   - Tree: parent[n] (int32, -1 = root; forests allowed), node_len[n] (int32
 *     tokens, >= 0), query_node[q] (int32 node index).  Host memory.
 *   - KV cache (device, bf16, caller-owned): k_pages and v_pages are
 *     [num_pages][num_kv_heads][page_size][head_dim].  Token t of node n lives
 *     in physical page page_id[node_page_off[n] + t / page_size], slot
 *     t % page_size.  node_page_off is int32 [num_nodes + 1], page_id int32
 *     (both device memory).  Slots past a node's last token are never read.
 *   - q: bf16 [num_queries][num_q_heads][head_dim] (device).
 *   - out: [num_queries][num_q_heads][head_dim], bf16 (DEFT_OUT_BF16) or fp32
 *     (DEFT_OUT_F32); lse: fp32 [num_queries][num_q_heads], natural log of
 *     the softmax normaliser of the scaled logits (device).  A query whose
 *     path holds no token gets out = 0 and lse = -inf.
 *   - Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   - Every call returns a deft_status; none aborts or prints.
 */
#ifndef DEFT_H
#define DEFT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum deft_status {
    DEFT_OK = 0,
    DEFT_EINVAL = -1,        /* null pointer, non-positive size or bad enum value   */
    DEFT_ECYCLE = -2,        /* parent[] does not describe a forest                 */
    DEFT_ERANGE = -3,        /* an index (parent, query_node, ...) is out of range  */
    DEFT_ENOMEM = -4,        /* host or device allocation failed                    */
    DEFT_EUNSUPPORTED = -5,  /* head_dim / page_size / GQA group not compiled in    */
    DEFT_ECUDA = -6,         /* a CUDA runtime call or kernel launch failed          */
    DEFT_EWORKSPACE = -7,    /* workspace null, too small or not 256-byte aligned   */
    DEFT_ESTATE = -8,        /* plan not uploaded, built for another GQA group, or  */
                             /* (deft_naive_attn) built without the naive partition */
    DEFT_EDEVICE = -9        /* deft_step_status: a kernel reported a failed wait   */
} deft_status;

enum { DEFT_OUT_BF16 = 0, DEFT_OUT_F32 = 1 };

/* deft_plan_ex flags. */
enum { DEFT_PLAN_TREE_ONLY = 1, DEFT_PLAN_TENSOR_PACK = 2 };

/* deft_tree_attn_ex flags. */
enum {
    DEFT_STEP_NAIVE = 1,          /* run the naive per-query partition (deft_naive_attn)          */
    DEFT_STEP_CUDA_CORES = 2,     /* run >= 16-row chunks on the CUDA-core kernel too, in items   */
                                  /* of at most 16 rows (same results; a comparison of the paths) */
    DEFT_STEP_SEPARATE_MERGE = 4  /* every query through the partials and the merge launch        */
};

/* Opaque plan: the flattened chunk list, segment bitmasks and per-query
 * partial-slot lists of one tree.  Library-owned; free with deft_plan_free. */
typedef struct deft_plan_t deft_plan_t;

typedef struct deft_plan_stats {
    int32_t num_nodes;
    int32_t num_queries;
    int32_t gqa_group;
    int32_t chunk_target;
    int32_t mask_words;          /* ceil(num_queries / 64): words per bitmask           */
    int32_t num_chunks;          /* KV chunks of the tree plan                          */
    int32_t num_segments;        /* (node, token range) pieces; never cross a node      */
    int32_t num_slots;           /* sum over chunks of |Q_c|: partial results per head  */
    int32_t num_fma_items;       /* phase-1 work items with < 16 rows (CUDA-core path)  */
    int32_t num_mma_items;       /* phase-1 work items with >= 16 rows (tensor path)    */
    int32_t num_fallback_items;  /* the >= 16-row chunks cut into <= 16-row items       */
    int32_t max_chunk_tokens;
    int32_t max_slots_per_query;
    int32_t naive_num_chunks;    /* per-query flash-decoding partition (0 if tree-only) */
    int32_t naive_num_slots;
    int32_t naive_num_segments;
    int32_t num_merge_queries;   /* queries of the tree plan the merge launch handles     */
    int32_t reserved0;
    int64_t unique_tokens;       /* tokens on at least one query path                   */
    int64_t naive_tokens;        /* sum over queries of their path tokens               */
    int64_t planned_tokens;      /* sum of chunk lengths; equals unique_tokens          */
    int64_t pair_tokens;         /* sum over chunks of tokens * |Q_c| (incl. masked)    */
    int64_t device_bytes;        /* size of the device copy deft_plan_upload makes      */
} deft_plan_stats;

/* Arrays a plan exposes through deft_plan_get (host copies, for tests and
 * tools).  Element type and count are given beside each name. */
typedef enum deft_plan_array {
    DEFT_A_CHUNK_SEG_OFF = 0,   /* int32  [num_chunks + 1]  segment range of chunk c          */
    DEFT_A_CHUNK_Q_OFF = 1,     /* int32  [num_chunks + 1]  range of chunk c in CHUNK_Q       */
    DEFT_A_CHUNK_Q = 2,         /* int32  [num_slots]       query ids; the index is the slot  */
    DEFT_A_SEG_NODE = 3,        /* int32  [num_segments]                                      */
    DEFT_A_SEG_TOK_BEGIN = 4,   /* int32  [num_segments]    first token inside the node       */
    DEFT_A_SEG_TOK_LEN = 5,     /* int32  [num_segments]                                      */
    DEFT_A_SEG_MASK = 6,        /* uint64 [num_segments * mask_words]  queries that see it    */
    DEFT_A_CHUNK_MASK = 7,      /* uint64 [num_chunks * mask_words]    union over segments    */
    DEFT_A_Q_SLOT_OFF = 8,      /* int32  [num_queries + 1]                                   */
    DEFT_A_Q_SLOT = 9,          /* int32  [num_slots]       partial slots of each query       */
    DEFT_A_NODE_COVER = 10,     /* uint64 [num_nodes * mask_words]     coverage bitsets       */
    DEFT_A_NODE_ORDER = 11,     /* int32  [num_nodes]       DFS preorder of all nodes         */
    DEFT_A_FMA_ITEMS = 12,      /* int32  [num_fma_items * 3]  (chunk, q_begin, q_end)        */
    DEFT_A_MMA_ITEMS = 13,      /* int32  [num_mma_items * 3]  q range local to the chunk     */
    DEFT_A_FALLBACK_ITEMS = 14, /* int32  [num_fallback_items * 3]                            */
    DEFT_A_NAIVE_CHUNK_SEG_OFF = 15, /* int32 [naive_num_chunks + 1]                          */
    DEFT_A_NAIVE_CHUNK_Q = 16,       /* int32 [naive_num_slots] (one query per chunk)         */
    DEFT_A_NAIVE_SEG_NODE = 17,      /* int32 [naive_num_segments]                            */
    DEFT_A_NAIVE_SEG_TOK_BEGIN = 18, /* int32 [naive_num_segments]                            */
    DEFT_A_NAIVE_SEG_TOK_LEN = 19,   /* int32 [naive_num_segments]                            */
    DEFT_A_NAIVE_Q_SLOT_OFF = 20,    /* int32 [num_queries + 1]                               */
    DEFT_A_NAIVE_Q_SLOT = 21,        /* int32 [naive_num_slots]                               */
    DEFT_A_FMA_DIRECT = 22,     /* uint32 [num_fma_items]   bit r: row r goes to out directly */
    DEFT_A_FALLBACK_DIRECT = 23,/* uint32 [num_fallback_items]  (always 0)                    */
    DEFT_A_MERGE_Q = 24,        /* int32  [num_merge_queries]  queries the merge launch takes */
    DEFT_A_COUNT = 25
} deft_plan_array;

/*
 * deft_plan -- build the plan of one tree (host only, no CUDA call).
 * Follows the DeFT abstract (KV-Guided Grouping; Flattened Tree KV
 * Splitting) and the Guide's section "The DeFT Architecture".
 *   - Validates the tree: parent in [-1, num_nodes) (DEFT_ERANGE) and not a
 *     cycle (DEFT_ECYCLE), node_len >= 0 (DEFT_EINVAL), query_node in
 *     [0, num_nodes) (DEFT_ERANGE), num_nodes >= 1, num_queries >= 0.
 *   - cover[n]: bit q set iff n lies on query q's root-to-node path.
 *   - Flattens nodes in DFS preorder (roots, then children, ascending id),
 *     cuts every node's tokens into segments and packs short segments into
 *     chunks of at most chunk_target tokens (1 <= chunk_target <= 8192); a
 *     heavily shared node gets longer chunks so that its partial-result
 *     traffic stays small next to its KV traffic.  Every (query, node on its
 *     path, token) triple lands in exactly one chunk that lists the query.
 *   - gqa_group = num_q_heads / num_kv_heads of the layer the plan will run
 *     (decides which chunks reach 16 rows = |Q_c| * gqa_group); 1..64 (a
 *     query's whole group shares one tensor-core item of at most 64 rows;
 *     above 64, DEFT_EINVAL).
 *   - The naive per-query partition (deft_naive_attn) cuts each query's
 *     path tokens into pieces of chunk_target tokens.
 * On success *out owns the plan (free with deft_plan_free).  The input arrays
 * are not retained.
 */
int deft_plan(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
              const int32_t *query_node, int32_t num_queries, int32_t chunk_target,
              int32_t gqa_group, deft_plan_t **out);

/*
 * deft_plan_at -- deft_plan for queries that sit at token positions of their
 * nodes (tree verification or prefill with multi-token nodes; the Guide's
 * causal tree mask, section "Deep Dive", taken at token granularity).
 *   query_pos[q] in [-1, node_len[query_node[q]]): the query attends tokens
 *   0..query_pos[q] of its own node and every token of the nodes above it;
 *   -1 means the node's last token, as in deft_plan.  query_pos NULL: all
 *   -1 (exactly deft_plan).  A position outside its node: DEFT_ERANGE.
 * A node holding queries at several positions is cut where each query's
 * part ends, so that every segment keeps one query set; the kernels run the
 * plan unchanged.  Other arguments, results and errors as deft_plan.
 */
int deft_plan_at(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
                 const int32_t *query_node, const int32_t *query_pos, int32_t num_queries,
                 int32_t chunk_target, int32_t gqa_group, deft_plan_t **out);

/*
 * deft_plan_ex -- deft_plan_at with option flags (0 = exactly deft_plan_at).
 *   DEFT_PLAN_TREE_ONLY: skip the naive per-query partition (a plan for
 *   deft_tree_attn alone: about half the planning time and a smaller device
 *   copy).  Its naive partition is empty (naive_num_* = 0, the naive arrays
 *   have no element but naive_q_slot_off's num_queries + 1 zeros) and
 *   deft_naive_attn on it returns DEFT_ESTATE.  naive_tokens is still
 *   counted.
 *   DEFT_PLAN_TENSOR_PACK: for layers run at head_dim 128 (the tensor-core
 *   path).  Segments whose queries make fewer than 16 rows (queries x
 *   gqa_group) are laid side by side in chunks of 16 to 64 rows, a piece of
 *   about chunk_target / m tokens from each of m consecutive such segments
 *   (the Guide's flattened-tree tile shared by several branches, other
 *   branches' queries masked), so that they run on the tensor cores instead
 *   of the CUDA cores.  Every token is still read once; a query gets one
 *   partial per piece.  At other head sizes the packed chunks run on CUDA
 *   cores at their full row count: leave the flag off there.
 * Unknown flag bits: DEFT_EINVAL.  Other arguments, results and errors as
 * deft_plan_at.
 */
int deft_plan_ex(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
                 const int32_t *query_node, const int32_t *query_pos, int32_t num_queries,
                 int32_t chunk_target, int32_t gqa_group, int32_t flags, deft_plan_t **out);

/*
 * deft_plan_rebuild -- re-plan a new tree into an existing plan (a decode
 * loop, whose tree changes every step): the same arguments, checks and
 * results as deft_plan_ex, but the plan keeps its device allocation (grown
 * only when the new plan needs more) and its pinned staging buffer, so the
 * next deft_plan_upload allocates nothing.  On success the plan is marked
 * not uploaded (deft_tree_attn returns DEFT_ESTATE until deft_plan_upload);
 * on error the plan is left exactly as it was.  The device copy of the old
 * plan stays valid until the next upload, which is stream-ordered: a step
 * still reading it must be ordered before that upload (same stream, or
 * synchronised streams).  A CUDA graph that captured a step of this plan
 * holds the old launch shapes and device addresses: capture it again after
 * a rebuild.  The new host arrays are built in a spare host plan of the
 * calling thread and swapped in; the spare keeps the replaced arrays, whose
 * storage the thread's next rebuild (of any plan) reuses, until the thread
 * exits.  DEFT_EINVAL for a null plan.
 */
int deft_plan_rebuild(deft_plan_t *plan, const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
                      const int32_t *query_node, const int32_t *query_pos, int32_t num_queries,
                      int32_t chunk_target, int32_t gqa_group, int32_t flags);

/*
 * deft_plan_update -- re-plan the plan's tree after its node lengths changed
 * (DeFT Guide, "Production Engineering and Kernel Deployment Best
 * Practices": the tree grows and is pruned between decode steps): tokens
 * appended to nodes, or subtrees pruned by setting their nodes' lengths to
 * 0 (a pruned node produces no segment; a query whose whole path is pruned
 * gets out = 0, lse = -inf).  The parents, queries, positions, chunk_target,
 * gqa_group and flags stay those of the last build; a change to any of them
 * (new nodes, queries moved) goes through deft_plan_rebuild.
 *   - The result equals, array for array, what deft_plan_rebuild makes of
 *     the same tree.  The work done is smaller: the forest check, coverage
 *     bitsets and DFS order are kept, and the chunks are re-emitted from the
 *     last point at or before the first changed node (in DFS order) where no
 *     chunk was open; the query lists, work items and the naive partition
 *     are recomputed.
 *   - num_nodes must be the plan's; node_len >= 0 (DEFT_EINVAL); a query
 *     position beyond its node's new length: DEFT_ERANGE.  On these errors
 *     the plan is left as it was.  DEFT_ENOMEM leaves it unusable until a
 *     deft_plan_rebuild (steps on it return DEFT_ESTATE).
 *   - When a length changed, the plan is marked not uploaded (upload again
 *     before the next step); when none did, nothing changes.
 */
int deft_plan_update(deft_plan_t *plan, const int32_t *node_len, int32_t num_nodes);

/* Plan statistics (host).  DEFT_EINVAL on null arguments. */
int deft_plan_stats_get(const deft_plan_t *plan, deft_plan_stats *out);

/* Copy one plan array (see deft_plan_array for type and length) to host
 * memory `dst` of `bytes` bytes.  DEFT_EINVAL if `bytes` is smaller than the
 * array or `which` is unknown. */
int deft_plan_get(const deft_plan_t *plan, int32_t which, void *dst, size_t bytes);

/* Copy the plan to device memory owned by the plan (allocated on the first
 * call, on the current device, and re-allocated only when a rebuilt plan
 * needs more or the device changes).  The copy goes through a pinned host
 * staging buffer owned by the plan (allocated on the first call, grown when
 * needed) and is enqueued on `stream` (a cudaStream_t, NULL = legacy
 * default stream); the call returns before it ends, after waiting for the
 * plan's previous upload copy, if any, to finish.  Call before
 * deft_tree_attn / deft_naive_attn on the same device.  DEFT_ENOMEM when an
 * allocation fails, DEFT_ECUDA when a copy or event call fails. */
int deft_plan_upload(deft_plan_t *plan, void *stream);

/* Bytes of device workspace deft_tree_attn and deft_naive_attn need for this
 * plan: fp32 partial outputs and lse values for every slot and query head of
 * either partition (the larger).  Returns 0 on bad arguments. */
size_t deft_workspace_bytes(const deft_plan_t *plan, int32_t num_q_heads, int32_t head_dim);

/*
 * deft_tree_attn -- one tree-attention decode step (DeFT Guide, "Deep Dive":
 * online-softmax tile accumulation; DeFT abstract: partial results merged
 * per query).  Phase 1 reads every chunk's KV once per KV head and writes
 * (o, lse) partials for each (chunk, query, query head) into the
 * workspace; phase 2 merges each query's partials by lse weight into out
 * and lse.  A query whose whole path lies in one chunk of fewer than 16 rows
 * has a single partial: the CUDA-core kernel writes its rows to out / lse
 * directly, and phase 2 runs only over the other queries (and not at all
 * when there are none).  Chunks with >= 16 rows run on tcgen05 tensor cores
 * (head_dim 128), the others on CUDA-core FMA.
 *   q, k_pages, v_pages, node_page_off, page_id, out, lse, workspace: device
 *     pointers as described at the top of this file; q, k_pages and v_pages
 *     must be 16-byte aligned (else DEFT_EINVAL); workspace must be
 *     256-byte aligned and hold deft_workspace_bytes(plan, num_q_heads,
 *     head_dim) bytes; its contents need not be initialised.  num_pages is the
 *     number of pages of k_pages / v_pages (it sizes the tensor maps); the
 *     kernels do not check page_id's values or node_page_off against it:
 *     deft_check_pages checks a layout on the host, once per change.
 *   head_dim in {64, 128}; page_size 16; num_q_heads a multiple of
 *     num_kv_heads whose quotient equals the plan's gqa_group (else
 *     DEFT_ESTATE); scale > 0 multiplies q.k (pass 1/sqrt(head_dim)).
 * Never allocates, never synchronises the host; stream-ordered on `stream`.
 * The plan's device copy holds the phase-1 launches' work queues, so one
 * plan serves one step at a time: steps that use the same plan must be
 * ordered (one stream, or synchronised streams).  Launch failures return
 * DEFT_ECUDA.
 */
int deft_tree_attn(const void *q, const void *k_pages, const void *v_pages,
                   const int32_t *node_page_off, const int32_t *page_id, int32_t num_pages,
                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                   int32_t page_size, float scale, const deft_plan_t *plan, void *out,
                   int32_t out_dtype, float *lse, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * deft_naive_attn -- the same step computed the per-query flash-decoding way
 * (DeFT Guide, "The Tree-Attention Bottleneck": every branch re-reads the
 * shared prefix): each query's path is split into pieces of chunk_target
 * tokens, each piece read for that query alone, then the same merge.  Same
 * arguments, results and rules as deft_tree_attn; the in-run IO comparison.
 * A plan made with DEFT_PLAN_TREE_ONLY: DEFT_ESTATE.
 */
int deft_naive_attn(const void *q, const void *k_pages, const void *v_pages,
                    const int32_t *node_page_off, const int32_t *page_id, int32_t num_pages,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t page_size, float scale, const deft_plan_t *plan, void *out,
                    int32_t out_dtype, float *lse, void *workspace, size_t workspace_bytes,
                    void *stream);

/*
 * deft_tree_attn_ex -- deft_tree_attn / deft_naive_attn with option flags
 * (DEFT_STEP_*; 0 = deft_tree_attn).  DEFT_STEP_CUDA_CORES runs the
 * tensor-core chunks on the CUDA-core kernel (head_dim 128 only needs it to
 * compare the two paths; a GQA group above 16 returns DEFT_EUNSUPPORTED),
 * DEFT_STEP_SEPARATE_MERGE sends every query, single-chunk ones included,
 * through the partials and the merge launch.  Results equal those without
 * flags within the tolerances of floating point (SEPARATE_MERGE gives the
 * same values: a single partial merges to itself).  Unknown flag bits: DEFT_EINVAL.  Other arguments and errors as
 * deft_tree_attn.
 */
int deft_tree_attn_ex(const void *q, const void *k_pages, const void *v_pages,
                      const int32_t *node_page_off, const int32_t *page_id, int32_t num_pages,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                      float scale, const deft_plan_t *plan, void *out, int32_t out_dtype, float *lse,
                      void *workspace, size_t workspace_bytes, int32_t flags, void *stream);

/*
 * deft_tree_attn_host -- deft_tree_attn with the step's per-call inputs and
 * outputs in host memory (no counterpart on the pages; the decode loop's
 * round trip in one call).  On `stream`, in order: q_host (num_queries x
 * num_q_heads x head_dim bf16) is copied into q, the step runs as
 * deft_tree_attn, and out and lse are copied into out_host (out_dtype
 * elements) and lse_host.  q, out, lse and workspace are device buffers as
 * for deft_tree_attn; the KV cache and page table stay on the device.  With
 * pinned host memory the copies are asynchronous and the call returns before
 * they finish: synchronise the stream before reading out_host / lse_host and
 * keep q_host unchanged until then.  Pageable host memory works too (CUDA
 * then stages the copies, which may wait for the stream).  Null host
 * pointers: DEFT_EINVAL; a failed copy: DEFT_ECUDA; other arguments and
 * errors as deft_tree_attn (checked before anything is enqueued).
 */
int deft_tree_attn_host(const void *q_host, void *q, const void *k_pages, const void *v_pages,
                        const int32_t *node_page_off, const int32_t *page_id, int32_t num_pages,
                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                        float scale, const deft_plan_t *plan, void *out, int32_t out_dtype, float *lse,
                        void *workspace, size_t workspace_bytes, void *out_host, float *lse_host,
                        void *stream);

/*
 * deft_step_status -- device-side failures of earlier steps of this plan (no
 * counterpart on the pages).  Every wait of a kernel on another part of its
 * CTA is bounded; one that runs out writes NaN into the rows of its launch
 * and records a code in the plan's device memory.  This call copies the
 * codes of both partitions back on `stream`, waits for that copy (it
 * synchronises the host with the stream) and clears them.  *code = 0 and
 * DEFT_OK when no step failed; otherwise *code = the first failing wait's
 * code and DEFT_EDEVICE: out / lse of the failed steps are not valid.
 * Steps of deft_tree_attn_noalloc are not covered (see there).
 * DEFT_ESTATE if the plan was never uploaded, DEFT_ECUDA if a copy fails.
 */
int deft_step_status(deft_plan_t *plan, void *stream, int32_t *code);

/*
 * deft_check_pages -- host check of a paged KV layout (DeFT Guide,
 * "Production Engineering", paged KV-cache compatibility): for every node
 * with tokens, its ceil(node_len / page_size) page-table entries
 * node_page_off[n] .. lie inside page_id[0 .. num_page_ids) and each names a
 * page in [0, num_pages).  All arrays are host memory (node_len and
 * node_page_off have num_nodes entries at least).  DEFT_OK, DEFT_ERANGE at
 * the first violation, DEFT_EINVAL on bad arguments.  The kernels read
 * page_id without checking it: run this once whenever the layout changes.
 */
int deft_check_pages(const int32_t *node_len, int32_t num_nodes, const int32_t *node_page_off,
                     const int32_t *page_id, int64_t num_page_ids, int32_t num_pages, int32_t page_size);

/*
 * deft_tree_attn_noalloc -- deft_tree_attn for callers that cannot allocate
 * device memory.  The paper has no counterpart; this is a library service.
 *
 * deft_tree_attn needs a workspace and an uploaded plan, and uploading calls
 * cudaMalloc.  Some callers may not do either: a runtime that reserves all
 * device memory for its own pool allocator and gives its kernels no way to
 * take more (a cudaMalloc there fails, or takes memory the pool counts on),
 * a plugin interface that hands the plugin its buffers and forbids it to
 * allocate during execution, and a serving loop that cannot afford the
 * device-wide synchronisation a cudaMalloc or cudaFree may cause.  This call
 * takes the same inputs and outputs as deft_tree_attn but no workspace, and
 * the plan need not be uploaded: the plan's tree arrays are copied, with one
 * cudaMemcpyAsync on `stream` from a host image the plan keeps (pageable
 * memory: CUDA may wait for the stream's earlier work before it stages the
 * bytes, and returns once they are staged), into
 * one static device array of DEFT_NOALLOC_SCRATCH_BYTES (64 MiB) that every
 * GPU loading the library holds until the process exits; the partials live
 * there too.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - A plan whose arrays plus partials (slots * num_q_heads * (head_dim + 1)
 *     fp32 values), in 256-byte aligned pieces, exceed the array is rejected
 *     with DEFT_EWORKSPACE before anything is enqueued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.
 *   - All calls share the array and it keeps the last call's contents: each
 *     call rewrites the plan arrays (work queues included) before its
 *     kernels run, and nothing else in it has to start at zero.  Calls that
 *     may overlap on the GPU (other streams, unsynchronised host threads)
 *     race and must not be made.
 *   - A failed wait inside a kernel shows only as NaN in out / lse (the
 *     status words live in the array; deft_step_status does not see them).
 * Results are those of deft_tree_attn; other arguments and errors as there.
 */
#define DEFT_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int deft_tree_attn_noalloc(const void *q, const void *k_pages, const void *v_pages,
                           const int32_t *node_page_off, const int32_t *page_id,
                           int32_t num_pages, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t page_size, float scale,
                           const deft_plan_t *plan, void *out, int32_t out_dtype, float *lse,
                           void *stream);

/*
 * Per-launch kernel timing, for measurement tools (no counterpart on the
 * pages).  While enabled, every kernel launch made by deft_tree_attn and
 * deft_naive_attn is bracketed by two CUDA events recorded on the launch
 * stream.  deft_trace_read waits for those events, writes up to `cap`
 * records (in launch order) to `out`, sets *count to the number written and
 * forgets all pending records.  Events are created on first use and reused;
 * the library is not thread-safe while tracing is on.
 */
typedef struct deft_trace_record {
    int32_t kernel;   /* DEFT_K_* */
    int32_t family;   /* 0 tree partition, 1 naive partition                  */
    int32_t bucket;   /* row bucket b (rows <= 2^b) of a CUDA-core launch     */
    int32_t fallback; /* 1 if the launch ran >= 16-row chunks on CUDA cores   */
    int32_t items;    /* work items (grid = items * num_kv_heads for phase 1) */
    float ms;         /* event-measured duration                              */
} deft_trace_record;

enum { DEFT_K_PHASE1_FMA = 0, DEFT_K_PHASE1_MMA = 1, DEFT_K_PHASE2 = 2 };

int deft_trace_enable(int32_t on);
int deft_trace_read(deft_trace_record *out, int32_t cap, int32_t *count);

/*
 * KV page pool with reference counts (DeFT Guide, "Production Engineering
 * and Kernel Deployment Best Practices", "Paged KV-Cache Compatibility" and
 * "Tree Pruning Memory Management": the pages of pruned branches go back to
 * the pool at once, O(1) a page, without copying).  Host bookkeeping only:
 * the pool hands out page numbers of the caller's k_pages / v_pages, and the
 * caller builds node_page_off / page_id from them.  A page holds one
 * reference per owner (deft_pages_retain adds one: a page shared by two page
 * tables); it is free again when the last is released.
 *   deft_pages_create: a pool of num_pages pages, all free (page 0 handed out
 *     first).  DEFT_EINVAL for num_pages < 1.
 *   deft_pages_alloc: n free pages, each with one reference, into page_ids;
 *     DEFT_ENOMEM if fewer than n are free (nothing taken).
 *   deft_pages_retain / deft_pages_release: one more / one less reference on
 *     each listed page (a page may be listed more than once).  A page id out
 *     of range: DEFT_ERANGE; a free page, or more releases than references:
 *     DEFT_ESTATE.  On an error nothing changes.
 *   deft_pages_free_count: free pages (-1 for a null pool).
 *   deft_pages_refcount: references of one page (-1 out of range).
 * Not thread-safe; deft_pages_free(NULL) is a no-op.
 */
typedef struct deft_pages_t deft_pages_t;
int deft_pages_create(int32_t num_pages, deft_pages_t **out);
void deft_pages_free(deft_pages_t *pool);
int deft_pages_alloc(deft_pages_t *pool, int32_t n, int32_t *page_ids);
int deft_pages_retain(deft_pages_t *pool, int32_t n, const int32_t *page_ids);
int deft_pages_release(deft_pages_t *pool, int32_t n, const int32_t *page_ids);
int32_t deft_pages_free_count(const deft_pages_t *pool);
int32_t deft_pages_refcount(const deft_pages_t *pool, int32_t page);

/* Free a plan and its device copy (the caller must ensure no kernel using it
 * is still running).  NULL is a no-op. */
void deft_plan_free(deft_plan_t *plan);

/* Static English text of a status code. */
const char *deft_status_str(int status);

/* Library version as major * 10000 + minor * 100 + patch. */
int deft_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DEFT_H */
