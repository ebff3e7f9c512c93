// planner.cpp -- host tree planner: validation, coverage bitsets, DFS
// flattening, segment/chunk construction and work items.
//
// KV-Guided Grouping (DeFT abstract; DeFT Guide, "The DeFT Architecture",
// item 1): work is grouped by KV, not by query.  A node's KV is read once
// for every query whose root-to-node path contains it; the set of those
// queries is the node's coverage bitset, and a chunk lists the union of its
// segments' sets.
//
// Flattened Tree KV Splitting (DeFT abstract; Guide, item 2, where chunks of
// B_KV = 128 tokens are the example): the tree is flattened into one token
// sequence (DFS preorder) and cut into chunks of roughly equal size.  Here a
// chunk is made of segments, each a token range of a single node, so that the
// per-segment query set is exact.  Readings taken where the pages are silent:
//   * Order: roots by ascending id, each subtree in preorder with children by
//     ascending id.  The order changes only the partition, never a result.
//   * Short nodes (at most chunk_target / 2 tokens) are packed, in preorder,
//     into chunks of at most chunk_target tokens and at most
//     kMaxSegsPerChunk segments; a node whose query set and the chunk's are
//     not one within the other joins only if it is tiny (at most
//     chunk_target / 4 tokens), since the chunk's rows, and with them the
//     work on every token of it, grow by its queries.
//   * A longer node is cut into equal page-aligned pieces of about
//     T = max(chunk_target, kSharedTokensPerRow * rows) tokens, rows being
//     |cover| * gqa_group.  Each (chunk, query, head) writes one fp32
//     partial of head_dim + 1 values, so keeping T >= 16 rows bounds the
//     partial-result write plus read to about 1/8 of the chunk's KV bytes.
//     (The Guide's claim that partials vanish entirely, section "Fused
//     In-SRAM Online Softmax Merging", is read as "made small", which is what
//     the abstract's "nearly 100% IO reduction for partial results" says.)
//   * Nodes with no token or no query on them produce no segment.
//   * With tensor packing (DEFT_PLAN_TENSOR_PACK, for head_dim 128), the
//     segments of kMmaMinRows / 4 to kMmaMinRows - 1 rows and more than
//     chunk_target / 4 tokens (tiny ones pack as above), which would run on
//     CUDA cores at a cost per token that grows with their rows, are instead
//     laid side by side: a chunk takes a piece of max(kTensorPiece,
//     chunk_target / m) tokens from each of the next m such segments
//     (longest first), m the fewest that bring
//     the chunk to kMmaMinRows rows (at most kMmaMaxRows), so that it runs
//     on the tensor cores, each row masked to its own segments.  This is the
//     Guide's tile of the flattened tree shared by several branches, the
//     queries of the other branches masked ("Deep Dive", the fused tiling
//     layout; "Flattened Tree KV Splitting": equal-sized tiles).  Each token
//     is still read once; a query gets one partial per piece of its
//     segments.
#include <algorithm>
#include <cstring>
#include <numeric>

#include "deft_internal.h"

namespace deft {
namespace {

int popcount_words(const uint64_t *w, int32_t words)
{
    int c = 0;
    for (int32_t i = 0; i < words; ++i)
        c += __builtin_popcountll(w[i]);
    return c;
}

struct Builder {
    Partition &p;
    int32_t W;
    int32_t cur_chunk_tokens = 0;
    int32_t cur_chunk_segs = 0;
    bool open = false;
    std::vector<uint64_t> cur_mask;

    // Capacity for about `chunks` chunks of `segs` segments in all.
    Builder(Partition &part, int32_t words, int64_t chunks, int64_t segs)
        : p(part), W(words), cur_mask(words, 0)
    {
        p.chunk_seg_off.reserve(chunks + 1);
        p.chunk_tokens.reserve(chunks);
        p.chunk_mask.reserve(chunks * W);
        p.seg_node.reserve(segs);
        p.seg_tok_begin.reserve(segs);
        p.seg_tok_len.reserve(segs);
        p.seg_chunk_pos.reserve(segs);
        p.seg_mask.reserve(segs * W);
        p.chunk_seg_off.push_back(0);
    }
    // Resumes `part` with its first `chunks` chunks and `segs` segments, no
    // chunk open (a checkpoint of an earlier build).
    Builder(Partition &part, int32_t words, int32_t chunks, int32_t segs, bool)
        : p(part), W(words), cur_mask(words, 0)
    {
        p.chunk_seg_off.resize((size_t)chunks + 1);
        p.chunk_tokens.resize(chunks);
        p.chunk_mask.resize((size_t)chunks * W);
        p.seg_node.resize(segs);
        p.seg_tok_begin.resize(segs);
        p.seg_tok_len.resize(segs);
        p.seg_chunk_pos.resize(segs);
        p.seg_mask.resize((size_t)segs * W);
    }
    // When some whole page of the open chunk sits at a position that is not
    // a multiple of kPageSize (after another segment's partial page), lays
    // the whole pages first: each segment's page-aligned part in order, then
    // the tokens before and after those parts.  The phase-1 kernels copy a
    // whole page at an aligned position with one bulk or tensor copy, the
    // rest row by row.  A chunk's result does not depend on the order of its
    // tokens.  Skipped when the chunk would pass kMaxSegsPerChunk segments.
    // realign's scratch, kept across chunks.
    struct Rec { int32_t node, begin, len; size_t src; };
    std::vector<Rec> whole, rest;
    std::vector<uint64_t> masks;
    void realign()
    {
        const size_t s0 = p.chunk_seg_off.back(), s1 = p.seg_node.size();
        whole.clear();
        rest.clear();
        bool moved = false;
        for (size_t s = s0; s < s1; ++s) {
            const int32_t n = p.seg_node[s], b = p.seg_tok_begin[s], L = p.seg_tok_len[s];
            const int32_t h = std::min(L, (kPageSize - b % kPageSize) % kPageSize);
            const int32_t w = (L - h) / kPageSize * kPageSize;
            if (w == 0) {
                rest.push_back({n, b, L, s});
                continue;
            }
            if (h > 0)
                rest.push_back({n, b, h, s});
            whole.push_back({n, b + h, w, s});
            if (L - h - w > 0)
                rest.push_back({n, b + h + w, L - h - w, s});
            moved = moved || (p.seg_chunk_pos[s] + h) % kPageSize != 0;
        }
        if (!moved || whole.size() + rest.size() > (size_t)kMaxSegsPerChunk)
            return;
        masks.assign(p.seg_mask.begin() + (std::ptrdiff_t)(s0 * W), p.seg_mask.end());
        p.seg_node.resize(s0);
        p.seg_tok_begin.resize(s0);
        p.seg_tok_len.resize(s0);
        p.seg_chunk_pos.resize(s0);
        p.seg_mask.resize(s0 * W);
        int32_t pos = 0;
        for (const std::vector<Rec> *v : {&whole, &rest})
            for (const Rec &r : *v) {
                p.seg_node.push_back(r.node);
                p.seg_tok_begin.push_back(r.begin);
                p.seg_tok_len.push_back(r.len);
                p.seg_chunk_pos.push_back(pos);
                const uint64_t *m = &masks[(r.src - s0) * W];
                p.seg_mask.insert(p.seg_mask.end(), m, m + W);
                pos += r.len;
            }
    }
    void close()
    {
        if (!open)
            return;
        realign();
        p.chunk_seg_off.push_back((int32_t)p.seg_node.size());
        p.chunk_tokens.push_back(cur_chunk_tokens);
        p.chunk_mask.insert(p.chunk_mask.end(), cur_mask.begin(), cur_mask.end());
        std::fill(cur_mask.begin(), cur_mask.end(), 0);
        cur_chunk_tokens = 0;
        cur_chunk_segs = 0;
        open = false;
    }
    // The open chunk's query set and `mask` are one within the other.
    bool nested(const uint64_t *mask) const
    {
        bool sub = true, sup = true;
        for (int32_t i = 0; i < W; ++i) {
            sub = sub && (mask[i] & ~cur_mask[i]) == 0;
            sup = sup && (cur_mask[i] & ~mask[i]) == 0;
        }
        return sub || sup;
    }
    void add_segment(int32_t node, int32_t begin, int32_t len, const uint64_t *mask)
    {
        open = true;
        p.seg_node.push_back(node);
        p.seg_tok_begin.push_back(begin);
        p.seg_tok_len.push_back(len);
        p.seg_chunk_pos.push_back(cur_chunk_tokens);
        p.seg_mask.insert(p.seg_mask.end(), mask, mask + W);
        for (int32_t i = 0; i < W; ++i)
            cur_mask[i] |= mask[i];
        cur_chunk_tokens += len;
        cur_chunk_segs += 1;
    }
};

// Query lists, slot lists and work items of a finished partition.
void finish_partition(Partition &p, int32_t num_queries, int32_t W, int32_t G)
{
    const int32_t C = p.num_chunks();
    p.chunk_q_off.assign(1, 0);
    p.chunk_q.clear();
    for (int32_t c = 0; c < C; ++c) {
        const uint64_t *m = &p.chunk_mask[(size_t)c * W];
        for (int32_t w = 0; w < W; ++w)
            for (uint64_t bits = m[w]; bits; bits &= bits - 1)
                p.chunk_q.push_back(w * 64 + __builtin_ctzll(bits));
        p.chunk_q_off.push_back((int32_t)p.chunk_q.size());
    }
    // Local masks: bit k of segment s = the chunk's k-th query sees s.  A
    // segment's queries are among its chunk's, so each set bit of its
    // global mask maps to a local index (loc, filled per chunk).
    p.seg_lmask_off.assign(1, 0);
    p.seg_lmask.clear();
    {
        std::vector<int32_t> loc(num_queries > 0 ? num_queries : 1);
        for (int32_t c = 0; c < C; ++c) {
            const int32_t q0 = p.chunk_q_off[c], nq = p.chunk_q_off[c + 1] - q0;
            const int32_t words = (nq + 31) / 32;
            for (int32_t k = 0; k < nq; ++k)
                loc[p.chunk_q[q0 + k]] = k;
            for (int32_t s = p.chunk_seg_off[c]; s < p.chunk_seg_off[c + 1]; ++s) {
                const uint64_t *m = &p.seg_mask[(size_t)s * W];
                const size_t at = p.seg_lmask.size();
                p.seg_lmask.resize(at + words, 0u);
                for (int32_t w = 0; w < W; ++w)
                    for (uint64_t bits = m[w]; bits; bits &= bits - 1) {
                        const int32_t k = loc[w * 64 + __builtin_ctzll(bits)];
                        p.seg_lmask[at + k / 32] |= 1u << (k % 32);
                    }
                p.seg_lmask_off.push_back((int32_t)p.seg_lmask.size());
            }
        }
    }
    // Per-query slot CSR, slots in chunk order.
    std::vector<int32_t> cnt(num_queries + 1, 0);
    for (int32_t s = 0; s < p.num_slots(); ++s)
        cnt[p.chunk_q[s] + 1] += 1;
    p.q_slot_off.assign(num_queries + 1, 0);
    for (int32_t q = 0; q < num_queries; ++q)
        p.q_slot_off[q + 1] = p.q_slot_off[q] + cnt[q + 1];
    p.q_slot.assign(p.num_slots(), 0);
    std::vector<int32_t> fill(p.q_slot_off.begin(), p.q_slot_off.end() - 1);
    for (int32_t s = 0; s < p.num_slots(); ++s)
        p.q_slot[fill[p.chunk_q[s]]++] = s;
    // A query whose path lies in one chunk of fewer than kMmaMinRows rows
    // (a CUDA-core chunk) has its rows written to out / lse by phase 1; the
    // merge launch takes every other query.
    std::vector<uint8_t> direct_q(num_queries, 0);
    for (int32_t c = 0; c < C; ++c) {
        const int32_t k = p.chunk_q_off[c + 1] - p.chunk_q_off[c];
        if ((int64_t)k * G >= kMmaMinRows)
            continue;
        for (int32_t s = p.chunk_q_off[c]; s < p.chunk_q_off[c + 1]; ++s) {
            const int32_t q = p.chunk_q[s];
            direct_q[q] = p.q_slot_off[q + 1] - p.q_slot_off[q] == 1 ? 1 : 0;
        }
    }
    p.merge_q.clear();
    for (int32_t q = 0; q < num_queries; ++q)
        if (!direct_q[q])
            p.merge_q.push_back(q);

    // Work items.  rows = queries * G.  Chunks under kMmaMinRows rows run on
    // the CUDA-core kernel in row blocks of at most kFmaItemRows rows (whole
    // queries): above 8 rows the kernel's per-token work outgrows what one
    // SM streams, and two blocks run on two SMs at once, the second reading
    // the chunk from L2.  The others run on the tensor-core kernel in row
    // blocks of at most kMmaMaxRows rows, and are also cut into items of at
    // most kFmaMaxRows rows for head sizes without a tensor path.
    struct Item { int32_t c, b, e; int64_t cost; int32_t bucket = 0; };
    std::vector<Item> fma, mma, fb;
    const int32_t qmax_mma = std::max(1, kMmaMaxRows / G);
    const int32_t qmax_fb = std::max(1, kFmaMaxRows / G);
    for (int32_t c = 0; c < C; ++c) {
        const int32_t k = p.chunk_q_off[c + 1] - p.chunk_q_off[c];
        const int64_t tok = p.chunk_tokens[c];
        if ((int64_t)k * G < kMmaMinRows) {
            const int32_t qmax = std::max(1, kFmaItemRows / G);
            const int32_t nb = (k + qmax - 1) / qmax, per = (k + nb - 1) / nb;
            for (int32_t b = 0; b < k; b += per)
                fma.push_back({c, b, std::min(k, b + per), tok, row_bucket((std::min(k, b + per) - b) * G)});
            continue;
        }
        const int32_t nb = (k + qmax_mma - 1) / qmax_mma;
        const int32_t per = (k + nb - 1) / nb;
        // Within a width (row bucket) a unit's time follows its tokens, not
        // its rows: the order of the launch's queue and of its static blocks.
        for (int32_t b = 0; b < k; b += per)
            mma.push_back({c, b, std::min(k, b + per), tok, mma_bucket((std::min(k, b + per) - b) * G)});
        const int32_t nf = (k + qmax_fb - 1) / qmax_fb;
        const int32_t perf = (k + nf - 1) / nf;
        for (int32_t b = 0; b < k; b += perf)
            fb.push_back({c, b, std::min(k, b + perf), tok, row_bucket((std::min(k, b + perf) - b) * G)});
    }
    // Tensor-core items of both widths run as one launch at 32 columns a
    // warpgroup when that costs little more (kCollapseMma); their row masks are
    // then laid out for that width.
    {
        double tok[2] = {0.0, 0.0};
        for (const Item &it : mma)
            tok[it.bucket] += (double)p.chunk_tokens[it.c];
        const double split = tok[0] * mma_ns_per_token(0) + tok[1] * mma_ns_per_token(1);
        const double one = (tok[0] + tok[1]) * mma_ns_per_token(1);
        if (tok[0] > 0.0 && tok[1] > 0.0 && one <= kCollapseMma * split)
            for (Item &it : mma)
                it.bucket = 1;
    }
    // Largest first, so the hardware block scheduler starts the long items
    // early (a longest-processing-time order).
    auto by_cost = [](const Item &x, const Item &y) {
        if (x.bucket != y.bucket)
            return x.bucket < y.bucket;
        return x.cost != y.cost ? x.cost > y.cost : (x.c != y.c ? x.c < y.c : x.b < y.b);
    };
    auto bucket_offsets = [](const std::vector<Item> &v, auto &off) {
        off.fill(0);
        for (const Item &it : v)
            off[it.bucket + 1] += 1;
        for (size_t b = 0; b + 1 < off.size(); ++b)
            off[b + 1] += off[b];
    };
    std::stable_sort(fma.begin(), fma.end(), by_cost);
    std::stable_sort(mma.begin(), mma.end(), by_cost);
    std::stable_sort(fb.begin(), fb.end(), by_cost);
    auto emit = [](const std::vector<Item> &v, std::vector<int32_t> &out) {
        out.clear();
        for (const Item &it : v) {
            out.push_back(it.c);
            out.push_back(it.b);
            out.push_back(it.e);
        }
    };
    emit(fma, p.fma_items);
    emit(mma, p.mma_items);
    emit(fb, p.fallback_items);

    // Row masks per (item, segment): row r of an item is its query
    // b + r / G, present in segment s when s's query mask has that bit.
    // qbits: local bits b .. b + n - 1 of segment s (n <= 64);
    // row_bits: those queries' rows, G bits each (at most 64 rows).
    auto qbits = [&](int32_t s, int32_t b, int32_t n) -> uint64_t {
        const int32_t w0 = p.seg_lmask_off[s], nw = p.seg_lmask_off[s + 1] - w0;
        const int32_t i = b / 32, sh = b % 32;
        auto word = [&](int32_t j) -> uint64_t { return j < nw ? p.seg_lmask[w0 + j] : 0u; };
        uint64_t x = (word(i) | (word(i + 1) << 32)) >> sh;
        if (sh > 0)
            x |= word(i + 2) << (64 - sh);
        return n >= 64 ? x : x & ((1ull << n) - 1);
    };
    auto row_bits = [&](uint64_t qb) -> uint64_t {
        if (G == 1)
            return qb;
        uint64_t r = 0;
        const uint64_t g = G >= 64 ? ~0ull : (1ull << G) - 1;
        for (; qb; qb &= qb - 1)
            r |= g << (__builtin_ctzll(qb) * G);
        return r;
    };
    auto row_masks = [&](const std::vector<Item> &v, std::vector<uint32_t> &mask, std::vector<int32_t> &off) {
        mask.clear();
        off.assign(1, 0);
        for (const Item &it : v) {
            for (int32_t s = p.chunk_seg_off[it.c]; s < p.chunk_seg_off[it.c + 1]; ++s)
                mask.push_back((uint32_t)row_bits(qbits(s, it.b, it.e - it.b)));
            off.push_back((int32_t)mask.size());
        }
    };
    row_masks(fma, p.fma_rmask, p.fma_rmask_off);
    row_masks(fb, p.fallback_rmask, p.fallback_rmask_off);
    p.mma_rmask.clear();
    p.mma_rmask_off.assign(1, 0);
    for (const Item &it : mma) {
        // Rows 0 .. nph-1 are warpgroup 0's columns (bits 0-63), the rest
        // warpgroup 1's (bits 64-127).
        const int32_t nph = 16 * (it.bucket + 1);
        for (int32_t s = p.chunk_seg_off[it.c]; s < p.chunk_seg_off[it.c + 1]; ++s) {
            const uint64_t r = row_bits(qbits(s, it.b, it.e - it.b));
            const uint64_t lo = nph >= 64 ? r : r & ((1ull << nph) - 1), hi = nph >= 64 ? 0 : r >> nph;
            const uint32_t w[4] = {(uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32)};
            p.mma_rmask.insert(p.mma_rmask.end(), w, w + 4);
        }
        p.mma_rmask_off.push_back((int32_t)(p.mma_rmask.size() / 4));
    }
    // Rows of the direct queries (none in the fallback items: their chunks
    // have kMmaMinRows rows or more).
    auto direct_rows = [&](const std::vector<Item> &v, std::vector<uint32_t> &out) {
        out.assign(v.size(), 0u);
        for (size_t i = 0; i < v.size(); ++i) {
            const Item &it = v[i];
            const int32_t rows = (it.e - it.b) * G;
            for (int32_t r = 0; r < rows; ++r)
                if (direct_q[p.chunk_q[p.chunk_q_off[it.c] + it.b + r / G]])
                    out[i] |= 1u << r;
        }
    };
    direct_rows(fma, p.fma_direct);
    direct_rows(fb, p.fallback_direct);
    bucket_offsets(fma, p.fma_bucket_off);
    bucket_offsets(fb, p.fallback_bucket_off);
    bucket_offsets(mma, p.mma_bucket_off);
    // KV tokens each bucket's launch reads (per KV head): the dispatcher
    // shares the SMs among concurrent launches in proportion.
    auto bucket_tokens = [&](const std::vector<Item> &v, auto &tok) {
        tok.fill(0);
        for (const Item &it : v)
            tok[it.bucket] += p.chunk_tokens[it.c];
    };
    bucket_tokens(fma, p.fma_bucket_tok);
    bucket_tokens(fb, p.fallback_bucket_tok);
    bucket_tokens(mma, p.mma_bucket_tok);
}

}  // namespace

namespace {

// The per-query parts of a plan that depend on the node lengths: the
// queries sitting inside each node (CSR, for the cuts of positioned
// queries) and the token counts.
void query_parts(deft_plan_t *plan, int64_t &naive_tokens, int64_t &path_nodes)
{
    const int32_t N = plan->num_nodes, Q = plan->num_queries;
    const int32_t *parent = plan->in_parent.data(), *node_len = plan->in_len.data();
    const int32_t *query_node = plan->in_qnode.data();
    const int32_t *query_pos = plan->in_qpos.empty() ? nullptr : plan->in_qpos.data();
    auto taken = [&](int32_t q, int32_t n) {
        return (query_pos && n == query_node[q] && query_pos[q] >= 0) ? query_pos[q] + 1 : node_len[n];
    };
    naive_tokens = path_nodes = 0;
    for (int32_t q = 0; q < Q; ++q)
        for (int32_t cur = query_node[q]; cur != -1; cur = parent[cur]) {
            naive_tokens += taken(q, cur);
            path_nodes += 1;
        }
    // Per node, the queries that sit at a position before its last token
    // (their part of the node ends there).
    plan->own_off.assign((size_t)N + 1, 0);
    plan->own_q.clear();
    if (query_pos) {
        for (int32_t q = 0; q < Q; ++q)
            if (query_pos[q] >= 0 && query_pos[q] + 1 < node_len[query_node[q]])
                plan->own_off[query_node[q] + 1] += 1;
        for (int32_t n = 0; n < N; ++n)
            plan->own_off[n + 1] += plan->own_off[n];
        plan->own_q.resize(plan->own_off[N]);
        std::vector<int32_t> fill(plan->own_off.begin(), plan->own_off.end() - 1);
        for (int32_t q = 0; q < Q; ++q)
            if (query_pos[q] >= 0 && query_pos[q] + 1 < node_len[query_node[q]])
                plan->own_q[fill[query_node[q]]++] = q;
    }
}

// The tree partition's segments and chunks, emitted from DFS position
// `start` on (0: from scratch), with the partition, the unique-token count
// and the tensor-packing list as the checkpoint at `start` recorded them
// (which must be clean: no chunk open).  Records a checkpoint before every
// position.
int64_t emit_tree(deft_plan_t *plan, size_t start)
{
    const int32_t N = plan->num_nodes, W = plan->mask_words;
    const int32_t chunk_target = plan->chunk_target, gqa_group = plan->gqa_group;
    const bool tensor_pack = plan->in_tensor_pack;
    const int32_t *node_len = plan->in_len.data();
    const int32_t *query_pos = plan->in_qpos.empty() ? nullptr : plan->in_qpos.data();
    const std::vector<int32_t> &own_off = plan->own_off, &own_q = plan->own_q;
    Partition &part = plan->tree;
    std::vector<ThinSeg> &thin = plan->thin;
    std::vector<uint64_t> &thin_mask = plan->thin_mask;
    int64_t unique_tokens = 0;
    std::vector<EmitCkpt> &ck = plan->ckpt;
    int64_t tokens = 0;
    for (int32_t n = 0; n < N; ++n)
        tokens += node_len[n];
    if (start == 0) {
        part.reset();
        thin.clear();
        thin_mask.clear();
    } else {
        unique_tokens = ck[start].unique;
        thin.resize(ck[start].thin);
        thin_mask.resize((size_t)ck[start].thin * W);
    }
    Builder b = start == 0 ? Builder(part, W, tokens / chunk_target + N, tokens / chunk_target + 2 * (int64_t)N)
                           : Builder(part, W, ck[start].chunks, ck[start].segs, true);
    ck.resize((size_t)N + 1);
    // Tokens [b0, b0 + L) of node n, attended by the queries in m (k of them).
    auto emit = [&](int32_t n, int32_t b0, int32_t L, const uint64_t *m, int k) {
        unique_tokens += L;
        if (tensor_pack && (int64_t)k * gqa_group < kMmaMinRows && (int64_t)k * gqa_group >= kMmaMinRows / 4 &&
            4 * (int64_t)L > chunk_target) {
            thin.push_back(ThinSeg{n, b0, L, (int32_t)(thin_mask.size() / W)});
            thin_mask.insert(thin_mask.end(), m, m + W);
            return;
        }
        if (2 * (int64_t)L <= chunk_target) {
            // A segment that would add queries to the open chunk (its
            // rows grow for every token of it) joins only when tiny.
            const bool tiny = 4 * (int64_t)L <= chunk_target;
            if (b.open && (b.cur_chunk_tokens + L > chunk_target ||
                           b.cur_chunk_segs >= kMaxSegsPerChunk || (!tiny && !b.nested(m))))
                b.close();
            b.add_segment(n, b0, L, m);
            return;
        }
        b.close();
        int64_t T = std::max<int64_t>(chunk_target, (int64_t)kSharedTokensPerRow * k * gqa_group);
        T = (T + kPageSize - 1) / kPageSize * kPageSize;
        const int64_t pieces = (L + T - 1) / T;
        int64_t piece = (L + pieces - 1) / pieces;
        piece = (piece + kPageSize - 1) / kPageSize * kPageSize;
        for (int64_t s = 0; s < L; s += piece) {
            b.add_segment(n, (int32_t)(b0 + s), (int32_t)std::min<int64_t>(piece, L - s), m);
            b.close();
        }
    };
    auto checkpoint = [&](size_t pos) {
        ck[pos] = EmitCkpt{(int32_t)part.chunk_tokens.size(), (int32_t)part.seg_node.size(), (int32_t)thin.size(),
                           unique_tokens, !b.open};
    };
    std::vector<int32_t> cuts;
    std::vector<uint64_t> pm(W, 0);
    for (size_t pos = start; pos < (size_t)N; ++pos) {
        checkpoint(pos);
        const int32_t n = plan->order[pos];
        const int32_t L = node_len[n];
        const uint64_t *m = &plan->cover[(size_t)n * W];
        const int k = popcount_words(m, W);
        if (L == 0 || k == 0)
            continue;
        if (own_off[n] == own_off[n + 1]) {
            emit(n, 0, L, m, k);
            continue;
        }
        // Queries sitting inside the node cut it where their part ends:
        // every piece has one query set (the node's, less the queries
        // whose position lies before the piece).
        cuts.clear();
        for (int32_t i = own_off[n]; i < own_off[n + 1]; ++i)
            cuts.push_back(query_pos[own_q[i]] + 1);
        std::sort(cuts.begin(), cuts.end());
        cuts.erase(std::unique(cuts.begin(), cuts.end()), cuts.end());
        cuts.push_back(L);
        int32_t b0 = 0;
        for (int32_t e : cuts) {
            std::copy(m, m + W, pm.begin());
            for (int32_t i = own_off[n]; i < own_off[n + 1]; ++i) {
                const int32_t q = own_q[i];
                if (query_pos[q] < b0)
                    pm[q / 64] &= ~(1ull << (q % 64));
            }
            const int kp = popcount_words(pm.data(), W);
            if (kp > 0)
                emit(n, b0, e - b0, pm.data(), kp);
            b0 = e;
        }
    }
    b.close();
    checkpoint((size_t)N);
    // Tensor packing of the thin segments, longest first, so that the
    // segments of a chunk run out together and the last ones, which may
    // not reach kMmaMinRows rows together, are the shortest.  (The list
    // keeps emission order for later resumes; the packing walks a sorted
    // index.)
    std::vector<size_t> byl(thin.size());
    std::iota(byl.begin(), byl.end(), (size_t)0);
    std::stable_sort(byl.begin(), byl.end(), [&](size_t x, size_t y) { return thin[x].L > thin[y].L; });
    std::vector<int32_t> left(thin.size());
    for (size_t i = 0; i < thin.size(); ++i)
        left[i] = thin[i].L;
    std::vector<uint64_t> um(W, 0);
    std::vector<size_t> group;
    size_t head = 0;
    while (true) {
        while (head < byl.size() && left[byl[head]] == 0)
            ++head;
        if (head == byl.size())
            break;
        // The next segments with tokens left, until their queries make
        // kMmaMinRows rows (never more than kMmaMaxRows).
        group.clear();
        std::fill(um.begin(), um.end(), 0);
        for (size_t h = head; h < byl.size() && (int)group.size() < kMaxSegsPerChunk; ++h) {
            const size_t i = byl[h];
            if (left[i] == 0)
                continue;
            const uint64_t *m = &thin_mask[(size_t)thin[i].mask * W];
            int k = 0;
            for (int32_t w = 0; w < W; ++w)
                k += __builtin_popcountll(um[w] | m[w]);
            if (!group.empty() && (int64_t)k * gqa_group > kMmaMaxRows)
                break;
            group.push_back(i);
            for (int32_t w = 0; w < W; ++w)
                um[w] |= m[w];
            if ((int64_t)k * gqa_group >= kMmaMinRows)
                break;
        }
        int64_t piece = std::max<int64_t>(kTensorPiece, chunk_target / (int64_t)group.size());
        piece = piece / kPageSize * kPageSize;
        for (size_t i : group) {
            const ThinSeg &t = thin[i];
            const int32_t take = (int32_t)std::min<int64_t>(piece, left[i]);
            b.add_segment(t.n, t.b0 + (t.L - left[i]), take, &thin_mask[(size_t)t.mask * W]);
            left[i] -= take;
        }
        b.close();
    }
    return unique_tokens;
}

// Naive partition, query lists of both partitions, work items, statistics.
void finish_plan(deft_plan_t *plan, int64_t unique_tokens, int64_t naive_tokens, int64_t path_nodes)
{
    const int32_t N = plan->num_nodes, Q = plan->num_queries, W = plan->mask_words;
    const int32_t chunk_target = plan->chunk_target, gqa_group = plan->gqa_group;
    const int32_t *parent = plan->in_parent.data(), *node_len = plan->in_len.data();
    const int32_t *query_node = plan->in_qnode.data();
    const int32_t *query_pos = plan->in_qpos.empty() ? nullptr : plan->in_qpos.data();
    auto taken = [&](int32_t q, int32_t n) {
        return (query_pos && n == query_node[q] && query_pos[q] >= 0) ? query_pos[q] + 1 : node_len[n];
    };
    finish_partition(plan->tree, Q, W, gqa_group);

    // Naive partition: each query's path (root first) cut every chunk_target
    // tokens; every chunk serves that one query.  Left empty (no chunk) when
    // the caller will not run it.
    plan->naive.reset();
    if (!plan->has_naive) {
        Builder b(plan->naive, W, 0, 0);
    } else {
        Builder b(plan->naive, W, naive_tokens / chunk_target + Q, naive_tokens / chunk_target + Q + path_nodes);
        std::vector<int32_t> path;
        std::vector<uint64_t> m(W, 0);
        for (int32_t q = 0; q < Q; ++q) {
            path.clear();
            for (int32_t cur = query_node[q]; cur != -1; cur = parent[cur])
                path.push_back(cur);
            std::reverse(path.begin(), path.end());
            std::fill(m.begin(), m.end(), 0);
            m[q / 64] = 1ull << (q % 64);
            for (int32_t n : path) {
                const int32_t len = taken(q, n);
                int32_t t = 0;
                while (t < len) {
                    if (b.open && (b.cur_chunk_tokens == chunk_target ||
                                   b.cur_chunk_segs >= kMaxSegsPerChunk))
                        b.close();
                    const int32_t take = std::min(len - t, chunk_target - b.cur_chunk_tokens);
                    b.add_segment(n, t, take, m.data());
                    t += take;
                }
            }
            b.close();
        }
    }
    finish_partition(plan->naive, Q, W, gqa_group);

    // Statistics.
    deft_plan_stats &st = plan->stats;
    std::memset(&st, 0, sizeof st);
    st.num_nodes = N;
    st.num_queries = Q;
    st.gqa_group = gqa_group;
    st.chunk_target = chunk_target;
    st.mask_words = W;
    st.num_chunks = plan->tree.num_chunks();
    st.num_segments = plan->tree.num_segments();
    st.num_slots = plan->tree.num_slots();
    st.num_fma_items = (int32_t)plan->tree.fma_items.size() / 3;
    st.num_mma_items = (int32_t)plan->tree.mma_items.size() / 3;
    st.num_fallback_items = (int32_t)plan->tree.fallback_items.size() / 3;
    for (int32_t c = 0; c < st.num_chunks; ++c) {
        st.max_chunk_tokens = std::max(st.max_chunk_tokens, plan->tree.chunk_tokens[c]);
        st.planned_tokens += plan->tree.chunk_tokens[c];
        st.pair_tokens += (int64_t)plan->tree.chunk_tokens[c] *
                          (plan->tree.chunk_q_off[c + 1] - plan->tree.chunk_q_off[c]);
    }
    for (int32_t q = 0; q < Q; ++q)
        st.max_slots_per_query = std::max(st.max_slots_per_query,
                                          plan->tree.q_slot_off[q + 1] - plan->tree.q_slot_off[q]);
    st.naive_num_chunks = plan->naive.num_chunks();
    st.naive_num_slots = plan->naive.num_slots();
    st.naive_num_segments = plan->naive.num_segments();
    st.num_merge_queries = (int32_t)plan->tree.merge_q.size();
    st.unique_tokens = unique_tokens;
    st.naive_tokens = naive_tokens;
}

}  // namespace

int build_plan(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
               const int32_t *query_node, const int32_t *query_pos, int32_t num_queries,
               int32_t chunk_target, int32_t gqa_group, bool with_naive, bool tensor_pack,
               deft_plan_t *plan)
{
    if (!parent || !node_len || !plan || num_nodes < 1 || num_queries < 0 ||
        (num_queries > 0 && !query_node))
        return DEFT_EINVAL;
    if (chunk_target < 1 || chunk_target > kMaxChunkTarget || gqa_group < 1 || gqa_group > 128)
        return DEFT_EINVAL;
    const int32_t N = num_nodes, Q = num_queries;
    for (int32_t n = 0; n < N; ++n) {
        if (parent[n] < -1 || parent[n] >= N)
            return DEFT_ERANGE;
        if (node_len[n] < 0)
            return DEFT_EINVAL;
    }
    for (int32_t q = 0; q < Q; ++q)
        if (query_node[q] < 0 || query_node[q] >= N)
            return DEFT_ERANGE;
    // A query at position p of its node attends tokens 0..p of it (-1: all).
    for (int32_t q = 0; q < Q && query_pos; ++q)
        if (query_pos[q] < -1 || query_pos[q] >= node_len[query_node[q]])
            return DEFT_ERANGE;

    // Forest check by colouring: 0 unseen, 1 on the current upward walk, 2 done.
    {
        std::vector<uint8_t> colour(N, 0);
        std::vector<int32_t> walk;
        for (int32_t n = 0; n < N; ++n) {
            int32_t cur = n;
            walk.clear();
            while (cur != -1 && colour[cur] == 0) {
                colour[cur] = 1;
                walk.push_back(cur);
                cur = parent[cur];
            }
            if (cur != -1 && colour[cur] == 1)
                return DEFT_ECYCLE;
            for (int32_t x : walk)
                colour[x] = 2;
        }
    }

    const int32_t W = (Q + 63) / 64;
    plan->num_nodes = N;
    plan->num_queries = Q;
    plan->gqa_group = gqa_group;
    plan->chunk_target = chunk_target;
    plan->mask_words = W;
    plan->has_naive = with_naive;
    plan->in_tensor_pack = tensor_pack;
    plan->in_parent.assign(parent, parent + N);
    plan->in_len.assign(node_len, node_len + N);
    plan->in_qnode.assign(query_node, query_node + Q);
    if (query_pos)
        plan->in_qpos.assign(query_pos, query_pos + Q);
    else
        plan->in_qpos.clear();

    // Coverage bitsets: walk every query's path.
    plan->cover.assign((size_t)N * W, 0);
    for (int32_t q = 0; q < Q; ++q)
        for (int32_t cur = query_node[q]; cur != -1; cur = parent[cur])
            plan->cover[(size_t)cur * W + q / 64] |= 1ull << (q % 64);
    int64_t naive_tokens = 0, path_nodes = 0;
    query_parts(plan, naive_tokens, path_nodes);

    // Children lists (ascending ids) and DFS preorder.
    std::vector<int32_t> child_off(N + 1, 0), child(N > 0 ? N : 1);
    for (int32_t n = 0; n < N; ++n)
        if (parent[n] >= 0)
            child_off[parent[n] + 1] += 1;
    for (int32_t n = 0; n < N; ++n)
        child_off[n + 1] += child_off[n];
    {
        std::vector<int32_t> fill(child_off.begin(), child_off.end() - 1);
        for (int32_t n = 0; n < N; ++n)
            if (parent[n] >= 0)
                child[fill[parent[n]]++] = n;
    }
    plan->order.clear();
    {
        std::vector<int32_t> stack;
        for (int32_t r = N - 1; r >= 0; --r)
            if (parent[r] == -1)
                stack.push_back(r);
        while (!stack.empty()) {
            int32_t n = stack.back();
            stack.pop_back();
            plan->order.push_back(n);
            for (int32_t i = child_off[n + 1] - 1; i >= child_off[n]; --i)
                stack.push_back(child[i]);
        }
    }
    plan->order_pos.assign(N, 0);
    for (int32_t i = 0; i < N; ++i)
        plan->order_pos[plan->order[i]] = i;

    // DeFT partition, then the rest.
    const int64_t unique_tokens = emit_tree(plan, 0);
    finish_plan(plan, unique_tokens, naive_tokens, path_nodes);
    return DEFT_OK;
}

int update_plan(deft_plan_t *plan, const int32_t *node_len, int32_t num_nodes)
{
    if (!plan || !node_len || num_nodes != plan->num_nodes)
        return DEFT_EINVAL;
    const int32_t N = num_nodes, Q = plan->num_queries;
    for (int32_t n = 0; n < N; ++n)
        if (node_len[n] < 0)
            return DEFT_EINVAL;
    const int32_t *query_node = plan->in_qnode.data();
    for (int32_t q = 0; q < Q && !plan->in_qpos.empty(); ++q)
        if (plan->in_qpos[q] >= node_len[query_node[q]])
            return DEFT_ERANGE;
    // The first changed node in DFS order.
    size_t first = (size_t)N;
    for (int32_t n = 0; n < N; ++n)
        if (node_len[n] != plan->in_len[n])
            first = std::min(first, (size_t)plan->order_pos[n]);
    plan->in_len.assign(node_len, node_len + N);
    if (first == (size_t)N)
        return DEFT_OK;   // nothing changed
    // Resume at the last position at or before it where no chunk was open:
    // everything emitted before it is what a fresh plan emits.
    size_t start = first;
    while (start > 0 && !plan->ckpt[start].clean)
        --start;
    int64_t naive_tokens = 0, path_nodes = 0;
    query_parts(plan, naive_tokens, path_nodes);
    const int64_t unique_tokens = emit_tree(plan, start);
    finish_plan(plan, unique_tokens, naive_tokens, path_nodes);
    return DEFT_OK;
}

}  // namespace deft
