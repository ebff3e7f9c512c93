/*
 * deft_oracle.c -- plain fp64 CPU oracle for DeFT tree-attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA library: it is written directly from
 * the definition of the operation so that a reader can check it by eye.
 *
 * What it computes (DeFT paper, arXiv 2404.00242, abstract; aifetchly "DeFT
 * Guide", section "Deep Dive: Mathematical Formulation", tree-constrained
 * attention formula and causal tree mask):
 *
 *   A query q sits at tree node n = query_node[q].  It attends to every token
 *   of every node on the root-to-n path, n itself included (the Guide's
 *   ancestor map starts each node's list with the node itself, section
 *   "End-to-End Implementation", TreeTopologyManager).  Tokens outside that
 *   path are masked to -inf.  A query may instead sit at token position
 *   p = query_pos[q] of its node (tree verification with multi-token
 *   nodes): the node's tokens are a chain, so it attends tokens 0..p of its
 *   own node and every token of the nodes above (the Guide's causal tree
 *   mask, section "Deep Dive", taken at token granularity); query_pos NULL
 *   or p < 0 means the node's last token.  For query head h (KV head h / G):
 *       s_j   = (q . k_j) * scale
 *       m     = max_j s_j,  l = sum_j exp(s_j - m)
 *       out   = sum_j exp(s_j - m) v_j / l
 *       lse   = m + ln l            (natural log; -inf and out = 0 for an
 *                                    empty path)
 *   All arithmetic is fp64 on the exact values of the bf16 inputs.
 *
 * It also produces the integer facts the planner must reproduce bit-exactly:
 * root-to-node paths, per-node coverage bitsets (bit q of node n set iff n is
 * on q's path: the query set that KV-Guided Grouping shares a node's KV
 * with), the unique-token count (tokens on at least one path) and the naive
 * per-query token count.
 *
 * Pins (tests/, run without a GPU): dense brute-force attention with an
 * explicit tree mask built by a different method, chain tree == causal decode
 * through a library attention routine, closed forms (single token, q = 0,
 * equal keys, empty path), node relabelling, the Guide's worked IO example.
 *
 * KV layout read here: bf16 [num_pages][num_kv_heads][page_size][head_dim];
 * token t of node n is in page page_id[node_page_off[n] + t / P], slot t % P.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Walk parent pointers from node n up to its root.  Writes the path root-first
 * into buf and returns its length, or -1 if an index is out of range or the
 * walk is longer than the node count (a cycle). */
static int32_t path_of(const int32_t *parent, int32_t num_nodes, int32_t n, int32_t *buf)
{
    int32_t len = 0;
    int32_t cur = n;
    while (cur != -1) {
        if (cur < 0 || cur >= num_nodes || len >= num_nodes)
            return -1;
        buf[len++] = cur;
        cur = parent[cur];
    }
    for (int32_t i = 0; i < len / 2; ++i) {
        int32_t t = buf[i];
        buf[i] = buf[len - 1 - i];
        buf[len - 1 - i] = t;
    }
    return len;
}

/* Root-to-node paths of all queries as CSR: path_off[q]..path_off[q+1] index
 * path_nodes.  Returns the total number of path entries, -1 on a bad tree, or
 * -2 if `cap` entries are not enough (path_off is still filled then). */
int64_t oracle_paths(const int32_t *parent, int32_t num_nodes, const int32_t *query_node,
                     int32_t num_queries, int64_t *path_off, int32_t *path_nodes, int64_t cap)
{
    int32_t *buf = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_nodes > 0 ? num_nodes : 1));
    int64_t total = 0;
    int overflow = 0;
    path_off[0] = 0;
    for (int32_t q = 0; q < num_queries; ++q) {
        int32_t len = path_of(parent, num_nodes, query_node[q], buf);
        if (len < 0) {
            free(buf);
            return -1;
        }
        for (int32_t i = 0; i < len; ++i) {
            if (total + i < cap)
                path_nodes[total + i] = buf[i];
            else
                overflow = 1;
        }
        total += len;
        path_off[q + 1] = total;
    }
    free(buf);
    return overflow ? -2 : total;
}

/* cover[n * words + q / 64] bit (q % 64) is set iff node n lies on the path
 * of query q.  words = ceil(num_queries / 64).  Returns 0 or -1. */
int oracle_cover(const int32_t *parent, int32_t num_nodes, const int32_t *query_node,
                 int32_t num_queries, uint64_t *cover)
{
    int32_t words = (num_queries + 63) / 64;
    int32_t *buf = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_nodes > 0 ? num_nodes : 1));
    memset(cover, 0, sizeof(uint64_t) * (size_t)num_nodes * (size_t)words);
    for (int32_t q = 0; q < num_queries; ++q) {
        int32_t len = path_of(parent, num_nodes, query_node[q], buf);
        if (len < 0) {
            free(buf);
            return -1;
        }
        for (int32_t i = 0; i < len; ++i)
            cover[(size_t)buf[i] * words + q / 64] |= (uint64_t)1 << (q % 64);
    }
    free(buf);
    return 0;
}

/* Tokens of `node` (on the path of a query at node qnode) that the query
 * attends: all of them, or 0..pos of its own node when it sits at pos. */
static int32_t tokens_taken(const int32_t *node_len, int32_t node, int32_t qnode, int32_t pos)
{
    if (node == qnode && pos >= 0)
        return pos + 1;
    return node_len[node];
}

/* Tokens on at least one query path (each counted once) and the sum over
 * queries of their path token counts.  query_pos may be NULL.  Returns 0 or
 * -1 (bad tree, or a position outside its node). */
int oracle_token_counts(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
                        const int32_t *query_node, const int32_t *query_pos, int32_t num_queries,
                        int64_t *unique_tokens, int64_t *naive_tokens)
{
    int32_t *buf = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_nodes > 0 ? num_nodes : 1));
    /* taken[n]: how many leading tokens of node n some query attends */
    int32_t *taken = (int32_t *)calloc((size_t)(num_nodes > 0 ? num_nodes : 1), sizeof(int32_t));
    int64_t uniq = 0, naive = 0;
    for (int32_t q = 0; q < num_queries; ++q) {
        int32_t len = path_of(parent, num_nodes, query_node[q], buf);
        int32_t pos = query_pos ? query_pos[q] : -1;
        if (len < 0 || pos >= node_len[query_node[q]]) {
            free(buf);
            free(taken);
            return -1;
        }
        for (int32_t i = 0; i < len; ++i) {
            int32_t take = tokens_taken(node_len, buf[i], query_node[q], pos);
            naive += take;
            if (take > taken[buf[i]])
                taken[buf[i]] = take;
        }
    }
    for (int32_t n = 0; n < num_nodes; ++n)
        uniq += taken[n];
    free(buf);
    free(taken);
    *unique_tokens = uniq;
    *naive_tokens = naive;
    return 0;
}

/* Address of element 0 of token t of node n, KV head kvh, in a paged buffer. */
static size_t token_offset(const int32_t *node_page_off, const int32_t *page_id, int32_t page_size,
                           int32_t num_kv_heads, int32_t head_dim, int32_t n, int32_t t, int32_t kvh)
{
    int32_t page = page_id[node_page_off[n] + t / page_size];
    int32_t slot = t % page_size;
    return (((size_t)page * num_kv_heads + kvh) * page_size + slot) * head_dim;
}

/* Attention of one (query, head) over an explicit list of tokens (node, t)
 * given as two arrays.  Writes out[head_dim] and returns lse. */
static double attend(const uint16_t *qv, const uint16_t *k_pages, const uint16_t *v_pages,
                     const int32_t *node_page_off, const int32_t *page_id, int32_t page_size,
                     int32_t num_kv_heads, int32_t head_dim, int32_t kvh, double scale,
                     const int32_t *tok_node, const int32_t *tok_idx, int64_t ntok,
                     double *scores, double *out)
{
    for (int32_t i = 0; i < head_dim; ++i)
        out[i] = 0.0;
    if (ntok == 0)
        return -INFINITY;
    double m = -INFINITY;
    for (int64_t j = 0; j < ntok; ++j) {
        size_t off = token_offset(node_page_off, page_id, page_size, num_kv_heads, head_dim,
                                  tok_node[j], tok_idx[j], kvh);
        double dot = 0.0;
        for (int32_t i = 0; i < head_dim; ++i)
            dot += bf16_value(qv[i]) * bf16_value(k_pages[off + i]);
        scores[j] = dot * scale;
        if (scores[j] > m)
            m = scores[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < ntok; ++j) {
        double p = exp(scores[j] - m);
        l += p;
        size_t off = token_offset(node_page_off, page_id, page_size, num_kv_heads, head_dim,
                                  tok_node[j], tok_idx[j], kvh);
        for (int32_t i = 0; i < head_dim; ++i)
            out[i] += p * bf16_value(v_pages[off + i]);
    }
    for (int32_t i = 0; i < head_dim; ++i)
        out[i] /= l;
    return m + log(l);
}

/* Expand query q's path into its token list (root first, tokens in order);
 * qpos >= 0: the query sits at that token of its node. */
static int64_t path_tokens(const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
                           int32_t qnode, int32_t qpos, int32_t *pathbuf, int32_t *tok_node,
                           int32_t *tok_idx)
{
    int32_t len = path_of(parent, num_nodes, qnode, pathbuf);
    if (len < 0 || qpos >= node_len[qnode])
        return -1;
    int64_t nt = 0;
    for (int32_t i = 0; i < len; ++i)
        for (int32_t t = 0; t < tokens_taken(node_len, pathbuf[i], qnode, qpos); ++t) {
            tok_node[nt] = pathbuf[i];
            tok_idx[nt] = t;
            ++nt;
        }
    return nt;
}

static int64_t longest_path_tokens(const int32_t *parent, const int32_t *node_len,
                                   int32_t num_nodes, const int32_t *query_node,
                                   int32_t num_queries, int32_t *pathbuf)
{
    int64_t best = 0;
    for (int32_t q = 0; q < num_queries; ++q) {
        int32_t len = path_of(parent, num_nodes, query_node[q], pathbuf);
        if (len < 0)
            return -1;
        int64_t nt = 0;
        for (int32_t i = 0; i < len; ++i)
            nt += node_len[pathbuf[i]];
        if (nt > best)
            best = nt;
    }
    return best;
}

/*
 * Tree attention for the listed queries (query_subset[i], i < n_subset; pass
 * NULL to mean all queries in order).  q: bf16 bits [Q][Hq][d].  out: fp64
 * [n_subset][Hq][d], lse: fp64 [n_subset][Hq].  Parallel over (query, head)
 * with `threads` OpenMP threads (<= 0: the runtime default).
 * Returns 0, or -1 for a bad tree / argument.
 */
int oracle_tree_attn_f64(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                         const int32_t *node_page_off, const int32_t *page_id, int32_t page_size,
                         const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
                         const int32_t *query_node, const int32_t *query_pos, int32_t num_queries,
                         const int32_t *query_subset, int32_t n_subset,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         double scale, double *out, double *lse, int32_t threads)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || page_size <= 0)
        return -1;
    int32_t group = num_q_heads / num_kv_heads;
    int32_t nsel = query_subset ? n_subset : num_queries;
    int32_t *pb = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_nodes > 0 ? num_nodes : 1));
    int64_t maxtok = longest_path_tokens(parent, node_len, num_nodes, query_node, num_queries, pb);
    free(pb);
    if (maxtok < 0)
        return -1;
    for (int32_t i = 0; i < nsel; ++i) {
        int32_t qi = query_subset ? query_subset[i] : i;
        if (qi < 0 || qi >= num_queries)
            return -1;
    }
    int bad = 0;
#ifdef _OPENMP
    int nthr = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel num_threads(nthr) reduction(| : bad)
#endif
    {
        int32_t *pathbuf = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_nodes > 0 ? num_nodes : 1));
        int32_t *tok_node = (int32_t *)malloc(sizeof(int32_t) * (size_t)(maxtok > 0 ? maxtok : 1));
        int32_t *tok_idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(maxtok > 0 ? maxtok : 1));
        double *scores = (double *)malloc(sizeof(double) * (size_t)(maxtok > 0 ? maxtok : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t w = 0; w < (int64_t)nsel * num_q_heads; ++w) {
            int32_t i = (int32_t)(w / num_q_heads);
            int32_t h = (int32_t)(w % num_q_heads);
            int32_t qi = query_subset ? query_subset[i] : i;
            int64_t nt = path_tokens(parent, node_len, num_nodes, query_node[qi],
                                     query_pos ? query_pos[qi] : -1, pathbuf, tok_node, tok_idx);
            if (nt < 0) {
                bad = 1;
                continue;
            }
            const uint16_t *qv = q + ((size_t)qi * num_q_heads + h) * head_dim;
            double *o = out + ((size_t)i * num_q_heads + h) * head_dim;
            lse[(size_t)i * num_q_heads + h] =
                attend(qv, k_pages, v_pages, node_page_off, page_id, page_size, num_kv_heads,
                       head_dim, h / group, scale, tok_node, tok_idx, nt, scores, o);
        }
        free(pathbuf);
        free(tok_node);
        free(tok_idx);
        free(scores);
    }
    return bad ? -1 : 0;
}

/*
 * The same result reached the split-K way the method uses (DeFT Guide,
 * section "Deep Dive", online-softmax tile accumulation; abstract: partial
 * results merged per query): each query's path-token sequence is cut into
 * pieces before every position i with cut[i] != 0 (cut has `cut_len`
 * entries; positions beyond it are never cut), each piece gives a normalised
 * partial output and its own lse, and the pieces are merged by their lse
 * weights:  M = max lse_p,  w_p = exp(lse_p - M),
 *           out = sum w_p o_p / sum w_p,   lse = M + ln sum w_p.
 * Single-threaded.  Same outputs as oracle_tree_attn_f64 over all queries.
 */
int oracle_tree_attn_pieces_f64(const uint16_t *q, const uint16_t *k_pages,
                                const uint16_t *v_pages, const int32_t *node_page_off,
                                const int32_t *page_id, int32_t page_size,
                                const int32_t *parent, const int32_t *node_len, int32_t num_nodes,
                                const int32_t *query_node, const int32_t *query_pos,
                                int32_t num_queries, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, double scale, const uint8_t *cut, int64_t cut_len,
                                double *out, double *lse)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || page_size <= 0)
        return -1;
    int32_t group = num_q_heads / num_kv_heads;
    int32_t *pathbuf = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_nodes > 0 ? num_nodes : 1));
    int64_t maxtok = longest_path_tokens(parent, node_len, num_nodes, query_node, num_queries, pathbuf);
    if (maxtok < 0) {
        free(pathbuf);
        return -1;
    }
    size_t cap = (size_t)(maxtok > 0 ? maxtok : 1);
    int32_t *tok_node = (int32_t *)malloc(sizeof(int32_t) * cap);
    int32_t *tok_idx = (int32_t *)malloc(sizeof(int32_t) * cap);
    double *scores = (double *)malloc(sizeof(double) * cap);
    double *piece_out = (double *)malloc(sizeof(double) * (size_t)head_dim * cap);
    double *piece_lse = (double *)malloc(sizeof(double) * cap);
    for (int32_t qi = 0; qi < num_queries; ++qi) {
        int64_t nt = path_tokens(parent, node_len, num_nodes, query_node[qi],
                                 query_pos ? query_pos[qi] : -1, pathbuf, tok_node, tok_idx);
        if (nt < 0) {
            free(pathbuf);
            free(tok_node);
            free(tok_idx);
            free(scores);
            free(piece_out);
            free(piece_lse);
            return -1;
        }
        for (int32_t h = 0; h < num_q_heads; ++h) {
            const uint16_t *qv = q + ((size_t)qi * num_q_heads + h) * head_dim;
            int64_t npieces = 0;
            int64_t start = 0;
            for (int64_t i = 1; i <= nt; ++i) {
                int end_here = (i == nt) || (i < cut_len && cut[i]);
                if (!end_here)
                    continue;
                piece_lse[npieces] =
                    attend(qv, k_pages, v_pages, node_page_off, page_id, page_size, num_kv_heads,
                           head_dim, h / group, scale, tok_node + start, tok_idx + start,
                           i - start, scores, piece_out + (size_t)npieces * head_dim);
                ++npieces;
                start = i;
            }
            double *o = out + ((size_t)qi * num_q_heads + h) * head_dim;
            for (int32_t i = 0; i < head_dim; ++i)
                o[i] = 0.0;
            double M = -INFINITY;
            for (int64_t p = 0; p < npieces; ++p)
                if (piece_lse[p] > M)
                    M = piece_lse[p];
            if (npieces == 0 || M == -INFINITY) {
                lse[(size_t)qi * num_q_heads + h] = -INFINITY;
                continue;
            }
            double wsum = 0.0;
            for (int64_t p = 0; p < npieces; ++p) {
                double w = exp(piece_lse[p] - M);
                wsum += w;
                for (int32_t i = 0; i < head_dim; ++i)
                    o[i] += w * piece_out[(size_t)p * head_dim + i];
            }
            for (int32_t i = 0; i < head_dim; ++i)
                o[i] /= wsum;
            lse[(size_t)qi * num_q_heads + h] = M + log(wsum);
        }
    }
    free(pathbuf);
    free(tok_node);
    free(tok_idx);
    free(scores);
    free(piece_out);
    free(piece_lse);
    return 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
