// phase1_fma.cu -- phase-1 partial attention on CUDA cores, for work items
// with fewer than 16 rows (rows = queries of the item x GQA group).
//
// What one thread block computes (DeFT Guide, "Deep Dive": tree-constrained
// attention and online-softmax tile accumulation; DeFT abstract: KV-Guided
// Grouping): for one chunk c, one KV head h and the item's rows r (query k,
// group member g, query head h*G+g), over the chunk's tokens j whose segment
// bitmask contains the row's query,
//     s_rj = (q_r . k_j) * scale,  m_r = max_j s_rj,  l_r = sum_j 2^... ,
//     o_r = sum_j exp(s_rj - m_r) v_j / l_r,  L_r = log-sum-exp of s_r,
// and stores o_r (fp32) and L_r (base 2) in the partial slot of (c, k).
// Logits are carried in base 2 (q pre-scaled by scale * log2 e) so that the
// exponentials are single exp2 instructions; phase 2 converts back.
//
// Data movement: the chunk's KV rows are fetched through the page table with
// 16-byte cp.async copies (coalesced: one token row of a page is 2*head_dim
// contiguous bytes) into a 3-stage shared-memory ring of 64-token tiles.
// Per-token page lookup makes ragged pages, 1-token nodes and arbitrary
// page order cost nothing extra.  The 16-byte chunks of each row are stored
// XOR-permuted so that both compute access patterns below are free of bank
// conflicts.
//
// Compute mapping (8 warps, each owning 8 tokens of a tile):
//   q.k   lane = 4 * token + quarter; each lane dots a quarter of head_dim
//         for every row (q broadcast from shared memory), then two xor
//         shuffles complete the dot;
//   p.v   lane owns head_dim/32 output elements of every row; the warp's 8
//         probabilities per row are broadcast through shared memory.
// Each warp keeps its own running max / sum / output per row; the 8 warp
// states are merged through shared memory at the end.
#include "common.cuh"
#include "deft_internal.h"
#include "kprof.cuh"

namespace deft {
namespace {

constexpr int kTile = 64;     // tokens per pipeline stage
constexpr int kStages = 3;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// Physical 16-byte chunk of logical chunk lc in token row `row`.
__device__ __forceinline__ int swz(int row, int lc)
{
    return lc ^ ((lc >> 3) << 1) ^ (row & 1);
}

template <int D, int RMAX>
struct FmaSmem {
    static constexpr int CH = D / 8;           // 16-byte chunks per token row
    static constexpr int QSTR = D / 4 + 4;     // padded quarter stride (floats)
    static constexpr int QROW = 4 * QSTR;
    static constexpr size_t kv_bytes = (size_t)kStages * 2 * kTile * D * 2;
    static constexpr size_t qs_off = kv_bytes;
    static constexpr size_t qs_bytes = (size_t)RMAX * QROW * 4;
    static constexpr size_t meta_off = qs_off + qs_bytes;
    static constexpr size_t meta_bytes = (size_t)kStages * kTile * 4;
    static constexpr size_t seg_off = meta_off + meta_bytes;
    static constexpr size_t seg_bytes = (size_t)kMaxSegsPerChunk * 4 * 4;
    static constexpr size_t ps_off = seg_off + seg_bytes;
    static constexpr size_t ps_bytes = (size_t)kWarps * 8 * RMAX * 4;
    static constexpr size_t total = ps_off + ps_bytes;
    static constexpr size_t merge_bytes = (size_t)kWarps * RMAX * (D + 2) * 4;
    static_assert(merge_bytes <= kv_bytes, "merge scratch must fit in the KV ring");
};

template <int D, int RMAX>
__global__ void __launch_bounds__(kThreads, (RMAX <= 8 ? 2 : 1))
phase1_fma_kernel(AttnArgs a, DevPartition p, const int32_t *__restrict__ items)
{
    using S = FmaSmem<D, RMAX>;
    constexpr int CH = S::CH;
    constexpr int E = D / 32;       // output elements per lane in p.v
    constexpr int QCH = CH / 4;     // chunks per lane in q.k
    extern __shared__ __align__(128) uint8_t smem[];
    float *qs = reinterpret_cast<float *>(smem + S::qs_off);
    uint32_t *meta = reinterpret_cast<uint32_t *>(smem + S::meta_off);
    int32_t *s_pos = reinterpret_cast<int32_t *>(smem + S::seg_off);
    int32_t *s_node = s_pos + kMaxSegsPerChunk;
    int32_t *s_tb = s_node + kMaxSegsPerChunk;
    uint32_t *s_rmask = reinterpret_cast<uint32_t *>(s_tb + kMaxSegsPerChunk);
    float *ps = reinterpret_cast<float *>(smem + S::ps_off);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        KPROF(a, 2000);
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads, G = a.gqa_group;
    const int item = blockIdx.x / Hkv;
    const int h = blockIdx.x - item * Hkv;
    const int c = items[3 * item], qb = items[3 * item + 1], qe = items[3 * item + 2];
    const int R = (qe - qb) * G;
    const int sb = p.chunk_seg_off[c], nseg = p.chunk_seg_off[c + 1] - sb;
    const int cq0 = p.chunk_q_off[c] + qb;
    const int T = p.chunk_tokens[c];
    const int ntiles = (T + kTile - 1) / kTile;

    // Segment table of the chunk, with each segment's row mask: bit r is set
    // iff row r's query is in the segment's query bitmask.
    for (int s = tid; s < nseg; s += kThreads) {
        s_pos[s] = p.seg_chunk_pos[sb + s];
        s_node[s] = a.node_page_off[p.seg_node[sb + s]];   // first page_id index of the node
        s_tb[s] = p.seg_tok_begin[sb + s];
        const uint32_t *lm = p.seg_lmask + p.seg_lmask_off[sb + s];
        uint32_t rm = 0;
        for (int r = 0; r < R; ++r) {
            const int k = qb + r / G;
            rm |= ((lm[k >> 5] >> (k & 31)) & 1u) << r;
        }
        s_rmask[s] = rm;
    }
    // Query rows, pre-scaled into base-2 logits, stored per head_dim quarter
    // with padding so the four quarters sit in different banks.
    const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    for (int i = tid; i < RMAX * D; i += kThreads) {
        const int r = i / D, e = i - r * D;
        float v = 0.f;
        if (r < R) {
            const int qid = p.chunk_q[cq0 + r / G];
            const int hq = h * G + (r % G);
            v = __bfloat162float(qg[((size_t)qid * Hq + hq) * D + e]) * a.scale_log2;
        }
        qs[r * S::QROW + (e / (D / 4)) * S::QSTR + (e % (D / 4))] = v;
    }
    __syncthreads();

    auto find_seg = [&](int pos) {
        int lo = 0, hi = nseg - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_pos[mid] <= pos)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    };
    const __nv_bfloat16 *kg = reinterpret_cast<const __nv_bfloat16 *>(a.k_pages);
    const __nv_bfloat16 *vg = reinterpret_cast<const __nv_bfloat16 *>(a.v_pages);
    auto kv_stage = [&](int st, int kv) { return smem + ((size_t)(st * 2 + kv) * kTile) * D * 2; };

    auto issue_tile = [&](int tile, int st) {
        const int base = tile * kTile;
        constexpr int NCOPY = kTile * 2 * CH;
        for (int i = tid; i < NCOPY; i += kThreads) {
            const int row = i / (2 * CH), idx = i - row * (2 * CH);
            const int kv = idx / CH, lc = idx - kv * CH;
            const int pos = base + row;
            if (pos < T) {
                const int s = find_seg(pos);
                const int t = s_tb[s] + pos - s_pos[s];
                const int page = a.page_id[s_node[s] + t / kPageSize];
                const size_t off =
                    (((size_t)page * Hkv + h) * kPageSize + (t % kPageSize)) * D + lc * 8;
                cp_async_16(smem_u32(kv_stage(st, kv) + (size_t)row * D * 2 + swz(row, lc) * 16),
                            (kv ? vg : kg) + off);
            }
        }
        if (tid < kTile) {
            const int pos = base + tid;
            meta[st * kTile + tid] = pos < T ? s_rmask[find_seg(pos)] : 0u;
        }
    };

    // Per-warp online-softmax state for every row.
    float m_run[RMAX], l_run[RMAX], o_acc[RMAX][E];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        m_run[r] = -INFINITY;
        l_run[r] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e)
            o_acc[r][e] = 0.f;
    }
    const int tok = lane >> 2, qtr = lane & 3;
    float *psw = ps + warp * 8 * RMAX;

#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) {
        if (st < ntiles)
            issue_tile(st, st);
        cp_async_commit();
    }
    if (tid == 0)
        KPROF(a, 2001);
    for (int tile = 0; tile < ntiles; ++tile) {
        const int nxt = tile + kStages - 1;
        if (nxt < ntiles)
            issue_tile(nxt, nxt % kStages);
        if (tid == 0)
            KPROF(a, 2100 + 4 * tile);
        cp_async_commit();
        cp_async_wait<kStages - 1>();
        __syncthreads();
        if (tid == 0)
            KPROF(a, 2101 + 4 * tile);

        const int st = tile % kStages;
        const uint8_t *Ks = kv_stage(st, 0);
        const uint8_t *Vs = kv_stage(st, 1);
        const int row = warp * 8 + tok;

        // q.k: this lane's quarter of head_dim, all rows.
        float s[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
            s[r] = 0.f;
#pragma unroll
        for (int c4 = 0; c4 < QCH; ++c4) {
            const int lc = qtr * QCH + c4;
            const uint4 kw = *reinterpret_cast<const uint4 *>(Ks + (size_t)row * D * 2 + swz(row, lc) * 16);
            const float2 k01 = bf16x2_to_float2(kw.x), k23 = bf16x2_to_float2(kw.y);
            const float2 k45 = bf16x2_to_float2(kw.z), k67 = bf16x2_to_float2(kw.w);
#pragma unroll
            for (int r = 0; r < RMAX; ++r) {
                if (r < R) {
                    const float *qp = qs + r * S::QROW + qtr * S::QSTR + c4 * 8;
                    const float4 qa = *reinterpret_cast<const float4 *>(qp);
                    const float4 qb4 = *reinterpret_cast<const float4 *>(qp + 4);
                    float acc = s[r];
                    acc = fmaf(qa.x, k01.x, acc);
                    acc = fmaf(qa.y, k01.y, acc);
                    acc = fmaf(qa.z, k23.x, acc);
                    acc = fmaf(qa.w, k23.y, acc);
                    acc = fmaf(qb4.x, k45.x, acc);
                    acc = fmaf(qb4.y, k45.y, acc);
                    acc = fmaf(qb4.z, k67.x, acc);
                    acc = fmaf(qb4.w, k67.y, acc);
                    s[r] = acc;
                }
            }
        }
        const uint32_t rmask = meta[st * kTile + row];
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            if (r < R) {
                float v = s[r];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v = ((rmask >> r) & 1u) ? v : -INFINITY;
                float mx = v;
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mnew = fmaxf(m_run[r], mx);
                float pr = 0.f, alpha = 1.f;
                if (mnew != -INFINITY) {
                    alpha = exp2f(m_run[r] - mnew);
                    pr = exp2f(v - mnew);
                }
                m_run[r] = mnew;
                l_run[r] = l_run[r] * alpha + (qtr == 0 ? pr : 0.f);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    o_acc[r][e] *= alpha;
                if (qtr == (r & 3))
                    psw[tok * RMAX + r] = pr;
            }
        }
        __syncwarp();
        // p.v over the warp's 8 tokens.
#pragma unroll 2
        for (int tt = 0; tt < 8; ++tt) {
            const int rt = warp * 8 + tt;
            if (meta[st * kTile + rt] == 0u)
                continue;
            float vf[E];
            const uint8_t *vrow = Vs + (size_t)rt * D * 2;
            if constexpr (E == 4) {
                const uint2 vw = *reinterpret_cast<const uint2 *>(vrow + swz(rt, lane >> 1) * 16 + (lane & 1) * 8);
                const float2 a01 = bf16x2_to_float2(vw.x), a23 = bf16x2_to_float2(vw.y);
                vf[0] = a01.x; vf[1] = a01.y; vf[2] = a23.x; vf[3] = a23.y;
            } else {
                const uint32_t vw = *reinterpret_cast<const uint32_t *>(vrow + swz(rt, lane >> 2) * 16 + (lane & 3) * 4);
                const float2 a01 = bf16x2_to_float2(vw);
                vf[0] = a01.x; vf[1] = a01.y;
            }
            const float *pp = psw + tt * RMAX;
#pragma unroll
            for (int r = 0; r < RMAX; ++r) {
                if (r < R) {
                    const float pr = pp[r];
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        o_acc[r][e] = fmaf(pr, vf[e], o_acc[r][e]);
                }
            }
        }
        __syncthreads();
        if (tid == 0)
            KPROF(a, 2102 + 4 * tile);
    }
    cp_async_wait<0>();
    __syncthreads();

    // Merge the 8 warp states of every row and store the partial.
    float *mw = reinterpret_cast<float *>(smem);          // [warps][RMAX]
    float *lw = mw + kWarps * RMAX;                      // [warps][RMAX]
    float *ow = lw + kWarps * RMAX;                      // [warps][RMAX][D]
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        if (r < R) {
            const float lt = warp_sum(l_run[r]);
            if (lane == 0) {
                mw[warp * RMAX + r] = m_run[r];
                lw[warp * RMAX + r] = lt;
            }
#pragma unroll
            for (int e = 0; e < E; ++e)
                ow[((size_t)warp * RMAX + r) * D + lane * E + e] = o_acc[r][e];
        }
    }
    __syncthreads();
    for (int i = tid; i < R * D; i += kThreads) {
        const int r = i / D, e = i - r * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            M = fmaxf(M, mw[w * RMAX + r]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float sc = exp2f(mw[w * RMAX + r] - M);
                L = fmaf(lw[w * RMAX + r], sc, L);
                O = fmaf(ow[((size_t)w * RMAX + r) * D + e], sc, O);
            }
        }
        const int slot = cq0 + r / G;
        const int hq = h * G + (r % G);
        const size_t prow = (size_t)slot * Hq + hq;
        a.o_part[prow * D + e] = L > 0.f ? O / L : 0.f;
        if (e == 0)
            a.lse_part[prow] = L > 0.f ? M + log2f(L) : -INFINITY;
    }
}

template <int D, int RMAX>
int launch_one(const AttnArgs &a, const DevPartition &p, const int32_t *items, int32_t n,
               cudaStream_t st)
{
    using S = FmaSmem<D, RMAX>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(phase1_fma_kernel<D, RMAX>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)S::total);
        if (e != cudaSuccess)
            return (int)e;
        configured = true;
    }
    const unsigned blocks = (unsigned)((int64_t)n * a.num_kv_heads);
    phase1_fma_kernel<D, RMAX><<<blocks, kThreads, S::total, st>>>(a, p, items);
    return (int)cudaGetLastError();
}

template <int D>
int launch_bucket(int bucket, const AttnArgs &a, const DevPartition &p, const int32_t *items,
                  int32_t n, cudaStream_t st)
{
    switch (bucket) {
    case 0: return launch_one<D, 1>(a, p, items, n, st);
    case 1: return launch_one<D, 2>(a, p, items, n, st);
    case 2: return launch_one<D, 4>(a, p, items, n, st);
    case 3: return launch_one<D, 8>(a, p, items, n, st);
    default: return launch_one<D, 16>(a, p, items, n, st);
    }
}

}  // namespace

int launch_phase1_fma(const AttnArgs &a, const DevPartition &p, const int32_t *items, int32_t n,
                      int bucket, void *stream)
{
    if (n <= 0)
        return 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return a.head_dim == 128 ? launch_bucket<128>(bucket, a, p, items, n, st)
                             : launch_bucket<64>(bucket, a, p, items, n, st);
}

}  // namespace deft
