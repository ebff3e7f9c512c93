// phase1_mma.cu -- phase-1 partial attention on tcgen05 tensor cores, for
// work items with 16..128 rows (rows = queries of the item x GQA group) and
// head_dim 128.
//
// Same result as phase1_fma.cu (DeFT Guide, "Deep Dive": tree-constrained
// attention, online-softmax tile accumulation; DeFT abstract: KV-Guided
// Grouping), for chunks shared by enough queries that the two products
// S = q.K^T and O = P.V are dense contractions worth the tensor cores.
//
// Formulation: KV tokens on the MMA M dimension (128-token tiles), query
// rows on N (R rounded up to 16):
//     S^T[128 tok x N]  = K_tile[128 x 128] . Q^T[128 x N]       (TMEM, fp32)
//     O^T[128 d   x N] += V_tile^T[128 x 128] . P^T[128 tok x N]   (TMEM, fp32)
// so one thread owns one token of S^T (and one output dimension of O^T),
// and the softmax work of a tile is spread over all 128 threads whatever
// the row count.  Column maxima and sums are warp butterflies
// (reduce-scatter: lane l ends with column l) plus a 4-way exchange in
// shared memory.  Logits are kept in base 2; phase 2 converts.
//
// Operands in shared memory use the canonical 128-byte-swizzled layouts:
// K tile, Q^T and P^T K-major (rows of 64 bf16 = 128 B, 16-byte chunk c of
// row r stored at chunk c ^ (r % 8), 8-row atoms 1024 B apart), V tile the
// same bytes read MN-major for V^T.  KV rows are fetched through the page
// table with 16-byte cp.async copies, one token row at a time, so ragged
// node tails and 1-token nodes cost nothing extra; one CTA runs one
// (chunk, KV head, row block) and prefetches tile t+1 while computing t.
//
// Every wait on an mbarrier is bounded; a CTA whose MMA never completes
// writes NaN partials (so the step's output shows the failure), waits for
// its own copies, frees its TMEM and returns.
#include "common.cuh"
#include "deft_internal.h"
#include "tcgen05.cuh"

namespace deft {
namespace {

constexpr int kD = 128;
constexpr int kTileTok = 128;
constexpr int kMStages = 2;
constexpr int kMThreads = 128;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kHalf = 128 * 128;       // one 64-wide half of a 128-row operand (16 KB)
constexpr uint32_t kTileBytes = 2 * kHalf;  // one 128 x 128 bf16 operand (32 KB)

struct MmaSmem {
    static constexpr uint32_t kv_off = 0;  // [stage][K, V]
    static constexpr uint32_t q_off = kv_off + kMStages * 2 * kTileBytes;
    static constexpr uint32_t p_off = q_off + kTileBytes;
    static constexpr uint32_t meta_off = p_off + kTileBytes;                  // [stage][128] uint4
    static constexpr uint32_t seg_off = meta_off + kMStages * kTileTok * 16;  // pos/node/tb + uint4 masks
    static constexpr uint32_t red_off = seg_off + kMaxSegsPerChunk * 12 + kMaxSegsPerChunk * 16;
    static constexpr uint32_t stat_off = red_off + 4 * 128 * 4;               // m, alpha, l
    static constexpr uint32_t misc_off = stat_off + 3 * 128 * 4;
    static constexpr uint32_t total = misc_off + 64;
    static constexpr uint32_t alloc = total + 1024;  // room to align the base to 1024 bytes
};

// Warp butterfly that leaves in every lane l the reduction over the warp of
// column l of v (32 columns).  v is destroyed.
template <bool kMax>
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = upper ? v[i] : v[i + o];
            const float keep = upper ? v[i + o] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, o);
            v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
    }
    return v[0];
}

__device__ __forceinline__ uint32_t mask_word(const uint4 &m, int w)
{
    return w == 0 ? m.x : w == 1 ? m.y : w == 2 ? m.z : m.w;
}

__global__ void __launch_bounds__(kMThreads, 1) phase1_mma_kernel(AttnArgs a, DevPartition p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    uint4 *meta = reinterpret_cast<uint4 *>(smem + MmaSmem::meta_off);
    int32_t *s_pos = reinterpret_cast<int32_t *>(smem + MmaSmem::seg_off);
    int32_t *s_node = s_pos + kMaxSegsPerChunk;
    int32_t *s_tb = s_node + kMaxSegsPerChunk;
    uint4 *s_rmask = reinterpret_cast<uint4 *>(smem + MmaSmem::seg_off + kMaxSegsPerChunk * 12);
    float *red = reinterpret_cast<float *>(smem + MmaSmem::red_off);
    float *m_s = reinterpret_cast<float *>(smem + MmaSmem::stat_off);
    float *alpha_s = m_s + 128;
    float *l_fin = alpha_s + 128;
    const uint32_t bar = base + MmaSmem::misc_off;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + MmaSmem::misc_off + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads, G = a.gqa_group;
    const int item = blockIdx.x / Hkv;
    const int h = blockIdx.x - item * Hkv;
    const int c = p.mma_items[3 * item], qb = p.mma_items[3 * item + 1], qe = p.mma_items[3 * item + 2];
    const int R = (qe - qb) * G;
    const int NP = (R + 15) & ~15;
    const int sb = p.chunk_seg_off[c], nseg = p.chunk_seg_off[c + 1] - sb;
    const int cq0 = p.chunk_q_off[c] + qb;
    const int T = p.chunk_tokens[c];
    const int ntiles = (T + kTileTok - 1) / kTileTok;
    const int W = p.mask_words;

    if (warp == 0) {
        tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(bar, 1);
        tc::fence_mbar_init();
    }
    // Zero the operand buffers once: rows no token fills (chunk tails) and
    // padded query rows must hold finite values.
    for (uint32_t i = tid; i < MmaSmem::meta_off / 16; i += kMThreads)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    for (int s = tid; s < nseg; s += kMThreads) {
        s_pos[s] = p.seg_chunk_pos[sb + s];
        s_node[s] = p.seg_node[sb + s];
        s_tb[s] = p.seg_tok_begin[sb + s];
        const uint64_t *m = p.seg_mask + (size_t)(sb + s) * W;
        uint32_t rm[4] = {0, 0, 0, 0};
        for (int r = 0; r < R; ++r) {
            const int qid = p.chunk_q[cq0 + r / G];
            rm[r >> 5] |= (uint32_t)((m[qid >> 6] >> (qid & 63)) & 1ull) << (r & 31);
        }
        s_rmask[s] = make_uint4(rm[0], rm[1], rm[2], rm[3]);
    }
    m_s[tid] = -INFINITY;
    alpha_s[tid] = 1.f;
    __syncthreads();
    // Q^T operand: row r = (query, group member), K-major, swizzled.
    const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    for (int i = tid; i < R * 16; i += kMThreads) {
        const int r = i >> 4, ch = i & 15;
        const int qid = p.chunk_q[cq0 + r / G];
        const int hq = h * G + (r % G);
        const uint4 v = *reinterpret_cast<const uint4 *>(qg + ((size_t)qid * Hq + hq) * kD + ch * 8);
        *reinterpret_cast<uint4 *>(smem + MmaSmem::q_off + (ch >> 3) * kHalf + r * 128 +
                                   (((ch & 7) ^ (r & 7)) << 4)) = v;
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t tmem_S = tmem_base;
    const uint32_t tmem_O = tmem_base + 128;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

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

    // Copies of tile `tile` into stage `st`: warp w moves rows w, w+4, ...;
    // lane l resolves row w + 4l through the page table once, then the warp
    // copies one row per step (lanes 0-15 the K row, 16-31 the V row).
    auto issue_tile = [&](int tile, int st) {
        const int rl = warp + 4 * lane;
        const int pos = tile * kTileTok + rl;
        long long off = -1;
        uint4 rm = make_uint4(0, 0, 0, 0);
        if (pos < T) {
            const int s = find_seg(pos);
            const int t = s_tb[s] + pos - s_pos[s];
            const int page = a.page_id[a.node_page_off[s_node[s]] + t / kPageSize];
            off = (((long long)page * Hkv + h) * kPageSize + (t % kPageSize)) * kD;
            rm = s_rmask[s];
        }
        meta[st * kTileTok + rl] = rm;
        const int kv = lane >> 4, ch = lane & 15;
        const uint32_t dst0 = base + MmaSmem::kv_off + (uint32_t)(st * 2 + kv) * kTileBytes +
                              (ch >> 3) * kHalf;
        const __nv_bfloat16 *src0 = (kv ? vg : kg) + ch * 8;
#pragma unroll 4
        for (int k = 0; k < 32; ++k) {
            const int row = warp + 4 * k;
            const long long o = __shfl_sync(0xffffffffu, off, k);
            if (o >= 0)
                cp_async_16(dst0 + row * 128 + (((ch & 7) ^ (row & 7)) << 4), src0 + o);
        }
    };

    const uint32_t idesc_s = tc::idesc_bf16(128, NP, 0, 0);
    const uint32_t idesc_o = tc::idesc_bf16(128, NP, 1, 0);
    const float sc = a.scale_log2;
    float l_own[4] = {0.f, 0.f, 0.f, 0.f};  // column sums of columns 32*g + lane
    uint32_t phase = 0;
    bool ok = true;

#pragma unroll
    for (int st = 0; st < kMStages - 1; ++st) {
        if (st < ntiles)
            issue_tile(st, st);
        cp_async_commit();
    }
    for (int t = 0; t < ntiles && ok; ++t) {
        const int st = t % kMStages;
        if (t + kMStages - 1 < ntiles)
            issue_tile(t + kMStages - 1, (t + kMStages - 1) % kMStages);
        cp_async_commit();
        cp_async_wait<kMStages - 1>();
        tc::fence_proxy_async();
        __syncthreads();

        // S^T = K_t . Q^T
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t kb = base + MmaSmem::kv_off + (uint32_t)(st * 2) * kTileBytes;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t ad = tc::smem_desc(kb + (s >> 2) * kHalf + (s & 3) * 32, 16, 1024);
                const uint64_t bd =
                    tc::smem_desc(base + MmaSmem::q_off + (s >> 2) * kHalf + (s & 3) * 32, 16, 1024);
                tc::mma_bf16(tmem_S, ad, bd, idesc_s, s > 0 ? 1u : 0u);
            }
            tc::mma_commit(bar);
        }
        ok = __syncthreads_and(tc::mbar_wait(bar, phase & 1));
        ++phase;
        if (!ok)
            break;
        tc::fence_after_sync();

        // Column maxima of the tile.
        const uint4 rm = meta[st * kTileTok + tid];
        for (int g = 0; g < NP; g += 32) {
            float v[32];
            tc::tmem_ld32(tmem_S + lane_off + g, v);
            const uint32_t w = mask_word(rm, g >> 5);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                v[i] = ((w >> i) & 1u) && (g + i < R) ? v[i] * sc : -INFINITY;
            red[warp * 128 + g + lane] = reduce_scatter32<true>(v, lane);
        }
        __syncthreads();
        bool need = false;
        if (tid < NP) {
            const float mt = fmaxf(fmaxf(red[tid], red[128 + tid]), fmaxf(red[256 + tid], red[384 + tid]));
            const float mo = m_s[tid];
            const float mn = fmaxf(mo, mt);
            const float al = mn == -INFINITY ? 1.f : exp2f(mo - mn);
            m_s[tid] = mn;
            alpha_s[tid] = al;
            need = al != 1.f;
        }
        const bool rescale = __syncthreads_or(need && t > 0) != 0;
        if (rescale) {
            for (int g = 0; g < NP; g += 32) {
                float v[32];
                tc::tmem_ld32(tmem_O + lane_off + g, v);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] *= alpha_s[g + i];
                tc::tmem_st32(tmem_O + lane_off + g, v);
                l_own[g >> 5] *= alpha_s[g + lane];
            }
        }

        // Probabilities -> P^T (bf16, K-major over tokens) and column sums.
        {
            const int j = tid;
            const uint32_t prow = base + MmaSmem::p_off + (j >> 6) * kHalf + ((j & 63) & 7) * 2;
            const int pch = (j & 63) >> 3;
            for (int g = 0; g < NP; g += 32) {
                float v[32];
                tc::tmem_ld32(tmem_S + lane_off + g, v);
                const uint32_t w = mask_word(rm, g >> 5);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int r = g + i;
                    float pr = 0.f;
                    if (((w >> i) & 1u) && r < R) {
                        // The normaliser sums the fp32 probabilities; only the
                        // P.V operand is rounded to bf16.
                        pr = exp2f(fmaf(v[i], sc, -m_s[r]));
                        const __nv_bfloat16 b = __float2bfloat16_rn(pr);
                        uint8_t *dst = smem + (prow - base) + r * 128 + ((pch ^ (r & 7)) << 4);
                        *reinterpret_cast<__nv_bfloat16 *>(dst) = b;
                    } else if (r < NP) {
                        uint8_t *dst = smem + (prow - base) + r * 128 + ((pch ^ (r & 7)) << 4);
                        *reinterpret_cast<__nv_bfloat16 *>(dst) = __float2bfloat16_rn(0.f);
                    }
                    v[i] = pr;
                }
                l_own[g >> 5] += reduce_scatter32<false>(v, lane);
            }
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();

        // O^T += V_t^T . P^T
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t vb = base + MmaSmem::kv_off + (uint32_t)(st * 2 + 1) * kTileBytes;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t ad = tc::smem_desc(vb + s * 2048, kHalf, 1024);
                const uint64_t bd =
                    tc::smem_desc(base + MmaSmem::p_off + (s >> 2) * kHalf + (s & 3) * 32, 16, 1024);
                tc::mma_bf16(tmem_O, ad, bd, idesc_o, (t > 0 || s > 0) ? 1u : 0u);
            }
            tc::mma_commit(bar);
        }
        ok = __syncthreads_and(tc::mbar_wait(bar, phase & 1));
        ++phase;
        tc::fence_after_sync();
    }
    cp_async_wait<0>();

    if (ok) {
        // Normalisers, then O^T / l written as fp32 partials (lane = dimension).
        for (int g = 0; g < NP; g += 32)
            red[warp * 128 + g + lane] = l_own[g >> 5];
        __syncthreads();
        if (tid < NP)
            l_fin[tid] = red[tid] + red[128 + tid] + red[256 + tid] + red[384 + tid];
        __syncthreads();
        for (int g = 0; g < NP; g += 32) {
            float v[32];
            tc::tmem_ld32(tmem_O + lane_off + g, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int r = g + i;
                if (r < R) {
                    const size_t prow = (size_t)(cq0 + r / G) * Hq + h * G + (r % G);
                    a.o_part[prow * kD + tid] = v[i] / l_fin[r];
                }
            }
        }
        if (tid < R) {
            const size_t prow = (size_t)(cq0 + tid / G) * Hq + h * G + (tid % G);
            a.lse_part[prow] = m_s[tid] + log2f(l_fin[tid]);
        }
    } else {
        for (int r = 0; r < R; ++r) {
            const size_t prow = (size_t)(cq0 + r / G) * Hq + h * G + (r % G);
            a.o_part[prow * kD + tid] = __int_as_float(0x7fc00000);
            if (tid == 0)
                a.lse_part[prow] = __int_as_float(0x7fc00000);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0)
        tc::tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

bool mma_supported(int32_t head_dim) { return head_dim == kD; }

int launch_phase1_mma(const AttnArgs &a, const DevPartition &p, void *stream)
{
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(
            phase1_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MmaSmem::alloc);
        if (e != cudaSuccess)
            return (int)e;
        configured = true;
    }
    if (p.num_mma_items <= 0)
        return 0;
    const unsigned blocks = (unsigned)((int64_t)p.num_mma_items * a.num_kv_heads);
    phase1_mma_kernel<<<blocks, kMThreads, MmaSmem::alloc, reinterpret_cast<cudaStream_t>(stream)>>>(a, p);
    return (int)cudaGetLastError();
}

}  // namespace deft
