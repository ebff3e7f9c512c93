// phase1_mma.cu -- phase-1 partial attention on tcgen05 tensor cores, for
// work items with 16..64 rows (rows = queries of the item x GQA group) and
// head_dim 128.  Chunks with more rows are cut into several items, each
// reading the chunk (the others mostly from L2): a wider item would cost
// more in its softmax, at 48 or 64 columns a warpgroup, than the re-read.
//
// Same result as phase1_fma.cu (DeFT Guide, "Deep Dive": tree-constrained
// attention, online-softmax tile accumulation; DeFT abstract: KV-Guided
// Grouping), for chunks shared by enough queries that S = q.K^T and O = P.V
// are dense contractions worth the tensor cores.
//
// Formulation: KV tokens on the MMA M dimension (128-token tiles), the
// item's query rows on N (RP = 2 NPH columns, NPH a template parameter;
// columns past the item's rows are masked):
//     S^T[128 tok x RP]  = K_tile . Q^T            (TMEM, fp32, 2 buffers)
//     O^T[128 d   x RP] += V_tile^T . P^T          (TMEM, fp32, 2 buffers)
// Eight MMAs (K = 16 each) per product and tile.  Two softmax warpgroups
// split the RP columns (NPH each); a thread owns one token of S^T and, at
// the end, one output dimension of O^T.  The column maximum is exact after
// a unit's first tile and afterwards only raised (with a rescale of O and
// of the per-thread column sums) when a logit exceeds it by more than 2^8,
// decided by a warpgroup vote.  Logits are base 2.
//
// Persistent CTAs (one per SM): the launch's early CTAs, those that start
// with the step, first take a contiguous block of units (unit = item x KV
// head, item-major, largest items first; 9/10 of an even share of the
// estimated cost among them); then every CTA takes units one at a time from the launch's work
// queue (an atomic counter), so a CTA that starts late or runs fast takes
// more;
// all roles walk the CTA's units in order and its tiles form one sequence
// through the stages, so the next unit's loads and its first S overlap the
// end of the current one.
// Roles (16 warps; the softmax warpgroups run with 168 registers a thread,
// the other two with 88):
//   warps 0-3, 4-7  softmax warpgroups 0 and 1 (column halves); at a unit's
//                   end they reduce their column sums and hand them, with
//                   the partial rows, to the epilogue warpgroup;
//   warps 8, 10     K and V producers: resolve a tile's pages through the
//                   page table one tile ahead, load full aligned pages with
//                   TMA (one box for eight consecutive pages, a 4 KB box a
//                   page otherwise) and ragged
//                   rows (node tails, packed one-token nodes) with 16-byte
//                   cp.async at the exact token count; K of a stage is
//                   refilled as soon as S of the tile two back is done, V
//                   once its P.V is done;
//   warp 9          allocates TMEM; lane 0 issues the MMAs, S(t) and P.V(t-1)
//                   in whichever order their inputs become ready;
//   warp 11         takes the next unit from the queue and passes its number
//                   to the producers through a shared-memory ring; per
//                   item, the segment table (positions, page bases, row
//                   masks); per unit, Q^T (two buffers, so the next unit's
//                   Q^T loads meanwhile);
//   warps 12-15     epilogue: O^T / l out of TMEM (two O buffers) into the
//                   fp32 partials while the softmax warpgroups go on with
//                   the next unit; it waits for the unit's last P.V itself
//                   (the softmax warpgroups hand over their column sums
//                   without waiting for it).
// Every hand-off is an mbarrier, every wait on one is bounded.  A CTA whose
// wait runs out writes NaN partials for its units (the step's output then
// shows the failure), waits for its own copies, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "merge.cuh"
#include "tcgen05.cuh"

namespace deft {
namespace {

constexpr int kD = 128;
constexpr int kTileTok = 128;
constexpr int kThreadsMma = 512;
// Registers per thread: the launch gives 128; the softmax warpgroups take
// 168 and the other two 88 (2 x 128 x 168 + 2 x 128 x 88 = 512 x 128).
constexpr uint32_t kRegsSoftmax = 168, kRegsOther = 88;
static_assert(2 * 128 * kRegsSoftmax + 2 * 128 * kRegsOther == kThreadsMma * 128, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kHalf = 128 * 128;       // one 64-wide half of a 128-row operand (16 KB)
constexpr uint32_t kTileBytes = 2 * kHalf;  // one 128 x 128 bf16 operand (32 KB)
// K and V tiles: [16 groups of 8 tokens][d half][8 tokens][128 B], 128-byte
// swizzled.  A group is two 1 KB swizzle atoms (dims 0-63, 64-127), so a
// 16-token page is 4 KB contiguous in the tile and lands with one TMA box.
constexpr uint32_t kRowGroup = 2048;        // 8 tokens x 128 dims
constexpr uint32_t kPageBytes = 4096;       // K (or V) of one 16-token page
constexpr int kSegInts = 7 * kMaxSegsPerChunk;  // pos, page base, token begin, row mask (4)

constexpr int kUnitQueue = 8;   // unit numbers passed from the metadata warp to the producers

struct UnitInfo {
    int32_t R;       // rows
    int32_t cq0;     // first slot of the unit's rows
    int32_t h;       // KV head
    int32_t ntiles;  // -1: no more units
    int32_t pad[4];
};

struct ItemInfo {
    int32_t nseg;
    int32_t T;       // chunk tokens
    int32_t pad[2];
};

// Shared-memory layout for NPH columns per warpgroup (RP = 2 NPH, NPH 16
// or 32).  Q^T is sized by RP, which leaves room for a third V stage when
// NPH = 16: a V stage is held through its tile's softmax, K only until S.
template <int NPH>
struct Smem {
    static_assert(NPH == 16 || NPH == 32, "16 or 32 columns a warpgroup");
    static constexpr int RP = 2 * NPH;
    static constexpr int VST = NPH <= 16 ? 3 : 2;                    // V stages (K has 2)
    static constexpr int QB = 2;                                     // Q^T buffers
    static constexpr uint32_t q_half = RP * 128;                     // one 64-wide half of Q^T
    static constexpr uint32_t k_off = 0;                             // [2] K operands
    static constexpr uint32_t v_off = k_off + 2 * kTileBytes;       // [VST] V operands
    static constexpr uint32_t q_off = v_off + VST * kTileBytes;     // [QB] Q^T: [d half][RP rows][128 B]
    static constexpr uint32_t p_off = q_off + QB * 2 * q_half;      // P^T: [col block][128 tok][128 B]
    static constexpr uint32_t meta_off = p_off + kHalf;              // [4 slots][128] uint4 row masks
    static constexpr uint32_t seg_off = meta_off + 4 * kTileTok * 16;  // [2][kSegInts]
    static constexpr uint32_t red_off = seg_off + 2 * kSegInts * 4;  // [wg][warp][64]
    static constexpr uint32_t stat_off = red_off + 2 * 4 * 64 * 4;  // [wg][m, alpha, 1/l, out row][64]
    static constexpr uint32_t epi_off = stat_off + 2 * 4 * 64 * 4;   // [ob][wg][1/l 64, out row 64]; [ob][R, fail0, fail1, -]
    static constexpr uint32_t uinfo_off = epi_off + 2 * 2 * 128 * 4 + 2 * 16;  // [2] UnitInfo
    static constexpr uint32_t iinfo_off = uinfo_off + 2 * 32;         // [2] ItemInfo
    static constexpr uint32_t useq_off = iinfo_off + 2 * 16;         // [kUnitQueue] unit numbers
    static constexpr uint32_t bar_off = useq_off + kUnitQueue * 4;   // mbarriers
    static constexpr uint32_t misc_off = bar_off + 48 * 8;          // tmem base, error flag, queue flags
    static constexpr uint32_t total = misc_off + 16;
    static constexpr uint32_t alloc = total + 1024;
    static_assert(alloc <= 227 * 1024, "shared memory of one CTA");
    static_assert(q_off % 1024 == 0 && p_off % 1024 == 0, "128-byte-swizzle atoms");
};

// mbarrier slots
constexpr int kBarFullK = 0;     // [2] K of a stage landed (producer: 32 lanes + tx)
constexpr int kBarFullV = 2;     // [3] V of a stage landed
constexpr int kBarEmptyK = 5;    // [2] S of the stage's tile finished (MMA commit)
constexpr int kBarEmptyV = 7;    // [3] P.V of the stage's tile finished (MMA commit)
constexpr int kBarSFull = 10;    // [2] S buffer ready (MMA commit)
constexpr int kBarSFree = 12;    // [2] S buffer read (one arrival per warpgroup)
constexpr int kBarPFull = 14;    // P written (one arrival per warpgroup)
constexpr int kBarPvDone = 15;   // P.V finished (MMA commit)
constexpr int kBarSegFull = 16;  // [2] an item's segment table written (32 lanes)
constexpr int kBarSegEmpty = 18; // [2] ... no longer read (both producers, 32 lanes each)
constexpr int kBarUFull = 20;    // [2] a unit's description and Q^T written (32 lanes)
constexpr int kBarUEmpty = 22;   // [2] ... description read (MMA issuer + 2 warpgroups)
constexpr int kBarQFree = 24;    // the unit's last S finished: its Q^T buffer may be replaced (MMA commit)
constexpr int kBarOFree = 25;    // [2] O buffer read out by the epilogue warpgroup
constexpr int kBarQFull = 27;    // [kUnitQueue] a unit number written (metadata lane 0)
constexpr int kBarQEmpty = 35;   // [kUnitQueue] ... read (lane 0 of each producer)
constexpr int kBarQFree1 = 43;   // ... the same for Q^T buffer 1
constexpr int kBarEpiFull = 44;  // [2] a unit's column sums and rows handed to the epilogue (one per warpgroup)
constexpr int kBarOFull = 46;    // [2] a unit's last P.V finished: its O buffer holds the unit's output (MMA commit)
constexpr int kNumBars = 48;
__device__ __forceinline__ int qfree_bar(int qb) { return qb == 0 ? kBarQFree : kBarQFree1; }
static_assert(kNumBars * 8 <= Smem<16>::misc_off - Smem<16>::bar_off, "mbarrier space");

// Tensor maps over the paged K and V, both viewing the pool [pages][Hkv][16]
// [128] as five dimensions, innermost first: 64 dims (one 128-byte swizzle
// row), 8 tokens (256 B apart), the two d halves (128 B apart), 2 Hkv token
// groups (head h's two groups of 8 at 2h, 2h + 1; 2 KB apart) and pages.  A
// box lands in the tile layout above.  *1: boxes of one page of one head;
// *8: of eight consecutive pages of one head (a tile whose pages were
// allocated back to back in one copy).
struct KvMaps {
    CUtensorMap k1, v1, k8, v8;
};

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

template <int NPH>
__global__ void __launch_bounds__(kThreadsMma, 1)
phase1_mma_kernel(AttnArgs a, DevPartition p, const int32_t *__restrict__ items,
                  const uint4 *__restrict__ rmask, const int32_t *__restrict__ rmask_off,
                  int32_t n_units, int32_t static_units, int32_t early, uint32_t *__restrict__ queue,
                  const __grid_constant__ KvMaps maps)
{
    using L = Smem<NPH>;
    constexpr int RP = L::RP;     // MMA N: both warpgroups' columns
    constexpr int VST = L::VST;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    uint4 *meta = reinterpret_cast<uint4 *>(smem + L::meta_off);
    float *red = reinterpret_cast<float *>(smem + L::red_off);
    float *stat = reinterpret_cast<float *>(smem + L::stat_off);
    UnitInfo *uinfo = reinterpret_cast<UnitInfo *>(smem + L::uinfo_off);
    ItemInfo *iinfo = reinterpret_cast<ItemInfo *>(smem + L::iinfo_off);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc_off);
    volatile int *err = reinterpret_cast<volatile int *>(smem + L::misc_off + 4);
    // qdone[0]: this CTA has counted itself done with the queue; qdone[1]:
    // it was the launch's last to do so.
    volatile int *qdone = reinterpret_cast<volatile int *>(smem + L::misc_off + 8);
    auto bar = [&](int i) { return base + L::bar_off + 8u * (uint32_t)i; };
    // Segment table of buffer sb: s_pos, s_pgb (first page_id index of the
    // node), s_tb (token begin in the node), s_rmask (columns of warpgroup 0
    // in bits 0-63, of warpgroup 1 in bits 64-127).
    auto seg_tab = [&](int sbuf) { return reinterpret_cast<int32_t *>(smem + L::seg_off) + sbuf * kSegInts; };

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads, G = a.gqa_group;
    constexpr int UQ = kUnitQueue;
    volatile int32_t *useq = reinterpret_cast<volatile int32_t *>(smem + L::useq_off);

    // ---------------- set-up ----------------
    // The tensor maps are kernel parameters: fetch them before anything else.
    if (warp == 8 && lane < 4)
        tc::prefetch_tmap(lane == 0 ? &maps.k1 : lane == 1 ? &maps.k8 : lane == 2 ? &maps.v1 : &maps.v8);
    // Then warm L2 with this CTA's share of the plan's arrays, the node page
    // offsets and q, which the metadata warp and the producers walk in
    // chains of dependent loads as soon as the set-up is done.  Prefetches
    // change no data, so they go out before the wait for the stream's
    // earlier work (a later write to these lines lands in L2 all the same).
    prefetch_l2_share(p.arrays, p.array_bytes, blockIdx.x, gridDim.x, tid, kThreadsMma);
    prefetch_l2_share(a.node_page_off, (size_t)(p.num_nodes + 1) * 4, blockIdx.x, gridDim.x, tid, kThreadsMma);
    prefetch_l2_share(a.q, (size_t)p.num_queries * Hq * kD * 2, blockIdx.x, gridDim.x, tid, kThreadsMma);
    if (a.wait_prior)
        grid_dep_wait();
    // A CTA that starts late, when the queue has nothing left, leaves now.
    if ((int)blockIdx.x >= early &&
        __syncthreads_or(tid == 0 && queue_drained(queue, n_units, early * static_units))) {
        if (tid == 0)
            queue_done_idle(queue);
        return;
    }
    if (tid == 0) {
        grid_dep_launch();
    }
    if (warp == 9) {
        tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = kBarFullK; i < kBarEmptyK; ++i)
            tc::mbar_init(bar(i), 33);
        for (int i = kBarEmptyK; i < kBarSFree; ++i)
            tc::mbar_init(bar(i), 1);
        tc::mbar_init(bar(kBarSFree + 0), 2);
        tc::mbar_init(bar(kBarSFree + 1), 2);
        tc::mbar_init(bar(kBarPFull), 2);
        tc::mbar_init(bar(kBarPvDone), 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(kBarSegFull + i), 32);
            tc::mbar_init(bar(kBarSegEmpty + i), 64);
            tc::mbar_init(bar(kBarUFull + i), 32);
            tc::mbar_init(bar(kBarUEmpty + i), 3);
            tc::mbar_init(bar(kBarOFree + i), 1);
            tc::mbar_init(bar(kBarEpiFull + i), 2);
            tc::mbar_init(bar(kBarOFull + i), 1);
        }
        tc::mbar_init(bar(kBarQFree), 1);
        tc::mbar_init(bar(kBarQFree1), 1);
        for (int i = 0; i < UQ; ++i) {
            tc::mbar_init(bar(kBarQFull + i), 1);
            tc::mbar_init(bar(kBarQEmpty + i), 2);
        }
        *err = 0;
        qdone[0] = 0;
        qdone[1] = 0;
        tc::fence_mbar_init();
    }
    // Operands start finite: rows past a chunk's end are never loaded and
    // their P is 0, which must not meet a NaN.
    for (uint32_t i = tid; i < L::meta_off / 16; i += kThreadsMma)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    float *epi = reinterpret_cast<float *>(smem + L::epi_off);
    volatile int32_t *epi_info = reinterpret_cast<volatile int32_t *>(smem + L::epi_off + 2 * 2 * 128 * 4);

    if (warp >= 8) {
        // Warps 8-11 and the epilogue warpgroup give registers to the
        // softmax warpgroups (each warpgroup as a whole, before its roles).
        tc::setmaxnreg_dec<kRegsOther>();
        if (warp == 11) {
            // ---------------- metadata: segment tables and Q^T ----------------
            // Per unit, Q^T is copied into buffer i % QB once the last S of the
            // unit QB back has read it (with two buffers, while the previous
            // unit runs); the rows of the unit after it are prefetched into L2
            // meanwhile.  A new item's Q^T copy is issued before its segment
            // table is built, so the two chains of dependent loads overlap.
            const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(a.q);
            int iseq = -1, prev_item = -1, R = 0, cq0 = 0, ntiles = 0;
            // qrow[k]: q row of item row lane + 32 k without the head term
            // (query * Hq + group member), loaded once per item in parallel.
            int qrow[4] = {0, 0, 0, 0};
            auto issue_q = [&](int h, int qb) {
                // Row r's 16 chunks go to lanes 16 (r & 1) ... + 15 in step r / 2.
    #pragma unroll 4
                for (int x0 = 0; x0 < R * 16; x0 += 32) {
                    const int x = x0 + lane, r = x >> 4, ch = x & 15;
                    const int src = r & 31;
                    const int qr0 = __shfl_sync(0xffffffffu, qrow[0], src), qr1 = __shfl_sync(0xffffffffu, qrow[1], src);
                    const int qr2 = __shfl_sync(0xffffffffu, qrow[2], src), qr3 = __shfl_sync(0xffffffffu, qrow[3], src);
                    const int k = r >> 5;
                    const int qr = k == 0 ? qr0 : k == 1 ? qr1 : k == 2 ? qr2 : qr3;
                    if (x < R * 16)
                        cp_async_16(base + L::q_off + (uint32_t)qb * 2 * L::q_half + (ch >> 3) * L::q_half + r * 128 +
                                        (((ch & 7) ^ (r & 7)) << 4),
                                    qg + (size_t)(qr + h * G) * kD + ch * 8);
                }
                cp_async_commit();
            };
            auto prefetch_q = [&](int h) {
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (lane + 32 * k < R) {
                        const char *addr = reinterpret_cast<const char *>(qg + (size_t)(qrow[k] + h * G) * kD);
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(addr));
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(addr + 128));
                    }
                }
            };
            // Only the launch's early CTAs own a block: the others start when
            // the step's earlier launches leave their SMs.
            const int own_units = (int)blockIdx.x < early ? static_units : 0;
            for (int i = 0;; ++i) {
                // The next unit: first the CTA's own contiguous block (runs of
                // one item's heads share its tables), then the launch's queue.
                int u = (int)blockIdx.x * static_units + i;
                if (i >= own_units) {
                    if (lane == 0)
                        u = early * static_units + (int)atomicAdd(queue, 1u);
                    u = __shfl_sync(0xffffffffu, u, 0);
                }
                const bool last = u >= n_units;
                const int ub = i & 1;
                // Pass it (or the end, -1) to the producers.
                const int qslot = i % UQ;
                if (i >= UQ &&
                    !__all_sync(0xffffffffu, tc::mbar_wait(bar(kBarQEmpty + qslot), ((i / UQ) - 1) & 1))) {
                    if (!*err) *err = 201;
                    break;
                }
                if (lane == 0) {
                    useq[qslot] = last ? -1 : u;
                    tc::mbar_arrive(bar(kBarQFull + qslot));
                }
                if (last) {
                    if (lane == 0)
                        queue_done(queue, qdone);
                    // End mark for the MMA issuer and the softmax warpgroups.
                    if (i >= 2 && !__all_sync(0xffffffffu, tc::mbar_wait(bar(kBarUEmpty + ub), ((i - 2) >> 1) & 1))) {
                        if (!*err) *err = 202;
                        break;
                    }
                    if (lane == 0)
                        uinfo[ub].ntiles = -1;
                    __syncwarp();
                    tc::mbar_arrive(bar(kBarUFull + ub));
                    break;
                }
                const int item = u / Hkv, h = u - item * Hkv;
                bool q_issued = false;
                if (item != prev_item) {
                    prev_item = item;
                    ++iseq;
                    const int sbuf = iseq & 1;
                    const int c = items[3 * item], qb = items[3 * item + 1], qe = items[3 * item + 2];
                    R = (qe - qb) * G;
                    const int sb = p.chunk_seg_off[c], nseg = p.chunk_seg_off[c + 1] - sb;
                    cq0 = p.chunk_q_off[c] + qb;
                    const int T = p.chunk_tokens[c];
                    ntiles = (T + kTileTok - 1) / kTileTok;
    #pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = lane + 32 * k;
                        qrow[k] = r < R ? p.chunk_q[cq0 + r / G] * Hq + r % G : 0;
                    }
                    if (i == 0) {
                        issue_q(h, 0);
                        q_issued = true;
                    }
                    if (iseq >= 2 &&
                        !__all_sync(0xffffffffu, tc::mbar_wait(bar(kBarSegEmpty + sbuf), ((iseq - 2) >> 1) & 1))) {
                        if (!*err) *err = 203;
                        break;
                    }
                    int32_t *tab = seg_tab(sbuf);
                    uint4 *s_rmask = reinterpret_cast<uint4 *>(tab + 3 * kMaxSegsPerChunk);
                    const uint4 *item_rm = rmask + rmask_off[item];
                    for (int s = lane; s < nseg; s += 32) {
                        const int pgb = a.node_page_off[p.seg_node[sb + s]];
                        const int tb = p.seg_tok_begin[sb + s];
                        tab[s] = p.seg_chunk_pos[sb + s];
                        tab[kMaxSegsPerChunk + s] = pgb;
                        tab[2 * kMaxSegsPerChunk + s] = tb;
                        // The producers' first page-table reads for this segment.
                        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a.page_id + pgb + tb / kPageSize));
                        s_rmask[s] = item_rm[s];
                    }
                    if (lane == 0)
                        iinfo[sbuf] = ItemInfo{nseg, T, {0, 0}};
                    __syncwarp();
                    tc::mbar_arrive(bar(kBarSegFull + sbuf));
                }
                if (!q_issued) {
                    // Q^T buffer i % QB, once unit i - QB's last S has read it.
                    const int qb = i % L::QB;
                    bool okw = i < 2 || tc::mbar_wait(bar(kBarUEmpty + ub), ((i - 2) >> 1) & 1);
                    okw = okw && (i < L::QB || tc::mbar_wait(bar(qfree_bar(qb)), ((i - L::QB) / L::QB) & 1));
                    if (!__all_sync(0xffffffffu, okw)) {
                        if (!*err) *err = 204;
                        break;
                    }
                    issue_q(h, qb);
                }
                cp_async_wait<0>();
                tc::fence_proxy_async();
                if (lane == 0)
                    uinfo[ub] = UnitInfo{R, cq0, h, ntiles, {0, 0, 0, 0}};
                __syncwarp();
                tc::mbar_arrive(bar(kBarUFull + ub));
                // Warm L2 with the rows of the item's next KV head, likely this
                // CTA's next unit (the queue hands out units in order).
                if (h + 1 < Hkv)
                    prefetch_q(h + 1);
            }
        } else if (warp == 8 || warp == 10) {
            // ---------------- producers (warp 8: K, warp 10: V) ----------------
            const int kv = warp == 8 ? 0 : 1;
            const int NS = kv ? VST : 2;   // stages of this operand
            const __nv_bfloat16 *src_base = reinterpret_cast<const __nv_bfloat16 *>(kv ? a.v_pages : a.k_pages);
            const CUtensorMap *tm = kv ? &maps.v1 : &maps.k1;
            const CUtensorMap *tm8 = kv ? &maps.v8 : &maps.k8;
            const uint64_t kv_pol = tc::l2_kv_policy(a.kv_once != 0);
            // One tile's resolution: rows lane + 32k (k < 4) and pages 0..7.
            struct Res {
                int seg[4], tok[4], pid[4];   // per row; pid only for ragged rows
                int page_y;                   // lane < 8: page id of page `lane` when it goes by TMA
                uint32_t tma_pages;
            };
            const int32_t *s_pos = nullptr, *s_pgb = nullptr, *s_tb = nullptr;
            const uint4 *s_rmask = nullptr;
            int T = 0, nseg = 0;
            // Segment of the current tile's first token: tiles go in order, so
            // it only moves forward (reset to 0 at each unit's first tile).
            int cur = 0;
            auto resolve = [&](int t, Res &r) {
                const int p0 = t * kTileTok;
                if (t == 0)
                    cur = 0;
                while (cur + 1 < nseg && s_pos[cur + 1] <= p0)
                    ++cur;
                const int sga = cur;
                const int tka = s_tb[sga] + p0 - s_pos[sga];
                const int send = sga + 1 < nseg ? s_pos[sga + 1] : T;   // segment sga ends before send
                if (T - p0 >= kTileTok && (tka % kPageSize) == 0 && send >= p0 + kTileTok) {
                    // Fast path: eight whole pages of one segment.
    #pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        r.seg[k] = sga;
                        r.tok[k] = tka + lane + 32 * k;
                        r.pid[k] = -1;
                    }
                    r.tma_pages = 0xffu;
                    r.page_y = lane < 8 ? a.page_id[s_pgb[sga] + tka / kPageSize + lane] : -1;
                    return;
                }
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int pos = t * kTileTok + lane + 32 * k;
                    r.seg[k] = -1;
                    r.tok[k] = 1;
                    if (pos < T) {
                        int lo = sga, hi = nseg - 1;
                        while (lo < hi) {
                            const int mid = (lo + hi + 1) >> 1;
                            if (s_pos[mid] <= pos)
                                lo = mid;
                            else
                                hi = mid - 1;
                        }
                        r.seg[k] = lo;
                        r.tok[k] = s_tb[lo] + pos - s_pos[lo];
                    }
                }
                uint32_t tp = 0;
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int s_first = __shfl_sync(0xffffffffu, r.seg[k], lane & 16);
                    const int t_first = __shfl_sync(0xffffffffu, r.tok[k], lane & 16);
                    const bool ok = r.seg[k] >= 0 && r.seg[k] == s_first && (t_first % kPageSize) == 0;
                    const uint32_t bal = __ballot_sync(0xffffffffu, ok);
                    if ((bal & 0xffffu) == 0xffffu)
                        tp |= 1u << (2 * k);
                    if ((bal >> 16) == 0xffffu)
                        tp |= 1u << (2 * k + 1);
                }
                r.tma_pages = tp;
                // Page ids: one load per TMA page (lanes 0-7), one per ragged row.
                int pseg = -1, ptok = 0;
    #pragma unroll
                for (int pg = 0; pg < 8; ++pg) {
                    const int sg = __shfl_sync(0xffffffffu, r.seg[pg >> 1], 16 * (pg & 1));
                    const int tk = __shfl_sync(0xffffffffu, r.tok[pg >> 1], 16 * (pg & 1));
                    if (lane == pg) {
                        pseg = sg;
                        ptok = tk;
                    }
                }
                r.page_y = -1;
                if (lane < 8 && ((tp >> lane) & 1u))
                    r.page_y = a.page_id[s_pgb[pseg] + ptok / kPageSize];
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    r.pid[k] = -1;
                    if (r.seg[k] >= 0 && !((tp >> ((lane + 32 * k) >> 4)) & 1u))
                        r.pid[k] = a.page_id[s_pgb[r.seg[k]] + r.tok[k] / kPageSize];
                }
            };
            int iseq = -1, prev_item = -1, gseq = 0, sbuf = 0;
            int st = 0;          // stage of tile gseq (gseq % NS)
            uint32_t wrap = 0;   // parity of gseq / NS
            bool ok = true;
            for (int i = 0; ok; ++i) {
                // The next unit number from the metadata warp (-1: no more).
                const int qslot = i % UQ;
                if (!__all_sync(0xffffffffu, tc::mbar_wait(bar(kBarQFull + qslot), (i / UQ) & 1))) {
                    if (!*err) *err = 205;
                    break;
                }
                const int u = useq[qslot];
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(bar(kBarQEmpty + qslot));
                const int item = u < 0 ? -1 : u / Hkv;
                if (u < 0 || item != prev_item) {
                    // Release the previous item's segment table, then wait for this one's.
                    if (prev_item >= 0) {
                        __syncwarp();
                        tc::mbar_arrive(bar(kBarSegEmpty + sbuf));
                    }
                    if (u < 0)
                        break;
                    prev_item = item;
                    ++iseq;
                    sbuf = iseq & 1;
                    if (!__all_sync(0xffffffffu, tc::mbar_wait(bar(kBarSegFull + sbuf), (iseq >> 1) & 1))) {
                        if (!*err) *err = 206;
                        break;
                    }
                }
                const int h = u - item * Hkv;
                const int32_t *tab = seg_tab(sbuf);
                s_pos = tab;
                s_pgb = tab + kMaxSegsPerChunk;
                s_tb = tab + 2 * kMaxSegsPerChunk;
                s_rmask = reinterpret_cast<const uint4 *>(tab + 3 * kMaxSegsPerChunk);
                const ItemInfo ii = iinfo[sbuf];
                T = ii.T;
                nseg = ii.nseg;
                const int ntiles = (T + kTileTok - 1) / kTileTok;
                Res res;
                resolve(0, res);
                for (int t = 0; t < ntiles; ++t, ++gseq) {
                    if (gseq >= NS) {
                        const bool okw = __all_sync(
                            0xffffffffu, tc::mbar_wait(bar((kv ? kBarEmptyV : kBarEmptyK) + st), wrap ^ 1u));
                        if (!okw) {
                            if (!*err) *err = 207;
                            ok = false;
                            break;
                        }
                    }
                    if (kv == 0) {
    #pragma unroll
                        for (int k = 0; k < 4; ++k)
                            meta[(gseq & 3) * kTileTok + lane + 32 * k] =
                                res.seg[k] >= 0 ? s_rmask[res.seg[k]] : make_uint4(0, 0, 0, 0);
                    }
                    const uint32_t full = bar((kv ? kBarFullV : kBarFullK) + st);
                    const uint32_t dst = base + (kv ? L::v_off : L::k_off) + (uint32_t)st * kTileBytes;
                    // Lane 0's arrival releases the row masks of the whole
                    // warp (the lanes' own arrivals below may be deferred).
                    __syncwarp();
                    if (lane == 0)
                        tc::mbar_arrive_expect_tx(full, __popc(res.tma_pages) * kPageBytes);
                    __syncwarp();
                    // Eight whole, consecutive pages: one box; else one box a page.
                    bool run8 = false;
                    const int pg0 = __shfl_sync(0xffffffffu, res.page_y, 0);
                    if (res.tma_pages == 0xffu)
                        run8 = __all_sync(0xffffffffu, lane >= 8 || res.page_y == pg0 + lane);
                    if (run8) {
                        if (lane == 0)
                            tc::tma_load_5d(dst, tm8, 0, 0, 0, 2 * h, pg0, full, kv_pol);
                    } else if (res.page_y >= 0) {
                        tc::tma_load_5d(dst + (uint32_t)lane * kPageBytes, tm, 0, 0, 0, 2 * h, res.page_y, full,
                                        kv_pol);
                    }
                    // Ragged rows: two rows per warp step, 16 lanes (16-byte chunks) each.
                    bool any_cp = false;
                    const __nv_bfloat16 *src0 = src_base + (lane & 15) * 8;
                    const uint32_t dst0 = dst + ((lane & 15) >> 3) * 1024u;
    #pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t nb = __ballot_sync(0xffffffffu, res.pid[k] >= 0);
                        any_cp |= nb != 0;
                        while (nb) {
                            const int l0 = __ffs(nb) - 1;
                            nb &= nb - 1;
                            int l1 = -1;
                            if (nb) {
                                l1 = __ffs(nb) - 1;
                                nb &= nb - 1;
                            }
                            const int mine = lane < 16 ? l0 : l1;
                            const int p0 = __shfl_sync(0xffffffffu, res.pid[k], l0);
                            const int t0 = __shfl_sync(0xffffffffu, res.tok[k], l0);
                            const int p1 = __shfl_sync(0xffffffffu, res.pid[k], l1 < 0 ? l0 : l1);
                            const int t1 = __shfl_sync(0xffffffffu, res.tok[k], l1 < 0 ? l0 : l1);
                            if (mine >= 0) {
                                const int row = mine + 32 * k;
                                const int pg = lane < 16 ? p0 : p1;
                                const int tk = lane < 16 ? t0 : t1;
                                const long long o = (((long long)pg * Hkv + h) * kPageSize + (tk % kPageSize)) * kD;
                                const int ch = lane & 7;
                                cp_async_16(dst0 + (uint32_t)(row >> 3) * kRowGroup + (row & 7) * 128 +
                                                ((ch ^ (row & 7)) << 4),
                                            src0 + o);
                            }
                        }
                    }
                    // With ragged rows, each lane's arrival waits for its own
                    // copies to land (the producer goes on with the next
                    // tile meanwhile); the MMA issuer makes them visible to
                    // the tensor core with a proxy fence after its wait.
                    if (any_cp)
                        cp_async_mbar_arrive_noinc(full);
                    else
                        tc::mbar_arrive(full);
                    if (++st == NS) {
                        st = 0;
                        wrap ^= 1u;
                    }
                    if (t + 1 < ntiles)
                        resolve(t + 1, res);
                }
            }
            cp_async_wait<0>();
            // Do not leave while a TMA copy of ours may still be landing.
            for (int s2 = 0; s2 < NS && s2 < gseq; ++s2) {
                const int last = gseq - 1 - ((gseq - 1 - s2) % NS);
                tc::mbar_wait(bar((kv ? kBarFullV : kBarFullK) + s2), (last / NS) & 1);
            }
        } else if (warp == 9) {
            // ---------------- MMA issue ----------------
            if (lane == 0) {
                const uint32_t idesc_s = tc::idesc_bf16(128, RP, 0, 0);
                const uint32_t idesc_o = tc::idesc_bf16(128, RP, 1, 1);
                // Descriptors of k-step 0; step s adds an address offset (16-byte units).
                const uint64_t dq = tc::smem_desc(base + L::q_off, 16, 1024);
                const uint64_t dp = tc::smem_desc(base + L::p_off, kHalf, 1024);
                // K: K-major, 8-token groups kRowGroup apart; V: MN-major, its
                // d halves 1 KB apart and its 8-token groups kRowGroup apart.
                const uint64_t dk0 = tc::smem_desc(base + L::k_off, 16, kRowGroup);
                const uint64_t dv0 = tc::smem_desc(base + L::v_off, 1024, kRowGroup);
                constexpr uint64_t kStageStep = kTileBytes >> 4;   // descriptor address units
                int nunits = 0x7fffffff;   // known once the end mark is read
                // S cursor: unit is, its tile ts (nts tiles, -1 before its
                // description is read), CTA tile gs.  P.V cursor: ip, tp, gp.
                int is = 0, ts = 0, nts = -1, gs = 0;
                int ip = 0, tp = 0, gp = 0;
                int ntq0 = 0, ntq1 = 0;   // tiles of the units in flight, by unit parity
                bool ok = true;
                uint32_t polls = 0;
                while (ip < nunits && ok) {
                    bool progressed = false;
                    // S(gs): needs the unit's Q^T, K(gs) and S buffer gs % 2
                    // released by tile gs - 2; at most one tile ahead of P.V.
                    if (is < nunits && gs <= gp + 1) {
                        if (nts < 0 && tc::mbar_test(bar(kBarUFull + (is & 1)), (is >> 1) & 1)) {
                            nts = uinfo[is & 1].ntiles;
                            if (nts < 0)
                                nunits = is;   // no more units
                            if (is & 1)
                                ntq1 = nts;
                            else
                                ntq0 = nts;
                            tc::mbar_arrive(bar(kBarUEmpty + (is & 1)));
                        }
                        const int st = gs & 1, b = gs & 1;
                        if (nts > 0 && tc::mbar_test(bar(kBarFullK + st), (gs >> 1) & 1) &&
                            (gs < 2 || tc::mbar_test(bar(kBarSFree + b), ((gs - 2) >> 1) & 1))) {
                            tc::fence_after_sync();
                            tc::fence_proxy_async();   // ragged rows came by cp.async (generic proxy)
                            const uint32_t d_s = tmem + (uint32_t)(b * 128);
    #pragma unroll
                            for (int s = 0; s < 8; ++s) {
                                const uint64_t ko = (uint64_t)(((s >> 2) * 1024 + (s & 3) * 32) >> 4);
                                const uint64_t qo = (uint64_t)(((is % L::QB) * 2 * L::q_half + (s >> 2) * L::q_half +
                                                                (s & 3) * 32) >> 4);
                                tc::mma_bf16(d_s, dk0 + (uint64_t)st * kStageStep + ko, dq + qo, idesc_s, s > 0 ? 1u : 0u);
                            }
                            tc::mma_commit(bar(kBarSFull + b));
                            tc::mma_commit(bar(kBarEmptyK + st));
                            ++gs;
                            if (++ts == nts) {
                                tc::mma_commit(bar(qfree_bar(is % L::QB)));
                                ++is;
                                ts = 0;
                                nts = -1;
                            }
                            progressed = true;
                        }
                    }
                    // P.V(gp): needs V(gp), P(gp) and, for a unit's first tile,
                    // its O buffer read out by the epilogue of the unit two back.
                    if (gp < gs) {
                        const int stp = gp % VST, ob = ip & 1;
                        if (tc::mbar_test(bar(kBarFullV + stp), (gp / VST) & 1) &&
                            tc::mbar_test(bar(kBarPFull), gp & 1) &&
                            (tp > 0 || ip < 2 || tc::mbar_test(bar(kBarOFree + ob), ((ip - 2) >> 1) & 1))) {
                            tc::fence_after_sync();
                            tc::fence_proxy_async();
                            const uint32_t d_o = tmem + 256 + (uint32_t)(ob * 128);
    #pragma unroll
                            for (int s = 0; s < 8; ++s) {
                                // k-step s: tokens 16 s .. 16 s + 15 (two groups of V, 2 KB of P^T).
                                const uint64_t sv = (uint64_t)((s * 2 * kRowGroup) >> 4);
                                const uint64_t sp = (uint64_t)((s * 2048) >> 4);
                                tc::mma_bf16(d_o, dv0 + (uint64_t)stp * kStageStep + sv, dp + sp, idesc_o,
                                             (tp > 0 || s > 0) ? 1u : 0u);
                            }
                            tc::mma_commit(bar(kBarPvDone));
                            tc::mma_commit(bar(kBarEmptyV + stp));
                            ++gp;
                            if (++tp == ((ip & 1) ? ntq1 : ntq0)) {
                                tc::mma_commit(bar(kBarOFull + ob));   // the unit's O is complete
                                ++ip;
                                tp = 0;
                            }
                            progressed = true;
                        }
                    }
                    // An idle pass naps briefly: a lane spinning at full rate
                    // takes issue slots from the softmax warps that share its
                    // scheduler (speculative forest 128.1 -> 126.2 us).
                    if (progressed)
                        polls = 0;
                    else if (++polls > (1u << 24))
                        ok = false;
                    else
                        __nanosleep(32);
                }
                if (!ok)
                    if (!*err) *err = 208;
            }
        } else if (warp >= 12) {
            // ---------------- epilogue warpgroup ----------------
            // Per unit, once both softmax warpgroups have handed over their
            // column sums: O^T / l from TMEM buffer ob into the fp32 partials
            // (thread je owns head dim je, the TMEM lane of its warp quarter),
            // then the buffer is free for the unit two on.
            const int je = tid - 384;
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            // One thread waits on each mbarrier and the named barrier
            // releases the others, so that 128 spinning threads do not take
            // issue slots from the softmax warps on the same schedulers.
            for (int i = 0;; ++i) {
                const int ob = i & 1;
                const bool okw = je != 0 || tc::mbar_wait(bar(kBarEpiFull + ob), (i >> 1) & 1);
                if (tc::named_sync_or(3, 128, !okw)) {
                    if (!*err) *err = 211;
                    break;
                }
                tc::fence_after_sync();
                const int R = epi_info[ob * 4];
                if (R == -1)
                    break;
                if (R >= 0) {
                    // The unit's last P.V (the softmax warpgroups do not wait for it).
                    const bool okf = je != 0 || tc::mbar_wait(bar(kBarOFull + ob), (i >> 1) & 1);
                    if (tc::named_sync_or(3, 128, !okf)) {
                        if (!*err) *err = 213;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t tmem_ob = tmem + 256 + (uint32_t)(ob * 128) + lane_off;
    #pragma unroll
                    for (int w = 0; w < 2; ++w) {
                        const int rows_w = w == 0 ? (R < NPH ? R : NPH) : (R > NPH ? R - NPH : 0);
                        if (epi_info[ob * 4 + 1 + w])
                            continue;
                        const float *linv_e = epi + (ob * 2 + w) * 128;
                        const int32_t *orow_e = reinterpret_cast<const int32_t *>(linv_e + 64);
    #pragma unroll
                        for (int g = 0; g < NPH; g += 16) {
                            if (g >= rows_w)
                                break;
                            float o[16];
                            tc::tmem_ld16(tmem_ob + (uint32_t)(w * NPH + g), o);
    #pragma unroll
                            for (int c2 = 0; c2 < 16; ++c2) {
                                const int cc = g + c2;
                                if (cc < rows_w)
                                    a.o_part[(size_t)orow_e[cc] * kD + je] = o[c2] * linv_e[cc];
                            }
                        }
                    }
                }
                tc::fence_before_sync();
                tc::named_sync(3, 128);
                if (je == 0)
                    tc::mbar_arrive(bar(kBarOFree + ob));
                if (R < 0)
                    break;
            }
    }
    } else {
        tc::setmaxnreg_inc<kRegsSoftmax>();
        // ---------------- softmax warpgroups ----------------
        // Warpgroup w owns columns [w*NPH, w*NPH + NPH) of S^T and O^T.
        const int w = warp >> 2, wt = warp & 3, j = tid & 127;
        const uint32_t nb_id = 1 + (uint32_t)w;
        float *m_s = stat + w * 256, *alpha_s = m_s + 64;
        float *redw = red + w * 256;
        const uint32_t lane_off = (uint32_t)(wt * 32) << 16;
        const uint32_t col0 = (uint32_t)(w * NPH);
        uint8_t *prow_ptr = smem + L::p_off + (j >> 3) * 1024 + (j & 7) * 128;
        const float sc = a.scale_log2;
        constexpr float kSlack = 8.f;   // rescale only when 2^(s - m) would exceed 2^8
        auto load_cols = [&](uint32_t taddr, float *v) {
#pragma unroll
            for (int g = 0; g + 32 <= NPH; g += 32) {
                float tmp[32];
                tc::tmem_ld32(taddr + g, tmp);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[g + i] = tmp[i];
            }
            if constexpr (NPH % 32 != 0)
                tc::tmem_ld16(taddr + (NPH & ~31), v + (NPH & ~31));
        };
        auto tile_max_to_smem = [&](const float *v) {
#pragma unroll
            for (int g = 0; g < NPH; g += 32) {
                float tmp[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    tmp[i] = (g + i < NPH) ? v[g + i] : -INFINITY;
                redw[wt * 64 + g + lane] = reduce_scatter32<true>(tmp, lane);
            }
        };
        // Tells the epilogue warpgroup that no unit follows (R = -1) or that
        // this one failed and none follows (R = -2), at unit index i: first
        // waits until the epilogue has read unit i - 2 out of buffer ob (a
        // real unit is held back by its P.V; this mark is not), so that the
        // mark neither overwrites that unit's description nor completes a
        // second phase of the buffer's barrier ahead of the epilogue.
        auto end_epilogue = [&](int i, int code) {
            const int ob = i & 1;
            if (j == 0) {
                if (i >= 2 && !tc::mbar_wait(bar(kBarOFree + ob), ((i - 2) >> 1) & 1))
                    if (!*err) *err = 212;
                if (w == 0)
                    epi_info[ob * 4] = code;
                tc::mbar_arrive(bar(kBarEpiFull + ob));
            }
        };
        int gseq = 0;
        // Unit -1 is a dry run of one tile (and, at 32 columns, a unit's
        // end), made while the first tile loads: it runs the same
        // instructions on whatever TMEM and shared memory hold, with no
        // waits, signals or global stores, so that the instruction fetches
        // of this code are not paid again on the real first tile.
        for (int i = -1;; ++i) {
            const bool dry = i < 0;
            const int ub = i & 1, ob = i & 1;
            const bool okw = dry || tc::mbar_wait(bar(kBarUFull + ub), (i >> 1) & 1);
            if (tc::named_sync_or(nb_id, 128, !okw)) {
                if (!*err) *err = 209;
                end_epilogue(i, -2);
                break;
            }
            const UnitInfo ui = dry ? UnitInfo{2 * NPH, 0, 0, 1, {0, 0, 0, 0}} : uinfo[ub];
            tc::named_sync(nb_id, 128);
            if (ui.ntiles < 0) {
                end_epilogue(i, -1);   // no more units
                break;
            }
            if (j == 0 && !dry)
                tc::mbar_arrive(bar(kBarUEmpty + ub));
            const int R = ui.R, ntiles = ui.ntiles;
            const int rows_w = w == 0 ? (R < NPH ? R : NPH) : (R > NPH ? R - NPH : 0);
            const uint32_t tmem_o = tmem + 256 + (uint32_t)(ob * 128) + lane_off + col0;
            float l[NPH];
#pragma unroll
            for (int c2 = 0; c2 < NPH; ++c2)
                l[c2] = 0.f;
            if (j < 64) {
                m_s[j] = -INFINITY;
                alpha_s[j] = 1.f;
            }
            tc::named_sync(nb_id, 128);
            bool ok = true;
            for (int t = 0; t < ntiles; ++t, ++gseq) {
                const int b = gseq & 1;
                ok = dry || tc::mbar_wait(bar(kBarSFull + b), (gseq >> 1) & 1);
                tc::fence_after_sync();
                float s[NPH];
                load_cols(tmem + (uint32_t)(b * 128) + lane_off + col0, s);
                const uint4 mk = meta[(gseq & 3) * kTileTok + j];
                const uint32_t mw0 = w == 0 ? mk.x : mk.z, mw1 = w == 0 ? mk.y : mk.w;
#pragma unroll
                for (int c2 = 0; c2 < NPH; ++c2) {
                    const uint32_t mword = c2 < 32 ? mw0 : mw1;
                    s[c2] = ((mword >> (c2 & 31)) & 1u) ? s[c2] * sc : -INFINITY;
                }
                tc::fence_before_sync();
                bool slow = t == 0;
                if (t > 0) {
                    bool flag = false;
#pragma unroll
                    for (int c2 = 0; c2 < NPH; c2 += 4) {
                        const float4 m4 = *reinterpret_cast<const float4 *>(m_s + c2);
                        flag |= (s[c2] > m4.x + kSlack) | (s[c2 + 1] > m4.y + kSlack) |
                                (s[c2 + 2] > m4.z + kSlack) | (s[c2 + 3] > m4.w + kSlack);
                    }
                    if (tc::named_sync_or(nb_id, 128, flag || !ok)) {
                        if (tc::named_sync_or(nb_id, 128, !ok)) {
                            ok = false;
                            break;
                        }
                        slow = true;
                    }
                }
                if (slow) {
                    tile_max_to_smem(s);
                    if (tc::named_sync_or(nb_id, 128, !ok)) {
                        ok = false;
                        break;
                    }
                    if (j < NPH) {
                        const float mt = fmaxf(fmaxf(redw[j], redw[64 + j]), fmaxf(redw[128 + j], redw[192 + j]));
                        const float mo = m_s[j];
                        const float mn = fmaxf(mo, mt);
                        alpha_s[j] = mn == -INFINITY ? 1.f : tc::ex2(mo - mn);
                        m_s[j] = mn;
                    }
                    tc::named_sync(nb_id, 128);
                }
                if (j == 0 && !dry)
                    tc::mbar_arrive(bar(kBarSFree + b));
                // P (one buffer) may be rewritten once the previous tile's
                // P.V is done; that P.V also finishes O before a rescale.
                bool ok2 = true;
                if (gseq >= 1) {
                    ok2 = tc::mbar_wait(bar(kBarPvDone), (gseq - 1) & 1);
                    tc::fence_after_sync();
                }
                if (slow && t >= 1) {
#pragma unroll
                    for (int g = 0; g < NPH; g += 16) {
                        float o[16];
                        tc::tmem_ld16(tmem_o + g, o);
#pragma unroll
                        for (int c2 = 0; c2 < 16; ++c2) {
                            o[c2] *= alpha_s[g + c2];
                            l[g + c2] *= alpha_s[g + c2];
                        }
                        tc::tmem_st16(tmem_o + g, o);
                    }
                }
                // Probabilities: fp32 column sums, bf16 P^T (MN-major: token
                // row j holds the columns, 16-byte chunks swizzled by j % 8).
#pragma unroll
                for (int ch = 0; ch < NPH / 8; ++ch) {
                    const float4 ma = *reinterpret_cast<const float4 *>(m_s + 8 * ch);
                    const float4 mb = *reinterpret_cast<const float4 *>(m_s + 8 * ch + 4);
                    const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
                    float pv[8];
#pragma unroll
                    for (int c2 = 0; c2 < 8; ++c2) {
                        const float x = s[8 * ch + c2];
                        pv[c2] = x == -INFINITY ? 0.f : tc::ex2(x - mm[c2]);
                        l[8 * ch + c2] += pv[c2];
                    }
                    uint4 packed;
                    packed.x = tc::pack_bf16x2(pv[0], pv[1]);
                    packed.y = tc::pack_bf16x2(pv[2], pv[3]);
                    packed.z = tc::pack_bf16x2(pv[4], pv[5]);
                    packed.w = tc::pack_bf16x2(pv[6], pv[7]);
                    const int q8 = (int)(col0 >> 3) + ch;   // global 8-column chunk
                    *reinterpret_cast<uint4 *>(prow_ptr + (q8 >> 3) * kHalf + (((q8 & 7) ^ (j & 7)) << 4)) = packed;
                }
                tc::fence_proxy_async();
                tc::fence_before_sync();
                if (tc::named_sync_or(nb_id, 128, !ok2)) {
                    ok = false;
                    break;
                }
                if (j == 0 && !dry)
                    tc::mbar_arrive(bar(kBarPFull));
            }
            // At 16 columns the dry run stops here: the unit-end code's
            // first fetch then overlaps the first unit's last tiles, which
            // measured faster than fetching it before the first tile (few-
            // shot tree 49.4 -> 48.4 us); at 32 columns the full dry unit
            // measured faster (speculative forest 132.2 -> 130.8 us).
            if (dry && NPH == 16) {
                gseq = 0;
                continue;
            }
            // 1 / l and the rows for the epilogue warpgroup, which waits for
            // the unit's last P.V itself: the column sums are this
            // warpgroup's own, so it goes on to the next unit meanwhile.
            if (!ok)
                if (!*err) *err = 210;
            const bool failed = tc::named_sync_or(nb_id, 128, !ok || *err != 0);
#pragma unroll
            for (int g = 0; g < NPH; g += 32) {
                float tmp[32];
#pragma unroll
                for (int c2 = 0; c2 < 32; ++c2)
                    tmp[c2] = (g + c2 < NPH) ? l[g + c2] : 0.f;
                redw[wt * 64 + g + lane] = reduce_scatter32<false>(tmp, lane);
            }
            tc::named_sync(nb_id, 128);
            // Column sums and partial rows for the epilogue warpgroup, which
            // reads O (buffer ob) out of TMEM; the lse partials go out here.
            float *linv_e = epi + (ob * 2 + w) * 128;
            int32_t *orow_e = reinterpret_cast<int32_t *>(linv_e + 64);
            if (j < NPH) {
                const float li = 1.f / (redw[j] + redw[64 + j] + redw[128 + j] + redw[192 + j]);
                const int r = w * NPH + j;
                const int orow = (ui.cq0 + r / G) * Hq + ui.h * G + (r % G);
                linv_e[j] = li;
                orow_e[j] = orow;
                if (j < rows_w && !failed && !dry)
                    a.lse_part[orow] = m_s[j] - log2f(li);
            }
            if (j == 0 && !dry) {
                epi_info[ob * 4 + 1 + w] = failed ? 1 : 0;
                if (w == 0)
                    epi_info[ob * 4] = failed ? -2 : R;
            }
            tc::named_sync(nb_id, 128);
            if (j == 0 && !dry)
                tc::mbar_arrive(bar(kBarEpiFull + ob));
            if (dry) {
                gseq = 0;
            }
            if (failed)
                break;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (*err && tid < 128) {
        // A wait ran out: record it in the partition's status word and mark
        // every partial of the launch as failed (the merged output then
        // shows it); the units are not tracked per CTA.
        if (tid == 0)
            report_failure(p.status, *err);
        for (int u = 0; u < n_units; ++u) {
            const int item = u / Hkv, h = u - item * Hkv;
            const int c = items[3 * item], qb = items[3 * item + 1], qe = items[3 * item + 2];
            const int cq0 = p.chunk_q_off[c] + qb;
            for (int r = 0; r < (qe - qb) * G; ++r) {
                const size_t prw = (size_t)(cq0 + r / G) * Hq + h * G + (r % G);
                a.o_part[prw * kD + tid] = __int_as_float(0x7fc00000);
                if (tid == 0)
                    a.lse_part[prw] = __int_as_float(0x7fc00000);
            }
        }
    }
    if (warp == 9)
        tc::tmem_dealloc(tmem, kTmemCols);
    if (tid == 0) {
        // The CTA that counted itself last waits, before it exits, for the
        // launch before this one: the grid completes only after that one
        // has, while the other CTAs leave their SMs at once.
        if (!qdone[0])
            queue_done(queue, qdone);
        if (qdone[1])
            grid_dep_wait();
    }
}

// ---- host: tensor maps over the paged KV ----
PFN_cuTensorMapEncodeTiled_v12000 get_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Encodes the *1 (run8 = false) or *8 view of a page pool.
bool encode_pool_map(const void *ptr, int32_t pages, int32_t hkv, bool run8, CUtensorMap *m)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encoder();
    if (!enc)
        return false;
    static_assert(kPageSize == 16 && kD == 128, "a page is two groups of 8 tokens x 128 dims");
    const cuuint64_t row = (cuuint64_t)kD * 2;
    const cuuint64_t dims[5] = {64, 8, 2, 2 * (cuuint64_t)hkv, (cuuint64_t)pages};
    const cuuint64_t strides[4] = {row, 128, 8 * row, row * kPageSize * hkv};
    const cuuint32_t box[5] = {64, 8, 2, 2, run8 ? 8u : 1u};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The four maps of (k, v, pages, hkv), cached per host thread for the last
// pools seen.
bool kv_maps(const void *k, const void *v, int32_t pages, int32_t hkv, KvMaps *out)
{
    struct Cache {
        const void *k = nullptr, *v = nullptr;
        int32_t pages = 0, hkv = 0;
        KvMaps maps;
    };
    thread_local Cache c;
    if (c.k != k || c.v != v || c.pages != pages || c.hkv != hkv) {
        KvMaps m;
        if (!encode_pool_map(k, pages, hkv, false, &m.k1) || !encode_pool_map(v, pages, hkv, false, &m.v1) ||
            !encode_pool_map(k, pages, hkv, true, &m.k8) || !encode_pool_map(v, pages, hkv, true, &m.v8))
            return false;
        c.k = k;
        c.v = v;
        c.pages = pages;
        c.hkv = hkv;
        c.maps = m;
    }
    *out = c.maps;
    return true;
}

template <int NPH>
int launch_cols(const AttnArgs &a, const DevPartition &p, const int32_t *items, const uint32_t *rmask,
                const int32_t *rmask_off, int32_t n, uint32_t *queue, LaunchShape sh, const KvMaps &maps,
                cudaStream_t st)
{
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(phase1_mma_kernel<NPH>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Smem<NPH>::alloc);
        if (e != cudaSuccess)
            return (int)e;
        configured = true;
    }
    const int32_t units = n * a.num_kv_heads;
    const int32_t grid = sh.grid < units ? sh.grid : units;
    const int32_t early = sh.early < grid ? sh.early : grid;
    return (int)launch_dependent(phase1_mma_kernel<NPH>, dim3(grid), dim3(kThreadsMma), Smem<NPH>::alloc, st, a, p,
                                 items, reinterpret_cast<const uint4 *>(rmask), rmask_off, units,
                                 static_block(units, early, sh.block), early, queue, maps);
}

}  // namespace

bool mma_supported(int32_t head_dim) { return head_dim == kD; }

int launch_phase1_mma(const AttnArgs &a, const DevPartition &p, const int32_t *items, const uint32_t *rmask,
                      const int32_t *rmask_off, int32_t n, int bucket, uint32_t *queue, LaunchShape shape,
                      void *stream)
{
    if (n <= 0)
        return 0;
    if ((int64_t)n * a.num_kv_heads > INT32_MAX || !queue || shape.grid < 1 || shape.early < 1)
        return (int)cudaErrorInvalidValue;
    KvMaps maps;
    if (!kv_maps(a.k_pages, a.v_pages, a.num_pages, a.num_kv_heads, &maps))
        return (int)cudaErrorInvalidValue;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (bucket) {
    case 0: return launch_cols<16>(a, p, items, rmask, rmask_off, n, queue, shape, maps, st);
    case 1: return launch_cols<32>(a, p, items, rmask, rmask_off, n, queue, shape, maps, st);
    default: return (int)cudaErrorInvalidValue;   // items have at most kMmaMaxRows = 64 rows
    }
}

}  // namespace deft
