// phase1_fma.cu -- phase-1 partial attention on CUDA cores, for work items
// with fewer than 16 rows (rows = queries of the item x GQA group).
//
// What a work unit (item = chunk + query range, one KV head h) computes
// (DeFT Guide, "Deep Dive": tree-constrained attention and online-softmax
// tile accumulation; DeFT abstract: KV-Guided Grouping): for the unit's rows
// r (query k, group member g, query head h*G+g), over the chunk's tokens j
// whose segment bitmask contains the row's query,
//     s_rj = (q_r . k_j) * scale,  o_r = softmax_j(s_r) . v,  L_r = lse(s_r)
// stored as an fp32 partial (o_r, L_r in base 2) in the unit's slot.
// Logits are carried in base 2 (q pre-scaled by scale * log2 e).
//
// Persistent CTAs (one per SM): the launch's early CTAs, those that start
// with the step, first take a contiguous block of units (9/10 of an even
// share of the estimated cost among them; units are item-major, so the block holds runs of
// one item's KV heads, which share the item's segment table and page list);
// then every CTA takes units one at a time from the launch's work queue (an
// atomic counter), so a CTA that starts late or runs fast takes more.  Each
// compute group has its own ring of 64-token stages through which the tiles
// of its units stream continuously, so the loads of its next unit overlap
// the end of the current one and the groups never wait on each other's
// tiles.
//   warp 0            metadata: runs ahead; takes the next unit from the
//                     queue and passes its number to the copy warps through a
//                     shared-memory ring; per item it builds the segment
//                     table (positions, page bases, row masks) and gathers
//                     the item's page ids, per unit it stages the q rows
//                     (cp.async, completion signalled on the unit's
//                     mbarrier, so the warp never waits on them);
//   warps 1, 2        copies: with two groups, warp 1 + g fills group g's
//                     ring; with one, the two alternate tiles.  A copy warp
//                     resolves a tile's pages through the page list (a
//                     fast path when the tile is four whole pages of one
//                     segment), loads every 16-token slot that is one whole page
//                     of one segment as a single contiguous bulk copy (a
//                     page holds a head's 16 rows back to back) and ragged
//                     rows (node tails, one-token nodes) with 16-byte
//                     cp.async at the exact token count;
//   warps 3..         NG groups of 8 compute warps; group g takes whole units
//                     g, g+NG, ... of the CTA; a warp owns 8 tokens of a tile:
//                       q.k  lane = 8 * quarter + token: each lane dots a
//                            quarter of head_dim for every row, its 16-byte
//                            chunks rotated by the token so that the 8
//                            tokens of a shared-memory phase hit 8 different
//                            bank groups; xor-shuffles finish the dot;
//                       p.v  lane owns head_dim/32 outputs of every row.
// Stages hold K and V rows unswizzled, [64 tokens][head_dim] bf16 each.
// Every warp keeps its own running max / sum / output per row; at the end
// of a unit the group's warp states are merged through shared-memory
// atomics.
// Every wait on an mbarrier is bounded.
#include "merge.cuh"
#include "tcgen05.cuh"

namespace deft {
namespace {

constexpr int kTile = 64;   // tokens per stage
constexpr int kPageList = 512;  // page ids staged per item (larger items look pages up in global memory)

// Bytes of everything but the stage ring, for NG compute groups.
template <int D, int RMAX>
constexpr uint32_t fma_fixed_bytes(int NG)
{
    return 2 * NG * RMAX * D * 2 + 2 * NG * 32 + NG * RMAX * D * 4 + 3 * 8 * NG * RMAX * 4 + NG * 8 * (RMAX < 8 ? RMAX : 8) * D * 4 +
           2 * kMaxSegsPerChunk * 20 +
           2 * kPageList * 4 + 2 * 16 + 64 + 384 + 1024 + NG * 16 + 2 * NG * 8 + 4 * NG * RMAX * 4;
}

template <int D, int RMAX>
struct FmaCfg {
    static constexpr int NG = RMAX <= 4 ? 2 : 1;       // compute groups
    static constexpr int NCW = 8 * NG;                 // compute warps
    static constexpr int THREADS = 32 * (NCW + 4);     // + metadata, two copy and a merge warp
    // Stages in the ring: as many as fit next to the fixed buffers, at most 6
    // and even: two groups get half each; one group's ring is filled by the two
    // copy warps alternately (copy warp w always serves the stages of parity w).
    static constexpr uint32_t stage_bytes = 2 * kTile * D * 2 + kTile * 4 + 16;
    static constexpr int ST_FIT = (int)((227u * 1024u - fma_fixed_bytes<D, RMAX>(NG)) / stage_bytes);
    static constexpr int ST = (ST_FIT < 6 ? ST_FIT : 6) & ~1;
    static_assert(ST >= 4, "at least four stages");
    static constexpr int RST = ST / NG;                // stages per group ring
    static constexpr int UB = 2 * NG;                  // unit slots (q rows, description)
    static constexpr uint32_t op_bytes = kTile * D * 2;           // K (or V) of one stage
    static constexpr uint32_t stage_off = 0;                      // [stage][K,V]
    static constexpr uint32_t meta_off = ST * 2 * op_bytes;       // [stage][64] row masks
    static constexpr uint32_t qst_off = meta_off + ST * kTile * 4;            // [UB][RMAX][D] bf16
    static constexpr uint32_t info_off = qst_off + UB * RMAX * D * 2;         // [UB] unit info
    static constexpr uint32_t qs_off = info_off + UB * 32;                     // [NG][RMAX][D] f32
    static constexpr uint32_t ml_off = qs_off + NG * RMAX * D * 4;             // [3][NCW][RMAX] m, l, weight
    static constexpr int MRB = RMAX < 8 ? RMAX : 8;                            // rows per merge round
    static constexpr uint32_t obuf_off = ml_off + 3 * NCW * RMAX * 4;         // [NG][8 warps][MRB][D] f32
    static constexpr uint32_t mdesc_off = obuf_off + NG * 8 * MRB * D * 4;     // [NG] MergeDesc
    static constexpr uint32_t seg_off = mdesc_off + NG * 16;                   // [2][5][256]
    static constexpr uint32_t pl_off = seg_off + 2 * kMaxSegsPerChunk * 20;    // [2][kPageList]
    static constexpr uint32_t iinfo_off = pl_off + 2 * kPageList * 4;          // [2] ItemInfo
    // Row r's query (bit 31: its only slot) per unit slot [UB][RMAX], the
    // group's copy handed to the merge warp [NG][RMAX], and the merge warp's
    // destination row of each row [NG][RMAX].
    static constexpr uint32_t urow_off = iinfo_off + 2 * 16;
    static constexpr uint32_t mrow_off = urow_off + UB * RMAX * 4;
    static constexpr uint32_t mdst_off = mrow_off + NG * RMAX * 4;
    static constexpr uint32_t useq_off = mdst_off + NG * RMAX * 4;             // [UQ] unit numbers, error and queue flags
    static constexpr uint32_t bar_off = useq_off + 16 * 4;
    static constexpr uint32_t nbars = 2 * ST + 2 * UB + 4 + 2 * 8 + 2 * NG;
    static constexpr uint32_t total = bar_off + nbars * 8;
    static constexpr uint32_t alloc = total + 1024;
    static_assert(alloc <= 227 * 1024, "shared memory of one CTA");
};

__device__ __forceinline__ uint32_t fbar(uint32_t base, int i) { return base + 8u * (uint32_t)i; }

constexpr int kUnitQueue = 8;   // unit numbers passed from the metadata warp to the copy warps

struct UnitInfo {
    int32_t R;       // rows (-1: no more units)
    int32_t cq0;     // first slot of the unit's rows
    int32_t h;       // KV head
    int32_t ntiles;
    int32_t seq0;    // position of the unit's first tile in the CTA's tile stream
    int32_t pad[3];
};

struct ItemInfo {
    int32_t nseg;
    int32_t T;       // chunk tokens
    int32_t listed;  // 1: the item's page ids are in the shared page list
    int32_t npages;  // page-list entries of the item
};

// A compute group's states of one unit, handed to the merge warp: rows
// rb .. rb + MRB - 1 of the unit (R rows, first slot cq0, KV head h); R < 0:
// the group has finished.
struct MergeDesc {
    int32_t R, cq0, h, rb;
};

template <int D, int RMAX>
__global__ void __launch_bounds__(FmaCfg<D, RMAX>::THREADS, 1)
phase1_fma_kernel(AttnArgs a, DevPartition p, const int32_t *__restrict__ items,
                  const uint32_t *__restrict__ rmask, const int32_t *__restrict__ rmask_off,
                  const uint32_t *__restrict__ direct, int32_t n_units, int32_t static_units, int32_t early,
                  uint32_t *__restrict__ queue)
{
    using C = FmaCfg<D, RMAX>;
    constexpr int NG = C::NG, NCW = C::NCW, ST = C::ST, RST = C::RST, UB = C::UB;
    constexpr int E = D / 32;       // p.v outputs per lane
    constexpr int QCH = D / 32;     // 16-byte chunks per lane in q.k (a quarter of the row)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    uint32_t *meta = reinterpret_cast<uint32_t *>(smem + C::meta_off);
    UnitInfo *info = reinterpret_cast<UnitInfo *>(smem + C::info_off);
    const uint32_t bars = base + C::bar_off;
    // mbarriers: full[ST], empty[ST], unit_full[UB], unit_empty[UB], seg_full[2], seg_empty[2],
    // queue_full[UQ], queue_empty[UQ]
    constexpr int UQ = kUnitQueue;
    const int kFull = 0, kEmpty = ST, kUFull = 2 * ST, kUEmpty = 2 * ST + UB;
    const int kSFull = 2 * ST + 2 * UB, kSEmpty = kSFull + 2;
    const int kQFull = kSEmpty + 2, kQEmpty = kQFull + UQ;
    const int kMFull = kQEmpty + UQ, kMEmpty = kMFull + NG;   // [NG] each: states written / read

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads, G = a.gqa_group;
    ItemInfo *iinfo = reinterpret_cast<ItemInfo *>(smem + C::iinfo_off);
    volatile MergeDesc *mdesc = reinterpret_cast<volatile MergeDesc *>(smem + C::mdesc_off);
    volatile int32_t *useq = reinterpret_cast<volatile int32_t *>(smem + C::useq_off);
    int32_t *urow = reinterpret_cast<int32_t *>(smem + C::urow_off);
    int32_t *mrow = reinterpret_cast<int32_t *>(smem + C::mrow_off);
    volatile int32_t *err = useq + UQ;
    // qdone[0]: this CTA has counted itself done with the queue; qdone[1]:
    // it was the launch's last to do so.
    volatile int32_t *qdone = useq + UQ + 1;

    // Warm L2 with this CTA's share of the plan's arrays, the node page
    // offsets and q, which the metadata and copy warps walk in chains of
    // dependent loads as soon as the set-up is done.  Prefetches change no
    // data, so they go out before the wait for the stream's earlier work.
    prefetch_l2_share(p.arrays, p.array_bytes, blockIdx.x, gridDim.x, tid, C::THREADS);
    prefetch_l2_share(a.node_page_off, (size_t)(p.num_nodes + 1) * 4, blockIdx.x, gridDim.x, tid, C::THREADS);
    prefetch_l2_share(a.q, (size_t)p.num_queries * Hq * D * 2, blockIdx.x, gridDim.x, tid, C::THREADS);
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
        for (int s = 0; s < ST; ++s) {
            tc::mbar_init(fbar(bars, kFull + s), 33);
            tc::mbar_init(fbar(bars, kEmpty + s), 8);
        }
        for (int u = 0; u < UB; ++u) {
            tc::mbar_init(fbar(bars, kUFull + u), 33);   // 32 cp.async arrivals + the description
            tc::mbar_init(fbar(bars, kUEmpty + u), 8);
        }
        for (int u = 0; u < 2; ++u) {
            tc::mbar_init(fbar(bars, kSFull + u), 32);
            tc::mbar_init(fbar(bars, kSEmpty + u), 64);
        }
        for (int u = 0; u < UQ; ++u) {
            tc::mbar_init(fbar(bars, kQFull + u), 1);
            tc::mbar_init(fbar(bars, kQEmpty + u), 2);   // lane 0 of each copy warp
        }
        for (int g = 0; g < NG; ++g) {
            tc::mbar_init(fbar(bars, kMFull + g), 1);
            tc::mbar_init(fbar(bars, kMEmpty + g), 1);
        }
        *err = 0;
        qdone[0] = 0;
        qdone[1] = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------- metadata (runs ahead)
        const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(a.q);
        constexpr int QJ = (RMAX * (D / 8) + 31) / 32;   // q chunks per lane
        int qrow[QJ];   // per q chunk of this lane: query * Hq + group member, or -1
        int rseq0 = 0, rseq1 = 0;   // next tile of each group's ring
        int iseq = -1, prev_item = -1, R = 0, cq0 = 0, ntiles = 0;
        int qf = 0;   // urow entry of row `lane` of the current item
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
            // Pass it (or the end, -1) to the copy warps.
            const int qslot = i % UQ;
            if (i >= UQ &&
                !__all_sync(0xffffffffu, tc::mbar_wait(fbar(bars, kQEmpty + qslot), ((i / UQ) - 1) & 1))) {
                if (!*err) *err = 101;
                break;
            }
            if (lane == 0) {
                useq[qslot] = last ? -1 : u;
                tc::mbar_arrive(fbar(bars, kQFull + qslot));
            }
            if (last) {
                if (lane == 0)
                    queue_done(queue, qdone);
                // One end mark for each compute group (local units i .. i + NG - 1).
                for (int k = 0; k < NG; ++k) {
                    const int ub = (i + k) % UB;
                    if (i + k >= UB &&
                        !__all_sync(0xffffffffu,
                                    tc::mbar_wait(fbar(bars, kUEmpty + ub), (((i + k) - UB) / UB) & 1))) {
                        if (!*err) *err = 102;
                        break;
                    }
                    if (lane == 0)
                        info[ub].R = -1;
                    __syncwarp();
                    tc::mbar_arrive(fbar(bars, kUFull + ub));
                    if (lane == 0)
                        tc::mbar_arrive(fbar(bars, kUFull + ub));
                }
                break;
            }
            const int item = u / Hkv, h = u - item * Hkv;
            if (item != prev_item) {
                // A new item: its segment table and page list.
                prev_item = item;
                ++iseq;
                const int sbuf = iseq & 1;
                const int c = items[3 * item], qb = items[3 * item + 1], qe = items[3 * item + 2];
                R = (qe - qb) * G;
                const int sb = p.chunk_seg_off[c], nseg = p.chunk_seg_off[c + 1] - sb;
                cq0 = p.chunk_q_off[c] + qb;
                const int T = p.chunk_tokens[c];
                ntiles = (T + kTile - 1) / kTile;
#pragma unroll
                for (int j = 0; j < QJ; ++j) {
                    const int r = (lane + 32 * j) / (D / 8);
                    qrow[j] = r < R ? p.chunk_q[cq0 + r / G] * Hq + r % G : -1;
                }
                if (lane < R)
                    qf = p.chunk_q[cq0 + lane / G] | (int)(((direct[item] >> lane) & 1u) << 31);
                if (iseq >= 2 &&
                    !__all_sync(0xffffffffu, tc::mbar_wait(fbar(bars, kSEmpty + sbuf), ((iseq - 2) >> 1) & 1))) {
                    if (!*err) *err = 103;
                    break;
                }
                int32_t *seg = reinterpret_cast<int32_t *>(smem + C::seg_off) + sbuf * 1280;
                const uint32_t *item_rm = rmask + rmask_off[item];
                int32_t *plist = reinterpret_cast<int32_t *>(smem + C::pl_off) + sbuf * kPageList;
                int npages = 0;   // page-list entries of the segments handled so far
                for (int s0 = 0; s0 < nseg; s0 += 32) {
                    const int s = s0 + lane;
                    int np = 0, tb = 0, pgb = 0;
                    if (s < nseg) {
                        const int len = p.seg_tok_len[sb + s];
                        tb = p.seg_tok_begin[sb + s];
                        pgb = a.node_page_off[p.seg_node[sb + s]];
                        np = (tb + len - 1) / kPageSize - tb / kPageSize + 1;
                        seg[s] = p.seg_chunk_pos[sb + s];
                        seg[256 + s] = pgb;
                        seg[512 + s] = tb;
                        seg[768 + s] = (int32_t)item_rm[s];
                    }
                    // Exclusive prefix sum of page counts across the warp.
                    int incl = np;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o)
                            incl += y;
                    }
                    const int ex = incl - np;
                    if (s < nseg)
                        seg[1024 + s] = npages + ex;
                    // Gather the batch's page ids, one entry per lane: entry j
                    // belongs to the last segment (lane) whose first entry is <= j.
                    const int tot = __shfl_sync(0xffffffffu, incl, 31);
                    const int pfirst = pgb + tb / kPageSize;
                    for (int j0 = 0; j0 < tot && npages + j0 < kPageList; j0 += 32) {
                        const int j = j0 + lane;
                        int lo = 0;
#pragma unroll
                        for (int step = 16; step > 0; step >>= 1)
                            if (__shfl_sync(0xffffffffu, ex, lo + step) <= j)
                                lo += step;
                        const int src = __shfl_sync(0xffffffffu, pfirst, lo) + j - __shfl_sync(0xffffffffu, ex, lo);
                        if (j < tot && npages + j < kPageList)
                            plist[npages + j] = a.page_id[src];
                    }
                    npages += tot;
                }
                if (lane == 0)
                    iinfo[sbuf] = ItemInfo{nseg, T, npages <= kPageList ? 1 : 0, npages};
                __syncwarp();
                tc::mbar_arrive(fbar(bars, kSFull + sbuf));
            }
            // The unit's q rows (bf16) and description for its compute group.
            const int ub = i % UB;
            if (i >= UB && !__all_sync(0xffffffffu, tc::mbar_wait(fbar(bars, kUEmpty + ub), ((i - UB) / UB) & 1))) {
                if (!*err) *err = 104;
                break;
            }
            const uint32_t qdst = base + C::qst_off + (uint32_t)ub * RMAX * D * 2;
#pragma unroll
            for (int j = 0; j < QJ; ++j) {
                const int x = lane + 32 * j;
                if (qrow[j] >= 0) {
                    const int r = x / (D / 8), ch = x - r * (D / 8);
                    cp_async_16(qdst + (uint32_t)(r * D + ch * 8) * 2, qg + (size_t)(qrow[j] + h * G) * D + ch * 8);
                }
            }
            cp_async_mbar_arrive_noinc(fbar(bars, kUFull + ub));
            if (lane < R)
                urow[ub * RMAX + lane] = qf;
            __syncwarp();
            if (lane == 0) {
                info[ub] = UnitInfo{R, cq0, h, ntiles, (i % NG) ? rseq1 : rseq0, {0, 0, 0}};
                tc::mbar_arrive(fbar(bars, kUFull + ub));
            }
            if (i % NG)
                rseq1 += ntiles;
            else
                rseq0 += ntiles;
        }
        cp_async_commit();
        cp_async_wait<0>();
    } else if (warp <= 2) {
        // ------------------------------------------------------- copy warps
        // Copy warp w (0, 1) loads the tiles of sequence number = w mod 2, so
        // one resolves its tile's pages while the other issues its copies.
        const int cpw = warp - 1;
        const int ring = NG == 2 ? cpw : 0;
        const __nv_bfloat16 *kg = reinterpret_cast<const __nv_bfloat16 *>(a.k_pages);
        const __nv_bfloat16 *vg = reinterpret_cast<const __nv_bfloat16 *>(a.v_pages);
        const uint64_t kv_pol = tc::l2_kv_policy(a.kv_once != 0);
        constexpr uint32_t kRowBytes = D * 2;
        constexpr uint32_t kPageBytes = kPageSize * kRowBytes;   // one head's rows of a page
        int seq = 0, iseq = -1, prev_item = -1, sbuf = 0;
        bool ok = true;
        for (int i = 0; ok; ++i) {
            // The next unit number from the metadata warp (-1: no more).
            const int qslot = i % UQ;
            if (!__all_sync(0xffffffffu, tc::mbar_wait(fbar(bars, kQFull + qslot), (i / UQ) & 1))) {
                if (!*err) *err = 105;
                break;
            }
            const int u = useq[qslot];
            __syncwarp();
            if (lane == 0)
                tc::mbar_arrive(fbar(bars, kQEmpty + qslot));
            const int item = u < 0 ? -1 : u / Hkv;
            if (u < 0 || item != prev_item) {
                // Release the previous item's segment table, then wait for this one's.
                if (prev_item >= 0) {
                    __syncwarp();
                    tc::mbar_arrive(fbar(bars, kSEmpty + sbuf));
                }
                if (u < 0)
                    break;
                prev_item = item;
                ++iseq;
                sbuf = iseq & 1;
                if (!__all_sync(0xffffffffu, tc::mbar_wait(fbar(bars, kSFull + sbuf), (iseq >> 1) & 1))) {
                    if (!*err) *err = 106;
                    break;
                }
            }
            const int h = u - item * Hkv;
            const int32_t *seg = reinterpret_cast<const int32_t *>(smem + C::seg_off) + sbuf * 1280;
            const int32_t *plist = reinterpret_cast<const int32_t *>(smem + C::pl_off) + sbuf * kPageList;
            const ItemInfo ii = iinfo[sbuf];
            (void)i;
            // Physical page of token tk of segment sg.
            auto page_of = [&](int sg, int tk) {
                return ii.listed ? plist[seg[1024 + sg] + tk / kPageSize - seg[512 + sg] / kPageSize]
                                 : a.page_id[seg[256 + sg] + tk / kPageSize];
            };
            const int nseg = ii.nseg, T = ii.T, ntiles = (T + kTile - 1) / kTile;
            const bool mine = NG == 1 || (i % NG) == cpw;   // the unit goes through this warp's ring
            for (int t = 0; t < (mine ? ntiles : 0); ++t, ++seq) {
                if (NG == 1 && (seq & 1) != cpw)
                    continue;
                const int st = ring * RST + seq % RST;
                const uint32_t full = fbar(bars, kFull + st);
                const uint32_t kdst = base + C::stage_off + (uint32_t)(st * 2) * C::op_bytes;
                const uint32_t vdst = kdst + C::op_bytes;
                // Segment holding position pos (warp-uniform: broadcast reads).
                auto seg_at = [&](int pos) {
                    int lo = 0, hi = nseg - 1;
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (seg[mid] <= pos)
                            lo = mid;
                        else
                            hi = mid - 1;
                    }
                    return lo;
                };
                const int p0 = t * kTile, nvalid = min(kTile, T - p0);
                const int sga = seg_at(p0);
                const int tka = seg[512 + sga] + p0 - seg[sga];
                if (nvalid == kTile && (tka % kPageSize) == 0 && seg_at(p0 + kTile - 1) == sga) {
                    // Fast path: four whole pages of one segment.
                    const int pg = lane < 4 ? page_of(sga, tka + kPageSize * lane) : -1;
                    if (seq >= RST &&
                        !__all_sync(0xffffffffu, tc::mbar_wait(fbar(bars, kEmpty + st), ((seq / RST) - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    const uint32_t mrow = (uint32_t)seg[768 + sga];
                    meta[st * kTile + lane] = mrow;
                    meta[st * kTile + lane + 32] = mrow;
                    if (lane == 0)
                        tc::mbar_arrive_expect_tx(full, 4 * 2 * kPageBytes);
                    __syncwarp();
                    if (lane < 4) {
                        const size_t o = ((size_t)pg * Hkv + h) * kPageSize * D;
                        const uint32_t rb = (uint32_t)lane * kPageBytes;
                        tc::bulk_load(kdst + rb, kg + o, kPageBytes, full, kv_pol);
                        tc::bulk_load(vdst + rb, vg + o, kPageBytes, full, kv_pol);
                    }
                    tc::mbar_arrive(full);
                    continue;
                }
                // General path: segment and token of the tile positions lane and lane + 32.
                int sgk[2], tkk[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int pos = p0 + lane + 32 * k;
                    sgk[k] = -1;
                    tkk[k] = 1;
                    if (pos < T) {
                        int lo = 0, hi = nseg - 1;
                        while (lo < hi) {
                            const int mid = (lo + hi + 1) >> 1;
                            if (seg[mid] <= pos)
                                lo = mid;
                            else
                                hi = mid - 1;
                        }
                        sgk[k] = lo;
                        tkk[k] = seg[512 + lo] + pos - seg[lo];
                    }
                }
                // Slot j (tile rows 16j..16j+15) goes by bulk copy when its 16
                // positions are one whole page of one segment.
                uint32_t tp = 0;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int s_first = __shfl_sync(0xffffffffu, sgk[k], lane & 16);
                    const int t_first = __shfl_sync(0xffffffffu, tkk[k], lane & 16);
                    const bool okp = sgk[k] >= 0 && sgk[k] == s_first && (t_first % kPageSize) == 0;
                    const uint32_t bal = __ballot_sync(0xffffffffu, okp);
                    if ((bal & 0xffffu) == 0xffffu)
                        tp |= 1u << (2 * k);
                    if ((bal >> 16) == 0xffffu)
                        tp |= 1u << (2 * k + 1);
                }
                // Lane j < 4 resolves slot j's page (position 16j is lane
                // 16 * (j & 1)'s entry k = j >> 1).
                const int src = 16 * (lane & 1);
                const int s_a = __shfl_sync(0xffffffffu, sgk[0], src), s_b = __shfl_sync(0xffffffffu, sgk[1], src);
                const int t_a = __shfl_sync(0xffffffffu, tkk[0], src), t_b = __shfl_sync(0xffffffffu, tkk[1], src);
                int pg_lane = -1;
                if (lane < 4 && ((tp >> lane) & 1u))
                    pg_lane = (lane & 2) ? page_of(s_b, t_b) : page_of(s_a, t_a);
                int pid[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    pid[k] = -1;
                    if (sgk[k] >= 0 && !((tp >> ((lane + 32 * k) >> 4)) & 1u))
                        pid[k] = page_of(sgk[k], tkk[k]);
                }
                if (seq >= RST &&
                    !__all_sync(0xffffffffu, tc::mbar_wait(fbar(bars, kEmpty + st), ((seq / RST) - 1) & 1))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    meta[st * kTile + lane + 32 * k] = sgk[k] >= 0 ? (uint32_t)seg[768 + sgk[k]] : 0u;
                // Rows past the chunk's end: zero V so that p.v may run over
                // all 64 rows (their p is 0; stale shared memory could be NaN).
                if (nvalid < kTile) {
                    uint4 *vz = reinterpret_cast<uint4 *>(smem + (vdst - base) + nvalid * kRowBytes);
                    for (int x = lane; x < (kTile - nvalid) * (D / 8); x += 32)
                        vz[x] = make_uint4(0u, 0u, 0u, 0u);
                }
                // Lane 0's arrival releases the warp's row masks and zeros
                // (the lanes' own arrivals below may be deferred).
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive_expect_tx(full, __popc(tp) * 2 * kPageBytes);
                __syncwarp();
                if (pg_lane >= 0) {
                    const size_t o = ((size_t)pg_lane * Hkv + h) * kPageSize * D;
                    const uint32_t rb = (uint32_t)lane * kPageBytes;
                    tc::bulk_load(kdst + rb, kg + o, kPageBytes, full, kv_pol);
                    tc::bulk_load(vdst + rb, vg + o, kPageBytes, full, kv_pol);
                }
                // Ragged rows: one row per warp step; lanes cover K and V chunks.
                bool any_cp = false;
                constexpr int CPR = D / 8;  // 16-byte chunks per row per operand
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    uint32_t nb = __ballot_sync(0xffffffffu, pid[k] >= 0);
                    any_cp |= nb != 0;
                    while (nb) {
                        const int sl = __ffs(nb) - 1;
                        nb &= nb - 1;
                        const int row = sl + 32 * k;
                        const int pgr = __shfl_sync(0xffffffffu, pid[k], sl);
                        const int tk = __shfl_sync(0xffffffffu, tkk[k], sl);
                        const long long o = (((long long)pgr * Hkv + h) * kPageSize + (tk % kPageSize)) * D;
                        for (int x = lane; x < 2 * CPR; x += 32) {
                            const int kv = x / CPR, ch = x - kv * CPR;
                            cp_async_16((kv ? vdst : kdst) + row * kRowBytes + ch * 16, (kv ? vg : kg) + o + ch * 8);
                        }
                    }
                }
                // With ragged rows, each lane's arrival waits for its own
                // copies to land; the warp goes on with the next tile.
                if (any_cp)
                    cp_async_mbar_arrive_noinc(full);
                else
                    tc::mbar_arrive(full);
            }
            if (!ok)
                if (!*err) *err = 107;
        }
        cp_async_wait<0>();
        // Do not leave while bulk copies of ours may still be landing: wait for
        // the last use of every stage.
        for (int s = 0; s < RST && s < seq; ++s) {
            const int last = seq - 1 - ((seq - 1 - s) % RST);
            tc::mbar_wait(fbar(bars, kFull + ring * RST + s), (last / RST) & 1);
        }
    } else if (warp < 3 + NCW) {
        // ------------------------------------------------------------ compute
        // Group g takes the CTA's units g, g + NG, ... whole; warp lw of the
        // group takes tokens 8 lw .. 8 lw + 7 of every tile.  Lane layout:
        //   part = lane % NPART   owns the head dims of 16-byte chunks part,
        //                         part + NPART, ... (DP dims; the part lanes
        //                         read contiguous bytes of a K or V row);
        //   rg                    row group: rows rg RL .. rg RL + RL - 1;
        //   ts                    token slot: token 8 lw + step TS + ts.
        // A lane keeps its q rows and its share of the output rows in
        // registers and works on fp32 pairs (f32x2 FMAs).  NPART is 16 at
        // head_dim 128 with 3-8 rows (one row group holds all rows, so each
        // K and V element is widened from bf16 once), else 8.
        constexpr int NPART = (D == 128 && (RMAX == 4 || RMAX == 8)) ? 16 : 8;
        constexpr int LP = NPART == 16 ? 4 : 3;        // log2 NPART
        constexpr int DP = D / NPART;                  // dims per lane
        constexpr int NCH = DP / 8;                    // 16-byte chunks per lane and row
        constexpr int NRG = NPART == 16 ? (RMAX == 8 ? 2 : 1) : (RMAX <= 2 ? 1 : RMAX == 4 ? 2 : 4);
        constexpr int RL = RMAX / NRG;                 // rows per lane
        constexpr int TS = 32 / (NPART * NRG);         // token slots per step
        constexpr int NSTEP = 8 / TS;                  // steps per tile
        constexpr int SUB = NSTEP < 4 ? NSTEP : 4;   // steps per maximum update
        static_assert(NCH >= 1 && TS >= 1 && NPART * NRG * TS == 32, "lane layout");
        const int cw = warp - 3;          // compute warp 0..NCW-1
        const int g = cw >> 3, lw = cw & 7;
        const int part = lane & (NPART - 1), rg = (lane >> LP) % NRG, ts = (lane >> LP) / NRG;
        // Rows whose softmax state a lane keeps.  With RL = 2 or 4 rows per
        // lane the part lanes split the first log2 RL steps of the
        // dot-product sums between the rows (a reduce-scatter over the part
        // bits RS_SH .. LP - 1) and finish one row each, hr: a lane keeps
        // only that row's logits, maximum and sum (1/RL of the
        // exponentials) and fetches the other rows' probabilities for p.v
        // from the lanes that finished them.  With one row per lane every
        // part lane keeps the row.
        constexpr bool SPLIT = RL >= 2;
        constexpr int RS = SPLIT ? 1 : RL;
        constexpr int RS_SH = LP - (RL == 4 ? 2 : RL == 2 ? 1 : 0);   // lowest row bit of part
        constexpr int ROWBITS = (RL - 1) << RS_SH;                    // part bits naming hr
        const int hr = SPLIT ? (part >> RS_SH) & (RL - 1) : 0;
        float *qs = reinterpret_cast<float *>(smem + C::qs_off) + g * RMAX * D;
        float *mw = reinterpret_cast<float *>(smem + C::ml_off) + g * 8 * RMAX;
        float *lwb = reinterpret_cast<float *>(smem + C::ml_off) + NCW * RMAX + g * 8 * RMAX;
        float *obuf = reinterpret_cast<float *>(smem + C::obuf_off) + g * 8 * C::MRB * D;
        const uint32_t bar_id = 1 + (uint32_t)g, nthr = 256;
        const int gtid = tid - 96 - g * 256;   // thread index within the group
        int mseq = 0;                          // states handed to the merge warp
        for (int i = g;; i += NG) {
            const int ub = i % UB;
            const bool okw = tc::mbar_wait(fbar(bars, kUFull + ub), (i / UB) & 1);
            if (tc::named_sync_or(bar_id, nthr, !okw)) {
                if (!*err) *err = 108;
                break;
            }
            const UnitInfo ui = info[ub];
            if (ui.R < 0)
                break;   // no more units
            const int R = ui.R;
            const __nv_bfloat16 *qst = reinterpret_cast<const __nv_bfloat16 *>(smem + C::qst_off) + ub * RMAX * D;
            // qs[r][e]: q pre-scaled by scale * log2 e; rows past R are 0.
            for (int x = gtid; x < RMAX * D; x += nthr)
                qs[x] = x < R * D ? __bfloat162float(qst[x]) * a.scale_log2 : 0.f;
            tc::named_sync(bar_id, nthr);
            f32x2 qv[RL][NCH * 4];
#pragma unroll
            for (int rl = 0; rl < RL; ++rl)
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    const float *qp = qs + (rg * RL + rl) * D + (part + NPART * c) * 8;
                    const ulonglong2 a0 = *reinterpret_cast<const ulonglong2 *>(qp);
                    const ulonglong2 a1 = *reinterpret_cast<const ulonglong2 *>(qp + 4);
                    qv[rl][4 * c + 0] = a0.x;
                    qv[rl][4 * c + 1] = a0.y;
                    qv[rl][4 * c + 2] = a1.x;
                    qv[rl][4 * c + 3] = a1.y;
                }
            float m_run[RS], l_run[RS];
            f32x2 o_acc[RL][NCH * 4];
#pragma unroll
            for (int k = 0; k < RS; ++k) {
                m_run[k] = -INFINITY;
                l_run[k] = 0.f;
            }
#pragma unroll
            for (int rl = 0; rl < RL; ++rl)
#pragma unroll
                for (int e = 0; e < NCH * 4; ++e)
                    o_acc[rl][e] = 0ull;   // (+0, +0)
            bool tile_ok = true;
            for (int t = 0; t < ui.ntiles; ++t) {
                const int sq = ui.seq0 + t, st = g * RST + sq % RST;
                // One consumer per ring, in order: the parity names the use.
                const bool got = tc::mbar_wait(fbar(bars, kFull + st), (sq / RST) & 1);
                if (!__all_sync(0xffffffffu, got)) {
                    tile_ok = false;
                    break;
                }
                const uint8_t *Ks = smem + C::stage_off + (size_t)(st * 2) * C::op_bytes;
                const uint8_t *Vs = Ks + C::op_bytes;
#pragma unroll
                for (int s0 = 0; s0 < NSTEP; s0 += SUB) {
                    // Logits of the lane's state rows for the SUB tokens of its slot.
                    float sv[SUB][RS];
#pragma unroll
                    for (int s = 0; s < SUB; ++s) {
                        const int tok = lw * 8 + (s0 + s) * TS + ts;
                        f32x2 acc[RL];
#pragma unroll
                        for (int rl = 0; rl < RL; ++rl)
                            acc[rl] = 0ull;
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            const uint4 kw =
                                *reinterpret_cast<const uint4 *>(Ks + tok * (D * 2) + (part + NPART * c) * 16);
                            const f32x2 k0 = bf16x2_to_f2(kw.x), k1 = bf16x2_to_f2(kw.y);
                            const f32x2 k2 = bf16x2_to_f2(kw.z), k3 = bf16x2_to_f2(kw.w);
#pragma unroll
                            for (int rl = 0; rl < RL; ++rl) {
                                acc[rl] = f2_fma(qv[rl][4 * c + 0], k0, acc[rl]);
                                acc[rl] = f2_fma(qv[rl][4 * c + 1], k1, acc[rl]);
                                acc[rl] = f2_fma(qv[rl][4 * c + 2], k2, acc[rl]);
                                acc[rl] = f2_fma(qv[rl][4 * c + 3], k3, acc[rl]);
                            }
                        }
                        const uint32_t mrow = meta[st * kTile + tok];
                        if constexpr (SPLIT) {
                            float v[RL];
#pragma unroll
                            for (int rl = 0; rl < RL; ++rl) {
                                const float2 a2 = f2_unpack(acc[rl]);
                                v[rl] = a2.x + a2.y;
                            }
                            // Lane and lane ^ NPART/2 swap halves of their
                            // rows: each adds the partner's share of the
                            // half it keeps (upper half if the bit is set).
                            {
                                constexpr int o1 = NPART / 2;
                                const bool up = (part & o1) != 0;
#pragma unroll
                                for (int j = 0; j < RL / 2; ++j) {
                                    const float keep = up ? v[j + RL / 2] : v[j];
                                    const float send = up ? v[j] : v[j + RL / 2];
                                    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o1);
                                }
                            }
                            if constexpr (RL == 4) {
                                constexpr int o2 = NPART / 4;
                                const bool up = (part & o2) != 0;
                                const float keep = up ? v[1] : v[0];
                                const float send = up ? v[0] : v[1];
                                v[0] = keep + __shfl_xor_sync(0xffffffffu, send, o2);
                            }
#pragma unroll
                            for (int o = NPART / (2 * RL); o >= 1; o >>= 1)
                                v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
                            sv[s][0] = ((mrow >> (rg * RL + hr)) & 1u) ? v[0] : -INFINITY;
                        } else {
#pragma unroll
                            for (int rl = 0; rl < RL; ++rl) {
                                const float2 a2 = f2_unpack(acc[rl]);
                                float v = a2.x + a2.y;
                                v += __shfl_xor_sync(0xffffffffu, v, 1);
                                v += __shfl_xor_sync(0xffffffffu, v, 2);
                                v += __shfl_xor_sync(0xffffffffu, v, 4);
                                sv[s][rl] = ((mrow >> (rg * RL + rl)) & 1u) ? v : -INFINITY;
                            }
                        }
                    }
                    // Running maximum over the warp's tokens (the slot lanes
                    // differ in lane bits 3 + log2 NRG and up), rescale, and
                    // the probabilities.
#pragma unroll
                    for (int k = 0; k < RS; ++k) {
                        float mx = sv[0][k];
#pragma unroll
                        for (int s = 1; s < SUB; ++s)
                            mx = fmaxf(mx, sv[s][k]);
#pragma unroll
                        for (int o = NPART * NRG; o < 32; o <<= 1)
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                        const float mnew = fmaxf(m_run[k], mx);
                        // Rescale the sums where the maximum grew (m_run may
                        // be -inf: alpha = 0 then, on zero sums); the warp
                        // skips it when no lane's maximum moved.
                        const bool grew = mnew > m_run[k];
                        if (__any_sync(0xffffffffu, grew)) {
                            const float alpha = grew ? tc::ex2(m_run[k] - mnew) : 1.f;
                            l_run[k] *= alpha;
                            if constexpr (SPLIT) {
#pragma unroll
                                for (int j = 0; j < RL; ++j) {
                                    const float aj =
                                        __shfl_sync(0xffffffffu, alpha, (lane & ~ROWBITS) | (j << RS_SH));
                                    const f32x2 aa = f2_pack(aj, aj);
#pragma unroll
                                    for (int e = 0; e < NCH * 4; ++e)
                                        o_acc[j][e] = f2_mul(o_acc[j][e], aa);
                                }
                            } else {
                                const f32x2 aa = f2_pack(alpha, alpha);
#pragma unroll
                                for (int e = 0; e < NCH * 4; ++e)
                                    o_acc[k][e] = f2_mul(o_acc[k][e], aa);
                            }
                        }
                        if (mnew != -INFINITY) {
#pragma unroll
                            for (int s = 0; s < SUB; ++s) {
                                const float pr = tc::ex2(sv[s][k] - mnew);
                                sv[s][k] = pr;
                                l_run[k] += pr;
                            }
                        } else {
#pragma unroll
                            for (int s = 0; s < SUB; ++s)
                                sv[s][k] = 0.f;
                        }
                        m_run[k] = mnew;
                    }
                    // p.v (p = 0 for masked and absent tokens, whose V rows
                    // are finite or zero).
#pragma unroll
                    for (int s = 0; s < SUB; ++s) {
                        const int tok = lw * 8 + (s0 + s) * TS + ts;
                        float pr[RL];
                        if constexpr (SPLIT) {
#pragma unroll
                            for (int j = 0; j < RL; ++j)
                                pr[j] = __shfl_sync(0xffffffffu, sv[s][0], (lane & ~ROWBITS) | (j << RS_SH));
                        } else {
#pragma unroll
                            for (int rl = 0; rl < RL; ++rl)
                                pr[rl] = sv[s][rl];
                        }
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            const uint4 vw =
                                *reinterpret_cast<const uint4 *>(Vs + tok * (D * 2) + (part + NPART * c) * 16);
                            const f32x2 v0 = bf16x2_to_f2(vw.x), v1 = bf16x2_to_f2(vw.y);
                            const f32x2 v2 = bf16x2_to_f2(vw.z), v3 = bf16x2_to_f2(vw.w);
#pragma unroll
                            for (int rl = 0; rl < RL; ++rl) {
                                const f32x2 pp = f2_pack(pr[rl], pr[rl]);
                                o_acc[rl][4 * c + 0] = f2_fma(pp, v0, o_acc[rl][4 * c + 0]);
                                o_acc[rl][4 * c + 1] = f2_fma(pp, v1, o_acc[rl][4 * c + 1]);
                                o_acc[rl][4 * c + 2] = f2_fma(pp, v2, o_acc[rl][4 * c + 2]);
                                o_acc[rl][4 * c + 3] = f2_fma(pp, v3, o_acc[rl][4 * c + 3]);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(fbar(bars, kEmpty + st));
            }
            if (tc::named_sync_or(bar_id, nthr, !tile_ok)) {
                if (!*err) *err = 109;
                break;
            }
            // The warp's state per row: sums over its token slots (lanes that
            // differ in the slot bits), the same on all part lanes.
#pragma unroll
            for (int k = 0; k < RS; ++k)
#pragma unroll
                for (int o = NPART * NRG; o < 32; o <<= 1)
                    l_run[k] += __shfl_xor_sync(0xffffffffu, l_run[k], o);
#pragma unroll
            for (int rl = 0; rl < RL; ++rl) {
#pragma unroll
                for (int o = NPART * NRG; o < 32; o <<= 1) {
#pragma unroll
                    for (int e = 0; e < NCH * 4; ++e)
                        o_acc[rl][e] = f2_add(o_acc[rl][e], __shfl_xor_sync(0xffffffffu, o_acc[rl][e], o));
                }
            }
            // Hand the states to the merge warp, MRB rows at a time, each
            // time after it has read the previous ones; the group goes on
            // with its next unit meanwhile.
            bool merr = false;
            for (int rb = 0; rb < R; rb += C::MRB) {
                const bool okm = mseq == 0 || tc::mbar_wait(fbar(bars, kMEmpty + g), (mseq - 1) & 1);
                if (tc::named_sync_or(bar_id, nthr, !okm)) {
                    if (!*err) *err = 110;
                    merr = true;
                    break;
                }
#pragma unroll
                for (int k = 0; k < RS; ++k) {
                    const int r = rg * RL + (SPLIT ? hr : k);
                    if (rb == 0 && ts == 0 && (part & ~ROWBITS) == 0 && r < R) {
                        mw[lw * RMAX + r] = m_run[k];
                        lwb[lw * RMAX + r] = l_run[k];
                    }
                }
                if (rb == 0 && gtid < R)
                    mrow[g * RMAX + gtid] = urow[ub * RMAX + gtid];
#pragma unroll
                for (int rl = 0; rl < RL; ++rl) {
                    const int r = rg * RL + rl;
                    if (ts == 0 && r >= rb && r < rb + C::MRB && r < R) {
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            float *dst = obuf + (lw * C::MRB + (r - rb)) * D + (part + NPART * c) * 8;
                            *reinterpret_cast<ulonglong2 *>(dst) =
                                make_ulonglong2(o_acc[rl][4 * c + 0], o_acc[rl][4 * c + 1]);
                            *reinterpret_cast<ulonglong2 *>(dst + 4) =
                                make_ulonglong2(o_acc[rl][4 * c + 2], o_acc[rl][4 * c + 3]);
                        }
                    }
                }
                if (gtid == 0) {
                    mdesc[g].R = R;
                    mdesc[g].cq0 = ui.cq0;
                    mdesc[g].h = ui.h;
                    mdesc[g].rb = rb;
                }
                tc::named_sync(bar_id, nthr);
                if (gtid == 0)
                    tc::mbar_arrive(fbar(bars, kMFull + g));
                ++mseq;
            }
            if (merr)
                break;
            if (lane == 0)
                tc::mbar_arrive(fbar(bars, kUEmpty + ub));
        }
        // The group is done: tell the merge warp, once it has read the last
        // states.
        if (gtid == 0) {
            if (mseq > 0 && !tc::mbar_wait(fbar(bars, kMEmpty + g), (mseq - 1) & 1))
                if (!*err) *err = 110;
            mdesc[g].R = -1;
            tc::mbar_arrive(fbar(bars, kMFull + g));
        }
    } else {
        // -------------------------------------------------------------- merge
        // Merges each unit's 8 warp states per row in a fixed order (the step
        // is bitwise repeatable): the max M over the warps, each warp's
        // weight 2^(m_w - M) / L with L the weighted sum of the warps' sums,
        // the lse partial M + log2 L, then each output element as the
        // weighted sum of the warps' values (a lane takes 4 elements).
        int ms[2] = {0, 0};
        bool live[2] = {true, NG == 2};
        uint32_t idle = 0;
        while (live[0] || live[1]) {
            bool any = false;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                if (!live[g] || !tc::mbar_test(fbar(bars, kMFull + g), ms[g] & 1))
                    continue;
                any = true;
                const MergeDesc md{mdesc[g].R, mdesc[g].cq0, mdesc[g].h, mdesc[g].rb};
                if (md.R < 0) {
                    live[g] = false;
                    continue;
                }
                const float *mw = reinterpret_cast<const float *>(smem + C::ml_off) + g * 8 * RMAX;
                const float *lwb = mw + NCW * RMAX;
                float *wts = reinterpret_cast<float *>(smem + C::ml_off) + 2 * NCW * RMAX + g * 8 * RMAX;
                const float *obuf = reinterpret_cast<const float *>(smem + C::obuf_off) + g * 8 * C::MRB * D;
                int32_t *mdst = reinterpret_cast<int32_t *>(smem + C::mdst_off) + g * RMAX;
                const int32_t *mq = mrow + g * RMAX;
                if (md.rb == 0 && lane < md.R) {
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < 8; ++w)
                        M = fmaxf(M, mw[w * RMAX + lane]);
                    float L = 0.f, c[8];
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const float mwv = mw[w * RMAX + lane];
                        c[w] = (M == -INFINITY || mwv == -INFINITY) ? 0.f : tc::ex2(mwv - M);
                        L += lwb[w * RMAX + lane] * c[w];
                    }
                    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w)
                        wts[w * RMAX + lane] = c[w] * inv;
                    const float l2 = L > 0.f ? M + log2f(L) : -INFINITY;
                    const int head = md.h * G + (lane % G), qf = mq[lane];
                    // Destination row: the partial slot's, or (a query with
                    // this one slot) -1 - the output row.
                    if (a.direct && qf < 0) {
                        const int orow = (qf & 0x7fffffff) * Hq + head;
                        a.lse_out[orow] = direct_lse(l2);
                        mdst[lane] = -1 - orow;
                    } else {
                        const int prow = (md.cq0 + lane / G) * Hq + head;
                        a.lse_part[prow] = l2;
                        mdst[lane] = prow;
                    }
                }
                __syncwarp();
                const int rows = md.R - md.rb < C::MRB ? md.R - md.rb : C::MRB;
                for (int x = lane; x < rows * (D / 4); x += 32) {
                    const int r = x / (D / 4), e4 = (x - r * (D / 4)) * 4;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const float4 v = *reinterpret_cast<const float4 *>(obuf + (w * C::MRB + r) * D + e4);
                        const float wt = wts[w * RMAX + md.rb + r];
                        acc.x = fmaf(v.x, wt, acc.x);
                        acc.y = fmaf(v.y, wt, acc.y);
                        acc.z = fmaf(v.z, wt, acc.z);
                        acc.w = fmaf(v.w, wt, acc.w);
                    }
                    const int dr = mdst[md.rb + r];
                    if (dr >= 0) {
                        *reinterpret_cast<float4 *>(a.o_part + (size_t)dr * D + e4) = acc;
                    } else {
                        const size_t orow = (size_t)(-1 - dr);
                        store_out(a, orow, e4 + 0, D, acc.x);
                        store_out(a, orow, e4 + 1, D, acc.y);
                        store_out(a, orow, e4 + 2, D, acc.z);
                        store_out(a, orow, e4 + 3, D, acc.w);
                    }
                }
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(fbar(bars, kMEmpty + g));
                ++ms[g];
            }
            if (any)
                idle = 0;
            else if (++idle > (1u << 24)) {
                if (!*err) *err = 111;
                break;
            }
        }
    }
    __syncthreads();
    if (*err) {
        // A wait ran out: record it in the partition's status word and mark
        // every partial and output row of the launch's units as failed (the
        // step's output then shows it); the units are not tracked per CTA.
        if (tid == 0)
            report_failure(p.status, *err);
        for (int u = 0; u < n_units; ++u) {
            const int item = u / Hkv, h = u - item * Hkv;
            const int c = items[3 * item], qb = items[3 * item + 1], qe = items[3 * item + 2];
            const int cq0 = p.chunk_q_off[c] + qb;
            for (int x = tid; x < (qe - qb) * G * D; x += C::THREADS) {
                const int r = x / D, e = x - r * D;
                const size_t prw = (size_t)(cq0 + r / G) * Hq + h * G + (r % G);
                const size_t orw = (size_t)p.chunk_q[cq0 + r / G] * Hq + h * G + (r % G);
                a.o_part[prw * D + e] = __int_as_float(0x7fc00000);
                store_out(a, orw, e, D, __int_as_float(0x7fc00000));
                if (e == 0) {
                    a.lse_part[prw] = __int_as_float(0x7fc00000);
                    a.lse_out[orw] = __int_as_float(0x7fc00000);
                }
            }
        }
    }
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


template <int D, int RMAX>
int launch_one(const AttnArgs &a, const DevPartition &p, const int32_t *items, const uint32_t *rmask,
               const int32_t *rmask_off, const uint32_t *direct, int32_t n, uint32_t *queue, LaunchShape sh,
               cudaStream_t st)
{
    using C = FmaCfg<D, RMAX>;
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(phase1_fma_kernel<D, RMAX>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::alloc);
        if (e != cudaSuccess)
            return (int)e;
        configured = true;
    }
    const int32_t units = n * a.num_kv_heads;
    const int32_t grid = sh.grid < units ? sh.grid : units;
    const int32_t early = sh.early < grid ? sh.early : grid;
    return (int)launch_dependent(phase1_fma_kernel<D, RMAX>, dim3(grid), dim3(C::THREADS), C::alloc, st, a, p,
                                 items, rmask, rmask_off, direct, units, static_block(units, early, sh.block), early,
                                 queue);
}

template <int D>
int launch_bucket(int bucket, const AttnArgs &a, const DevPartition &p, const int32_t *items,
                  const uint32_t *rmask, const int32_t *rmask_off, const uint32_t *direct, int32_t n,
                  uint32_t *queue, LaunchShape sh, cudaStream_t st)
{
    switch (bucket) {
    case 0: return launch_one<D, 1>(a, p, items, rmask, rmask_off, direct, n, queue, sh, st);
    case 1: return launch_one<D, 2>(a, p, items, rmask, rmask_off, direct, n, queue, sh, st);
    case 2: return launch_one<D, 4>(a, p, items, rmask, rmask_off, direct, n, queue, sh, st);
    case 3: return launch_one<D, 8>(a, p, items, rmask, rmask_off, direct, n, queue, sh, st);
    default: return launch_one<D, 16>(a, p, items, rmask, rmask_off, direct, n, queue, sh, st);
    }
}

}  // namespace

int launch_phase1_fma(const AttnArgs &a, const DevPartition &p, const int32_t *items, const uint32_t *rmask,
                      const int32_t *rmask_off, const uint32_t *direct, int32_t n, int bucket, uint32_t *queue,
                      LaunchShape shape, void *stream)
{
    if (n <= 0)
        return 0;
    if ((int64_t)n * a.num_kv_heads > INT32_MAX || !queue || shape.grid < 1 || shape.early < 1)
        return (int)cudaErrorInvalidValue;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return a.head_dim == 128 ? launch_bucket<128>(bucket, a, p, items, rmask, rmask_off, direct, n, queue, shape, st)
                             : launch_bucket<64>(bucket, a, p, items, rmask, rmask_off, direct, n, queue, shape, st);
}

}  // namespace deft
