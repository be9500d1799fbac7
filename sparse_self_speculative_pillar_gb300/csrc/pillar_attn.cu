// pillar_attn.cu -- the persistent unified draft/verify attention kernel and
// the merge of its partial results.
//
// What it computes ("SparseSpec-MLSys26", 核心方法 / PillarAttn):
//   draft request, KV head g: every query head h of group g attends exactly
//     the listed positions I = sparse_idx[b, g, :cnt]:
//       out[h] = sum_{t in I} softmax_t(scale * q_h . k_t) v_t
//   verify request, row j in 0..k: full causal attention over positions
//     [0, L-(k+1)+j], writing the scaled logits of every position (-inf past
//     the row's limit) and the row's natural-log LSE.
// Both go through the same page-size-1 gather: position t of request b lives
// in slot slot_table[kv_off[b] + t], its K/V row at k_pool[slot, g, :]
// (same page, "Unified batch scheduler + fused attention kernel": page size 1
// unifies sparse and full attention in one pipeline).
//
// GB300 design: a persistent grid of one CTA per SM (the CTA owns the SM's
// 512 tensor-memory columns and a ring of up to eight 64-key K/V stages in
// shared memory), sixteen warps per CTA in four groups (registers move to
// the softmax group with setmaxnreg):
//   * resolver warp: pops work items from a global atomic counter, reads the
//     item's records and translates its positions into pool slots (a verify
//     item's slots are one run of the slot table, read 32 per lane in one
//     round trip; a draft list is read 16 per lane, list -> slot) into a ring
//     of three row lists, up to two items ahead of the loaders;
//   * four loader warps: gather the item's K/V rows into the stage ring with
//     TMA tile::gather4 (four 256-byte page-size-1 rows per copy) in the
//     swizzled layout the tensor cores read, completion counted in bytes on
//     the stage's mbarrier; the item's query rows go to their operand slots
//     with the first tile and its metadata travels in the stage record;
//   * MMA warp (one thread): issues all tensor-core work -- S = Q K^T
//     (M = 64 query-row slots, N = 64 keys) into one of four S buffers in
//     tensor memory as soon as a tile has landed, and O += P V with P read
//     straight from tensor memory once the softmax has written it; a
//     finished P V releases the stage and the S buffer through
//     tcgen05.commit, so the tensor pipe runs up to four tiles ahead of the
//     softmax;
//   * four consumer warps, for draft and verify items alike.  An item's query
//     rows (the G heads of a draft token, the (k+1)*G rows of a verify
//     request) are spread over the four TMEM lane quadrants; each warp reads
//     its rows with the 16x256b shape, four threads per row, masks (list
//     validity; for verify rows also causality), dumps the verify logits,
//     keeps a running maximum and sum, and writes the bf16 probabilities back
//     over the scores for the P V MMA.  O is rescaled only when a row's
//     maximum grows by more than 2^8, so the exponentials stay bounded
//     without touching O on most tiles.  Two items have query operands of
//     their own (alternating between items) and their O
//     accumulators sit in separate TMEM columns, so an item's epilogue
//     overlaps the next item's MMAs;
//   * four epilogue warps, one per quadrant: the softmax warps hand each
//     finished item over (a two-slot shared-memory mailbox per quadrant);
//     once the item's last P V has completed, the epilogue warp reads its O
//     columns, normalises, writes the rows and releases the columns;
//   * a (request, KV head) split over several items (long contexts, long
//     critical lists) writes normalised partials (o, lse) per item, combined
//     afterwards by merge_kernel, a flat bandwidth pass:
//     o = sum_i e^{lse_i - lse} o_i, lse = log sum_i e^{lse_i};
//   * every wait is bounded (1 s unless the shape sets a bound); a timeout raises PILLAR_FLAG_TIMEOUT,
//     the loaders wait for their copies still in flight, the MMA thread for
//     its MMAs, the tensor memory is freed and the CTA returns.
#include <cuda.h>  // CUtensorMap (the encoder is resolved at run time through the runtime)

#include "pillar_device.cuh"

namespace pillar {

struct AttnParams {
    CUtensorMap tmap_k, tmap_v;  // the pools as [num_slots * Hkv rows, D] bf16, box 64 x 1, 128-byte swizzle
    const uint16_t *q, *k_pool, *v_pool;
    const int *slot_table, *sparse_idx;
    const int *sparse_slot;  // null, or the draft lists' slots (same layout as sparse_idx)
    uint16_t *out;
    float *logits, *lse;
    WsHeader *hdr;
    const ReqInfo *req;
    const long long *kv_off, *logit_off;
    const UnitInfo *unit;
    const MergeUnit *merge_units;
    const Item *items;
    float *part_o, *part_lse;
    long long num_slots;
    int Hq, Hkv, G, k, M, max_sparse;
    int RQ, RQd;  // query rows per TMEM lane quadrant: verify ceil(M / 4), draft ceil(G / 4)
    int static_units;  // 1: the naive joint batch (CTA c takes units c, c + grid, ...; no queue)
    float scale;
    unsigned long long wait_ns;  // bound of every pipeline wait (the drains keep kWaitTimeoutNs)
};

enum : int { kFirst = 1, kLast = 2, kStop = 4 };

// Everything the consumers need to know about a work item.
struct ItemInfo {
    int it;          // work item index (-1: no more work)
    int mode;        // 1 verify, otherwise draft
    int b, g;        // request, KV head
    int n, begin;    // keys of the item, first key (verify: position; draft: list index)
    int q_off, vidx; // first query row, verify index
    int L, nsplit, split, rec;  // context length, items of the unit, this item's index, first partial row
    long long logit_off, kv_off;
};

struct StageMeta {
    ItemInfo info;             // meaningful on the first tile of an item
    int nk;                    // keys in this tile (0..64)
    int flags;                 // kFirst / kLast / kStop
    int pos0;                  // logical position of key 0 (verify)
    int qb;                    // query buffer of the item
    unsigned long long valid;  // bit i: key i has an in-range position and slot
    int mode;                  // the item's mode, on every tile
    int pad;
};

constexpr int kSBuf = 4;                  // S/P buffers in tensor memory
constexpr int kRowLists = 3;              // resolved items in flight between the resolver and the loaders
constexpr int kMaxStages = 8;             // K/V stages in shared memory
constexpr int kSmemBudget = 227 * 1024;   // dynamic shared memory of one CTA
constexpr int kMinSmem = 120 * 1024;      // never two CTAs on one SM: each takes all 512 TMEM columns
constexpr uint32_t kTmemCols = 512;       // 4 S/P buffers x 64 columns, then O of the two query buffers

template <int D>
struct Smem {
    static constexpr int KCH = D / 8;              // 16-byte chunks per row
    static constexpr int CORE_SBO = KCH * 128;     // core-matrix stride along rows (verify Q, K and V tiles)
    static constexpr int QHALF = 64 * D * 2;       // the 64 query-row slots of one item's S MMA (M = 64)
    static constexpr int QREG = 2 * QHALF;         // two items' query operands
    static constexpr int ROWS = kTileKeys * D * 2;  // the K (or V) rows of one tile
    static constexpr int STAGE = 2 * ROWS;
    static constexpr int off_q = 0;
    static constexpr int off_rows = QREG;
    static constexpr int off_info = off_rows + kRowLists * kMaxChunk * 4;
    static constexpr int off_meta = off_info + kRowLists * (int)sizeof(ItemInfo);
    static constexpr int off_pend = off_meta + kMaxStages * (int)sizeof(StageMeta);
    static constexpr int off_bar = off_pend + kSBuf * 16;
    // full and empty [kMaxStages], qempty[2], rfull and rempty [kRowLists], s_full, s_free and p_full [kSBuf],
    // o_free[2], cexit, drain, o_done[2], epi_full and epi_empty [2 * kEpiWarps]
    static constexpr int NBAR = 2 * kMaxStages + 2 + 2 * kRowLists + 3 * kSBuf + 2 + 2 + 2 + 4 * kEpiWarps;
    static constexpr int off_misc = off_bar + NBAR * 8;
    static constexpr int off_epi = off_misc + 16;  // per (epilogue warp, slot): EpiRec + 32 float2
    static constexpr int EPI_BYTES = kEpiWarps * 2 * (32 + 32 * 8);
    static constexpr int off_stage = (off_epi + EPI_BYTES + 1023) / 1024 * 1024;
    static constexpr int NSTAGE = (kSmemBudget - off_stage) / STAGE < kMaxStages ? (kSmemBudget - off_stage) / STAGE
                                                                                 : kMaxStages;
    static constexpr int used = off_stage + NSTAGE * STAGE;
    static constexpr int total = used < kMinSmem ? kMinSmem : used;
    static constexpr uint32_t tO = kSBuf * kTileKeys;  // TMEM column of O for query buffer 0 (+D for buffer 1)
};
static_assert(Smem<128>::NSTAGE >= 4 && Smem<64>::NSTAGE >= 4, "stage ring depth");
static_assert(Smem<128>::total <= kSmemBudget && Smem<64>::total <= kSmemBudget, "shared memory budget");
static_assert(Smem<128>::tO + 2 * 128 <= kTmemCols, "tensor memory budget");
static_assert(sizeof(StageMeta) % 16 == 0 && sizeof(ItemInfo) == 64, "record layout");

// An item whose O rows an epilogue warp is to write (handed over by the
// consumer warp of the same quadrant through a two-slot mailbox).
struct EpiRec {
    int mode, g, q_off, nsplit, rec, qb;
    int stop;  // no more items
    int pad;
};
static_assert(sizeof(EpiRec) == 32, "epilogue record");

struct Ctx {
    char *smem;
    StageMeta *meta;
    ItemInfo *iinfo;
    int *rowlist;  // [kRowLists][kMaxChunk]
    uint64_t *full, *empty, *qempty, *rfull, *rempty;
    uint64_t *s_full, *s_free, *p_full, *o_free, *cexit, *drain;
    uint64_t *o_done;                // [2]: an item's last P V has completed (per O buffer)
    uint64_t *epi_full, *epi_empty;  // [kEpiWarps * 2]: mailbox slots
    EpiRec *epi;                     // [kEpiWarps * 2]
    float2 *epi_l;                   // [kEpiWarps * 2][32]: the softmax sums l of each thread's two rows
    int4 *pend;  // [kSBuf] tiles between their S and P V MMAs (MMA thread only)
    volatile int *abort;
    uint32_t *tmem_slot;
    int *err;
    unsigned long long wait_ns;  // bound of every pipeline wait
};

template <int D>
__device__ __forceinline__ Ctx make_ctx(char *smem, const AttnParams &p) {
    using S = Smem<D>;
    Ctx c;
    c.smem = smem;
    c.meta = reinterpret_cast<StageMeta *>(smem + S::off_meta);
    c.iinfo = reinterpret_cast<ItemInfo *>(smem + S::off_info);
    c.rowlist = reinterpret_cast<int *>(smem + S::off_rows);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::off_bar);
    c.full = bars;
    c.empty = bars + kMaxStages;
    c.qempty = bars + 2 * kMaxStages;
    c.rfull = c.qempty + 2;
    c.rempty = c.rfull + kRowLists;
    c.s_full = c.rempty + kRowLists;
    c.s_free = c.s_full + kSBuf;
    c.p_full = c.s_free + kSBuf;
    c.o_free = c.p_full + kSBuf;
    c.cexit = c.o_free + 2;
    c.drain = c.cexit + 1;
    c.o_done = c.drain + 1;
    c.epi_full = c.o_done + 2;
    c.epi_empty = c.epi_full + 2 * kEpiWarps;
    c.epi = reinterpret_cast<EpiRec *>(smem + S::off_epi);
    c.epi_l = reinterpret_cast<float2 *>(smem + S::off_epi + 2 * kEpiWarps * 32);
    c.pend = reinterpret_cast<int4 *>(smem + S::off_pend);
    c.abort = reinterpret_cast<volatile int *>(smem + S::off_misc);
    c.tmem_slot = reinterpret_cast<uint32_t *>(smem + S::off_misc + 4);
    c.err = &p.hdr->err;
    c.wait_ns = p.wait_ns;
    return c;
}

// Bounded wait that ignores the abort flag: used only to let copies or MMAs
// already in flight finish before the CTA exits (always the one-second
// bound, whatever the pipeline waits' bound).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kWaitTimeoutNs) return;
}

// Slot of an item's query row r in the 64-row operand of the S MMA.  With
// M = 64 the MMA keeps operand row a in TMEM lane 32 (a / 16) + a % 16, so
// slot 16 q + i lands in lane i of quadrant q: row r goes to quadrant r / RQ,
// lane r % RQ (RQ <= 16).  The S, P and O rows share those lanes.  Verify row
// r = j*G + gi, draft row r = gi.
__device__ __forceinline__ int row_slot(int r, int RQ) {
    const int q = r / RQ;
    return 16 * q + (r - q * RQ);
}

// ============================================================== resolver warp

// The next item of a CTA under the naive joint batch: the items of units
// blockIdx.x, blockIdx.x + gridDim.x, ... in order (unit cursor u, split s);
// num_items when none is left.  A verify unit's items are listed head-minor
// by the planner: split s of unit (b, g) is item item_base - g*ns + g + s*Hkv.
__device__ __forceinline__ int static_next_item(const AttnParams &p, int num_items, int &u, int &s) {
    const int U = *reinterpret_cast<volatile int *>(&p.hdr->num_units);
    for (; u < U; u += gridDim.x, s = 0) {
        const UnitInfo ui = p.unit[u];
        if (s >= ui.nsplit) continue;
        const int b = u / p.Hkv, g = u - b * p.Hkv;
        const int it = p.req[b].mode == 1 ? ui.item_base - g * ui.nsplit + g + s * p.Hkv : ui.item_base + s;
        ++s;
        return it;
    }
    return num_items;
}

__device__ void resolver(const AttnParams &p, const Ctx &c, int lane) {
    const int num_items = *reinterpret_cast<volatile int *>(&p.hdr->num_items);
    uint32_t eph = 0;
    int su = blockIdx.x, ss = 0;  // the naive joint batch's cursor
    for (int rb = 0;; rb = rb + 1 == kRowLists ? 0 : rb + 1) {
        if (!mbar_wait(&c.rempty[rb], ((eph >> rb) & 1) ^ 1, c.abort, c.err, c.wait_ns)) return;
        eph ^= 1u << rb;
        int it = 0;
        if (lane == 0) it = p.static_units ? static_next_item(p, num_items, su, ss) : atomicAdd(&p.hdr->item_counter, 1);
        it = __shfl_sync(0xffffffffu, it, 0);
        if (it >= num_items) {
            if (lane == 0) c.iinfo[rb].it = -1;
            mbar_arrive(&c.rfull[rb]);
            return;
        }
        const Item itm = p.items[it];
        const int b = itm.unit / p.Hkv, g = itm.unit - b * p.Hkv;
        const ReqInfo ri = p.req[b];
        const UnitInfo ui = p.unit[itm.unit];
        const long long kvo = p.kv_off[b];
        const long long lgo = p.logit_off[b];
        const bool verify = ri.mode == 1;
        const int n = itm.end - itm.begin;
        const long long lrow = ((long long)b * p.Hkv + g) * p.max_sparse + itm.begin;
        const int *list = p.sparse_idx + lrow;
        // draft lists with their slots already translated: the slot is read beside the position
        // instead of through the slot table (one round trip instead of two dependent ones)
        const int *slist = (!verify && p.sparse_slot) ? p.sparse_slot + lrow : nullptr;
        int *rows = c.rowlist + rb * kMaxChunk;
        int bad = 0;
        if (verify) {
            // a verify item's slots are one contiguous run of the slot table: 32 independent
            // loads per lane, one round trip for the 1024 keys of a default item
            for (int base = 0; base < n; base += 32 * 32) {
                int slot[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const int i = base + r * 32 + lane;
                    slot[r] = i < n ? __ldg(p.slot_table + kvo + itm.begin + i) : -1;
                }
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const int i = base + r * 32 + lane;
                    if (i < n) {
                        int s = slot[r];
                        if (s < 0 || (long long)s >= p.num_slots) {
                            bad |= PILLAR_FLAG_SLOT;
                            s = -1;
                        }
                        rows[i] = s;
                    }
                }
            }
        } else
        // draft lists: 16 independent loads per lane keep the dependent list -> slot chain short
        for (int base = 0; base < n; base += 32 * 16) {
            int pos[16], slot[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int i = base + r * 32 + lane;
                pos[r] = i < n ? __ldg(list + i) : -1;
                if (slist) slot[r] = i < n ? __ldg(slist + i) : -1;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int i = base + r * 32 + lane;
                const bool inpos = pos[r] >= 0 && pos[r] < ri.len;
                if (i < n && !inpos) bad |= PILLAR_FLAG_INDEX;
                if (!slist) slot[r] = (i < n && inpos) ? __ldg(p.slot_table + kvo + pos[r]) : -1;
                else if (!inpos) slot[r] = -1;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int i = base + r * 32 + lane;
                if (i < n) {
                    int s = slot[r];
                    if (pos[r] >= 0 && pos[r] < ri.len && (s < 0 || (long long)s >= p.num_slots)) {
                        bad |= PILLAR_FLAG_SLOT;
                        s = -1;
                    }
                    rows[i] = s;
                }
            }
        }
        if (bad) atomicOr(c.err, bad);
        if (lane == 0) {
            ItemInfo info;
            info.it = it;
            info.mode = ri.mode;
            info.b = b;
            info.g = g;
            info.n = n;
            info.begin = itm.begin;
            info.q_off = ri.q_off;
            info.vidx = ri.vidx;
            info.L = ri.len;
            info.nsplit = ui.nsplit;
            info.split = itm.split;
            info.rec = ui.rec_base + itm.split * ui.rec_rows;
            info.logit_off = lgo;
            info.kv_off = kvo;
            c.iinfo[rb] = info;
        }
        mbar_arrive(&c.rfull[rb]);  // every lane: releases its own row-list writes
    }
}

// L2 cache policy: lines of a single-use stream, evicted before other lines.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_gather4 with an L2 cache policy for the rows it reads.
__device__ __forceinline__ void tma_gather4_hint(void *dst, const void *tmap, int col, int r0, int r1, int r2, int r3,
                                                 uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// mbar_wait for the loader warps: the first test inline, the bounded polling out of line (a
// function of their own: one called from warps at different register counts does not allocate;
// measured on back-to-back steps, -0.5 us on the Qwen3-8B shape and -1.7 us on the stress batch,
// while the same for the epilogue warps as well cost +9 us).
__device__ __noinline__ bool mbar_wait_poll80(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                                              unsigned long long limit_ns) {
    return mbar_wait(bar, parity, abort, err, limit_ns);
}
__device__ __forceinline__ bool mbar_wait_80(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                                             unsigned long long limit_ns) {
    return mbar_try_wait(bar, parity) || mbar_wait_poll80(bar, parity, abort, err, limit_ns);
}

// ============================================================== loader warps

// The loader warps share every tile: warp li fetches rows [RW li, RW li + RW),
// RW = 64 / kLoaderWarps, of K and of V by TMA tile::gather4 (four rows per
// copy, each lane issuing its own) into the 128-byte-swizzled layout the
// tensor cores read, split in 64-column halves; each announces its bytes on
// the stage barrier.  All loaders run the same deterministic sequence and
// share the query rows of an item's first tile (16-byte cp.async); loader 0
// writes the stage record.
template <int D>
__device__ void loader(const AttnParams &p, const Ctx &c, int lane, int li) {
    using S = Smem<D>;
    constexpr int NH = D / 64;                  // 64-column halves of a row
    constexpr int RW = kTileKeys / kLoaderWarps;  // rows of a tile per loader warp
    constexpr int GW = RW / 4;                  // gather4 row groups per loader warp
    static_assert(GW * 2 * NH <= 32, "one gather4 per lane");
    int stage = 0, qn = 0;
    uint32_t phase = 0, qph = 0, fph = 0, issued = 0, issued_par = 0;
    bool ok = true;
    // this lane's gather4: row group rgl of the warp's rows, K (kv 0) or V (kv 1), column half h.
    // The column halves of a row group go to adjacent lanes, so the two 128-byte halves of each
    // 256-byte row are requested back to back and reach DRAM as one access (halves requested
    // apart behave as random 128-byte reads, which DRAM serves far below its copy rate).
    const int h = lane % NH, kv = (lane / NH) & 1, rgl = lane / (2 * NH);
    const bool gl = rgl < GW;
    // K and V rows are read once: evicted first, so that the verify logits written meanwhile
    // are still in L2 when the Top-K pass reads them
    const uint64_t kv_policy = l2_evict_first_policy();
    for (int rb = 0;; rb = rb + 1 == kRowLists ? 0 : rb + 1) {
        ok = mbar_wait_80(&c.rfull[rb], (fph >> rb) & 1, c.abort, c.err, c.wait_ns);
        if (!ok) break;
        fph ^= 1u << rb;
        const ItemInfo info = c.iinfo[rb];
        if (info.it < 0) {
            ok = mbar_wait_80(&c.empty[stage], phase ^ 1, c.abort, c.err, c.wait_ns);
            if (ok) {
                cp_async_arrive_noinc(&c.full[stage]);
                __syncwarp();
                if (lane == 0) {
                    if (li == 0) c.meta[stage].flags = kStop;
                    mbar_arrive(&c.full[stage]);
                }
            }
            break;
        }
        const int *rows = c.rowlist + rb * kMaxChunk;
        const bool verify = info.mode == 1;
        const int n = info.n, g = info.g;
        const int ntiles = n > 0 ? (n + kTileKeys - 1) / kTileKeys : 1;
        const int qb = qn & 1;  // two query buffers: this item's may still hold the one before last
        ++qn;
        for (int t = 0; t < ntiles; ++t) {
            ok = mbar_wait_80(&c.empty[stage], phase ^ 1, c.abort, c.err, c.wait_ns);
            if (!ok) break;
            if (t == 0) {  // every loader writes query rows: the buffer's previous item must be done with it
                ok = mbar_wait_80(&c.qempty[qb], ((qph >> qb) & 1) ^ 1, c.abort, c.err, c.wait_ns);
                if (!ok) break;
                qph ^= 1u << qb;
            }
            const int k0 = t * kTileKeys;
            const int nk = max(0, min(kTileKeys, n - k0));
            const int r0 = lane < nk ? rows[k0 + lane] : -1;
            const int r1 = lane + 32 < nk ? rows[k0 + lane + 32] : -1;
            const unsigned v0 = __ballot_sync(0xffffffffu, r0 >= 0);
            const unsigned v1 = __ballot_sync(0xffffffffu, r1 >= 0);
            const unsigned long long valid = ((unsigned long long)v1 << 32) | v0;
            if (lane == 0) {
                if (li == 0) {  // the stage record
                    StageMeta &m = c.meta[stage];
                    if (t == 0) m.info = info;
                    m.nk = nk;
                    m.flags = (t == 0 ? kFirst : 0) | (t == ntiles - 1 ? kLast : 0);
                    m.pos0 = verify ? info.begin + k0 : 0;
                    m.qb = qb;
                    m.valid = valid;
                    m.mode = info.mode;
                }
                mbar_arrive_expect_tx(&c.full[stage], valid ? (uint32_t)(RW * D * 2 * 2) : 0u);  // this warp's rows of K and V
            }
            __syncwarp();
            if (valid) {
                // Keys that are invalid or past the tail still get a real row (the
                // first valid key's): every staged row then holds finite pool data
                // and a zero probability can never meet a NaN.
                const int f = __ffsll((long long)valid) - 1;
                const int fb = __shfl_sync(0xffffffffu, f < 32 ? r0 : r1, f & 31);
                const int sown = (RW * li < 32) ? (r0 >= 0 ? r0 : fb) : (r1 >= 0 ? r1 : fb);
                int rr[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = RW * li + 4 * rgl + e;  // the warp's rows lie on one side of 32
                    rr[e] = __shfl_sync(0xffffffffu, sown, i & 31) * p.Hkv + g;
                }
                if (gl) {
                    char *dst = c.smem + S::off_stage + stage * S::STAGE + kv * S::ROWS + h * (kTileKeys * 128) +
                                (RW * li + 4 * rgl) * 128;
                    tma_gather4_hint(dst, kv ? (const void *)&p.tmap_v : (const void *)&p.tmap_k, 64 * h, rr[0], rr[1],
                                     rr[2], rr[3], &c.full[stage], kv_policy);
                }
            }
            if (t == 0) {  // query rows into their operand slots (core-matrix layout), shared by the loaders
                char *qreg = c.smem + S::off_q + qb * S::QHALF;
                const int nchunks = (verify ? p.M : p.G) * S::KCH;
                const int rq = verify ? p.RQ : p.RQd;
                for (int i = li * 32 + lane; i < nchunks; i += 32 * kLoaderWarps) {
                    const int r = i / S::KCH, cc = i - r * S::KCH;
                    const int j = verify ? r / p.G : 0, gi = r - j * p.G;
                    const int a = row_slot(r, rq);
                    cp_async16(qreg + (a >> 3) * S::CORE_SBO + cc * 128 + (a & 7) * 16,
                               p.q + ((size_t)(info.q_off + j) * p.Hq + (size_t)g * p.G + gi) * D + cc * 8);
                }
            }
            cp_async_arrive_noinc(&c.full[stage]);  // lands with this lane's query copies (if any)
            issued |= 1u << stage;
            issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
            if (++stage == S::NSTAGE) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (!ok) break;
        __syncwarp();
        mbar_arrive(&c.rempty[rb]);  // every lane is done reading this row list
    }
    if (!ok) {
        // Let every copy this warp started land before the CTA can exit.
        for (int s2 = 0; s2 < S::NSTAGE; ++s2)
            if ((issued >> s2) & 1) drain_wait(&c.full[s2], (issued_par >> s2) & 1);
    }
}

// ============================================================== MMA warp

// One thread issues every tensor-core operation of the CTA.  It walks the
// stage ring in order and keeps two cursors: vs, the next tile whose
// S = Q K^T to issue (needs the tile landed and its S buffer released by the
// P V four tiles back), and vp, the next tile whose O += P V to issue (needs
// the softmax's P, and for an item's first tile its O columns read out by the
// epilogue two items back).
// Both are polled with non-blocking tests, so neither waits behind the other.
template <int D>
__device__ void mma_issuer(const AttnParams &p, const Ctx &c, uint32_t tbase) {
    using S = Smem<D>;
    constexpr uint32_t idS = umma_idesc_bf16(64, kTileKeys, 0, 0);  // M = 64 query-row slots
    constexpr uint32_t idO = umma_idesc_bf16(64, D, 0, 1);
    const uint32_t sq0 = smem_u32(c.smem + S::off_q);
    int stage = 0;
    uint32_t phase = 0, vs = 0, vp = 0;
    uint32_t ocount0 = 0, ocount1 = 0;  // items finished per query buffer (scalars: no local-memory array)
    bool stopped = false, started = false, issued = false;
    unsigned long long t_idle = 0;
    for (uint32_t spin = 0;; ++spin) {
        bool progress = false;
        if (!stopped && vs - vp < (uint32_t)kSBuf && mbar_test_wait(&c.full[stage], phase)) {
            const StageMeta &m = c.meta[stage];
            const int flags = m.flags;
            bool advance = false;
            if (flags & kStop) {
                stopped = true;
            } else {
                const uint32_t sb = vs % kSBuf;
                if (mbar_test_wait(&c.s_free[sb], ((vs / kSBuf) & 1) ^ 1)) {
                    fence_proxy_async_smem();  // cp.async data seen through the stage barrier -> tensor-core reads
                    tc_fence_after();
                    const int qb = m.qb;
                    const int valid = m.valid != 0ull;
                    if (valid) {
                        const uint32_t sk = smem_u32(c.smem + S::off_stage + stage * S::STAGE);
                        const uint32_t sq = sq0 + qb * S::QHALF;
                        // descriptors advance by start address (16-byte units): Q 256 B per K step,
                        // K 32 B per K step inside a 64-column half of 8 KB
                        const uint64_t da = umma_sdesc(sq, 128, S::CORE_SBO), db = umma_sdesc_sw128(sk, 16, 1024);
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks)
                            umma_bf16(tbase + sb * kTileKeys, da + (uint64_t)(ks * 16),
                                      db + (uint64_t)((ks >> 2) * (kTileKeys * 8) + (ks & 3) * 2), idS, ks > 0 ? 1u : 0u);
                    }
                    umma_commit(&c.s_full[sb]);
                    if (flags & kLast) {  // the item's query rows are free once its last S has completed
                        mbar_arrive_cnt(&c.qempty[qb], kConsumerWarps - 1);
                        umma_commit(&c.qempty[qb]);
                    }
                    c.pend[sb] = make_int4(stage, qb, flags, valid);  // (shared memory: no local-memory stack)
                    ++vs;
                    issued = true;
                    advance = true;
                }
            }
            if (advance && ++stage == S::NSTAGE) {
                stage = 0;
                phase ^= 1;
            }
            progress = advance || stopped;
        }
        if (vp < vs) {
            const uint32_t sb = vp % kSBuf;
            const int4 pe = c.pend[sb];  // stage, query buffer, flags, valid of the tile
            const int e_stage = pe.x, e_qb = pe.y, e_flags = pe.z, e_valid = pe.w;
            bool ready = mbar_test_wait(&c.p_full[sb], (vp / kSBuf) & 1);
            if (ready && (e_flags & kFirst))
                ready = mbar_test_wait(&c.o_free[e_qb], ((e_qb ? ocount1 : ocount0) & 1) ^ 1);
            if (ready) {
                tc_fence_after();
                if (e_valid) {
                    const uint32_t sv = smem_u32(c.smem + S::off_stage + e_stage * S::STAGE + S::ROWS);
                    const uint32_t tO = tbase + S::tO + (uint32_t)e_qb * D;
                    const uint64_t dv = umma_sdesc_sw128(sv, kTileKeys * 128, 1024);
#pragma unroll
                    for (int ks = 0; ks < kTileKeys / 16; ++ks)  // V: 16 keys = two 8-key atoms = 2048 B
                        umma_bf16_ts(tO, tbase + sb * kTileKeys + ks * 8, dv + (uint64_t)(ks * 128), idO,
                                     (started || ks > 0) ? 1u : 0u);
                    started = true;
                }
                umma_commit(&c.s_free[sb]);      // S/P buffer free, and the O of this tile final
                umma_commit(&c.empty[e_stage]);  // K and V rows consumed
                if (e_flags & kLast) {
                    umma_commit(&c.o_done[e_qb]);  // the item's O is final: its epilogue may read it
                    started = false;
                    if (e_qb) ++ocount1; else ++ocount0;
                }
                ++vp;
                progress = true;
            }
        }
        if (stopped && vp == vs) break;
        if (progress) {
            t_idle = 0;
            continue;
        }
        __nanosleep(20);  // idle: leave the issue slots to the warps sharing this sub-partition
        if ((spin & 63) == 0) {
            if (*c.abort) break;
            const unsigned long long now = global_timer_ns();
            if (t_idle == 0) {
                t_idle = now;
            } else if (now - t_idle > c.wait_ns) {
                atomicOr(c.err, PILLAR_FLAG_TIMEOUT);
                *c.abort = 1;
                break;
            }
        }
    }
    if (issued) {  // every MMA issued has completed before the tensor memory can be freed
        umma_commit(c.drain);
        drain_wait(c.drain, 0);
    }
}

// ============================================================== consumer warps

// Consumer state that persists across items.
struct CState {
    int stage;
    uint32_t phase;
    uint32_t vt;      // tiles this CTA has processed (selects S buffers and barrier parities)
    uint32_t tbase;   // TMEM base address
    uint32_t items;   // items handed to the epilogue warp (their mailbox slot alternates)
};

// The softmax warps' code is kept small: their loop slows with every instruction it holds, taken
// or not (instruction-fetch stalls; measured on the Qwen3-8B-shaped step, where the rare paths
// below moved out of line, the visibility test made one 64-bit mask applied after one multiply
// path and the division moved to the epilogue warps took the step from 202.7 to 197.2 us).
// Hence mbar_wait for these warps: the first test inline, the bounded polling out of line.
__device__ __noinline__ bool mbar_wait_poll(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                                            unsigned long long limit_ns) {
    return mbar_wait(bar, parity, abort, err, limit_ns);
}
__device__ __forceinline__ bool mbar_wait_c(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                                            unsigned long long limit_ns) {
    return mbar_try_wait(bar, parity) || mbar_wait_poll(bar, parity, abort, err, limit_ns);
}

// Hands the next mailbox slot of this warp's quadrant to its epilogue warp
// (waiting, bounded, for the slot to have been taken two records back).
__device__ __forceinline__ bool post_epilogue(const Ctx &c, int warp, int lane, CState &cs, const EpiRec &e, float2 l) {
    const int slot = warp * 2 + (int)(cs.items & 1);
    const uint32_t use = cs.items >> 1;  // earlier uses of this slot
    if (!mbar_wait_c(&c.epi_empty[slot], (use & 1) ^ 1, c.abort, c.err, c.wait_ns)) return false;
    if (lane == 0) c.epi[slot] = e;
    c.epi_l[slot * 32 + lane] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.epi_full[slot]);
    ++cs.items;
    return true;
}

constexpr float kRescaleLog2 = 8.f;  // O is rescaled once a row maximum has grown by more than 2^8

// One query row of an item as seen by one of the four threads that share it.
struct VRow {
    bool act;
    int row, j, gi, lim;
    long long lb;   // offset of the row's logits at position 0 (verify)
    float m, l;     // reference maximum of P, and the sum of this thread's probabilities
};

// Row i of the warp's quadrant: verify row r = j*G + gi sees positions up to
// L-(k+1)+j; a draft row r = gi sees every listed position.
__device__ __forceinline__ VRow item_row(const AttnParams &p, const ItemInfo &in, bool verify, int warp, int i) {
    VRow r;
    const int rq = verify ? p.RQ : p.RQd;
    r.row = warp * rq + i;
    r.act = i < rq && r.row < (verify ? p.M : p.G);
    r.j = 0;
    r.gi = r.row;
    r.lim = 0x7fffffff;
    r.lb = 0;
    r.m = neg_inf();
    r.l = 0.f;
    if (r.act && verify) {
        const int kk1 = p.k + 1;
        int j = 0, gi = r.row;  // row / G by subtraction (at most k+1 steps; less code than a division)
        while (gi >= p.G) gi -= p.G, ++j;
        r.j = j;
        r.gi = gi;
        r.lim = in.L - kk1 + r.j;
        r.lb = in.logit_off + ((long long)(in.g * p.G + r.gi) * kk1 + r.j) * in.L;
    }
    return r;
}

// This thread's 16 scores of one row (chunk c, pair e <-> key 8c + cq + e,
// held in s[4c + OFF + e]): scale, mask, dump the logits of verify rows;
// returns their max.
template <int OFF>
__device__ __forceinline__ float row_scores(const AttnParams &p, const StageMeta &cur, const VRow &r, float *s, int cq,
                                            bool verify) {
    if (!r.act) return neg_inf();
    // the row's visible keys of the tile: listed with a valid slot (the valid mask has no bit at or
    // past nk) and, for a verify row, at or before its causal limit
    const int span = r.lim - cur.pos0;
    const unsigned long long vis = cur.valid & (span >= 63 ? ~0ull : span < 0 ? 0ull : (2ull << span) - 1);
    const float2 sc = make_float2(p.scale, p.scale);
#pragma unroll
    for (int c = 0; c < 8; ++c) {  // packed pairs: one fp32x2 multiply per two scores
        const float2 v = fmul2(make_float2(s[4 * c + OFF], s[4 * c + OFF + 1]), sc);
        s[4 * c + OFF] = v.x;
        s[4 * c + OFF + 1] = v.y;
    }
    if (vis != ~0ull) {  // keys this row does not see
        const unsigned long long m = vis >> cq;
#pragma unroll
        for (int c = 0; c < 8; ++c)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                if (!((m >> (8 * c + e)) & 1ull)) s[4 * c + OFF + e] = neg_inf();
    }
    // maximum as a tree (short dependency chains)
    float m8[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) m8[c] = fmaxf(s[4 * c + OFF], s[4 * c + OFF + 1]);
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int c = 0; c < w; ++c) m8[c] = fmaxf(m8[c], m8[c + w]);
    const float mt = m8[0];
    if (!verify) return mt;
    // the row's four threads write 8 consecutive positions per chunk
    float *dst = p.logits + r.lb + cur.pos0 + cq;
    if (cur.nk == kTileKeys && ((r.lb + cur.pos0) & 1) == 0) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float2 *>(dst + 8 * c) = make_float2(s[4 * c + OFF], s[4 * c + OFF + 1]);
    } else {  // a row that starts on an odd float, or the keys of a partial tile: one float at a time
        const int lim = cur.nk - cq;
#pragma unroll
        for (int c = 0; c < 8; ++c)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                if (8 * c + e < lim) dst[8 * c + e] = s[4 * c + OFF + e];
    }
    return mt;
}

// Probabilities of one row as bf16 pairs (P column 4c + t%4 <-> keys 8c + cq, +1).
template <int OFF>
__device__ __forceinline__ void row_probs(VRow &r, const float *s, uint32_t *pw) {
    if (r.act) {
        const float nb = -(r.m == neg_inf() ? 0.f : r.m) * kLog2e;
        const float2 k2 = make_float2(kLog2e, kLog2e), b2 = make_float2(nb, nb);
        float2 l4[4];
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // packed pairs: exponent arguments and sums two at a time
            const float2 a = ffma2(make_float2(s[4 * c + OFF], s[4 * c + OFF + 1]), k2, b2);
            const float2 pe = make_float2(ex2_approx(a.x), ex2_approx(a.y));
            l4[c & 3] = c < 4 ? pe : fadd2(l4[c & 3], pe);
            pw[2 * c + OFF / 2] = pack_bf16x2(pe.x, pe.y);
        }
        const float2 l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
        r.l += l2.x + l2.y;
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) pw[2 * c + OFF / 2] = 0u;
    }
}

// The normalised output of one row from this thread's O columns (c0 + 8c + cq, +1).
template <int D, int OFF>
__device__ __forceinline__ void row_output(const AttnParams &p, const ItemInfo &in, const VRow &r, const float *ov, int c0,
                                           int cq, float inv) {
    if (!r.act) return;
    if (in.nsplit == 1) {
        uint16_t *dst = p.out + ((size_t)(in.q_off + r.j) * p.Hq + (size_t)in.g * p.G + r.gi) * D + c0 + cq;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint32_t *>(dst + 8 * c) = pack_bf16x2(ov[4 * c + OFF] * inv, ov[4 * c + OFF + 1] * inv);
    } else {
        float *dst = p.part_o + ((size_t)in.rec + r.row) * D + c0 + cq;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float2 *>(dst + 8 * c) = make_float2(ov[4 * c + OFF] * inv, ov[4 * c + OFF + 1] * inv);
    }
}

// Scales this thread's two O rows by aa (row A) and ab (row B) after a running maximum grew by
// more than 2^8 (rare; out of line).
template <int D>
__device__ __noinline__ bool rescale_o(uint64_t *sfree, uint32_t par, volatile int *abort, int *err,
                                       unsigned long long wait_ns, uint32_t taddr, float aa, float ab) {
    // O holds this item's earlier tiles (a grow needs one): the last P V must have completed
    if (!mbar_wait(sfree, par, abort, err, wait_ns)) return false;
    tc_fence_after();
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 64) {
        float ov[32];
        tmem_ld16x256b_x8(taddr + c0, ov);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            ov[4 * q] *= aa;
            ov[4 * q + 1] *= aa;
            ov[4 * q + 2] *= ab;
            ov[4 * q + 3] *= ab;
        }
        tmem_st16x256b_x8(taddr + c0, ov);
    }
    return true;
}

// A row's LSE from its running maximum and sum (once per item; out of line).
__device__ __noinline__ void put_lse(float *dst, float m, float l) { *dst = l > 0.f ? m + logf(l) : neg_inf(); }

// The consumer side of an item.  The warp reads lanes 0-15 of
// its TMEM quadrant with the 16x256b shape: each row (lane) is shared by four
// threads, sixteen columns each; thread t holds rows t/4 ("A") and 8 + t/4
// ("B", present when a quadrant holds more than eight rows).
template <int D>
__device__ bool attn_item(const AttnParams &p, const Ctx &c, int warp, int lane, CState &cs, StageMeta cur) {
    using S = Smem<D>;
    const ItemInfo in = cur.info;
    const bool verify = in.mode == 1;
    const int qb = cur.qb;
    const int cq = 2 * (lane & 3);
    VRow ra = item_row(p, in, verify, warp, lane >> 2);
    VRow rb = item_row(p, in, verify, warp, 8 + (lane >> 2));
    const bool have_b = (verify ? p.RQ : p.RQd) > 8;  // warp-uniform
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;  // lanes 0-15 of the warp's quadrant (M = 64)
    const uint32_t tO = cs.tbase + S::tO + (uint32_t)qb * D;
    uint32_t last_vt = 0;

    for (;;) {
        const uint32_t vt = cs.vt, sb = vt % kSBuf;
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.empty[cs.stage]);  // the stage is read by the tensor cores only
        if (!mbar_wait_c(&c.s_full[sb], (vt / kSBuf) & 1, c.abort, c.err, c.wait_ns)) return false;
        tc_fence_after();
        const uint32_t tS = cs.tbase + sb * kTileKeys;
        float s[32];
        tmem_ld16x256b_x8(tS + lane_base, s);
        float mta = row_scores<0>(p, cur, ra, s, cq, verify);
        float mtb = have_b ? row_scores<2>(p, cur, rb, s, cq, verify) : neg_inf();
        mta = fmaxf(mta, __shfl_xor_sync(0xffffffffu, mta, 1));
        mta = fmaxf(mta, __shfl_xor_sync(0xffffffffu, mta, 2));
        if (have_b) {
            mtb = fmaxf(mtb, __shfl_xor_sync(0xffffffffu, mtb, 1));
            mtb = fmaxf(mtb, __shfl_xor_sync(0xffffffffu, mtb, 2));
        }
        // running maxima: rescale O only when one grows by more than 2^8
        const float mna = fmaxf(ra.m, mta), mnb = fmaxf(rb.m, mtb);
        const bool grow_a = ra.act && ra.m != neg_inf() && (mna - ra.m) * kLog2e > kRescaleLog2;
        const bool grow_b = rb.act && rb.m != neg_inf() && (mnb - rb.m) * kLog2e > kRescaleLog2;
        float aa = 1.f, ab = 1.f;  // rescale factors, computed only on the rare growth
        if (grow_a) {
            aa = exp2f((ra.m - mna) * kLog2e);
            ra.l *= aa;
            ra.m = mna;
        }
        if (grow_b) {
            ab = exp2f((rb.m - mnb) * kLog2e);
            rb.l *= ab;
            rb.m = mnb;
        }
        if (ra.act && ra.m == neg_inf()) ra.m = mna;  // first visible keys of the row
        if (rb.act && rb.m == neg_inf()) rb.m = mnb;
        // P (bf16 pairs) over the scores, for the P V MMA
        uint32_t pw[16];
        row_probs<0>(ra, s, pw);
        if (have_b) {
            row_probs<2>(rb, s, pw);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) pw[2 * q + 1] = 0u;
        }
        if (__any_sync(0xffffffffu, grow_a || grow_b)) {
            const uint32_t pv = vt - 1;
            if (!rescale_o<D>(&c.s_free[pv % kSBuf], (pv / kSBuf) & 1, c.abort, c.err, c.wait_ns, tO + lane_base, aa, ab))
                return false;
        }
        tmem_st16x128b_x8(tS + lane_base, pw);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.p_full[sb]);
        last_vt = vt;
        cs.vt = vt + 1;
        const bool last = cur.flags & kLast;
        if (++cs.stage == S::NSTAGE) {
            cs.stage = 0;
            cs.phase ^= 1;
        }
        if (last) break;
        if (!mbar_wait_c(&c.full[cs.stage], cs.phase, c.abort, c.err, c.wait_ns)) return false;
        cur = c.meta[cs.stage];
    }

    // epilogue: row sums and LSEs first, then the O rows once the item's last P V has completed
    ra.l += __shfl_xor_sync(0xffffffffu, ra.l, 1);
    ra.l += __shfl_xor_sync(0xffffffffu, ra.l, 2);
    rb.l += __shfl_xor_sync(0xffffffffu, rb.l, 1);
    rb.l += __shfl_xor_sync(0xffffffffu, rb.l, 2);
    if ((lane & 3) == 0 && (verify || in.nsplit > 1)) {
        const int kk1 = p.k + 1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const VRow &r = h ? rb : ra;
            if (!r.act) continue;
            put_lse(in.nsplit == 1 ? p.lse + ((size_t)in.vidx * p.Hq + (size_t)in.g * p.G + r.gi) * kk1 + r.j
                                   : p.part_lse + (size_t)in.rec + r.row,
                    r.m, r.l);
        }
    }
    // the O rows are written by the epilogue warp of this quadrant once the item's last P V has
    // completed; this warp goes on with the next item
    (void)last_vt;
    EpiRec e;
    e.mode = in.mode;
    e.g = in.g;
    e.q_off = in.q_off;
    e.nsplit = in.nsplit;
    e.rec = in.rec;
    e.qb = qb;
    e.stop = 0;
    e.pad = 0;
    return post_epilogue(c, warp, lane, cs, e, make_float2(ra.l, rb.l));
}

// The epilogue warp of quadrant q: for each item of the consumer warp of its
// quadrant, in order, wait until the item's last P V has completed, read its
// O columns, normalise, write the rows (or the partial record of a split
// item) and release the columns.
template <int D>
__device__ void epilogue_warp(const AttnParams &p, const Ctx &c, int q, int lane, uint32_t tbase) {
    using S = Smem<D>;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;  // lanes 0-15 of quadrant q (M = 64)
    const int cq = 2 * (lane & 3);
    uint32_t odone = 0;  // bit b: parity of O buffer b's next completion
    for (uint32_t n = 0;; ++n) {
        const int slot = q * 2 + (int)(n & 1);
        if (!mbar_wait(&c.epi_full[slot], (n >> 1) & 1, c.abort, c.err, c.wait_ns)) break;
        const EpiRec e = c.epi[slot];
        const float2 l = c.epi_l[slot * 32 + lane];  // (the division is done here, off the softmax warps' code)
        const float2 inv = make_float2(l.x > 0.f ? 1.f / l.x : 0.f, l.y > 0.f ? 1.f / l.y : 0.f);
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.epi_empty[slot]);  // the record is copied: the slot may be reused
        if (e.stop) break;
        if (!mbar_wait(&c.o_done[e.qb], (odone >> e.qb) & 1, c.abort, c.err, c.wait_ns)) break;
        odone ^= 1u << e.qb;
        tc_fence_after();
        ItemInfo in;
        in.mode = e.mode;
        in.g = e.g;
        in.q_off = e.q_off;
        in.nsplit = e.nsplit;
        in.rec = e.rec;
        in.L = 0;  // (row limits and logit offsets are not used here)
        in.logit_off = 0;
        const bool verify = e.mode == 1;
        const VRow ra = item_row(p, in, verify, q, lane >> 2);
        const VRow rb = item_row(p, in, verify, q, 8 + (lane >> 2));
        const bool have_b = (verify ? p.RQ : p.RQd) > 8;
        const uint32_t tO = tbase + S::tO + (uint32_t)e.qb * D;
#pragma unroll 1  // (rolled: less code beside the softmax warps' on each sub-partition)
        for (int c0 = 0; c0 < D; c0 += 64) {
            float ov[32];
            tmem_ld16x256b_x8(tO + lane_base + c0, ov);  // warp-collective: every lane loads
            row_output<D, 0>(p, in, ra, ov, c0, cq, inv.x);
            if (have_b) row_output<D, 2>(p, in, rb, ov, c0, cq, inv.y);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.o_free[e.qb]);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(c.cexit);
}

template <int D>
__device__ void consumer(const AttnParams &p, const Ctx &c, int warp, int lane, uint32_t tbase) {
    CState cs;
    cs.stage = 0;
    cs.phase = 0;
    cs.vt = 0;
    cs.tbase = tbase;
    cs.items = 0;
    for (;;) {
        if (!mbar_wait_c(&c.full[cs.stage], cs.phase, c.abort, c.err, c.wait_ns)) break;
        const StageMeta m = c.meta[cs.stage];
        if (m.flags & kStop) break;
        if (!attn_item<D>(p, c, warp, lane, cs, m)) break;
    }
    EpiRec stop = {};
    stop.stop = 1;
    post_epilogue(c, warp, lane, cs, stop, make_float2(0.f, 0.f));  // (returns at once on an abort)
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(c.cexit);
}

// ============================================================== kernel

// Per-warp-group register reallocation (every warp of the group executes it).
template <uint32_t R>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <uint32_t R>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) unified_attn_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ __align__(1024) char smem[];
    using S = Smem<D>;
    const Ctx c = make_ctx<D>(smem, p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S::NSTAGE; ++s) {
            mbar_init(&c.full[s], kLoaderWarps * 33);  // per loader: a byte-count arrival + its lanes' query-copy arrivals
            mbar_init(&c.empty[s], kConsumerWarps + 1);    // one per consumer warp + the MMA thread
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&c.qempty[i], kConsumerWarps);
            mbar_init(&c.o_free[i], kConsumerWarps);
        }
        for (int i = 0; i < kRowLists; ++i) {
            mbar_init(&c.rfull[i], 32);
            mbar_init(&c.rempty[i], kLoaderWarps * 32);
        }
        for (int i = 0; i < kSBuf; ++i) {
            mbar_init(&c.s_full[i], 1);
            mbar_init(&c.s_free[i], 1);
            mbar_init(&c.p_full[i], kConsumerWarps);
        }
        mbar_init(c.cexit, kConsumerWarps + 1 + kEpiWarps);
        mbar_init(c.drain, 1);
        for (int i = 0; i < 2; ++i) mbar_init(&c.o_done[i], 1);
        for (int i = 0; i < 2 * kEpiWarps; ++i) {
            mbar_init(&c.epi_full[i], 1);
            mbar_init(&c.epi_empty[i], 1);
        }
        *c.abort = 0;
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(c.tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *c.tmem_slot;
    // Everything above is private to the CTA; the plan's output is read only from here on.
    pdl_wait_prerequisites();
    pdl_launch_dependents();  // the merge kernel waits for this kernel's completion itself
    // Registers move to the softmax warps: the CTA is launched with 128 per thread; the
    // other three warp groups drop to 80 and the softmax group rises to 232
    // (4*128*128 = 65536 >= 128*232 + 3*128*80 = 60416).
    const int wg = warp >> 2;
    if (wg == 0) {
        regs_increase<232>();
        consumer<D>(p, c, warp, lane, tbase);
    } else if (wg == 1) {
        regs_decrease<80>();
        loader<D>(p, c, lane, warp - kConsumerWarps);
    } else if (wg == 2) {
        regs_decrease<80>();
        if (warp == 8) {
            resolver(p, c, lane);
        } else if (warp == 9) {
            if (lane == 0) {
                mma_issuer<D>(p, c, tbase);
                tc_fence_before();
                mbar_arrive(c.cexit);
            }
            __syncwarp();
        }
    } else {
        regs_decrease<80>();
        epilogue_warp<D>(p, c, warp - 12, lane, tbase);
    }
    if (warp == 0) {  // the consumers and the MMA thread are done with the tensor memory (bounded wait), then free it
        drain_wait(c.cexit, 0);
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// ============================================================== merge of partials

constexpr int kMergeThreads = 1024;
constexpr int kMergeBatch = 4;     // records whose loads are in flight together
constexpr int kMergeCtasPerSm = 1;  // one large CTA per SM: the whole grid is resident when the attention kernel ends

// Combines the partial rows of every split (request, KV head).  A split unit
// has nrec records of nrows rows (M for verify, G for draft); the work is
// flattened over (listed unit, row, four output dimensions), one thread each,
// so that few, long units still spread over the whole GPU: the verify units
// (listed from the bottom of the merge list) with M rows each, then the
// draft units (listed from the top) with their G rows.  The planner's
// MergeUnit record holds everything a task needs, so a thread loads the unit
// counts, its record, and then all its partials at once.  A thread merges its records in batches, carrying a running
// max and sums between batches.
template <int D>
__global__ void __launch_bounds__(kMergeThreads, kMergeCtasPerSm) merge_kernel(const AttnParams p) {
    pdl_wait_prerequisites();  // the partials come from the attention kernel
    // the attention kernel is complete: its work queue is reset for the next run on the same plan
    if (blockIdx.x == 0 && threadIdx.x == 0) p.hdr->item_counter = 0;
    constexpr int C4 = D / 4;
    const int vslot = p.M * C4, dslot = p.G * C4;  // thread slots of a verify unit, of a draft unit
    const int nv = p.hdr->num_merge, nd = p.hdr->num_merge_draft, U = p.hdr->num_units;
    const long long vtotal = (long long)nv * vslot, total = vtotal + (long long)nd * dslot;
    for (long long w = (long long)blockIdx.x * kMergeThreads + threadIdx.x; w < total;
         w += (long long)gridDim.x * kMergeThreads) {
        int li, idx;
        if (w < vtotal) {
            li = (int)(w / vslot);
            idx = (int)(w - (long long)li * vslot);
        } else {
            const long long w2 = w - vtotal;
            const int k = (int)(w2 / dslot);
            idx = (int)(w2 - (long long)k * dslot);
            li = U - 1 - k;
        }
        const MergeUnit mu = p.merge_units[li];
        const int row = idx / C4, c4 = idx - row * C4;
        const float *pl = p.part_lse + (size_t)mu.rec_base + row;
        const float4 *po = reinterpret_cast<const float4 *>(p.part_o + ((size_t)mu.rec_base + row) * D) + c4;
        const size_t so = (size_t)mu.nrows * C4;
        float mx = neg_inf(), den = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r0 = 0; r0 < mu.nrec; r0 += kMergeBatch) {
            float ls[kMergeBatch];
            float4 v[kMergeBatch];
#pragma unroll
            for (int q = 0; q < kMergeBatch; ++q) {
                const int r = r0 + q;
                if (r < mu.nrec) {
                    ls[q] = __ldcg(pl + (size_t)r * mu.nrows);
                    v[q] = __ldcg(po + r * so);
                } else {
                    ls[q] = neg_inf();
                    v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            float bm = mx;
#pragma unroll
            for (int q = 0; q < kMergeBatch; ++q) bm = fmaxf(bm, ls[q]);
            if (bm == neg_inf()) continue;
            const float a = ex2_approx((mx - bm) * kLog2e);  // rescale what was merged so far (0 when empty)
            den *= a;
            o = make_float4(o.x * a, o.y * a, o.z * a, o.w * a);
#pragma unroll
            for (int q = 0; q < kMergeBatch; ++q) {
                const float wq = ex2_approx((ls[q] - bm) * kLog2e);
                den += wq;
                o.x += wq * v[q].x;
                o.y += wq * v[q].y;
                o.z += wq * v[q].z;
                o.w += wq * v[q].w;
            }
            mx = bm;
        }
        float lse = neg_inf();
        if (den > 0.f) {
            const float inv = 1.f / den;
            o = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
            lse = mx + logf(den);
        }
        const int j = mu.verify ? row / p.G : 0, gi = row - j * p.G;
        const long long orow = mu.orow0 + (long long)j * p.Hq + gi;
        uint2 pk;
        pk.x = pack_bf16x2(o.x, o.y);
        pk.y = pack_bf16x2(o.z, o.w);
        *reinterpret_cast<uint2 *>(p.out + orow * D + 4 * c4) = pk;
        if (mu.verify && c4 == 0) p.lse[mu.lse0 + (long long)gi * (p.k + 1) + j] = lse;
    }
}

// ------------------------------------------------------------------ host-side launch helpers

template <int D>
cudaError_t launch_unified_t(const AttnParams &p, int nsm, cudaStream_t st) {
    // launch attributes, once per device context
    static unsigned long long configured[kMaxDevices] = {};
    int dev = 0;
    unsigned long long ctx = 0;
    cudaError_t e = current_device_context(&dev, &ctx);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (ctx == 0 || __atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE) != ctx) {
        e = cudaFuncSetAttribute(unified_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<D>::total);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, unified_attn_kernel<D>, kThreads, Smem<D>::total);
        if (e != cudaSuccess) return e;
        // exactly one CTA per SM: it allocates all of the SM's tensor memory
        if (n != 1) return cudaErrorInvalidConfiguration;
        e = current_device_context(&dev, &ctx);  // (the calls above made a context current)
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[dev], ctx, __ATOMIC_RELEASE);
    }
    // Both kernels are launched as programmatic dependents of the one before
    // them on the stream: their launch and prologue overlap its tail.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nsm);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Smem<D>::total;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, unified_attn_kernel<D>, p);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(nsm * kMergeCtasPerSm);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, merge_kernel<D>, p);
}

// The tensor-map encoder of the driver, resolved once through the runtime
// (no link-time dependency on the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiledFn) nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// A pool [num_slots, Hkv, D] bf16 as the 2-D tensor [num_slots * Hkv rows, D]:
// boxes of 64 columns x 1 row (the gather4 shape), 128-byte swizzle.
static cudaError_t pool_tensor_map(CUtensorMap *m, const void *pool, long long num_slots, int Hkv, int D) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)num_slots * (cuuint64_t)Hkv};
    const cuuint64_t gstride[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, 1}, estride[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), gdim, gstride, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_attn(const AttnArgs &a, int nsm, cudaStream_t st) {
    AttnParams p;
    cudaError_t e = pool_tensor_map(&p.tmap_k, a.k_pool, a.num_slots, a.Hkv, a.D);
    if (e != cudaSuccess) return e;
    e = pool_tensor_map(&p.tmap_v, a.v_pool, a.num_slots, a.Hkv, a.D);
    if (e != cudaSuccess) return e;
    p.q = a.q;
    p.k_pool = a.k_pool;
    p.v_pool = a.v_pool;
    p.slot_table = a.slot_table;
    p.sparse_idx = a.sparse_idx;
    p.sparse_slot = a.sparse_slot;
    p.out = a.out;
    p.logits = a.logits;
    p.lse = a.lse;
    p.hdr = reinterpret_cast<WsHeader *>(a.ws);
    p.req = reinterpret_cast<const ReqInfo *>(a.ws + a.lay.req);
    p.kv_off = reinterpret_cast<const long long *>(a.ws + a.lay.kv_off);
    p.logit_off = reinterpret_cast<const long long *>(a.ws + a.lay.logit_off);
    p.unit = reinterpret_cast<const UnitInfo *>(a.ws + a.lay.unit);
    p.merge_units = reinterpret_cast<const MergeUnit *>(a.ws + a.lay.merge_units);
    p.items = reinterpret_cast<const Item *>(a.ws + a.lay.items);
    p.part_o = reinterpret_cast<float *>(a.ws + a.lay.part_o);
    p.part_lse = reinterpret_cast<float *>(a.ws + a.lay.part_lse);
    p.num_slots = a.num_slots;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.k = a.k;
    p.M = (a.k + 1) * p.G;
    p.RQ = (p.M + kConsumerWarps - 1) / kConsumerWarps;
    // draft items spread their G rows over the four quadrants, except in the
    // uniform-rows schedule and the naive joint batch, where they take the verify row layout
    const bool naive = a.schedule == PILLAR_SCHEDULE_NAIVE_JOINT;
    p.RQd = (a.schedule == PILLAR_SCHEDULE_UNIFORM_ROWS || naive) ? p.RQ : (p.G + kConsumerWarps - 1) / kConsumerWarps;
    p.static_units = naive ? 1 : 0;
    p.max_sparse = a.max_sparse;
    p.scale = a.scale;
    p.wait_ns = a.wait_ns;
    return a.D == 128 ? launch_unified_t<128>(p, nsm, st) : launch_unified_t<64>(p, nsm, st);
}

}  // namespace pillar
