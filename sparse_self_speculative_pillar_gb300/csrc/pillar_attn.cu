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
// GB300 design: a persistent grid, two CTAs per SM (two independent
// pipelines per SM), six warps per CTA:
//   * resolver warp: pops work items from a global atomic counter, reads the
//     item's records and translates its positions into pool slots (list ->
//     slot, many independent loads per lane) into one of two row lists, one
//     item ahead of the loader;
//   * loader warp: gathers the item's K/V rows into a ring of shared-memory
//     stages with 16-byte cp.async (a 256-byte page-size-1 row is far too
//     small a unit for a TMA transfer), completion tracked on the stage's
//     mbarrier, and bulk-copies the item's query rows; the item's metadata
//     travels in the stage record, so consumers never read global memory
//     between items;
//   * four consumer warps, which never wait on each other: a verify item is a
//     dense (k+1)*G x 64 tile per stage on the tensor cores (mma.sync bf16 ->
//     fp32, one 16-row slice per warp, online softmax, logits dumped from the
//     same accumulators); a draft item runs on the CUDA cores, each warp
//     taking 16 of the 64 staged keys, each lane owning D/32 dimensions,
//     sixteen keys reduced at once by a transpose reduction across lanes,
//     packed fp32x2 FMAs;
//   * results that need combining -- the four warps' states of a draft item,
//     the pieces of a verify request split over several items -- are written
//     as normalised partials (o, lse) and combined afterwards by merge_kernel,
//     a flat bandwidth pass: o = sum_i e^{lse_i - lse} o_i, lse = log sum_i
//     e^{lse_i};
//   * every wait is bounded (about 1 s); a timeout raises PILLAR_FLAG_TIMEOUT,
//     the loader waits for its copies still in flight, and the CTA returns.
#include "pillar_device.cuh"

namespace pillar {

struct AttnParams {
    const uint16_t *q, *k_pool, *v_pool;
    const int *slot_table, *sparse_idx;
    uint16_t *out;
    float *logits, *lse;
    WsHeader *hdr;
    const ReqInfo *req;
    const long long *kv_off, *logit_off;
    const UnitInfo *unit;
    const int *merge_list;
    const Item *items;
    float *part_o, *part_lse;
    long long num_slots;
    int Hq, Hkv, G, k, M, max_sparse;
    float scale;
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
    long long pad2;
};

template <int D>
struct Smem {
    static constexpr int KSTR = D * 2 + 16;  // padded row stride: ldmatrix rows hit distinct banks
    static constexpr int ROWS = kTileKeys * KSTR;
    static constexpr int STAGE = 2 * ROWS;    // K rows, then V rows
    static constexpr int NSTAGE = 2;
    static constexpr int QBUF = kMaxRows * D * 2;
    static constexpr int off_q = NSTAGE * STAGE;
    static constexpr int off_rows = off_q + 2 * QBUF;
    static constexpr int off_info = off_rows + 2 * kMaxChunk * 4;
    static constexpr int off_meta = off_info + 2 * (int)sizeof(ItemInfo);
    static constexpr int off_bar = off_meta + NSTAGE * (int)sizeof(StageMeta);
    static constexpr int NBAR = 2 * NSTAGE + 2 + 4;  // full, empty, qempty[2], rfull[2], rempty[2]
    static constexpr int off_ps = off_bar + NBAR * 8;
    static constexpr int off_misc = off_ps + kConsumerWarps * 16 * kMaxG * 4;
    static constexpr int total = off_misc + 16;
};
// two CTAs share an SM's 228 KB
static_assert(Smem<128>::total <= 113 * 1024, "shared memory budget of two CTAs per SM");
static_assert(sizeof(StageMeta) % 16 == 0 && sizeof(ItemInfo) == 64, "record layout");

struct Ctx {
    char *smem;
    StageMeta *meta;
    ItemInfo *iinfo;
    int *rowlist;  // [2][kMaxChunk]
    uint64_t *full, *empty, *qempty, *rfull, *rempty;
    float *ps;
    volatile int *abort;
    int *err;
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
    c.empty = bars + S::NSTAGE;
    c.qempty = bars + 2 * S::NSTAGE;
    c.rfull = bars + 2 * S::NSTAGE + 2;
    c.rempty = bars + 2 * S::NSTAGE + 4;
    c.ps = reinterpret_cast<float *>(smem + S::off_ps);
    c.abort = reinterpret_cast<volatile int *>(smem + S::off_misc);
    c.err = &p.hdr->err;
    return c;
}

// Bounded wait that ignores the abort flag: used only to let copies already
// in flight land before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kWaitTimeoutNs) return;
}

// ============================================================== resolver warp

__device__ void resolver(const AttnParams &p, const Ctx &c, int lane) {
    const int num_items = *reinterpret_cast<volatile int *>(&p.hdr->num_items);
    uint32_t eph = 0;
    for (int rb = 0;; rb ^= 1) {
        if (!mbar_wait(&c.rempty[rb], ((eph >> rb) & 1) ^ 1, c.abort, c.err)) return;
        eph ^= 1u << rb;
        int it = 0;
        if (lane == 0) it = atomicAdd(&p.hdr->item_counter, 1);
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
        const int *list = p.sparse_idx + ((long long)b * p.Hkv + g) * p.max_sparse + itm.begin;
        int *rows = c.rowlist + rb * kMaxChunk;
        int bad = 0;
        // 16 independent loads per lane keep the dependent list -> slot chain short
        for (int base = 0; base < n; base += 32 * 16) {
            int pos[16], slot[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int i = base + r * 32 + lane;
                pos[r] = i < n ? (verify ? itm.begin + i : __ldg(list + i)) : -1;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int i = base + r * 32 + lane;
                const bool inpos = pos[r] >= 0 && pos[r] < ri.len;
                if (i < n && !inpos) bad |= PILLAR_FLAG_INDEX;
                slot[r] = (i < n && inpos) ? __ldg(p.slot_table + kvo + pos[r]) : -1;
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

// ============================================================== loader warp

template <int D>
__device__ void loader(const AttnParams &p, const Ctx &c, int lane) {
    using S = Smem<D>;
    int stage = 0, qn = 0;
    uint32_t phase = 0, qph = 0, fph = 0, issued = 0, issued_par = 0;
    bool ok = true;
    for (int rb = 0;; rb ^= 1) {
        ok = mbar_wait(&c.rfull[rb], (fph >> rb) & 1, c.abort, c.err);
        if (!ok) break;
        fph ^= 1u << rb;
        const ItemInfo info = c.iinfo[rb];
        if (info.it < 0) {
            ok = mbar_wait(&c.empty[stage], phase ^ 1, c.abort, c.err);
            if (ok) {
                cp_async_arrive_noinc(&c.full[stage]);
                __syncwarp();
                if (lane == 0) {
                    c.meta[stage].flags = kStop;
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
        for (int t = 0; t < ntiles; ++t) {
            ok = mbar_wait(&c.empty[stage], phase ^ 1, c.abort, c.err);
            if (!ok) break;
            if (t == 0) {
                ok = mbar_wait(&c.qempty[qb], ((qph >> qb) & 1) ^ 1, c.abort, c.err);
                if (!ok) break;
                qph ^= 1u << qb;
                ++qn;
            }
            const int k0 = t * kTileKeys;
            const int nk = max(0, min(kTileKeys, n - k0));
            const int r0 = lane < nk ? rows[k0 + lane] : -1;
            const int r1 = lane + 32 < nk ? rows[k0 + lane + 32] : -1;
            const unsigned v0 = __ballot_sync(0xffffffffu, r0 >= 0);
            const unsigned v1 = __ballot_sync(0xffffffffu, r1 >= 0);
            const unsigned long long valid = ((unsigned long long)v1 << 32) | v0;
            // Keys that are invalid or past the tail still get a real row (the
            // first valid key's): every staged row then holds finite pool data
            // and a zero probability can never meet a NaN.
            int fb = 0;
            if (valid) {
                const int f = __ffsll((long long)valid) - 1;
                fb = __shfl_sync(0xffffffffu, f < 32 ? r0 : r1, f & 31);
            }
            char *sK = c.smem + stage * S::STAGE;
            char *sV = sK + S::ROWS;
            if (valid) {
                // 16-byte cp.async: D/8 lanes per row, 256/D rows per warp pass
                constexpr int LPR = D / 8, RPP = 32 / LPR;
                const int cch = lane % LPR, rsub = lane / LPR;
                const int s0 = r0 >= 0 ? r0 : fb, s1 = r1 >= 0 ? r1 : fb;
                const char *kpool = reinterpret_cast<const char *>(p.k_pool);
                const char *vpool = reinterpret_cast<const char *>(p.v_pool);
#pragma unroll 4
                for (int i = 0; i < kTileKeys / RPP; ++i) {
                    const int row = RPP * i + rsub;  // the rows of one pass lie on the same side of 32
                    const int sl = __shfl_sync(0xffffffffu, row < 32 ? s0 : s1, row & 31);
                    const size_t off = ((size_t)sl * p.Hkv + g) * (D * 2) + cch * 16;
                    cp_async16(sK + row * S::KSTR + cch * 16, kpool + off);
                    cp_async16(sV + row * S::KSTR + cch * 16, vpool + off);
                }
            }
            cp_async_arrive_noinc(&c.full[stage]);  // lands with this lane's copies
            __syncwarp();
            const int qrows = verify ? p.k + 1 : 1;
            const uint32_t qbytes = (uint32_t)p.G * D * 2;
            if (lane == 0) {
                StageMeta &m = c.meta[stage];
                if (t == 0) m.info = info;
                m.nk = nk;
                m.flags = (t == 0 ? kFirst : 0) | (t == ntiles - 1 ? kLast : 0);
                m.pos0 = verify ? info.begin + k0 : 0;
                m.qb = qb;
                m.valid = valid;
                if (t == 0)
                    mbar_arrive_expect_tx(&c.full[stage], (uint32_t)qrows * qbytes);
                else
                    mbar_arrive(&c.full[stage]);
            }
            __syncwarp();
            if (t == 0) {
                char *qdst = c.smem + S::off_q + qb * S::QBUF;
                for (int j = lane; j < qrows; j += 32)
                    bulk_g2s(qdst + j * qbytes, p.q + ((size_t)(info.q_off + j) * p.Hq + (size_t)g * p.G) * D, qbytes,
                             &c.full[stage]);
            }
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
        for (int s = 0; s < S::NSTAGE; ++s)
            if ((issued >> s) & 1) drain_wait(&c.full[s], (issued_par >> s) & 1);
    }
}

// ============================================================== verify items (tensor cores)

template <int D>
__device__ bool verify_item(const AttnParams &p, const Ctx &c, int warp, int lane, int &stage, uint32_t &phase,
                            StageMeta cur) {
    using S = Smem<D>;
    const ItemInfo in = cur.info;
    const int G = p.G, M = p.M, kk1 = p.k + 1, L = in.L, g = in.g;
    const bool active = warp * 16 < M;
    const int row0 = warp * 16 + (lane >> 2), row1 = row0 + 8;
    const int j0 = row0 / G, gi0 = row0 - j0 * G, j1 = row1 / G, gi1 = row1 - j1 * G;
    const int lim0 = L - kk1 + j0, lim1 = L - kk1 + j1;
    const long long lb0 = in.logit_off + ((long long)(g * G + gi0) * kk1 + j0) * L;
    const long long lb1 = in.logit_off + ((long long)(g * G + gi1) * kk1 + j1) * L;
    const int c0 = 2 * (lane & 3);

    // Query rows stay in this item's shared-memory buffer; each tile reloads
    // the warp's A fragments from it (rows >= M read as zero).
    const int qb = cur.qb;
    const uint32_t qaddr = smem_u32(c.smem + S::off_q + qb * S::QBUF) +
                           (uint32_t)(min(warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), kMaxRows - 1) * D * 2 +
                                      (lane >> 4) * 16);

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = neg_inf(), m1 = neg_inf(), l0 = 0.f, l1 = 0.f;

    for (;;) {
        if (active && cur.valid) {
            const uint32_t kb = smem_u32(c.smem + stage * S::STAGE);
            const uint32_t vb = kb + S::ROWS;
            float s[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
            // S = Q K^T over the 64 staged keys
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(qaddr + ks * 32, a0, a1, a2, a3);
                if (row0 >= M) a0 = a2 = 0u;
                if (row1 >= M) a1 = a3 = 0u;
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const int key = 16 * np + ((lane >> 4) << 3) + (lane & 7);
                    ldsm_x4(kb + key * S::KSTR + (2 * ks + ((lane >> 3) & 1)) * 16, b0, b1, b2, b3);
                    mma_bf16_16816(s[2 * np], a0, a1, a2, a3, b0, b1);
                    mma_bf16_16816(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }
            // scale, mask, dump the logits, row maxima.  Interior tiles (every key
            // valid and visible to every row) skip the masking; the dump uses
            // 8-byte stores when the row offset is even.
            float mx0 = neg_inf(), mx1 = neg_inf();
            const bool interior = cur.nk == kTileKeys && cur.valid == ~0ull && cur.pos0 + kTileKeys - 1 <= L - kk1;
            if (interior) {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[nt][e] *= p.scale;
                    mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
                    mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
                }
                const long long t0 = cur.pos0 + c0;
                if (row0 < M) {
                    float *dst = p.logits + lb0 + t0;
                    if (((lb0 + t0) & 1) == 0) {
#pragma unroll
                        for (int nt = 0; nt < 8; ++nt)
                            *reinterpret_cast<float2 *>(dst + 8 * nt) = make_float2(s[nt][0], s[nt][1]);
                    } else {
#pragma unroll
                        for (int nt = 0; nt < 8; ++nt) {
                            dst[8 * nt] = s[nt][0];
                            dst[8 * nt + 1] = s[nt][1];
                        }
                    }
                }
                if (row1 < M) {
                    float *dst = p.logits + lb1 + t0;
                    if (((lb1 + t0) & 1) == 0) {
#pragma unroll
                        for (int nt = 0; nt < 8; ++nt)
                            *reinterpret_cast<float2 *>(dst + 8 * nt) = make_float2(s[nt][2], s[nt][3]);
                    } else {
#pragma unroll
                        for (int nt = 0; nt < 8; ++nt) {
                            dst[8 * nt] = s[nt][2];
                            dst[8 * nt + 1] = s[nt][3];
                        }
                    }
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = 8 * nt + c0 + (e & 1);
                        const int t = cur.pos0 + key;
                        const bool inkey = key < cur.nk;
                        const bool kv = inkey && ((cur.valid >> key) & 1ull);
                        const bool hi = e >= 2;
                        const bool vis = kv && t <= (hi ? lim1 : lim0);
                        const float x = vis ? s[nt][e] * p.scale : neg_inf();
                        s[nt][e] = x;
                        if (inkey) {
                            if (!hi && row0 < M) p.logits[lb0 + t] = x;
                            if (hi && row1 < M) p.logits[lb1 + t] = x;
                        }
                        if (hi)
                            mx1 = fmaxf(mx1, x);
                        else
                            mx0 = fmaxf(mx0, x);
                    }
                }
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float u0 = n0 == neg_inf() ? 0.f : n0, u1 = n1 == neg_inf() ? 0.f : n1;
            const float a0 = exp2f((m0 - u0) * kLog2e), a1 = exp2f((m1 - u1) * kLog2e);
            m0 = n0;
            m1 = n1;
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                s[nt][0] = exp2f((s[nt][0] - u0) * kLog2e);
                s[nt][1] = exp2f((s[nt][1] - u0) * kLog2e);
                s[nt][2] = exp2f((s[nt][2] - u1) * kLog2e);
                s[nt][3] = exp2f((s[nt][3] - u1) * kLog2e);
                ls0 += s[nt][0] + s[nt][1];
                ls1 += s[nt][2] + s[nt][3];
            }
            l0 = l0 * a0 + ls0;
            l1 = l1 * a1 + ls1;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                o[i][0] *= a0;
                o[i][1] *= a0;
                o[i][2] *= a1;
                o[i][3] *= a1;
            }
            // O += P V
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t pa0 = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
                const uint32_t pa1 = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
                const uint32_t pa2 = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
                const uint32_t pa3 = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
                const int key = 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vb + key * S::KSTR + (2 * dp + (lane >> 4)) * 16, b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * dp], pa0, pa1, pa2, pa3, b0, b1);
                    mma_bf16_16816(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2, b3);
                }
            }
        }
        mbar_arrive(&c.empty[stage]);
        const bool last = cur.flags & kLast;
        if (++stage == S::NSTAGE) {
            stage = 0;
            phase ^= 1;
        }
        if (last) break;
        if (!mbar_wait(&c.full[stage], phase, c.abort, c.err)) return false;
        cur = c.meta[stage];
    }

    mbar_arrive(&c.qempty[qb]);  // done with this item's query rows

    // Epilogue: normalise; write the output (or the item's partial) and the LSE.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const float e0 = l0 > 0.f ? m0 + logf(l0) : neg_inf();
    const float e1 = l1 > 0.f ? m1 + logf(l1) : neg_inf();
    if (active) {
        if (in.nsplit == 1) {
            const size_t or0 = ((size_t)(in.q_off + j0) * p.Hq + (size_t)g * G + gi0) * D;
            const size_t or1 = ((size_t)(in.q_off + j1) * p.Hq + (size_t)g * G + gi1) * D;
#pragma unroll
            for (int dn = 0; dn < D / 8; ++dn) {
                const int d = 8 * dn + c0;
                if (row0 < M)
                    *reinterpret_cast<uint32_t *>(p.out + or0 + d) = pack_bf16x2(o[dn][0] * i0, o[dn][1] * i0);
                if (row1 < M)
                    *reinterpret_cast<uint32_t *>(p.out + or1 + d) = pack_bf16x2(o[dn][2] * i1, o[dn][3] * i1);
            }
            if ((lane & 3) == 0) {
                if (row0 < M) p.lse[((size_t)in.vidx * p.Hq + (size_t)g * G + gi0) * kk1 + j0] = e0;
                if (row1 < M) p.lse[((size_t)in.vidx * p.Hq + (size_t)g * G + gi1) * kk1 + j1] = e1;
            }
        } else {
            const size_t pr0 = (size_t)in.rec + row0, pr1 = (size_t)in.rec + row1;
#pragma unroll
            for (int dn = 0; dn < D / 8; ++dn) {
                const int d = 8 * dn + c0;
                if (row0 < M)
                    *reinterpret_cast<float2 *>(p.part_o + pr0 * D + d) = make_float2(o[dn][0] * i0, o[dn][1] * i0);
                if (row1 < M)
                    *reinterpret_cast<float2 *>(p.part_o + pr1 * D + d) = make_float2(o[dn][2] * i1, o[dn][3] * i1);
            }
            if ((lane & 3) == 0) {
                if (row0 < M) p.part_lse[pr0] = e0;
                if (row1 < M) p.part_lse[pr1] = e1;
            }
        }
    }
    return true;
}

// ============================================================== draft items (CUDA cores)

// Sixteen per-lane partial sums v[0..16) (one per key) are reduced across the
// 32 lanes so that every lane ends with the full sum of key lane >> 1: each
// butterfly stage sends half of the lane's values to its partner and keeps
// the other half -- 16 shuffles for 16 keys instead of 5 per key.
__device__ __forceinline__ float transpose_reduce16(float (&v)[16], int lane) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool up = lane & 16;
        const float send = up ? v[i] : v[i + 8], keep = up ? v[i + 8] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = lane & 8;
        const float send = up ? v[i] : v[i + 4], keep = up ? v[i + 4] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = lane & 4;
        const float send = up ? v[i] : v[i + 2], keep = up ? v[i + 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    {
        const bool up = lane & 2;
        const float send = up ? v[0] : v[1], keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// This lane's D/32 bf16 elements of a shared-memory row, as fp32 pairs.
template <int D>
__device__ __forceinline__ void load_dims(const char *row, int lane, float2 (&x)[D / 64]) {
    if constexpr (D == 128) {
        const uint2 w = *reinterpret_cast<const uint2 *>(row + lane * 8);
        x[0] = make_float2(bf16lo(w.x), bf16hi(w.x));
        x[1] = make_float2(bf16lo(w.y), bf16hi(w.y));
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(row + lane * 4);
        x[0] = make_float2(bf16lo(w), bf16hi(w));
    }
}

template <int D, int GMAX>
__device__ bool draft_item(const AttnParams &p, const Ctx &c, int warp, int lane, int &stage, uint32_t &phase,
                           StageMeta cur) {
    using S = Smem<D>;
    constexpr int NP = D / 64;                 // fp32 pairs per lane (D/32 dimensions)
    constexpr int HC = GMAX < 4 ? GMAX : 4;    // heads reduced together
    const ItemInfo in = cur.info;
    const int G = p.G;

    float2 qf[GMAX][NP];
    {
        const char *qbuf = c.smem + S::off_q + cur.qb * S::QBUF;
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            if (h < G) {
                load_dims<D>(qbuf + h * D * 2, lane, qf[h]);
            } else {
#pragma unroll
                for (int e = 0; e < NP; ++e) qf[h][e] = make_float2(0.f, 0.f);
            }
        }
    }
    mbar_arrive(&c.qempty[cur.qb]);
    float2 o[GMAX][NP];
    float mw[GMAX], lp[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
        mw[h] = neg_inf();
        lp[h] = 0.f;
#pragma unroll
        for (int e = 0; e < NP; ++e) o[h][e] = make_float2(0.f, 0.f);
    }
    float *ps = c.ps + warp * 16 * kMaxG;   // [16 keys][kMaxG] probabilities of this warp's keys
    const int key_l = lane >> 1;

    for (;;) {
        if (cur.valid) {
            const char *sK = c.smem + stage * S::STAGE + (16 * warp) * S::KSTR;
            const char *sV = sK + S::ROWS;
            const int key = 16 * warp + key_l;
            const bool kv = key < cur.nk && ((cur.valid >> key) & 1ull);
            float sv[GMAX];
#pragma unroll
            for (int hc = 0; hc < GMAX; hc += HC) {
                if (hc < G) {
                    float part[HC][16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float2 kf[NP];
                        load_dims<D>(sK + j * S::KSTR, lane, kf);
#pragma unroll
                        for (int h = 0; h < HC; ++h) {
                            float2 a = make_float2(0.f, 0.f);
#pragma unroll
                            for (int e = 0; e < NP; ++e) a = ffma2(qf[hc + h][e], kf[e], a);
                            part[h][j] = a.x + a.y;
                        }
                    }
#pragma unroll
                    for (int h = 0; h < HC; ++h) {
                        const float d = transpose_reduce16(part[h], lane);
                        sv[hc + h] = kv ? d * p.scale : neg_inf();
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < HC; ++h) sv[hc + h] = neg_inf();
                }
            }
            // online softmax over this warp's 16 keys (lane pairs hold the same key)
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                if (h < G) {
                    float mt = sv[h];
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
                    const float mn = fmaxf(mw[h], mt);
                    const float mu = mn == neg_inf() ? 0.f : mn;
                    const float a = exp2f((mw[h] - mu) * kLog2e);
                    mw[h] = mn;
                    const float pr = exp2f((sv[h] - mu) * kLog2e);
                    lp[h] = lp[h] * a + ((lane & 1) ? 0.f : pr);
#pragma unroll
                    for (int e = 0; e < NP; ++e) o[h][e] = make_float2(o[h][e].x * a, o[h][e].y * a);
                    if ((lane & 1) == 0) ps[key_l * kMaxG + h] = pr;
                }
            }
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float2 vf[NP];
                load_dims<D>(sV + j * S::KSTR, lane, vf);
                float pj[GMAX];
                if constexpr (GMAX >= 4) {
#pragma unroll
                    for (int h4 = 0; h4 < GMAX; h4 += 4) {
                        const float4 w4 = *reinterpret_cast<const float4 *>(ps + j * kMaxG + h4);
                        pj[h4] = w4.x;
                        pj[h4 + 1] = w4.y;
                        pj[h4 + 2] = w4.z;
                        pj[h4 + 3] = w4.w;
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < GMAX; ++h) pj[h] = ps[j * kMaxG + h];
                }
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    if (h < G) {
                        const float2 pp = make_float2(pj[h], pj[h]);
#pragma unroll
                        for (int e = 0; e < NP; ++e) o[h][e] = ffma2(pp, vf[e], o[h][e]);
                    }
                }
            }
            __syncwarp();  // the probabilities are rewritten by the next tile
        }
        mbar_arrive(&c.empty[stage]);
        const bool last = cur.flags & kLast;
        if (++stage == S::NSTAGE) {
            stage = 0;
            phase ^= 1;
        }
        if (last) break;
        if (!mbar_wait(&c.full[stage], phase, c.abort, c.err)) return false;
        cur = c.meta[stage];
    }

    // This warp's partial: normalised over its own keys, with its LSE.
    const size_t rec = (size_t)in.rec + (size_t)warp * G;
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
        if (h < G) {
            float l = lp[h];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float2 *dst = reinterpret_cast<float2 *>(p.part_o + (rec + h) * D + lane * (D / 32));
#pragma unroll
            for (int e = 0; e < NP; ++e) dst[e] = make_float2(o[h][e].x * inv, o[h][e].y * inv);
            if (lane == 0) p.part_lse[rec + h] = l > 0.f ? mw[h] + logf(l) : neg_inf();
        }
    }
    return true;
}

// ============================================================== kernel

template <int D, int GMAX>
__device__ void consumer(const AttnParams &p, const Ctx &c, int warp, int lane) {
    int stage = 0;
    uint32_t phase = 0;
    for (;;) {
        if (!mbar_wait(&c.full[stage], phase, c.abort, c.err)) return;
        const StageMeta m = c.meta[stage];
        if (m.flags & kStop) return;
        const bool ok = m.info.mode == 1 ? verify_item<D>(p, c, warp, lane, stage, phase, m)
                                         : draft_item<D, GMAX>(p, c, warp, lane, stage, phase, m);
        if (!ok) return;
    }
}

template <int D, int GMAX>
__global__ void __launch_bounds__(kThreads, 2) unified_attn_kernel(const AttnParams p) {
    extern __shared__ __align__(1024) char smem[];
    using S = Smem<D>;
    const Ctx c = make_ctx<D>(smem, p);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S::NSTAGE; ++s) {
            mbar_init(&c.full[s], 32 + 1);  // the loader lanes' copy arrivals + its metadata arrival
            mbar_init(&c.empty[s], kConsumerWarps * 32);
        }
        mbar_init(&c.qempty[0], kConsumerWarps * 32);
        mbar_init(&c.qempty[1], kConsumerWarps * 32);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&c.rfull[i], 32);
            mbar_init(&c.rempty[i], 32);
        }
        *c.abort = 0;
        mbar_init_fence();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == kConsumerWarps)
        loader<D>(p, c, lane);
    else if (warp == kConsumerWarps + 1)
        resolver(p, c, lane);
    else
        consumer<D, GMAX>(p, c, warp, lane);
}

// ============================================================== merge of partials

constexpr int kMergeThreads = 256;

// For every listed (request, KV head): combine its partial rows.  Draft units
// have nsplit items x 4 warp records of G rows; split verify units have
// nsplit records of M rows.  Four output dimensions per thread.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const AttnParams p) {
    const int nm = p.hdr->num_merge;
    for (int li = blockIdx.x; li < nm; li += gridDim.x) {
        const int u = p.merge_list[li];
        const int b = u / p.Hkv, g = u - b * p.Hkv;
        const ReqInfo ri = p.req[b];
        const UnitInfo ui = p.unit[u];
        const bool verify = ri.mode == 1;
        const int nrows = verify ? p.M : p.G;
        const int nrec = verify ? ui.nsplit : ui.nsplit * kConsumerWarps;
        for (int idx = threadIdx.x; idx < nrows * (D / 4); idx += kMergeThreads) {
            const int row = idx / (D / 4), c4 = idx - row * (D / 4);
            float mx = neg_inf();
            for (int r = 0; r < nrec; ++r) {
                const size_t pr = verify ? (size_t)ui.rec_base + (size_t)r * p.M + row
                                         : (size_t)ui.rec_base + (size_t)(r / kConsumerWarps) * ui.rec_rows +
                                               (size_t)(r % kConsumerWarps) * p.G + row;
                mx = fmaxf(mx, p.part_lse[pr]);
            }
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            float lse = neg_inf();
            if (mx != neg_inf()) {
                float den = 0.f;
                for (int r = 0; r < nrec; ++r) {
                    const size_t pr = verify ? (size_t)ui.rec_base + (size_t)r * p.M + row
                                             : (size_t)ui.rec_base + (size_t)(r / kConsumerWarps) * ui.rec_rows +
                                                   (size_t)(r % kConsumerWarps) * p.G + row;
                    const float w = expf(p.part_lse[pr] - mx);
                    const float4 v = *reinterpret_cast<const float4 *>(p.part_o + pr * D + 4 * c4);
                    den += w;
                    o.x += w * v.x;
                    o.y += w * v.y;
                    o.z += w * v.z;
                    o.w += w * v.w;
                }
                const float inv = 1.f / den;
                o = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
                lse = mx + logf(den);
            }
            int j = 0, gi = row;
            if (verify) {
                j = row / p.G;
                gi = row - j * p.G;
            }
            const size_t orow = (size_t)(ri.q_off + j) * p.Hq + (size_t)g * p.G + gi;
            uint2 pk;
            pk.x = pack_bf16x2(o.x, o.y);
            pk.y = pack_bf16x2(o.z, o.w);
            *reinterpret_cast<uint2 *>(p.out + orow * D + 4 * c4) = pk;
            if (verify && c4 == 0) p.lse[((size_t)ri.vidx * p.Hq + (size_t)g * p.G + gi) * (p.k + 1) + j] = lse;
        }
    }
}

// ------------------------------------------------------------------ host-side launch helpers

template <int D, int GMAX>
cudaError_t launch_unified_t(const AttnParams &p, int nsm, cudaStream_t st) {
    static int configured_mask = 0;  // one bit per device (up to 32)
    static int blocks_per_sm[32];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int bit = 1 << (dev & 31);
    if (!(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(unified_attn_kernel<D, GMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Smem<D>::total);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, unified_attn_kernel<D, GMAX>, kThreads,
                                                          Smem<D>::total);
        if (e != cudaSuccess) return e;
        blocks_per_sm[dev & 31] = n > 0 ? n : 1;
        __atomic_fetch_or(&configured_mask, bit, __ATOMIC_RELEASE);
    }
    unified_attn_kernel<D, GMAX><<<nsm * blocks_per_sm[dev & 31], kThreads, Smem<D>::total, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    merge_kernel<D><<<nsm * 4, kMergeThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_attn(const AttnArgs &a, int nsm, cudaStream_t st) {
    AttnParams p;
    p.q = a.q;
    p.k_pool = a.k_pool;
    p.v_pool = a.v_pool;
    p.slot_table = a.slot_table;
    p.sparse_idx = a.sparse_idx;
    p.out = a.out;
    p.logits = a.logits;
    p.lse = a.lse;
    p.hdr = reinterpret_cast<WsHeader *>(a.ws);
    p.req = reinterpret_cast<const ReqInfo *>(a.ws + a.lay.req);
    p.kv_off = reinterpret_cast<const long long *>(a.ws + a.lay.kv_off);
    p.logit_off = reinterpret_cast<const long long *>(a.ws + a.lay.logit_off);
    p.unit = reinterpret_cast<const UnitInfo *>(a.ws + a.lay.unit);
    p.merge_list = reinterpret_cast<const int *>(a.ws + a.lay.merge_list);
    p.items = reinterpret_cast<const Item *>(a.ws + a.lay.items);
    p.part_o = reinterpret_cast<float *>(a.ws + a.lay.part_o);
    p.part_lse = reinterpret_cast<float *>(a.ws + a.lay.part_lse);
    p.num_slots = a.num_slots;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.k = a.k;
    p.M = (a.k + 1) * p.G;
    p.max_sparse = a.max_sparse;
    p.scale = a.scale;
    const bool small_g = p.G <= 4;
    if (a.D == 128) return small_g ? launch_unified_t<128, 4>(p, nsm, st) : launch_unified_t<128, 8>(p, nsm, st);
    return small_g ? launch_unified_t<64, 4>(p, nsm, st) : launch_unified_t<64, 8>(p, nsm, st);
}

}  // namespace pillar
