// pillar_attn.cu -- the persistent unified draft/verify attention kernel.
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
// GB300 design:
//   * one CTA per SM, persistent: a producer warp pops work items from a
//     global atomic counter and streams their K/V rows into a ring of
//     shared-memory stages with 1-D bulk (TMA) copies, one 256-byte row per
//     copy, completion counted on an mbarrier; the next item's rows are
//     resolved (list -> slot) while earlier stages are still being consumed,
//     so the pipeline does not drain between items;
//   * four consumer warps: a verify item is a dense (k+1)*G x 64 tile per
//     stage on the tensor cores (mma.sync bf16 -> fp32, one 16-row slice per
//     warp, FA2-style online softmax with the logits dump from the same
//     accumulators); a draft item (G query rows) runs on the CUDA cores, 16
//     lanes per key with warp-shuffle dot products and softmax, merged over
//     the four warps at the end;
//   * a (request, KV head) whose keys were split over several items writes
//     normalised partials (o, lse); the last item to finish (detected with an
//     atomic counter, never a wait) merges them by LSE weights;
//   * every wait is bounded (about 1 s); a timeout raises PILLAR_FLAG_TIMEOUT,
//     the producer waits for its copies still in flight, and the CTA returns.
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
    int *arrive;
    const Item *items;
    float *part_o, *part_lse;
    long long num_slots;
    int Hq, Hkv, G, k, M, max_sparse, rows;
    float scale;
};

enum : int { kFirst = 1, kLast = 2, kStop = 4 };

struct StageMeta {
    int item;   // work item index
    int nk;     // keys in this tile (0..64)
    int flags;  // kFirst / kLast / kStop
    int qb;     // query buffer of the item
    int pos0;   // logical position of key 0 (verify)
    int pad;
    unsigned long long valid;  // bit i: key i has an in-range position and slot
};

template <int D>
struct Smem {
    static constexpr int KSTR = D * 2 + 16;  // padded row stride: ldmatrix rows hit distinct banks
    static constexpr int ROWS = kTileKeys * KSTR;
    static constexpr int STAGE = 2 * ROWS;    // K rows, then V rows
    static constexpr int NSTAGE = 5;
    static constexpr int QBUF = kMaxRows * D * 2;
    static constexpr int off_q = NSTAGE * STAGE;
    static constexpr int off_rows = off_q + 2 * QBUF;
    static constexpr int off_meta = off_rows + kMaxChunk * 4;
    static constexpr int off_bar = off_meta + NSTAGE * (int)sizeof(StageMeta);
    static constexpr int NBAR = 2 * NSTAGE + 2 + 1;  // full, empty, qempty[2], cbar
    static constexpr int off_ml = off_bar + NBAR * 8;
    static constexpr int off_misc = off_ml + kConsumerWarps * kMaxG * 2 * 4;
    static constexpr int total = off_misc + 16;
};
static_assert(Smem<128>::total <= 227 * 1024, "shared memory budget");
static_assert(Smem<128>::QBUF >= kConsumerWarps * kMaxG * 128 * 4, "draft merge scratch fits a query buffer");

struct Ctx {
    char *smem;
    StageMeta *meta;
    uint64_t *full, *empty, *qempty, *cbar;
    float *ml;
    volatile int *abort;
    int *is_last;
    int *err;
};

template <int D>
__device__ __forceinline__ Ctx make_ctx(char *smem, const AttnParams &p) {
    using S = Smem<D>;
    Ctx c;
    c.smem = smem;
    c.meta = reinterpret_cast<StageMeta *>(smem + S::off_meta);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::off_bar);
    c.full = bars;
    c.empty = bars + S::NSTAGE;
    c.qempty = bars + 2 * S::NSTAGE;
    c.cbar = bars + 2 * S::NSTAGE + 2;
    c.ml = reinterpret_cast<float *>(smem + S::off_ml);
    c.abort = reinterpret_cast<volatile int *>(smem + S::off_misc);
    c.is_last = reinterpret_cast<int *>(smem + S::off_misc + 4);
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

// All 128 consumer threads meet (bounded).
__device__ __forceinline__ bool consumer_sync(const Ctx &c, uint32_t &cph) {
    mbar_arrive(c.cbar);
    const bool ok = mbar_wait(c.cbar, cph, c.abort, c.err);
    cph ^= 1;
    return ok;
}

// ============================================================== producer

template <int D>
__device__ void producer(const AttnParams &p, const Ctx &c, int lane) {
    using S = Smem<D>;
    int *rowlist = reinterpret_cast<int *>(c.smem + S::off_rows);
    const int num_items = *reinterpret_cast<volatile int *>(&p.hdr->num_items);
    int stage = 0;
    uint32_t phase = 0, qph = 0, issued = 0, issued_par = 0;
    int qn = 0;
    bool ok = true;
    while (ok) {
        int it = 0;
        if (lane == 0) it = atomicAdd(&p.hdr->item_counter, 1);
        it = __shfl_sync(0xffffffffu, it, 0);
        if (it >= num_items) {
            ok = mbar_wait(&c.empty[stage], phase ^ 1, c.abort, c.err);
            if (ok && lane == 0) {
                c.meta[stage].flags = kStop;
                mbar_arrive(&c.full[stage]);
            }
            break;
        }
        const Item itm = p.items[it];
        const int b = itm.unit / p.Hkv, g = itm.unit - b * p.Hkv;
        const ReqInfo ri = p.req[b];
        const bool verify = ri.mode == 1;
        const int n = itm.end - itm.begin;
        const long long kvo = p.kv_off[b];
        const int *list = p.sparse_idx + ((long long)b * p.Hkv + g) * p.max_sparse + itm.begin;

        // Resolve positions -> slots for the whole item; 8 independent loads
        // per lane at a time keep the dependent index->slot chain short.
        int bad = 0;
        for (int base = 0; base < n; base += 32 * 8) {
            int pos[8], slot[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = base + r * 32 + lane;
                pos[r] = i < n ? (verify ? itm.begin + i : __ldg(list + i)) : -1;
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = base + r * 32 + lane;
                const bool inpos = pos[r] >= 0 && pos[r] < ri.len;
                if (i < n && !inpos) bad |= PILLAR_FLAG_INDEX;
                slot[r] = (i < n && inpos) ? __ldg(p.slot_table + kvo + pos[r]) : -1;
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = base + r * 32 + lane;
                if (i < n) {
                    int s = slot[r];
                    if (pos[r] >= 0 && pos[r] < ri.len && (s < 0 || (long long)s >= p.num_slots)) {
                        bad |= PILLAR_FLAG_SLOT;
                        s = -1;
                    }
                    rowlist[i] = s;
                }
            }
        }
        if (bad) atomicOr(c.err, bad);
        __syncwarp();

        const int qb = qn & 1;
        ok = mbar_wait(&c.qempty[qb], ((qph >> qb) & 1) ^ 1, c.abort, c.err);
        if (!ok) break;
        qph ^= 1u << qb;
        ++qn;

        const int ntiles = n > 0 ? (n + kTileKeys - 1) / kTileKeys : 1;
        for (int t = 0; t < ntiles; ++t) {
            ok = mbar_wait(&c.empty[stage], phase ^ 1, c.abort, c.err);
            if (!ok) break;
            const int k0 = t * kTileKeys;
            const int nk = max(0, min(kTileKeys, n - k0));
            const int r0 = lane < nk ? rowlist[k0 + lane] : -1;
            const int r1 = lane + 32 < nk ? rowlist[k0 + lane + 32] : -1;
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
            const int flags = (t == 0 ? kFirst : 0) | (t == ntiles - 1 ? kLast : 0);
            const int qrows = verify ? p.k + 1 : 1;
            const uint32_t qbytes = (uint32_t)p.G * D * 2;
            uint32_t tx = valid ? 2u * kTileKeys * D * 2 : 0u;
            if (t == 0) tx += (uint32_t)qrows * qbytes;
            if (lane == 0) {
                StageMeta m;
                m.item = it;
                m.nk = nk;
                m.flags = flags;
                m.qb = qb;
                m.pos0 = verify ? itm.begin + k0 : 0;
                m.pad = 0;
                m.valid = valid;
                c.meta[stage] = m;
                if (tx)
                    mbar_arrive_expect_tx(&c.full[stage], tx);
                else
                    mbar_arrive(&c.full[stage]);
            }
            __syncwarp();
            char *sK = c.smem + stage * S::STAGE;
            char *sV = sK + S::ROWS;
            if (valid) {
                const size_t a0 = ((size_t)(r0 >= 0 ? r0 : fb) * p.Hkv + g) * D;
                const size_t a1 = ((size_t)(r1 >= 0 ? r1 : fb) * p.Hkv + g) * D;
                bulk_g2s(sK + lane * S::KSTR, p.k_pool + a0, D * 2, &c.full[stage]);
                bulk_g2s(sK + (lane + 32) * S::KSTR, p.k_pool + a1, D * 2, &c.full[stage]);
                bulk_g2s(sV + lane * S::KSTR, p.v_pool + a0, D * 2, &c.full[stage]);
                bulk_g2s(sV + (lane + 32) * S::KSTR, p.v_pool + a1, D * 2, &c.full[stage]);
            }
            if (t == 0) {
                char *qdst = c.smem + S::off_q + qb * S::QBUF;
                for (int j = lane; j < qrows; j += 32)
                    bulk_g2s(qdst + j * qbytes, p.q + ((size_t)(ri.q_off + j) * p.Hq + (size_t)g * p.G) * D,
                             qbytes, &c.full[stage]);
            }
            issued |= 1u << stage;
            issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
            if (++stage == S::NSTAGE) {
                stage = 0;
                phase ^= 1;
            }
        }
    }
    if (!ok) {
        // Let every copy this warp started land before the CTA can exit.
        for (int s = 0; s < S::NSTAGE; ++s)
            if ((issued >> s) & 1) drain_wait(&c.full[s], (issued_par >> s) & 1);
    }
}

// ============================================================== merge of split items

// The last item of a split (request, KV head) combines the normalised partials
// o_i with weights exp(lse_i - lse), lse = log sum_i exp(lse_i).
__device__ void merge_unit(const AttnParams &p, int u, const UnitInfo &ui, const ReqInfo &ri, int ctid, int D) {
    const int b = u / p.Hkv, g = u - b * p.Hkv;
    const bool verify = ri.mode == 1;
    const int nrows = verify ? p.M : p.G;
    for (int idx = ctid; idx < nrows * D; idx += kConsumerWarps * 32) {
        const int row = idx / D, d = idx - row * D;
        float mx = neg_inf();
        for (int s = 0; s < ui.nsplit; ++s)
            mx = fmaxf(mx, __ldcg(p.part_lse + (size_t)(ui.item_base + s) * p.rows + row));
        float o = 0.f, lse = neg_inf();
        if (mx != neg_inf()) {
            float den = 0.f, num = 0.f;
            for (int s = 0; s < ui.nsplit; ++s) {
                const size_t pr = (size_t)(ui.item_base + s) * p.rows + row;
                const float w = expf(__ldcg(p.part_lse + pr) - mx);
                den += w;
                num += w * __ldcg(p.part_o + pr * D + d);
            }
            o = num / den;
            lse = mx + logf(den);
        }
        int j = 0, gi = row;
        if (verify) {
            j = row / p.G;
            gi = row - j * p.G;
        }
        const size_t orow = (size_t)(ri.q_off + j) * p.Hq + (size_t)g * p.G + gi;
        __nv_bfloat16 ob = __float2bfloat16_rn(o);
        p.out[orow * D + d] = *reinterpret_cast<uint16_t *>(&ob);
        if (verify && d == 0) p.lse[((size_t)ri.vidx * p.Hq + (size_t)g * p.G + gi) * (p.k + 1) + j] = lse;
    }
}

// After an item's partial is written: count arrivals; the last one merges.
__device__ bool finish_split(const AttnParams &p, const Ctx &c, uint32_t &cph, int it_unit, const UnitInfo &ui,
                             const ReqInfo &ri, int ctid, int D) {
    __threadfence();
    if (!consumer_sync(c, cph)) return false;
    if (ctid == 0) {
        const int old = atomicAdd(p.arrive + it_unit, 1);
        *c.is_last = old == ui.nsplit - 1;
    }
    if (!consumer_sync(c, cph)) return false;
    if (*c.is_last) {
        __threadfence();
        merge_unit(p, it_unit, ui, ri, ctid, D);
    }
    return true;
}

// ============================================================== verify items (tensor cores)

template <int D>
__device__ bool verify_item(const AttnParams &p, const Ctx &c, int warp, int lane, int &stage, uint32_t &phase,
                            uint32_t &cph, StageMeta cur) {
    using S = Smem<D>;
    const int it = cur.item;
    const Item itm = p.items[it];
    const int u = itm.unit, b = u / p.Hkv, g = u - b * p.Hkv;
    const ReqInfo ri = p.req[b];
    const UnitInfo ui = p.unit[u];
    const int G = p.G, M = p.M, kk1 = p.k + 1, L = ri.len;
    const bool active = warp * 16 < M;
    const int row0 = warp * 16 + (lane >> 2), row1 = row0 + 8;
    const int j0 = row0 / G, gi0 = row0 - j0 * G, j1 = row1 / G, gi1 = row1 - j1 * G;
    const int lim0 = L - kk1 + j0, lim1 = L - kk1 + j1;
    const long long lgb = p.logit_off[b];
    const long long lb0 = lgb + ((long long)(g * G + gi0) * kk1 + j0) * L;
    const long long lb1 = lgb + ((long long)(g * G + gi1) * kk1 + j1) * L;
    const int c0 = 2 * (lane & 3);

    // Query A fragments for this warp's 16 rows (rows >= M are zero).
    uint32_t qa[D / 16][4];
    {
        const uint32_t qbase = smem_u32(c.smem + S::off_q + cur.qb * S::QBUF);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int r = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            ldsm_x4(qbase + (uint32_t)(min(r, kMaxRows - 1) * D * 2 + (2 * ks + (lane >> 4)) * 16), qa[ks][0],
                    qa[ks][1], qa[ks][2], qa[ks][3]);
            if (row0 >= M) qa[ks][0] = qa[ks][2] = 0u;
            if (row1 >= M) qa[ks][1] = qa[ks][3] = 0u;
        }
    }
    // The query buffer is free once every consumer holds its fragments.
    mbar_arrive(&c.qempty[cur.qb]);

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
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const int key = 16 * np + ((lane >> 4) << 3) + (lane & 7);
                    ldsm_x4(kb + key * S::KSTR + (2 * ks + ((lane >> 3) & 1)) * 16, b0, b1, b2, b3);
                    mma_bf16_16816(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                    mma_bf16_16816(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
                }
            }
            // scale, mask, dump the logits, row maxima
            float mx0 = neg_inf(), mx1 = neg_inf();
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

    // Epilogue: normalise; write the output (or the partial) and the LSE.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const float e0 = l0 > 0.f ? m0 + logf(l0) : neg_inf();
    const float e1 = l1 > 0.f ? m1 + logf(l1) : neg_inf();
    if (active) {
        if (ui.nsplit == 1) {
            const size_t or0 = ((size_t)(ri.q_off + j0) * p.Hq + (size_t)g * G + gi0) * D;
            const size_t or1 = ((size_t)(ri.q_off + j1) * p.Hq + (size_t)g * G + gi1) * D;
#pragma unroll
            for (int dn = 0; dn < D / 8; ++dn) {
                const int d = 8 * dn + c0;
                if (row0 < M)
                    *reinterpret_cast<uint32_t *>(p.out + or0 + d) = pack_bf16x2(o[dn][0] * i0, o[dn][1] * i0);
                if (row1 < M)
                    *reinterpret_cast<uint32_t *>(p.out + or1 + d) = pack_bf16x2(o[dn][2] * i1, o[dn][3] * i1);
            }
            if ((lane & 3) == 0) {
                if (row0 < M) p.lse[((size_t)ri.vidx * p.Hq + (size_t)g * G + gi0) * kk1 + j0] = e0;
                if (row1 < M) p.lse[((size_t)ri.vidx * p.Hq + (size_t)g * G + gi1) * kk1 + j1] = e1;
            }
        } else {
            const size_t pr0 = (size_t)it * p.rows + row0, pr1 = (size_t)it * p.rows + row1;
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
    if (ui.nsplit > 1) return finish_split(p, c, cph, u, ui, ri, warp * 32 + lane, D);
    return true;
}

// ============================================================== draft items (CUDA cores)

template <int D, int GMAX>
__device__ bool draft_item(const AttnParams &p, const Ctx &c, int warp, int lane, int &stage, uint32_t &phase,
                           uint32_t &cph, StageMeta cur) {
    using S = Smem<D>;
    constexpr int LPK = D / 8;         // lanes per key: each holds 8 of the D elements
    constexpr int KPP = 32 / LPK;      // keys per warp pass
    constexpr int PASSES = 16 / KPP;   // a warp covers 16 of the 64 staged keys
    const int it = cur.item;
    const Item itm = p.items[it];
    const int u = itm.unit, b = u / p.Hkv, g = u - b * p.Hkv;
    const ReqInfo ri = p.req[b];
    const UnitInfo ui = p.unit[u];
    const int G = p.G;
    const int grp = lane / LPK, cl = lane % LPK;
    const int qb = cur.qb;
    char *qbuf = c.smem + S::off_q + qb * S::QBUF;

    float qf[GMAX][8];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
        if (h < G) {
            const uint4 w = *reinterpret_cast<const uint4 *>(qbuf + h * D * 2 + cl * 16);
            qf[h][0] = bf16lo(w.x); qf[h][1] = bf16hi(w.x);
            qf[h][2] = bf16lo(w.y); qf[h][3] = bf16hi(w.y);
            qf[h][4] = bf16lo(w.z); qf[h][5] = bf16hi(w.z);
            qf[h][6] = bf16lo(w.w); qf[h][7] = bf16hi(w.w);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[h][e] = 0.f;
        }
    }
    float o[GMAX][8], mr[GMAX], lr[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
        mr[h] = neg_inf();
        lr[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] = 0.f;
    }

    for (;;) {
        if (cur.valid) {
            const char *sK = c.smem + stage * S::STAGE;
            const char *sV = sK + S::ROWS;
            float s[PASSES][GMAX];
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps) {
                const int key = 16 * warp + ps * KPP + grp;
                const bool kv = key < cur.nk && ((cur.valid >> key) & 1ull);
                const uint4 w = *reinterpret_cast<const uint4 *>(sK + key * S::KSTR + cl * 16);
                const float kf[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                                     bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    if (h < G) {
                        float d = 0.f;
#pragma unroll
                        for (int e = 0; e < 8; ++e) d = fmaf(qf[h][e], kf[e], d);
#pragma unroll
                        for (int off = LPK / 2; off >= 1; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
                        s[ps][h] = kv ? d * p.scale : neg_inf();
                    } else {
                        s[ps][h] = neg_inf();
                    }
                }
            }
            float mu[GMAX];
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                float mt = s[0][h];
#pragma unroll
                for (int ps = 1; ps < PASSES; ++ps) mt = fmaxf(mt, s[ps][h]);
                const float mn = fmaxf(mr[h], mt);
                mu[h] = mn == neg_inf() ? 0.f : mn;
                const float a = exp2f((mr[h] - mu[h]) * kLog2e);
                mr[h] = mn;
                lr[h] *= a;
#pragma unroll
                for (int e = 0; e < 8; ++e) o[h][e] *= a;
            }
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps) {
                const int key = 16 * warp + ps * KPP + grp;
                const uint4 w = *reinterpret_cast<const uint4 *>(sV + key * S::KSTR + cl * 16);
                const float vf[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                                     bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    if (h < G) {
                        const float pr = exp2f((s[ps][h] - mu[h]) * kLog2e);
                        lr[h] += pr;
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[h][e] = fmaf(pr, vf[e], o[h][e]);
                    }
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

    // Merge the key groups of this warp (they saw different keys).
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            if (h < G) {
                const float mo = __shfl_xor_sync(0xffffffffu, mr[h], off);
                const float lo = __shfl_xor_sync(0xffffffffu, lr[h], off);
                const float mn = fmaxf(mr[h], mo);
                const float mu = mn == neg_inf() ? 0.f : mn;
                const float a = exp2f((mr[h] - mu) * kLog2e), bb = exp2f((mo - mu) * kLog2e);
                lr[h] = lr[h] * a + lo * bb;
#pragma unroll
                for (int e = 0; e < 8; ++e) o[h][e] = o[h][e] * a + __shfl_xor_sync(0xffffffffu, o[h][e], off) * bb;
                mr[h] = mn;
            }
        }
    }
    // Every warp has read its query fragments: the query buffer becomes the
    // merge scratch [warp][h][D] (fp32) for the four warps' states.
    if (!consumer_sync(c, cph)) return false;
    float *so = reinterpret_cast<float *>(qbuf);
    if (grp == 0) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            if (h < G) {
                float4 *dst = reinterpret_cast<float4 *>(so + ((size_t)warp * G + h) * D + cl * 8);
                dst[0] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
                dst[1] = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
                if (cl == 0) {
                    c.ml[(warp * kMaxG + h) * 2 + 0] = mr[h];
                    c.ml[(warp * kMaxG + h) * 2 + 1] = lr[h];
                }
            }
        }
    }
    if (!consumer_sync(c, cph)) return false;
    const int ctid = warp * 32 + lane;
    for (int idx = ctid; idx < G * D; idx += kConsumerWarps * 32) {
        const int h = idx / D, d = idx - h * D;
        float mx = neg_inf();
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) mx = fmaxf(mx, c.ml[(w * kMaxG + h) * 2]);
        float ov = 0.f, lse = neg_inf();
        if (mx != neg_inf()) {
            float den = 0.f, num = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float wt = exp2f((c.ml[(w * kMaxG + h) * 2] - mx) * kLog2e);
                den += wt * c.ml[(w * kMaxG + h) * 2 + 1];
                num += wt * so[((size_t)w * G + h) * D + d];
            }
            if (den > 0.f) {
                ov = num / den;
                lse = mx + logf(den);
            }
        }
        if (ui.nsplit == 1) {
            __nv_bfloat16 ob = __float2bfloat16_rn(ov);
            p.out[((size_t)ri.q_off * p.Hq + (size_t)g * G + h) * D + d] = *reinterpret_cast<uint16_t *>(&ob);
        } else {
            const size_t pr = (size_t)it * p.rows + h;
            p.part_o[pr * D + d] = ov;
            if (d == 0) p.part_lse[pr] = lse;
        }
    }
    // The scratch will next be overwritten by a bulk copy (async proxy).
    fence_proxy_async_smem();
    mbar_arrive(&c.qempty[qb]);
    if (ui.nsplit > 1) return finish_split(p, c, cph, u, ui, ri, ctid, D);
    return true;
}

// ============================================================== kernel

template <int D, int GMAX>
__device__ void consumer(const AttnParams &p, const Ctx &c, int warp, int lane) {
    int stage = 0;
    uint32_t phase = 0, cph = 0;
    for (;;) {
        if (!mbar_wait(&c.full[stage], phase, c.abort, c.err)) return;
        const StageMeta m = c.meta[stage];
        if (m.flags & kStop) return;
        const Item itm = p.items[m.item];
        const int mode = p.req[itm.unit / p.Hkv].mode;
        const bool ok = mode == 1 ? verify_item<D>(p, c, warp, lane, stage, phase, cph, m)
                                  : draft_item<D, GMAX>(p, c, warp, lane, stage, phase, cph, m);
        if (!ok) return;
    }
}

template <int D, int GMAX>
__global__ void __launch_bounds__(kThreads, 1) unified_attn_kernel(const AttnParams p) {
    extern __shared__ __align__(1024) char smem[];
    using S = Smem<D>;
    const Ctx c = make_ctx<D>(smem, p);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S::NSTAGE; ++s) {
            mbar_init(&c.full[s], 1);
            mbar_init(&c.empty[s], kConsumerWarps * 32);
        }
        mbar_init(&c.qempty[0], kConsumerWarps * 32);
        mbar_init(&c.qempty[1], kConsumerWarps * 32);
        mbar_init(c.cbar, kConsumerWarps * 32);
        *c.abort = 0;
        *c.is_last = 0;
        mbar_init_fence();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == kConsumerWarps)
        producer<D>(p, c, lane);
    else
        consumer<D, GMAX>(p, c, warp, lane);
}

// ------------------------------------------------------------------ host-side launch helpers

template <int D, int GMAX>
cudaError_t launch_unified_t(const AttnParams &p, int grid, cudaStream_t st) {
    static int configured_mask = 0;  // one bit per device (up to 32)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int bit = 1 << (dev & 31);
    if (!(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(unified_attn_kernel<D, GMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Smem<D>::total);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured_mask, bit, __ATOMIC_RELEASE);
    }
    unified_attn_kernel<D, GMAX><<<grid, kThreads, Smem<D>::total, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_attn(const AttnArgs &a, int grid, cudaStream_t st) {
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
    p.arrive = reinterpret_cast<int *>(a.ws + a.lay.arrive);
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
    p.rows = a.lay.rows;
    p.scale = a.scale;
    const bool small_g = p.G <= 4;
    if (a.D == 128) return small_g ? launch_unified_t<128, 4>(p, grid, st) : launch_unified_t<128, 8>(p, grid, st);
    return small_g ? launch_unified_t<64, 4>(p, grid, st) : launch_unified_t<64, 8>(p, grid, st);
}

}  // namespace pillar
