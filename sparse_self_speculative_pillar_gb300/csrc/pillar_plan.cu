// pillar_plan.cu -- device-side planner of the unified step.
//
// One CTA turns the batch description (req_mode, req_len, sparse_cnt) into
// the per-request offsets and the work list of the persistent attention
// kernel.  A work item is (request, KV head, key range): verify requests are
// split over their context into near-equal chunks of about verify_chunk keys,
// draft lists into chunks of about draft_chunk listed keys.  Verify items are
// listed first (they are the heavy ones), then draft items, so the work queue
// is consumed roughly heaviest-first.  The draft/verify mix in one batch is
// the unified batch of "SparseSpec-MLSys26" (Unified batch scheduler + fused
// attention kernel); splitting long contexts over CTAs and merging the pieces
// by their LSE is this implementation's own load balancing.
//
// The planner also places the partial records: every draft item writes one
// record of G rows per consumer warp, a verify request split over several
// items writes M = (k+1)*G rows per item; the units that need combining are
// listed for the merge kernel.
#include "pillar_device.cuh"

namespace pillar {

struct PlanParams {
    const int *req_mode, *req_len, *sparse_cnt;
    WsHeader *hdr;
    ReqInfo *req;
    long long *kv_off, *logit_off;
    UnitInfo *unit;
    int *merge_list;
    Item *items;
    int B, Hq, Hkv, k, max_sparse, max_len, vchunk, dchunk;
};

// Exclusive scan over the CTA (kPlanThreads threads); *total gets the sum.
__device__ long long block_exclusive_scan(long long v, long long *total) {
    __shared__ long long warp_sums[kPlanThreads / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        long long s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            long long y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    const long long base = wid ? warp_sums[wid - 1] : 0;
    *total = warp_sums[kPlanThreads / 32 - 1];
    __syncthreads();
    return base + x - v;
}

// Near-equal chunking of n keys into pieces of at most `chunk` keys, rounded
// up to whole 64-key tiles.  Returns the chunk size; *ns gets the count (>=1).
__device__ __forceinline__ int chunking(int n, int chunk, int *ns) {
    if (n <= 0) {
        *ns = 1;
        return 0;
    }
    int n0 = (n + chunk - 1) / chunk;
    int cs = (n + n0 - 1) / n0;
    cs = (cs + kTileKeys - 1) / kTileKeys * kTileKeys;
    *ns = (n + cs - 1) / cs;
    return cs;
}

// Keys, split count and chunk size of unit u (request b = u / Hkv).
__device__ __forceinline__ int unit_split(const PlanParams &p, const ReqInfo &r, int u, int *n, int *ns, int *bad) {
    if (r.mode == 1) {
        *n = r.len;
        return chunking(r.len, p.vchunk, ns);
    }
    int c = r.mode == 0 ? p.sparse_cnt[u] : 0;
    if (c < 0 || c > p.max_sparse) *bad |= PILLAR_FLAG_COUNT;
    c = c < 0 ? 0 : (c > p.max_sparse ? p.max_sparse : c);
    *n = c;
    return chunking(c, p.dchunk, ns);
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanParams p) {
    const int tid = threadIdx.x;
    const int G = p.Hq / p.Hkv, M = (p.k + 1) * G;
    if (tid == 0) {
        p.hdr->err = 0;
        p.hdr->item_counter = 0;
    }
    int bad = 0;

    // Requests: query-row, KV, verify-index and logits offsets.
    long long cq = 0, ckv = 0, cv = 0, clg = 0;
    for (int base = 0; base < p.B; base += kPlanThreads) {
        const int b = base + tid;
        int mode = 0, len = 0;
        if (b < p.B) {
            mode = p.req_mode[b];
            len = p.req_len[b];
        }
        int eff_mode = mode, proc_len = len;
        if (b < p.B) {
            if (mode != 0 && mode != 1) bad |= PILLAR_FLAG_REQUEST, eff_mode = -1;
            if (len < 0) bad |= PILLAR_FLAG_REQUEST, proc_len = 0, len = 0;
            if (proc_len > p.max_len) bad |= PILLAR_FLAG_REQUEST, proc_len = p.max_len;
            if (eff_mode == 1 && len < p.k + 1) bad |= PILLAR_FLAG_REQUEST;
        }
        const long long nq = b < p.B ? (eff_mode == 1 ? p.k + 1 : 1) : 0;
        const long long kvl = b < p.B ? len : 0;
        const long long isv = (b < p.B && eff_mode == 1) ? 1 : 0;
        const long long lg = isv ? (long long)p.Hq * (p.k + 1) * len : 0;
        long long tq, tkv, tv, tlg;
        const long long oq = block_exclusive_scan(nq, &tq);
        const long long okv = block_exclusive_scan(kvl, &tkv);
        const long long ov = block_exclusive_scan(isv, &tv);
        const long long olg = block_exclusive_scan(lg, &tlg);
        if (b < p.B) {
            ReqInfo r;
            r.q_off = (int)(cq + oq);
            r.vidx = (int)(cv + ov);
            r.len = proc_len;
            r.mode = eff_mode;
            p.req[b] = r;
            p.kv_off[b] = ckv + okv;
            p.logit_off[b] = clg + olg;
        }
        cq += tq;
        ckv += tkv;
        cv += tv;
        clg += tlg;
    }
    __syncthreads();

    // Units (request, KV head): item bases (verify units first), partial-row
    // bases and the merge list.
    const int U = p.B * p.Hkv;
    long long c_ver_items = 0;
    {   // pass 0: verify item bases
        long long carry = 0;
        for (int base = 0; base < U; base += kPlanThreads) {
            const int u = base + tid;
            long long cnt = 0;
            int n = 0, ns = 1;
            bool isv = false;
            if (u < U) {
                const ReqInfo r = p.req[u / p.Hkv];
                unit_split(p, r, u, &n, &ns, &bad);
                isv = r.mode == 1;
                cnt = isv ? ns : 0;
            }
            long long tot;
            const long long off = block_exclusive_scan(cnt, &tot);
            if (u < U && isv) p.unit[u].item_base = (int)(carry + off);
            carry += tot;
        }
        c_ver_items = carry;
    }
    long long c_items = c_ver_items, c_rec = 0, c_merge = 0;
    for (int base = 0; base < U; base += kPlanThreads) {   // pass 1: the rest
        const int u = base + tid;
        long long dcnt = 0, recs = 0, mflag = 0;
        int n = 0, ns = 1, rec_rows = 0;
        bool isv = false;
        if (u < U) {
            const ReqInfo r = p.req[u / p.Hkv];
            int dummy = 0;
            unit_split(p, r, u, &n, &ns, &dummy);
            isv = r.mode == 1;
            dcnt = isv ? 0 : ns;
            rec_rows = isv ? (ns > 1 ? M : 0) : kConsumerWarps * G;
            recs = (long long)ns * rec_rows;
            mflag = rec_rows > 0 ? 1 : 0;
        }
        long long td, tr, tm;
        const long long od = block_exclusive_scan(dcnt, &td);
        const long long orr = block_exclusive_scan(recs, &tr);
        const long long om = block_exclusive_scan(mflag, &tm);
        if (u < U) {
            UnitInfo ui;
            ui.nsplit = ns;
            ui.item_base = isv ? p.unit[u].item_base : (int)(c_items + od);
            ui.rec_base = (int)(c_rec + orr);
            ui.rec_rows = rec_rows;
            p.unit[u] = ui;
            if (mflag) p.merge_list[c_merge + om] = u;
        }
        c_items += td;
        c_rec += tr;
        c_merge += tm;
    }
    if (tid == 0) {
        p.hdr->num_items = (int)c_items;
        p.hdr->num_units = U;
        p.hdr->num_merge = (int)c_merge;
    }
    __syncthreads();

    // Emit the items.
    for (int u = tid; u < U; u += kPlanThreads) {
        const ReqInfo r = p.req[u / p.Hkv];
        const UnitInfo ui = p.unit[u];
        int n, ns, dummy = 0;
        const int cs = unit_split(p, r, u, &n, &ns, &dummy);
        for (int s = 0; s < ns; ++s) {
            Item it;
            it.unit = u;
            it.begin = s * cs;
            it.end = min(n, (s + 1) * cs);
            it.split = s;
            p.items[ui.item_base + s] = it;
        }
    }
    if (bad) atomicOr(&p.hdr->err, bad);
}

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t st) {
    PlanParams p;
    p.req_mode = a.req_mode;
    p.req_len = a.req_len;
    p.sparse_cnt = a.sparse_cnt;
    p.hdr = reinterpret_cast<WsHeader *>(a.ws);
    p.req = reinterpret_cast<ReqInfo *>(a.ws + a.lay.req);
    p.kv_off = reinterpret_cast<long long *>(a.ws + a.lay.kv_off);
    p.logit_off = reinterpret_cast<long long *>(a.ws + a.lay.logit_off);
    p.unit = reinterpret_cast<UnitInfo *>(a.ws + a.lay.unit);
    p.merge_list = reinterpret_cast<int *>(a.ws + a.lay.merge_list);
    p.items = reinterpret_cast<Item *>(a.ws + a.lay.items);
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.k = a.k;
    p.max_sparse = a.max_sparse;
    p.max_len = a.max_len;
    p.vchunk = a.vchunk;
    p.dchunk = a.dchunk;
    plan_kernel<<<1, kPlanThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace pillar
