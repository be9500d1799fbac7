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
// attention kernel); splitting long contexts over CTAs with an LSE merge is
// this kernel's own load balancing.
#include "pillar_device.cuh"

namespace pillar {

struct PlanParams {
    const int *req_mode, *req_len, *sparse_cnt;
    WsHeader *hdr;
    ReqInfo *req;
    long long *kv_off, *logit_off;
    UnitInfo *unit;
    int *arrive;
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

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanParams p) {
    const int tid = threadIdx.x;
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

    // Units (request, KV head): split counts, then item bases (verify first).
    const int U = p.B * p.Hkv;
    long long cver = 0;
    for (int pass = 0; pass < 2; ++pass) {
        long long carry = pass ? cver : 0;
        for (int base = 0; base < U; base += kPlanThreads) {
            const int u = base + tid;
            long long cnt = 0;
            int ns = 1;
            bool isv = false;
            if (u < U) {
                const int b = u / p.Hkv;
                const ReqInfo r = p.req[b];
                isv = r.mode == 1;
                if (isv) {
                    chunking(r.len, p.vchunk, &ns);
                } else {
                    int n = r.mode == 0 ? p.sparse_cnt[u] : 0;
                    if (n < 0 || n > p.max_sparse) {
                        if (pass == 0) bad |= PILLAR_FLAG_COUNT;
                    }
                    n = n < 0 ? 0 : (n > p.max_sparse ? p.max_sparse : n);
                    chunking(n, p.dchunk, &ns);
                }
                cnt = (pass == 0) == isv ? ns : 0;
            }
            long long tot;
            const long long off = block_exclusive_scan(cnt, &tot);
            if (u < U && ((pass == 0) == isv)) {
                UnitInfo ui;
                ui.nsplit = ns;
                ui.item_base = (int)(carry + off);
                p.unit[u] = ui;
                p.arrive[u] = 0;
            }
            carry += tot;
        }
        if (pass == 0) cver = carry;
        else if (tid == 0) {
            p.hdr->num_items = (int)carry;
            p.hdr->num_units = U;
        }
    }
    __syncthreads();

    // Emit the items.
    for (int u = tid; u < U; u += kPlanThreads) {
        const int b = u / p.Hkv;
        const ReqInfo r = p.req[b];
        const UnitInfo ui = p.unit[u];
        int n, ns, cs;
        if (r.mode == 1) {
            n = r.len;
            cs = chunking(n, p.vchunk, &ns);
        } else {
            n = r.mode == 0 ? p.sparse_cnt[u] : 0;
            n = n < 0 ? 0 : (n > p.max_sparse ? p.max_sparse : n);
            cs = chunking(n, p.dchunk, &ns);
        }
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
    p.arrive = reinterpret_cast<int *>(a.ws + a.lay.arrive);
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
