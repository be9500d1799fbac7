// pillar_plan.cu -- device-side planner of the unified step.
//
// One CTA turns the batch description (req_mode, req_len, sparse_cnt) into
// the per-request offsets and the work list of the persistent attention
// kernel.  A work item is (request, KV head, key range): verify requests are
// split over their context into near-equal chunks of about verify_chunk keys,
// draft lists into chunks of about draft_chunk listed keys.  Verify items are
// listed first (they are the heavy ones), then draft items by size, largest
// first, so the work queue is consumed heaviest-first and the last items
// taken are the shortest (the longest-processing-time rule: the CTAs finish
// close together); a verify request's items are listed chunk by chunk with
// the KV heads innermost, so the CTAs that read the same positions
// (neighbouring 256-byte rows of the same slot blocks, one per head) run at
// the same time.  The draft/verify mix in one batch is
// the unified batch of "SparseSpec-MLSys26" (Unified batch scheduler + fused
// attention kernel); splitting long contexts over CTAs and merging the pieces
// by their LSE is this implementation's own load balancing.
//
// The planner also places the partial records: a (request, KV head) split
// over several items writes one record per item, M = (k+1)*G rows for a
// verify request, G rows for a draft token; the units that need combining
// are listed for the merge kernel, the verify units from the start of the
// list and the draft units from its end, so that the merge gives each unit
// threads for its own rows only.
#include "pillar_device.cuh"

namespace pillar {

struct PlanParams {
    const int *req_mode, *req_len, *sparse_cnt;
    WsHeader *hdr;
    ReqInfo *req;
    long long *kv_off, *logit_off;
    UnitInfo *unit;
    MergeUnit *merge_units;
    Item *items;
    int B, Hq, Hkv, k, max_sparse, max_len, vchunk, dchunk;
    int schedule;  // PILLAR_SCHEDULE_*
};

constexpr int kScanN = 8;

// Size bins of the draft items: bin i holds the items of the draft units whose
// chunk spans kSizeBins - i tiles, so the bins in order are largest first.
constexpr int kSizeBins = kMaxChunk / kTileKeys;

// Size bin of a draft unit's items from its chunk size cs (an empty list
// counts as one tile: its item still passes through the pipeline once).
__device__ __forceinline__ int size_bin(int cs) {
    const int tiles = cs > kTileKeys ? (cs + kTileKeys - 1) / kTileKeys : 1;
    return kSizeBins - (tiles < kSizeBins ? tiles : kSizeBins);
}

// Units a planner thread keeps in registers between the scan and the item
// emission (one per chunk of kPlanThreads units); beyond that many chunks
// the emission re-reads its inputs.  Two measured slower than one: the
// registers they hold cost the whole kernel more than the re-reads.
constexpr int kRegChunks = 1;

// Exclusive scan of kScanN values per thread over the CTA (kPlanThreads
// threads), all at once; tot[] gets the CTA totals.
__device__ void block_scan8(long long (&v)[kScanN], long long (&tot)[kScanN]) {
    __shared__ long long warp_sums[kPlanThreads / 32][kScanN];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    long long x[kScanN];
#pragma unroll
    for (int i = 0; i < kScanN; ++i) x[i] = v[i];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int i = 0; i < kScanN; ++i) {
            const long long y = __shfl_up_sync(0xffffffffu, x[i], o);
            if (lane >= o) x[i] += y;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int i = 0; i < kScanN; ++i) warp_sums[wid][i] = x[i];
    }
    __syncthreads();
    if (wid == 0) {
        // the columns in two halves, each loaded first and scanned together:
        // independent shuffle chains within the 64 registers a thread has here
#pragma unroll
        for (int h = 0; h < kScanN; h += kScanN / 2) {
            long long t[kScanN / 2];
#pragma unroll
            for (int i = 0; i < kScanN / 2; ++i) t[i] = warp_sums[lane][h + i];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                for (int i = 0; i < kScanN / 2; ++i) {
                    const long long y = __shfl_up_sync(0xffffffffu, t[i], o);
                    if (lane >= o) t[i] += y;
                }
            }
#pragma unroll
            for (int i = 0; i < kScanN / 2; ++i) warp_sums[lane][h + i] = t[i];
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kScanN; ++i) {
        const long long base = wid ? warp_sums[wid - 1][i] : 0;
        tot[i] = warp_sums[kPlanThreads / 32 - 1][i];
        v[i] = base + x[i] - v[i];
    }
    __syncthreads();
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

// Keys, split count and chunk size of a unit of a request with record r;
// cnt is the unit's sparse_cnt entry (used by draft units only).  A request
// that the schedule leaves out of this call has no items (ns = 0).
__device__ __forceinline__ int unit_split(const PlanParams &p, const ReqInfo &r, int cnt, int *n, int *ns, int *bad) {
    if ((p.schedule == PILLAR_SCHEDULE_DRAFT_ONLY && r.mode == 1) ||
        (p.schedule == PILLAR_SCHEDULE_VERIFY_ONLY && r.mode == 0)) {
        *n = 0;
        *ns = 0;
        return 0;
    }
    if (r.mode == 1) {
        *n = r.len;
        const int vc = p.vchunk > 0 ? p.vchunk : (r.len >= kLongContext ? kLongVerifyChunk : kDefaultVerifyChunk);
        return chunking(r.len, vc, ns);
    }
    int c = r.mode == 0 ? cnt : 0;
    if (c < 0 || c > p.max_sparse) *bad |= PILLAR_FLAG_COUNT;
    c = c < 0 ? 0 : (c > p.max_sparse ? p.max_sparse : c);
    *n = c;
    return chunking(c, p.dchunk, ns);
}

// Request record from a request's mode and length (validated).
__device__ __forceinline__ ReqInfo check_request(const PlanParams &p, int mode, int len, int *bad, int *len_out) {
    ReqInfo r;
    r.q_off = r.vidx = 0;
    r.mode = mode;
    if (mode != 0 && mode != 1) *bad |= PILLAR_FLAG_REQUEST, r.mode = -1;
    if (len < 0) *bad |= PILLAR_FLAG_REQUEST, len = 0;
    r.len = len;
    if (r.len > p.max_len) *bad |= PILLAR_FLAG_REQUEST, r.len = p.max_len;
    if (r.mode == 1 && len < p.k + 1) *bad |= PILLAR_FLAG_REQUEST;
    *len_out = len;
    return r;
}

// The work items of unit u.  A verify request's Hkv units all have ns items;
// they are listed chunk by chunk, head-minor (request, chunk, head), so the
// Hkv items reading the same positions are taken up together.  Draft items
// stay per unit.
__device__ __forceinline__ void emit_items(const PlanParams &p, int u, int mode, int n, int ns, int cs, int item_base) {
    const int g = u - (u / p.Hkv) * p.Hkv;
    const int first = mode == 1 ? item_base - g * ns + g : item_base;
    const int step = mode == 1 ? p.Hkv : 1;
    for (int s = 0; s < ns; ++s) {
        Item it;
        it.unit = u;
        it.begin = s * cs;
        it.end = min(n, (s + 1) * cs);
        it.split = s;
        p.items[first + s * step] = it;
    }
}

// One thread per unit (request, KV head), chunks of kPlanThreads units; the
// unit with g == 0 also carries its request's counts, so one fused scan per
// chunk gives every offset.  A draft unit's items are placed in two steps:
// its place inside its size bin while the chunks are scanned, the bin's
// first index once every unit has been counted.
__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanParams p) {
    // launched as a programmatic dependent of the kernel before it on the stream (the last
    // step's Top-K, or another layer's run on this workspace): nothing is read or written
    // before the kernels ahead are complete.  The inputs' lines are only prefetched into L2
    // meanwhile (a hint: the loads below read them after the wait, through the coherent L2).
    {
        const int U0 = p.B * p.Hkv;
        const int t = threadIdx.x;
        for (int l = t; l * 32 < U0; l += kPlanThreads) l2_prefetch(p.sparse_cnt + l * 32);
        if (t * 32 < p.B) {
            l2_prefetch(p.req_mode + t * 32);
            l2_prefetch(p.req_len + t * 32);
        }
    }
    pdl_wait_prerequisites();
    // the attention kernel may start its prologue (barriers, tensor memory) now;
    // it reads nothing of this kernel's output before this kernel completes
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const int G = p.Hq / p.Hkv, M = (p.k + 1) * G;
    const int U = p.B * p.Hkv;
    if (tid == 0) {
        p.hdr->err = 0;
        p.hdr->item_counter = 0;
    }
    int bad = 0;
    // When at most kRegChunks chunks cover every unit, each thread keeps its
    // units' records and emits their items without reading anything back.
    const bool in_regs = U <= kRegChunks * kPlanThreads;
    int modek[kRegChunks], nk[kRegChunks], nsk[kRegChunks], csk[kRegChunks], itemk[kRegChunks];
    // running totals of the chunks before (shared memory: no registers held across the scans):
    // q rows, kv positions, verify requests, logits, verify items, draft items, partial rows, merges
    __shared__ long long carry[kScanN];
    __shared__ int s_bin[kSizeBins];  // draft items per size bin, then each bin's first item
    __shared__ int s_mdraft;          // split draft units: listed from the top of the merge list down
    // the naive joint batch walks each unit's items in place, so its drafts stay unit by unit
    const bool by_size = p.schedule != PILLAR_SCHEDULE_NAIVE_JOINT;
    if (tid < kScanN) carry[tid] = 0;
    if (tid < kSizeBins) s_bin[tid] = 0;
    if (tid == 0) s_mdraft = 0;
    __syncthreads();
#pragma unroll 1
    for (int base = 0, ci = 0; base < U; base += kPlanThreads, ++ci) {
        const int u = base + tid;
        const bool live = u < U;
        const int b = live ? u / p.Hkv : 0, g = live ? u - b * p.Hkv : 0;
        // the unit's three inputs in one round trip
        const int in_mode = live ? p.req_mode[b] : 0, in_len = live ? p.req_len[b] : 0;
        const int in_cnt = live ? p.sparse_cnt[u] : 0;
        long long v[kScanN] = {0, 0, 0, 0, 0, 0, 0, 0};
        ReqInfo r;
        int len = 0, n = 0, ns = 1, cs = 0, rec_rows = 0;
        if (live) {
            int ignored = 0;
            r = check_request(p, in_mode, in_len, g == 0 ? &bad : &ignored, &len);  // request problems flagged once
            cs = unit_split(p, r, in_cnt, &n, &ns, &bad);
            rec_rows = ns > 1 ? (r.mode == 1 ? M : G) : 0;
            if (g == 0) {
                v[0] = r.mode == 1 ? p.k + 1 : 1;
                v[1] = len;
                v[2] = r.mode == 1;
                v[3] = r.mode == 1 ? (long long)p.Hq * (p.k + 1) * len : 0;
            }
            if (r.mode == 1) v[4] = ns; else v[5] = ns;
            v[6] = (long long)ns * rec_rows;
            v[7] = rec_rows > 0 && r.mode == 1;
        }
        long long tot[kScanN];
        block_scan8(v, tot);
        // A draft unit's place in its size bin.  The units of a warp with the same bin and split
        // count take consecutive places through one shared atomic (the whole warp is here,
        // converged after the scan), so the bin counters see a few atomics per warp and the
        // items of neighbouring units are written next to each other.
        int bin_place = 0;
        if (by_size) {
            const bool placed = live && r.mode != 1 && ns > 0;
            const int bin = placed ? size_bin(cs) : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, bin) & __match_any_sync(0xffffffffu, placed ? ns : -1);
            if (placed) {
                const int lane = tid & 31, leader = __ffs(peers) - 1;
                int first = 0;
                if (lane == leader) first = atomicAdd(&s_bin[bin], __popc(peers) * ns);
                bin_place = __shfl_sync(peers, first, leader) + __popc(peers & ((1u << lane) - 1)) * ns;
            }
        }
        if (live) {
            if (g == 0) {
                r.q_off = (int)(carry[0] + v[0]);
                r.vidx = (int)(carry[2] + v[2]);
                p.req[b] = r;
                p.kv_off[b] = carry[1] + v[1];
                p.logit_off[b] = carry[3] + v[3];
            }
            UnitInfo ui;
            ui.nsplit = ns;
            ui.rec_rows = rec_rows;
            ui.rec_base = (int)(carry[6] + v[6]);
            // draft items follow every verify item; their bases are relative here (the place
            // in the size bin, or among the drafts in unit order) and fixed up below
            if (r.mode == 1)
                ui.item_base = (int)(carry[4] + v[4]);
            else if (by_size)
                ui.item_base = bin_place;
            else
                ui.item_base = (int)(carry[5] + v[5]);
            p.unit[u] = ui;
            if (in_regs) {
#pragma unroll
                for (int k = 0; k < kRegChunks; ++k)
                    if (k == ci) {
                        modek[k] = r.mode;
                        nk[k] = n;
                        nsk[k] = ns;
                        csk[k] = cs;
                        itemk[k] = ui.item_base;
                    }
            }
            if (rec_rows > 0) {
                // the request's first query row and verify index: the exclusive prefixes at
                // its g = 0 unit, which precedes this one in the scan
                const int qrows = r.mode == 1 ? p.k + 1 : 1;
                const long long q_off = carry[0] + v[0] - (g > 0 ? qrows : 0);
                const long long vidx = carry[2] + v[2] - (g > 0 ? (r.mode == 1) : 0);
                MergeUnit mu;
                mu.rec_base = ui.rec_base;
                mu.nrows = rec_rows;
                mu.nrec = ns;
                mu.verify = r.mode == 1;
                mu.orow0 = q_off * p.Hq + (long long)g * G;
                mu.lse0 = r.mode == 1 ? (vidx * p.Hq + (long long)g * G) * (p.k + 1) : -1;
                p.merge_units[r.mode == 1 ? carry[7] + v[7] : U - 1 - atomicAdd(&s_mdraft, 1)] = mu;
            }
        }
        __syncthreads();  // every thread has read this chunk's carries
        if (tid == 0) {
#pragma unroll
            for (int i = 0; i < kScanN; ++i) carry[i] += tot[i];
        }
        __syncthreads();
    }
    const long long ver_items = carry[4];
    if (by_size && tid < 32) {  // each size bin's first item: after the verify items, largest bin first
        static_assert(kSizeBins <= 32, "one warp lays out the bins");
        const int own = tid < kSizeBins ? s_bin[tid] : 0;
        int x = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (tid >= o) x += y;
        }
        if (tid < kSizeBins) s_bin[tid] = x - own + (int)ver_items;
    }
    __syncthreads();
    if (tid == 0) {
        p.hdr->num_items = (int)(carry[4] + carry[5]);
        p.hdr->num_units = U;
        p.hdr->num_merge = (int)carry[7];
        p.hdr->num_merge_draft = s_mdraft;
    }
    // Emit the items, with the draft units' bases made absolute.
    if (in_regs) {
#pragma unroll
        for (int k = 0; k < kRegChunks; ++k) {
            const int u = k * kPlanThreads + tid;
            if (u < U) {
                int item = itemk[k];
                if (modek[k] != 1) {
                    item += by_size ? s_bin[size_bin(csk[k])] : (int)ver_items;
                    p.unit[u].item_base = item;
                }
                emit_items(p, u, modek[k], nk[k], nsk[k], csk[k], item);
            }
        }
    } else {
        for (int u = tid; u < U; u += kPlanThreads) {  // each thread re-reads only the unit it wrote itself
            const int b = u / p.Hkv;
            int len, dummy = 0;
            const ReqInfo r = check_request(p, p.req_mode[b], p.req_len[b], &dummy, &len);
            UnitInfo ui = p.unit[u];
            int n, ns;
            const int cs = unit_split(p, r, p.sparse_cnt[u], &n, &ns, &dummy);
            if (r.mode != 1) {
                ui.item_base += by_size ? s_bin[size_bin(cs)] : (int)ver_items;
                p.unit[u].item_base = ui.item_base;
            }
            emit_items(p, u, r.mode, n, ns, cs, ui.item_base);
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
    p.merge_units = reinterpret_cast<MergeUnit *>(a.ws + a.lay.merge_units);
    p.items = reinterpret_cast<Item *>(a.ws + a.lay.items);
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.k = a.k;
    p.max_sparse = a.max_sparse;
    p.max_len = a.max_len;
    p.vchunk = a.vchunk;
    p.dchunk = a.dchunk;
    p.schedule = a.schedule;
    // a programmatic dependent of the kernel before it: its launch overlaps that kernel's tail
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, plan_kernel, p);
}

}  // namespace pillar
