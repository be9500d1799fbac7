// pillar_topk.cu -- next critical lists from the verify dump.
//
// "SparseSpec-MLSys26", 核心方法 / PillarAttn: the verify kernel dumps logits
// and LSE; exact softmax scores are rematerialised from them, averaged over
// the k draft rows and the query heads of one GQA group, and the Top-K
// positions (K = ceil(s*len)) are the critical set of the next k draft steps.
//
//   score[v][g][t] = 1/(R*G) * sum_{r in [row_lo,row_hi)} sum_{h in group g}
//                    exp(logit[v][h][r][t] - lse[v][h][r])
//
// Two kernels:
//   1. topk_scores: a flat, bandwidth-bound pass over the R*G logit rows of
//      every (verify request, KV head), 2048 positions per CTA, coalesced
//      loads; writes fp32 scores (scratch in the workspace, L2-resident for
//      the next kernel at the usual sizes).
//   2. topk_select: one CTA per (verify request, KV head): the K-th largest
//      score, on the order-preserving uint32 key of the (non-negative) fp32
//      score, by a radix select whose first digit is the key's top 11 bits
//      (exponent and three mantissa bits), histogrammed while the keys are
//      loaded; the keys of the bucket that holds the K-th largest are then
//      gathered and the two remaining 10-bit digits are resolved on them alone
//      (a byte-wise radix select over every key stands in when that bucket is
//      too large to gather).  An ordered compaction then keeps everything
//      above the threshold plus the lowest positions equal to it -- the output
//      comes out ascending with no sort.
// The two are chained by programmatic dependent launch: the select grid is
// scheduled while the scores finish and waits for them before reading.
#include "pillar_device.cuh"

namespace pillar {

struct TopkParams {
    const float *logits, *lse;
    const int *req_len, *group_map, *K;
    int *next_idx, *next_cnt;
    WsHeader *hdr;
    TopkRow *rows;
    float *scores;
    int B, V, Hq, Hkv, G, k, row_lo, row_hi, max_topk, max_len, smem_keys;
};

// L_v of verify request v, or -1 when group_map[v] names no request of the
// batch (that request is then skipped and flagged).
__device__ __forceinline__ int verify_len(const TopkParams &p, int v) {
    const int b = p.group_map[v];
    return (b >= 0 && b < p.B) ? p.req_len[b] : -1;
}

constexpr int kScoreThreads = 256;
constexpr int kScorePerThread = 2;
constexpr int kScoreRowBatch = 8;  // logit rows whose loads are in flight together
constexpr int kScoreChunk = kScoreThreads * kScorePerThread;
constexpr int kSelectThreads = 1024;
constexpr int kSelectSmemKeys = 40 * 1024;  // keys kept in shared memory (160 KB); longer rows stay in global
constexpr int kSelectWarps = kSelectThreads / 32;
constexpr int kCoarseShift = 20;                   // first digit: key bits 30..20
constexpr int kCoarseBins = 1 << (31 - kCoarseShift);
constexpr int kFineBins = 1 << 10;                 // then bits 19..10 and 9..0
constexpr int kCandCap = 4096;                     // keys of the first digit's bucket kept for the fine digits
// shared memory after the keys: coarse histogram, two fine histograms, candidates, per-warp byte histograms
constexpr size_t kSelectScratchBytes =
    sizeof(uint32_t) * (kCoarseBins + 2 * kFineBins + kCandCap + kSelectWarps * 256);

// Offsets of verify request v in the packed logits (sums over v' < v of
// Hq*(k+1)*max(L_v', 0), the offsets the attention planner gives the dump)
// and in the scores scratch (sums of Hkv*min(max(L_v', 0), max_len), so that
// a bad length can never push a later request past the workspace).  A request
// whose group_map entry is out of range counts as length 0.
// Warp 0 computes them; every thread of the block gets them.
__device__ void verify_offsets(const TopkParams &p, int v, long long *lg_off, long long *sc_off) {
    __shared__ long long s_off[2];
    if (threadIdx.x < 32) {
        long long s = 0, c = 0;
        for (int i = threadIdx.x; i < v; i += 32) {
            const int l = verify_len(p, i);
            s += l < 0 ? 0 : l;
            c += l < 0 ? 0 : (l > p.max_len ? p.max_len : l);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            s += __shfl_xor_sync(0xffffffffu, s, o);
            c += __shfl_xor_sync(0xffffffffu, c, o);
        }
        if (threadIdx.x == 0) {
            s_off[0] = s * p.Hq * (p.k + 1);
            s_off[1] = c * p.Hkv;
        }
    }
    __syncthreads();
    *lg_off = s_off[0];
    *sc_off = s_off[1];
}

// Exponent offset of the score pass: each term is formed as
// 2^(24 + (logit - lse) log2 e) and the sum is scaled by 2^-24 at the end, so
// the fast base-2 exponential (which flushes results below 2^-126) still
// yields every term that is representable in fp32 after the scaling.
constexpr float kExpOffset = 24.f;

// Accumulates this thread's positions t0 + threadIdx.x + e*kScoreThreads over
// the (padded) rows; kWhole: every position is inside the row.
template <bool kWhole>
__device__ __forceinline__ void score_rows(const TopkParams &p, const float *s_c, const long long *s_row,
                                           int nrows_pad, int t0, int L, float (&acc)[kScorePerThread]) {
    const float *base = p.logits + t0 + threadIdx.x;
    for (int i0 = 0; i0 < nrows_pad; i0 += kScoreRowBatch) {
        float x[kScoreRowBatch][kScorePerThread];
#pragma unroll
        for (int ii = 0; ii < kScoreRowBatch; ++ii) {
            const float *row = base + s_row[i0 + ii];
#pragma unroll
            for (int e = 0; e < kScorePerThread; ++e)
                x[ii][e] = (kWhole || t0 + e * kScoreThreads + (int)threadIdx.x < L) ? __ldcs(row + e * kScoreThreads)
                                                                                      : neg_inf();
        }
#pragma unroll
        for (int ii = 0; ii < kScoreRowBatch; ++ii) {
            const float c = s_c[i0 + ii];
#pragma unroll
            for (int e = 0; e < kScorePerThread; ++e) acc[e] += ex2_approx(fmaf(x[ii][e], kLog2e, c));
        }
    }
}

__global__ void __launch_bounds__(kScoreThreads) topk_scores_kernel(const TopkParams p) {
    // The select kernel may be scheduled now; it reads the scores only after
    // this grid has completed.  Nothing here is read or written before the
    // kernels ahead on the stream are complete.
    pdl_launch_dependents();
    pdl_wait_prerequisites();
    // The workspace's error word starts the call at zero: no block of this grid writes it, and
    // the select (the only kernel of the call that flags) runs once this grid has completed.
    // No memset has to come between the attention's kernels and this one.
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) p.hdr->err = 0;
    // the verify requests in the reverse of the order in which the attention pass wrote their
    // logits: the most recently written rows, the likeliest to be still in L2, are read first,
    // before the pass's own reads push them out
    const int v = (int)(gridDim.z - 1 - blockIdx.z), g = blockIdx.y;
    const int L = verify_len(p, v);
    const int t0 = blockIdx.x * kScoreChunk;
    const bool recorder = blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0;  // writes the request's record
    if (L < 0 || L > p.max_len) {  // skipped; the select flags it from the record
        if (recorder) p.rows[v] = TopkRow{-1, 0, 0};
        return;
    }
    if (L == 0 && recorder) p.rows[v] = TopkRow{0, p.K[v], 0};
    if (t0 >= L) return;
    long long lg_off, sc_off;
    verify_offsets(p, v, &lg_off, &sc_off);
    if (recorder) p.rows[v] = TopkRow{L, p.K[v], sc_off};
    const int R = p.row_hi - p.row_lo, nrows = R * p.G;
    const int nrows_pad = (nrows + kScoreRowBatch - 1) / kScoreRowBatch * kScoreRowBatch;
    // per averaged row: its offset in the logits and 24 - lse*log2(e); the
    // padding rows repeat row 0's offset and contribute 2^-inf = 0, and so
    // does a row that saw no position (LSE -inf, every logit -inf)
    __shared__ float s_c[kMaxRows];
    __shared__ long long s_row[kMaxRows];
    static_assert(kMaxRows % kScoreRowBatch == 0 && kMaxRows <= kScoreThreads, "row tables");
    if (threadIdx.x < nrows_pad) {
        const int i = threadIdx.x, ir = i < nrows ? i : 0;
        const int h = g * p.G + ir / R, r = p.row_lo + ir % R;
        const float lse = i < nrows ? p.lse[((long long)v * p.Hq + h) * (p.k + 1) + r] : neg_inf();
        s_c[i] = lse > neg_inf() ? kExpOffset - lse * kLog2e : neg_inf();
        s_row[i] = lg_off + ((long long)h * (p.k + 1) + r) * L;
    }
    __syncthreads();
    float acc[kScorePerThread];
#pragma unroll
    for (int e = 0; e < kScorePerThread; ++e) acc[e] = 0.f;
    if (t0 + kScoreChunk <= L)
        score_rows<true>(p, s_c, s_row, nrows_pad, t0, L, acc);
    else
        score_rows<false>(p, s_c, s_row, nrows_pad, t0, L, acc);
    const float scale = 0x1p-24f / (float)nrows;  // undo the exponent offset; mean over the R*G rows
    float *dst = p.scores + sc_off + (long long)g * L;
#pragma unroll
    for (int e = 0; e < kScorePerThread; ++e) {
        const int t = t0 + e * kScoreThreads + threadIdx.x;
        if (t < L) dst[t] = acc[e] * scale;
    }
}

// Exclusive scans of two ints per thread over the select block, together
// (one set of shuffles and barriers); *total gets the block totals.
__device__ int2 select_block_scan2(int a, int b, int2 *total) {
    __shared__ int2 ws[kSelectWarps];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int xa = a, xb = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, xa, o), yb = __shfl_up_sync(0xffffffffu, xb, o);
        if (lane >= o) xa += ya, xb += yb;
    }
    if (lane == 31) ws[wid] = make_int2(xa, xb);
    __syncthreads();
    if (wid == 0) {
        int2 t = ws[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ya = __shfl_up_sync(0xffffffffu, t.x, o), yb = __shfl_up_sync(0xffffffffu, t.y, o);
            if (lane >= o) t.x += ya, t.y += yb;
        }
        ws[lane] = t;
    }
    __syncthreads();
    const int2 base = wid ? ws[wid - 1] : make_int2(0, 0);
    *total = ws[kSelectWarps - 1];
    __syncthreads();
    return make_int2(base.x + xa - a, base.y + xb - b);
}

__device__ __forceinline__ uint32_t score_key(float s) { return __float_as_uint(s) & 0x7fffffffu; }
// The key of position t (rows too long for shared memory are read from the scores themselves).
__device__ __forceinline__ uint32_t key_at(const uint32_t *keys, int t) { return keys[t] & 0x7fffffffu; }

// The bin of hist[0, NB) that holds the rem-th largest key (rem >= 1, bins
// walked from the top) and the key's rank inside that bin, found by the whole
// block: thread i owns the NB/1024 bins below NB-1-i*NB/1024, a warp scan and a
// scan of the 32 warp totals give every thread the count above its bins, and
// the thread whose bins cross rem writes the results (read after the closing
// barrier).  s_wsum: 32 words of scratch.
template <int NB>
__device__ __forceinline__ void block_find_bin(const uint32_t *hist, uint32_t rem, uint32_t *s_wsum, uint32_t *s_bin,
                                               uint32_t *s_rank) {
    constexpr int kPer = NB / kSelectThreads;
    static_assert(kPer == 1 || kPer == 2, "bins per thread");
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int top = NB - 1 - tid * kPer;
    uint32_t c[kPer];
    if (kPer == 2) {  // the thread's two bins in one 8-byte load
        const uint2 pr = *reinterpret_cast<const uint2 *>(hist + top - 1);
        c[0] = pr.y;
        c[kPer - 1] = pr.x;
    } else {
        c[0] = hist[top];
    }
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) sum += c[j];
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[w] = incl;
    __syncthreads();
    const uint32_t ws = s_wsum[lane];
    uint32_t wincl = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, wincl, o);
        if (lane >= o) wincl += y;
    }
    const uint32_t above_warp = __shfl_sync(0xffffffffu, wincl - ws, w);
    uint32_t cum = above_warp + incl - sum;
    if (cum < rem && cum + sum >= rem) {
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (cum + c[j] >= rem) {
                *s_bin = (uint32_t)(top - j);
                *s_rank = rem - cum;
                break;
            }
            cum += c[j];
        }
    }
    __syncthreads();
}

// Byte-wise radix select of the rem-th largest of L keys (every key visited in
// each of four passes): the stand-in for a first-digit bucket too large to
// gather.  Returns the key; *rank gets its rank among the keys equal to it.
__device__ uint32_t radix_select_bytes(const uint32_t *keys, int L, uint32_t rem, uint32_t (*whist)[256],
                                       uint32_t *rank) {
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_prefix, s_mask, s_remaining;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_prefix = 0;
        s_mask = 0;
        s_remaining = rem;
    }
    __syncthreads();
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t *myhist = whist[tid >> 5];
        for (int i = tid & 31; i < 256; i += 32) myhist[i] = 0;
        __syncwarp();
        const uint32_t prefix = s_prefix, mask = s_mask;
        for (int t = tid; t < L; t += blockDim.x) {
            const uint32_t key = key_at(keys, t);
            if ((key & mask) == prefix) atomicAdd(&myhist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t c = 0;
#pragma unroll 8
            for (int w = 0; w < kSelectWarps; ++w) c += whist[w][tid];
            hist[tid] = c;
        }
        __syncthreads();
        if (tid < 32) {
            const uint32_t r = s_remaining;
            __syncwarp();  // every lane has read s_remaining before it changes
            uint32_t bin = 0, rk = 0;
            bool mine = false;
            {
                // (find_bin writes from one lane; the lane also updates the prefix)
                constexpr int kPer = 8;
                const int lane = tid, top = 255 - lane * kPer;
                uint32_t sum = 0;
#pragma unroll
                for (int i = 0; i < kPer; ++i) sum += hist[top - i];
                uint32_t incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const uint32_t before = incl - sum;
                if (before < r && incl >= r) {
                    uint32_t cum = before;
                    for (int i = 0; i < kPer; ++i) {
                        const uint32_t c = hist[top - i];
                        if (cum + c >= r) {
                            bin = (uint32_t)(top - i);
                            rk = r - cum;
                            mine = true;
                            break;
                        }
                        cum += c;
                    }
                }
            }
            if (mine) {
                s_prefix = prefix | (bin << shift);
                s_mask = mask | (255u << shift);
                s_remaining = rk;
            }
        }
        __syncthreads();
    }
    *rank = s_remaining;
    return s_prefix;
}

__global__ void __launch_bounds__(kSelectThreads, 1) topk_select_kernel(const TopkParams p) {
    extern __shared__ uint32_t smem[];
    uint32_t *skeys = smem;
    uint32_t *coarse = smem + p.smem_keys;
    uint32_t *fine_a = coarse + kCoarseBins, *fine_b = fine_a + kFineBins;
    uint32_t *cand = fine_b + kFineBins;
    uint32_t(*whist)[256] = reinterpret_cast<uint32_t(*)[256]>(cand + kCandCap);
    __shared__ uint32_t s_bin, s_rank, s_ncand, s_wsum[kSelectWarps];
    pdl_launch_dependents();   // the next kernel (the next step's planner) may be scheduled now
    pdl_wait_prerequisites();  // the scores and the score pass's records are complete and visible
    const int v = blockIdx.y, g = blockIdx.x, tid = threadIdx.x;
    const TopkRow rec = p.rows[v];
    const int L = rec.L;
    if (L < 0 || L > p.max_len) {  // a request the score pass skipped (group_map entry or length)
        if (tid == 0) {
            p.next_cnt[v * p.Hkv + g] = 0;
            if (g == 0) atomicOr(&p.hdr->err, PILLAR_FLAG_REQUEST);
        }
        return;
    }
    int K = rec.K;
    K = K < 0 ? 0 : (K > L ? L : K);
    if (K > p.max_topk) {
        if (tid == 0) atomicOr(&p.hdr->err, PILLAR_FLAG_TOPK);
        K = p.max_topk;
    }
    int *dst = p.next_idx + ((long long)v * p.Hkv + g) * p.max_topk;
    if (tid == 0) p.next_cnt[v * p.Hkv + g] = K;
    if (K == 0) return;
    if (K == L) {
        for (int t = tid; t < L; t += blockDim.x) dst[t] = t;
        return;
    }
    const float *sc = p.scores + rec.sc_off + (long long)g * L;
    for (int i = tid; i < kCoarseBins; i += kSelectThreads) coarse[i] = 0;
    for (int i = tid; i < 2 * kFineBins; i += kSelectThreads) fine_a[i] = 0;
    if (tid == 0) s_ncand = 0;
    __syncthreads();
    // The keys (kept in shared memory when they fit) and the histogram of their first digit.
    const bool in_smem = L <= p.smem_keys;
    {
        constexpr int kU = 8;  // independent loads in flight per thread
        for (int t0 = 0; t0 < L; t0 += kU * kSelectThreads) {
            float x[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int t = t0 + u * kSelectThreads + tid;
                x[u] = t < L ? sc[t] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int t = t0 + u * kSelectThreads + tid;
                if (t < L) {
                    const uint32_t key = score_key(x[u]);
                    if (in_smem) skeys[t] = key;
                    atomicAdd(&coarse[key >> kCoarseShift], 1u);
                }
            }
        }
    }
    // (scores are >= 0: their keys need no sign fix)
    const uint32_t *keys = in_smem ? skeys : reinterpret_cast<const uint32_t *>(sc);
    __syncthreads();
    block_find_bin<kCoarseBins>(coarse, (uint32_t)K, s_wsum, &s_bin, &s_rank);
    const uint32_t b1 = s_bin, r1 = s_rank;
    // Gather the keys of that bucket.
    for (int t = tid; t < L; t += kSelectThreads) {
        const uint32_t key = key_at(keys, t);
        if ((key >> kCoarseShift) == b1) {
            const uint32_t i = atomicAdd(&s_ncand, 1u);
            if (i < (uint32_t)kCandCap) cand[i] = key;
        }
    }
    __syncthreads();
    const int ncand = (int)s_ncand;
    uint32_t T;
    int need_eq;
    if (ncand <= kCandCap) {
        // the two fine digits, on the candidates alone
        for (int i = tid; i < ncand; i += kSelectThreads) atomicAdd(&fine_a[(cand[i] >> 10) & 1023u], 1u);
        __syncthreads();
        block_find_bin<kFineBins>(fine_a, r1, s_wsum, &s_bin, &s_rank);
        const uint32_t b2 = s_bin, r2 = s_rank;
        for (int i = tid; i < ncand; i += kSelectThreads) {
            const uint32_t key = cand[i];
            if (((key >> 10) & 1023u) == b2) atomicAdd(&fine_b[key & 1023u], 1u);
        }
        __syncthreads();  // (also: every thread has read s_bin and s_rank before they change)
        block_find_bin<kFineBins>(fine_b, r2, s_wsum, &s_bin, &s_rank);
        T = (b1 << kCoarseShift) | (b2 << 10) | s_bin;
        need_eq = (int)s_rank;
    } else {
        uint32_t rk;
        T = radix_select_bytes(keys, L, (uint32_t)K, whist, &rk);
        need_eq = (int)rk;
    }

    // Ordered compaction: each thread owns a contiguous run of positions (an odd run length, so
    // that the 32 lanes of a warp read 32 different shared-memory banks).
    const int per = ((L + blockDim.x - 1) / blockDim.x) | 1;
    const int tb = min(L, tid * per), te = min(L, tb + per);
    int cgt = 0, ceq = 0;
    for (int t = tb; t < te; ++t) {
        const uint32_t key = key_at(keys, t);
        cgt += key > T;
        ceq += key == T;
    }
    int2 tot;
    const int2 before = select_block_scan2(cgt, ceq, &tot);
    int out = before.x + min(before.y, need_eq);
    int eq_rank = before.y;
    for (int t = tb; t < te; ++t) {
        const uint32_t key = key_at(keys, t);
        if (key > T) {
            dst[out++] = t;
        } else if (key == T) {
            if (eq_rank < need_eq) dst[out++] = t;
            ++eq_rank;
        }
    }
}

cudaError_t launch_topk_select(const TopkArgs &a, cudaStream_t st) {
    TopkParams p;
    p.logits = a.logits;
    p.lse = a.lse;
    p.req_len = a.req_len;
    p.group_map = a.group_map;
    p.K = a.K;
    p.next_idx = a.next_idx;
    p.next_cnt = a.next_cnt;
    p.hdr = reinterpret_cast<WsHeader *>(a.ws);
    p.rows = a.rows;
    p.scores = a.scores;
    p.B = a.B;
    p.V = a.V;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.k = a.k;
    p.row_lo = a.row_lo;
    p.row_hi = a.row_hi;
    p.max_topk = a.max_topk;
    p.max_len = a.max_len;
    p.smem_keys = min((a.max_len + 3) & ~3, kSelectSmemKeys);  // (a multiple of 4: the histograms after the keys are 16-byte aligned)
    if (p.V == 0) return cudaSuccess;
    // launch attributes, once per device context
    static unsigned long long configured[kMaxDevices] = {};
    int dev = 0;
    unsigned long long ctx = 0;
    cudaError_t e = current_device_context(&dev, &ctx);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const size_t sel_smem = sizeof(uint32_t) * (size_t)p.smem_keys + kSelectScratchBytes;
    if (ctx == 0 || __atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE) != ctx) {
        e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(sizeof(uint32_t) * kSelectSmemKeys + kSelectScratchBytes));
        if (e != cudaSuccess) return e;
        e = current_device_context(&dev, &ctx);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[dev], ctx, __ATOMIC_RELEASE);
    }
    // Both kernels are programmatic dependents of the one before them on the
    // stream: their launch overlaps its tail, and each waits for it to
    // complete before touching memory.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.max_len + kScoreChunk - 1) / kScoreChunk, p.Hkv, p.V);
    cfg.blockDim = dim3(kScoreThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, topk_scores_kernel, p);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(p.Hkv, p.V);
    cfg.blockDim = dim3(kSelectThreads);
    cfg.dynamicSmemBytes = sel_smem;
    return cudaLaunchKernelEx(&cfg, topk_select_kernel, p);
}

}  // namespace pillar
