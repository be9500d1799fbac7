// pillar_internal.h -- workspace layout and launch constants shared by the
// planner, the unified attention kernel, the Top-K kernels and the host API.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/pillar.h"

namespace pillar {

constexpr int kTileKeys = 64;          // keys staged per pipeline stage
constexpr int kConsumerWarps = 4;      // compute warps per CTA (one per TMEM lane quadrant)
constexpr int kLoaderWarps = 4;        // gather warps per CTA (each fetches 64 / kLoaderWarps rows of a tile)
constexpr int kEpiWarps = 4;           // O-epilogue warps (one per TMEM lane quadrant)
// four warp groups: consumers | loaders | resolver, MMA issuer and two spare warps | epilogue warps
constexpr int kThreads = 16 * 32;
constexpr int kMaxRows = 64;           // (k+1)*G bound of a verify tile
constexpr int kMaxG = 8;               // query heads per KV head
// Default verify item size: 1024 keys for contexts shorter than kLongContext
// positions, 2048 from there on (fewer items and partial records where the
// per-item cost weighs, enough items to balance the CTAs below).
constexpr int kDefaultVerifyChunk = 1024;
constexpr int kLongVerifyChunk = 2048;
constexpr int kLongContext = 8192;
constexpr int kDefaultDraftChunk = 2048;
constexpr int kMaxChunk = 2048;        // item key bound (sizes the resolved row lists in shared memory)
constexpr int kPlanThreads = 1024;
constexpr unsigned long long kWaitTimeoutNs = 1000ull * 1000ull * 1000ull;  // 1 s: the default wait bound, and the drains'

// Request and unit records written by the planner.
struct ReqInfo {
    int q_off;      // first query row
    int vidx;       // index among verify requests (verify only)
    int len;        // L_b, clamped to [0, max_len]
    int mode;       // 0 draft, 1 verify, -1 invalid (skipped)
};

struct UnitInfo {
    int nsplit;     // work items of this (request, KV head)
    int item_base;  // index of its first item
    int rec_base;   // first partial row of its items (see AttnLayout)
    int rec_rows;   // partial rows written per item of a split unit: M (verify), G (draft); 0 if not split
};

// A split (request, KV head) as the merge sees it: where its partial rows
// are and where the combined rows go.
struct MergeUnit {
    int rec_base;    // first partial row of its first item
    int nrows;       // rows per item: M (verify), G (draft)
    int nrec;        // items (partial records per row)
    int verify;
    long long orow0;  // output row of its row 0: q_off*Hq + g*G (row j*G + gi -> orow0 + j*Hq + gi)
    long long lse0;   // verify: LSE index of its row 0, (vidx*Hq + g*G)*(k+1) (row j*G + gi -> lse0 + gi*(k+1) + j)
};

struct Item {
    int unit;       // b * Hkv + g
    int begin;      // first key (verify: position; draft: list index)
    int end;        // one past the last key
    int split;      // index among the unit's items
};

struct WsHeader {
    int err;        // PILLAR_FLAG_* bits
    int num_items;
    int item_counter;
    int num_units;
    int num_merge;        // verify units whose partials the merge kernel combines (merge_units[0, num_merge))
    int num_merge_draft;  // draft units it combines (merge_units[num_units - num_merge_draft, num_units))
    int pad[58];          // keeps the arrays 256-byte aligned
};

// Byte offsets of the attention workspace sections.
struct AttnLayout {
    size_t req, kv_off, logit_off, unit, merge_units, items, part_o, part_lse, total;
    long long max_items, max_rec_rows;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// One-time per-context set-up (launch attributes, symbol addresses).  A
// device's context is told apart by its process-unique id (cuCtxGetId), so
// a context re-created after cudaDeviceReset is set up again.
constexpr int kMaxDevices = 64;

// The current device and the unique id of the context current on it (0
// when no context is current yet: the caller then sets up and asks again).
cudaError_t current_device_context(int *dev, unsigned long long *ctx_id);

// 0: the default, chosen per request by its context length (see kLongContext)
inline int verify_chunk_of(const pillar_shape_t &s) { return s.verify_chunk > 0 ? s.verify_chunk : 0; }
inline int draft_chunk_of(const pillar_shape_t &s) { return s.draft_chunk > 0 ? s.draft_chunk : kDefaultDraftChunk; }

// Partials: an item of a (request, KV head) split over several items writes
// its rows (M = (k+1)*G for verify, G for draft); each partial row is D fp32
// values (the normalised output) plus one fp32 LSE.
inline AttnLayout attn_layout(const pillar_shape_t &s) {
    AttnLayout l{};
    const long long B = s.B, U = (long long)s.B * s.Hkv;
    const int G = s.Hq / s.Hkv;
    // (the default verify chunk is bounded by its smaller size: the most items)
    const long long vc = verify_chunk_of(s) > 0 ? verify_chunk_of(s) : kDefaultVerifyChunk, dc = draft_chunk_of(s);
    long long per_unit = (s.max_len + vc - 1) / vc;
    long long dsplit = (s.max_sparse + dc - 1) / dc;
    if (dsplit > per_unit) per_unit = dsplit;
    if (per_unit < 1) per_unit = 1;
    l.max_items = U * per_unit;
    const long long per_item = (long long)(s.k + 1) * G;
    l.max_rec_rows = l.max_items * per_item;
    size_t off = sizeof(WsHeader);
    l.req = off;        off = align256(off + sizeof(ReqInfo) * B);
    l.kv_off = off;     off = align256(off + sizeof(long long) * B);
    l.logit_off = off;  off = align256(off + sizeof(long long) * B);
    l.unit = off;       off = align256(off + sizeof(UnitInfo) * U);
    l.merge_units = off; off = align256(off + sizeof(MergeUnit) * U);
    l.items = off;      off = align256(off + sizeof(Item) * l.max_items);
    l.part_o = off;     off = align256(off + sizeof(float) * (size_t)l.max_rec_rows * s.D);
    l.part_lse = off;   off = align256(off + sizeof(float) * (size_t)l.max_rec_rows);
    l.total = off;
    return l;
}

// Top-K workspace: header (error word), one record per verify request (what
// the score pass found out about it, for the select), then the packed scores
// [V][Hkv][L_v].
struct TopkRow {
    int L;            // L_v, or -1 when the request is skipped
    int K;            // its budget as given
    long long sc_off; // offset of its scores [Hkv][L_v] in the scores scratch
};
inline size_t topk_rows_offset() { return sizeof(WsHeader); }
inline size_t topk_scores_offset(int V) { return align256(sizeof(WsHeader) + sizeof(TopkRow) * (size_t)V); }
inline size_t topk_ws_bytes(const pillar_shape_t &s, int V) {
    return align256(topk_scores_offset(V) + sizeof(float) * (size_t)V * s.Hkv * (size_t)s.max_len);
}

// ------------------------------------------------------------------ launchers
// (host side; each kernel translation unit turns these into its kernel
// parameters and enqueues on the given stream)

struct PlanArgs {
    const int *req_mode, *req_len, *sparse_cnt;
    char *ws;
    AttnLayout lay;
    int B, Hq, Hkv, k, max_sparse, max_len, vchunk, dchunk;
    int schedule;  // PILLAR_SCHEDULE_*
};
cudaError_t launch_plan(const PlanArgs &a, cudaStream_t st);

struct AttnArgs {
    const uint16_t *q, *k_pool, *v_pool;
    const int *slot_table, *sparse_idx;
    const int *sparse_slot;  // null, or the slots of the draft lists (layout of sparse_idx)
    uint16_t *out;
    float *logits, *lse;
    char *ws;
    AttnLayout lay;
    long long num_slots;
    int Hq, Hkv, D, k, max_sparse;
    int schedule;  // PILLAR_SCHEDULE_*
    float scale;
    unsigned long long wait_ns;  // bound of every pipeline wait
};
cudaError_t launch_attn(const AttnArgs &a, int grid, cudaStream_t st);

struct TopkArgs {
    const float *logits, *lse;
    const int *req_len, *group_map, *K;
    int *next_idx, *next_cnt;
    char *ws;
    TopkRow *rows;
    float *scores;
    int B, V, Hq, Hkv, k, row_lo, row_hi, max_topk, max_len;
};
cudaError_t launch_topk_select(const TopkArgs &a, cudaStream_t st);

}  // namespace pillar
