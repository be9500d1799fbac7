/*
 * pillar.h -- C ABI of the GB300 (sm_103a) PillarAttn unified step.
 *
 * The method ("SparseSpec-MLSys26", section 核心方法 / PillarAttn):
 *   - a draft request (one query token) attends only its critical-token list,
 *     one list per (request, KV head);
 *   - a verify request (k+1 query tokens, causal among themselves) attends
 *     its full context and, in the same pass, dumps the raw attention logits
 *     and the log-sum-exp of every row;
 *   - from that dump the exact softmax scores are rematerialised, averaged
 *     over the k draft rows and the GQA group's query heads, and the Top-K
 *     positions (K = ceil(s*len)) become the next stride's critical list.
 * With a page-size-1 KV pool every position reaches its K/V row through a
 * per-request slot table, so sparse and full attention share one pipeline
 * and mix freely in one batch (same page, section "Unified batch scheduler
 * + fused attention kernel").
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller (the
 *     phase-bucket functions at the end work on host memory).  The library
 *     allocates nothing and keeps no state between calls, except the launch
 *     attributes it sets once per device context (up to 64 devices) and the
 *     scratch array of pillar_topk_select_noalloc.  Scratch lives in the
 *     caller's workspace (sized by the *_workspace_bytes functions); the
 *     device error word sits inside that workspace.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream: a return of PILLAR_OK means the work was
 *     validated and enqueued.  Data-dependent problems found on the device
 *     (an index or slot out of range, a bad mode or length) are skipped and
 *     recorded in the error word; read it with pillar_get_error.
 *   - Nothing on the device waits without a bound: a wait that runs past
 *     its bound (one second, or the shape's wait_timeout_us) records
 *     PILLAR_FLAG_TIMEOUT and the kernel returns.  The device error word
 *     of the workspace is cleared by every call and reports that call only.
 */
#ifndef PILLAR_H
#define PILLAR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PILLAR_API __attribute__((visibility("default")))
#else
#define PILLAR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define PILLAR_OK 0
#define PILLAR_ERR_ARG (-1)         /* null pointer, bad dimension or unsupported shape */
#define PILLAR_ERR_WORKSPACE (-2)   /* workspace null, misaligned or too small */
#define PILLAR_ERR_CUDA (-3)        /* a CUDA runtime call or launch failed */
#define PILLAR_ERR_DEVICE (-4)      /* pillar_get_error: the device error word is non-zero */
#define PILLAR_ERR_SCRATCH (-5)     /* pillar_topk_select_noalloc: the shape needs more than its built-in scratch */

/* Size of the scratch array compiled into the library for
 * pillar_topk_select_noalloc (16 MiB of scores plus a 256-byte header). */
#define PILLAR_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u + 256u)

/* Bits of the device error word. */
#define PILLAR_FLAG_INDEX 1         /* a critical-list position outside [0, L_b) was skipped */
#define PILLAR_FLAG_SLOT 2          /* a slot outside [0, num_slots) was skipped */
#define PILLAR_FLAG_REQUEST 4       /* req_mode not 0/1, L_b < 0, L_b > max_len, or verify L_b < k+1 */
#define PILLAR_FLAG_COUNT 8         /* sparse_cnt outside [0, max_sparse] (clamped) */
#define PILLAR_FLAG_TIMEOUT 16      /* a bounded device wait gave up; outputs are incomplete */
#define PILLAR_FLAG_TOPK 32         /* a Top-K budget exceeded max_topk (clamped) */

typedef struct pillar_shape {
    int32_t B;             /* requests in the batch (>= 0) */
    int32_t Hq;            /* query heads */
    int32_t Hkv;           /* KV heads; G = Hq / Hkv query heads share one (1 <= G <= 8) */
    int32_t D;             /* head dimension: 64 or 128 */
    int32_t k;             /* stride: a verify request carries k+1 query rows; (k+1)*G <= 64 */
    int32_t max_sparse;    /* row stride of sparse_idx (>= 0) */
    int32_t max_len;       /* upper bound on every req_len; sizes the workspace (>= 1) */
    int32_t row_lo;        /* verify rows [row_lo, row_hi) are averaged by Top-K; */
    int32_t row_hi;        /*   the k draft rows are [1, k+1) */
    int32_t max_topk;      /* row stride of next_idx (>= 1) */
    int32_t verify_chunk;  /* keys per verify work item (multiple of 64, <= 2048); 0: 1024 for
                              contexts under 8192 positions, 2048 from 8192 on */
    int32_t draft_chunk;   /* listed keys per draft work item (multiple of 64, <= 2048; 0 = 2048) */
    int64_t num_slots;     /* rows of k_pool / v_pool */
    float sm_scale;        /* logit scale; 0 means 1/sqrt(D) */
    int32_t schedule;      /* PILLAR_SCHEDULE_* (0: the unified pass) */
    int32_t wait_timeout_us; /* bound on every pipeline wait of pillar_attn_unified, in
                              microseconds (>= 0; 0 means 1000000, one second); a wait that
                              runs past it records PILLAR_FLAG_TIMEOUT and the kernel
                              returns with incomplete outputs.  The waits that let copies
                              and tensor-core work already in flight finish before a CTA
                              exits keep their own one-second bound. */
    int32_t reserved;      /* set to 0 */
} pillar_shape_t;

/*
 * Schedules of pillar_attn_unified.  The unified pass is the method's design
 * ("SparseSpec-MLSys26", Unified batch scheduler + fused attention kernel:
 * one persistent kernel serves draft and verify requests of one batch).  The
 * other schedules exist to measure it against the two alternatives that
 * section compares it with; all of them compute the same outputs.
 *   UNIFIED       draft and verify requests in one persistent pass.
 *   DRAFT_ONLY    the draft requests only; the outputs of verify requests
 *                 (their out rows, logits and LSEs) are left untouched.
 *   VERIFY_ONLY   the verify requests only; draft outputs left untouched.  A
 *                 DRAFT_ONLY call followed by a VERIFY_ONLY call on the same
 *                 buffers is the sequential two-kernel schedule; it writes
 *                 the same values as one UNIFIED call.
 *   UNIFORM_ROWS  one pass in which a draft item takes the verify item's row
 *                 layout (its G rows as the first G of the (k+1)*G row slots,
 *                 the slots of one TMEM lane quadrant) instead of its own
 *                 spread of the G rows over the four quadrants: a joint batch
 *                 without per-mode dispatch.
 *   NAIVE_JOINT   the naive joint batch: the UNIFORM_ROWS row layout for every
 *                 request, work items of the largest size the pipeline takes
 *                 (2048 keys, whatever verify_chunk and draft_chunk say), and
 *                 no dynamic load balancing -- each CTA of the persistent grid
 *                 takes the (request, KV head) units c, c + grid, c + 2 grid,
 *                 ... in batch order and works through all of their items.
 * The device error word is cleared by every call; it reports that call only.
 */
#define PILLAR_SCHEDULE_UNIFIED 0
#define PILLAR_SCHEDULE_DRAFT_ONLY 1
#define PILLAR_SCHEDULE_VERIFY_ONLY 2
#define PILLAR_SCHEDULE_UNIFORM_ROWS 3
#define PILLAR_SCHEDULE_NAIVE_JOINT 4

/*
 * pillar_attn_workspace_bytes -- bytes of workspace pillar_attn_unified
 * needs for this shape (a bound over every batch with req_len <= max_len and
 * sparse_cnt <= max_sparse).  Returns PILLAR_OK or PILLAR_ERR_ARG (a bad
 * shape, or one whose workspace bound would pass 2^50 bytes).
 */
PILLAR_API int pillar_attn_workspace_bytes(const pillar_shape_t *shape, size_t *bytes);

/*
 * pillar_attn_unified -- one unified draft/verify attention step.
 * ("SparseSpec-MLSys26", 核心方法 / PillarAttn: sparse draft attention over
 * the critical set, full verify attention with the logits/LSE dump; and the
 * unified-batch section: page size 1, one fused pass over mixed requests.)
 *
 *   q            [T_q, Hq, D] bf16.  Requests packed in batch order: one row
 *                for a draft request, k+1 rows for a verify request.
 *   k_pool,
 *   v_pool       [num_slots, Hkv, D] bf16: one slot = one token, all heads.
 *   slot_table   int32; request b's L_b slots start at sum_{b'<b} L_b'.
 *                slot_table[off_b + t] is the slot of position t.
 *   req_mode     [B] int32: 0 draft, 1 verify.
 *   req_len      [B] int32: L_b, the context length including the request's
 *                own new tokens.  Verify row j (0..k) sits at position
 *                L_b-(k+1)+j and attends positions [0, L_b-(k+1)+j].
 *   sparse_idx   [B, Hkv, max_sparse] int32 logical positions (draft only);
 *   sparse_cnt   [B, Hkv] int32 list lengths.  Query head h uses KV head
 *                h / G and that head's list, taken literally (a repeated
 *                position counts twice).  An empty list gives a zero output.
 *   out          [T_q, Hq, D] bf16: attention output of every query row.
 *   verify_logits  fp32, packed over the verify requests in batch order:
 *                [V][Hq][k+1][L_v], the scaled logits q.k*scale, -inf where
 *                the row may not look (t beyond its causal limit).
 *   verify_lse   [V][Hq][k+1] fp32: natural-log LSE of each verify row.
 *   workspace    device scratch of at least pillar_attn_workspace_bytes,
 *                256-byte aligned.  Must not be shared by concurrent calls.
 * All pointers are device memory.  Alignment: q, k_pool and v_pool 16 bytes,
 * verify_logits 8 bytes (pairs of logits are stored together), out and the
 * int32 and fp32 arrays 4 bytes; a misaligned pointer is PILLAR_ERR_ARG.
 *
 * Returns PILLAR_OK, PILLAR_ERR_ARG, PILLAR_ERR_WORKSPACE or PILLAR_ERR_CUDA.
 * With B == 0 nothing is launched.
 */
PILLAR_API int pillar_attn_unified(const pillar_shape_t *shape, const uint16_t *q, const uint16_t *k_pool,
                        const uint16_t *v_pool, const int32_t *slot_table, const int32_t *req_mode,
                        const int32_t *req_len, const int32_t *sparse_idx, const int32_t *sparse_cnt,
                        uint16_t *out, float *verify_logits, float *verify_lse, void *workspace,
                        size_t ws_bytes, void *stream);

/*
 * pillar_attn_unified_slotted -- pillar_attn_unified whose draft lists come
 * with their pool slots already translated (as pillar_draft_lists writes
 * them), so that a draft key's K/V rows are reached without the dependent
 * slot-table load ("SparseSpec-MLSys26", Unified batch scheduler + fused
 * attention kernel: page size 1 -- every listed position is one slot).
 *
 *   sparse_slot  [B, Hkv, max_sparse] int32, device memory, 4-byte aligned,
 *                or NULL (then exactly pillar_attn_unified): entry i of
 *                request b's list of KV head h is the slot of position
 *                sparse_idx[b, h, i], i.e. slot_table[off_b + that position].
 *                The positions are still read: one outside [0, L_b) is
 *                skipped and flagged (PILLAR_FLAG_INDEX), and a slot outside
 *                [0, num_slots) is skipped and flagged (PILLAR_FLAG_SLOT).
 *                Verify requests use slot_table as before.
 * All other arguments, results and return codes as pillar_attn_unified.
 */
PILLAR_API int pillar_attn_unified_slotted(const pillar_shape_t *shape, const uint16_t *q, const uint16_t *k_pool,
                                           const uint16_t *v_pool, const int32_t *slot_table,
                                           const int32_t *req_mode, const int32_t *req_len,
                                           const int32_t *sparse_idx, const int32_t *sparse_cnt,
                                           const int32_t *sparse_slot, uint16_t *out, float *verify_logits,
                                           float *verify_lse, void *workspace, size_t ws_bytes, void *stream);

/*
 * pillar_attn_plan + pillar_attn_run -- pillar_attn_unified in two calls, so
 * that one plan serves several runs.  The plan depends only on the batch
 * description (req_mode, req_len, sparse_cnt), which is the same for every
 * layer of a model step; the runs take what differs per layer (q, the pools,
 * the lists, the outputs).  pillar_attn_unified(_slotted) is exactly a plan
 * followed by a run.
 *
 * pillar_attn_plan(shape, req_mode, req_len, sparse_cnt, workspace, ...)
 *   launches the device planner: it clears the workspace's error word and
 *   writes the offsets, work items and partial-record layout into the
 *   workspace.  Arguments as in pillar_attn_unified; with B == 0 it only
 *   clears the error word.
 * pillar_attn_run(shape, q, k_pool, v_pool, slot_table, sparse_idx,
 *                 sparse_slot, out, verify_logits, verify_lse, workspace, ...)
 *   launches the attention kernel and the merge of split units on the plan in
 *   the workspace; sparse_slot may be NULL (as pillar_attn_unified_slotted).
 *   The shape must be the one the plan was made with, the inputs must have the
 *   plan's batch description (the same modes, lengths and list counts), and the
 *   plan must precede the run on the stream (or be complete).  Any number of
 *   runs may follow one plan, one after the other on a stream; the error word
 *   collects the flags of the plan and of every run until pillar_get_error
 *   reads and clears it.
 * Return codes as pillar_attn_unified; a run with B == 0 does nothing.
 */
PILLAR_API int pillar_attn_plan(const pillar_shape_t *shape, const int32_t *req_mode, const int32_t *req_len,
                                const int32_t *sparse_cnt, void *workspace, size_t ws_bytes, void *stream);
PILLAR_API int pillar_attn_run(const pillar_shape_t *shape, const uint16_t *q, const uint16_t *k_pool,
                               const uint16_t *v_pool, const int32_t *slot_table, const int32_t *sparse_idx,
                               const int32_t *sparse_slot, uint16_t *out, float *verify_logits, float *verify_lse,
                               void *workspace, size_t ws_bytes, void *stream);

/*
 * pillar_topk_workspace_bytes -- workspace of pillar_topk_select for V
 * verify requests of length <= max_len.  Returns PILLAR_OK or PILLAR_ERR_ARG
 * (a bad shape, V < 0, or V * Hkv * max_len fp32 scores past 2^50 bytes).
 */
PILLAR_API int pillar_topk_workspace_bytes(const pillar_shape_t *shape, int32_t V, size_t *bytes);

/*
 * pillar_topk_select -- the next stride's critical lists from one verify
 * pass ("SparseSpec-MLSys26", 核心方法 / PillarAttn: rematerialise exact
 * scores from the dumped logits and LSE, average over the k draft rows and
 * the GQA group's heads, take Top-K).
 *
 *   V              number of verify requests (host value).
 *   verify_logits,
 *   verify_lse     as written by pillar_attn_unified.
 *   req_len        [B] int32, as given to pillar_attn_unified.
 *   group_map      [V] int32: batch index b of the v-th verify request, in
 *                  increasing order (it fixes L_v and the logits offsets).
 *                  A request whose entry lies outside [0, B), or whose
 *                  length is negative or above max_len, is skipped
 *                  (next_cnt 0) and flagged PILLAR_FLAG_REQUEST; it counts
 *                  as length 0 in the offsets of the requests after it.
 *   K              [V] int32: K_v, the number of positions to keep; clamped
 *                  to [0, L_v], and to max_topk with PILLAR_FLAG_TOPK.
 *   next_idx       [V, Hkv, max_topk] int32: the selected positions of KV
 *                  head g, ascending; entries past next_cnt are untouched.
 *   next_cnt       [V, Hkv] int32: number of selected positions.
 * For KV head g and position t in [0, L_v):
 *   score[t] = 1/((row_hi-row_lo)*G) * sum_{r in [row_lo,row_hi)}
 *              sum_{h in group g} exp(logit[h][r][t] - lse[h][r])
 * (masked logits contribute 0, and so does a row that saw no position,
 * whose LSE is -inf).  The K_v largest scores are kept, equal scores taken
 * lowest position first.  Scores are formed in fp32.
 */
PILLAR_API int pillar_topk_select(const pillar_shape_t *shape, int32_t V, const float *verify_logits,
                       const float *verify_lse, const int32_t *req_len, const int32_t *group_map,
                       const int32_t *K, int32_t *next_idx, int32_t *next_cnt, void *workspace,
                       size_t ws_bytes, void *stream);

/*
 * pillar_topk_select_noalloc -- pillar_topk_select without a workspace.
 * (The paper has no counterpart: this is a convenience of this library.)
 *
 * For callers that cannot allocate device memory themselves -- their HBM is
 * owned by another allocator (a framework's caching allocator, an inference
 * server that reserves the whole budget up front), or they sit on a
 * latency-critical path where cudaMalloc's implicit device synchronisation
 * is not acceptable.  It computes exactly what pillar_topk_select computes,
 * with the same kernels; its scratch (error word and fp32 score rows) is one
 * array of PILLAR_NOALLOC_SCRATCH_BYTES compiled into the library, which
 * every GPU that loads the library holds until the process exits.  Nothing
 * is allocated or freed by this call.
 *
 *   arguments 1-9   as for pillar_topk_select (inputs and outputs, caller-owned
 *                   device memory);
 *   device_flags    NULL or a device int32 that receives the call's device
 *                   error word (PILLAR_FLAG_* bits) when the call completes.
 *
 * Returns PILLAR_ERR_SCRATCH, with nothing enqueued, when the shape needs
 * more scratch than the array holds (pillar_topk_workspace_bytes(shape, V)
 * > PILLAR_NOALLOC_SCRATCH_BYTES, about V * Hkv * max_len > 4M scores);
 * otherwise as pillar_topk_select.
 *
 * The first call in a device's context looks up the array's device address
 * (once per device context, with that device current: a context created
 * anew, after cudaDeviceReset for instance, gets a lookup of its own); make
 * that first call before any stream capture.  Every call shares the one array: calls whose work overlaps on
 * the GPU (different streams, or different host threads on one device) race
 * on it and must be serialised by the caller.  Each call clears the error
 * word itself; the score rows are fully rewritten before they are read.
 */
PILLAR_API int pillar_topk_select_noalloc(const pillar_shape_t *shape, int32_t V, const float *verify_logits,
                                          const float *verify_lse, const int32_t *req_len,
                                          const int32_t *group_map, const int32_t *K, int32_t *next_idx,
                                          int32_t *next_cnt, int32_t *device_flags, void *stream);

/*
 * pillar_draft_lists -- the critical lists of a draft step that follows a
 * verify step ("SparseSpec-MLSys26", 核心方法 / PillarAttn: the Top-K of the
 * verify step is the critical set of the next k draft steps; the tokens
 * appended since the verify step are attended as well).
 *
 * For verify request v of the earlier step, b = group_map[v] is its row in
 * the draft step's batch and p = req_len[b] - verify_len[v] the tokens it has
 * appended since; for every KV head h the kernel writes
 *   sparse_idx[b, h, :] = next_idx[v, h, :next_cnt[v, h]],
 *                         then verify_len[v], ..., verify_len[v] + p - 1
 *   sparse_cnt[b, h]    = next_cnt[v, h] + p
 * (ascending: the Top-K positions all lie below verify_len[v]), and with
 * sparse_slot non-NULL, sparse_slot[b, h, i] = slot_table[off_b + that
 * position], off_b = sum over b' < b of max(req_len[b'], 0), for
 * pillar_attn_unified_slotted.  Rows of other requests are left untouched.
 *
 *   V              number of verify requests (host value).
 *   next_idx,
 *   next_cnt       [V, Hkv, max_topk], [V, Hkv] int32 as pillar_topk_select
 *                  wrote them (shape->max_topk is the row stride).
 *   group_map      [V] int32: batch index of request v in the draft step.
 *   verify_len     [V] int32: request v's length at its verify step.
 *   req_len        [B] int32: the draft step's lengths (shape->B requests).
 *   slot_table     the draft step's slot table (needed with sparse_slot).
 *   sparse_idx,
 *   sparse_cnt,
 *   sparse_slot    the draft step's lists: [B, Hkv, max_sparse] (stride
 *                  shape->max_sparse), [B, Hkv], [B, Hkv, max_sparse] or NULL.
 *   device_flags   NULL or a device int32 the kernel OR-s flags into:
 *                  PILLAR_FLAG_REQUEST for a group_map entry outside [0, B)
 *                  or a length that shrank since the verify step (no list is
 *                  written; sparse_cnt 0 for the latter), PILLAR_FLAG_COUNT
 *                  for a list longer than max_sparse (cut to max_sparse) or a
 *                  next_cnt outside [0, max_topk] (clamped), PILLAR_FLAG_INDEX
 *                  / PILLAR_FLAG_SLOT for a position or slot out of range
 *                  (slot -1 written).
 * All arrays are device memory, 4-byte aligned.  Asynchronous on `stream`;
 * allocates nothing.  Returns PILLAR_OK, PILLAR_ERR_ARG or PILLAR_ERR_CUDA.
 */
PILLAR_API int pillar_draft_lists(const pillar_shape_t *shape, int32_t V, const int32_t *next_idx,
                                  const int32_t *next_cnt, const int32_t *group_map, const int32_t *verify_len,
                                  const int32_t *req_len, const int32_t *slot_table, int32_t *sparse_idx,
                                  int32_t *sparse_cnt, int32_t *sparse_slot, int32_t *device_flags, void *stream);

/*
 * pillar_get_error -- synchronises `stream`, then copies the device error
 * word of a workspace (either entry point's) into *flags and clears it.
 * Returns PILLAR_OK if it was zero, PILLAR_ERR_DEVICE if not,
 * PILLAR_ERR_ARG / PILLAR_ERR_CUDA on failure.
 */
PILLAR_API int pillar_get_error(void *workspace, void *stream, int32_t *flags);

/* pillar_status_string -- a static English description of a return code. */
PILLAR_API const char *pillar_status_string(int status);

/*
 * pillar_kv_append -- writes n new tokens' K and V rows into their page-size-1
 * slots (the step before the unified pass: the token a draft step appends or
 * the k+1 tokens of a verify step go to whatever slots the caller's allocator
 * handed out; "SparseSpec-MLSys26", Unified batch scheduler + fused attention
 * kernel: page size 1):
 *   k_pool[slots[i], h, :] = k_new[i, h, :],  v_pool[slots[i], h, :] = v_new[i, h, :]
 * for i < n and h < Hkv.  Only shape->Hkv, D and num_slots are used.
 *   k_new, v_new   [n, Hkv, D] bf16, device memory, 16-byte aligned
 *   slots          [n] int32, device memory; distinct (for a repeated slot one
 *                  of the writes wins)
 *   k_pool, v_pool [num_slots, Hkv, D] bf16, device memory, 16-byte aligned
 *   device_flags   device int32 or null: PILLAR_FLAG_SLOT is or-ed into it
 *                  when a slot lies outside [0, num_slots); that token is
 *                  skipped and no other row is touched
 * Asynchronous on `stream`; allocates nothing.  Returns PILLAR_OK,
 * PILLAR_ERR_ARG (bad shape, n < 0, a null or misaligned pointer) or
 * PILLAR_ERR_CUDA.
 */
PILLAR_API int pillar_kv_append(const pillar_shape_t *shape, const uint16_t *k_new, const uint16_t *v_new,
                                const int32_t *slots, int32_t n, uint16_t *k_pool, uint16_t *v_pool,
                                int32_t *device_flags, void *stream);

/*
 * Phase buckets of the unified batch (host side; "SparseSpec-MLSys26",
 * Unified batch scheduler + fused attention kernel, load balancing).  Every
 * request runs a cycle of k+1 steps: k draft steps (phases 1..k), then one
 * verify step (phase 0).  A request in bucket c is in phase (c + t) mod (k+1)
 * at step t, so the requests of one bucket verify together.  A new request
 * joins the bucket with the fewest requests (ties to the lowest index), which
 * keeps the verify requests of a step near B/(k+1) and the step's query rows
 * near (2k+1)/(k+1)*B instead of alternating between B and (k+1)*B.
 *
 * The state is a plain caller-owned struct; nothing is allocated and no GPU
 * is touched.  Every function returns PILLAR_OK or PILLAR_ERR_ARG (a null
 * pointer, k outside [0, PILLAR_MAX_BUCKETS - 1], a bucket outside
 * [0, k], retiring from an empty bucket, n < 0) and changes nothing on error.
 */
#define PILLAR_MAX_BUCKETS 64
typedef struct pillar_buckets {
    int32_t nbuckets;                    /* k + 1 */
    int32_t count[PILLAR_MAX_BUCKETS];   /* requests in each bucket */
} pillar_buckets_t;

/* pillar_buckets_init -- k+1 empty buckets. */
PILLAR_API int pillar_buckets_init(pillar_buckets_t *pb, int32_t k);

/* pillar_buckets_admit -- places a new request: *bucket gets the least
 * loaded bucket (the lowest index among equals), whose count grows by one. */
PILLAR_API int pillar_buckets_admit(pillar_buckets_t *pb, int32_t *bucket);

/* pillar_buckets_retire -- a request of `bucket` has finished. */
PILLAR_API int pillar_buckets_retire(pillar_buckets_t *pb, int32_t bucket);

/*
 * pillar_buckets_step -- the inputs of step `step` for n requests whose
 * buckets are bucket[0..n): req_mode[i] = 1 (verify) when the request's phase
 * is 0, else 0 (draft), and phase[i] in [0, k] (either output may be null).
 * *q_rows (nullable) gets the step's query rows, k+1 per verify request and
 * one per draft request (the T_q of pillar_attn_unified).  All pointers are
 * host memory.
 */
PILLAR_API int pillar_buckets_step(const pillar_buckets_t *pb, const int32_t *bucket, int32_t n, int64_t step,
                                   int32_t *req_mode, int32_t *phase, int64_t *q_rows);

/*
 * Host offload of KV ("SparseSpec-MLSys26", 动态 KV 管理 / the dynamic KV
 * manager: when device memory runs short, requests' KV goes to host memory
 * chunk by chunk, asynchronously, first in first out; requests that were
 * offloaded are scheduled again, ahead of new ones, as soon as device memory
 * is free).  Two parts: the copies of slot blocks between the page-size-1
 * pools and packed rows in host memory (device kernels), and the FIFO of
 * offloaded chunks (plain host code, caller-owned state).
 */

/*
 * pillar_kv_offload -- packs n slot blocks of the pools into rows of host
 * memory:
 *   host_k[i, h, :] = k_pool[slots[i], h, :],  host_v[i, h, :] = v_pool[slots[i], h, :]
 * for i < n and h < Hkv.  Only shape->Hkv, D and num_slots are used.
 *   k_pool, v_pool [num_slots, Hkv, D] bf16, device memory, 16-byte aligned
 *   slots          [n] int32, device memory (the slots of a request's chunk of
 *                  positions, in position order)
 *   host_k, host_v [n, Hkv, D] bf16, 16-byte aligned, page-locked host memory
 *                  (cudaHostAlloc / cudaMallocHost / cudaHostRegister; the
 *                  kernel writes it through its device mapping, over
 *                  NVLink-C2C on a Grace-Blackwell node) or device memory
 *   device_flags   device int32 or null: PILLAR_FLAG_SLOT is or-ed into it
 *                  for a slot outside [0, num_slots); that row is not written
 * Asynchronous on `stream` (the host rows are complete once the stream has
 * reached the call); allocates nothing.  Returns PILLAR_OK, PILLAR_ERR_ARG
 * (bad shape, n < 0, a null or misaligned pointer, or a host buffer the
 * device cannot address: pageable host memory is refused) or PILLAR_ERR_CUDA.
 */
PILLAR_API int pillar_kv_offload(const pillar_shape_t *shape, const uint16_t *k_pool, const uint16_t *v_pool,
                                 const int32_t *slots, int32_t n, uint16_t *host_k, uint16_t *host_v,
                                 int32_t *device_flags, void *stream);

/*
 * pillar_kv_reload -- the way back: the packed rows go to (new) slots,
 *   k_pool[slots[i], h, :] = host_k[i, h, :],  v_pool[slots[i], h, :] = host_v[i, h, :]
 * with the buffers, alignment, flags and status codes of pillar_kv_offload
 * (host_k and host_v are read, the pools written).  It is pillar_kv_append
 * with its new rows in host memory.
 */
PILLAR_API int pillar_kv_reload(const pillar_shape_t *shape, const uint16_t *host_k, const uint16_t *host_v,
                                const int32_t *slots, int32_t n, uint16_t *k_pool, uint16_t *v_pool,
                                int32_t *device_flags, void *stream);

/*
 * The FIFO of offloaded chunks.  The state counts the device slots held by
 * resident requests against a capacity, and queues the chunks of offloaded
 * requests (a request's positions [0, len) in chunks of `chunk` positions,
 * the last one possibly shorter) in the order they were offloaded.  A
 * request comes back whole: pillar_offload_reload pops the chunks of the
 * oldest offloaded requests while they fit in the free capacity, so a request
 * offloaded earlier is always reloaded earlier, and a request never runs
 * with part of its KV on the host.  Which request to offload is the caller's
 * choice (the pages leave it open).  Every function returns PILLAR_OK or
 * PILLAR_ERR_ARG (a null pointer or out-of-range argument) and changes
 * nothing on error.  Nothing is allocated and no GPU is touched.
 */
#define PILLAR_OFFLOAD_QUEUE 1024
typedef struct pillar_offload_chunk {
    int32_t req;    /* the caller's request id */
    int32_t first;  /* first position of the chunk */
    int32_t n;      /* positions in the chunk (chunk, or fewer for the request's last) */
    int32_t last;   /* 1 on the request's last chunk */
} pillar_offload_chunk_t;
typedef struct pillar_offload_fifo {
    int64_t capacity;  /* device slots available to requests' KV */
    int64_t resident;  /* slots held by resident requests */
    int32_t chunk;     /* positions per chunk (>= 1) */
    int32_t head;      /* queue index of the oldest chunk */
    int32_t count;     /* chunks queued */
    int32_t pad;
    pillar_offload_chunk_t q[PILLAR_OFFLOAD_QUEUE];
} pillar_offload_fifo_t;

/* pillar_offload_init -- no request resident, nothing queued. */
PILLAR_API int pillar_offload_init(pillar_offload_fifo_t *f, int64_t capacity, int32_t chunk);

/*
 * pillar_offload_reserve -- asks for n more device slots (a new request's KV,
 * or the tokens a running request appends).  *granted = 1 and the slots are
 * counted as resident if they fit; *granted = 0 otherwise, and also, for a
 * new request (new_request != 0), while offloaded requests wait: they are
 * brought back first.
 */
PILLAR_API int pillar_offload_reserve(pillar_offload_fifo_t *f, int64_t n, int32_t new_request, int32_t *granted);

/* pillar_offload_release -- a resident request finished: its n slots are free. */
PILLAR_API int pillar_offload_release(pillar_offload_fifo_t *f, int64_t n);

/*
 * pillar_offload_evict -- request `req` with len resident positions goes to
 * the host: its chunks join the queue (*nchunks of them, nullable) and its
 * slots stop counting as resident.  The caller copies each chunk's slot blocks
 * with pillar_kv_offload before it hands those slots out again.  Refused
 * (PILLAR_ERR_ARG) when the queue has no room for the chunks or len exceeds
 * the resident count.
 */
PILLAR_API int pillar_offload_evict(pillar_offload_fifo_t *f, int32_t req, int32_t len, int32_t *nchunks);

/*
 * pillar_offload_reload -- the chunks to bring back now: those of the oldest
 * offloaded requests, whole requests only, while their positions fit in the
 * free capacity and their chunks in out[0, max_out).  They leave the queue and
 * count as resident; *nout gets the number of chunks written (0: nothing fits
 * yet).  The caller allocates slots for them and copies with pillar_kv_reload.
 */
PILLAR_API int pillar_offload_reload(pillar_offload_fifo_t *f, pillar_offload_chunk_t *out, int32_t max_out,
                                     int32_t *nout);

#ifdef __cplusplus
}
#endif

#endif /* PILLAR_H */
