// pillar_api.cu -- the C ABI declared in include/pillar.h: argument checks,
// workspace carving, launches.  Every check that can be made on the host is
// made here, before anything is enqueued; data-dependent checks are made on
// the device and reported through the workspace error word.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cuda.h>  // CUcontext, CUresult (driver entry points are resolved through the runtime)
#include <cuda_runtime.h>

#include "pillar_internal.h"
#include "pillar_kv.h"
#include "pillar_lists.h"

namespace pillar {

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

void *driver_entry(const char *name, int version) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return f;
}
}  // namespace

cudaError_t current_device_context(int *dev, unsigned long long *ctx_id) {
    static const CtxGetCurrentFn get_current = reinterpret_cast<CtxGetCurrentFn>(driver_entry("cuCtxGetCurrent", 4000));
    static const CtxGetIdFn get_id = reinterpret_cast<CtxGetIdFn>(driver_entry("cuCtxGetId", 12000));
    *ctx_id = 0;
    const cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    CUcontext c = nullptr;
    if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c) return cudaSuccess;
    unsigned long long id = 0;
    if (get_id(c, &id) == CUDA_SUCCESS) *ctx_id = id;
    return cudaSuccess;
}

}  // namespace pillar

namespace {

using namespace pillar;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_shape(const pillar_shape_t *s) {
    if (!s) return PILLAR_ERR_ARG;
    if (s->B < 0 || s->Hq <= 0 || s->Hkv <= 0 || s->Hq % s->Hkv != 0) return PILLAR_ERR_ARG;
    const int G = s->Hq / s->Hkv;
    if (G > kMaxG) return PILLAR_ERR_ARG;
    if (s->D != 64 && s->D != 128) return PILLAR_ERR_ARG;
    if (s->k < 0 || (long long)(s->k + 1) * G > kMaxRows) return PILLAR_ERR_ARG;
    if (s->max_sparse < 0 || s->max_len < 1 || s->num_slots < 1 || s->max_topk < 1) return PILLAR_ERR_ARG;
    // the pools are addressed as num_slots * Hkv rows with 32-bit row coordinates
    if (s->Hkv > 0 && s->num_slots > 0x7fffffffll / s->Hkv) return PILLAR_ERR_ARG;
    if (s->row_lo < 0 || s->row_hi > s->k + 1 || s->row_lo >= s->row_hi) return PILLAR_ERR_ARG;
    if (s->schedule < PILLAR_SCHEDULE_UNIFIED || s->schedule > PILLAR_SCHEDULE_NAIVE_JOINT) return PILLAR_ERR_ARG;
    if (s->wait_timeout_us < 0) return PILLAR_ERR_ARG;
    if (!(s->sm_scale >= 0.f) || std::isinf(s->sm_scale)) return PILLAR_ERR_ARG;
    for (int c : {s->verify_chunk, s->draft_chunk})
        if (c != 0 && (c < kTileKeys || c > kMaxChunk || c % kTileKeys != 0)) return PILLAR_ERR_ARG;
    if ((long long)s->B * s->Hkv > (1ll << 30) || (long long)s->max_len * s->Hq * (s->k + 1) > (1ll << 40))
        return PILLAR_ERR_ARG;
    // The attention workspace must be sizeable in 64 bits with room to spare: its largest
    // section holds, per work item, (k+1)*G partial rows of D fp32 values (+ LSE), and a
    // (request, KV head) has at most max(max_len / verify chunk, max_sparse / draft chunk) + 1
    // items.  Shapes whose bound passes 2^50 bytes are refused rather than wrapped.
    const long double vc = s->verify_chunk > 0 ? s->verify_chunk : kTileKeys;
    const long double dc = s->draft_chunk > 0 ? s->draft_chunk : kTileKeys;
    const long double per_unit = std::max((long double)s->max_len / vc, (long double)s->max_sparse / dc) + 2.0L;
    const long double rows = (long double)(s->k + 1) * G;
    const long double bound = (long double)s->B * s->Hkv * per_unit * (rows * (s->D + 1) * 4.0L + 64.0L) +
                              (long double)s->B * 64.0L + 65536.0L;
    if (bound > 1125899906842624.0L) return PILLAR_ERR_ARG;  // 2^50
    return PILLAR_OK;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

}  // namespace

extern "C" {

int pillar_attn_workspace_bytes(const pillar_shape_t *shape, size_t *bytes) {
    const int st = check_shape(shape);
    if (st != PILLAR_OK) return st;
    if (!bytes) return PILLAR_ERR_ARG;
    *bytes = attn_layout(*shape).total;
    return PILLAR_OK;
}

// The host checks of an attention run (everything but the planner's inputs).
static int attn_run_checks(const pillar_shape_t *shape, const uint16_t *q, const uint16_t *k_pool,
                           const uint16_t *v_pool, const int32_t *slot_table, const int32_t *sparse_idx,
                           const int32_t *sparse_slot, const uint16_t *out, const float *verify_logits,
                           const float *verify_lse, const void *workspace, size_t ws_bytes) {
    const int st = check_shape(shape);
    if (st != PILLAR_OK) return st;
    const pillar_shape_t &s = *shape;
    if (s.B == 0) return PILLAR_OK;
    if (!q || !k_pool || !v_pool || !slot_table || !out || !verify_logits || !verify_lse) return PILLAR_ERR_ARG;
    if (s.max_sparse > 0 && !sparse_idx) return PILLAR_ERR_ARG;
    // TMA and 16-byte copies need 16-byte aligned rows; the logit dump stores pairs (8 bytes);
    // everything else is read or written in 4-byte words
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 4) ||
        !aligned(verify_logits, 8) || !aligned(verify_lse, 4) || !aligned(slot_table, 4) ||
        (sparse_idx && !aligned(sparse_idx, 4)) || (sparse_slot && !aligned(sparse_slot, 4)))
        return PILLAR_ERR_ARG;
    if (sparse_slot && !sparse_idx) return PILLAR_ERR_ARG;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < attn_layout(s).total) return PILLAR_ERR_WORKSPACE;
    return PILLAR_OK;
}

int pillar_attn_unified(const pillar_shape_t *shape, const uint16_t *q, const uint16_t *k_pool,
                        const uint16_t *v_pool, const int32_t *slot_table, const int32_t *req_mode,
                        const int32_t *req_len, const int32_t *sparse_idx, const int32_t *sparse_cnt,
                        uint16_t *out, float *verify_logits, float *verify_lse, void *workspace,
                        size_t ws_bytes, void *stream) {
    return pillar_attn_unified_slotted(shape, q, k_pool, v_pool, slot_table, req_mode, req_len, sparse_idx,
                                       sparse_cnt, nullptr, out, verify_logits, verify_lse, workspace, ws_bytes,
                                       stream);
}

int pillar_attn_unified_slotted(const pillar_shape_t *shape, const uint16_t *q, const uint16_t *k_pool,
                                const uint16_t *v_pool, const int32_t *slot_table, const int32_t *req_mode,
                                const int32_t *req_len, const int32_t *sparse_idx, const int32_t *sparse_cnt,
                                const int32_t *sparse_slot, uint16_t *out, float *verify_logits,
                                float *verify_lse, void *workspace, size_t ws_bytes, void *stream) {
    // the run's checks first, so that a bad call enqueues nothing
    const int st = attn_run_checks(shape, q, k_pool, v_pool, slot_table, sparse_idx, sparse_slot, out, verify_logits,
                                   verify_lse, workspace, ws_bytes);
    if (st != PILLAR_OK) return st;
    const int sp = pillar_attn_plan(shape, req_mode, req_len, sparse_cnt, workspace, ws_bytes, stream);
    if (sp != PILLAR_OK) return sp;
    return pillar_attn_run(shape, q, k_pool, v_pool, slot_table, sparse_idx, sparse_slot, out, verify_logits,
                           verify_lse, workspace, ws_bytes, stream);
}

int pillar_attn_plan(const pillar_shape_t *shape, const int32_t *req_mode, const int32_t *req_len,
                     const int32_t *sparse_cnt, void *workspace, size_t ws_bytes, void *stream) {
    int st = check_shape(shape);
    if (st != PILLAR_OK) return st;
    const pillar_shape_t &s = *shape;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (s.B == 0) {
        // nothing to plan; a workspace passed in still reads back as clean
        if (workspace && ws_bytes >= sizeof(WsHeader) && cudaMemsetAsync(workspace, 0, sizeof(int), cs) != cudaSuccess)
            return PILLAR_ERR_CUDA;
        return PILLAR_OK;
    }
    if (!req_mode || !req_len || !sparse_cnt) return PILLAR_ERR_ARG;
    if (!aligned(req_mode, 4) || !aligned(req_len, 4) || !aligned(sparse_cnt, 4)) return PILLAR_ERR_ARG;
    const AttnLayout lay = attn_layout(s);
    if (!workspace || !aligned(workspace, 256) || ws_bytes < lay.total) return PILLAR_ERR_WORKSPACE;
    PlanArgs pa;
    pa.req_mode = req_mode;
    pa.req_len = req_len;
    pa.sparse_cnt = sparse_cnt;
    pa.ws = static_cast<char *>(workspace);
    pa.lay = lay;
    pa.B = s.B;
    pa.Hq = s.Hq;
    pa.Hkv = s.Hkv;
    pa.k = s.k;
    pa.max_sparse = s.max_sparse;
    pa.max_len = s.max_len;
    const bool naive = s.schedule == PILLAR_SCHEDULE_NAIVE_JOINT;  // the largest items the pipeline takes
    pa.vchunk = naive ? kMaxChunk : verify_chunk_of(s);
    pa.dchunk = naive ? kMaxChunk : draft_chunk_of(s);
    pa.schedule = s.schedule;
    return launch_plan(pa, cs) == cudaSuccess ? PILLAR_OK : PILLAR_ERR_CUDA;
}

int pillar_attn_run(const pillar_shape_t *shape, const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                    const int32_t *slot_table, const int32_t *sparse_idx, const int32_t *sparse_slot, uint16_t *out,
                    float *verify_logits, float *verify_lse, void *workspace, size_t ws_bytes, void *stream) {
    const int st = attn_run_checks(shape, q, k_pool, v_pool, slot_table, sparse_idx, sparse_slot, out, verify_logits,
                                   verify_lse, workspace, ws_bytes);
    if (st != PILLAR_OK) return st;
    const pillar_shape_t &s = *shape;
    if (s.B == 0) return PILLAR_OK;
    const int nsm = sm_count();
    if (nsm <= 0) return PILLAR_ERR_CUDA;
    AttnArgs aa;
    aa.q = q;
    aa.k_pool = k_pool;
    aa.v_pool = v_pool;
    aa.slot_table = slot_table;
    aa.sparse_idx = sparse_idx;
    aa.sparse_slot = sparse_slot;
    aa.out = out;
    aa.logits = verify_logits;
    aa.lse = verify_lse;
    aa.ws = static_cast<char *>(workspace);
    aa.lay = attn_layout(s);
    aa.num_slots = s.num_slots;
    aa.Hq = s.Hq;
    aa.Hkv = s.Hkv;
    aa.D = s.D;
    aa.k = s.k;
    aa.max_sparse = s.max_sparse;
    aa.schedule = s.schedule;
    aa.scale = s.sm_scale > 0.f ? s.sm_scale : 1.0f / std::sqrt((float)s.D);
    aa.wait_ns = s.wait_timeout_us > 0 ? (unsigned long long)s.wait_timeout_us * 1000ull : kWaitTimeoutNs;
    return launch_attn(aa, nsm, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PILLAR_OK : PILLAR_ERR_CUDA;
}

int pillar_topk_workspace_bytes(const pillar_shape_t *shape, int32_t V, size_t *bytes) {
    const int st = check_shape(shape);
    if (st != PILLAR_OK) return st;
    if (!bytes || V < 0) return PILLAR_ERR_ARG;
    if ((long double)V * shape->Hkv * shape->max_len * 4.0L > 1125899906842624.0L) return PILLAR_ERR_ARG;  // 2^50
    *bytes = topk_ws_bytes(*shape, V);
    return PILLAR_OK;
}

int pillar_topk_select(const pillar_shape_t *shape, int32_t V, const float *verify_logits,
                       const float *verify_lse, const int32_t *req_len, const int32_t *group_map,
                       const int32_t *K, int32_t *next_idx, int32_t *next_cnt, void *workspace,
                       size_t ws_bytes, void *stream) {
    int st = check_shape(shape);
    if (st != PILLAR_OK) return st;
    if (V < 0) return PILLAR_ERR_ARG;
    if (V == 0) {
        if (workspace && ws_bytes >= sizeof(WsHeader) &&
            cudaMemsetAsync(workspace, 0, sizeof(int), static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return PILLAR_ERR_CUDA;
        return PILLAR_OK;
    }
    if (!verify_logits || !verify_lse || !req_len || !group_map || !K || !next_idx || !next_cnt)
        return PILLAR_ERR_ARG;
    if (!aligned(verify_logits, 4) || !aligned(verify_lse, 4) || !aligned(req_len, 4) || !aligned(group_map, 4) ||
        !aligned(K, 4) || !aligned(next_idx, 4) || !aligned(next_cnt, 4))
        return PILLAR_ERR_ARG;  // every array is read or written in 4-byte words
    if (!workspace || !aligned(workspace, 256) || ws_bytes < topk_ws_bytes(*shape, V)) return PILLAR_ERR_WORKSPACE;
    if ((long long)V * shape->Hkv > 65535ll * 65535ll || V > 65535) return PILLAR_ERR_ARG;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    TopkArgs ta;
    ta.logits = verify_logits;
    ta.lse = verify_lse;
    ta.req_len = req_len;
    ta.group_map = group_map;
    ta.K = K;
    ta.next_idx = next_idx;
    ta.next_cnt = next_cnt;
    ta.ws = static_cast<char *>(workspace);
    ta.rows = reinterpret_cast<TopkRow *>(ta.ws + topk_rows_offset());
    ta.scores = reinterpret_cast<float *>(ta.ws + topk_scores_offset(V));
    ta.B = shape->B;
    ta.V = V;
    ta.Hq = shape->Hq;
    ta.Hkv = shape->Hkv;
    ta.k = shape->k;
    ta.row_lo = shape->row_lo;
    ta.row_hi = shape->row_hi;
    ta.max_topk = shape->max_topk;
    ta.max_len = shape->max_len;
    // (the score kernel clears the error word itself: no memset between the attention and the Top-K)
    if (launch_topk_select(ta, cs) != cudaSuccess) return PILLAR_ERR_CUDA;
    return PILLAR_OK;
}

int pillar_kv_append(const pillar_shape_t *shape, const uint16_t *k_new, const uint16_t *v_new,
                     const int32_t *slots, int32_t n, uint16_t *k_pool, uint16_t *v_pool, int32_t *device_flags,
                     void *stream) {
    const int st = check_shape(shape);
    if (st != PILLAR_OK) return st;
    if (n < 0) return PILLAR_ERR_ARG;
    if (n == 0) return PILLAR_OK;
    if (!k_new || !v_new || !slots || !k_pool || !v_pool) return PILLAR_ERR_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(slots, 4) || (device_flags && !aligned(device_flags, 4)))
        return PILLAR_ERR_ARG;
    const int nsm = sm_count();
    if (nsm <= 0) return PILLAR_ERR_CUDA;
    KvAppendArgs a;
    a.k_new = k_new;
    a.v_new = v_new;
    a.slots = slots;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.flags = device_flags;
    a.num_slots = shape->num_slots;
    a.n = n;
    a.Hkv = shape->Hkv;
    a.D = shape->D;
    return launch_kv_append(a, nsm, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PILLAR_OK : PILLAR_ERR_CUDA;
}

// The device address of a buffer the offload copies read or write: device
// memory as it is, page-locked host memory through its mapping; anything else
// (pageable host memory) is refused rather than handed to a kernel.
static void *device_address(void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();  // (the failed query leaves an error that the next check would see)
        return nullptr;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return p;
    if (at.type == cudaMemoryTypeHost) return at.devicePointer;
    return nullptr;
}

static int kv_copy_checks(const pillar_shape_t *shape, int32_t n, const void *a, const void *b, const void *c,
                          const void *d, const int32_t *slots, const int32_t *device_flags) {
    const int st = check_shape(shape);
    if (st != PILLAR_OK) return st;
    if (n < 0) return PILLAR_ERR_ARG;
    if (n == 0) return PILLAR_OK;
    if (!a || !b || !c || !d || !slots) return PILLAR_ERR_ARG;
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(c, 16) || !aligned(d, 16) || !aligned(slots, 4) ||
        (device_flags && !aligned(device_flags, 4)))
        return PILLAR_ERR_ARG;
    return PILLAR_OK;
}

int pillar_kv_offload(const pillar_shape_t *shape, const uint16_t *k_pool, const uint16_t *v_pool,
                      const int32_t *slots, int32_t n, uint16_t *host_k, uint16_t *host_v, int32_t *device_flags,
                      void *stream) {
    const int st = kv_copy_checks(shape, n, k_pool, v_pool, host_k, host_v, slots, device_flags);
    if (st != PILLAR_OK || n == 0) return st;
    void *ko = device_address(host_k), *vo = device_address(host_v);
    if (!ko || !vo) return PILLAR_ERR_ARG;
    const int nsm = sm_count();
    if (nsm <= 0) return PILLAR_ERR_CUDA;
    KvOffloadArgs a;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.slots = slots;
    a.k_out = static_cast<uint16_t *>(ko);
    a.v_out = static_cast<uint16_t *>(vo);
    a.flags = device_flags;
    a.num_slots = shape->num_slots;
    a.n = n;
    a.Hkv = shape->Hkv;
    a.D = shape->D;
    return launch_kv_offload(a, nsm, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PILLAR_OK : PILLAR_ERR_CUDA;
}

int pillar_kv_reload(const pillar_shape_t *shape, const uint16_t *host_k, const uint16_t *host_v,
                     const int32_t *slots, int32_t n, uint16_t *k_pool, uint16_t *v_pool, int32_t *device_flags,
                     void *stream) {
    const int st = kv_copy_checks(shape, n, host_k, host_v, k_pool, v_pool, slots, device_flags);
    if (st != PILLAR_OK || n == 0) return st;
    void *ki = device_address(const_cast<uint16_t *>(host_k)), *vi = device_address(const_cast<uint16_t *>(host_v));
    if (!ki || !vi) return PILLAR_ERR_ARG;
    // the reload is the append's scatter, its packed rows read through their device address
    return pillar_kv_append(shape, static_cast<const uint16_t *>(ki), static_cast<const uint16_t *>(vi), slots, n,
                            k_pool, v_pool, device_flags, stream);
}

int pillar_draft_lists(const pillar_shape_t *shape, int32_t V, const int32_t *next_idx, const int32_t *next_cnt,
                       const int32_t *group_map, const int32_t *verify_len, const int32_t *req_len,
                       const int32_t *slot_table, int32_t *sparse_idx, int32_t *sparse_cnt, int32_t *sparse_slot,
                       int32_t *device_flags, void *stream) {
    const int st = check_shape(shape);
    if (st != PILLAR_OK) return st;
    if (V < 0 || V > 65535 * 32) return PILLAR_ERR_ARG;
    if (V == 0) return PILLAR_OK;
    if (!next_idx || !next_cnt || !group_map || !verify_len || !req_len || !sparse_idx || !sparse_cnt)
        return PILLAR_ERR_ARG;
    if (shape->max_sparse < 1 || (sparse_slot && !slot_table)) return PILLAR_ERR_ARG;
    for (const void *ptr : {(const void *)next_idx, (const void *)next_cnt, (const void *)group_map,
                            (const void *)verify_len, (const void *)req_len, (const void *)slot_table,
                            (const void *)sparse_idx, (const void *)sparse_cnt, (const void *)sparse_slot,
                            (const void *)device_flags})
        if (!aligned(ptr, 4)) return PILLAR_ERR_ARG;  // 4-byte words throughout
    ListsArgs a;
    a.next_idx = next_idx;
    a.next_cnt = next_cnt;
    a.group_map = group_map;
    a.verify_len = verify_len;
    a.req_len = req_len;
    a.slot_table = slot_table;
    a.sparse_idx = sparse_idx;
    a.sparse_cnt = sparse_cnt;
    a.sparse_slot = sparse_slot;
    a.flags = device_flags;
    a.num_slots = shape->num_slots;
    a.V = V;
    a.B = shape->B;
    a.Hkv = shape->Hkv;
    a.max_topk = shape->max_topk;
    a.max_sparse = shape->max_sparse;
    return launch_draft_lists(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PILLAR_OK : PILLAR_ERR_CUDA;
}

int pillar_get_error(void *workspace, void *stream, int32_t *flags) {
    if (!workspace || !flags) return PILLAR_ERR_ARG;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return PILLAR_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), cs) != cudaSuccess) return PILLAR_ERR_CUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return PILLAR_ERR_CUDA;
    *flags = v;
    return v ? PILLAR_ERR_DEVICE : PILLAR_OK;
}

const char *pillar_status_string(int status) {
    switch (status) {
        case PILLAR_OK: return "ok";
        case PILLAR_ERR_ARG: return "bad argument (null pointer, dimension or unsupported shape)";
        case PILLAR_ERR_WORKSPACE: return "workspace null, misaligned or too small";
        case PILLAR_ERR_CUDA: return "CUDA runtime or launch error";
        case PILLAR_ERR_DEVICE: return "device reported an out-of-range index, slot, length or a timeout";
        case PILLAR_ERR_SCRATCH: return "shape exceeds the built-in scratch of pillar_topk_select_noalloc";
        default: return "unknown status";
    }
}

}  // extern "C"
