// pillar_sched.cu -- host-side phase buckets of the unified batch, and the
// FIFO of host-offloaded KV chunks (at the end of the file).
//
// The buckets ("SparseSpec-MLSys26", Unified batch scheduler + fused attention
// kernel, load balancing): requests are kept in k+1 buckets by the step of
// their cycle at which they verify; a new request joins the least loaded
// bucket.  Plain host code: no allocation, no GPU.
#include <cstdint>

#include "../../include/pillar.h"

namespace {

bool valid(const pillar_buckets_t *pb) {
    return pb && pb->nbuckets >= 1 && pb->nbuckets <= PILLAR_MAX_BUCKETS;
}

}  // namespace

extern "C" {

int pillar_buckets_init(pillar_buckets_t *pb, int32_t k) {
    if (!pb || k < 0 || k + 1 > PILLAR_MAX_BUCKETS) return PILLAR_ERR_ARG;
    pb->nbuckets = k + 1;
    for (int i = 0; i < PILLAR_MAX_BUCKETS; ++i) pb->count[i] = 0;
    return PILLAR_OK;
}

int pillar_buckets_admit(pillar_buckets_t *pb, int32_t *bucket) {
    if (!valid(pb) || !bucket) return PILLAR_ERR_ARG;
    int best = 0;
    for (int c = 1; c < pb->nbuckets; ++c)
        if (pb->count[c] < pb->count[best]) best = c;  // strict: ties keep the lower index
    if (pb->count[best] == INT32_MAX) return PILLAR_ERR_ARG;
    ++pb->count[best];
    *bucket = best;
    return PILLAR_OK;
}

int pillar_buckets_retire(pillar_buckets_t *pb, int32_t bucket) {
    if (!valid(pb) || bucket < 0 || bucket >= pb->nbuckets || pb->count[bucket] <= 0) return PILLAR_ERR_ARG;
    --pb->count[bucket];
    return PILLAR_OK;
}

int pillar_buckets_step(const pillar_buckets_t *pb, const int32_t *bucket, int32_t n, int64_t step,
                        int32_t *req_mode, int32_t *phase, int64_t *q_rows) {
    if (!valid(pb) || n < 0 || (n > 0 && !bucket)) return PILLAR_ERR_ARG;
    const int64_t nb = pb->nbuckets;
    for (int32_t i = 0; i < n; ++i)
        if (bucket[i] < 0 || bucket[i] >= nb) return PILLAR_ERR_ARG;
    const int64_t t = ((step % nb) + nb) % nb;  // the step's place in the cycle (any sign of step)
    int64_t rows = 0;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t ph = (int32_t)((bucket[i] + t) % nb);
        if (phase) phase[i] = ph;
        if (req_mode) req_mode[i] = ph == 0 ? 1 : 0;
        rows += ph == 0 ? nb : 1;
    }
    if (q_rows) *q_rows = rows;
    return PILLAR_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- host offload FIFO
//
// The dynamic KV manager's queue ("SparseSpec-MLSys26", 动态 KV 管理): the
// chunks of offloaded requests wait in the order they were offloaded and come
// back whole requests at a time, oldest first.

namespace {

bool valid(const pillar_offload_fifo_t *f) {
    return f && f->chunk >= 1 && f->capacity >= 0 && f->resident >= 0 && f->resident <= f->capacity &&
           f->head >= 0 && f->head < PILLAR_OFFLOAD_QUEUE && f->count >= 0 && f->count <= PILLAR_OFFLOAD_QUEUE;
}

const pillar_offload_chunk_t &at(const pillar_offload_fifo_t *f, int32_t i) {
    return f->q[(f->head + i) % PILLAR_OFFLOAD_QUEUE];
}

}  // namespace

extern "C" {

int pillar_offload_init(pillar_offload_fifo_t *f, int64_t capacity, int32_t chunk) {
    if (!f || capacity < 0 || chunk < 1) return PILLAR_ERR_ARG;
    f->capacity = capacity;
    f->resident = 0;
    f->chunk = chunk;
    f->head = 0;
    f->count = 0;
    f->pad = 0;
    return PILLAR_OK;
}

int pillar_offload_reserve(pillar_offload_fifo_t *f, int64_t n, int32_t new_request, int32_t *granted) {
    if (!valid(f) || n < 0 || !granted) return PILLAR_ERR_ARG;
    const bool fits = n <= f->capacity - f->resident;
    const bool ok = fits && !(new_request && f->count > 0);  // offloaded requests come back before new ones
    if (ok) f->resident += n;
    *granted = ok ? 1 : 0;
    return PILLAR_OK;
}

int pillar_offload_release(pillar_offload_fifo_t *f, int64_t n) {
    if (!valid(f) || n < 0 || n > f->resident) return PILLAR_ERR_ARG;
    f->resident -= n;
    return PILLAR_OK;
}

int pillar_offload_evict(pillar_offload_fifo_t *f, int32_t req, int32_t len, int32_t *nchunks) {
    if (!valid(f) || len < 1 || len > f->resident) return PILLAR_ERR_ARG;
    const int32_t nc = (int32_t)((len + (int64_t)f->chunk - 1) / f->chunk);
    if (nc > PILLAR_OFFLOAD_QUEUE - f->count) return PILLAR_ERR_ARG;
    for (int32_t c = 0; c < nc; ++c) {
        pillar_offload_chunk_t &e = f->q[(f->head + f->count + c) % PILLAR_OFFLOAD_QUEUE];
        e.req = req;
        e.first = c * f->chunk;
        e.n = c + 1 < nc ? f->chunk : len - c * f->chunk;
        e.last = c + 1 == nc;
    }
    f->count += nc;
    f->resident -= len;
    if (nchunks) *nchunks = nc;
    return PILLAR_OK;
}

int pillar_offload_reload(pillar_offload_fifo_t *f, pillar_offload_chunk_t *out, int32_t max_out, int32_t *nout) {
    if (!valid(f) || max_out < 0 || (max_out > 0 && !out) || !nout) return PILLAR_ERR_ARG;
    int32_t taken = 0;
    int64_t free_slots = f->capacity - f->resident;
    while (taken < f->count) {
        // the next request: its chunks up to its last one
        int32_t end = taken;
        int64_t len = 0;
        while (end < f->count) {
            const pillar_offload_chunk_t &e = at(f, end++);
            len += e.n;
            if (e.last) break;
        }
        if (len > free_slots || end > max_out) break;
        for (int32_t i = taken; i < end; ++i) out[i] = at(f, i);
        free_slots -= len;
        taken = end;
    }
    f->head = (f->head + taken) % PILLAR_OFFLOAD_QUEUE;
    f->count -= taken;
    f->resident = f->capacity - free_slots;
    *nout = taken;
    return PILLAR_OK;
}

}  // extern "C"
