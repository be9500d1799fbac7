// pillar_sched.cu -- host-side phase buckets of the unified batch
// ("SparseSpec-MLSys26", Unified batch scheduler + fused attention kernel,
// load balancing): requests are kept in k+1 buckets by the step of their
// cycle at which they verify; a new request joins the least loaded bucket.
// Plain host code: no allocation, no GPU.
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
