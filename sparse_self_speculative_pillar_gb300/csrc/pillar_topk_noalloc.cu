// pillar_topk_noalloc.cu -- pillar_topk_select for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand this library a workspace: their device
// memory is owned by another allocator (a framework's caching allocator or
// an inference server that reserves the whole HBM budget up front and must
// not see foreign cudaMalloc calls), or they run on a latency-critical path
// where cudaMalloc's implicit device synchronisation is not acceptable.
// This entry point runs the same Top-K kernels as pillar_topk_select, but
// its scratch (the error word and the fp32 score rows) lives in one
// fixed-size array compiled into the library, so the caller passes only
// inputs and outputs.  Every GPU that loads the library holds the array
// until the process exits.
#include <cstdint>
#include <initializer_list>
#include <cuda_runtime.h>
#include <mutex>

#include "pillar_internal.h"

namespace {

using namespace pillar;

// The built-in scratch: the Top-K workspace layout (header with the error
// word, per-request records, then the packed scores [V][Hkv][max_len]) capped at
// PILLAR_NOALLOC_SCRATCH_BYTES.  In host code this name is only a stand-in
// for the device copy; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_topk_scratch[PILLAR_NOALLOC_SCRATCH_BYTES];

std::mutex g_setup_mutex;
struct ScratchAddr {
    unsigned long long ctx;  // unique id of the context the address belongs to (0: none yet)
    void *ptr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

// The device address of the scratch array in the context current on the
// current device, looked up once per device context (so a context created
// anew after cudaDeviceReset gets its own lookup).  Returns nullptr if the
// runtime cannot provide it.
void *scratch_for_current_device() {
    int dev = 0;
    unsigned long long ctx = 0;
    if (current_device_context(&dev, &ctx) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    ScratchAddr &a = g_scratch_addr[dev];
    if (ctx == 0 || a.ctx != ctx || !a.ptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess) return nullptr;
        if (current_device_context(&dev, &ctx) != cudaSuccess) return nullptr;  // the lookup made a context current
        a.ctx = ctx;
        a.ptr = p;
    }
    return a.ptr;
}

}  // namespace

extern "C" {

int pillar_topk_select_noalloc(const pillar_shape_t *shape, int32_t V, const float *verify_logits,
                               const float *verify_lse, const int32_t *req_len, const int32_t *group_map,
                               const int32_t *K, int32_t *next_idx, int32_t *next_cnt, int32_t *device_flags,
                               void *stream) {
    if (!shape || V < 0) return PILLAR_ERR_ARG;
    size_t need = 0;
    const int st = pillar_topk_workspace_bytes(shape, V, &need);
    if (st != PILLAR_OK) return st;
    if (need > (size_t)PILLAR_NOALLOC_SCRATCH_BYTES) return PILLAR_ERR_SCRATCH;
    if (V > 0 && (!verify_logits || !verify_lse || !req_len || !group_map || !K || !next_idx || !next_cnt))
        return PILLAR_ERR_ARG;
    for (const void *ptr : {(const void *)verify_logits, (const void *)verify_lse, (const void *)req_len,
                            (const void *)group_map, (const void *)K, (const void *)next_idx,
                            (const void *)next_cnt, (const void *)device_flags})
        if (reinterpret_cast<uintptr_t>(ptr) & 3u) return PILLAR_ERR_ARG;  // 4-byte words throughout
    if ((long long)V * shape->Hkv > 65535ll * 65535ll || V > 65535) return PILLAR_ERR_ARG;
    char *ws = static_cast<char *>(scratch_for_current_device());
    if (!ws) return PILLAR_ERR_CUDA;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: the error word must start at zero (the score
    // kernel clears it when there is a verify request)
    if (V == 0 && cudaMemsetAsync(ws, 0, sizeof(int), cs) != cudaSuccess) return PILLAR_ERR_CUDA;
    if (V > 0) {
        TopkArgs ta;
        ta.logits = verify_logits;
        ta.lse = verify_lse;
        ta.req_len = req_len;
        ta.group_map = group_map;
        ta.K = K;
        ta.next_idx = next_idx;
        ta.next_cnt = next_cnt;
        ta.ws = ws;
        ta.rows = reinterpret_cast<TopkRow *>(ws + topk_rows_offset());
        ta.scores = reinterpret_cast<float *>(ws + topk_scores_offset(V));
        ta.B = shape->B;
        ta.V = V;
        ta.Hq = shape->Hq;
        ta.Hkv = shape->Hkv;
        ta.k = shape->k;
        ta.row_lo = shape->row_lo;
        ta.row_hi = shape->row_hi;
        ta.max_topk = shape->max_topk;
        ta.max_len = shape->max_len;
        if (launch_topk_select(ta, cs) != cudaSuccess) return PILLAR_ERR_CUDA;
    }
    if (device_flags &&
        cudaMemcpyAsync(device_flags, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
        return PILLAR_ERR_CUDA;
    return PILLAR_OK;
}

}  // extern "C"
