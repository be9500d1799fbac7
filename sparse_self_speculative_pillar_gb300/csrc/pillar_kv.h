// pillar_kv.h -- host-side launches of the slot-block copies (pillar_kv.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pillar {

struct KvAppendArgs {
    const uint16_t *k_new, *v_new;
    const int *slots;
    uint16_t *k_pool, *v_pool;
    int *flags;  // device error word, or null
    long long num_slots;
    int n, Hkv, D;
};
cudaError_t launch_kv_append(const KvAppendArgs &a, int nsm, cudaStream_t st);
struct KvOffloadArgs {
    const uint16_t *k_pool, *v_pool;
    const int *slots;
    uint16_t *k_out, *v_out;  // packed rows [n, Hkv, D]: device addresses (of host memory, for an offload)
    int *flags;               // device error word, or null
    long long num_slots;
    int n, Hkv, D;
};
cudaError_t launch_kv_offload(const KvOffloadArgs &a, int nsm, cudaStream_t st);

}  // namespace pillar
