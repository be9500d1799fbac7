// pillar_lists.h -- launch declaration of the next-draft-list kernel
// (pillar_lists.cu), called by the C ABI in pillar_api.cu.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pillar {

struct ListsArgs {
    const int32_t *next_idx, *next_cnt, *group_map, *verify_len, *req_len, *slot_table;
    int32_t *sparse_idx, *sparse_cnt, *sparse_slot, *flags;
    long long num_slots;
    int V, B, Hkv, max_topk, max_sparse;
};

cudaError_t launch_draft_lists(const ListsArgs &a, cudaStream_t st);

}  // namespace pillar
