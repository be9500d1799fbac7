// pillar_lists.cu -- the critical lists of the draft steps that follow a
// verify step.
//
// "SparseSpec-MLSys26", 核心方法 / PillarAttn: the Top-K of the verify step's
// exact scores is the critical set of the next k draft steps; the tokens the
// request has appended since the verify step are attended as well.  For
// verify request v (batch index b = group_map[v], length L_v at its verify
// step, length req_len[b] now, so p = req_len[b] - L_v tokens appended) and KV
// head h, the draft step's list is
//     next_idx[v, h, :next_cnt[v, h]]  (ascending, all below L_v)
//     then L_v, L_v + 1, ..., L_v + p - 1
// which is ascending as a whole.  Optionally each listed position is also
// translated to its pool slot, slot_table[kv_off[b] + pos] with kv_off the
// CSR offsets of the current lengths, so that the draft step's gather does
// not have to chase the slot table.
//
// One CTA per (verify request, KV head): a list is short (about K + p
// entries), so the kernel is one coalesced pass per CTA; the request's CSR
// offset is a block reduction over the lengths before it.
#include "pillar_device.cuh"
#include "pillar_lists.h"

namespace pillar {

namespace {

constexpr int kListThreads = 256;

__global__ void __launch_bounds__(kListThreads) draft_lists_kernel(const ListsArgs a) {
    const int v = blockIdx.x, h = blockIdx.y;
    __shared__ long long s_red[kListThreads / 32];
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    // the loads that do not depend on one another go out together
    const int b = a.group_map[v];
    const int Lv = a.verify_len[v];
    int c = a.next_cnt[(long long)v * a.Hkv + h];
    const bool b_ok = b >= 0 && b < a.B;
    // CSR offset of request b under the current lengths (a negative length counts as 0, as in the
    // attention planner)
    long long part = 0;
    if (b_ok)
        for (int i = threadIdx.x; i < b; i += kListThreads) {
            const int l = a.req_len[i];
            part += l > 0 ? l : 0;
        }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = part;
    __syncthreads();
    if (!b_ok) {
        if (threadIdx.x == 0 && h == 0 && a.flags) atomicOr(a.flags, PILLAR_FLAG_REQUEST);
        return;
    }
    long long kv_off = 0;
#pragma unroll
    for (int i = 0; i < kListThreads / 32; ++i) kv_off += s_red[i];
    const int Lb = a.req_len[b];
    const int p = Lb - Lv;
    int32_t *cnt_row = a.sparse_cnt + (long long)b * a.Hkv;
    if (Lv < 0 || p < 0) {  // a length that went down since the verify step: no list
        if (threadIdx.x == 0) {
            cnt_row[h] = 0;
            if (a.flags) atomicOr(a.flags, PILLAR_FLAG_REQUEST);
        }
        return;
    }
    int bad = 0;
    {
        if (c < 0 || c > a.max_topk) bad |= PILLAR_FLAG_COUNT, c = c < 0 ? 0 : a.max_topk;
        long long n = (long long)c + p;
        if (n > a.max_sparse) bad |= PILLAR_FLAG_COUNT, n = a.max_sparse;
        const int32_t *src = a.next_idx + ((long long)v * a.Hkv + h) * a.max_topk;
        const long long row = ((long long)b * a.Hkv + h) * a.max_sparse;
        for (int i = threadIdx.x; i < n; i += kListThreads) {
            const int pos = i < c ? __ldg(src + i) : Lv + (i - c);
            a.sparse_idx[row + i] = pos;
            if (a.sparse_slot) {
                int slot = -1;
                if (pos >= 0 && pos < Lb) {
                    slot = __ldg(a.slot_table + kv_off + pos);
                    if (slot < 0 || (long long)slot >= a.num_slots) bad |= PILLAR_FLAG_SLOT, slot = -1;
                } else {
                    bad |= PILLAR_FLAG_INDEX;
                }
                a.sparse_slot[row + i] = slot;
            }
        }
        if (threadIdx.x == 0) cnt_row[h] = (int)n;
    }
    if (bad) atomicOr(&s_bad, bad);
    __syncthreads();
    if (threadIdx.x == 0 && s_bad && a.flags) atomicOr(a.flags, s_bad);
}

}  // namespace

cudaError_t launch_draft_lists(const ListsArgs &a, cudaStream_t st) {
    if (a.V == 0) return cudaSuccess;
    draft_lists_kernel<<<dim3(a.V, a.Hkv), kListThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace pillar
