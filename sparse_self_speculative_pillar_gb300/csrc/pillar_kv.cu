// pillar_kv.cu -- moving whole slot blocks of the page-size-1 pools.
//
// With page size 1 ("SparseSpec-MLSys26", Unified batch scheduler + fused
// attention kernel) every token owns one slot of the pools [num_slots, Hkv,
// D]: token i's Hkv*D bf16 values of K (and of V) are one contiguous block.
//   * append: a scatter of packed rows into their slots (the new tokens of a
//     step); the reload of offloaded KV is the same scatter, its packed rows
//     read from host memory;
//   * offload: the gather of slots into packed rows in host memory (the
//     dynamic KV manager's chunk-wise offload, "SparseSpec-MLSys26", 动态 KV
//     管理: on device-memory pressure a request's KV goes to the host in
//     chunks, and comes back before the request is scheduled again).  The
//     host rows are written by the kernel itself, through their device
//     address (NVLink-C2C on a Grace-Blackwell node).
// Flat grid-stride copies in 16-byte pieces: reads and writes are coalesced
// within a slot's block (2 KB at Hkv = 8, D = 128).
#include <cstdint>
#include <cuda_runtime.h>

#include "pillar_internal.h"
#include "pillar_kv.h"

namespace pillar {

__global__ void kv_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                 const int *__restrict__ slots, int n, int row_chunks, long long num_slots,
                                 uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool, int *flags) {
    const long long total = (long long)n * row_chunks;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / row_chunks);
        const int c = (int)(i - (long long)t * row_chunks);
        const int s = __ldg(slots + t);
        if (s < 0 || (long long)s >= num_slots) {
            if (c == 0 && flags) atomicOr(flags, PILLAR_FLAG_SLOT);
            continue;
        }
        const size_t dst = (size_t)s * (size_t)row_chunks + (size_t)c;
        const uint4 kv = __ldg(k_new + i), vv = __ldg(v_new + i);
        k_pool[dst] = kv;
        v_pool[dst] = vv;
    }
}

__global__ void kv_offload_kernel(const uint4 *__restrict__ k_pool, const uint4 *__restrict__ v_pool,
                                  const int *__restrict__ slots, int n, int row_chunks, long long num_slots,
                                  uint4 *__restrict__ k_out, uint4 *__restrict__ v_out, int *flags) {
    const long long total = (long long)n * row_chunks;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / row_chunks);
        const int c = (int)(i - (long long)t * row_chunks);
        const int s = __ldg(slots + t);
        if (s < 0 || (long long)s >= num_slots) {  // nothing is read; the packed row is left as it was
            if (c == 0 && flags) atomicOr(flags, PILLAR_FLAG_SLOT);
            continue;
        }
        const size_t src = (size_t)s * (size_t)row_chunks + (size_t)c;
        const uint4 kv = __ldg(k_pool + src), vv = __ldg(v_pool + src);
        k_out[i] = kv;
        v_out[i] = vv;
    }
}

cudaError_t launch_kv_offload(const KvOffloadArgs &a, int nsm, cudaStream_t st) {
    if (a.n == 0) return cudaSuccess;
    const int row_chunks = a.Hkv * a.D * 2 / 16;
    const long long total = (long long)a.n * row_chunks;
    constexpr int kThreadsPerCta = 256;
    long long blocks = (total + kThreadsPerCta - 1) / kThreadsPerCta;
    const long long cap = (long long)nsm * 8;
    if (blocks > cap) blocks = cap;
    kv_offload_kernel<<<(unsigned)blocks, kThreadsPerCta, 0, st>>>(
        reinterpret_cast<const uint4 *>(a.k_pool), reinterpret_cast<const uint4 *>(a.v_pool), a.slots, a.n,
        row_chunks, a.num_slots, reinterpret_cast<uint4 *>(a.k_out), reinterpret_cast<uint4 *>(a.v_out), a.flags);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(const KvAppendArgs &a, int nsm, cudaStream_t st) {
    if (a.n == 0) return cudaSuccess;
    const int row_chunks = a.Hkv * a.D * 2 / 16;  // 16-byte pieces of one slot's block
    const long long total = (long long)a.n * row_chunks;
    constexpr int kThreadsPerCta = 256;
    long long blocks = (total + kThreadsPerCta - 1) / kThreadsPerCta;
    const long long cap = (long long)nsm * 8;  // grid-stride beyond eight CTAs per SM
    if (blocks > cap) blocks = cap;
    kv_append_kernel<<<(unsigned)blocks, kThreadsPerCta, 0, st>>>(
        reinterpret_cast<const uint4 *>(a.k_new), reinterpret_cast<const uint4 *>(a.v_new), a.slots, a.n,
        row_chunks, a.num_slots, reinterpret_cast<uint4 *>(a.k_pool), reinterpret_cast<uint4 *>(a.v_pool),
        a.flags);
    return cudaGetLastError();
}

}  // namespace pillar
