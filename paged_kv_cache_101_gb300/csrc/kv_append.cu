// kv_append.cu -- write this step's new K/V rows into their slots of the paged pool.
//
// "LLM Inference Serving", block-table pseudo-code: a generated token is
// appended in place into its sequence's last block (the host allocates a new
// block first when that one is full). The host hands over one slot per new
// token (physical_block * 16 + offset); since the pool is
// [num_blocks][16][Hkv][D], slot * Hkv * D is the row's element offset.
//
// One CTA per new token; its threads move the token's K and V rows (2*Hkv*D
// bf16) as 16-byte vectors, fully coalesced on both sides. A negative slot is
// padding; a slot past the pool is skipped, never written.
#include "pkv_internal.h"

namespace pkv {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4 *__restrict__ k_new,
                                                        const uint4 *__restrict__ v_new,
                                                        const int64_t *__restrict__ slot_mapping,
                                                        uint4 *__restrict__ k_cache,
                                                        uint4 *__restrict__ v_cache,
                                                        int64_t total_slots, int row_vec)
{
    // a dependent launched with programmatic serialization (the attention
    // kernel) may start its prologue now; it waits for this grid's completion
    // before it reads anything from global memory
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t i = blockIdx.x;
    const int64_t slot = __ldg(slot_mapping + i);
    if (slot < 0 || slot >= total_slots)
        return;
    const uint4 *ks = k_new + i * row_vec;
    const uint4 *vs = v_new + i * row_vec;
    uint4 *kd = k_cache + slot * row_vec;
    uint4 *vd = v_cache + slot * row_vec;
    for (int e = threadIdx.x; e < 2 * row_vec; e += blockDim.x) {
        if (e < row_vec)
            kd[e] = __ldg(ks + e);
        else
            vd[e - row_vec] = __ldg(vs + (e - row_vec));
    }
}

cudaError_t launch_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                             int64_t n_new, void *k_cache, void *v_cache, int64_t num_blocks,
                             int num_kv_heads, int head_dim, cudaStream_t stream)
{
    const int row_vec = num_kv_heads * head_dim / 8;  // 16-byte vectors per K row
    int threads = 2 * row_vec;
    if (threads > 256)
        threads = 256;
    threads = (threads + 31) / 32 * 32;
    // grid.x is limited to 2^31 - 1 blocks; the host checks n_new against it.
    kv_append_kernel<<<static_cast<unsigned>(n_new), threads, 0, stream>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping,
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
        num_blocks * kBlockSize, row_vec);
    return cudaGetLastError();
}

}  // namespace pkv
