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
#include "pkv_common.cuh"
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

// E4M3 pools ("ML Interview Prep, Lesson 13" section 3.7: an fp8 KV cache; "07 --
// Inference" section 4.3: E4M3, max 448, scales per channel). Each code is the
// new bf16 value divided by its kv head's scale (float, round to nearest) and
// rounded to the nearest E4M3 value, ties to even, saturating at +-448. A
// thread turns 8 bf16 (16 bytes) into 8 codes (8 bytes).
__device__ __forceinline__ uint32_t quantise4(uint32_t a, uint32_t b, float s)
{
    const uint32_t lo = pack_e4m3x2(__fdiv_rn(bf16lo_f32(a), s), __fdiv_rn(bf16hi_f32(a), s));
    const uint32_t hi = pack_e4m3x2(__fdiv_rn(bf16lo_f32(b), s), __fdiv_rn(bf16hi_f32(b), s));
    return lo | (hi << 16);
}

__global__ void __launch_bounds__(256) kv_append_fp8_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    const int64_t *__restrict__ slot_mapping, uint2 *__restrict__ k_cache,
    uint2 *__restrict__ v_cache, const float *__restrict__ k_scale,
    const float *__restrict__ v_scale, int64_t total_slots, int row_vec, int head_dim)
{
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t i = blockIdx.x;
    const int64_t slot = __ldg(slot_mapping + i);
    if (slot < 0 || slot >= total_slots)
        return;
    for (int e = threadIdx.x; e < 2 * row_vec; e += blockDim.x) {
        const bool is_v = e >= row_vec;
        const int c = is_v ? e - row_vec : e;  // 8-element group within the token row
        const int h = (c * 8) / head_dim;
        const float s = __ldg((is_v ? v_scale : k_scale) + h);
        const uint4 x = __ldg((is_v ? v_new : k_new) + i * row_vec + c);
        uint2 q;
        q.x = quantise4(x.x, x.y, s);
        q.y = quantise4(x.z, x.w, s);
        (is_v ? v_cache : k_cache)[slot * row_vec + c] = q;
    }
}

cudaError_t launch_kv_append_fp8(const void *k_new, const void *v_new,
                                 const int64_t *slot_mapping, int64_t n_new, void *k_cache,
                                 void *v_cache, int64_t num_blocks, int num_kv_heads,
                                 int head_dim, const float *k_scale, const float *v_scale,
                                 cudaStream_t stream)
{
    const int row_vec = num_kv_heads * head_dim / 8;  // 8-element groups per token row
    int threads = 2 * row_vec;
    if (threads > 256)
        threads = 256;
    threads = (threads + 31) / 32 * 32;
    kv_append_fp8_kernel<<<static_cast<unsigned>(n_new), threads, 0, stream>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping,
        static_cast<uint2 *>(k_cache), static_cast<uint2 *>(v_cache), k_scale, v_scale,
        num_blocks * kBlockSize, row_vec, head_dim);
    return cudaGetLastError();
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
