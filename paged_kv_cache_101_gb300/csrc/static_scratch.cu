// static_scratch.cu -- pkv_paged_decode_attention_static: decode attention for
// callers that cannot allocate device memory.
//
// The scratch the attention kernels need (split-K partials, the merge's piece
// records, error word) lives in a file-scope device array instead of a caller-provided
// workspace. Host code cannot use the array's name as a device address (on the
// host it is only a stand-in symbol), so the first call on each device looks up
// the real address with cudaGetSymbolAddress, with that device current, and the
// kernels are handed that pointer. Nothing here allocates: no cudaMalloc,
// cudaFree or allocating library routine.
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

// Shared by every call on a device; keeps the previous call's contents.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void *g_static_ptr[64] = {};

// Device address of g_static_scratch on the current device (looked up once per
// device). Returns null if the lookup fails.
void *static_scratch_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (g_static_ptr[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || p == nullptr)
            return nullptr;
        g_static_ptr[dev] = p;
    }
    return g_static_ptr[dev];
}

bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" pkv_status pkv_paged_decode_attention_static(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
    int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, float scale, void *out, int32_t out_dtype, void *stream)
{
    // Let the regular entry point report invalid arguments (it checks them all
    // before touching the device); only then set up and clear the scratch.
    const bool plausible = num_seqs > 0 && q && k_cache && v_cache && block_tables &&
                           context_lens && out && num_blocks >= 1 && max_blocks_per_seq >= 1 &&
                           (out_dtype == PKV_BF16 || out_dtype == PKV_FP32) &&
                           aligned_to(q, 16) && aligned_to(k_cache, 16) && aligned_to(v_cache, 16) &&
                           aligned_to(out, 16) && aligned_to(block_tables, 4) &&
                           aligned_to(context_lens, 4) && max_blocks_per_seq <= (1 << 26) &&
                           num_blocks <= 0x7fffffffLL && num_seqs <= (1 << 24) &&
                           num_kv_heads <= 65535;
    if (!plausible)
        return pkv_paged_decode_attention(q, k_cache, v_cache, num_blocks, block_tables,
                                          max_blocks_per_seq, context_lens, num_seqs,
                                          n_query_per_seq, num_q_heads, num_kv_heads, head_dim,
                                          scale, out, out_dtype, nullptr, 0, stream);
    const size_t need = pkv_workspace_size(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads,
                                           head_dim);
    if (need == 0)  // unsupported geometry or no usable device: full validation says which
        return pkv_paged_decode_attention(q, k_cache, v_cache, num_blocks, block_tables,
                                          max_blocks_per_seq, context_lens, num_seqs,
                                          n_query_per_seq, num_q_heads, num_kv_heads, head_dim,
                                          scale, out, out_dtype, nullptr, 0, stream);
    if (need > kStaticScratchBytes)
        return PKV_ERR_WORKSPACE;  // this geometry needs more than the static maximum
    void *scratch = static_scratch_address();
    if (scratch == nullptr)
        return PKV_ERR_CUDA;
    // The header (device error word, work counters) must start at zero; every
    // other byte of the scratch is written by the kernels before it is read.
    const size_t zero = pkv::workspace_zero_prefix(num_seqs, n_query_per_seq, num_q_heads,
                                                   num_kv_heads, head_dim);
    if (zero == 0 || zero > kStaticScratchBytes)
        return PKV_ERR_CUDA;
    if (cudaMemsetAsync(scratch, 0, zero, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return pkv_paged_decode_attention(q, k_cache, v_cache, num_blocks, block_tables,
                                      max_blocks_per_seq, context_lens, num_seqs, n_query_per_seq,
                                      num_q_heads, num_kv_heads, head_dim, scale, out, out_dtype,
                                      scratch, kStaticScratchBytes, stream);
}
