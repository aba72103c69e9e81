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

}  // namespace

extern "C" pkv_status pkv_paged_decode_attention_static(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
    int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, float scale, void *out, int32_t out_dtype, void *stream)
{
    // Every host check of the workspace entry point, in its order, and the
    // scratch bytes of the very plan the call below will run (grid, options).
    size_t need = 0;
    const pkv_status st = pkv::attention_need(q, k_cache, v_cache, num_blocks, block_tables,
                                              max_blocks_per_seq, context_lens, num_seqs,
                                              n_query_per_seq, num_q_heads, num_kv_heads,
                                              head_dim, out, out_dtype, &need);
    if (st != PKV_OK || need == 0)
        return st;  // an invalid argument, or nothing to do (num_seqs == 0)
    if (need > kStaticScratchBytes)
        return PKV_ERR_WORKSPACE;  // this geometry needs more than the static maximum
    void *scratch = static_scratch_address();
    if (scratch == nullptr)
        return PKV_ERR_CUDA;
    // The header (device error word, work counters) must start at zero; every
    // other byte of the scratch is written by the kernels before it is read.
    if (cudaMemsetAsync(scratch, 0, pkv::kWsHeaderBytes, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    return pkv_paged_decode_attention(q, k_cache, v_cache, num_blocks, block_tables,
                                      max_blocks_per_seq, context_lens, num_seqs, n_query_per_seq,
                                      num_q_heads, num_kv_heads, head_dim, scale, out, out_dtype,
                                      scratch, kStaticScratchBytes, stream);
}

extern "C" pkv_status pkv_static_error_word(uint32_t *host_word, void *stream)
{
    if (host_word == nullptr)
        return PKV_ERR_NULL;
    void *scratch = static_scratch_address();
    if (scratch == nullptr)
        return PKV_ERR_CUDA;
    // A plain 4-byte read of the header's first word after the stream's work.
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host_word, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}
