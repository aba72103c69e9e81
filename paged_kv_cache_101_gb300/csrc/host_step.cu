// host_step.cu -- one decode step from host memory through the C ABI: one
// host-to-device copy of the step's inputs (packed in one arena), the KV append
// and the attention on views of the device arena, one device-to-host copy of
// the output.
#include <cuda_runtime.h>

#include <stdint.h>

#include "pkv.h"

namespace {

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Byte sizes of the six inputs, in arena order; false for an unsupported geometry.
bool input_sizes(int32_t S, int32_t nq, int32_t Hq, int32_t Hkv, int32_t D, int32_t MB,
                 size_t sz[6])
{
    if (S < 0 || nq < 1 || nq > 4 || Hkv < 1 || Hq < 1 || Hq % Hkv != 0 ||
        (D != 64 && D != 128) || MB < 1 || (Hq / Hkv) * nq > 32 || S > (1 << 24) ||
        MB > (1 << 26))
        return false;
    const size_t rows = size_t(S) * size_t(nq);
    sz[0] = rows * size_t(Hq) * size_t(D) * 2;   // q, bf16
    sz[1] = rows * size_t(Hkv) * size_t(D) * 2;  // k_new, bf16
    sz[2] = sz[1];                               // v_new
    sz[3] = rows * 8;                            // slot_mapping, int64
    sz[4] = size_t(S) * size_t(MB) * 4;          // block_tables, int32
    sz[5] = size_t(S) * 4;                       // context_lens, int32
    return true;
}

}  // namespace

extern "C" {

size_t pkv_step_arena_layout(int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t max_blocks_per_seq,
                             size_t offsets[6])
{
    size_t sz[6];
    if (!input_sizes(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim,
                     max_blocks_per_seq, sz))
        return 0;
    size_t off = 0;
    for (int i = 0; i < 6; ++i) {
        if (offsets)
            offsets[i] = off;
        off = up256(off + sz[i]);
    }
    return off;
}

pkv_status pkv_decode_step_host(const void *host_arena, void *device_arena, size_t arena_bytes,
                                void *k_cache, void *v_cache, int64_t num_blocks,
                                int32_t max_blocks_per_seq, int32_t num_seqs,
                                int32_t n_query_per_seq, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim, float scale,
                                void *out_device, void *out_host, int32_t out_dtype,
                                void *workspace, size_t workspace_bytes, void *stream)
{
    size_t sz[6], off[6];
    if (!input_sizes(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim,
                     max_blocks_per_seq, sz))
        return num_seqs < 0 || max_blocks_per_seq < 1 ? PKV_ERR_SHAPE : PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0)
        return PKV_OK;
    const size_t need = pkv_step_arena_layout(num_seqs, n_query_per_seq, num_q_heads,
                                              num_kv_heads, head_dim, max_blocks_per_seq, off);
    if (!host_arena || !device_arena || !out_host)
        return PKV_ERR_NULL;
    if (arena_bytes < need)
        return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(device_arena) % 256 != 0)
        return PKV_ERR_ALIGN;
    if (out_dtype != PKV_BF16 && out_dtype != PKV_FP32)
        return PKV_ERR_DTYPE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t *d = static_cast<const uint8_t *>(device_arena);
    const int64_t n_new = int64_t(num_seqs) * n_query_per_seq;
    const size_t out_bytes = size_t(n_new) * size_t(num_q_heads) * size_t(head_dim) *
                             (out_dtype == PKV_FP32 ? 4 : 2);

    // the device-side checks of both calls first, so a refused step enqueues nothing
    if (!out_device || !k_cache || !v_cache)
        return PKV_ERR_NULL;
    if (num_blocks < 1)
        return PKV_ERR_SHAPE;
    if (!workspace)
        return PKV_ERR_WORKSPACE;
    if (workspace_bytes < pkv_workspace_size(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads,
                                             head_dim))
        return PKV_ERR_WORKSPACE;

    if (cudaMemcpyAsync(device_arena, host_arena, need, cudaMemcpyHostToDevice, st) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    pkv_status s = pkv_kv_append(d + off[1], d + off[2], reinterpret_cast<const int64_t *>(d + off[3]),
                                 n_new, k_cache, v_cache, num_blocks, num_kv_heads, head_dim,
                                 stream);
    if (s != PKV_OK)
        return s;
    s = pkv_paged_decode_attention(d + off[0], k_cache, v_cache, num_blocks,
                                   reinterpret_cast<const int32_t *>(d + off[4]),
                                   max_blocks_per_seq,
                                   reinterpret_cast<const int32_t *>(d + off[5]), num_seqs,
                                   n_query_per_seq, num_q_heads, num_kv_heads, head_dim, scale,
                                   out_device, out_dtype, workspace, workspace_bytes, stream);
    if (s != PKV_OK)
        return s;
    if (cudaMemcpyAsync(out_host, out_device, out_bytes, cudaMemcpyDeviceToHost, st) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // extern "C"
