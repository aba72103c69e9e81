// host_step.cu -- one decode step from host memory through the C ABI: one
// host-to-device copy of the step's inputs (packed in one arena), the KV append
// and the attention on views of the device arena, one device-to-host copy of
// the output. The pipelined form puts the two copies and the kernels on three
// streams, ordered by the caller's events, so that a loop over steps overlaps
// each step's copies with its neighbours' kernels.
#include <cuda_runtime.h>

#include <stdint.h>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Byte sizes of the six inputs, in arena order; false for an unsupported geometry.
bool input_sizes(int32_t S, int32_t nq, int32_t Hq, int32_t Hkv, int32_t D, int32_t MB,
                 size_t sz[6])
{
    if (S < 0 || nq < 1 || nq > 4 || Hkv < 1 || Hq < 1 || Hq % Hkv != 0 ||
        (D != 64 && D != 128) || MB < 1 || (Hq / Hkv) * nq > 64 || S > (1 << 24) ||
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

}  // extern "C"

namespace {

// A validated step: the arena offsets and the output's bytes.
struct StepPlan {
    size_t off[6];
    size_t need, out_bytes;
    int64_t n_new;
};

// The checks of both calls that do not depend on device data, so that a refused
// step enqueues nothing.
pkv_status plan_step(const void *host_arena, const void *device_arena, size_t arena_bytes,
                     const void *k_cache, const void *v_cache, int64_t num_blocks,
                     int32_t max_blocks_per_seq, int32_t num_seqs, int32_t n_query_per_seq,
                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                     const void *out_device, const void *out_host, int32_t out_dtype,
                     const void *workspace, size_t workspace_bytes, StepPlan *sp)
{
    size_t sz[6];
    if (!input_sizes(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim,
                     max_blocks_per_seq, sz))
        return num_seqs < 0 || max_blocks_per_seq < 1 ? PKV_ERR_SHAPE : PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0)
        return PKV_OK;
    sp->need = pkv_step_arena_layout(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads,
                                     head_dim, max_blocks_per_seq, sp->off);
    if (!host_arena || !device_arena || !out_host)
        return PKV_ERR_NULL;
    if (arena_bytes < sp->need)
        return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(device_arena) % 256 != 0)
        return PKV_ERR_ALIGN;
    if (out_dtype != PKV_BF16 && out_dtype != PKV_FP32)
        return PKV_ERR_DTYPE;
    sp->n_new = int64_t(num_seqs) * n_query_per_seq;
    sp->out_bytes = size_t(sp->n_new) * size_t(num_q_heads) * size_t(head_dim) *
                    (out_dtype == PKV_FP32 ? 4 : 2);
    if (!out_device || !k_cache || !v_cache)
        return PKV_ERR_NULL;
    if (num_blocks < 1)
        return PKV_ERR_SHAPE;
    if (!workspace)
        return PKV_ERR_WORKSPACE;
    if (workspace_bytes < pkv_workspace_size(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads,
                                             head_dim))
        return PKV_ERR_WORKSPACE;
    return PKV_OK;
}

// Steps 2 and 3 on `stream`: the append and the attention on the arena's views
// (E4M3 pools when both scales are given).
pkv_status compute_step(const StepPlan &sp, const void *device_arena, void *k_cache,
                        void *v_cache, int64_t num_blocks, int32_t max_blocks_per_seq,
                        int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                        int32_t num_kv_heads, int32_t head_dim, float scale, void *out_device,
                        int32_t out_dtype, void *workspace, size_t workspace_bytes,
                        const float *k_scale, const float *v_scale, void *stream)
{
    const uint8_t *d = static_cast<const uint8_t *>(device_arena);
    if (k_scale && v_scale) {
        pkv_status s = pkv_kv_append_fp8(d + sp.off[1], d + sp.off[2],
                                         reinterpret_cast<const int64_t *>(d + sp.off[3]),
                                         sp.n_new, k_cache, v_cache, num_blocks, num_kv_heads,
                                         head_dim, k_scale, v_scale, stream);
        if (s != PKV_OK)
            return s;
        // the append just enqueued writes only the pool; the arena was in place before it
        pkv::set_meta_ready(true);
        s = pkv_paged_decode_attention_fp8(
            d + sp.off[0], k_cache, v_cache, num_blocks, k_scale, v_scale,
            reinterpret_cast<const int32_t *>(d + sp.off[4]), max_blocks_per_seq,
            reinterpret_cast<const int32_t *>(d + sp.off[5]), num_seqs, n_query_per_seq,
            num_q_heads, num_kv_heads, head_dim, scale, out_device, out_dtype, workspace,
            workspace_bytes, stream);
        pkv::set_meta_ready(false);
        return s;
    }
    pkv_status s = pkv_kv_append(d + sp.off[1], d + sp.off[2],
                                 reinterpret_cast<const int64_t *>(d + sp.off[3]), sp.n_new,
                                 k_cache, v_cache, num_blocks, num_kv_heads, head_dim, stream);
    if (s != PKV_OK)
        return s;
    pkv::set_meta_ready(true);
    s = pkv_paged_decode_attention(d + sp.off[0], k_cache, v_cache, num_blocks,
                                   reinterpret_cast<const int32_t *>(d + sp.off[4]),
                                   max_blocks_per_seq,
                                   reinterpret_cast<const int32_t *>(d + sp.off[5]), num_seqs,
                                   n_query_per_seq, num_q_heads, num_kv_heads, head_dim, scale,
                                   out_device, out_dtype, workspace, workspace_bytes, stream);
    pkv::set_meta_ready(false);
    return s;
}

}  // namespace

extern "C" {

pkv_status pkv_decode_step(const void *q, const void *k_new, const void *v_new,
                           const int64_t *slot_mapping, void *k_cache, void *v_cache,
                           int64_t num_blocks, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, float scale, void *out,
                           int32_t out_dtype, void *workspace, size_t workspace_bytes,
                           const float *k_scale, const float *v_scale, void *stream)
{
    if ((k_scale == nullptr) != (v_scale == nullptr))
        return PKV_ERR_NULL;
    const int kv8 = k_scale ? 1 : 0;
    // every check of both calls before anything is enqueued: the attention's (with
    // the workspace its plan needs), then the append's own (it checks before it
    // enqueues)
    size_t need = 0;
    pkv_status s = pkv::attention_check(q, k_cache, v_cache, num_blocks, kv8, k_scale, v_scale,
                                        block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                        n_query_per_seq, num_q_heads, num_kv_heads, head_dim, out,
                                        out_dtype, &need);
    if (s != PKV_OK)
        return s;
    if (need > 0) {
        if (!workspace || workspace_bytes < need)
            return PKV_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
            return PKV_ERR_ALIGN;
    }
    const int64_t n_new = int64_t(num_seqs) * n_query_per_seq;
    s = kv8 ? pkv_kv_append_fp8(k_new, v_new, slot_mapping, n_new, k_cache, v_cache, num_blocks,
                                num_kv_heads, head_dim, k_scale, v_scale, stream)
            : pkv_kv_append(k_new, v_new, slot_mapping, n_new, k_cache, v_cache, num_blocks,
                            num_kv_heads, head_dim, stream);
    if (s != PKV_OK)
        return s;
    // the append just enqueued writes only the pools, and the caller's q, tables and
    // lengths were complete before it ran: the attention plans its cells while the
    // append runs and waits for it only before its first read of the pool
    pkv::set_meta_ready(true);
    s = kv8 ? pkv_paged_decode_attention_fp8(q, k_cache, v_cache, num_blocks, k_scale, v_scale,
                                             block_tables, max_blocks_per_seq, context_lens,
                                             num_seqs, n_query_per_seq, num_q_heads, num_kv_heads,
                                             head_dim, scale, out, out_dtype, workspace,
                                             workspace_bytes, stream)
            : pkv_paged_decode_attention(q, k_cache, v_cache, num_blocks, block_tables,
                                         max_blocks_per_seq, context_lens, num_seqs,
                                         n_query_per_seq, num_q_heads, num_kv_heads, head_dim,
                                         scale, out, out_dtype, workspace, workspace_bytes, stream);
    pkv::set_meta_ready(false);
    return s;
}

pkv_status pkv_decode_step_host(const void *host_arena, void *device_arena, size_t arena_bytes,
                                void *k_cache, void *v_cache, int64_t num_blocks,
                                int32_t max_blocks_per_seq, int32_t num_seqs,
                                int32_t n_query_per_seq, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim, float scale,
                                void *out_device, void *out_host, int32_t out_dtype,
                                void *workspace, size_t workspace_bytes, void *stream)
{
    StepPlan sp;
    pkv_status s = plan_step(host_arena, device_arena, arena_bytes, k_cache, v_cache, num_blocks,
                             max_blocks_per_seq, num_seqs, n_query_per_seq, num_q_heads,
                             num_kv_heads, head_dim, out_device, out_host, out_dtype, workspace,
                             workspace_bytes, &sp);
    if (s != PKV_OK || num_seqs == 0)
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(device_arena, host_arena, sp.need, cudaMemcpyHostToDevice, st) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    s = compute_step(sp, device_arena, k_cache, v_cache, num_blocks, max_blocks_per_seq, num_seqs,
                     n_query_per_seq, num_q_heads, num_kv_heads, head_dim, scale, out_device,
                     out_dtype, workspace, workspace_bytes, nullptr, nullptr, stream);
    if (s != PKV_OK)
        return s;
    if (cudaMemcpyAsync(out_host, out_device, sp.out_bytes, cudaMemcpyDeviceToHost, st) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

pkv_status pkv_decode_step_host_pipelined(
    const void *host_arena, void *device_arena, size_t arena_bytes, void *k_cache, void *v_cache,
    int64_t num_blocks, int32_t max_blocks_per_seq, int32_t num_seqs, int32_t n_query_per_seq,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale, void *out_device,
    void *out_host, int32_t out_dtype, void *workspace, size_t workspace_bytes,
    const float *k_scale, const float *v_scale, void *upload_stream, void *compute_stream,
    void *download_stream, void *uploaded, void *computed, void *downloaded)
{
    StepPlan sp;
    pkv_status s = plan_step(host_arena, device_arena, arena_bytes, k_cache, v_cache, num_blocks,
                             max_blocks_per_seq, num_seqs, n_query_per_seq, num_q_heads,
                             num_kv_heads, head_dim, out_device, out_host, out_dtype, workspace,
                             workspace_bytes, &sp);
    if (s != PKV_OK || num_seqs == 0)
        return s;
    if (!uploaded || !computed || !downloaded || (!k_scale) != (!v_scale))
        return PKV_ERR_NULL;
    if (k_scale && head_dim != 128)
        return PKV_ERR_UNSUPPORTED;  // E4M3 rows are one 128-byte row
    cudaStream_t up = static_cast<cudaStream_t>(upload_stream);
    cudaStream_t comp = static_cast<cudaStream_t>(compute_stream);
    cudaStream_t down = static_cast<cudaStream_t>(download_stream);
    cudaEvent_t e_up = static_cast<cudaEvent_t>(uploaded);
    cudaEvent_t e_comp = static_cast<cudaEvent_t>(computed);
    cudaEvent_t e_down = static_cast<cudaEvent_t>(downloaded);
    // 1. upload, once this slot's previous step has read its device arena
    if (cudaStreamWaitEvent(up, e_comp, 0) != cudaSuccess ||
        cudaMemcpyAsync(device_arena, host_arena, sp.need, cudaMemcpyHostToDevice, up) !=
            cudaSuccess ||
        cudaEventRecord(e_up, up) != cudaSuccess)
        return PKV_ERR_CUDA;
    // 2-3. append and attention, after the upload and after this slot's previous
    // output has left out_device
    if (cudaStreamWaitEvent(comp, e_up, 0) != cudaSuccess ||
        cudaStreamWaitEvent(comp, e_down, 0) != cudaSuccess)
        return PKV_ERR_CUDA;
    s = compute_step(sp, device_arena, k_cache, v_cache, num_blocks, max_blocks_per_seq, num_seqs,
                     n_query_per_seq, num_q_heads, num_kv_heads, head_dim, scale, out_device,
                     out_dtype, workspace, workspace_bytes, k_scale, v_scale, compute_stream);
    if (s != PKV_OK)
        return s;
    if (cudaEventRecord(e_comp, comp) != cudaSuccess)
        return PKV_ERR_CUDA;
    // 4. download
    if (cudaStreamWaitEvent(down, e_comp, 0) != cudaSuccess ||
        cudaMemcpyAsync(out_host, out_device, sp.out_bytes, cudaMemcpyDeviceToHost, down) !=
            cudaSuccess ||
        cudaEventRecord(e_down, down) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // extern "C"
