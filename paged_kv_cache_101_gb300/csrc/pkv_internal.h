// pkv_internal.h -- shapes shared by the host API and the kernels of libpkv.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kBlockSize = 16;          // tokens per physical block
constexpr int kTileBytes = 16 * 128;    // one (head, 64-column half) tile: 16 rows x 128 B
constexpr int kMaxRows = 64;            // query rows per kv head: G * n_query_per_seq
constexpr int kMaxConsumerWarps = 8;
// warp 0 produces, warps 1..ncw consume
constexpr int kThreadsMax = 32 * (1 + kMaxConsumerWarps);
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits: 2 s
// per-CTA trace words: entry, first TMA issued, first stage consumed, last TMA
// issued, last stage consumed (ns, %globaltimer), units, segments, SM id,
// paced stages, 7 spare
constexpr int kTraceWords = 16;
constexpr int kMaxPreChunks = 4;  // cascade: prefix partials per row

// device error word codes (workspace offset 0)
enum : uint32_t {
    kErrConsumerWait = 1u,  // a consumer warp gave up waiting for a stage
    kErrProducerWait = 2u,  // the producer gave up waiting for a free stage
    kErrDrainWait = 4u,     // a copy did not land while unwinding
    kErrBadBlock = 8u,      // a block-table entry outside [0, num_blocks) (read as zeros)
    kErrBadQuery = 16u,     // variable query counts: a sequence's rows or table row invalid
    kErrBadGroup = 32u      // cascade: a prefix group outside the batch or the tables
};

// Split of the work of one call (computed on the host from the shapes).
struct DecodePlan {
    int D;           // head_dim
    int G;           // query heads per kv head
    int rows;        // G * nq: query rows per kv head
    int wph;         // consumer warps per kv head (1 or 2)
    int ntw;         // 8-row n-tiles per consumer warp (0: CUDA-core consumers)
    int rows_pad;    // wph * ntw * 8
    int HG;          // kv heads per head group (one CTA streams one group)
    int n_hg;        // Hkv / HG
    int threads;     // 32 * (1 + HG * wph)
    int stage_bytes; // K + V of one 16-token block for HG heads
    int nst;         // pipeline stages
    int whole_box;   // 1: one TMA box per block for K (and V) of all HG heads
    int kv8;         // 1: E4M3 pools (one 128-byte tile per head row), 0: bf16
    int fma;         // 1: CUDA-core (fp32 FMA) consumers instead of tensor cores
    int rw;          // CUDA-core consumers: query rows per warp (4 or 8)
    int prefix;      // 1: the cascade's prefix pass (one head per CTA, 8 warps x 16 rows)
    int umma;        // 1: tcgen05 consumers (one head per CTA, rows padded to rows_pad = N)
    int grid;        // persistent CTAs
    int ctas_per_sm; // CTAs of the grid resident per SM (1, or 2 for the E4M3 5-8-row shape)
    int tickets_max; // cap on dynamically claimed tickets (0: static chunks only)
    int tail_div;    // the last 1/tail_div of the units go out as tickets (0: none)
    size_t smem;     // dynamic shared memory bytes
    // workspace layout (byte offsets)
    size_t off_rec, off_ml, off_part, ws_bytes;
};

// Workspace header words (uint32 at byte offset 4*i).
// kWsUnits: blocks of all sequences (per head group); kWsDense: 1 if no cell is
// empty (both written by CTA 0 of the main pass for the merge).
enum {
    kWsErr = 0,
    kWsTicket = 2,
    kWsDone = 3,
    kWsProgress = 4,
    kWsUnits = 5,
    kWsDense = 6,
    kWsHeaderBytes = 256
};
struct DecodeParams {
    const uint16_t *q;
    void *out;
    const int32_t *block_tables;
    const int32_t *context_lens;
    uint32_t *ws;          // workspace header: error word, ticket, done and progress counters
    int2 *pieces;          // [S][n_hg] cells of the first and last piece (for the merge)
    float *ml;             // [cells][2][HG][rows] (m, l) partial states
    float *part;           // [cells][2][HG][rows][D] unnormalised partial acc
    uint64_t *trace;       // optional per-CTA timeline [grid][kTraceWords] (null: off)
    int64_t num_blocks;
    int S, MB, nq, Hq, Hkv, G, rows, rows_pad, HG, n_hg, out_f32;
    int stage_bytes, nst;
    int whole_box;         // 1: the tensor maps box a whole block (HG heads) at once
    int ncw;               // consumer warps per CTA (HG * wph)
    int tickets_max;       // dynamic tickets: at most this many (0: none)
    int ticket_div;        // the last F / ticket_div units go to tickets
    int ticket_units;      // at least this many units per ticket
    float scale_log2;      // scale * log2(e)
    int pace;              // pacing: one stage fewer in flight while ahead of the grid (0: off)
    int meta_ready;        // 1: the kernel before this one on the stream writes none of the
                           // lengths, tables and queries (the library's own KV append in a
                           // host step): the producer reads them before the grid dependency
                           // wait and waits only before its first read of the pool
    float pace_margin;     // pacing: lead (fraction of the work) allowed before pacing
    int pf_units;          // tcgen05 kernel: blocks prefetched into L2 ahead of the loads
    const float *k_scale;  // E4M3 pools: [Hkv] dequantisation scales (null for bf16)
    const float *v_scale;
    // variable query counts (all null for a fixed n_query_per_seq = nq, causal):
    const int32_t *q_start;     // [S + 1] first query row of each sequence
    const uint32_t *tree_mask;  // [total_q] per-row visibility bits over the window
    const int32_t *tree_len;    // [S] mask window (positions T - W .. T - 1)
    const int32_t *table_row;   // [S] block-table row of each sequence
    int total_q;                // rows of q and out
    int table_rows;             // rows of block_tables
    // shared-prefix cascade (null / 0 without): groups [num_groups][3] = (first
    // sequence, sequences, prefix blocks), members consecutive, groups ascending
    const int32_t *prefix_groups;
    int num_groups;
    int prefix_pass;            // 1: this launch attends the groups' prefixes
    int pre_tiles;              // prefix pass: row tiles per group
    int pre_qrows;              // prefix pass: query rows per tile
    int pre_chunks;             // prefix pass: each group's prefix cut into this many
                                // block ranges (one partial each, at most kMaxPreChunks)
    float *pre_ml;              // [chunk][total_q][Hq][2] (m, l) of each row over a prefix chunk
    float *pre_acc;             // [chunk][total_q][Hq][D] unnormalised acc over the chunk
};

// Host steps (host_step.cu) mark the attention call that follows their own KV
// append on the calling thread: its metadata is in place before that append runs.
void set_meta_ready(bool ready);

// umma = 1: kv heads with 17..64 query rows (bf16 pools, head_dim 128) take the
// tcgen05 kernel; 0: the mma.sync kernels serve every shape.
int plan_decode(int S, int nq, int Hq, int Hkv, int D, int MB, int num_sms, int opt_ctas,
                int opt_stages, int opt_heads, int opt_tail, int smem_optin, int kv8, int fma,
                int umma, DecodePlan *plan);

// The tcgen05 kernel (paged_decode_umma.cu): shared memory and super-stages for
// N = 32 or 64 padded rows; the launch of it and its merge. qmap views q as
// (64, 2, Hq, rows, 1) with a box of (64, 1, G, n_query_per_seq, 1).
size_t umma_smem_bytes(int n);
int umma_stages(int n);
cudaError_t launch_decode_umma(const DecodePlan &plan, const DecodeParams &p,
                               const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const CUtensorMap &qmap, cudaStream_t stream, cudaEvent_t ev_before,
                               cudaEvent_t ev_after);

// The merge of the split sequences' partials (a programmatic dependent).
cudaError_t launch_merge(const DecodePlan &plan, const DecodeParams &p, cudaStream_t stream);

// The cascade's prefix pass (one head per CTA, 128 score rows per tile); returns
// the row tiles per group, or -1 if unsupported.
int plan_prefix(int D, int G, int Hkv, int num_groups, int max_group_seqs, int nq,
                int smem_optin, DecodePlan *plan);

// ev_before/ev_after (may be null) are recorded around the kernel.
cudaError_t launch_decode(const DecodePlan &plan, const DecodeParams &p, const CUtensorMap &kmap,
                          const CUtensorMap &vmap, cudaStream_t stream, cudaEvent_t ev_before,
                          cudaEvent_t ev_after);

// The host-side checks of pkv_paged_decode_attention, in its order, with the
// workspace taken as given; on PKV_OK *need holds the workspace bytes the call's
// plan needs (0 when there is nothing to do). Enqueues nothing.
pkv_status attention_need(const void *q, const void *k_cache, const void *v_cache,
                          int64_t num_blocks,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs, int32_t n_query_per_seq,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, void *out,
                          int32_t out_dtype, size_t *need);
// The same checks for either pool type (kv8: E4M3 pools with per-head scales), with
// the workspace taken as given: the bytes the call's plan needs go to *need.
pkv_status attention_check(const void *q, const void *k_cache, const void *v_cache,
                           int64_t num_blocks, int kv8, const float *k_scale,
                           const float *v_scale, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, void *out, int32_t out_dtype,
                           size_t *need);

cudaError_t launch_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                             int64_t n_new, void *k_cache, void *v_cache, int64_t num_blocks,
                             int num_kv_heads, int head_dim, cudaStream_t stream);

// E4M3 pools: quantise the new rows with per-kv-head scales.
cudaError_t launch_kv_append_fp8(const void *k_new, const void *v_new,
                                 const int64_t *slot_mapping, int64_t n_new, void *k_cache,
                                 void *v_cache, int64_t num_blocks, int num_kv_heads,
                                 int head_dim, const float *k_scale, const float *v_scale,
                                 cudaStream_t stream);

}  // namespace pkv
