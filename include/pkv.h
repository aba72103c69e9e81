/*
 * pkv.h -- C ABI of the paged KV-cache decode library for one NVIDIA GB300
 * (sm_103a).
 *
 * Two operations make up one decode step of PagedAttention-style serving:
 *
 *   pkv_kv_append                writes the step's new K/V rows into their
 *                                slots of the paged pool;
 *   pkv_paged_decode_attention   attends one or a few query tokens per
 *                                sequence over the pool, through per-sequence
 *                                block tables.
 *
 * When sequences share blocks, pkv_copy_blocks first gives a writer its
 * private copy of a shared block (copy-on-write). The host-side block
 * manager that decides slots, tables and copies is in pkv_block_manager.h.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named as device buffers must point to memory of the current
 *    CUDA device; the library never allocates, frees or copies them to the
 *    host. The caller owns every buffer.
 *  - `stream` is a cudaStream_t (passed as void* so this header needs no CUDA
 *    include); NULL means the legacy default stream. Work is enqueued
 *    asynchronously on it; a return of PKV_OK means the launch was accepted.
 *  - Arguments are validated on the host before anything is enqueued; an
 *    invalid argument returns its status code and enqueues nothing.
 *    Values that live in device memory (block ids, slots, context lengths)
 *    cannot be checked without a device-to-host copy: the kernels clamp or
 *    skip out-of-range values instead of faulting (documented per call), and
 *    the results for such inputs are unspecified.
 *  - bf16 is IEEE bfloat16 (the upper half of a binary32), little endian.
 *  - Physical block size is fixed at 16 tokens (vLLM's default, "ML Interview
 *    Prep, Lesson 13" section 3.5; "Chapter 18" section 18.2.2 on why 16).
 *  - KV pool layout ("LLM Inference Serving", KV-cache shape section): K and V
 *    are separate buffers, each [num_blocks][16][num_kv_heads][head_dim] bf16,
 *    row-major. Token slot `slot = physical_block * 16 + offset`.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_NULL = 1,        /* a required pointer is NULL                     */
    PKV_ERR_SHAPE = 2,       /* inconsistent or non-positive sizes             */
    PKV_ERR_DTYPE = 3,       /* unknown output dtype                           */
    PKV_ERR_ALIGN = 4,       /* a buffer is not aligned as required            */
    PKV_ERR_RANGE = 5,       /* a size is beyond what the library supports     */
    PKV_ERR_WORKSPACE = 6,   /* workspace missing or smaller than required     */
    PKV_ERR_CUDA = 7,        /* a CUDA runtime/driver call or launch failed    */
    PKV_ERR_UNSUPPORTED = 8, /* a valid shape the library has no kernel for   */
    PKV_ERR_NO_BLOCKS = 9,   /* block manager: not enough free blocks          */
    PKV_ERR_SEQUENCE = 10    /* block manager: unknown or duplicate sequence id */
} pkv_status;

typedef enum pkv_dtype {
    PKV_BF16 = 0,
    PKV_FP32 = 1
} pkv_dtype;

/*
 * pkv_kv_append -- write this step's new K/V rows into the paged pool.
 *
 * Passage: "LLM Inference Serving", block-table pseudo-code (when a token is
 * generated it is appended in place into the last block's free slot, a new
 * physical block being allocated first when that block is full) and "LLM
 * Serving: Continuous Batching & PagedAttention", section 4.1 (a new 16-token
 * block is taken from the free list when the sequence crosses a block
 * boundary). Block allocation is the caller's host-side job; this call only
 * writes rows: for every i in [0, n_new) with slot_mapping[i] >= 0,
 *     k_cache[slot/16][slot%16][h][:] = k_new[i][h][:]   for every kv head h,
 *     v_cache[slot/16][slot%16][h][:] = v_new[i][h][:].
 * The copy is bit-exact.
 *
 *   k_new, v_new   device, bf16 [n_new][num_kv_heads][head_dim], 16-byte aligned
 *   slot_mapping   device, int64 [n_new]; < 0 means "skip" (padding).
 *                  A slot >= num_blocks*16 is skipped as well (no write, no fault).
 *                  Two entries naming the same slot give an unspecified row.
 *   k_cache,v_cache device, bf16 [num_blocks][16][num_kv_heads][head_dim],
 *                  16-byte aligned; rows not named by slot_mapping are untouched.
 *   head_dim       a multiple of 8 (rows move in 16-byte vectors), <= 1024.
 *   n_new == 0     is a no-op returning PKV_OK.
 * Writing into a block shared by several sequences (reference count > 1) is
 * the caller's error: copy-on-write must happen first ("ML Interview Prep,
 * Lesson 13" section 3.5).
 */
pkv_status pkv_kv_append(const void *k_new, const void *v_new,
                         const int64_t *slot_mapping, int64_t n_new,
                         void *k_cache, void *v_cache, int64_t num_blocks,
                         int32_t num_kv_heads, int32_t head_dim, void *stream);

/*
 * pkv_copy_blocks -- copy whole physical blocks of the pool (copy-on-write).
 *
 * Passage: "ML Interview Prep, Lesson 13" section 3.5 "Sharing" (before a
 * sequence writes into a block whose reference count is above 1 it gets a
 * private copy, and the shared block's count drops by one) and "LLM Serving:
 * Continuous Batching & PagedAttention" section 4.2 (copy-on-write prefix
 * sharing). The host block manager (pkv_block_manager.h) decides the pairs;
 * this call moves the bytes: for every i in [0, num_pairs),
 *     k_cache[block_dst[i]][:] = k_cache[block_src[i]][:]   (all 16 token rows,
 *     v_cache[block_dst[i]][:] = v_cache[block_src[i]][:]    every kv head)
 * bit-exact. Enqueue it before the pkv_kv_append of the same step: the append
 * may write into a source block (its last sharer writes in place).
 *
 *   k_cache,v_cache device pool as described above, 16-byte aligned.
 *   block_src, block_dst device, int32 [num_pairs], 4-byte aligned. A pair
 *                  naming a block outside [0, num_blocks), or with src == dst,
 *                  is skipped (no write, no fault). The destinations must be
 *                  distinct and no destination may be another pair's source
 *                  (the pairs of one block-manager step always are); otherwise
 *                  the result is unspecified.
 *   head_dim       a multiple of 8, <= 1024 (16-byte vectors), as for the append.
 *   num_pairs == 0 is a no-op returning PKV_OK.
 */
pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, int64_t num_blocks,
                           int32_t num_kv_heads, int32_t head_dim,
                           const int32_t *block_src, const int32_t *block_dst,
                           int32_t num_pairs, void *stream);

/*
 * pkv_workspace_size -- bytes of device workspace pkv_paged_decode_attention
 * needs for this geometry on the CURRENT CUDA device (the size depends on its
 * SM count). n_query_per_seq may be up to 64 / (num_q_heads / num_kv_heads)
 * (the max_q_len of pkv_paged_decode_attention_varlen). Returns 0 if the geometry is unsupported or no device is usable.
 * The workspace holds the split-K partial states (m, l, acc) that the merge
 * step combines, per (sequence, kv-head group) the cells holding its first and
 * last partial, and a 4-byte device error word at offset 0 (see
 * pkv_paged_decode_attention).
 */
size_t pkv_workspace_size(int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim);

/*
 * pkv_paged_decode_attention -- decode attention over the paged pool.
 *
 * Passages: "ML Interview Prep, Lesson 13" section 3.5 (the kernel follows the
 * block table and reads keys and values one block at a time) and section 3.3
 * (grouped-query heads); "07 -- Inference" section 5.1 (online softmax, exact)
 * and section 5.3 (FlashDecoding: split the KV sequence into chunks handled by
 * separate thread blocks, each giving a partial (m, l, acc), merged with the
 * online-softmax rescaling rule); "LLM Serving: Continuous Batching &
 * PagedAttention", speculative decoding mechanics (the target scores all draft
 * positions in one pass under a causal mask).
 *
 * For every sequence s, query j in [0, n_query_per_seq), query head qh:
 *     T   = context_lens[s]          (tokens INCLUDING this step's nq new ones)
 *     lim = T - n_query_per_seq + j  (last position query j may see)
 *     x_t = scale * <q[s*nq+j][qh], K_s[t][qh/G]>   for t in [0, lim]
 *     out[s*nq+j][qh] = sum_t softmax(x)_t * V_s[t][qh/G]
 * with G = num_q_heads / num_kv_heads and K_s[t] the row at
 * block_tables[s][t/16], offset t%16. A row with lim < 0 is all zeros.
 * Accumulation is fp32 from bf16 inputs; the result matches the fp64
 * definition within |err| <= 2e-3 + 1e-2*|ref| (bf16 output) and is
 * deterministic for a given device and input (no atomics in any reduction).
 *
 *   q              device, bf16 [num_seqs*n_query_per_seq][num_q_heads][head_dim],
 *                  16-byte aligned; row s*nq+j is query j of sequence s.
 *   k_cache,v_cache device pool as described above, 16-byte aligned.
 *   num_blocks     pool size in blocks, 1 .. 2^31-1. A table entry outside
 *                  [0, num_blocks) reads zeros (no fault) and ORs 8 into the
 *                  workspace error word.
 *   block_tables   device, int32 [num_seqs][max_blocks_per_seq]; entries at and
 *                  past ceil(T/16) are never read (any value, e.g. -1).
 *   context_lens   device, int32 [num_seqs]; a value above 16*max_blocks_per_seq
 *                  is clamped to it, a negative value counts as 0.
 *   n_query_per_seq 1..4; num_q_heads % num_kv_heads == 0;
 *                  (num_q_heads/num_kv_heads) * n_query_per_seq <= 64.
 *   head_dim       64 or 128.
 *   scale          usually 1/sqrt(head_dim).
 *   out            device, [num_seqs*n_query_per_seq][num_q_heads][head_dim] of
 *                  out_dtype (PKV_BF16 rounds to nearest even), 16-byte aligned.
 *   workspace      device, >= pkv_workspace_size(...) bytes, 256-byte aligned,
 *                  ZERO-FILLED before its first use; every call leaves the
 *                  counters it uses at zero again, so one workspace serves any
 *                  sequence of calls (of any shapes that fit it). It holds a
 *                  256-byte header, the merge's piece records and the split-K
 *                  partial states (m, l, acc) per cell (a fixed slice of the
 *                  batch's blocks). Its first 4
 *                  bytes are a sticky device error word: a kernel that gives up
 *                  on a wait (never expected; a bounded wait guards against a
 *                  hang) ORs a nonzero code there and returns early; zero the
 *                  workspace again after such a call. Calls sharing a
 *                  workspace must be ordered on one stream (or otherwise
 *                  serialised).
 *   num_seqs == 0  is a no-op returning PKV_OK.
 */
pkv_status pkv_paged_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                                      int64_t num_blocks, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      int32_t num_seqs, int32_t n_query_per_seq,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      float scale, void *out, int32_t out_dtype, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * pkv_paged_decode_attention_cascade -- pkv_paged_decode_attention for a batch
 * whose sequences share prefixes, with each shared prefix attended once per
 * group of sequences instead of once per sequence.
 *
 * Passages: "ML Interview Prep, Lesson 13" section 3.5 "Sharing" (parallel
 * samples and a common system prompt share physical blocks) and "07 --
 * Inference" section 5.3 (a partial (m, l, acc) over any token range merges
 * exactly with the others by the online-softmax rescaling rule). The result is
 * the same function as pkv_paged_decode_attention on the same inputs (within
 * the same tolerance); only the work differs.
 *
 *   prefix_groups   device int32 [num_groups][3]: (first sequence, number of
 *                   sequences, prefix blocks P). A group's sequences are
 *                   consecutive in the batch, groups ascend by first sequence and
 *                   do not overlap, and every member's block-table row starts with
 *                   the same P physical ids (its first P blocks are the shared
 *                   prefix); P <= max_blocks_per_seq.
 *   max_group_seqs  host bound on the sequences of any group (it sizes the grid
 *                   of the prefix pass).
 *   workspace       >= pkv_workspace_size_cascade(...) bytes (zero-filled before
 *                   first use, as for pkv_paged_decode_attention).
 * A member whose query rows do not all see the whole prefix (16*P > T - nq) or
 * whose context is the prefix alone is attended without the cascade; a group
 * outside the batch or the tables is skipped and ORs 32 into the workspace
 * error word. num_groups == 0 is the plain call. bf16 pools only.
 *
 * How: a prefix pass (one kv head per CTA; 128 score rows = 128/G members'
 * queries per row tile) streams each group's prefix blocks once per row tile
 * and leaves every member row's partial (m, l, acc); the main pass streams only
 * the members' own blocks; the merge starts each member row from its prefix
 * partial.
 */
size_t pkv_workspace_size_cascade(int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim);

/*
 * pkv_cascade_pays -- host planner: 1 if pkv_paged_decode_attention_cascade is
 * expected to beat pkv_paged_decode_attention for this batch, 0 if not, -1 for
 * invalid input (a negative count, a NULL array with a nonzero count, a group
 * outside the batch, non-positive head sizes).
 *
 * Passage: "ML Interview Prep, Lesson 13" section 3.5 "Sharing" (shared blocks
 * are read by every sharer). The plain call reads every member's copy of the
 * shared prefix; after the first, those reads mostly hit L2, so they cost
 * little while they are few, and bound the kernel once they are not. The
 * cascade avoids them for a roughly fixed price (a second launch, its prefix
 * pass, one partial fold per member row). The rule, with repeated prefix tokens
 * = the sum over groups of (members whose context extends past the prefix - 1)
 * * 16 * P and unique tokens = all context tokens minus the repeated ones:
 * repeated >= unique, and the repeated tokens' K and V (num_kv_heads * head_dim
 * bf16 each) weigh at least 1.5 GB. Measured on GB300 (256 sequences, 8 kv
 * heads of 128 dims): a 4,096-token prompt with suffixes under 512 tokens runs
 * 1.7x faster with the cascade; 512-token prompts and the 70B-shaped mix run
 * faster without.
 *
 *   context_lens   host int32 [num_seqs], as the attention call's
 *   prefix_groups  host int32 [num_groups][3], as the cascade call's
 */
int32_t pkv_cascade_pays(const int32_t *context_lens, int32_t num_seqs,
                         const int32_t *prefix_groups, int32_t num_groups,
                         int32_t num_kv_heads, int32_t head_dim);

pkv_status pkv_paged_decode_attention_cascade(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
    int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, float scale, const int32_t *prefix_groups, int32_t num_groups,
    int32_t max_group_seqs, void *out, int32_t out_dtype, void *workspace,
    size_t workspace_bytes, void *stream);

/*
 * pkv_paged_decode_attention_varlen -- per-sequence query counts, optional
 * tree masks, optional shared block-table rows.
 *
 * Passages: "Chapter 18" section 18.1.2 (tree-based speculative decoding: all
 * candidate nodes are scored in one pass, each seeing its own ancestors) and
 * section 18.2 (variable-length attention, no padding); "07 -- Inference"
 * section 2.4 (chunked prefill: attending a prompt chunk by chunk gives the
 * one-pass result).
 *
 * Sequence s owns query rows q_start[s] .. q_start[s+1]-1 of q and out
 * (q_len_s of them, 0 <= q_len_s <= max_q_len) and T_s = context_lens[s]
 * tokens read through block-table row table_row[s] (or s when table_row is
 * NULL). Without masks query j sees positions 0 .. T_s - q_len_s + j (causal
 * over the sequence's last q_len_s tokens). With masks the last
 * W_s = tree_len[s] (0..32) positions form a window: query row r sees every
 * position before T_s - W_s and window position i iff bit i of tree_mask[r].
 * A row that sees nothing is zeros.
 *
 *   q, out          [total_q][num_q_heads][head_dim] (bf16 / out_dtype).
 *   block_tables    device int32 [num_table_rows][max_blocks_per_seq].
 *   table_row       device int32 [num_seqs] or NULL (then num_table_rows >= num_seqs).
 *   context_lens    device int32 [num_seqs].
 *   q_start         device int32 [num_seqs + 1], nondecreasing, q_start[num_seqs] <= total_q.
 *   tree_mask       device uint32 [total_q] or NULL; tree_len device int32
 *                   [num_seqs], given together with tree_mask.
 *   max_q_len       >= 1 with (num_q_heads/num_kv_heads) * max_q_len <= 64 (the
 *                   kernel's score rows per kv head; unlike the fixed-count call,
 *                   more than 4 is allowed); the workspace is
 *                   pkv_workspace_size(num_seqs, max_q_len, ...).
 * Device values that break these rules (rows outside [0, total_q), more than
 * max_q_len rows, a table row outside the tables) give that sequence no output
 * and OR 16 into the workspace error word. Other arguments and errors as
 * pkv_paged_decode_attention. Longer query runs go through pkv_split_queries.
 */
pkv_status pkv_paged_decode_attention_varlen(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    const int32_t *block_tables, int32_t max_blocks_per_seq, int32_t num_table_rows,
    const int32_t *table_row, const int32_t *context_lens, const int32_t *q_start,
    const uint32_t *tree_mask, const int32_t *tree_len, int32_t num_seqs, int32_t max_q_len,
    int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
    void *out, int32_t out_dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * pkv_split_queries -- host arrays in and out: cut every sequence's query rows
 * into runs of at most max_rows rows ("virtual sequences") for
 * pkv_paged_decode_attention_varlen, so prefill chunks and large candidate
 * trees fit its row limit. Run k of sequence s covers rows
 * q_start[s] + k*max_rows .. (exclusive) min(q_start[s+1], ...), reads table row
 * s, and keeps every row's visibility: without tree_len its context length is
 * T_s - q_len_s + (its end row - q_start[s]) (causal); with tree_len its context
 * is T_s and its window tree_len[s] (the rows keep their mask words).
 * Sequences with no query row produce no run. Writes v_q_start[0..V],
 * v_context_lens[0..V-1], v_table_row[0..V-1] and (with tree_len) v_tree_len;
 * *num_virtual = V. PKV_ERR_RANGE (and *num_virtual = the V needed) when
 * capacity < V; PKV_ERR_SHAPE for negative counts or max_rows < 1.
 */
pkv_status pkv_split_queries(const int32_t *q_start, const int32_t *context_lens,
                             const int32_t *tree_len, int32_t num_seqs, int32_t max_rows,
                             int32_t *v_q_start, int32_t *v_context_lens, int32_t *v_tree_len,
                             int32_t *v_table_row, int32_t capacity, int32_t *num_virtual);

/*
 * FP8 (E4M3) pools -- the same two operations on a cache stored in 8 bits.
 *
 * Passages: "ML Interview Prep, Lesson 13" section 3.7 (an fp8 KV cache stores
 * keys and values in 8 bits while the matmuls run at 16 bits: twice the tokens
 * in memory, half the KV bytes read per step) and "07 -- Inference" section
 * 4.3 (E4M3 for inference, largest magnitude 448; per-tensor, per-channel or
 * per-block scales). Here each kv head h has one float scale for K and one for
 * V: a stored code c stands for e4m3(c) * scale[h].
 *
 * Pools: k_cache, v_cache are uint8 [num_blocks][16][num_kv_heads][head_dim]
 * of E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; S.1111.111 is NaN), 16-byte aligned. k_scale, v_scale: device
 * float [num_kv_heads], 4-byte aligned, finite and nonzero.
 *
 * pkv_kv_append_fp8 -- for every i with slot_mapping[i] >= 0 and every head h:
 *     k_cache[slot/16][slot%16][h][d] = E4M3(k_new[i][h][d] / k_scale[h])
 * (the quotient in float, round to nearest; then the nearest E4M3 value, ties
 * to even, magnitudes beyond 448 saturate to 448, NaN stays NaN); V likewise.
 * Bit-exact. Other arguments, limits and errors as pkv_kv_append (head_dim a
 * multiple of 8; caches 8-byte aligned at least).
 *
 * pkv_paged_decode_attention_fp8 -- pkv_paged_decode_attention over E4M3
 * pools: K_s[t] = e4m3(code) * k_scale[h], V likewise, everything else as
 * there (causality, GQA, output layout and dtype, workspace, errors; the
 * workspace size is pkv_workspace_size's). head_dim must be 128
 * (PKV_ERR_UNSUPPORTED otherwise). The kernels dequantise exactly to fp16 and
 * multiply in fp16 with fp32 accumulation: q is rounded to fp16 (|q| must stay
 * below 65504) and the softmax weights P are rounded to fp16 (relative error
 * <= 2^-12) before the PV product. Against the fp64 definition on the
 * dequantised pool the result is within |err| <= 2e-3 + 1e-2*|ref| for the
 * bf16 output.
 */
pkv_status pkv_kv_append_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                             int64_t n_new, void *k_cache, void *v_cache, int64_t num_blocks,
                             int32_t num_kv_heads, int32_t head_dim, const float *k_scale,
                             const float *v_scale, void *stream);

pkv_status pkv_paged_decode_attention_fp8(const void *q, const void *k_cache, const void *v_cache,
                                          int64_t num_blocks, const float *k_scale,
                                          const float *v_scale, const int32_t *block_tables,
                                          int32_t max_blocks_per_seq,
                                          const int32_t *context_lens, int32_t num_seqs,
                                          int32_t n_query_per_seq, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim, float scale,
                                          void *out, int32_t out_dtype, void *workspace,
                                          size_t workspace_bytes, void *stream);

/*
 * pkv_paged_decode_attention_static -- pkv_paged_decode_attention without a
 * caller-provided workspace, for callers that cannot allocate device memory.
 *
 * The pages have no counterpart: this is a packaging variant, not a step of
 * the method. Some callers of this library cannot call cudaMalloc (or any
 * allocator): plugins hosted by a framework that owns all device memory and
 * hands its plugins no allocator, and serving loops whose device memory is
 * fixed when they start (cudaMalloc/cudaFree synchronise the device and
 * fragment the pool, so such loops forbid them after start-up). This entry point
 * allocates nothing -- no cudaMalloc, cudaFree or allocating library routine --
 * and the caller still passes every input and output buffer.
 *
 * Arguments, results and errors are those of pkv_paged_decode_attention
 * without `workspace`/`workspace_bytes`: the same host checks run in the same
 * order and return the same status. The scratch instead lives in one
 * static device array of 32 MiB (32 * 2^20 bytes), which every GPU that loads
 * the library's module holding it keeps until the process exits (with CUDA's
 * default lazy module loading: from this entry point's first call on that
 * GPU). A call whose plan (sized as the workspace call would size it, tuning
 * options included) needs more than 32 MiB of scratch returns
 * PKV_ERR_WORKSPACE before anything is enqueued; on a 152-SM GB300 a
 * geometry with up to 32 query rows per kv head needs at most ~21 MiB plus 8
 * bytes per (sequence, group of up to 8 kv heads), one with 33 to 64 rows up
 * to ~42 MiB (those above 32 MiB take the workspace call).
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it; make that
 * first call before any stream capture. Each call clears the array's
 * 256-byte header (device error word, work counters; one cudaMemsetAsync on
 * `stream`) before its kernels; they write every other byte they read. All calls share the one array and
 * it keeps the last call's contents: calls that overlap on the GPU (on
 * different streams, or from several threads) race on it and give
 * unspecified results. Serialise them, e.g. on one stream.
 *
 * Device-side problems (a block-table entry outside [0, num_blocks), a bounded
 * wait that gave up) are recorded in the array's error word, as in a caller's
 * workspace: read it with pkv_static_error_word after the call and before the
 * next static call, which clears it.
 */
pkv_status pkv_paged_decode_attention_static(const void *q, const void *k_cache,
                                             const void *v_cache, int64_t num_blocks,
                                             const int32_t *block_tables,
                                             int32_t max_blocks_per_seq,
                                             const int32_t *context_lens, int32_t num_seqs,
                                             int32_t n_query_per_seq, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t head_dim, float scale,
                                             void *out, int32_t out_dtype, void *stream);

/*
 * pkv_static_error_word -- the device error word of the static scratch that
 * pkv_paged_decode_attention_static uses on the current device: the bits a
 * workspace's first 4 bytes hold after pkv_paged_decode_attention (8 = a
 * block-table entry outside [0, num_blocks), read as zeros; 1, 2, 4 = a
 * bounded wait gave up).
 *
 * No counterpart on the pages either: it lets a caller that cannot allocate
 * see device-side errors of its static calls. Enqueues one 4-byte
 * device-to-host copy on `stream` (after the stream's earlier work) into
 * `host_word` and waits for the stream; allocates nothing. PKV_ERR_NULL for a
 * NULL `host_word`, PKV_ERR_CUDA if the copy fails. The word is cleared by
 * the next static call.
 */
pkv_status pkv_static_error_word(uint32_t *host_word, void *stream);

/*
 * pkv_step_arena_layout -- byte layout of one decode step's inputs in a single
 * buffer: q, k_new, v_new, slot_mapping, block_tables, context_lens, in that
 * order, each at a 256-byte aligned offset, with the shapes and types of
 * pkv_kv_append (n_new = num_seqs * n_query_per_seq new tokens, one per query
 * row) and pkv_paged_decode_attention. Writes the six offsets to `offsets`
 * (may be NULL) and returns the total bytes: 0 for num_seqs == 0, an
 * unsupported geometry (pkv_paged_decode_attention's rules) or
 * max_blocks_per_seq < 1.
 */
size_t pkv_step_arena_layout(int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t max_blocks_per_seq,
                             size_t offsets[6]);

/*
 * pkv_decode_step -- one decode step on device buffers: the step's new K/V rows
 * are appended (pkv_kv_append, or pkv_kv_append_fp8 with scales), then the
 * attention runs over the updated pool (pkv_paged_decode_attention, or
 * pkv_paged_decode_attention_fp8), both on `stream`.
 *
 * Passage: "ML Interview Prep, Lesson 13" section 3.5 and "LLM Inference Serving"
 * (block-table pseudo-code): each decode step writes the new token's K/V into
 * its slot, then attends over the sequence's blocks.
 *
 *   q, block_tables, context_lens, out, workspace: as pkv_paged_decode_attention
 *   k_new, v_new   device [num_seqs * n_query_per_seq, num_kv_heads, head_dim]
 *                  bf16 (one new row per query row, in row order)
 *   slot_mapping   device int64 [num_seqs * n_query_per_seq], as pkv_kv_append
 *   k_scale, v_scale  device float [num_kv_heads]: E4M3 pools (head_dim 128);
 *                  both NULL: bf16 pools; one alone: PKV_ERR_NULL
 *
 * Same results, bit for bit, as the two calls in turn. The difference is
 * timing: the append writes only the pools, and q, the tables and the lengths
 * must be complete when the call's work starts on `stream`, so the attention
 * kernel reads the lengths and tables and plans its work while the append
 * still runs, and waits for the append only before its first read of the pool.
 * q, the tables, the lengths and out must not overlap the pools.
 *
 * Errors: every argument check of both calls (and the workspace size and
 * alignment the attention's plan needs) runs before anything is enqueued; on an
 * error nothing is enqueued and the pools are unchanged. PKV_ERR_CUDA if a
 * launch fails (the append may then have run).
 */
pkv_status pkv_decode_step(const void *q, const void *k_new, const void *v_new,
                           const int64_t *slot_mapping, void *k_cache, void *v_cache,
                           int64_t num_blocks, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, float scale, void *out,
                           int32_t out_dtype, void *workspace, size_t workspace_bytes,
                           const float *k_scale, const float *v_scale, void *stream);

/*
 * pkv_decode_step_host -- one decode step from host memory: the step's inputs
 * cross to the device, the new tokens are appended, the attention runs, and
 * its output comes back to the host. Enqueued on `stream` in this order:
 *   1. one host-to-device copy of `host_arena` (pkv_step_arena_layout's
 *      layout, arena_bytes long) into `device_arena`;
 *   2. pkv_kv_append of the arena's k_new / v_new rows at its slot_mapping;
 *   3. pkv_paged_decode_attention over the arena's q, block_tables and
 *      context_lens into `out_device`;
 *   4. one device-to-host copy of `out_device` into `out_host`.
 * The step is the pair of calls a decode loop makes ("LLM Serving: Continuous
 * Batching & PagedAttention": each iteration writes the new token's K/V into
 * its block slot, then attends over the block table); the pages give no host
 * interface, so this one is the plainest: one copy each way.
 *
 *   host_arena     host, arena_bytes >= pkv_step_arena_layout(...) bytes; page-
 *                  locked (cudaHostAlloc / cudaHostRegister) for the copy to be
 *                  asynchronous; must stay unchanged until the copy has run.
 *   device_arena   device, same size, 256-byte aligned; the library reads it
 *                  only through steps 1-3.
 *   out_device     device output of step 3 (pkv_paged_decode_attention's `out`).
 *   out_host       host, num_seqs*n_query_per_seq*num_q_heads*head_dim elements
 *                  of out_dtype; valid once the stream has reached step 4.
 *   other arguments as pkv_kv_append and pkv_paged_decode_attention.
 * Errors: those of the two calls (checked before anything is enqueued where
 * they do not depend on device data), PKV_ERR_NULL for a missing arena or host
 * output, PKV_ERR_WORKSPACE if arena_bytes is below the layout's size,
 * PKV_ERR_CUDA if a copy cannot be enqueued.
 */
pkv_status pkv_decode_step_host(const void *host_arena, void *device_arena, size_t arena_bytes,
                                void *k_cache, void *v_cache, int64_t num_blocks,
                                int32_t max_blocks_per_seq, int32_t num_seqs,
                                int32_t n_query_per_seq, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim, float scale,
                                void *out_device, void *out_host, int32_t out_dtype,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * pkv_decode_step_host_pipelined -- pkv_decode_step_host with its phases on
 * three streams, so that in a loop over steps the copies of a step run while
 * the kernels of its neighbours stream the pool (the copy engines move host
 * memory while the SMs read HBM). A buffer slot is (host_arena, device_arena,
 * out_device, out_host) with three events of its own (cudaEvent_t, e.g. created
 * with cudaEventDisableTiming; an event never recorded is no wait):
 *   upload_stream:   waits `computed` (the slot's previous step has read its
 *                    device arena), copies host_arena -> device_arena, records
 *                    `uploaded`;
 *   compute_stream:  waits `uploaded` and `downloaded` (the slot's previous
 *                    output has left out_device), runs pkv_kv_append and
 *                    pkv_paged_decode_attention as pkv_decode_step_host does,
 *                    records `computed`;
 *   download_stream: waits `computed`, copies out_device -> out_host, records
 *                    `downloaded`.
 * With two slots used in turn, step n+1's upload and step n-1's download
 * overlap step n's kernels, and the kernels of consecutive steps stay in order
 * on compute_stream (one workspace serves them all). The three streams may be
 * the same stream (then it is pkv_decode_step_host). out_host is valid once
 * `downloaded` has completed. With k_scale and v_scale (device float [Hkv]) the
 * pools are E4M3 and the step calls pkv_kv_append_fp8 and
 * pkv_paged_decode_attention_fp8 (head_dim 128); both NULL: bf16 pools.
 * Arguments and errors otherwise as pkv_decode_step_host; PKV_ERR_NULL for a
 * missing event or only one scale.
 */
pkv_status pkv_decode_step_host_pipelined(
    const void *host_arena, void *device_arena, size_t arena_bytes, void *k_cache, void *v_cache,
    int64_t num_blocks, int32_t max_blocks_per_seq, int32_t num_seqs, int32_t n_query_per_seq,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale, void *out_device,
    void *out_host, int32_t out_dtype, void *workspace, size_t workspace_bytes,
    const float *k_scale, const float *v_scale, void *upload_stream, void *compute_stream,
    void *download_stream, void *uploaded, void *computed, void *downloaded);

/* Text for a status code (static storage; never NULL). */
const char *pkv_status_string(int32_t status);

/*
 * Tuning options (process-wide, not thread-safe against concurrent calls):
 *   PKV_OPT_NUM_CTAS     persistent grid size of the attention kernel; 0 = one
 *                        CTA per SM (default). Any value >= 1 gives the same
 *                        result up to fp32 rounding order.
 *   PKV_OPT_STAGES       pipeline depth (K/V stages in shared memory); 0 = as
 *                        many as fit (default), else clamped to [2, 8].
 *   PKV_OPT_HEADS_PER_CTA cap on the kv heads one CTA streams together (each
 *                        stage holds one 16-token block of that many heads);
 *                        0 = up to 8 (default).
 *   PKV_OPT_TMA_BOX      0 = one TMA box per block when the driver accepts the
 *                        tensor map, else one per (head, 64-column half) tile
 *                        (default); 1 = always per tile; 2 = always per block
 *                        (PKV_ERR_UNSUPPORTED if the driver refuses the map).
 *   PKV_OPT_TAIL         0 or 1 = no dynamic tail (default); n >= 2 = the last
 *                        1/n of the work goes out as dynamically claimed
 *                        tickets to the CTAs that finish their static share
 *                        first. Ticket boundaries depend on the sizes only, so
 *                        results stay deterministic.
 *   PKV_OPT_PACE         0 = off (default); 1 = pace the attention kernel's
 *                        static chunks: a CTA whose share of its chunk runs
 *                        ahead of the grid's share of all work (one progress
 *                        counter in the workspace header) keeps one stage fewer
 *                        in flight, so where HBM is saturated the SMs that
 *                        stream slower get more of it and the chunks end closer
 *                        together (measured on GB300: within 1 % on HBM-bound
 *                        batches, slower where L2 serves shared blocks or the
 *                        math bounds the kernel). Timing only: results are
 *                        bit-identical with pacing on or off.
 *   PKV_OPT_PACE_MARGIN  the lead allowed before pacing, in 1/10000 of the
 *                        work; 0..10000, default 0.
 *   PKV_OPT_MATH         0 = tensor cores (default); 1 = the same
 *                        pipeline with the scores and P.V on the CUDA cores
 *                        (fp32 FMA, shuffle reductions), kept as the reference
 *                        point for that choice. It applies to
 *                        pkv_paged_decode_attention with head_dim 128 only
 *                        (the other entry points always use tensor cores).
 *   PKV_OPT_UMMA         0 = the warp-level mma.sync kernels for every shape
 *                        (default); 1 = kv heads with 17 to 64 query rows on bf16
 *                        pools with head_dim 128 use the fifth-generation tensor
 *                        cores instead (tcgen05: MMAs from shared memory into
 *                        tensor memory; measured slower on this KV layout, kept
 *                        for comparison). The cascade always runs on mma.sync.
 *   PKV_OPT_PREFETCH     tcgen05 kernel: 0 = prefetch the K/V tiles into L2 64
 *                        blocks ahead of their loads into shared memory
 *                        (default); n >= 1 = n - 1 blocks ahead (1 = none).
 * All settings give the same result up to fp32 rounding order.
 * Returns the previous value, or -1 for an unknown option or an invalid value.
 */
enum { PKV_OPT_NUM_CTAS = 1, PKV_OPT_STAGES = 2, PKV_OPT_HEADS_PER_CTA = 3, PKV_OPT_TMA_BOX = 4,
       PKV_OPT_TAIL = 5, PKV_OPT_PACE = 6, PKV_OPT_PACE_MARGIN = 7, PKV_OPT_MATH = 8,
       PKV_OPT_UMMA = 9, PKV_OPT_PREFETCH = 10 };
int32_t pkv_set_option(int32_t option, int32_t value);

/*
 * pkv_set_profiling_events -- measurement hook (process-wide). When both are
 * non-NULL, every later pkv_paged_decode_attention call records `before` (a
 * cudaEvent_t) on its stream just before its main attention kernel and `after`
 * just after it, before the merge kernel; cudaEventElapsedTime of the pair is
 * that kernel's device time. NULL, NULL turns the hook off. The events stay
 * owned by the caller and must belong to the stream's device.
 */
void pkv_set_profiling_events(void *before, void *after);

/*
 * pkv_set_trace_buffer -- per-CTA timeline of the attention kernel (process-
 * wide; NULL turns it off). When set, every later pkv_paged_decode_attention
 * call whose grid fits writes, for each CTA c, 16 uint64 words at
 * device_buffer[16c ..]: [0] entry, [1] first K/V copy issued, [2] first stage
 * consumed, [3] last copy issued, [4] last stage consumed (ns of the GPU's
 * global timer), [5] 16-token blocks streamed, [6] sequence segments
 * started, [7] SM id; the counters add to the existing values; [8..15]
 * are reserved. The caller zeroes the buffer before a call; a
 * buffer smaller than grid*128 bytes disables the trace.
 */
void pkv_set_trace_buffer(void *device_buffer, size_t bytes);

/* Library version as an integer (major*10000 + minor*100 + patch). */
int32_t pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
