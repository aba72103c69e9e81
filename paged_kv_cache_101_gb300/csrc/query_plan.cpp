// query_plan.cpp -- host-side planners (see include/pkv.h): the split of long
// query runs into virtual sequences for pkv_paged_decode_attention_varlen, and the
// rule that picks the shared-prefix cascade or the plain call.
//
// The attention kernel holds at most 64 score rows per kv head (G * q_len), so a
// prefill chunk or a large candidate tree is cut into runs of at most max_rows
// query rows. A causal run keeps its rows' causal limits by ending its context
// where its last row sits ("07 -- Inference" section 2.4: chunked prefill gives
// the one-pass result); a masked run keeps the whole context and the sequence's
// window, its rows keeping their own mask words. Every run reads its source
// sequence's block-table row.
#include <stdint.h>

#include "pkv.h"

namespace {
// The cascade pays once the repeated prefix bytes reach the step's unique bytes and
// 1.5 GB: below that the plain call re-reads the prefix from L2 faster than the
// cascade's prefix pass and member seeding cost (measured on GB300, 256 sequences
// with 8 kv heads of 128 dims: prefixes of 512 to 4,096 tokens, suffixes up to
// 4,096 tokens).
constexpr double kCascadeMinRepeatedBytes = 1.5e9;
}  // namespace

extern "C" pkv_status pkv_split_queries(const int32_t *q_start, const int32_t *context_lens,
                                        const int32_t *tree_len, int32_t num_seqs,
                                        int32_t max_rows, int32_t *v_q_start,
                                        int32_t *v_context_lens, int32_t *v_tree_len,
                                        int32_t *v_table_row, int32_t capacity,
                                        int32_t *num_virtual)
{
    if (!num_virtual)
        return PKV_ERR_NULL;
    *num_virtual = 0;
    if (num_seqs < 0 || max_rows < 1 || capacity < 0)
        return PKV_ERR_SHAPE;
    if (num_seqs > 0 && (!q_start || !context_lens))
        return PKV_ERR_NULL;
    int64_t need = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int64_t ql = int64_t(q_start[s + 1]) - q_start[s];
        if (ql < 0 || q_start[s] < 0)
            return PKV_ERR_SHAPE;
        if (tree_len && (tree_len[s] < 0 || tree_len[s] > 32))
            return PKV_ERR_RANGE;
        need += (ql + max_rows - 1) / max_rows;
    }
    if (need > INT32_MAX - 1)
        return PKV_ERR_RANGE;
    if (need > capacity) {
        *num_virtual = int32_t(need);
        return PKV_ERR_RANGE;
    }
    if (need > 0 && (!v_q_start || !v_context_lens || !v_table_row || (tree_len && !v_tree_len)))
        return PKV_ERR_NULL;
    int32_t v = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t a = q_start[s], ql = q_start[s + 1] - q_start[s];
        for (int32_t r = 0; r < ql; r += max_rows) {
            const int32_t end = r + max_rows < ql ? r + max_rows : ql;
            v_q_start[v] = a + r;
            v_table_row[v] = s;
            if (tree_len) {
                v_context_lens[v] = context_lens[s];
                v_tree_len[v] = tree_len[s];
            } else {
                v_context_lens[v] = context_lens[s] - ql + end;  // the run's last row's position + 1
            }
            ++v;
            v_q_start[v] = a + end;
        }
    }
    *num_virtual = v;
    return PKV_OK;
}

// Whether the shared-prefix cascade is expected to beat the plain call. The
// plain call streams every member's copy of its group's prefix: the first copy
// from HBM, the others mostly from L2 while the prefix stays resident. Those
// repeated prefix reads cost L2 bandwidth and, once they rival the step's unique
// bytes, they bound the plain kernel; the cascade reads each prefix once per row
// tile instead, for the price of a second launch, its prefix pass and one
// partial fold per member row. So the rule compares the repeated prefix bytes
// with the unique bytes and with that fixed price.
extern "C" int32_t pkv_cascade_pays(const int32_t *context_lens, int32_t num_seqs,
                                    const int32_t *prefix_groups, int32_t num_groups,
                                    int32_t num_kv_heads, int32_t head_dim)
{
    if (num_seqs < 0 || num_groups < 0 || num_kv_heads < 1 || head_dim < 1)
        return -1;
    if (num_seqs == 0 || num_groups == 0)
        return 0;
    if (!context_lens || !prefix_groups)
        return -1;
    int64_t total = 0;
    for (int32_t s = 0; s < num_seqs; ++s)
        total += context_lens[s] > 0 ? context_lens[s] : 0;
    int64_t repeated = 0;
    for (int32_t g = 0; g < num_groups; ++g) {
        const int32_t f = prefix_groups[3 * g], cnt = prefix_groups[3 * g + 1];
        const int32_t P = prefix_groups[3 * g + 2];
        if (f < 0 || cnt < 0 || P < 0 || int64_t(f) + cnt > num_seqs)
            return -1;
        // members that attend the prefix through the cascade: those whose context
        // holds more than the prefix (the others fall back to the plain path)
        int64_t members = 0;
        for (int32_t s = f; s < f + cnt; ++s)
            members += int64_t(context_lens[s]) > int64_t(16) * P ? 1 : 0;
        if (members > 1)
            repeated += (members - 1) * int64_t(16) * P;
    }
    const int64_t unique = total - repeated;
    const double token_bytes = 2.0 * 2.0 * double(num_kv_heads) * double(head_dim);  // K + V, bf16
    const double rep_bytes = double(repeated) * token_bytes;
    return repeated >= unique && rep_bytes >= kCascadeMinRepeatedBytes ? 1 : 0;
}
