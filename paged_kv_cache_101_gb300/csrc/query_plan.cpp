// query_plan.cpp -- host-side split of long query runs into virtual sequences
// for pkv_paged_decode_attention_varlen (see include/pkv.h).
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
