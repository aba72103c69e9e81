// pkv_cells.cuh -- the work partition shared by the attention kernels: the flat
// unit space of a call cut into cells (one contiguous chunk per CTA of the
// persistent grid, optionally followed by dynamically claimed tickets), and the
// per-sequence view of the inputs (rows, table row, mask window, cascade prefix).
#pragma once

#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {

// Stage flags. F_FIRST / F_LAST: the first / last stage of a segment (a
// sequence's blocks inside one cell); F_DIRECT: that segment is the whole sequence
// (finished in place); F_END: no more work. F_PREFIX: a stage of the cascade's
// prefix pass; F_PRE: the first stage of a cascade member's own blocks, whose
// running state starts from its prefix partial.
enum : int32_t { F_FIRST = 1, F_LAST = 2, F_DIRECT = 4, F_END = 8, F_PREFIX = 16, F_PRE = 32 };

// The fixed partition of the flat unit space [0, F): cells 0..G-1 split
// [0, F1) evenly (cell c is CTA c's chunk); cells G..G+NT-1 split [F1, F) evenly
// (tickets, claimed dynamically).
struct Cells {
    int64_t F, F1, F2;
    int32_t G, NT;

    __device__ __forceinline__ int64_t start(int64_t k) const
    {
        return k <= G ? k * F1 / G : F1 + (k - G) * F2 / NT;
    }
    __device__ __forceinline__ bool empty(int64_t k) const { return start(k) == start(k + 1); }
    // the cell holding unit f (0 <= f < F)
    __device__ __forceinline__ int64_t cell_of(int64_t f) const
    {
        if (f < F1)
            return ((f + 1) * G + F1 - 1) / F1 - 1;
        return G + ((f - F1 + 1) * NT + F2 - 1) / F2 - 1;
    }
};

// The cells of a call: G static chunks, then up to tickets_max tickets over the
// last F / ticket_div units. A function of the sizes only (the merge kernel
// rebuilds the same cells).
__device__ __forceinline__ Cells make_cells(const DecodeParams &p, int nb_total, int grid)
{
    Cells C;
    C.F = int64_t(p.n_hg) * nb_total;
    C.G = grid;
    C.NT = 0;
    C.F2 = 0;
    if (p.tickets_max > 0 && p.ticket_div > 0) {
        const int64_t f2 = C.F / p.ticket_div;
        const int64_t nt = f2 / (p.ticket_units > 0 ? p.ticket_units : 1);
        if (nt > 0) {
            C.NT = int(nt < p.tickets_max ? nt : p.tickets_max);
            C.F2 = f2;
        }
    }
    C.F1 = C.F - C.F2;
    return C;
}

__device__ __forceinline__ int seq_tokens(const DecodeParams &p, int s)
{
    int T = __ldg(p.context_lens + s);
    T = T < 0 ? 0 : T;
    const int cap = p.MB * kBlockSize;
    return T > cap ? cap : T;
}

// Per-sequence view of the inputs. Fixed query count: rows s*nq .. +nq, block
// table row s, causal. Variable counts (q_start): rows q_start[s] ..
// q_start[s+1]-1 (at most nq), table row table_row[s] (or s), and with tree
// masks a window of tree_len[s] positions. Inconsistent device values (rows
// outside [0, total_q), more rows than nq, a table row outside the tables)
// leave the sequence without queries and set kErrBadQuery.
struct SeqInfo {
    int T;   // tokens (clamped to the table)
    int nb;  // blocks to stream (0 if the sequence has no query rows)
    int q0;  // first query row
    int ql;  // query rows
    int W;   // mask window (causal: ql)
    int tr;  // block-table row
    int b0;  // first block streamed: a cascade member's prefix is attended apart
};

// Cascade: the group holding sequence s (groups ascending by first sequence),
// or -1. Each row of pre-computed groups is (first sequence, sequences, blocks).
__device__ __forceinline__ int group_of(const DecodeParams &p, int s)
{
    int lo = 0, hi = p.num_groups - 1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        const int f = __ldg(p.prefix_groups + 3 * mid);
        if (s < f) {
            hi = mid - 1;
        } else if (s >= f + __ldg(p.prefix_groups + 3 * mid + 1)) {
            lo = mid + 1;
        } else {
            return mid;
        }
    }
    return -1;
}

__device__ __forceinline__ SeqInfo seq_info(const DecodeParams &p, int s)
{
    SeqInfo i;
    i.T = seq_tokens(p, s);
    i.q0 = s * p.nq;
    i.ql = p.nq;
    i.tr = s;
    bool bad = false;
    if (p.q_start) {
        const int a = __ldg(p.q_start + s), e = __ldg(p.q_start + s + 1);
        bad = a < 0 || e < a || e > p.total_q || e - a > p.nq;
        i.q0 = a;
        i.ql = bad ? 0 : e - a;
    }
    if (p.table_row) {
        i.tr = __ldg(p.table_row + s);
        if (i.tr < 0 || i.tr >= p.table_rows) {
            bad = true;
            i.ql = 0;
        }
    }
    i.W = i.ql;
    if (p.tree_mask) {
        const int w = __ldg(p.tree_len + s);
        i.W = w < 0 ? 0 : (w > 32 ? 32 : w);
    }
    if (bad)
        atomicOr(p.ws + kWsErr, kErrBadQuery);
    const int nb = i.ql > 0 ? (i.T + kBlockSize - 1) / kBlockSize : 0;
    i.b0 = 0;
    if (p.prefix_groups && nb > 0) {
        // a member skips its group's prefix when every query row sees all of it
        const int gi = group_of(p, s);
        if (gi >= 0) {
            // the same validity rule as the prefix pass: a group it skips is not
            // skipped here either
            const int f = __ldg(p.prefix_groups + 3 * gi);
            const int cnt = __ldg(p.prefix_groups + 3 * gi + 1);
            const int P = __ldg(p.prefix_groups + 3 * gi + 2);
            const bool group_ok = f >= 0 && cnt >= 0 && f + cnt <= p.S && P >= 0 && P <= p.MB;
            if (group_ok && P > 0 && P < nb && kBlockSize * P <= i.T - i.ql)
                i.b0 = P;
        }
    }
    i.nb = nb - i.b0;  // blocks streamed by the main pass
    return i;
}

__device__ __forceinline__ int seq_blocks(const DecodeParams &p, int s) { return seq_info(p, s).nb; }

// A gpu-scope relaxed load (the L2 copy of a counter other CTAs update).
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *ptr)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

}  // namespace pkv
