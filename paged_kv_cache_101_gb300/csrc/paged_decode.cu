// paged_decode.cu -- paged decode attention for sm_103a.
//
// What is computed: for every sequence s, query j < nq and query head qh,
//   out = softmax_t(scale * <q, K_s[t]>) . V_s   over t <= T_s - nq + j,
// with K_s/V_s the sequence's tokens reached through its block table
// ("ML Interview Prep, Lesson 13" section 3.5: the kernel follows the block table
// and reads keys and values one block at a time; "07 -- Inference" section 5.1:
// online softmax with running max m, running sum l and a rescaled accumulator;
// section 5.3: FlashDecoding split + merge with the same rescaling rule).
//
// How (GB300 design, not the pages' kernel):
//  * Work space. Per head group (HG kv heads), the blocks of all sequences are
//    laid end to end: unit u = hg * NB_total + block_prefix[s] + b. This flat
//    space is cut into fixed cells: one equal contiguous chunk per CTA of the
//    persistent grid, optionally followed by a tail of smaller tickets that
//    CTAs claim dynamically once their chunk is done (so SMs that stream faster
//    take more of the tail). Cell boundaries depend only on the sizes, never on
//    which CTA runs a cell, so results are deterministic.
//  * Split-K. A sequence inside one cell is finished in place (normalised
//    output). A sequence cut by cell boundaries leaves one partial (m, l, acc)
//    per cell in the workspace; a small merge kernel, launched as a
//    programmatic dependent, combines them (same rescaling rule).
//  * Staging. The last warp is the producer: it walks its cells, reads block-table
//    entries 32 at a time (one coalesced load), and for each block issues TMA
//    tensor loads of K and V for its HG heads into a ring of shared-memory
//    stages (128-byte swizzle, mbarrier completion with byte counts). Stages are
//    recycled through "empty" mbarriers the consumers arrive on.
//  * Math. One, two or four consumer warps per kv head, bf16 mma.sync m16n8k16 with
//    fp32 accumulation, two orientations chosen by the query rows per kv head:
//    - up to 8 rows (one warp per head): S^T = K.Q^T with M = the block's 16
//      tokens, N = 8 rows, K = 16 head dims, so no mma work goes to padding
//      rows. The online softmax runs on the fragments (shuffles across the 8
//      token lanes); P is transposed in registers with movmatrix and
//      O^T += V^T.P^T takes V^T fragments from ldmatrix.trans.
//    - 9 to 64 rows (16 rows per warp): S = Q.K^T with M = 16 rows, N = 8
//      tokens, so the score fragments are the A operand of O += P.V as they
//      stand (no transposes), row reductions take two shuffles and outputs
//      leave as pairs.
//    In both, P is split into bf16 hi + lo parts (P = hi + lo to 2^-16). Rows
//    of a sequence's last block past T_s are masked in the scores and zeroed
//    in the V fragments, so stale or NaN pool contents never reach the output.
//  * Safety. Every mbarrier wait is bounded (2 s of %globaltimer); on timeout
//    the warp records a code in the workspace error word and unwinds; the
//    producer waits (bounded) for its own TMA copies before leaving. TMA reads
//    of an out-of-range block id return zeros instead of faulting.
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cstddef>
#include <type_traits>

#include "pkv_cells.cuh"
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

struct StageHdr {
    int32_t q0;     // the sequence's first query row
    int32_t b;      // logical block within the sequence
    int32_t T;      // context length (clamped)
    int32_t hg;     // head group
    int32_t flags;  // F_*
    int32_t slot;   // partial slot: 0 if the segment opens its cell, else 1
    int32_t cell;   // cell holding this block
    int16_t ql;     // the sequence's query rows (G * ql score rows per kv head)
    int16_t W;      // mask window: per-row masks rule the last W positions
};
static_assert(sizeof(StageHdr) == 32, "stage header: two 16-byte words");
static_assert(offsetof(StageHdr, hg) == 12 && offsetof(StageHdr, flags) == 16 &&
                  offsetof(StageHdr, cell) == 24 && offsetof(StageHdr, ql) == 28 &&
                  offsetof(StageHdr, W) == 30,
              "the producer writes the header as two int4 in field order");

struct Smem {
    uint8_t *stages;
    StageHdr *hdr;
    uint64_t *full;
    uint64_t *empty;
    Cells *cells;
};

__device__ __forceinline__ Smem carve(uint8_t *raw, const DecodeParams &p)
{
    uint8_t *base =
        reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    Smem s;
    s.stages = base;
    s.hdr = reinterpret_cast<StageHdr *>(base + size_t(p.nst) * p.stage_bytes);
    s.full = reinterpret_cast<uint64_t *>(s.hdr + p.nst);
    s.empty = s.full + p.nst;
    s.cells = reinterpret_cast<Cells *>(s.empty + p.nst);
    return s;
}

// ------------------------------------------------------------------ producer
template <int D, bool KV8>
__device__ void producer_warp(const CUtensorMap *kmap, const CUtensorMap *vmap,
                              const DecodeParams &p, const Smem &sm, int lane)
{
    constexpr int NH = KV8 ? 1 : D / 64;  // 16-row x 128-byte tiles per head
    const unsigned FULLMASK = 0xffffffffu;
    const int S = p.S;

    // ---- block prefix sums over sequences (lane l owns a contiguous range)
    const int per = (S + 31) / 32;
    const int s_lo = min(S, lane * per), s_hi = min(S, s_lo + per);
    int local = 0;
    for (int s = s_lo; s < s_hi; ++s)
        local += seq_blocks(p, s);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULLMASK, incl, o);
        if (lane >= o)
            incl += v;
    }
    const int base = incl - local;
    const int nb_total = __shfl_sync(FULLMASK, incl, 31);

    const Cells C = make_cells(p, nb_total, int(gridDim.x));
    if (lane == 0)
        *sm.cells = C;  // published to the consumers by the first stage's arrive
    if (blockIdx.x == 0 && lane == 0 && !p.prefix_pass) {
        // for the merge: the unit count, and whether every cell holds units
        p.ws[kWsUnits] = uint32_t(nb_total);
        p.ws[kWsDense] = (C.F1 >= C.G && (C.NT == 0 || C.F2 >= C.NT)) ? 1u : 0u;
    }

    uint32_t st = 0, phase = 0;  // ring position of the next stage to fill
    uint32_t issued = 0;         // stages filled so far
    bool ok = true;
    const uint64_t pol = policy_evict_first();

    // Fill the next stage with block `phys` (all HG heads of group hg) under the
    // given header; waits for the stage to be free first. False if that wait
    // gave up.
    auto issue = [&](int phys, int q0, int ql, int W, int b, int T, int hg, int flags, int cellv,
                     int slot, bool shallow) -> bool {
        if (issued >= uint32_t(p.nst)) {
            // the slot's previous fill must have been consumed; a paced CTA
            // (`shallow`) waits for the fill after it instead, keeping one stage
            // fewer in flight
            uint32_t ws = st, wpar = phase ^ 1u;
            if (shallow && ++ws == uint32_t(p.nst)) {
                ws = 0;
                wpar = phase;
            }
            int w_ok = 1;
            if (lane == 0)
                w_ok = mbar_wait(smem_u32(&sm.empty[ws]), wpar, kWaitLimitNs);
            if (!__shfl_sync(FULLMASK, w_ok, 0))
                return false;
        }
        if (lane == 0) {
            if (shallow && p.trace)
                p.trace[blockIdx.x * kTraceWords + 8] += 1;
            // the header in two 16-byte stores (field order of StageHdr)
            int4 *h = reinterpret_cast<int4 *>(&sm.hdr[st]);
            h[0] = make_int4(q0, b, T, hg);
            h[1] = make_int4(flags, slot, cellv,
                             int((uint32_t(uint16_t(ql))) | (uint32_t(uint16_t(W)) << 16)));
            const uint32_t bar = smem_u32(&sm.full[st]);
            mbar_arrive_expect_tx(bar, uint32_t(p.stage_bytes));
            const uint32_t kdst = smem_u32(sm.stages + size_t(st) * p.stage_bytes);
            const uint32_t vdst = kdst + uint32_t(p.HG * NH * kTileBytes);
            const int h0 = hg * p.HG;
            if (p.whole_box) {
                // map dims (d, token, half, head, block): one box = HG heads x 16 rows
                tma_load_5d_hint(kdst, kmap, bar, 0, 0, 0, h0, phys, pol);
                tma_load_5d_hint(vdst, vmap, bar, 0, 0, 0, h0, phys, pol);
            } else {
                // map dims (d, half, head, token, block): one box = one (head, half) tile
                for (int hl = 0; hl < p.HG; ++hl) {
#pragma unroll
                    for (int hf = 0; hf < NH; ++hf) {
                        const uint32_t off = uint32_t((hl * NH + hf) * kTileBytes);
                        tma_load_5d_hint(kdst + off, kmap, bar, 0, hf, h0 + hl, 0, phys, pol);
                        tma_load_5d_hint(vdst + off, vmap, bar, 0, hf, h0 + hl, 0, phys, pol);
                    }
                }
            }
            if (p.trace && issued == 0)
                p.trace[blockIdx.x * kTraceWords + 1] = global_timer_ns();
        }
        __syncwarp();
        ++issued;
        if (++st == uint32_t(p.nst)) {
            st = 0;
            phase ^= 1u;
        }
        return true;
    };
    // a block id outside the pool is flagged and read past the tensor's end (zeros)
    auto checked = [&](int phys) -> int {
        if (phys < 0 || int64_t(phys) >= p.num_blocks) {
            if (lane == 0)
                atomicOr(p.ws + kWsErr, kErrBadBlock);
            phys = int(p.num_blocks < 0x7fffffff ? p.num_blocks : 0x7fffffff);
        }
        return phys;
    };

    int64_t cell = blockIdx.x;       // phase 1: this CTA's own chunk
    int claim = -1;                  // lane 0: a ticket claimed ahead
    bool claimed = false;
    if (p.prefix_pass) {
        // Cascade prefix pass: CTA = (group, row tile, kv head); it streams the
        // group's prefix blocks once for the tile's query rows (up to 16 x 8 = 128
        // score rows, one consumer warp per 16), read through the first member's
        // table row, and leaves each row's partial over the prefix.
        const int head = int(blockIdx.x) % p.n_hg;
        const int rest = int(blockIdx.x) / p.n_hg;
        const int c = rest % p.pre_chunks;  // block range c of the prefix
        const int v = rest / p.pre_chunks;
        const int gi = v / p.pre_tiles, t = v - gi * p.pre_tiles;
        const int f = __ldg(p.prefix_groups + 3 * gi);
        const int cnt = __ldg(p.prefix_groups + 3 * gi + 1);
        int P = __ldg(p.prefix_groups + 3 * gi + 2);
        const bool bad = f < 0 || cnt < 0 || f + cnt > S || P < 0 || P > p.MB;
        if (bad && lane == 0)
            atomicOr(p.ws + kWsErr, kErrBadGroup);
        const int qrows = bad ? 0 : cnt * p.nq;
        const int q0 = f * p.nq + t * p.pre_qrows;
        int ql = qrows - t * p.pre_qrows;
        ql = ql < 0 ? 0 : (ql > p.pre_qrows ? p.pre_qrows : ql);
        if (ql == 0)
            P = 0;
        // blocks [c*P/C, (c+1)*P/C) of the prefix; the chunk index rides in `cell`
        const int b_lo = c * P / p.pre_chunks, b_hi = (c + 1) * P / p.pre_chunks;
        int bt_base = -(1 << 30), bt_val = 0;
        for (int b = b_lo; b < b_hi && ok; ++b) {
            if (b >= bt_base + 32) {
                bt_base = b;
                const int idx = b + lane;
                bt_val = idx < b_hi ? __ldg(p.block_tables + int64_t(f) * p.MB + idx) : 0;
            }
            const int phys = checked(__shfl_sync(FULLMASK, bt_val, b - bt_base));
            const int flags =
                F_PREFIX | (b == b_lo ? F_FIRST : 0) | (b == b_hi - 1 ? F_LAST : 0);
            ok = issue(phys, q0, ql, 0, b, P * kBlockSize, head, flags, c, 0, false);
        }
    }
    // Optional pacing of the static chunks: per-SM streaming rates differ by
    // several percent, so equal chunks end at different times. Every 4 units the
    // producer compares its chunk's progress with the grid's (units issued by all
    // CTAs, one counter in the workspace, read one round ahead so the load never
    // stalls the warp) and, while ahead by more than a margin, keeps one stage
    // fewer in flight: where HBM is saturated, the SMs behind get more of it.
    // Timing only: the partition, and so every result bit, is unchanged.
    uint32_t g_rd = 0;  // lane 0: the grid's units issued, as last read
    int64_t k_rd = 0;   // lane 0: this chunk's units issued at that read
    bool ahead = false;
    for (; !p.prefix_pass;) {
        const int64_t a = C.start(cell), e = C.start(cell + 1);
        const bool pace = p.pace != 0 && cell < C.G;
        const float inv_n = a < e ? 1.f / float(e - a) : 0.f, inv_f = 1.f / float(C.F);
        ahead = false;
        // locate unit f: head group, sequence and block within it
        auto locate = [&](int64_t f, int &hg_o, int &s_o, int &b_o) {
            hg_o = int(f / nb_total);
            const int r0 = int(f - int64_t(hg_o) * nb_total);
            const unsigned own =
                __ballot_sync(FULLMASK, local > 0 && r0 >= base && r0 < base + local);
            const int src = __ffs(own) - 1;
            int s_f = 0, b_f = 0;
            if (lane == src) {
                int run = base;
                for (int s = s_lo; s < s_hi; ++s) {
                    const int nb = seq_blocks(p, s);
                    if (r0 < run + nb) {
                        s_f = s;
                        b_f = r0 - run;
                        break;
                    }
                    run += nb;
                }
            }
            s_o = __shfl_sync(FULLMASK, s_f, src);
            b_o = __shfl_sync(FULLMASK, b_f, src);
        };
        if (a < e) {
            int hg, s, b;
            locate(a, hg, s, b);
            SeqInfo si = seq_info(p, s);
            b += si.b0;                  // locate counts streamed blocks only
            int b_end = si.b0 + si.nb;   // one past the sequence's last block
            int seg_b0 = b;
            bool cell_first = true;
            int bt_base = -(1 << 30);
            int bt_val = 0;
            if (p.meta_ready && issued == 0) {
                // the cell's first block-table entries, then the grid dependency wait
                // before the first copy from the pool
                bt_base = b;
                const int idx = b + lane;
                bt_val = idx < b_end ? __ldg(p.block_tables + int64_t(si.tr) * p.MB + idx) : 0;
                asm volatile("griddepcontrol.wait;" ::: "memory");
            }

            for (int64_t u = a; u < e; ++u) {
                if (b < bt_base || b >= bt_base + 32) {
                    bt_base = b;
                    const int idx = b + lane;
                    bt_val = idx < b_end ? __ldg(p.block_tables + int64_t(si.tr) * p.MB + idx) : 0;
                }
                const int phys = checked(__shfl_sync(FULLMASK, bt_val, b - bt_base));
                // claim the next ticket while the last few stages of this cell stream
                if (C.NT > 0 && !claimed && e - u <= 2) {
                    if (lane == 0)
                        claim = int(atomicAdd(p.ws + kWsTicket, 1u));
                    claimed = true;
                }
                const bool first = (u == a) || (b == si.b0);
                if (first)
                    seg_b0 = b;
                const bool last = (u == e - 1) || (b == b_end - 1);
                if (lane == 0) {
                    // the merge's record: cell (and slot) of the sequence's first
                    // piece, cell of its last
                    int2 *rec = p.pieces + int64_t(s) * p.n_hg + hg;
                    if (b == si.b0)
                        rec->x = int(cell) * 2 + (cell_first ? 0 : 1);
                    if (b == b_end - 1)
                        rec->y = int(cell);
                }
                int flags = (first ? F_FIRST : 0) | (last ? F_LAST : 0);
                // a cascade member's own blocks continue from its prefix partial
                if (first && si.b0 > 0 && b == si.b0)
                    flags |= F_PRE;
                // a whole sequence in one cell is finished in place
                if (last && seg_b0 == si.b0 && b == b_end - 1)
                    flags |= F_DIRECT;
                if (pace && lane == 0 && ((u - a) & 3) == 0) {
                    if (u > a)  // the read issued 4 units ago
                        ahead = float(k_rd) * inv_n > float(g_rd) * inv_f + p.pace_margin;
                    g_rd = ld_relaxed_gpu(p.ws + kWsProgress);
                    k_rd = u - a;
                }
                if (!issue(phys, si.q0, si.ql, si.W, b, si.T, hg, flags, int(cell),
                           cell_first ? 0 : 1, ahead)) {
                    ok = false;
                    break;
                }
                if (pace && lane == 0)
                    atomicAdd(p.ws + kWsProgress, 1u);  // result unused: a reduction
                if (last)
                    cell_first = false;
                // advance to the next unit
                ++b;
                if (b == b_end && u + 1 < e) {
                    do {
                        if (++s == S) {
                            s = 0;
                            ++hg;
                        }
                        si = seq_info(p, s);
                    } while (si.nb == 0);
                    b = si.b0;
                    b_end = si.b0 + si.nb;
                    bt_base = -(1 << 30);
                }
            }
            if (!ok)
                break;
        }
        // ---- the next cell: a ticket
        if (C.NT == 0)
            break;
        if (!claimed && lane == 0)
            claim = int(atomicAdd(p.ws + kWsTicket, 1u));
        const int t = __shfl_sync(FULLMASK, claim, 0);
        claimed = false;
        if (t >= C.NT)
            break;
        cell = int64_t(C.G) + t;
    }

    if (ok) {
        // end-of-work marker for the consumers (no bytes: a plain arrival)
        if (issued >= uint32_t(p.nst)) {
            int w_ok = 1;
            if (lane == 0)
                w_ok = mbar_wait(smem_u32(&sm.empty[st]), phase ^ 1u, kWaitLimitNs);
            ok = __shfl_sync(FULLMASK, w_ok, 0) != 0;
        }
        if (ok && lane == 0) {
            sm.hdr[st].flags = F_END;
            mbar_arrive(smem_u32(&sm.full[st]));
            if (p.trace) {
                p.trace[blockIdx.x * kTraceWords + 3] = global_timer_ns();
                p.trace[blockIdx.x * kTraceWords + 5] = issued;
            }
        }
    }
    if (lane == 0) {
        // the last CTA to finish claiming resets the ticket and progress counters
        // for the next call (the fence orders this CTA's progress updates first)
        __threadfence();
        if (atomicAdd(p.ws + kWsDone, 1u) == gridDim.x - 1) {
            atomicExch(p.ws + kWsTicket, 0u);
            atomicExch(p.ws + kWsProgress, 0u);
            atomicExch(p.ws + kWsDone, 0u);
        }
    }
    if (!ok && lane == 0) {
        atomicOr(p.ws + kWsErr, kErrProducerWait);
        // wait (bounded) for every copy this warp may still have in flight
        const uint32_t n = issued < uint32_t(p.nst) ? issued : uint32_t(p.nst);
        for (uint32_t k = 0; k < n; ++k) {
            // the k-th most recent fill: ring position and its phase parity
            uint32_t ps = st, pp = phase;
            for (uint32_t back = 0; back <= k; ++back) {
                if (ps == 0) {
                    ps = uint32_t(p.nst) - 1;
                    pp ^= 1u;
                } else {
                    --ps;
                }
            }
            if (!mbar_wait(smem_u32(&sm.full[ps]), pp, kWaitLimitNs))
                atomicOr(p.ws + kWsErr, kErrDrainWait);
        }
    }
}

// ------------------------------------------------------------------ consumers
// Consumer for warps that own at most 8 query rows (G*nq <= 8): scores in the
// tokens x rows orientation (M = the block's 16 tokens, N = 8 rows, K = 16
// dims), so a single n-tile covers the rows and no mma work is spent on
// padding rows; lane holds rows 2tq, 2tq+1.
template <int D, bool KV8>
__device__ void consumer_warp_m8(const DecodeParams &p, const Smem &sm, int cw, int lane)
{
    // bf16: a head row is D/64 tiles of 64 columns; E4M3: one 128-byte tile
    constexpr int NH = KV8 ? 1 : D / 64;
    constexpr int KS = D / 16;  // k-steps of the score mma
    constexpr int MT = D / 16;  // 16-dim m-tiles of the PV mma
    const int hl = cw;          // kv head within the group (one warp per head)
    const int g = lane >> 2, tq = lane & 3;

    // ldmatrix row addresses inside a (head, half) tile: [16 tokens][8 x 16 B], 128B swizzle
    const int k_tok = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int k_cadd = lane >> 4;
    const int v_tok = (lane & 7) + ((lane >> 4) & 1) * 8;
    const int v_cadd = (lane >> 3) & 1;
    const int sw = lane & 7;  // == k_tok & 7 == v_tok & 7

    float acc[MT][4];
    uint32_t qf[KS][2];
    float m_r[2], l_r[2];
    // E4M3: K's scale folds into the score scale, V's into the output
    float qscale = p.scale_log2, vscale = 1.f;

    // running state of the current segment
    auto reset_state = [&]() {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
            qf[ks][0] = qf[ks][1] = 0u;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            m_r[r] = -INFINITY;
            l_r[r] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                acc[i][e] = 0.f;
    };
    const uint32_t stage_base = smem_u32(sm.stages);
    uint32_t st = 0, phase = 0;
    for (;;) {
        if (!mbar_wait(smem_u32(&sm.full[st]), phase, kWaitLimitNs)) {
            if (lane == 0)
                atomicOr(p.ws + kWsErr, kErrConsumerWait);
            return;
        }
        const StageHdr h = sm.hdr[st];
        if (p.trace && cw == 0 && lane == 0) {
            uint64_t *tr = p.trace + blockIdx.x * kTraceWords;
            if (h.flags & F_END)
                tr[4] = global_timer_ns();
            else if (tr[2] == 0)
                tr[2] = global_timer_ns();
            if (h.flags & F_FIRST)
                tr[6] += 1;
        }
        if (h.flags & F_END)
            break;
        const int kvh = h.hg * p.HG + hl;

        if (h.flags & F_FIRST) {
            // a new segment: fresh running state and its query rows
            reset_state();
            if constexpr (KV8) {
                qscale = p.scale_log2 * __ldg(p.k_scale + kvh);
                vscale = __ldg(p.v_scale + kvh);
            }
            if constexpr (!KV8) {
                if (h.flags & F_PRE) {
                    // cascade member: continue from the prefix pass's (m, l, acc) of
                    // the lane's rows 2tq, 2tq+1 (l on one lane of the row's reduction)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int row = 2 * tq + r;
                        if (row >= p.G * h.ql)
                            continue;
                        const int j = row / p.G;
                        const int64_t pi0 =
                            (int64_t(h.q0) + j) * p.Hq + int64_t(kvh) * p.G + (row - j * p.G);
                        const int P = h.b;  // the member's first own block = prefix blocks
                        float M = -INFINITY, L = 0.f;
#pragma unroll
                        for (int c = 0; c < kMaxPreChunks; ++c) {
                            if (c >= p.pre_chunks ||
                                (c + 1) * P / p.pre_chunks == c * P / p.pre_chunks)
                                continue;  // no range, or an empty one that left no partial
                            const int64_t pi = int64_t(c) * p.total_q * p.Hq + pi0;
                            const float mc = __ldcg(p.pre_ml + pi * 2);
                            const float Mn = fmaxf(M, mc);
                            const float so = ex2(M - Mn), sn = ex2(mc - Mn);
                            L = L * so + __ldcg(p.pre_ml + pi * 2 + 1) * sn;
#pragma unroll
                            for (int i = 0; i < MT; ++i) {
                                acc[i][r] = acc[i][r] * so + __ldcg(p.pre_acc + pi * D + 16 * i + g) * sn;
                                acc[i][r + 2] =
                                    acc[i][r + 2] * so + __ldcg(p.pre_acc + pi * D + 16 * i + 8 + g) * sn;
                            }
                            M = Mn;
                        }
                        m_r[r] = M;
                        l_r[r] = g == 0 ? L : 0.f;
                    }
                }
            }
            if (g < p.G * h.ql) {
                const int j = g / p.G;
                const int gq = g - j * p.G;
                const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                    p.q + ((int64_t(h.q0) + j) * p.Hq + int64_t(kvh) * p.G + gq) * D);
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    if constexpr (KV8) {
                        // k-step ks = 16-byte chunk ks of the E4M3 row; lane tq holds
                        // dims 16ks+4tq .. +3 (k indices 2tq, 2tq+1 and 2tq+8, 2tq+9)
                        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(qrow) + ks * 4 + tq);
                        qf[ks][0] = bf16x2_to_f16x2(w.x);
                        qf[ks][1] = bf16x2_to_f16x2(w.y);
                    } else {
                        qf[ks][0] = __ldg(qrow + ks * 8 + tq);
                        qf[ks][1] = __ldg(qrow + ks * 8 + 4 + tq);
                    }
                }
            }
        }

        const uint32_t kb = stage_base + st * uint32_t(p.stage_bytes) + uint32_t(hl * NH * kTileBytes);
        const uint32_t vb = kb + uint32_t(p.HG * NH * kTileBytes);  // same head in the V half

        // ---- scores S^T[token][row] for the block's 16 tokens (two accumulation
        //      chains, even and odd k-steps, to halve the dependent-mma latency)
        float sc[4], sc2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            sc[e] = sc2[e] = 0.f;
        if constexpr (KV8) {
            // one ldmatrix brings chunks 2i and 2i+1 of tokens 0-7 and 8-15; a lane
            // gets 4 codes (dims 4tq..4tq+3 of its chunk) per matrix
#pragma unroll
            for (int i = 0; i < KS / 2; ++i) {
                const int chunk = 2 * i + k_cadd;
                const uint32_t addr = kb + uint32_t(k_tok * 128 + ((chunk ^ sw) << 4));
                uint32_t r[4];
                ldsm_x4(addr, r);
                uint32_t a0[4], a1[4];
                e4m3x4_to_f16x2x2(r[0], a0[0], a0[2]);
                e4m3x4_to_f16x2x2(r[1], a0[1], a0[3]);
                e4m3x4_to_f16x2x2(r[2], a1[0], a1[2]);
                e4m3x4_to_f16x2x2(r[3], a1[1], a1[3]);
                mma_f16_16816(sc, a0, qf[2 * i][0], qf[2 * i][1]);
                mma_f16_16816(sc2, a1, qf[2 * i + 1][0], qf[2 * i + 1][1]);
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int chunk = 2 * ks + k_cadd;
                const uint32_t addr = kb + uint32_t((chunk >> 3) * kTileBytes + k_tok * 128 +
                                                    (((chunk & 7) ^ sw) << 4));
                uint32_t a[4];
                ldsm_x4(addr, a);
                if (ks & 1)
                    mma_bf16_16816(sc2, a, qf[ks][0], qf[ks][1]);
                else
                    mma_bf16_16816(sc, a, qf[ks][0], qf[ks][1]);
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
            sc[e] += sc2[e];

        // ---- scale (log2 domain) and causal / tree / tail mask: positions
        //      before the first maskable one are seen by every row
        const int t0 = h.b * kBlockSize;
        const int w0 = p.tree_mask ? h.T - h.W : h.T - h.ql + 1;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            sc[e] *= qscale;
        if (__builtin_expect((t0 + kBlockSize - 1) >= w0, 0)) {
            // a sequence's last block(s): the lane's rows 2tq, 2tq+1 (the last query
            // index for padding rows) against the causal limit or their window bits
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                int j = (2 * tq + r) / p.G;
                j = j < h.ql ? j : h.ql - 1;
                if (p.tree_mask) {
                    const uint32_t bits = (2 * tq + r) < p.G * h.ql ? __ldg(p.tree_mask + h.q0 + j) : 0u;
#pragma unroll
                    for (int hi = 0; hi < 2; ++hi) {
                        const int tok = t0 + g + 8 * hi;
                        const bool vis = tok < w0 || (tok < h.T && ((bits >> (tok - w0)) & 1u));
                        if (!vis)
                            sc[2 * hi + r] = -INFINITY;
                    }
                } else {
#pragma unroll
                    for (int hi = 0; hi < 2; ++hi)
                        if (t0 + g + 8 * hi > h.T - h.ql + j)
                            sc[2 * hi + r] = -INFINITY;
                }
            }
        }

        // ---- online softmax (rows 2tq, 2tq+1 live in this lane). The running
        //      max is raised only once a score passes it by more than 2^8 (log2
        //      units), so most blocks skip the row reductions; P can reach 2^8 in
        //      between, and the result stays exact because the sum is taken
        //      against the same max. The accumulator is rescaled only when a row's
        //      max moves (otherwise every factor would be exactly 1).
        constexpr float kLazyLog2 = 8.f;
        bool lead = false;
#pragma unroll
        for (int r = 0; r < 2; ++r)
            lead |= fmaxf(sc[r], sc[r + 2]) > m_r[r] + kLazyLog2;
        if (__any_sync(0xffffffffu, lead)) {
            float corr[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float bm = fmaxf(sc[r], sc[r + 2]);
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
                const float mn = fmaxf(m_r[r], bm);
                const float mu = (mn == -INFINITY) ? 0.f : mn;
                corr[r] = ex2(m_r[r] - mu);
                m_r[r] = mn;
                l_r[r] *= corr[r];
            }
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                acc[i][0] *= corr[0];
                acc[i][1] *= corr[1];
                acc[i][2] *= corr[0];
                acc[i][3] *= corr[1];
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float mu = (m_r[r] == -INFINITY) ? 0.f : m_r[r];
            const float p0 = ex2(sc[r] - mu);
            const float p1 = ex2(sc[r + 2] - mu);
            l_r[r] += p0 + p1;
            sc[r] = p0;
            sc[r + 2] = p1;
        }

        // ---- P = hi + lo (bf16 each), transposed into mma B fragments
        //      (E4M3: P in f16, a single part: relative error <= 2^-11)
        uint32_t bh[2], bl[2];
        if constexpr (KV8) {
            bh[0] = movmatrix_trans(pack_f16x2(sc[0], sc[1]));
            bh[1] = movmatrix_trans(pack_f16x2(sc[2], sc[3]));
            bl[0] = bl[1] = 0u;
        } else {
            const uint32_t h01 = pack_bf16x2(sc[0], sc[1]);
            const uint32_t h23 = pack_bf16x2(sc[2], sc[3]);
            const uint32_t l01 = pack_bf16x2(sc[0] - bf16lo_f32(h01), sc[1] - bf16hi_f32(h01));
            const uint32_t l23 = pack_bf16x2(sc[2] - bf16lo_f32(h23), sc[3] - bf16hi_f32(h23));
            bh[0] = movmatrix_trans(h01);
            bh[1] = movmatrix_trans(h23);
            bl[0] = movmatrix_trans(l01);
            bl[1] = movmatrix_trans(l23);
        }

        // ---- V rows past the context (stale or NaN slots) are zeroed
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        const int vc = h.T - t0;
        if (vc < kBlockSize) {
            const int k0 = 2 * tq;
            mlo = (k0 < vc ? 0x0000ffffu : 0u) | (k0 + 1 < vc ? 0xffff0000u : 0u);
            mhi = (k0 + 8 < vc ? 0x0000ffffu : 0u) | (k0 + 9 < vc ? 0xffff0000u : 0u);
        }

        // ---- O^T[d][row] += V^T[d][tok] . P^T[tok][row]; the masks are applied
        //      in a sequence's last block only (MASKED = true)
        auto pv = [&](auto masked) {
            constexpr bool MASKED = decltype(masked)::value;
            if constexpr (KV8) {
                // ldmatrix.trans of chunks 2i, 2i+1 (tokens 0-7 and 8-15) gives a lane
                // tokens 2tq, 2tq+1 of the code pair (dims 2g, 2g+1); bytes 0,2 form
                // the even-dim m-tile 2i and bytes 1,3 the odd-dim m-tile 2i+1. In
                // both, M-row g is dim 32i+2g(+1) and M-row g+8 is dim 32i+16+2g(+1).
#pragma unroll
                for (int i = 0; i < MT / 2; ++i) {
                    const int chunk = 2 * i + v_cadd;
                    const uint32_t addr = vb + uint32_t(v_tok * 128 + ((chunk ^ sw) << 4));
                    uint32_t r[4];
                    ldsm_x4_trans(addr, r);
                    uint32_t ae[4], ao[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        // bytes 0,2 (even dims) then 1,3 (odd dims) in one permute
                        e4m3x4_to_f16x2x2(__byte_perm(r[m], 0u, 0x3120), ae[m], ao[m]);
                        if constexpr (MASKED) {
                            ae[m] &= m < 2 ? mlo : mhi;
                            ao[m] &= m < 2 ? mlo : mhi;
                        }
                    }
                    mma_f16_16816(acc[2 * i], ae, bh[0], bh[1]);
                    mma_f16_16816(acc[2 * i + 1], ao, bh[0], bh[1]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    const int chunk = 2 * i + v_cadd;
                    const uint32_t addr = vb + uint32_t((chunk >> 3) * kTileBytes + v_tok * 128 +
                                                        (((chunk & 7) ^ sw) << 4));
                    uint32_t a[4];
                    ldsm_x4_trans(addr, a);
                    if constexpr (MASKED) {
                        a[0] &= mlo;
                        a[1] &= mlo;
                        a[2] &= mhi;
                        a[3] &= mhi;
                    }
                    mma_bf16_16816(acc[i], a, bh[0], bh[1]);
                    mma_bf16_16816(acc[i], a, bl[0], bl[1]);
                }
            }
        };
        if (__builtin_expect(vc < kBlockSize, 0))
            pv(std::true_type());
        else
            pv(std::false_type());

        // the epilogue's header fields are read now (not kept live through the
        // stage); then the stage's shared memory goes back to the producer
        int e_q0 = 0, e_rows = 0, e_cell = 0, e_slot = 0;
        if (h.flags & F_LAST) {
            const StageHdr *hp = &sm.hdr[st];
            e_q0 = hp->q0;
            e_rows = p.G * hp->ql;
            e_cell = hp->cell;
            e_slot = hp->slot;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&sm.empty[st]));
        if (++st == uint32_t(p.nst)) {
            st = 0;
            phase ^= 1u;
        }

        if (h.flags & F_LAST) {
            // ---- finish the segment: full row sums, then output or partial
            float lf[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float v = l_r[r];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                lf[r] = v;
            }
            if (h.flags & F_DIRECT) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = 2 * tq + r;
                    if (row >= e_rows)
                        continue;
                    const int j = row / p.G;
                    const int gq = row - j * p.G;
                    const int64_t o = ((int64_t(e_q0) + j) * p.Hq + int64_t(kvh) * p.G + gq) * D;
                    const float inv = lf[r] > 0.f ? 1.f / lf[r] : 0.f;
                    if constexpr (KV8) {
                        const float f = inv * vscale;
#pragma unroll
                        for (int i = 0; i < MT / 2; ++i) {
                            const int d0 = 32 * i + 2 * g;  // and d0 + 16 for M-rows g+8
                            if (p.out_f32) {
                                float *out = static_cast<float *>(p.out) + o;
                                *reinterpret_cast<float2 *>(out + d0) =
                                    make_float2(acc[2 * i][r] * f, acc[2 * i + 1][r] * f);
                                *reinterpret_cast<float2 *>(out + d0 + 16) =
                                    make_float2(acc[2 * i][r + 2] * f, acc[2 * i + 1][r + 2] * f);
                            } else {
                                __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) + o;
                                *reinterpret_cast<__nv_bfloat162 *>(out + d0) =
                                    __floats2bfloat162_rn(acc[2 * i][r] * f, acc[2 * i + 1][r] * f);
                                *reinterpret_cast<__nv_bfloat162 *>(out + d0 + 16) =
                                    __floats2bfloat162_rn(acc[2 * i][r + 2] * f,
                                                          acc[2 * i + 1][r + 2] * f);
                            }
                        }
                    } else if (p.out_f32) {
                        float *out = static_cast<float *>(p.out) + o;
#pragma unroll
                        for (int i = 0; i < MT; ++i) {
                            out[16 * i + g] = acc[i][r] * inv;
                            out[16 * i + 8 + g] = acc[i][r + 2] * inv;
                        }
                    } else {
                        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) + o;
#pragma unroll
                        for (int i = 0; i < MT; ++i) {
                            out[16 * i + g] = __float2bfloat16_rn(acc[i][r] * inv);
                            out[16 * i + 8 + g] = __float2bfloat16_rn(acc[i][r + 2] * inv);
                        }
                    }
                }
            } else {
                // partial (m, l, acc) of this cell for the merge kernel
                const int64_t cellbase = (int64_t(e_cell) * 2 + e_slot) * p.HG + hl;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = 2 * tq + r;
                    if (row >= e_rows)
                        continue;
                    float *pa = p.part + (cellbase * p.rows + row) * D;
                    if constexpr (KV8) {
#pragma unroll
                        for (int i = 0; i < MT / 2; ++i) {
                            const int d0 = 32 * i + 2 * g;
                            *reinterpret_cast<float2 *>(pa + d0) =
                                make_float2(acc[2 * i][r] * vscale, acc[2 * i + 1][r] * vscale);
                            *reinterpret_cast<float2 *>(pa + d0 + 16) = make_float2(
                                acc[2 * i][r + 2] * vscale, acc[2 * i + 1][r + 2] * vscale);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < MT; ++i) {
                            pa[16 * i + g] = acc[i][r];
                            pa[16 * i + 8 + g] = acc[i][r + 2];
                        }
                    }
                    if (g == 0) {
                        float *ml = p.ml + (cellbase * p.rows + row) * 2;
                        ml[0] = m_r[r];
                        ml[1] = lf[r];
                    }
                }
            }
        }
    }
}

// Consumer for warps that own 16 query rows (G*nq > 8): scores in the
// rows x tokens orientation (M = the warp's 16 rows, N = 8 tokens, K = 16 dims),
// so the score fragments are directly the A operand of the PV mma and each lane
// holds two rows (g, g+8): no register transposes, two-shuffle row reductions,
// pairwise output stores. Same pipeline, masking, hi/lo split of P and lazy
// rescale as the 8-row consumer.
template <int D, int WPH, bool KV8>
__device__ void consumer_warp_m16(const DecodeParams &p, const Smem &sm, int cw, int lane)
{
    // bf16: a head row is D/64 tiles of 64 columns; E4M3: one 128-byte tile
    constexpr int NH = KV8 ? 1 : D / 64;
    constexpr int KS = D / 16;  // k-steps of the score mma
    constexpr int ND = D / 8;   // 8-dim n-tiles of the output
    const int hl = cw / WPH;    // kv head within the group
    const int r0 = (cw % WPH) * 16;
    // only the 8-warp instance runs the cascade's prefix pass
    constexpr bool kPrefixPass = (WPH == 8);
    const int g = lane >> 2, tq = lane & 3;

    // ldmatrix rows inside a (head, half) tile [16 tokens][8 x 16 B], 128B swizzle
    const int mi = lane >> 3;
    const int k_tok = (lane & 7) + ((mi >> 1) << 3);  // K: tokens 0-7 | 8-15, chunks c | c+1
    const int k_cadd = mi & 1;
    const int v_tok = (lane & 7) + ((mi & 1) << 3);   // V: tokens 0-7 | 8-15, chunks c | c+1
    const int v_cadd = mi >> 1;
    const int sw = lane & 7;

    float acc[ND][4];
    uint32_t qa[KS][4];
    float m_r[2], l_r[2];
    // E4M3: K's scale folds into the score scale, V's into the output
    float qscale = p.scale_log2, vscale = 1.f;
    auto reset_state = [&]() {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                qa[ks][e] = 0u;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            m_r[rr] = -INFINITY;
            l_r[rr] = 0.f;
        }
#pragma unroll
        for (int n = 0; n < ND; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                acc[n][e] = 0.f;
    };

    const uint32_t stage_base = smem_u32(sm.stages);
    uint32_t st = 0, phase = 0;
    for (;;) {
        if (!mbar_wait(smem_u32(&sm.full[st]), phase, kWaitLimitNs)) {
            if (lane == 0)
                atomicOr(p.ws + kWsErr, kErrConsumerWait);
            return;
        }
        const StageHdr h = sm.hdr[st];
        if (p.trace && cw == 0 && lane == 0) {
            uint64_t *tr = p.trace + blockIdx.x * kTraceWords;
            if (h.flags & F_END)
                tr[4] = global_timer_ns();
            else if (tr[2] == 0)
                tr[2] = global_timer_ns();
            if (h.flags & F_FIRST)
                tr[6] += 1;
        }
        if (h.flags & F_END)
            break;
        const int kvh = h.hg * p.HG + hl;

        if (h.flags & F_FIRST) {
            reset_state();
            if constexpr (KV8) {
                qscale = p.scale_log2 * __ldg(p.k_scale + kvh);
                vscale = __ldg(p.v_scale + kvh);
            }
            if constexpr (!KV8 && !kPrefixPass) {
                if (h.flags & F_PRE) {
                    // cascade member: continue from the prefix pass's (m, l, acc) of
                    // the lane's rows g, g+8 (l on one lane of the row's reduction)
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const int row = r0 + g + 8 * rr;
                        if (row >= p.G * h.ql)
                            continue;
                        const int j = row / p.G;
                        const int64_t pi0 =
                            (int64_t(h.q0) + j) * p.Hq + int64_t(kvh) * p.G + (row - j * p.G);
                        const int P = h.b;  // the member's first own block = prefix blocks
                        float M = -INFINITY, L = 0.f;
#pragma unroll
                        for (int c = 0; c < kMaxPreChunks; ++c) {
                            if (c >= p.pre_chunks ||
                                (c + 1) * P / p.pre_chunks == c * P / p.pre_chunks)
                                continue;  // no range, or an empty one that left no partial
                            const int64_t pi = int64_t(c) * p.total_q * p.Hq + pi0;
                            const float mc = __ldcg(p.pre_ml + pi * 2);
                            const float Mn = fmaxf(M, mc);
                            const float so = ex2(M - Mn), sn = ex2(mc - Mn);
                            L = L * so + __ldcg(p.pre_ml + pi * 2 + 1) * sn;
#pragma unroll
                            for (int n = 0; n < ND; ++n) {
                                const float2 v = __ldcg(reinterpret_cast<const float2 *>(
                                    p.pre_acc + pi * D + 8 * n + 2 * tq));
                                acc[n][2 * rr] = acc[n][2 * rr] * so + v.x * sn;
                                acc[n][2 * rr + 1] = acc[n][2 * rr + 1] * so + v.y * sn;
                            }
                            M = Mn;
                        }
                        m_r[rr] = M;
                        l_r[rr] = tq == 0 ? L : 0.f;
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int row = r0 + g + 8 * rr;
                if (row < p.G * h.ql) {
                    const int j = row / p.G;
                    const int gq = row - j * p.G;
                    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                        p.q + ((int64_t(h.q0) + j) * p.Hq + int64_t(kvh) * p.G + gq) * D);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        if constexpr (KV8) {
                            // k-step ks = 16-byte chunk ks of the E4M3 row: dims 16ks+4tq,
                            // +1 are k indices 2tq, 2tq+1; dims +2, +3 are 2tq+8, 2tq+9
                            const uint2 w =
                                __ldg(reinterpret_cast<const uint2 *>(qrow) + ks * 4 + tq);
                            qa[ks][rr] = bf16x2_to_f16x2(w.x);
                            qa[ks][2 + rr] = bf16x2_to_f16x2(w.y);
                        } else {
                            qa[ks][rr] = __ldg(qrow + ks * 8 + tq);          // dims 16ks+2tq..
                            qa[ks][2 + rr] = __ldg(qrow + ks * 8 + 4 + tq);  // 16ks+8+2tq..
                        }
                    }
                }
            }
        }

        const uint32_t kb = stage_base + st * uint32_t(p.stage_bytes) + uint32_t(hl * NH * kTileBytes);
        const uint32_t vb = kb + uint32_t(p.HG * NH * kTileBytes);  // same head in the V half

        // ---- scores S[row][token]: n-tile 0 = tokens 0-7, n-tile 1 = tokens 8-15
        float sc[2][4], sc2[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sc[n][e] = sc2[n][e] = 0.f;
        if constexpr (KV8) {
            // matrices: tokens 0-7 / chunk 2i, tokens 0-7 / 2i+1, tokens 8-15 / 2i,
            // tokens 8-15 / 2i+1; a lane gets dims 4tq..4tq+3 of token g
#pragma unroll
            for (int i = 0; i < KS / 2; ++i) {
                const int chunk = 2 * i + k_cadd;
                const uint32_t addr = kb + uint32_t(k_tok * 128 + ((chunk ^ sw) << 4));
                uint32_t r[4];
                ldsm_x4(addr, r);
                uint32_t b[4][2];
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    e4m3x4_to_f16x2x2(r[m], b[m][0], b[m][1]);
                mma_f16_16816(sc[0], qa[2 * i], b[0][0], b[0][1]);
                mma_f16_16816(sc[1], qa[2 * i], b[2][0], b[2][1]);
                mma_f16_16816(sc2[0], qa[2 * i + 1], b[1][0], b[1][1]);
                mma_f16_16816(sc2[1], qa[2 * i + 1], b[3][0], b[3][1]);
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int chunk = 2 * ks + k_cadd;
                const uint32_t addr = kb + uint32_t((chunk >> 3) * kTileBytes + k_tok * 128 +
                                                    (((chunk & 7) ^ sw) << 4));
                uint32_t b[4];
                ldsm_x4(addr, b);
                const uint32_t a[4] = {qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]};
                if (ks & 1) {
                    mma_bf16_16816(sc2[0], a, b[0], b[1]);
                    mma_bf16_16816(sc2[1], a, b[2], b[3]);
                } else {
                    mma_bf16_16816(sc[0], a, b[0], b[1]);
                    mma_bf16_16816(sc[1], a, b[2], b[3]);
                }
            }
        }
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sc[n][e] += sc2[n][e];

        // ---- scale (log2 domain) and causal / tree / tail mask: positions
        //      before the first maskable one are seen by every row
        const int t0 = h.b * kBlockSize;
        const int w0 = (kPrefixPass && (h.flags & F_PREFIX))
                           ? INT_MAX
                           : (p.tree_mask ? h.T - h.W : h.T - h.ql + 1);
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sc[n][e] *= qscale;
        if (__builtin_expect((t0 + kBlockSize - 1) >= w0, 0)) {
            // a sequence's last block(s): the lane's rows g, g+8 (the last query index
            // for padding rows) against the causal limit or their window bits
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int row = r0 + g + 8 * rr;
                int j = row / p.G;
                j = j < h.ql ? j : h.ql - 1;
                if (p.tree_mask) {
                    const uint32_t bits = row < p.G * h.ql ? __ldg(p.tree_mask + h.q0 + j) : 0u;
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const int tok = t0 + 8 * n + 2 * tq + c;
                            const bool vis = tok < w0 || (tok < h.T && ((bits >> (tok - w0)) & 1u));
                            if (!vis)
                                sc[n][2 * rr + c] = -INFINITY;
                        }
                } else {
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            if (t0 + 8 * n + 2 * tq + c > h.T - h.ql + j)
                                sc[n][2 * rr + c] = -INFINITY;
                }
            }
        }

        // ---- online softmax over the lane's two rows (g: e = 0,1; g+8: e = 2,3).
        //      The running max is raised only once a score passes it by more than
        //      2^8 (log2 units): most blocks then skip the row reductions. P can
        //      reach 2^8 in between, and the result stays exact because the sum is
        //      taken against the same max.
        constexpr float kLazyLog2 = 8.f;
        bool lead = false;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int n = 0; n < 2; ++n)
                lead |= fmaxf(sc[n][2 * rr], sc[n][2 * rr + 1]) > m_r[rr] + kLazyLog2;
        if (__any_sync(0xffffffffu, lead)) {
            float corr[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                float bm = fmaxf(fmaxf(sc[0][2 * rr], sc[0][2 * rr + 1]),
                                 fmaxf(sc[1][2 * rr], sc[1][2 * rr + 1]));
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
                const float mn = fmaxf(m_r[rr], bm);
                const float mu = (mn == -INFINITY) ? 0.f : mn;
                corr[rr] = ex2(m_r[rr] - mu);
                m_r[rr] = mn;
                l_r[rr] *= corr[rr];
            }
#pragma unroll
            for (int n = 0; n < ND; ++n) {
                acc[n][0] *= corr[0];
                acc[n][1] *= corr[0];
                acc[n][2] *= corr[1];
                acc[n][3] *= corr[1];
            }
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const float mu = (m_r[rr] == -INFINITY) ? 0.f : m_r[rr];
            float sum = 0.f;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 2 * rr; e < 2 * rr + 2; ++e) {
                    const float pv = ex2(sc[n][e] - mu);
                    sc[n][e] = pv;
                    sum += pv;
                }
            l_r[rr] += sum;
        }

        // ---- P (16 rows x 16 tokens) as the A operand, split into bf16 hi + lo
        //      (E4M3: P in f16, a single part: relative error <= 2^-11)
        uint32_t ph[4], plo[4];
        if constexpr (KV8) {
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
                    ph[2 * n + rr] = pack_f16x2(sc[n][2 * rr], sc[n][2 * rr + 1]);
        } else {
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const float x0 = sc[n][2 * rr], x1 = sc[n][2 * rr + 1];
                    const uint32_t hi = pack_bf16x2(x0, x1);
                    ph[2 * n + rr] = hi;  // a0 = (g, 0-7), a1 = (g+8, 0-7), a2 = (g, 8-15), a3 = (g+8, 8-15)
                    plo[2 * n + rr] = pack_bf16x2(x0 - bf16lo_f32(hi), x1 - bf16hi_f32(hi));
                }
        }

        // ---- V rows past the context (stale or NaN slots) are zeroed
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        const int vc = h.T - t0;
        if (vc < kBlockSize) {
            const int k0 = 2 * tq;
            mlo = (k0 < vc ? 0x0000ffffu : 0u) | (k0 + 1 < vc ? 0xffff0000u : 0u);
            mhi = (k0 + 8 < vc ? 0x0000ffffu : 0u) | (k0 + 9 < vc ? 0xffff0000u : 0u);
        }

        // ---- O[row][d] += P[row][tok] . V[tok][d]; the masks are applied in a
        //      sequence's last block only (MASKED = true)
        auto pv = [&](auto masked) {
            constexpr bool MASKED = decltype(masked)::value;
            if constexpr (KV8) {
                // ldmatrix.trans of chunks 2i, 2i+1 (tokens 0-7 and 8-15) gives a lane
                // tokens 2tq, 2tq+1 of the code pair (dims 2g, 2g+1): bytes 0,2 make
                // an n-tile of even dims, bytes 1,3 one of odd dims. n-tile 4i+2c+par
                // holds dims 16(2i+c) + 2n + par for its columns n = 0..7.
#pragma unroll
                for (int i = 0; i < D / 32; ++i) {
                    const int chunk = 2 * i + v_cadd;
                    const uint32_t addr = vb + uint32_t(v_tok * 128 + ((chunk ^ sw) << 4));
                    uint32_t r[4];
                    ldsm_x4_trans(addr, r);  // r0: tok 0-7 / 2i, r1: 8-15 / 2i, r2, r3: 2i+1
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t lo_t = r[2 * c], hi_t = r[2 * c + 1];
                        uint32_t e0, e1, o0, o1;  // even dims (bytes 0,2), odd (1,3)
                        e4m3x4_to_f16x2x2(__byte_perm(lo_t, 0u, 0x3120), e0, o0);
                        e4m3x4_to_f16x2x2(__byte_perm(hi_t, 0u, 0x3120), e1, o1);
                        if constexpr (MASKED) {
                            e0 &= mlo;
                            e1 &= mhi;
                            o0 &= mlo;
                            o1 &= mhi;
                        }
                        mma_f16_16816(acc[4 * i + 2 * c], ph, e0, e1);
                        mma_f16_16816(acc[4 * i + 2 * c + 1], ph, o0, o1);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < D / 16; ++i) {
                    const int chunk = 2 * i + v_cadd;
                    const uint32_t addr = vb + uint32_t((chunk >> 3) * kTileBytes + v_tok * 128 +
                                                        (((chunk & 7) ^ sw) << 4));
                    uint32_t b[4];
                    ldsm_x4_trans(addr, b);
                    if constexpr (MASKED) {
                        b[0] &= mlo;
                        b[1] &= mhi;
                        b[2] &= mlo;
                        b[3] &= mhi;
                    }
                    mma_bf16_16816(acc[2 * i], ph, b[0], b[1]);
                    mma_bf16_16816(acc[2 * i], plo, b[0], b[1]);
                    mma_bf16_16816(acc[2 * i + 1], ph, b[2], b[3]);
                    mma_bf16_16816(acc[2 * i + 1], plo, b[2], b[3]);
                }
            }
        };
        if (__builtin_expect(vc < kBlockSize, 0))
            pv(std::true_type());
        else
            pv(std::false_type());

        // the epilogue's header fields are read now (not kept live through the
        // stage); then the stage's shared memory goes back to the producer
        int e_q0 = 0, e_rows = 0, e_cell = 0, e_slot = 0;
        if (h.flags & F_LAST) {
            const StageHdr *hp = &sm.hdr[st];
            e_q0 = hp->q0;
            e_rows = p.G * hp->ql;
            e_cell = hp->cell;
            e_slot = hp->slot;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&sm.empty[st]));
        if (++st == uint32_t(p.nst)) {
            st = 0;
            phase ^= 1u;
        }

        if (h.flags & F_LAST) {
            float lf[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                float v = l_r[rr];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                lf[rr] = v;
            }
            if (h.flags & F_DIRECT) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int row = r0 + g + 8 * rr;
                    if (row >= e_rows)
                        continue;
                    const int j = row / p.G;
                    const int gq = row - j * p.G;
                    const int64_t o = ((int64_t(e_q0) + j) * p.Hq + int64_t(kvh) * p.G + gq) * D;
                    const float inv = lf[rr] > 0.f ? 1.f / lf[rr] : 0.f;
                    if constexpr (KV8) {
                        // chunk ch: dims 16ch + 4tq .. +3 from the even / odd n-tiles
                        const float f = inv * vscale;
#pragma unroll
                        for (int ch = 0; ch < D / 16; ++ch) {
                            const int te = 4 * (ch >> 1) + 2 * (ch & 1);
                            const float x0 = acc[te][2 * rr] * f, x1 = acc[te + 1][2 * rr] * f;
                            const float x2 = acc[te][2 * rr + 1] * f;
                            const float x3 = acc[te + 1][2 * rr + 1] * f;
                            if (p.out_f32) {
                                *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o +
                                                            16 * ch + 4 * tq) =
                                    make_float4(x0, x1, x2, x3);
                            } else {
                                const __nv_bfloat162 lo = __floats2bfloat162_rn(x0, x1);
                                const __nv_bfloat162 hi = __floats2bfloat162_rn(x2, x3);
                                uint2 w;
                                w.x = *reinterpret_cast<const uint32_t *>(&lo);
                                w.y = *reinterpret_cast<const uint32_t *>(&hi);
                                *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.out) +
                                                           o + 16 * ch + 4 * tq) = w;
                            }
                        }
                    } else if (p.out_f32) {
                        float *out = static_cast<float *>(p.out) + o;
#pragma unroll
                        for (int n = 0; n < ND; ++n)
                            *reinterpret_cast<float2 *>(out + 8 * n + 2 * tq) =
                                make_float2(acc[n][2 * rr] * inv, acc[n][2 * rr + 1] * inv);
                    } else {
                        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) + o;
#pragma unroll
                        for (int n = 0; n < ND; ++n)
                            *reinterpret_cast<__nv_bfloat162 *>(out + 8 * n + 2 * tq) =
                                __floats2bfloat162_rn(acc[n][2 * rr] * inv, acc[n][2 * rr + 1] * inv);
                    }
                }
            } else {
                // partial (m, l, acc) of this cell for the merge kernel, or of the whole
                // prefix (cascade prefix pass) for the row's (query row, head)
                const int64_t cellbase = (int64_t(e_cell) * 2 + e_slot) * p.HG + hl;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int row = r0 + g + 8 * rr;
                    if (row >= e_rows)
                        continue;
                    int64_t pidx = cellbase * p.rows + row;
                    float *pa = p.part;
                    float *pml = p.ml;
                    if (kPrefixPass && (h.flags & F_PREFIX)) {
                        const int j = row / p.G;
                        pidx = (int64_t(e_cell) * p.total_q + e_q0 + j) * p.Hq +
                               int64_t(kvh) * p.G + (row - j * p.G);
                        pa = p.pre_acc;
                        pml = p.pre_ml;
                    }
                    pa += pidx * D;
                    if constexpr (KV8) {
#pragma unroll
                        for (int ch = 0; ch < D / 16; ++ch) {
                            const int te = 4 * (ch >> 1) + 2 * (ch & 1);
                            *reinterpret_cast<float4 *>(pa + 16 * ch + 4 * tq) = make_float4(
                                acc[te][2 * rr] * vscale, acc[te + 1][2 * rr] * vscale,
                                acc[te][2 * rr + 1] * vscale, acc[te + 1][2 * rr + 1] * vscale);
                        }
                    } else {
#pragma unroll
                        for (int n = 0; n < ND; ++n)
                            *reinterpret_cast<float2 *>(pa + 8 * n + 2 * tq) =
                                make_float2(acc[n][2 * rr], acc[n][2 * rr + 1]);
                    }
                    if (tq == 0) {
                        pml[pidx * 2] = m_r[rr];
                        pml[pidx * 2 + 1] = lf[rr];
                    }
                }
            }
        }
    }
}

// MINB: CTAs per SM the plan runs (2 for the E4M3 5-8-row shape; registers are
// then capped so that two fit).
template <int D, int NTW, int WPH, bool KV8, int MINB = 1>
__global__ void __launch_bounds__(kThreadsMax, MINB)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p)
{
    static_assert(NTW == 2 || WPH == 1, "8-row warps each own a whole kv head");
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve(smem_raw, p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        for (int i = 0; i < p.nst; ++i) {
            mbar_init(smem_u32(&sm.full[i]), 1);
            mbar_init(smem_u32(&sm.empty[i]), uint32_t(p.HG * WPH));
        }
        fence_mbar_init();
    }
    // This grid may be launched while the previous kernel on the stream (e.g.
    // the KV append writing the pool) still runs: wait for it to complete and
    // its writes to be visible before reading any global memory. When that kernel
    // is known to write only the pool (meta_ready), the producer plans its cell
    // first and waits just before its first copy from the pool; the consumers
    // read nothing before the first stage lands.
    if (!p.meta_ready)
        asm volatile("griddepcontrol.wait;" ::: "memory");
    if (p.trace && threadIdx.x == 0) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        p.trace[blockIdx.x * kTraceWords + 0] = global_timer_ns();
        p.trace[blockIdx.x * kTraceWords + 7] = smid;
    }
    __syncthreads();
    // The producer is the last warp: it shares an SM sub-partition with two consumer
    // warps, and in the last slot the warp schedulers favour those consumers over it
    // (it has stages of slack); in warp 0 it slowed them (measured: speculative verify
    // 248.2 -> 243.6 us with the producer last).
    const int producer = int(blockDim.x >> 5) - 1;
    if (warp == producer) {
        producer_warp<D, KV8>(&kmap, &vmap, p, sm, lane);
    } else {
        if constexpr (NTW == 2)
            consumer_warp_m16<D, WPH, KV8>(p, sm, warp, lane);
        else
            consumer_warp_m8<D, KV8>(p, sm, warp, lane);
    }
}

// ------------------------------------------------------------------ CUDA-core consumer
// The same pipeline with the math on the CUDA cores (fp32 FMA): the reference
// point against which the tensor-core consumers were chosen. A warp owns RW
// query rows of one kv head (D = 128, bf16 pools, causal rows).
//  * Scores: lane (t, h) = (token, 64-dim half) dots its half of K row t with
//    the same half of every row's query (the queries sit in shared memory as
//    fp32 and are read as broadcasts); one shuffle joins the two halves.
//  * Online softmax per row with shuffle reductions over the 16 token lanes
//    (running max m, per-lane partial sums l, a lazily rescaled accumulator).
//  * P goes to shared memory token-major; lane i owns dims 4i..4i+3 and adds
//    P[t][r] * V[t][d] over the block's tokens (P read as broadcasts).
constexpr int kFmaHalfStride = 68;                // floats: 64 + 4 pad (no bank conflict)
constexpr int kFmaRowStride = 2 * kFmaHalfStride; // floats per staged query row

__host__ __device__ constexpr int fma_warp_bytes(int rw)
{
    return rw * kFmaRowStride * 4 + 16 * rw * 4;  // query rows + P[16][rw]
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

template <int RW>
__device__ void consumer_warp_fma(const DecodeParams &p, const Smem &sm, int cw, int lane,
                                  float *qs, float *ps)
{
    constexpr int D = 128, NH = 2;
    const unsigned FULL = 0xffffffffu;
    const int wph = p.ncw / p.HG;
    const int hl = cw / wph;              // kv head within the group
    const int r0 = (cw % wph) * RW;       // first row of this warp
    const int t = lane & 15, h = lane >> 4;  // score lanes: token, 64-dim half
    // PV lanes: dims 4*lane..+3 = half hv, 16-byte chunk cv, 8-byte sub-offset
    const int hv = lane >> 4, cv = (lane & 15) >> 1, sub = (lane & 1) * 8;

    float acc[RW][4], m_r[RW], l_r[RW];
    auto reset_state = [&]() {
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            m_r[r] = -INFINITY;
            l_r[r] = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                acc[r][e] = 0.f;
        }
    };
    auto unpack = [](uint32_t x, float &lo, float &hi) {
        lo = __uint_as_float(x << 16);
        hi = __uint_as_float(x & 0xffff0000u);
    };

    const uint32_t stage_base = smem_u32(sm.stages);
    uint32_t st = 0, phase = 0;
    for (;;) {
        if (!mbar_wait(smem_u32(&sm.full[st]), phase, kWaitLimitNs)) {
            if (lane == 0)
                atomicOr(p.ws + kWsErr, kErrConsumerWait);
            return;
        }
        const StageHdr hd = sm.hdr[st];
        if (p.trace && cw == 0 && lane == 0) {
            uint64_t *tr = p.trace + blockIdx.x * kTraceWords;
            if (hd.flags & F_END)
                tr[4] = global_timer_ns();
            else if (tr[2] == 0)
                tr[2] = global_timer_ns();
            if (hd.flags & F_FIRST)
                tr[6] += 1;
        }
        if (hd.flags & F_END)
            break;
        const int kvh = hd.hg * p.HG + hl;
        const int vrows = p.G * hd.ql;  // valid rows of this kv head

        if (hd.flags & F_FIRST) {
            // a new segment: fresh state; this warp's query rows into shared memory
            reset_state();
            __syncwarp();  // the previous segment's reads of qs are done
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int row = r0 + r;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (row < vrows) {
                    const int j = row / p.G, gq = row - j * p.G;
                    const uint2 w = __ldg(reinterpret_cast<const uint2 *>(
                        p.q + ((int64_t(hd.q0) + j) * p.Hq + int64_t(kvh) * p.G + gq) * D +
                        4 * lane));
                    unpack(w.x, v.x, v.y);
                    unpack(w.y, v.z, v.w);
                }
                *reinterpret_cast<float4 *>(qs + r * kFmaRowStride + hv * kFmaHalfStride +
                                            4 * (lane & 15)) = v;
            }
            __syncwarp();
        }

        const uint32_t kb =
            stage_base + st * uint32_t(p.stage_bytes) + uint32_t(hl * NH * kTileBytes);
        const uint32_t vb = kb + uint32_t(p.HG * NH * kTileBytes);

        // ---- scores: lane (t, h) over dims 64h .. 64h + 63, 8 at a time
        float s[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r)
            s[r] = 0.f;
        const uint32_t krow = kb + uint32_t(h * kTileBytes + t * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 kw = lds128(krow + uint32_t((c ^ (t & 7)) << 4));
            float kf[8];
            unpack(kw.x, kf[0], kf[1]);
            unpack(kw.y, kf[2], kf[3]);
            unpack(kw.z, kf[4], kf[5]);
            unpack(kw.w, kf[6], kf[7]);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const float4 *qv =
                    reinterpret_cast<const float4 *>(qs + r * kFmaRowStride + h * kFmaHalfStride + 8 * c);
                const float4 a = qv[0], b = qv[1];
                float x = s[r];
                x = fmaf(a.x, kf[0], x);
                x = fmaf(a.y, kf[1], x);
                x = fmaf(a.z, kf[2], x);
                x = fmaf(a.w, kf[3], x);
                x = fmaf(b.x, kf[4], x);
                x = fmaf(b.y, kf[5], x);
                x = fmaf(b.z, kf[6], x);
                x = fmaf(b.w, kf[7], x);
                s[r] = x;
            }
        }
        const int t0 = hd.b * kBlockSize;
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            s[r] += __shfl_xor_sync(FULL, s[r], 16);
            s[r] *= p.scale_log2;
        }
        if (__builtin_expect(t0 + kBlockSize - 1 >= hd.T - hd.ql + 1, 0)) {
            // a sequence's last block(s): causal limit per row (padding rows take
            // the last query's), which also masks tokens past the context
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                int j = (r0 + r) / p.G;
                j = j < hd.ql ? j : hd.ql - 1;
                if (t0 + t > hd.T - hd.ql + j)
                    s[r] = -INFINITY;
            }
        }

        // ---- online softmax: block max over the 16 token lanes of each half
        //      (both halves hold the same scores), rescale only when it grew
        bool grew = false;
        float corr[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            float bm = s[r];
            bm = fmaxf(bm, __shfl_xor_sync(FULL, bm, 1));
            bm = fmaxf(bm, __shfl_xor_sync(FULL, bm, 2));
            bm = fmaxf(bm, __shfl_xor_sync(FULL, bm, 4));
            bm = fmaxf(bm, __shfl_xor_sync(FULL, bm, 8));
            const float mn = fmaxf(m_r[r], bm);
            grew |= mn > m_r[r];
            const float mu = mn == -INFINITY ? 0.f : mn;
            corr[r] = ex2(m_r[r] - mu);  // 1 when the max did not grow, 0 from -inf
            m_r[r] = mn;
            const float pr = ex2(s[r] - mu);  // 0 for a masked token
            l_r[r] = l_r[r] * corr[r] + pr;
            s[r] = pr;
        }
        if (__any_sync(FULL, grew)) {
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[r][e] *= corr[r];
        }

        // ---- P to shared memory, token-major
        __syncwarp();  // the previous block's reads of ps are done
        if (h == 0) {
#pragma unroll
            for (int r4 = 0; r4 < RW / 4; ++r4)
                *reinterpret_cast<float4 *>(ps + t * RW + 4 * r4) =
                    make_float4(s[4 * r4], s[4 * r4 + 1], s[4 * r4 + 2], s[4 * r4 + 3]);
        }
        __syncwarp();

        // ---- O[r][4 lane .. +3] += P[t][r] * V[t][..]; slots past the context
        //      (stale or NaN) are zeroed in the last block
        const int vc = hd.T - t0;
        const uint32_t vrow = vb + uint32_t(hv * kTileBytes + sub);
        auto pv = [&](auto masked) {
            constexpr bool MASKED = decltype(masked)::value;
#pragma unroll
            for (int tt = 0; tt < kBlockSize; ++tt) {
                const uint2 vw = lds64(vrow + uint32_t(tt * 128 + ((cv ^ (tt & 7)) << 4)));
                float v[4];
                unpack(vw.x, v[0], v[1]);
                unpack(vw.y, v[2], v[3]);
                if constexpr (MASKED) {
                    if (tt >= vc)
                        v[0] = v[1] = v[2] = v[3] = 0.f;
                }
#pragma unroll
                for (int r4 = 0; r4 < RW / 4; ++r4) {
                    const float4 pr = *reinterpret_cast<const float4 *>(ps + tt * RW + 4 * r4);
                    const float pp[4] = {pr.x, pr.y, pr.z, pr.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            acc[4 * r4 + i][e] = fmaf(pp[i], v[e], acc[4 * r4 + i][e]);
                }
            }
        };
        if (__builtin_expect(vc < kBlockSize, 0))
            pv(std::true_type());
        else
            pv(std::false_type());

        // epilogue fields, then the stage goes back to the producer
        int e_q0 = 0, e_cell = 0, e_slot = 0;
        if (hd.flags & F_LAST) {
            const StageHdr *hp = &sm.hdr[st];
            e_q0 = hp->q0;
            e_cell = hp->cell;
            e_slot = hp->slot;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&sm.empty[st]));
        if (++st == uint32_t(p.nst)) {
            st = 0;
            phase ^= 1u;
        }

        if (hd.flags & F_LAST) {
            // full row sums over the 16 token lanes, then output or partial
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                float v = l_r[r];
                v += __shfl_xor_sync(FULL, v, 1);
                v += __shfl_xor_sync(FULL, v, 2);
                v += __shfl_xor_sync(FULL, v, 4);
                v += __shfl_xor_sync(FULL, v, 8);
                const int row = r0 + r;
                if (row >= vrows)
                    continue;
                if (hd.flags & F_DIRECT) {
                    const int j = row / p.G, gq = row - j * p.G;
                    const int64_t o =
                        ((int64_t(e_q0) + j) * p.Hq + int64_t(kvh) * p.G + gq) * D + 4 * lane;
                    const float inv = v > 0.f ? 1.f / v : 0.f;
                    if (p.out_f32) {
                        *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o) = make_float4(
                            acc[r][0] * inv, acc[r][1] * inv, acc[r][2] * inv, acc[r][3] * inv);
                    } else {
                        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[r][0] * inv, acc[r][1] * inv);
                        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[r][2] * inv, acc[r][3] * inv);
                        uint2 w;
                        w.x = *reinterpret_cast<const uint32_t *>(&lo);
                        w.y = *reinterpret_cast<const uint32_t *>(&hi);
                        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.out) + o) = w;
                    }
                } else {
                    // partial (m, l, acc) of this cell for the merge kernel
                    const int64_t pidx =
                        ((int64_t(e_cell) * 2 + e_slot) * p.HG + hl) * p.rows + row;
                    *reinterpret_cast<float4 *>(p.part + pidx * D + 4 * lane) =
                        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
                    if (lane == 0) {
                        p.ml[pidx * 2] = m_r[r];
                        p.ml[pidx * 2 + 1] = v;
                    }
                }
            }
        }
    }
}

template <int RW>
__global__ void __launch_bounds__(kThreadsMax, 1)
    paged_decode_fma_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve(smem_raw, p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        for (int i = 0; i < p.nst; ++i) {
            mbar_init(smem_u32(&sm.full[i]), 1);
            mbar_init(smem_u32(&sm.empty[i]), uint32_t(p.ncw));
        }
        fence_mbar_init();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        producer_warp<128, false>(&kmap, &vmap, p, sm, lane);
    } else {
        // per-warp query rows and P after the cells record (16-byte aligned)
        uint8_t *extra = reinterpret_cast<uint8_t *>(
            (reinterpret_cast<uintptr_t>(sm.cells + 1) + 15) & ~uintptr_t(15));
        float *qs = reinterpret_cast<float *>(extra + size_t(warp - 1) * fma_warp_bytes(RW));
        float *ps = qs + RW * kFmaRowStride;
        consumer_warp_fma<RW>(p, sm, warp - 1, lane, qs, ps);
    }
}

// ------------------------------------------------------------------ merge
// Combine the partials of every sequence that cell boundaries split. The main
// pass records, per (sequence, head group), the cell of the first piece (and
// its slot: 1 if the piece does not open its cell) and the cell of the last;
// the pieces are the cells between, each in slot 0 of its cell. Per output row:
//   M = max_k m_k,  f_k = 2^(m_k - M),  L = sum_k l_k f_k,  out = sum_k f_k acc_k / L
// ("07 -- Inference" section 5.3, m in the log2 domain). With M known first, the
// acc loads of all pieces are independent and go out together. One CTA per
// (sequence, head group, 8 * RPW rows): a warp takes RPW rows; lane k holds
// (m, l) of piece k (32 pieces a round, rescaled across rounds), then lane i owns
// dims 4i..4i+3 of every piece, PB pieces per batch of acc loads. Sequences with
// no token get zeros. Launched as a programmatic dependent of the main kernel: it
// waits (griddepcontrol) for it. Its time after the main kernel is a chain of L2
// round trips, so the registers are capped for three CTAs per SM (two rows per
// warp and four pieces per batch for up to 32 rows per head group, more CTAs for
// few rows; four rows per warp and two pieces per batch above, fewer CTAs).
template <int D, int RPW, int PB>
__global__ void __launch_bounds__(256, 3)
    paged_decode_merge_kernel(const DecodeParams p, int grid)
{
    const unsigned FULL = 0xffffffffu;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int s = blockIdx.x, hg = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrows = p.HG * p.rows;  // partial rows of this (sequence, head group)
    const int r0 = int(blockIdx.z) * (8 * RPW) + warp * RPW;
    if (r0 >= nrows)
        return;
    const SeqInfo si = seq_info(p, s);
    const int vrows = p.G * si.ql;  // rows of each kv head with a query
    const bool has_d = lane * 4 < D;

    auto valid = [&](int r) { return r < nrows && r - (r / p.rows) * p.rows < vrows; };
    auto out_offset = [&](int r) -> int64_t {  // r = hl * rows + row
        const int hl = r / p.rows, row = r - hl * p.rows;
        const int j = row / p.G, gq = row - j * p.G;
        return ((int64_t(si.q0) + j) * p.Hq + int64_t(hg * p.HG + hl) * p.G + gq) * D + lane * 4;
    };
    auto store = [&](int64_t o, float4 v) {
        if (p.out_f32) {
            *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o) = v;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&lo);
            u.y = *reinterpret_cast<uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.out) + o) = u;
        }
    };

    if (si.nb == 0) {  // no token (or no query rows): zeros
#pragma unroll
        for (int i = 0; i < RPW; ++i)
            if (has_d && valid(r0 + i))
                store(out_offset(r0 + i), make_float4(0.f, 0.f, 0.f, 0.f));
        return;
    }
    const int2 rec = __ldcg(p.pieces + int64_t(s) * p.n_hg + hg);
    const int kb = rec.x >> 1, ke = rec.y;
    if (ke <= kb)
        return;  // one piece: finished in place by the main kernel
    if (kb < 0 || ke >= grid + p.tickets_max)
        return;  // not a record of this call (a main pass that gave up): nothing to merge
    const int np = ke - kb + 1;
    // with fewer units than cells some cells are empty and hold no partial
    const bool dense = __ldcg(p.ws + kWsDense) != 0u;
    Cells C{};
    if (!dense)
        C = make_cells(p, int(__ldcg(p.ws + kWsUnits)), grid);
    // (cell, slot) base index of piece k, or -1 for an empty cell
    auto piece_base = [&](int k) -> int64_t {
        const int64_t cell = int64_t(kb) + k;
        if (!dense && C.empty(cell))
            return -1;
        return (cell * 2 + (k == 0 ? (rec.x & 1) : 0)) * p.HG;
    };

    float M[RPW], L[RPW];
    float4 a[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        M[i] = -INFINITY;
        L[i] = 0.f;
        a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k0 = 0; k0 < np; k0 += 32) {
        // ---- (m, l) of pieces k0 + lane: the round's max, weights and sums
        const int kn = np - k0 < 32 ? np - k0 : 32;
        const int64_t cb = lane < kn ? piece_base(k0 + lane) : -1;
        float f[RPW];
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const int r = r0 + i;
            const bool ok = cb >= 0 && r < nrows;
            const int64_t idx = cb * p.rows + r;
            const float m = ok ? __ldcg(p.ml + idx * 2) : -INFINITY;
            const float l = ok ? __ldcg(p.ml + idx * 2 + 1) : 0.f;
            float mr = m;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                mr = fmaxf(mr, __shfl_xor_sync(FULL, mr, o));
            const float Mn = fmaxf(M[i], mr);
            const float mu = Mn == -INFINITY ? 0.f : Mn;
            const float so = ex2(M[i] - mu);  // earlier rounds (0 while M is -inf)
            f[i] = ex2(m - mu);                // 0 for an absent piece
            float lr = l * f[i];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                lr += __shfl_xor_sync(FULL, lr, o);
            L[i] = L[i] * so + lr;
            a[i].x *= so;
            a[i].y *= so;
            a[i].z *= so;
            a[i].w *= so;
            M[i] = Mn;
        }
        // ---- acc of the round's pieces, PB at a time, all rows together
        for (int kk = 0; kk < kn; kk += PB) {
            float4 v[PB][RPW];
            float w[PB][RPW];
#pragma unroll
            for (int c = 0; c < PB; ++c) {
                const int k = kk + c;
                const int64_t cbk = __shfl_sync(FULL, cb, k & 31);
#pragma unroll
                for (int i = 0; i < RPW; ++i) {
                    const int r = r0 + i;
                    w[c][i] = __shfl_sync(FULL, f[i], k & 31);
                    const bool ok = k < kn && cbk >= 0 && r < nrows && has_d;
                    v[c][i] = ok ? __ldcg(reinterpret_cast<const float4 *>(
                                       p.part + (cbk * p.rows + r) * D) + lane)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                    if (!ok)
                        w[c][i] = 0.f;
                }
            }
#pragma unroll
            for (int c = 0; c < PB; ++c)
#pragma unroll
                for (int i = 0; i < RPW; ++i) {
                    a[i].x += w[c][i] * v[c][i].x;
                    a[i].y += w[c][i] * v[c][i].y;
                    a[i].z += w[c][i] * v[c][i].z;
                    a[i].w += w[c][i] * v[c][i].w;
                }
        }
    }
    if (!has_d)
        return;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        if (!valid(r0 + i))
            continue;
        const float inv = L[i] > 0.f ? 1.f / L[i] : 0.f;
        store(out_offset(r0 + i), make_float4(a[i].x * inv, a[i].y * inv, a[i].z * inv, a[i].w * inv));
    }
}

// ------------------------------------------------------------------ host side
static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int plan_decode(int S, int nq, int Hq, int Hkv, int D, int MB, int num_sms, int opt_ctas,
                int opt_stages, int opt_heads, int opt_tail, int smem_optin, int kv8, int fma,
                int umma, DecodePlan *pl)
{
    if (S < 1 || nq < 1 || Hkv < 1 || Hq % Hkv != 0 || (D != 64 && D != 128) || MB < 1)
        return -1;
    if (kv8 && D != 128)
        return -1;  // E4M3 rows are one 128-byte swizzle row
    if (fma && (kv8 || D != 128))
        return -1;  // the CUDA-core consumer: bf16 pools, head_dim 128
    DecodePlan P{};
    P.D = D;
    P.kv8 = kv8 ? 1 : 0;
    P.fma = fma ? 1 : 0;
    P.G = Hq / Hkv;
    P.rows = P.G * nq;
    if (P.rows > kMaxRows)
        return -1;
    if (umma && !P.kv8 && !P.fma && D == 128 && P.rows > 16) {
        // tcgen05 consumers: one kv head per CTA, super-stages of 8 blocks, the
        // query rows padded to the MMA's N (32 or 64)
        P.umma = 1;
        P.rows_pad = P.rows <= 32 ? 32 : 64;
        P.wph = 1;
        P.ntw = 0;
        P.HG = 1;
        P.n_hg = Hkv;
        P.threads = 352;
        P.stage_bytes = 65536;
        P.nst = umma_stages(P.rows_pad);
        P.smem = umma_smem_bytes(P.rows_pad);
        if (int(P.smem) > smem_optin)
            return -1;
        P.ctas_per_sm = 1;
        const int grid_cap = opt_ctas > 0 ? opt_ctas : num_sms;
        if (grid_cap < 1 || grid_cap > 16384)
            return -1;
        P.grid = int(std::min<int64_t>(grid_cap, int64_t(P.n_hg) * S * MB));
        P.tail_div = 0;
        P.tickets_max = 0;
        const size_t cells = size_t(grid_cap);
        P.off_rec = kWsHeaderBytes;
        P.off_ml = P.off_rec + round_up(size_t(S) * P.n_hg * 8, 256);
        P.off_part = P.off_ml + round_up(cells * 2 * P.rows * 2 * 4, 256);
        P.ws_bytes = P.off_part + round_up(cells * 2 * P.rows * size_t(D) * 4, 256);
        *pl = P;
        return 0;
    }
    if (P.fma) {
        // 4 or 8 rows per warp (fp32 registers: RW x 4 accumulators a lane)
        P.rw = P.rows <= 4 ? 4 : 8;
        P.wph = (P.rows + P.rw - 1) / P.rw;
        P.ntw = 0;
        P.rows_pad = P.wph * P.rw;
    } else {
        // up to 16 rows: one warp per kv head; above, 16-row warps (2 or 4 per head)
        const int nt_total = (P.rows + 7) / 8;
        if (nt_total <= 2) {
            P.wph = 1;
            P.ntw = nt_total;
        } else {
            P.wph = nt_total <= 4 ? 2 : 4;
            P.ntw = 2;
        }
        P.rows_pad = P.wph * P.ntw * 8;
    }
    int max_hg = kMaxConsumerWarps / P.wph;
    if (opt_heads > 0 && opt_heads < max_hg)
        max_hg = opt_heads;
    P.HG = 1;
    for (int h = std::min(max_hg, Hkv); h >= 1; --h)
        if (Hkv % h == 0) {
            P.HG = h;
            break;
        }
    P.n_hg = Hkv / P.HG;
    P.threads = 32 * (1 + P.HG * P.wph);
    P.stage_bytes = 2 * P.HG * (P.kv8 ? 1 : D / 64) * kTileBytes;
    const int per_stage = P.stage_bytes + int(sizeof(StageHdr)) + 16;
    int fixed = 1024 + int(sizeof(Cells)) + 64;
    if (P.fma)  // per consumer warp: its query rows and P in fp32
        fixed += 16 + P.HG * P.wph * fma_warp_bytes(P.rw);
    // E4M3 with 5 to 8 rows per kv head: two CTAs per SM. These consumers wait on
    // the latency of the conversions and the doubled math per byte, not on memory,
    // so twice the warps pay off more than deep rings (measured: 8 rows 130 -> 113
    // us on the 70B mix; with 4 rows the extra cells and shorter rings cost more).
    const bool two_per_sm = P.kv8 && P.ntw == 1 && P.wph == 1 && P.rows > 4;
    const int smem_budget = two_per_sm ? smem_optin / 2 - 1024 : smem_optin;
    int max_st = (smem_budget - fixed) / per_stage;
    if (max_st > 8)
        max_st = 8;
    if (max_st < 2)
        return -1;
    P.nst = opt_stages > 0 ? std::min(std::max(opt_stages, 2), max_st) : max_st;
    P.smem = size_t(fixed) + size_t(P.nst) * per_stage;
    P.ctas_per_sm = two_per_sm ? 2 : 1;
    const int grid_cap = opt_ctas > 0 ? opt_ctas : P.ctas_per_sm * num_sms;
    if (grid_cap < 1 || grid_cap > 16384)
        return -1;
    const int64_t f_max = int64_t(P.n_hg) * S * MB;
    P.grid = int(std::min<int64_t>(grid_cap, f_max));
    // Optional dynamic tail: the last 1/tail_div of the units go out as tickets
    // to the CTAs that finish their chunk first (per-SM streaming rates differ
    // by a few percent). Off by default: the extra cells cost the merge more
    // than the balance gains. Never with many query rows per kv head.
    P.tail_div = opt_tail <= 1 ? 0 : opt_tail;
    P.tickets_max = (P.tail_div > 0 && P.rows <= 16) ? 2 * grid_cap : 0;
    const size_t cells = size_t(grid_cap) + size_t(P.tickets_max);
    P.off_rec = kWsHeaderBytes;
    P.off_ml = P.off_rec + round_up(size_t(S) * P.n_hg * 8, 256);
    P.off_part = P.off_ml + round_up(cells * 2 * P.HG * P.rows * 2 * 4, 256);
    P.ws_bytes = P.off_part + round_up(cells * 2 * P.HG * P.rows * size_t(D) * 4, 256);
    *pl = P;
    return 0;
}

// The cascade's prefix pass: one kv head per CTA, 8 consumer warps of 16 score
// rows (128 rows: 128 / G queries of the group's members per row tile).
int plan_prefix(int D, int G, int Hkv, int num_groups, int max_group_seqs, int nq,
                int smem_optin, DecodePlan *pl)
{
    if ((D != 64 && D != 128) || G < 1 || G > 128 || Hkv < 1 || num_groups < 1 ||
        max_group_seqs < 1 || nq < 1)
        return -1;
    DecodePlan P{};
    P.D = D;
    P.G = G;
    P.prefix = 1;
    P.wph = 8;
    P.ntw = 2;
    P.rows = (128 / G) * G;  // score rows of a tile
    P.rows_pad = 128;
    P.HG = 1;
    P.n_hg = Hkv;
    P.threads = 32 * (1 + 8);
    P.stage_bytes = 2 * (D / 64) * kTileBytes;
    const int per_stage = P.stage_bytes + int(sizeof(StageHdr)) + 16;
    const int fixed = 1024 + int(sizeof(Cells)) + 64;
    P.nst = std::min(8, (smem_optin - fixed) / per_stage);
    if (P.nst < 2)
        return -1;
    P.smem = size_t(fixed) + size_t(P.nst) * per_stage;
    const int64_t tiles = (int64_t(max_group_seqs) * nq + (128 / G) - 1) / (128 / G);
    const int64_t grid = int64_t(num_groups) * tiles * Hkv;
    if (grid > 0x7fffffff)
        return -1;
    P.grid = int(grid);
    P.tickets_max = 0;
    P.tail_div = 0;
    *pl = P;
    return int(tiles);
}

// Launch one attention kernel (and, unless told not to, its merge) on `stream`;
// `configured_smem` is the kernel's own record of the shared memory it may use.
template <typename Kern>
static cudaError_t launch_kernel(Kern kern, int *configured_smem, const DecodePlan &pl,
                                 const DecodeParams &p, const CUtensorMap &kmap,
                                 const CUtensorMap &vmap, cudaStream_t stream,
                                 cudaEvent_t ev_before, cudaEvent_t ev_after, bool with_merge)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && configured_smem[dev] < int(pl.smem)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem));
        if (e != cudaSuccess)
            return e;
        configured_smem[dev] = int(pl.smem);
    }
    if (ev_before && (e = cudaEventRecord(ev_before, stream)) != cudaSuccess)
        return e;
    // programmatic serialization: the kernel's prologue may overlap the tail of
    // the previous kernel; it waits (griddepcontrol.wait) before any read
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(pl.grid));
    cfg.blockDim = dim3(unsigned(pl.threads));
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, kmap, vmap, p);
    if (e != cudaSuccess)
        return e;
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    if (ev_after && (e = cudaEventRecord(ev_after, stream)) != cudaSuccess)
        return e;
    if (!with_merge)
        return cudaSuccess;
    return launch_merge(pl, p, stream);
}

cudaError_t launch_merge(const DecodePlan &pl, const DecodeParams &p, cudaStream_t stream)
{
    // the merge: one CTA per (sequence, head group, 8 * RPW rows), a programmatic dependent
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaError_t e;
    const bool few_rows = p.HG * p.rows <= 32;
    // fewer (sequence, head group) pairs than cells: sequences span many cells, so a
    // merge folds many pieces; one row per warp and 8 pieces per batch of loads
    // halve its chain of L2 round trips
    const bool many_pieces = few_rows && int64_t(p.S) * p.n_hg < int64_t(pl.grid);
    const int cta_rows = many_pieces ? 8 : few_rows ? 16 : 32;
    cudaLaunchConfig_t mcfg = {};
    mcfg.gridDim = dim3(unsigned(p.S), unsigned(p.n_hg),
                        unsigned((p.HG * p.rows + cta_rows - 1) / cta_rows));
    mcfg.blockDim = dim3(256);
    mcfg.dynamicSmemBytes = 0;
    mcfg.stream = stream;
    mcfg.attrs = attr;
    mcfg.numAttrs = 1;
    if (pl.D == 64)
        e = few_rows ? cudaLaunchKernelEx(&mcfg, paged_decode_merge_kernel<64, 2, 4>, p, int(pl.grid))
                     : cudaLaunchKernelEx(&mcfg, paged_decode_merge_kernel<64, 4, 2>, p, int(pl.grid));
    else if (many_pieces)
        e = cudaLaunchKernelEx(&mcfg, paged_decode_merge_kernel<128, 1, 8>, p, int(pl.grid));
    else
        e = few_rows ? cudaLaunchKernelEx(&mcfg, paged_decode_merge_kernel<128, 2, 4>, p, int(pl.grid))
                     : cudaLaunchKernelEx(&mcfg, paged_decode_merge_kernel<128, 4, 2>, p, int(pl.grid));
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <int D, int NTW, int WPH, bool KV8, int MINB = 1>
static cudaError_t launch_one(const DecodePlan &pl, const DecodeParams &p, const CUtensorMap &kmap,
                              const CUtensorMap &vmap, cudaStream_t stream, cudaEvent_t ev_before,
                              cudaEvent_t ev_after, bool with_merge = true)
{
    static int configured_smem[64] = {0};  // per device ordinal
    return launch_kernel(paged_decode_kernel<D, NTW, WPH, KV8, MINB>, configured_smem, pl, p,
                         kmap, vmap, stream, ev_before, ev_after, with_merge);
}

template <int RW>
static cudaError_t launch_fma(const DecodePlan &pl, const DecodeParams &p, const CUtensorMap &kmap,
                              const CUtensorMap &vmap, cudaStream_t stream, cudaEvent_t ev_before,
                              cudaEvent_t ev_after)
{
    static int configured_smem[64] = {0};  // per device ordinal
    return launch_kernel(paged_decode_fma_kernel<RW>, configured_smem, pl, p, kmap, vmap, stream,
                         ev_before, ev_after, true);
}

cudaError_t launch_decode(const DecodePlan &pl, const DecodeParams &p, const CUtensorMap &kmap,
                          const CUtensorMap &vmap, cudaStream_t stream, cudaEvent_t eb,
                          cudaEvent_t ea)
{
    if (pl.prefix) {  // cascade prefix pass: no merge of its own
        if (pl.D == 64)
            return launch_one<64, 2, 8, false>(pl, p, kmap, vmap, stream, eb, ea, false);
        return launch_one<128, 2, 8, false>(pl, p, kmap, vmap, stream, eb, ea, false);
    }
    if (pl.fma) {  // CUDA-core consumers: bf16, D = 128
        if (pl.rw == 4)
            return launch_fma<4>(pl, p, kmap, vmap, stream, eb, ea);
        return launch_fma<8>(pl, p, kmap, vmap, stream, eb, ea);
    }
    if (pl.kv8) {  // E4M3 pools: D = 128 only
        if (pl.ctas_per_sm == 2)
            return launch_one<128, 1, 1, true, 2>(pl, p, kmap, vmap, stream, eb, ea);
        if (pl.wph == 4)
            return launch_one<128, 2, 4, true>(pl, p, kmap, vmap, stream, eb, ea);
        if (pl.wph == 2)
            return launch_one<128, 2, 2, true>(pl, p, kmap, vmap, stream, eb, ea);
        if (pl.ntw == 2)
            return launch_one<128, 2, 1, true>(pl, p, kmap, vmap, stream, eb, ea);
        return launch_one<128, 1, 1, true>(pl, p, kmap, vmap, stream, eb, ea);
    }
    if (pl.D == 64) {
        if (pl.wph == 4)
            return launch_one<64, 2, 4, false>(pl, p, kmap, vmap, stream, eb, ea);
        if (pl.wph == 2)
            return launch_one<64, 2, 2, false>(pl, p, kmap, vmap, stream, eb, ea);
        if (pl.ntw == 2)
            return launch_one<64, 2, 1, false>(pl, p, kmap, vmap, stream, eb, ea);
        return launch_one<64, 1, 1, false>(pl, p, kmap, vmap, stream, eb, ea);
    }
    if (pl.wph == 4)
        return launch_one<128, 2, 4, false>(pl, p, kmap, vmap, stream, eb, ea);
    if (pl.wph == 2)
        return launch_one<128, 2, 2, false>(pl, p, kmap, vmap, stream, eb, ea);
    if (pl.ntw == 2)
        return launch_one<128, 2, 1, false>(pl, p, kmap, vmap, stream, eb, ea);
    return launch_one<128, 1, 1, false>(pl, p, kmap, vmap, stream, eb, ea);
}

}  // namespace pkv
