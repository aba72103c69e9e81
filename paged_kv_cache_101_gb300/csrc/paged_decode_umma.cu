// paged_decode_umma.cu -- paged decode attention on the fifth-generation tensor
// cores (tcgen05) for kv heads with 17 to 64 query rows: speculative verification
// (nq draft tokens x G query heads per kv head) and tree verification.
//
// What is computed is the same function as paged_decode.cu's kernels: for every
// sequence, query row and query head, softmax_t(scale * <q, K_s[t]>) . V_s over the
// tokens the row sees, with K_s/V_s reached through the block table ("ML Interview
// Prep, Lesson 13" section 3.5), accumulated with the online-softmax rescaling rule
// ("07 -- Inference" section 5.1) and split into cells whose partials the merge
// kernel combines (section 5.3).
//
// Why a second kernel: with G * nq = 32 or more query rows per kv head, the warp
// MMA path spends more issue slots on mma.sync, ldmatrix and register-held
// accumulators than HBM needs to stream the tiles. Here one thread issues whole-tile
// MMAs from shared memory, the scores, probabilities and accumulators live in
// tensor memory (TMEM), and the CUDA cores keep only the softmax.
//
// Layout of the work:
//  * The unit space, cells and stages are those of paged_decode.cu: a unit is one
//    16-token block of HG = 2 kv heads (a head group), each CTA of the persistent
//    grid streams one contiguous cell, and a stage is one block of the group's K
//    and V ([head][64-dim half][16 tokens][64] bf16, the 128-byte swizzle TMA
//    writes) in a ring of shared-memory stages released block by block.
//  * Scores, rows on M: S_h[64 rows][16 tokens] = Q_h . K_h^T per head and block
//    (M = 64, N = 16, K = 128 dims) into TMEM. Q_h holds the sequence's G * nq
//    query rows (zero rows up to 64) and is staged by TMA at every segment's start.
//    Blocks go through scores, softmax and values in groups of two consecutive
//    blocks of a segment, and two groups are in flight (S and P double-buffered in
//    TMEM), so the MMA-softmax-MMA round trip is paid once per 32 KiB.
//  * Softmax: the thread of row r (lane r % 16 of the warp in TMEM lane quarter
//    r / 16, the M = 64 data-path layout) reads its 16 scores, masks, keeps the
//    row's running max m and sum l in registers, raises m only when a score exceeds
//    it by more than 2^8 (exact: the output is normalised by a sum taken with the
//    same max), and writes P = 2^(s - m) to TMEM as bf16 hi + lo parts (P = hi + lo
//    to 2^-16), double-buffered.
//  * Values: O_h[64 rows][128 dims] += P_hi . V_h + P_lo . V_h (M = 64, N = 128,
//    K = 16 tokens, A from TMEM, B the stage's V tile), accumulated across the
//    segment. In a sequence's last block the rows of slots past the context are
//    cleared first (the pool may hold anything there, NaN included).
//  * A segment's end: the row's thread reads its O_h row, divides by l and writes
//    the output (whole sequence in the cell), or the partial (m, l, acc) the merge
//    kernel folds.
//
// Warps: 0 produces (TMA), 1 issues the MMAs (one lane) and owns the TMEM
// allocation, 2-5 run the softmax and epilogue of the group's first head, 6-9 of
// its second. Every mbarrier wait is bounded (2 s); on a timeout a warp records the
// error and leaves its loop, and the MMA issuer waits for its last MMAs before the
// CTA tears down.
#include <cuda_bf16.h>

#include <climits>

#include "pkv_cells.cuh"
#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_umma.cuh"

namespace pkv {

namespace {

struct UHdr {
    int32_t q0;     // the sequence's first query row
    int32_t b;      // logical block within the sequence
    int32_t T;      // context length (clamped)
    int32_t hg;     // head group
    int32_t flags;  // F_*
    int32_t slot;   // partial slot: 0 if the segment opens its cell, else 1
    int32_t cell;   // cell holding this block
    int16_t ql;     // the sequence's query rows
    int16_t W;      // mask window: per-row masks rule the last W positions
};
static_assert(sizeof(UHdr) == 32, "stage header");

constexpr int kHG = 2;                      // kv heads per CTA (a head group)
constexpr int kM = 64;                      // MMA rows: up to 64 query rows per kv head
constexpr uint32_t kQHead = kM * 256;       // Q of one head: [2 halves][64 rows][128 B]
constexpr uint32_t kStageBytes = kHG * 8192;
constexpr float kLazyLog2 = 8.f;            // raise the running max past a 2^8 lead
// Blocks are scored, exponentiated and multiplied in groups of up to two
// consecutive blocks of a segment; a group's last block carries kGroupEnd.
constexpr int kNBG = 2;
constexpr int32_t kGroupEnd = 64;
// TMEM columns of head h: S [2 groups][2 blocks][16], P [2 groups][2 blocks]
// [hi 8 | lo 8], O [128]
constexpr uint32_t kColsHead = 256;
constexpr uint32_t kNCols = 512;
__host__ __device__ constexpr uint32_t col_s(int h, int g, int k) { return uint32_t(h) * kColsHead + uint32_t(g * kNBG + k) * 16; }
__host__ __device__ constexpr uint32_t col_p(int h, int g, int k) { return uint32_t(h) * kColsHead + 64 + uint32_t(g * kNBG + k) * 16; }
__host__ __device__ constexpr uint32_t col_o(int h) { return uint32_t(h) * kColsHead + 128; }

// Shared memory: NS stages, the group's Q, the stage headers and the barriers.
struct USmem {
    uint8_t *base;
    int ns;
    UHdr *hdr;
    uint64_t *bar;
    uint32_t *tslot;
    __device__ uint8_t *stage(int i) const { return base + uint32_t(i) * kStageBytes; }
    __device__ uint8_t *q(int h) const { return base + uint32_t(ns) * kStageBytes + uint32_t(h) * kQHead; }
    __device__ uint32_t full(int i) const { return smem_u32(bar + i); }
    __device__ uint32_t empty(int i) const { return smem_u32(bar + ns + i); }
    __device__ uint32_t q_full() const { return smem_u32(bar + 2 * ns); }
    __device__ uint32_t q_free() const { return smem_u32(bar + 2 * ns + 1); }
    __device__ uint32_t s_full(int b) const { return smem_u32(bar + 2 * ns + 2 + b); }
    __device__ uint32_t s_free(int b) const { return smem_u32(bar + 2 * ns + 4 + b); }
    __device__ uint32_t p_full(int b) const { return smem_u32(bar + 2 * ns + 6 + b); }
    __device__ uint32_t p_free(int b) const { return smem_u32(bar + 2 * ns + 8 + b); }
    __device__ uint32_t o_free() const { return smem_u32(bar + 2 * ns + 10); }
    __device__ uint32_t done() const { return smem_u32(bar + 2 * ns + 11); }
};
constexpr int kBarsFixed = 12;

__host__ __device__ constexpr uint32_t umma_smem_bytes_ns(int ns)
{
    return uint32_t(ns) * kStageBytes + kHG * kQHead + uint32_t(ns) * 32 +
           uint32_t(2 * ns + kBarsFixed) * 8 + 16 + 1024;  // + base alignment
}

__device__ __forceinline__ USmem ucarve(uint8_t *raw, int ns)
{
    USmem s;
    s.base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.ns = ns;
    s.hdr = reinterpret_cast<UHdr *>(s.base + uint32_t(ns) * kStageBytes + kHG * kQHead);
    s.bar = reinterpret_cast<uint64_t *>(s.hdr + ns);
    s.tslot = reinterpret_cast<uint32_t *>(s.bar + 2 * ns + kBarsFixed);
    return s;
}

// ------------------------------------------------------------------ producer
// Walks the CTA's cell like paged_decode.cu's producer: per block one TMA box of K
// and one of V for the group's two heads (or per-tile boxes when the driver refuses
// the whole-block map), and at every segment's start the segment's query rows for
// both heads, once the previous segment's scores have read the single Q buffer.
__device__ void producer_umma(const CUtensorMap *kmap, const CUtensorMap *vmap,
                              const CUtensorMap *qmap, const DecodeParams &p, const USmem &sm,
                              int lane)
{
    const unsigned FULLMASK = 0xffffffffu;
    const int S = p.S, NS = sm.ns;

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
    const Cells Cc = make_cells(p, nb_total, int(gridDim.x));
    if (blockIdx.x == 0 && lane == 0) {
        // for the merge: the unit count, and whether every cell holds units
        p.ws[kWsUnits] = uint32_t(nb_total);
        p.ws[kWsDense] = Cc.F1 >= Cc.G ? 1u : 0u;
    }

    uint32_t st = 0, phase = 0, issued = 0;
    int segs = 0;  // segments started (the Q buffer's uses)
    bool ok = true;
    const uint64_t pol = policy_evict_first();
    const uint32_t qbytes = uint32_t(2 * 128 * p.G * p.nq);  // both halves of one head

    const int64_t cell = blockIdx.x;
    const int64_t a = Cc.start(cell), e = Cc.start(cell + 1);
    if (a < e) {
        // locate unit a: head group, sequence and block within it
        const int hg0 = int(a / nb_total);
        const int r0 = int(a - int64_t(hg0) * nb_total);
        const unsigned own = __ballot_sync(FULLMASK, local > 0 && r0 >= base && r0 < base + local);
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
        int hg = hg0;
        int s = __shfl_sync(FULLMASK, s_f, src);
        SeqInfo si = seq_info(p, s);
        int b = __shfl_sync(FULLMASK, b_f, src) + si.b0;
        int b_end = si.b0 + si.nb;
        int seg_b0 = b;
        bool cell_first = true;
        int bt_base = -(1 << 30), bt_val = 0;
        for (int64_t u = a; u < e; ++u) {
            if (b < bt_base || b >= bt_base + 32) {
                bt_base = b;
                const int idx = b + lane;
                bt_val = idx < b_end ? __ldg(p.block_tables + int64_t(si.tr) * p.MB + idx) : 0;
            }
            int phys = __shfl_sync(FULLMASK, bt_val, b - bt_base);
            if (phys < 0 || int64_t(phys) >= p.num_blocks) {
                // read past the pool's end: zeros, and flagged
                if (lane == 0)
                    atomicOr(p.ws + kWsErr, kErrBadBlock);
                phys = int(p.num_blocks < 0x7fffffff ? p.num_blocks : 0x7fffffff);
            }
            const bool first = (u == a) || (b == si.b0);
            if (first)
                seg_b0 = b;
            const bool last = (u == e - 1) || (b == b_end - 1);
            int w_ok = 1;
            if (lane == 0) {
                if (issued >= uint32_t(NS))
                    w_ok = mbar_wait(sm.empty(int(st)), phase ^ 1u, kWaitLimitNs);
                if (w_ok && first)  // the previous segment's scores have read Q
                    w_ok = mbar_wait(sm.q_free(), uint32_t(segs & 1) ^ 1u, kWaitLimitNs);
            }
            if (!__shfl_sync(FULLMASK, w_ok, 0)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                // the merge's record: cell (and slot) of the sequence's first piece,
                // cell of its last
                int2 *rec = p.pieces + int64_t(s) * p.n_hg + hg;
                if (b == si.b0)
                    rec->x = int(cell) * 2 + (cell_first ? 0 : 1);
                if (b == b_end - 1)
                    rec->y = int(cell);
                UHdr *h = &sm.hdr[st];
                h->q0 = si.q0;
                h->b = b;
                h->T = si.T;
                h->hg = hg;
                h->flags = (first ? F_FIRST : 0) | (last ? F_LAST : 0) |
                           (last && seg_b0 == si.b0 && b == b_end - 1 ? F_DIRECT : 0) |
                           (last || ((b - seg_b0) % kNBG) == kNBG - 1 ? kGroupEnd : 0);
                h->slot = cell_first ? 0 : 1;
                h->cell = int(cell);
                h->ql = int16_t(si.ql);
                h->W = int16_t(si.W);
                if (first) {
                    // the segment's query rows [j][g] of both heads, both 64-dim halves
                    mbar_arrive_expect_tx(sm.q_full(), kHG * qbytes);
                    for (int hl = 0; hl < kHG; ++hl)
                        for (int hf = 0; hf < 2; ++hf)
                            tma_load_5d(smem_u32(sm.q(hl)) + uint32_t(hf) * (kM * 128), qmap,
                                        sm.q_full(), 0, hf, (hg * kHG + hl) * p.G, si.q0, 0);
                }
                const uint32_t bar = sm.full(int(st));
                mbar_arrive_expect_tx(bar, kStageBytes);
                const uint32_t kdst = smem_u32(sm.stage(int(st)));
                const uint32_t vdst = kdst + kStageBytes / 2;
                if (p.whole_box) {
                    // map dims (d, token, half, head, block): one box = the group's 2
                    // heads x 16 rows
                    tma_load_5d_hint(kdst, kmap, bar, 0, 0, 0, hg * kHG, phys, pol);
                    tma_load_5d_hint(vdst, vmap, bar, 0, 0, 0, hg * kHG, phys, pol);
                } else {
                    // map dims (d, half, head, token, block): one box = one (head, half)
                    for (int hl = 0; hl < kHG; ++hl)
                        for (int hf = 0; hf < 2; ++hf) {
                            const uint32_t off = uint32_t((hl * 2 + hf) * kTileBytes);
                            tma_load_5d_hint(kdst + off, kmap, bar, 0, hf, hg * kHG + hl, 0, phys,
                                             pol);
                            tma_load_5d_hint(vdst + off, vmap, bar, 0, hf, hg * kHG + hl, 0, phys,
                                             pol);
                        }
                }
            }
            __syncwarp();
            if (first)
                ++segs;
            ++issued;
            if (++st == uint32_t(NS)) {
                st = 0;
                phase ^= 1u;
            }
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
    }

    if (ok) {
        // end-of-work marker (no bytes: a plain arrival)
        int w_ok = 1;
        if (lane == 0 && issued >= uint32_t(NS))
            w_ok = mbar_wait(sm.empty(int(st)), phase ^ 1u, kWaitLimitNs);
        ok = __shfl_sync(FULLMASK, w_ok, 0) != 0;
        if (ok && lane == 0) {
            sm.hdr[st].flags = F_END;
            mbar_arrive(sm.full(int(st)));
        }
    }
    if (!ok && lane == 0) {
        atomicOr(p.ws + kWsErr, kErrProducerWait);
        // wait (bounded) for every copy this warp may still have in flight
        const uint32_t n = issued < uint32_t(NS) ? issued : uint32_t(NS);
        for (uint32_t k = 0; k < n; ++k) {
            uint32_t ps = st, pp = phase;
            for (uint32_t back = 0; back <= k; ++back) {
                if (ps == 0) {
                    ps = uint32_t(NS) - 1;
                    pp ^= 1u;
                } else {
                    --ps;
                }
            }
            if (!mbar_wait(sm.full(int(ps)), pp, kWaitLimitNs))
                atomicOr(p.ws + kWsErr, kErrDrainWait);
        }
        if (segs > 0 && !mbar_wait(sm.q_full(), uint32_t((segs - 1) & 1), kWaitLimitNs))
            atomicOr(p.ws + kWsErr, kErrDrainWait);
    }
}

// ------------------------------------------------------------------ MMA issue
// One thread issues, in order of readiness, the scores of the next block (once its
// tiles and, for a segment's first, the queries have landed and, for a group's
// first, the group's S buffer is free) and the values of the oldest scored group
// (once both heads' P of it is in TMEM): neither waits for the other's inputs.
// Polls never suspend the thread.
__device__ void mma_umma(const DecodeParams &p, const USmem &sm, uint32_t tmem)
{
    const int NS = sm.ns;
    constexpr uint32_t kIdS = umma_idesc_bf16(kM, 16, false, false);   // Q, K: K-major
    constexpr uint32_t kIdO = umma_idesc_bf16(kM, 128, false, true);   // P (TMEM), V: MN-major
    // descriptors at the tiles' starts; a step adds its byte offset >> 4 (no field
    // carries: every tile lies below 256 KiB)
    const uint64_t d_k0 = umma_sdesc(smem_u32(sm.stage(0)), 16, 1024, kSw128);
    const uint64_t d_v0 = umma_sdesc(smem_u32(sm.stage(0)) + kStageBytes / 2, 2048, 1024, kSw128);
    const uint64_t d_q0 = umma_sdesc(smem_u32(sm.q(0)), 16, 1024, kSw128);
    constexpr uint64_t kStageStep = kStageBytes >> 4;

    uint32_t nb = 0;            // blocks scored
    uint32_t gs = 0, kk_s = 0;  // groups whose scoring started; blocks of the open one
    uint32_t gpv = 0;           // groups whose values are issued
    int segs = -1;              // segments scored
    // per group buffer (parity): its stages, block count, segment, and whether it
    // opens its segment
    int g_st[2][kNBG] = {}, g_n[2] = {}, g_seg[2] = {};
    bool g_first[2] = {};
    bool end_seen = false, ok = true;
    uint64_t t_idle = 0;
    while (ok && !(end_seen && gpv == gs && kk_s == 0)) {
        bool progressed = false;
        // ---- scores of block nb: S_h = Q_h . K_h^T over the 8 16-dim steps
        if (!end_seen && (kk_s > 0 || gs - gpv < 2)) {
            const int st = int(nb % uint32_t(NS));
            if (mbar_test_wait(sm.full(st), (nb / uint32_t(NS)) & 1u)) {
                const UHdr h = sm.hdr[st];
                if (h.flags & F_END) {
                    end_seen = true;
                    progressed = true;
                } else {
                    const bool first = (h.flags & F_FIRST) != 0;
                    const int g = first ? segs + 1 : segs;
                    const uint32_t gb = gs & 1u;
                    if ((kk_s > 0 || mbar_test_wait(sm.s_free(int(gb)), ((gs >> 1) & 1u) ^ 1u)) &&
                        (!first || mbar_test_wait(sm.q_full(), uint32_t(g & 1)))) {
                        tc_fence_after();
                        segs = g;
                        const uint64_t dk = d_k0 + uint64_t(st) * kStageStep;
#pragma unroll
                        for (int hl = 0; hl < kHG; ++hl) {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                // K tile of head hl: [half][16 tokens][64], 4 KiB a head
                                const uint64_t ko = uint64_t(hl * 4096 + (kk >> 2) * 2048 +
                                                             (kk & 3) * 32) >> 4;
                                const uint64_t qo = uint64_t(hl * kQHead + (kk >> 2) * (kM * 128) +
                                                             (kk & 3) * 32) >> 4;
                                umma_bf16(tmem + col_s(hl, int(gb), int(kk_s)), d_q0 + qo, dk + ko,
                                          kIdS, kk > 0);
                            }
                        }
                        if (h.flags & F_LAST)
                            umma_commit(sm.q_free());  // the segment's Q is read
                        if (kk_s == 0) {
                            g_first[gb] = first;
                            g_seg[gb] = g;
                        }
                        g_st[gb][kk_s] = st;
                        ++kk_s;
                        ++nb;
                        if (h.flags & kGroupEnd) {
                            umma_commit(sm.s_full(int(gb)));
                            g_n[gb] = int(kk_s);
                            kk_s = 0;
                            ++gs;
                        }
                        progressed = true;
                    }
                }
            }
        }
        // ---- values of group gpv: O_h += P_hi . V_h + P_lo . V_h, block by block
        const uint32_t pb = gpv & 1u;
        if (gpv < gs && mbar_test_wait(sm.p_full(int(pb)), (gpv >> 1) & 1u) &&
            (!g_first[pb] || mbar_test_wait(sm.o_free(), uint32_t(g_seg[pb] & 1) ^ 1u))) {
            tc_fence_after();
            for (int k = 0; k < g_n[pb]; ++k) {
                const int st = g_st[pb][k];
                const uint64_t dv = d_v0 + uint64_t(st) * kStageStep;
#pragma unroll
                for (int hl = 0; hl < kHG; ++hl) {
                    const uint64_t dvh = dv + uint64_t(hl * 4096 >> 4);
                    const uint32_t pc = tmem + col_p(hl, int(pb), k);
                    umma_bf16_tmem_a(tmem + col_o(hl), pc, dvh, kIdO, !(g_first[pb] && k == 0));
                    umma_bf16_tmem_a(tmem + col_o(hl), pc + 8, dvh, kIdO, true);
                }
                umma_commit(sm.empty(st));
            }
            umma_commit(sm.p_free(int(pb)));
            ++gpv;
            progressed = true;
        }
        if (progressed) {
            t_idle = 0;
        } else if (t_idle == 0) {
            t_idle = global_timer_ns();
        } else if (global_timer_ns() - t_idle > kWaitLimitNs) {
            atomicOr(p.ws + kWsErr, kErrConsumerWait);
            ok = false;
        }
    }
    // every MMA issued has completed before the CTA tears down
    umma_commit(sm.done());
    if (!mbar_wait(sm.done(), 0, kWaitLimitNs))
        atomicOr(p.ws + kWsErr, kErrDrainWait);
}

// ------------------------------------------------------------------ softmax + epilogue
// Warp `warp` (2..9) serves head hl = (warp - 2) / 4 of the group; its lanes 0..15
// own rows 16 * (warp % 4) + lane (the M = 64 TMEM data-path layout); lanes 16..31
// take part in the warp-wide TMEM accesses only.
__device__ void softmax_umma(const DecodeParams &p, const USmem &sm, uint32_t tmem, int warp,
                             int lane)
{
    const int NS = sm.ns;
    const int hl = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = 16 * q4 + (lane & 15);  // the row (lanes >= 16: a copy of lane - 16's)
    const bool row_lane = lane < 16;
    const uint32_t lane_base = tmem + (uint32_t(q4 * 32) << 16);
    float m = -INFINITY, l = 0.f;
    bool wait_ok = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!mbar_wait(bar, parity, kWaitLimitNs) && wait_ok) {
            if (lane == 0)
                atomicOr(p.ws + kWsErr, kErrConsumerWait);
            wait_ok = false;
        }
        return wait_ok;
    };

    uint32_t i = 0;  // blocks consumed
    for (uint32_t g = 0;; ++g) {
        const uint32_t gb = g & 1u;
        // the group's blocks (one or two) and their headers
        int stk[kNBG];
        UHdr hk[kNBG];
        int n = 0;
        bool end = false;
        for (; n < kNBG; ++n) {
            const uint32_t bi = i + uint32_t(n);
            stk[n] = int(bi % uint32_t(NS));
            if (!wait(sm.full(stk[n]), (bi / uint32_t(NS)) & 1u)) {
                end = true;
                break;
            }
            hk[n] = sm.hdr[stk[n]];
            if (hk[n].flags & F_END) {
                end = true;
                break;
            }
            if (hk[n].flags & kGroupEnd) {
                ++n;
                break;
            }
        }
        if (end)
            break;
        const UHdr &h = hk[0];
        const UHdr &hl_last = hk[n - 1];
        const int kvh = h.hg * kHG + hl;
        if (!wait(sm.s_full(int(gb)), (g >> 1) & 1u))
            break;
        tc_fence_after();
        float x[32];
        tmem_ld32<0>(lane_base + col_s(hl, int(gb), 0), x);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(sm.s_free(int(gb)));
        const bool first = (h.flags & F_FIRST) != 0;
        if (first) {
            m = -INFINITY;
            l = 0.f;
        }
        // scale (log2 domain); tokens past the context, and positions the row does
        // not see, are masked
        int j = r / p.G;
        j = j < h.ql ? j : h.ql - 1;  // padding rows: the last query's rule
        const int w0 = p.tree_mask ? h.T - h.W : h.T - h.ql + 1;
        const int t_end = hk[n - 1].b * kBlockSize + kBlockSize;  // one past the group's tokens
        const bool masked_group = t_end - 1 >= w0;
        uint32_t bits = 0u;
        if (masked_group && p.tree_mask)
            bits = __ldg(p.tree_mask + h.q0 + j);
        float bm = -INFINITY;
#pragma unroll
        for (int k = 0; k < kNBG; ++k) {
            const int t0 = (k < n ? hk[k].b : 0) * kBlockSize;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int tok = t0 + c;
                bool vis = k < n && tok < h.T;
                if (masked_group && tok >= w0)
                    vis = vis && (p.tree_mask ? ((bits >> (tok - w0)) & 1u) != 0u
                                              : tok <= h.T - h.ql + j);
                float &v = x[16 * k + c];
                v = vis ? v * p.scale_log2 : -INFINITY;
                bm = fmaxf(bm, v);
            }
        }
        // raise the running max (the first group always sets it); an accumulator
        // holding earlier groups of the segment is rescaled by the same factor, once
        // the previous group's P.V has landed
        const bool need = bm > m + kLazyLog2 || (first && bm > m);
        float f = 1.f;
        if (need) {
            f = ex2(m - bm);  // 0 from -inf
            m = bm;
            l *= f;
        }
        if (__any_sync(0xffffffffu, need && row_lane && !first)) {
            if (g > 0)
                wait(sm.p_free(int((g - 1) & 1u)), ((g - 1) >> 1) & 1u);
            tc_fence_after();
            const uint32_t oc = lane_base + col_o(hl);
#pragma unroll 1
            for (int c32 = 0; c32 < 4; ++c32) {
                float o[32];
                tmem_ld32<0>(oc + 32 * c32, o);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    o[k] *= f;
                tmem_st32<0>(oc + 32 * c32, o);
                tmem_wait_st();
            }
        }
        // P = 2^(x - m) as bf16 hi + lo, block by block
        const float mu = m == -INFINITY ? 0.f : m;
        uint32_t phi[kNBG][8], plo[kNBG][8];
#pragma unroll
        for (int k = 0; k < kNBG; ++k)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float a0 = ex2(x[16 * k + 2 * c] - mu), a1 = ex2(x[16 * k + 2 * c + 1] - mu);
                l += a0 + a1;
                phi[k][c] = pack_bf16x2(a0, a1);
                plo[k][c] = pack_bf16x2(a0 - bf16lo_f32(phi[k][c]), a1 - bf16hi_f32(phi[k][c]));
            }
        if (g >= 2)  // the group two back has read this P buffer
            wait(sm.p_free(int(gb)), ((g - 2) >> 1) & 1u);
#pragma unroll
        for (int k = 0; k < kNBG; ++k) {
            if (k < n) {
                tmem_st8(lane_base + col_p(hl, int(gb), k), phi[k]);
                tmem_st8(lane_base + col_p(hl, int(gb), k) + 8, plo[k]);
            }
        }
        const int vc = h.T - hk[n - 1].b * kBlockSize;  // tokens of the last block in context
        if (__builtin_expect(vc < kBlockSize, 0)) {
            // the sequence's last block: its slots past the context (stale, or NaN)
            // must not reach P.V even times a zero weight. The head's 4 warps clear
            // those rows of its V tile (both halves; whole rows, so the swizzle does
            // not matter) and fence the writes for the tensor cores.
            uint8_t *vt = sm.stage(stk[n - 1]) + kStageBytes / 2 + uint32_t(hl) * 4096u;
            for (int k = q4 * 32 + lane; k < (kBlockSize - vc) * 16; k += 128) {
                const int row = vc + (k >> 4), c = k & 15;
                *reinterpret_cast<uint4 *>(vt + (c >> 3) * 2048 + row * 128 + (c & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(sm.p_full(int(gb)));
        i += uint32_t(n);

        if (hl_last.flags & F_LAST) {
            // ---- the segment's end: this row of O_h, over the row sum
            wait(sm.p_free(int(gb)), (g >> 1) & 1u);
            tc_fence_after();
            const UHdr &he = hl_last;
            const int rows_v = p.G * he.ql;
            const bool live = row_lane && r < rows_v;
            const int jr = r / p.G;
            const int64_t cb = int64_t(he.cell) * 2 + he.slot;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t orow = (int64_t(he.q0) + jr) * p.Hq + int64_t(kvh) * p.G + (r - jr * p.G);
            const int64_t prow = (cb * p.HG + hl) * p.rows + r;
            const uint32_t oc = lane_base + col_o(hl);
#pragma unroll 1
            for (int c32 = 0; c32 < 4; ++c32) {
                float o[32];
                tmem_ld32<0>(oc + 32 * c32, o);
                tmem_wait_ld();
                if (!live)
                    continue;
                if (he.flags & F_DIRECT) {
                    if (p.out_f32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) +
                                                                 orow * 128 + 32 * c32);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            dst[k] = make_float4(o[4 * k] * inv, o[4 * k + 1] * inv,
                                                 o[4 * k + 2] * inv, o[4 * k + 3] * inv);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            static_cast<__nv_bfloat16 *>(p.out) + orow * 128 + 32 * c32);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            dst[k] = make_uint4(pack_bf16x2(o[8 * k] * inv, o[8 * k + 1] * inv),
                                                pack_bf16x2(o[8 * k + 2] * inv, o[8 * k + 3] * inv),
                                                pack_bf16x2(o[8 * k + 4] * inv, o[8 * k + 5] * inv),
                                                pack_bf16x2(o[8 * k + 6] * inv, o[8 * k + 7] * inv));
                    }
                } else {
                    // partial (m, l, acc) of this cell for the merge kernel
                    float4 *dst = reinterpret_cast<float4 *>(p.part + prow * 128 + 32 * c32);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                }
            }
            if (live && !(he.flags & F_DIRECT)) {
                p.ml[prow * 2] = m;
                p.ml[prow * 2 + 1] = l;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(sm.o_free());
        }
    }
}

}  // namespace

__global__ void __launch_bounds__(320, 1)
    paged_decode_umma_kernel(const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap,
                             const __grid_constant__ CUtensorMap qmap, const DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const USmem sm = ucarve(smem_raw, p.nst);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        tma_prefetch_desc(&qmap);
        for (int i = 0; i < sm.ns; ++i) {
            mbar_init(sm.full(i), 1);
            mbar_init(sm.empty(i), 1);
        }
        mbar_init(sm.q_full(), 1);
        mbar_init(sm.q_free(), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.s_full(b), 1);
            mbar_init(sm.s_free(b), 8);
            mbar_init(sm.p_full(b), 8);
            mbar_init(sm.p_free(b), 1);
        }
        mbar_init(sm.o_free(), 8);
        mbar_init(sm.done(), 1);
        fence_mbar_init();
    }
    // Q rows past a segment's G * nq (padding up to 64) are never written by the
    // copies: they hold zeros so the padding scores stay finite
    for (uint32_t i = threadIdx.x; i < kHG * kQHead / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(sm.q(0))[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (warp == 1)
        tmem_alloc(smem_u32(sm.tslot), kNCols);
    // the previous kernel on the stream (e.g. the KV append) has finished writing
    asm volatile("griddepcontrol.wait;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tslot;
    if (warp == 0) {
        producer_umma(&kmap, &vmap, &qmap, p, sm, lane);
    } else if (warp == 1) {
        if (lane == 0)
            mma_umma(p, sm, tmem);
        __syncwarp();
    } else {
        softmax_umma(p, sm, tmem, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kNCols);
    }
}

size_t umma_smem_bytes(int ns) { return umma_smem_bytes_ns(ns); }

int umma_max_stages(int smem_optin)
{
    int ns = 2;
    while (ns < 16 && int(umma_smem_bytes_ns(ns + 1)) <= smem_optin)
        ++ns;
    return int(umma_smem_bytes_ns(ns)) <= smem_optin ? ns : 0;
}

cudaError_t launch_decode_umma(const DecodePlan &pl, const DecodeParams &p,
                               const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const CUtensorMap &qmap, cudaStream_t stream, cudaEvent_t ev_before,
                               cudaEvent_t ev_after)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && configured[dev] < int(pl.smem)) {
        e = cudaFuncSetAttribute(paged_decode_umma_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem));
        if (e != cudaSuccess)
            return e;
        configured[dev] = int(pl.smem);
    }
    if (ev_before && (e = cudaEventRecord(ev_before, stream)) != cudaSuccess)
        return e;
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
    e = cudaLaunchKernelEx(&cfg, paged_decode_umma_kernel, kmap, vmap, qmap, p);
    if (e != cudaSuccess)
        return e;
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    if (ev_after && (e = cudaEventRecord(ev_after, stream)) != cudaSuccess)
        return e;
    return launch_merge(pl, p, stream);
}

}  // namespace pkv
