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
// Why a second kernel: with G * nq = 32 or more query rows per kv head, the
// legacy warp MMA path spends more issue slots on mma.sync, ldmatrix and the
// register-held accumulators than HBM needs to stream the tiles. Here one thread
// issues whole-tile MMAs from shared memory, the accumulators live in tensor
// memory (TMEM), and the CUDA cores keep only the softmax.
//
// Layout of the work:
//  * The unit space is the one of paged_decode.cu with one kv head per unit (a
//    16-token block of one kv head); each CTA of the persistent grid streams one
//    contiguous cell. A super-stage is up to 8 consecutive blocks of one
//    (sequence, kv head): K and V as [2 halves][128 tokens][64 dims] bf16 tiles in
//    the 128-byte swizzle TMA writes (one 2 KiB box per block, half and tensor).
//  * Scores, tokens on M: S^T[128 tokens][N rows] = K . Q^T (M = 128, N = 32 or
//    64, K = 128 dims) into TMEM; Q [N rows][128 dims] is staged by TMA at the
//    start of every segment (double-buffered).
//  * Softmax: two teams of four warps each own half of the N rows; thread t of a
//    team owns token t: it reads its TMEM row of N/2 scores, masks, exponentiates
//    against a per-row running max that is raised only when a score exceeds it by
//    more than 2^8 (exact: the output is normalised by a sum taken with the same
//    max), and writes its part of the P^T row as a bf16 hi + lo pair (P = hi + lo
//    to 2^-16) to shared memory.
//    Row sums are reduced over each warp's 32 tokens by a butterfly and kept per
//    lane.
//  * Values, d on M: O^T[128 dims][hi | lo] += V^T . [P_hi | P_lo]^T (M = 128,
//    N = 2 x rows, K = 16 tokens per MMA), accumulated in TMEM across the segment.
//  * A segment's end: thread d of a team reads its TMEM rows of O^T (hi + lo),
//    divides by the row sums and writes the output (whole sequence in the cell),
//    or writes the partial (m, l, acc) the merge kernel folds.
//
// Warps: 0 produces (TMA), 1 issues the MMAs (one elected lane) and owns the TMEM
// allocation, 2-9 run the softmax and the epilogue, 10 prefetches the tiles into L2
// ahead of their loads. Every mbarrier wait is bounded
// (2 s); the softmax warps decide to leave their loop only at their per-stage
// named-barrier reduction, so no warp is left waiting on a named barrier.
//
// The kernel is opt-in (PKV_OPT_UMMA = 1): on GB300 the mma.sync kernels run the
// same 32- and 60-row batches faster. The tokens-on-M tile needs a uniform row
// stride across scattered blocks, so the TMA moves one 2 KiB box per (block, half,
// tensor): 32 boxes per super-stage against 2 for the mma.sync kernel's whole-block
// boxes, and each super-stage's softmax and values MMAs form one serial chain.
#include <cuda_bf16.h>

#include <climits>

#include "pkv_cells.cuh"
#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_umma.cuh"

namespace pkv {

namespace {

// One super-stage: up to 8 consecutive blocks of one (sequence, kv head).
struct UHdr {
    int32_t q0;     // the sequence's first query row
    int32_t b0;     // logical block of the stage's first token row
    int32_t T;      // context length (clamped)
    int32_t head;   // kv head
    int32_t flags;  // F_*
    int32_t cell;   // cell holding the stage (and the partial slot in bit 0 of `slot`)
    int16_t ql;     // the sequence's query rows
    int16_t W;      // mask window: per-row masks rule the last W positions
    int8_t nbv;     // blocks filled (1..8)
    int8_t qb;      // Q buffer of the segment
    int8_t slot;    // partial slot: 0 if the segment opens its cell, else 1
    int8_t pad;
};
static_assert(sizeof(UHdr) == 32, "super-stage header");

constexpr int kSsBlocks = 8;                 // blocks per super-stage (M = 128 tokens)
constexpr uint32_t kSsBytes = 65536;         // K [2][128][128 B] + V [2][128][128 B]
constexpr uint32_t kHalfBytes = 16384;       // one 64-dim half of 128 token rows
constexpr float kLazyLog2 = 8.f;             // raise the running max past a 2^8 lead

template <int N>
struct UCfg {
    static constexpr int NS = N == 32 ? 3 : 2;      // super-stages in flight
    static constexpr uint32_t QBUF = N * 256;        // [2 halves][N rows][128 B]
    // P^T [128 tokens][2N] bf16: the hi parts of the N rows, then their lo parts,
    // in MN-major 128-byte-swizzle atoms of 64 elements ([atom][128 tokens][128 B])
    static constexpr uint32_t PBUF = N * 512;
    static constexpr uint32_t P_ATOM = 16384;        // one 64-element atom of 128 token rows
    // TMEM columns: S^T x 2 [0, 2N); O^T hi | lo [2N, 4N)
    static constexpr uint32_t O_COL = 2 * N;
    static constexpr uint32_t NCOLS = 4 * N <= 128 ? 128 : 256;
    static constexpr uint32_t OFF_Q = NS * kSsBytes;
    static constexpr uint32_t OFF_P = OFF_Q + 2 * QBUF;
    // red_m [N][4], red_l [N][4], mrow [N], frow [N]
    static constexpr uint32_t OFF_RED = OFF_P + PBUF;
    static constexpr uint32_t OFF_HDR = OFF_RED + 10 * N * 4;
    // barriers: full[NS], empty[NS], q_full[2], q_free[2], s_full[2], s_free[2],
    // p_full, p_free, o_free, done
    static constexpr int NBAR = 2 * NS + 12;
    static constexpr uint32_t OFF_BAR = OFF_HDR + NS * 32;
    static constexpr uint32_t OFF_TSLOT = OFF_BAR + NBAR * 8;
    static constexpr uint32_t SMEM = OFF_TSLOT + 16 + 1024;  // + base alignment
};

template <int N>
struct USmem {
    uint8_t *base;
    UHdr *hdr;
    uint64_t *bar;
    uint32_t *tslot;
    float *red_m, *red_l, *mrow, *frow;
    volatile int *progress;  // blocks of the cell handed to shared memory (producer -> prefetch)
    __device__ uint8_t *stage(int i) const { return base + uint32_t(i) * kSsBytes; }
    __device__ uint8_t *qbuf(int b) const { return base + UCfg<N>::OFF_Q + uint32_t(b) * UCfg<N>::QBUF; }
    __device__ uint32_t full(int i) const { return smem_u32(bar + i); }
    __device__ uint32_t empty(int i) const { return smem_u32(bar + UCfg<N>::NS + i); }
    __device__ uint32_t q_full(int b) const { return smem_u32(bar + 2 * UCfg<N>::NS + b); }
    __device__ uint32_t q_free(int b) const { return smem_u32(bar + 2 * UCfg<N>::NS + 2 + b); }
    __device__ uint32_t s_full(int b) const { return smem_u32(bar + 2 * UCfg<N>::NS + 4 + b); }
    __device__ uint32_t s_free(int b) const { return smem_u32(bar + 2 * UCfg<N>::NS + 6 + b); }
    __device__ uint32_t p_full() const { return smem_u32(bar + 2 * UCfg<N>::NS + 8); }
    __device__ uint32_t p_free() const { return smem_u32(bar + 2 * UCfg<N>::NS + 9); }
    __device__ uint32_t o_free() const { return smem_u32(bar + 2 * UCfg<N>::NS + 10); }
    __device__ uint32_t done() const { return smem_u32(bar + 2 * UCfg<N>::NS + 11); }
};

template <int N>
__device__ __forceinline__ USmem<N> ucarve(uint8_t *raw)
{
    using C = UCfg<N>;
    USmem<N> s;
    s.base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.hdr = reinterpret_cast<UHdr *>(s.base + C::OFF_HDR);
    s.bar = reinterpret_cast<uint64_t *>(s.base + C::OFF_BAR);
    s.tslot = reinterpret_cast<uint32_t *>(s.base + C::OFF_TSLOT);
    s.progress = reinterpret_cast<volatile int *>(s.tslot + 2);
    float *red = reinterpret_cast<float *>(s.base + C::OFF_RED);
    s.red_m = red;
    s.red_l = red + 4 * N;
    s.mrow = red + 8 * N;
    s.frow = red + 9 * N;
    return s;
}

// ------------------------------------------------------------------ producer
template <int N>
__device__ void producer_umma(const CUtensorMap *kmap, const CUtensorMap *vmap,
                              const CUtensorMap *qmap, const DecodeParams &p, const USmem<N> &sm,
                              int lane)
{
    using C = UCfg<N>;
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
    const Cells Cc = make_cells(p, nb_total, int(gridDim.x));
    if (blockIdx.x == 0 && lane == 0) {
        // for the merge: the unit count, and whether every cell holds units
        p.ws[kWsUnits] = uint32_t(nb_total);
        p.ws[kWsDense] = Cc.F1 >= Cc.G ? 1u : 0u;
    }

    uint32_t st = 0, phase = 0, issued = 0;
    int handed = 0;  // blocks of the cell handed to shared memory so far
    int qseg = 0;    // segments started: Q buffer qseg & 1
    bool ok = true;
    const uint64_t pol = policy_evict_first();
    const uint32_t qbytes = uint32_t(2 * 128 * p.G * p.nq);

    const int64_t cell = blockIdx.x;
    const int64_t a = Cc.start(cell), e = Cc.start(cell + 1);
    if (a < e) {
        // locate unit a: kv head, sequence and block within it
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
        int b = __shfl_sync(FULLMASK, b_f, src);
        SeqInfo si = seq_info(p, s);
        b += si.b0;
        bool cell_first = true;
        for (int64_t u = a; u < e && ok;) {
            const int b_end = si.b0 + si.nb;
            const int64_t left = e - u;
            const int seg_len = int(int64_t(b_end - b) < left ? int64_t(b_end - b) : left);
            const bool seg_direct = b == si.b0 && b + seg_len == b_end;
            if (lane == 0) {
                // the merge's record: cell (and slot) of the sequence's first piece,
                // cell of its last
                int2 *rec = p.pieces + int64_t(s) * p.n_hg + hg;
                if (b == si.b0)
                    rec->x = int(cell) * 2 + (cell_first ? 0 : 1);
                if (b + seg_len == b_end)
                    rec->y = int(cell);
            }
            const int qb = qseg & 1;
            for (int c0 = 0; c0 < seg_len && ok; c0 += kSsBlocks) {
                const int nbv = min(kSsBlocks, seg_len - c0);
                // this chunk's physical block ids (lane j < nbv), loaded before the
                // wait for a free super-stage so the load overlaps it
                int phys = 0;
                if (lane < nbv) {
                    phys = __ldg(p.block_tables + int64_t(si.tr) * p.MB + b + c0 + lane);
                    if (phys < 0 || int64_t(phys) >= p.num_blocks) {
                        // read past the pool's end: zeros, and flagged
                        atomicOr(p.ws + kWsErr, kErrBadBlock);
                        phys = int(p.num_blocks < 0x7fffffff ? p.num_blocks : 0x7fffffff);
                    }
                }
                const bool first = c0 == 0, last = c0 + nbv == seg_len;
                int w_ok = 1;
                if (lane == 0) {
                    if (issued >= uint32_t(C::NS))
                        w_ok = mbar_wait(sm.empty(int(st)), phase ^ 1u, kWaitLimitNs);
                    if (w_ok && first)
                        w_ok = mbar_wait(sm.q_free(qb), uint32_t((qseg >> 1) & 1) ^ 1u, kWaitLimitNs);
                }
                if (!__shfl_sync(FULLMASK, w_ok, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    UHdr *h = &sm.hdr[st];
                    h->q0 = si.q0;
                    h->b0 = b + c0;
                    h->T = si.T;
                    h->head = hg;
                    h->flags = (first ? F_FIRST : 0) | (last ? F_LAST : 0) |
                               (last && seg_direct ? F_DIRECT : 0);
                    h->cell = int(cell);
                    h->ql = int16_t(si.ql);
                    h->W = int16_t(si.W);
                    h->nbv = int8_t(nbv);
                    h->qb = int8_t(qb);
                    h->slot = int8_t(cell_first ? 0 : 1);
                    if (first) {
                        // the segment's query rows [j][g] of both 64-dim halves
                        const uint32_t qbar = sm.q_full(qb);
                        mbar_arrive_expect_tx(qbar, qbytes);
                        const uint32_t qdst = smem_u32(sm.qbuf(qb));
                        tma_load_5d(qdst, qmap, qbar, 0, 0, hg * p.G, si.q0, 0);
                        tma_load_5d(qdst + uint32_t(N * 128), qmap, qbar, 0, 1, hg * p.G, si.q0, 0);
                    }
                    mbar_arrive_expect_tx(sm.full(int(st)), uint32_t(nbv) * 8192u);
                }
                __syncwarp();
                // lane 4j + 2t + h: block j, tensor t (K, V), 64-dim half h
                const int pj = __shfl_sync(FULLMASK, phys, lane >> 2);
                if (lane < 4 * nbv) {
                    const int j = lane >> 2, tv = (lane >> 1) & 1, hf = lane & 1;
                    const uint32_t dst = smem_u32(sm.stage(int(st))) + uint32_t(tv) * 32768u +
                                         uint32_t(hf) * kHalfBytes + uint32_t(j) * 2048u;
                    tma_load_5d_hint(dst, tv ? vmap : kmap, sm.full(int(st)), 0, hf, hg, 0, pj,
                                     pol);
                }
                __syncwarp();
                handed += nbv;
                if (lane == 0)
                    *sm.progress = handed;  // for the L2 prefetch warp
                ++issued;
                if (++st == uint32_t(C::NS)) {
                    st = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            ++qseg;
            cell_first = false;
            u += seg_len;
            b += seg_len;
            if (u < e) {
                // the next sequence (or kv head) with blocks to stream
                do {
                    if (++s == S) {
                        s = 0;
                        ++hg;
                    }
                    si = seq_info(p, s);
                } while (si.nb == 0);
                b = si.b0;
            }
        }
    }

    if (lane == 0)
        *sm.progress = INT_MAX;  // the prefetch warp may finish its walk
    if (ok) {
        // end-of-work marker (no bytes: a plain arrival)
        int w_ok = 1;
        if (lane == 0 && issued >= uint32_t(C::NS))
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
        const uint32_t n = issued < uint32_t(C::NS) ? issued : uint32_t(C::NS);
        for (uint32_t k = 0; k < n; ++k) {
            uint32_t ps = st, pp = phase;
            for (uint32_t back = 0; back <= k; ++back) {
                if (ps == 0) {
                    ps = uint32_t(C::NS) - 1;
                    pp ^= 1u;
                } else {
                    --ps;
                }
            }
            if (!mbar_wait(sm.full(int(ps)), pp, kWaitLimitNs))
                atomicOr(p.ws + kWsErr, kErrDrainWait);
        }
        // and for the last Q copies (each buffer's most recent fill)
        for (int k = 1; k <= 2 && k <= qseg; ++k) {
            const int g = qseg - k;
            if (!mbar_wait(sm.q_full(g & 1), uint32_t((g >> 1) & 1), kWaitLimitNs))
                atomicOr(p.ws + kWsErr, kErrDrainWait);
        }
    }
}

// ------------------------------------------------------------------ L2 prefetch
// Walks the same units as the producer, in the same order, and prefetches each
// block's K and V tiles into L2 (no shared memory, no completion) while keeping
// at most p.pf_units blocks ahead of the blocks the producer has handed to shared
// memory: the super-stages' loads then meet L2 latency rather than DRAM latency,
// so the few 64 KiB super-stages shared memory holds suffice. A hint only: a
// prefetch that is late, early or skipped changes no result.
template <int N>
__device__ void prefetch_umma(const CUtensorMap *kmap, const CUtensorMap *vmap,
                              const DecodeParams &p, const USmem<N> &sm, int lane)
{
    const unsigned FULLMASK = 0xffffffffu;
    const int S = p.S;
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
    const int64_t a = Cc.start(blockIdx.x), e = Cc.start(blockIdx.x + 1);
    if (a >= e || p.pf_units <= 0)
        return;
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
    int64_t u = a;
    uint64_t t0 = 0;
    while (u < e) {
        // stay within p.pf_units blocks of what the producer has handed over
        const int done = *sm.progress;
        if (int64_t(done) + p.pf_units <= u - a) {
            if (t0 == 0)
                t0 = global_timer_ns();
            else if (global_timer_ns() - t0 > kWaitLimitNs)
                return;  // the producer stopped: nothing left worth prefetching
            __nanosleep(256);
            continue;
        }
        t0 = 0;
        const int b_end = si.b0 + si.nb;
        const int64_t left = e - u;
        const int n0 = min(kSsBlocks, b_end - b);
        const int n = int64_t(n0) < left ? n0 : int(left);
        if (lane < 4 * n) {  // lane 4j + 2t + h: block j, tensor t, half h
            const int phys = __ldg(p.block_tables + int64_t(si.tr) * p.MB + b + (lane >> 2));
            if (phys >= 0 && int64_t(phys) < p.num_blocks)
                tma_prefetch_l2_5d((lane >> 1) & 1 ? vmap : kmap, 0, lane & 1, hg, 0, phys);
        }
        u += n;
        b += n;
        if (b == b_end && u < e) {
            do {
                if (++s == S) {
                    s = 0;
                    ++hg;
                }
                si = seq_info(p, s);
            } while (si.nb == 0);
            b = si.b0;
        }
    }
}

// ------------------------------------------------------------------ MMA issue
// One thread issues, in order of readiness, the scores of the next super-stage
// (once its tiles and, for a segment's first, its queries have landed and the S^T
// buffer is free) and the values of the oldest scored super-stage (once its P^T
// is written): neither waits for the other's inputs.
template <int N>
__device__ void mma_umma(const DecodeParams &p, const USmem<N> &sm, uint32_t tmem)
{
    using C = UCfg<N>;
    constexpr uint32_t kIdS = umma_idesc_bf16(128, N, false, false);       // K, Q: K-major
    constexpr uint32_t kIdO = umma_idesc_bf16(128, 2 * N, true, true);     // V^T, P^T: MN-major
    const uint32_t o_col = tmem + C::O_COL;
    // descriptors at the tiles' starts; a step adds its byte offset >> 4 (no field
    // carries: every tile lies below 256 KiB)
    const uint64_t d_p = umma_sdesc(smem_u32(sm.base + C::OFF_P), N == 32 ? 1024 : C::P_ATOM,
                                    1024, kSw128);
    const uint64_t d_v0 = umma_sdesc(smem_u32(sm.stage(0)) + 32768u, kHalfBytes, 1024, kSw128);
    const uint64_t d_k0 = umma_sdesc(smem_u32(sm.stage(0)), 16, 1024, kSw128);
    const uint64_t d_q0 = umma_sdesc(smem_u32(sm.qbuf(0)), 16, 1024, kSw128);
    constexpr uint64_t kStageStep = kSsBytes >> 4, kQStep = C::QBUF >> 4;

    uint32_t ns = 0, npv = 0;   // super-stages scored, and whose values are issued
    int g_s = -1;               // segment of the last scored super-stage
    // segment of, and whether it opens its segment, the (at most two) scored
    // super-stages npv .. ns - 1, by parity
    int seg_even = 0, seg_odd = 0;
    uint32_t first_of = 0;      // bit k & 1: super-stage k opens its segment
    bool end_seen = false, ok = true;
    uint64_t t_idle = 0;
    while (ok && !(end_seen && npv == ns)) {
        bool progressed = false;
        // ---- scores of super-stage ns
        if (!end_seen && ns - npv < 2) {
            const int st = int(ns % uint32_t(C::NS));
            if (mbar_test_wait(sm.full(st), (ns / uint32_t(C::NS)) & 1u)) {
                const UHdr h = sm.hdr[st];
                if (h.flags & F_END) {
                    end_seen = true;
                    progressed = true;
                } else {
                    const bool first = (h.flags & F_FIRST) != 0;
                    const int g = first ? g_s + 1 : g_s;
                    const uint32_t bsel = ns & 1u;
                    if ((!first || mbar_test_wait(sm.q_full(g & 1), uint32_t((g >> 1) & 1))) &&
                        mbar_test_wait(sm.s_free(int(bsel)), ((ns >> 1) & 1u) ^ 1u)) {
                        tc_fence_after();
                        g_s = g;
                        const uint64_t dk = d_k0 + uint64_t(st) * kStageStep;
                        const uint64_t dq = d_q0 + uint64_t(g & 1) * kQStep;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t ko = uint64_t((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                            const uint64_t qo = uint64_t((kk >> 2) * (N * 128) + (kk & 3) * 32) >> 4;
                            umma_bf16(tmem + bsel * N, dk + ko, dq + qo, kIdS, kk > 0);
                        }
                        umma_commit(sm.s_full(int(bsel)));
                        if (h.flags & F_LAST)
                            umma_commit(sm.q_free(g & 1));  // the segment's Q is read
                        if (ns & 1u)
                            seg_odd = g;
                        else
                            seg_even = g;
                        first_of = (first_of & ~(1u << (ns & 1u))) | (uint32_t(first) << (ns & 1u));
                        ++ns;
                        progressed = true;
                    }
                }
            }
        }
        // ---- values and row sums of super-stage npv
        if (npv < ns && mbar_test_wait(sm.p_full(), npv & 1u)) {
            const bool seg_first = (first_of >> (npv & 1u)) & 1u;
            const int g = (npv & 1u) ? seg_odd : seg_even;
            if (!seg_first || mbar_test_wait(sm.o_free(), uint32_t(g & 1) ^ 1u)) {
                tc_fence_after();
                const int st = int(npv % uint32_t(C::NS));
                const uint64_t dv = d_v0 + uint64_t(st) * kStageStep;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // 16 tokens a step
                    umma_bf16(o_col, dv + uint64_t(kk * 2048 >> 4), d_p + uint64_t(kk * 2048 >> 4),
                              kIdO, !(seg_first && kk == 0));
                umma_commit(sm.empty(st));
                umma_commit(sm.p_free());
                ++npv;
                progressed = true;
            }
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
// Row maxima (or sums) of R values per lane over the warp's 32 lanes (a butterfly
// that halves the values each step): on return v[0] holds the result of row
// (lane >> (5 - log2 R)), the same in the 32 / R lanes that share that row.
template <int R, bool SUM = false>
__device__ __forceinline__ void warp_row_reduce(float (&v)[R], int lane)
{
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int off = 16 >> step;
        const int len = R >> (step + 1);
        if (len >= 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int k = 0; k < R / 2; ++k) {
                if (k < len) {
                    const float send = upper ? v[k] : v[k + len];
                    const float keep = upper ? v[k + len] : v[k];
                    const float got = __shfl_xor_sync(0xffffffffu, send, off);
                    v[k] = SUM ? keep + got : fmaxf(keep, got);
                }
            }
        } else {
            const float got = __shfl_xor_sync(0xffffffffu, v[0], off);
            v[0] = SUM ? v[0] + got : fmaxf(v[0], got);
        }
    }
}

// Softmax team `team` (0, 1) of 4 warps owns rows team * N/2 .. + N/2 - 1; thread t
// of the team owns token t of a super-stage (and head dim t in the epilogue).
template <int N>
__device__ void softmax_umma(const DecodeParams &p, const USmem<N> &sm, uint32_t tmem, int warp,
                             int lane)
{
    using C = UCfg<N>;
    constexpr int R2 = N / 2;                  // rows of this team
    constexpr int LOG_R2 = R2 == 16 ? 4 : 5;   // rows per lane group after the butterfly
    const int team = (warp - 2) >> 2;
    const int q4 = warp & 3;                   // this warp's TMEM lane quarter
    const int t = q4 * 32 + lane;              // token row of a super-stage; head dim later
    const int tt = team * 128 + t;             // index among the 256 softmax threads
    const int row0 = team * R2;
    const uint32_t lane_base = tmem + (uint32_t(q4 * 32) << 16);
    // this team's rows in the hi and lo column halves of O^T
    const uint32_t o_col = lane_base + C::O_COL + uint32_t(row0);
    const int own = lane >> (5 - LOG_R2);  // the row (of the team's) whose sum this lane keeps
    float lsum = 0.f;                      // that row's sum over this warp's tokens
    uint8_t *pbuf = sm.base + C::OFF_P;
    volatile int *exit_flag = reinterpret_cast<volatile int *>(sm.tslot + 1);
    if (tt == 0)
        *exit_flag = 0;
    tc_fence_before();
    bar_sync_named(1, 256);

    // running max of the team's rows (log2 domain), the same in every thread: kept in
    // registers for 16 rows a team, read from sm.mrow (a broadcast) for 32
    constexpr bool kMReg = R2 == 16;
    float m[kMReg ? R2 : 1];
#pragma unroll
    for (int r = 0; r < (kMReg ? R2 : 1); ++r)
        m[r] = -INFINITY;
    auto mrow = [&](int r) -> float { return kMReg ? m[kMReg ? r : 0] : sm.mrow[row0 + r]; };
    bool wait_ok = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!mbar_wait(bar, parity, kWaitLimitNs) && wait_ok) {
            atomicOr(p.ws + kWsErr, kErrConsumerWait);
            wait_ok = false;
        }
    };

    for (uint32_t i = 0;; ++i) {
        const int st = int(i % uint32_t(C::NS));
        const uint32_t bsel = i & 1u;
        bool leave = false;
        UHdr h = {};
        float x[R2];
        if (!mbar_wait(sm.full(st), (i / uint32_t(C::NS)) & 1u, kWaitLimitNs)) {
            atomicOr(p.ws + kWsErr, kErrConsumerWait);
            leave = true;
        } else {
            h = sm.hdr[st];
            leave = (h.flags & F_END) != 0 || !wait_ok;
        }
        bool first = false, need = false, tok_ok = false;
        if (!leave) {
            wait(sm.s_full(int(bsel)), (i >> 1) & 1u);
            tc_fence_after();
            if constexpr (R2 == 16) {
                float v[32];
                tmem_ld16(lane_base + bsel * N + uint32_t(row0), v);
                tmem_wait_ld();
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    x[r] = v[r];
            } else {
                tmem_ld32<0>(lane_base + bsel * N + uint32_t(row0), x);
                tmem_wait_ld();
            }
            tc_fence_before();
            mbar_arrive(sm.s_free(int(bsel)));
            first = (h.flags & F_FIRST) != 0;
            if (first)
                lsum = 0.f;
            // scale (log2 domain); tokens outside the stage's blocks or past the
            // context, and positions a row does not see, are masked
            const int tok = h.b0 * kBlockSize + t;
            tok_ok = t < int(h.nbv) * kBlockSize && tok < h.T;
#pragma unroll
            for (int r = 0; r < R2; ++r)
                x[r] = tok_ok ? x[r] * p.scale_log2 : -INFINITY;
            const int w0 = p.tree_mask ? h.T - h.W : h.T - h.ql + 1;
            if (__builtin_expect(tok_ok && tok >= w0, 0)) {
#pragma unroll
                for (int r = 0; r < R2; ++r) {
                    int j = (row0 + r) / p.G;
                    j = j < h.ql ? j : h.ql - 1;  // padding rows: the last query's rule
                    bool vis;
                    if (p.tree_mask)
                        vis = (__ldg(p.tree_mask + h.q0 + j) >> (tok - w0)) & 1u;
                    else
                        vis = tok <= h.T - h.ql + j;
                    if (!vis)
                        x[r] = -INFINITY;
                }
            }
            need = first;  // a new segment always sets its running max
#pragma unroll
            for (int r = 0; r < R2; ++r)
                need |= x[r] > mrow(r) + kLazyLog2;
        }
        if (leave)
            *exit_flag = 1;
        // the stage's one reduction: leave together, or raise the running max
        if (bar_red_or_named(1, 256, leave || need)) {
            if (*exit_flag)
                break;
            // ---- raise the running max: block max per row over the 128 tokens
            float bm[R2];
#pragma unroll
            for (int r = 0; r < R2; ++r)
                bm[r] = x[r];
            warp_row_reduce<R2>(bm, lane);
            if ((lane & ((1 << (5 - LOG_R2)) - 1)) == 0)
                sm.red_m[(row0 + own) * 4 + q4] = bm[0];
            bar_sync_named(1, 256);
            if (tt < N) {
                const float4 w = *reinterpret_cast<const float4 *>(sm.red_m + 4 * tt);
                const float mo = first ? -INFINITY : sm.mrow[tt];
                const float mn = fmaxf(mo, fmaxf(fmaxf(w.x, w.y), fmaxf(w.z, w.w)));
                sm.frow[tt] = mn == mo ? 1.f : ex2(mo - mn);  // 0 from -inf
                sm.mrow[tt] = mn;
            }
            bar_sync_named(1, 256);
            bool changed = false;
#pragma unroll
            for (int r = 0; r < R2; ++r) {
                if constexpr (kMReg)
                    m[kMReg ? r : 0] = sm.mrow[row0 + r];
                changed |= sm.frow[row0 + r] != 1.f;
            }
            if (!first && changed) {
                // the accumulators hold earlier stages of this segment: rescale them
                // (O^T, then the row sums) once the previous stage's MMAs have landed
                wait(sm.p_free(), (i - 1) & 1u);
                tc_fence_after();
                lsum *= sm.frow[row0 + own];
#pragma unroll 1
                for (int acc = 0; acc < 2; ++acc) {  // O^T hi, lo
                    const uint32_t col = o_col + uint32_t(acc * N);
                    float a[32];
                    if constexpr (R2 == 16)
                        tmem_ld16(col, a);
                    else
                        tmem_ld32<0>(col, a);
                    tmem_wait_ld();
#pragma unroll
                    for (int r = 0; r < R2; ++r)
                        a[r] *= sm.frow[row0 + r];
                    if constexpr (R2 == 16)
                        tmem_st16(col, a);
                    else
                        tmem_st32<0>(col, a);
                    tmem_wait_st();
                }
                tc_fence_before();
            }
        }

        // ---- P = 2^(x - m) as P^T rows, bf16 hi + lo
#pragma unroll
        for (int r = 0; r < R2; ++r) {
            const float mr = mrow(r);
            const float mu = mr == -INFINITY ? 0.f : mr;
            x[r] = ex2(x[r] - mu);  // 0 for a masked token
        }
        {
            float rs[R2];
#pragma unroll
            for (int r = 0; r < R2; ++r)
                rs[r] = x[r];
            warp_row_reduce<R2, true>(rs, lane);
            lsum += rs[0];
        }
        if (i > 0)
            wait(sm.p_free(), (i - 1) & 1u);  // the previous stage's MMAs have read P^T
#pragma unroll
        for (int c = 0; c < R2 / 8; ++c) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float a0 = x[8 * c + 2 * k], a1 = x[8 * c + 2 * k + 1];
                hi[k] = pack_bf16x2(a0, a1);
                lo[k] = pack_bf16x2(a0 - bf16lo_f32(hi[k]), a1 - bf16hi_f32(hi[k]));
            }
            // P^T row t: element e (hi: row, lo: N + row) sits in atom e / 64, 16-byte
            // chunk (e % 64) / 8, swizzled by the row's low 3 bits
            const int eh = row0 + 8 * c, el = N + row0 + 8 * c;
            const uint32_t oh = uint32_t(eh >> 6) * C::P_ATOM + uint32_t(t) * 128u +
                                (uint32_t(((eh & 63) >> 3) ^ (t & 7)) << 4);
            const uint32_t ol = uint32_t(el >> 6) * C::P_ATOM + uint32_t(t) * 128u +
                                (uint32_t(((el & 63) >> 3) ^ (t & 7)) << 4);
            *reinterpret_cast<uint4 *>(pbuf + oh) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(pbuf + ol) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        if (!tok_ok && !leave) {
            // a slot past the context or outside the stage's blocks: its V row (stale
            // or NaN) must not reach the accumulator, even times a zero weight; each
            // team clears one 64-dim half
            uint8_t *vrow = sm.stage(st) + 32768u + uint32_t(team) * kHalfBytes + uint32_t(t) * 128u;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(vrow + c * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        mbar_arrive(sm.p_full());

        if (h.flags & F_LAST) {
            // ---- the segment's end: O^T row d = t of the team's rows, over the sums
            wait(sm.p_free(), i & 1u);
            tc_fence_after();
            // the hi and lo halves of O^T and of the row sums, added, 16 rows at a time;
            // the output (the whole sequence in this cell) or the partial (m, l, acc)
            // for the merge kernel leaves as each chunk is read
            if ((lane & ((1 << (5 - LOG_R2)) - 1)) == 0)
                sm.red_l[(row0 + own) * 4 + q4] = lsum;
            bar_sync_named(1, 256);
            const int rows_v = p.G * h.ql;
            const int d = t;
            const int64_t cb = int64_t(h.cell) * 2 + h.slot;
#pragma unroll
            for (int c16 = 0; c16 < R2 / 16; ++c16) {
                float o[16], l[16];
                {
                    float a[32], b[32];
                    tmem_ld16(o_col + 16 * c16, a);
                    tmem_ld16(o_col + N + 16 * c16, b);
                    tmem_wait_ld();
#pragma unroll
                    for (int r = 0; r < 16; ++r)
                        o[r] = a[r] + b[r];
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        const float4 w =
                            *reinterpret_cast<const float4 *>(sm.red_l + 4 * (row0 + 16 * c16 + r));
                        l[r] = (w.x + w.y) + (w.z + w.w);
                    }
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const int rr = 16 * c16 + r, row = row0 + rr;
                    if (row >= rows_v)
                        continue;
                    if (h.flags & F_DIRECT) {
                        const float v = o[r] * (l[r] > 0.f ? 1.f / l[r] : 0.f);
                        const int j = row / p.G;
                        const int64_t oi = ((int64_t(h.q0) + j) * p.Hq + int64_t(h.head) * p.G +
                                            (row - j * p.G)) * 128 + d;
                        if (p.out_f32)
                            static_cast<float *>(p.out)[oi] = v;
                        else
                            static_cast<__nv_bfloat16 *>(p.out)[oi] = __float2bfloat16_rn(v);
                    } else {
                        p.part[(cb * p.rows + row) * 128 + d] = o[r];
                        if (d == rr) {
                            float *ml = p.ml + (cb * p.rows + row) * 2;
                            ml[0] = mrow(rr);
                            ml[1] = l[r];
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(sm.o_free());
        }
    }
}

}  // namespace

template <int N>
__global__ void __launch_bounds__(352, 1)
    paged_decode_umma_kernel(const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap,
                             const __grid_constant__ CUtensorMap qmap, const DecodeParams p)
{
    using C = UCfg<N>;
    extern __shared__ uint8_t smem_raw[];
    const USmem<N> sm = ucarve<N>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        tma_prefetch_desc(&qmap);
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(sm.full(i), 1);
            mbar_init(sm.empty(i), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.q_full(b), 1);
            mbar_init(sm.q_free(b), 1);
            mbar_init(sm.s_full(b), 1);
            mbar_init(sm.s_free(b), 256);
        }
        mbar_init(sm.p_full(), 256);
        mbar_init(sm.p_free(), 1);
        mbar_init(sm.o_free(), 256);
        mbar_init(sm.done(), 1);
        fence_mbar_init();
        *sm.progress = 0;
    }
    // Q rows past a segment's G * nq (padding up to N) are never written by the
    // copies: they hold zeros so the padding scores stay finite
    for (uint32_t i = threadIdx.x; i < 2 * C::QBUF / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(sm.base + C::OFF_Q)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (warp == 1)
        tmem_alloc(smem_u32(sm.tslot), C::NCOLS);
    // the previous kernel on the stream (e.g. the KV append) has finished writing
    asm volatile("griddepcontrol.wait;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tslot;
    if (warp == 0) {
        producer_umma<N>(&kmap, &vmap, &qmap, p, sm, lane);
    } else if (warp == 1) {
        if (lane == 0)
            mma_umma<N>(p, sm, tmem);
        __syncwarp();
    } else if (warp < 10) {
        softmax_umma<N>(p, sm, tmem, warp, lane);
    } else {
        prefetch_umma<N>(&kmap, &vmap, p, sm, lane);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::NCOLS);
    }
}

size_t umma_smem_bytes(int n) { return n == 32 ? UCfg<32>::SMEM : UCfg<64>::SMEM; }
int umma_stages(int n) { return n == 32 ? UCfg<32>::NS : UCfg<64>::NS; }

template <int N>
static cudaError_t launch_umma_n(const DecodePlan &pl, const DecodeParams &p,
                                 const CUtensorMap &kmap, const CUtensorMap &vmap,
                                 const CUtensorMap &qmap, cudaStream_t stream,
                                 cudaEvent_t ev_before, cudaEvent_t ev_after)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && configured[dev] < int(pl.smem)) {
        e = cudaFuncSetAttribute(paged_decode_umma_kernel<N>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem));
        if (e != cudaSuccess)
            return e;
        configured[dev] = int(pl.smem);
    }
    if (ev_before && (e = cudaEventRecord(ev_before, stream)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(pl.grid));
    cfg.blockDim = dim3(352);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, paged_decode_umma_kernel<N>, kmap, vmap, qmap, p);
    if (e != cudaSuccess)
        return e;
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    if (ev_after && (e = cudaEventRecord(ev_after, stream)) != cudaSuccess)
        return e;
    return launch_merge(pl, p, stream);
}

cudaError_t launch_decode_umma(const DecodePlan &pl, const DecodeParams &p,
                               const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const CUtensorMap &qmap, cudaStream_t stream, cudaEvent_t eb,
                               cudaEvent_t ea)
{
    if (pl.rows_pad == 32)
        return launch_umma_n<32>(pl, p, kmap, vmap, qmap, stream, eb, ea);
    return launch_umma_n<64>(pl, p, kmap, vmap, qmap, stream, eb, ea);
}

}  // namespace pkv
