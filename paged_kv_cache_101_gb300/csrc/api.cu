// api.cu -- the extern "C" entry points of libpkv (see include/pkv.h).
//
// Every argument that lives on the host is validated before any CUDA call, so
// an invalid call returns its status without touching the device. Tensor maps
// (TMA descriptors) for the K/V pools are encoded on the host through the
// driver entry point the CUDA runtime exposes (no link-time libcuda
// dependency) and cached per (pointer, shape, device).
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace pkv {
// copy_blocks.cu
cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, int64_t num_blocks, int num_kv_heads,
                               int head_dim, const int32_t *src, const int32_t *dst,
                               int num_pairs, cudaStream_t stream);
}  // namespace pkv

namespace {

int32_t g_opt_num_ctas = 0;
int32_t g_opt_stages = 0;
int32_t g_opt_heads = 0;
int32_t g_opt_box = 0;
int32_t g_opt_tail = 0;
int32_t g_opt_pace = 0;
int32_t g_opt_math = 0;
int32_t g_opt_umma = 0;
int32_t g_opt_prefetch = 0;
thread_local bool t_meta_ready = false;  // set by a host step around its attention call
int32_t g_opt_pace_margin = 0;
cudaEvent_t g_ev_before = nullptr;
cudaEvent_t g_ev_after = nullptr;
void *g_trace = nullptr;
size_t g_trace_bytes = 0;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct DeviceInfo {
    bool valid = false;
    int num_sms = 0;
    int smem_optin = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[64];

cudaError_t device_info(DeviceInfo *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev[dev].valid) {
        DeviceInfo d;
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess)
            return e;
        d.valid = true;
        g_dev[dev] = d;
    }
    *out = g_dev[dev];
    return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode)
        return cudaSuccess;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess)
        return e;
    if (q != cudaDriverEntryPointSuccess || fn == nullptr)
        return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// A pool [num_blocks][16][Hkv][D] bf16 seen as 5-D (64, D/64, Hkv, 16, num_blocks);
// a box is one (head, 64-column half) tile of one block: 16 rows x 128 B,
// stored with the 128-byte swizzle.
CUresult encode_pool(CUtensorMap *map, const void *base, int64_t num_blocks, int Hkv, int D)
{
    const cuuint64_t dims[5] = {64, cuuint64_t(D / 64), cuuint64_t(Hkv), 16,
                                cuuint64_t(num_blocks)};
    const cuuint64_t strides[4] = {128, cuuint64_t(D) * 2, cuuint64_t(Hkv) * D * 2,
                                   cuuint64_t(16) * Hkv * D * 2};
    const cuuint32_t box[5] = {64, 1, 1, 16, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// The same pool seen as (64, 16, D/64, Hkv, num_blocks): token before half and
// head, so one box (64, 16, D/64, hg, 1) brings a whole block of hg heads and
// lands in shared memory as [head][half][token][64], the layout the tile boxes
// build. Returns non-success if the driver refuses this stride order.
CUresult encode_pool_block(CUtensorMap *map, const void *base, int64_t num_blocks, int Hkv, int D,
                           int hg)
{
    const cuuint64_t dims[5] = {64, 16, cuuint64_t(D / 64), cuuint64_t(Hkv),
                                cuuint64_t(num_blocks)};
    const cuuint64_t strides[4] = {cuuint64_t(Hkv) * D * 2, 128, cuuint64_t(D) * 2,
                                   cuuint64_t(16) * Hkv * D * 2};
    const cuuint32_t box[5] = {64, 16, cuuint32_t(D / 64), cuuint32_t(hg), 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// E4M3 pools [num_blocks][16][Hkv][128] of uint8: a head row is one 128-byte
// swizzle row. Tile boxes: (128, 1, Hkv, 16, num_blocks) with box (128,1,1,16,1);
// whole-block boxes: (128, 16, 1, Hkv, num_blocks) with box (128,16,1,hg,1), so
// shared memory holds [head][token][128 B] either way.
CUresult encode_pool_fp8(CUtensorMap *map, const void *base, int64_t num_blocks, int Hkv, int hg)
{
    const cuuint64_t row = 128, tok = cuuint64_t(Hkv) * 128, blk = 16 * tok;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (hg == 0) {
        const cuuint64_t dims[5] = {128, 1, cuuint64_t(Hkv), 16, cuuint64_t(num_blocks)};
        const cuuint64_t strides[4] = {row, row, tok, blk};
        const cuuint32_t box[5] = {128, 1, 1, 16, 1};
        return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    const cuuint64_t dims[5] = {128, 16, 1, cuuint64_t(Hkv), cuuint64_t(num_blocks)};
    const cuuint64_t strides[4] = {tok, row, row, blk};
    const cuuint32_t box[5] = {128, 16, 1, cuuint32_t(hg), 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

struct MapEntry {
    const void *base = nullptr;
    int64_t nb = 0;
    int hkv = 0, d = 0, dev = -1, kind = 0;  // kind 0: tile boxes, else heads per box
    int kv8 = 0;
    CUtensorMap map;
};
MapEntry g_maps[16];
int g_map_next = 0;

// kind 0: tile-box map; kind hg > 0: whole-block map with hg heads per box.
cudaError_t pool_map(const void *base, int64_t nb, int Hkv, int D, int kind, int kv8,
                     CUtensorMap *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = get_encoder();
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto &m : g_maps)
        if (m.base == base && m.nb == nb && m.hkv == Hkv && m.d == D && m.dev == dev &&
            m.kind == kind && m.kv8 == kv8) {
            *out = m.map;
            return cudaSuccess;
        }
    MapEntry &m = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % 16;
    const CUresult r = kv8         ? encode_pool_fp8(&m.map, base, nb, Hkv, kind)
                       : kind == 0 ? encode_pool(&m.map, base, nb, Hkv, D)
                                   : encode_pool_block(&m.map, base, nb, Hkv, D, kind);
    if (r != CUDA_SUCCESS) {
        m.base = nullptr;
        return cudaErrorInvalidValue;
    }
    m.base = base;
    m.nb = nb;
    m.hkv = Hkv;
    m.d = D;
    m.kv8 = kv8;
    m.dev = dev;
    m.kind = kind;
    *out = m.map;
    return cudaSuccess;
}

// q [rows][Hq][D] bf16 (D = 128) seen as (64, 2, Hq, rows, 1): one box (64, 1, G,
// box_rows, 1) brings one 64-dim half of box_rows queries x G heads as [row][g][64],
// stored with the 128-byte swizzle; rows past the end read as zeros.
CUresult encode_q(CUtensorMap *map, const void *q, int64_t rows, int Hq, int G, int box_rows)
{
    const cuuint64_t row = cuuint64_t(Hq) * 256;
    const cuuint64_t dims[5] = {64, 2, cuuint64_t(Hq), cuuint64_t(rows), 1};
    const cuuint64_t strides[4] = {128, 256, row, row * cuuint64_t(rows)};
    const cuuint32_t box[5] = {64, 1, cuuint32_t(G), cuuint32_t(box_rows), 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(q), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

struct QMapEntry {
    const void *q = nullptr;
    int64_t rows = 0;
    int hq = 0, g = 0, box_rows = 0, dev = -1;
    CUtensorMap map;
};
QMapEntry g_qmaps[8];
int g_qmap_next = 0;

cudaError_t q_map(const void *q, int64_t rows, int Hq, int G, int box_rows, CUtensorMap *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = get_encoder();
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto &m : g_qmaps)
        if (m.q == q && m.rows == rows && m.hq == Hq && m.g == G && m.box_rows == box_rows &&
            m.dev == dev) {
            *out = m.map;
            return cudaSuccess;
        }
    QMapEntry &m = g_qmaps[g_qmap_next];
    g_qmap_next = (g_qmap_next + 1) % 8;
    if (encode_q(&m.map, q, rows, Hq, G, box_rows) != CUDA_SUCCESS) {
        m.q = nullptr;
        return cudaErrorInvalidValue;
    }
    m.q = q;
    m.rows = rows;
    m.hq = Hq;
    m.g = G;
    m.box_rows = box_rows;
    m.dev = dev;
    *out = m.map;
    return cudaSuccess;
}

// Host-side checks shared by the workspace query and the attention calls. The
// fixed-count call takes 1..4 queries per sequence; the variable-count call any
// count whose score rows (G per query) fit the kernel's 64 rows per kv head.
pkv_status check_geometry(int32_t num_seqs, int32_t nq, int32_t Hq, int32_t Hkv, int32_t D,
                          bool varlen = false)
{
    if (num_seqs < 0 || nq < 1 || Hq < 1 || Hkv < 1)
        return PKV_ERR_SHAPE;
    if (Hq % Hkv != 0)
        return PKV_ERR_SHAPE;
    if (D != 64 && D != 128)
        return PKV_ERR_UNSUPPORTED;
    if (nq > 4 && !varlen)
        return PKV_ERR_UNSUPPORTED;
    if ((Hq / Hkv) * nq > pkv::kMaxRows)
        return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

}  // namespace

namespace pkv {

void set_meta_ready(bool ready) { t_meta_ready = ready; }

}  // namespace pkv

extern "C" {

const char *pkv_status_string(int32_t status)
{
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is NULL";
    case PKV_ERR_SHAPE: return "inconsistent or non-positive sizes";
    case PKV_ERR_DTYPE: return "unknown output dtype";
    case PKV_ERR_ALIGN: return "a buffer is not aligned as required";
    case PKV_ERR_RANGE: return "a size is beyond what the library supports";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case PKV_ERR_UNSUPPORTED: return "no kernel for this (valid) shape";
    case PKV_ERR_NO_BLOCKS: return "not enough free blocks in the pool";
    case PKV_ERR_SEQUENCE: return "unknown or duplicate sequence id";
    default: return "unknown status";
    }
}

int32_t pkv_version(void) { return 200; }

void pkv_set_trace_buffer(void *device_buffer, size_t bytes)
{
    g_trace = device_buffer;
    g_trace_bytes = device_buffer ? bytes : 0;
}

void pkv_set_profiling_events(void *before, void *after)
{
    if (before && after) {
        g_ev_before = static_cast<cudaEvent_t>(before);
        g_ev_after = static_cast<cudaEvent_t>(after);
    } else {
        g_ev_before = g_ev_after = nullptr;
    }
}

int32_t pkv_set_option(int32_t option, int32_t value)
{
    if (value < 0)
        return -1;
    int32_t prev;
    switch (option) {
    case PKV_OPT_NUM_CTAS:
        prev = g_opt_num_ctas;
        g_opt_num_ctas = value;
        return prev;
    case PKV_OPT_STAGES:
        prev = g_opt_stages;
        g_opt_stages = value;
        return prev;
    case PKV_OPT_HEADS_PER_CTA:
        prev = g_opt_heads;
        g_opt_heads = value;
        return prev;
    case PKV_OPT_TAIL:
        prev = g_opt_tail;
        g_opt_tail = value;
        return prev;
    case PKV_OPT_TMA_BOX:
        if (value > 2)
            return -1;
        prev = g_opt_box;
        g_opt_box = value;
        return prev;
    case PKV_OPT_PACE:
        if (value > 1)
            return -1;
        prev = g_opt_pace;
        g_opt_pace = value;
        return prev;
    case PKV_OPT_MATH:
        if (value > 1)
            return -1;
        prev = g_opt_math;
        g_opt_math = value;
        return prev;
    case PKV_OPT_UMMA:
        if (value > 1)
            return -1;
        prev = g_opt_umma;
        g_opt_umma = value;
        return prev;
    case PKV_OPT_PREFETCH:
        if (value > 4097)
            return -1;
        prev = g_opt_prefetch;
        g_opt_prefetch = value;
        return prev;
    case PKV_OPT_PACE_MARGIN:
        if (value > 10000)
            return -1;
        prev = g_opt_pace_margin;
        g_opt_pace_margin = value;
        return prev;
    default:
        return -1;
    }
}

pkv_status pkv_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                         int64_t n_new, void *k_cache, void *v_cache, int64_t num_blocks,
                         int32_t num_kv_heads, int32_t head_dim, void *stream)
{
    if (n_new < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1)
        return PKV_ERR_SHAPE;
    if (n_new == 0)
        return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache)
        return PKV_ERR_NULL;
    if (head_dim % 8 != 0)
        return PKV_ERR_UNSUPPORTED;
    if (head_dim > 1024 || num_kv_heads > 1024 || n_new > 0x7fffffffLL ||
        num_blocks > (int64_t(1) << 40))
        return PKV_ERR_RANGE;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
        return PKV_ERR_ALIGN;
    cudaError_t e = pkv::launch_kv_append(k_new, v_new, slot_mapping, n_new, k_cache, v_cache,
                                          num_blocks, num_kv_heads, head_dim,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, int64_t num_blocks,
                           int32_t num_kv_heads, int32_t head_dim, const int32_t *block_src,
                           const int32_t *block_dst, int32_t num_pairs, void *stream)
{
    if (num_pairs < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1)
        return PKV_ERR_SHAPE;
    if (num_pairs == 0)
        return PKV_OK;
    if (!k_cache || !v_cache || !block_src || !block_dst)
        return PKV_ERR_NULL;
    if (head_dim % 8 != 0)
        return PKV_ERR_UNSUPPORTED;
    if (head_dim > 1024 || num_kv_heads > 1024 || num_blocks > (int64_t(1) << 40))
        return PKV_ERR_RANGE;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_src, 4) ||
        !aligned(block_dst, 4))
        return PKV_ERR_ALIGN;
    cudaError_t e = pkv::launch_copy_blocks(k_cache, v_cache, num_blocks, num_kv_heads, head_dim,
                                            block_src, block_dst, num_pairs,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t pkv_workspace_size(int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim)
{
    if (check_geometry(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim, true) !=
        PKV_OK)
        return 0;
    if (num_seqs == 0)
        return 256;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess)
        return 0;
    pkv::DecodePlan pl;
    if (pkv::plan_decode(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim, 1,
                         d.num_sms, g_opt_num_ctas, g_opt_stages, g_opt_heads, g_opt_tail, d.smem_optin,
                         0, 0, 0, &pl) != 0)
        return 0;
    size_t bytes = pl.ws_bytes;
    // the tcgen05 kernel (one kv head per CTA) and the E4M3 call share this size:
    // their plans may need more records or cells
    pkv::DecodePlan alt;
    for (int kind = 0; kind < 2; ++kind)
        if (head_dim == 128 &&
            pkv::plan_decode(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim, 1,
                             d.num_sms, g_opt_num_ctas, g_opt_stages, g_opt_heads, g_opt_tail,
                             d.smem_optin, kind, 0, 1 - kind, &alt) == 0 &&
            alt.ws_bytes > bytes)
            bytes = alt.ws_bytes;
    return bytes;
}

}  // extern "C"

namespace {

// Shared-prefix cascade (null / 0 without).
struct Cascade {
    const int32_t *groups = nullptr;  // device [num_groups][3]
    int32_t num_groups = 0, max_group_seqs = 0;
};

// Bytes of the cascade's prefix partials: (m, l) and acc[D] per (prefix chunk,
// query row, head), for up to kMaxPreChunks chunks.
size_t prefix_region_bytes(int64_t total_q, int32_t Hq, int32_t D)
{
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t rows = size_t(pkv::kMaxPreChunks) * size_t(total_q) * Hq;
    return up(rows * 2 * 4) + up(rows * D * 4);
}

// Variable query counts (all null / 0 for the fixed-count call).
struct Varlen {
    const int32_t *q_start = nullptr;
    const uint32_t *tree_mask = nullptr;
    const int32_t *tree_len = nullptr;
    const int32_t *table_row = nullptr;
    int32_t total_q = 0, table_rows = 0;
};

// The attention call for bf16 (kv8 = 0) or E4M3 (kv8 = 1, with scales) pools;
// n_query_per_seq is the query count of every sequence, or with vl.q_start the
// largest one.
pkv_status attention(const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
                     int kv8, const float *k_scale, const float *v_scale,
                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                     const int32_t *context_lens, int32_t num_seqs, int32_t n_query_per_seq,
                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                     void *out, int32_t out_dtype, void *workspace, size_t workspace_bytes,
                     void *stream, const Varlen &vl = Varlen(), const Cascade &cc = Cascade(),
                     size_t *need_only = nullptr)
{
    // need_only != null: run every host check (a workspace taken as given and
    // aligned), store the workspace bytes the call's plan needs (0: nothing to
    // do) and return before any CUDA work is enqueued
    if (need_only)
        *need_only = 0;
    pkv_status st = check_geometry(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim,
                                   vl.q_start != nullptr);
    if (st != PKV_OK)
        return st;
    if (kv8 && head_dim != 128)
        return PKV_ERR_UNSUPPORTED;
    if (num_blocks < 1 || max_blocks_per_seq < 1)
        return PKV_ERR_SHAPE;
    if (out_dtype != PKV_BF16 && out_dtype != PKV_FP32)
        return PKV_ERR_DTYPE;
    if (num_seqs == 0)
        return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return PKV_ERR_NULL;
    if (kv8 && (!k_scale || !v_scale))
        return PKV_ERR_NULL;
    if (!workspace && !need_only)
        return PKV_ERR_WORKSPACE;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
        (!need_only && !aligned(workspace, 256)))
        return PKV_ERR_ALIGN;
    if (kv8 && (!aligned(k_scale, 4) || !aligned(v_scale, 4)))
        return PKV_ERR_ALIGN;
    if (max_blocks_per_seq > (1 << 26) || num_blocks > 0x7fffffffLL || num_seqs > (1 << 24) ||
        num_kv_heads > 65535)
        return PKV_ERR_RANGE;

    DeviceInfo d;
    if (device_info(&d) != cudaSuccess)
        return PKV_ERR_CUDA;
    // the CUDA-core consumers (PKV_OPT_MATH = 1) serve the plain bf16 call only
    const int fma = (g_opt_math == 1 && !kv8 && !vl.q_start && !cc.groups && head_dim == 128 &&
                     (num_q_heads / num_kv_heads) * n_query_per_seq <= 32)
                        ? 1
                        : 0;
    // the tcgen05 kernel (opt-in: measured slower than the mma.sync kernel on the
    // paged layout) serves 17..64 query rows per kv head, except for a cascade (its
    // members' running states start from prefix partials)
    const int umma = (g_opt_umma == 1 && !cc.groups) ? 1 : 0;
    pkv::DecodePlan pl;
    if (pkv::plan_decode(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim,
                         max_blocks_per_seq, d.num_sms, g_opt_num_ctas, g_opt_stages,
                         g_opt_heads, g_opt_tail, d.smem_optin, kv8, fma, umma, &pl) != 0)
        return PKV_ERR_UNSUPPORTED;
    // cascade: the prefix pass's plan and the prefix partials after the workspace
    pkv::DecodePlan ppl{};
    int pre_tiles = 0;
    size_t off_pre = 0;
    if (cc.groups) {
        if (kv8 || vl.q_start)
            return PKV_ERR_UNSUPPORTED;  // the cascade runs on bf16 pools, fixed counts
        pre_tiles = pkv::plan_prefix(head_dim, num_q_heads / num_kv_heads, num_kv_heads,
                                     cc.num_groups, cc.max_group_seqs, n_query_per_seq,
                                     d.smem_optin, &ppl);
        if (pre_tiles < 1)
            return PKV_ERR_UNSUPPORTED;
        off_pre = (pl.ws_bytes + 255) / 256 * 256;
    }
    const size_t need =
        cc.groups ? off_pre + prefix_region_bytes(int64_t(num_seqs) * n_query_per_seq,
                                                  num_q_heads, head_dim)
                  : pl.ws_bytes;
    if (need_only) {
        *need_only = need;
        return PKV_OK;
    }
    if (workspace_bytes < need)
        return PKV_ERR_WORKSPACE;
    uint64_t *trace = nullptr;
    if (g_trace && g_trace_bytes >= size_t(pl.grid) * pkv::kTraceWords * 8 &&
        aligned(g_trace, 8))
        trace = static_cast<uint64_t *>(g_trace);

    CUtensorMap kmap, vmap, qmap;
    int whole_box = 0;
    if (pl.umma) {
        // one (head, half) box per block: the tiles land in the super-stage's rows
        if (pool_map(k_cache, num_blocks, num_kv_heads, head_dim, 0, 0, &kmap) != cudaSuccess ||
            pool_map(v_cache, num_blocks, num_kv_heads, head_dim, 0, 0, &vmap) != cudaSuccess ||
            q_map(q, vl.q_start ? vl.total_q : int64_t(num_seqs) * n_query_per_seq, num_q_heads,
                  pl.G, n_query_per_seq, &qmap) != cudaSuccess)
            return PKV_ERR_CUDA;
    } else if (g_opt_box != 1 &&
        pool_map(k_cache, num_blocks, num_kv_heads, head_dim, pl.HG, kv8, &kmap) == cudaSuccess &&
        pool_map(v_cache, num_blocks, num_kv_heads, head_dim, pl.HG, kv8, &vmap) == cudaSuccess)
        whole_box = 1;
    if (!whole_box && !pl.umma) {
        if (g_opt_box == 2)
            return PKV_ERR_UNSUPPORTED;  // whole-block boxes requested but refused
        if (pool_map(k_cache, num_blocks, num_kv_heads, head_dim, 0, kv8, &kmap) != cudaSuccess ||
            pool_map(v_cache, num_blocks, num_kv_heads, head_dim, 0, kv8, &vmap) != cudaSuccess)
            return PKV_ERR_CUDA;
    }

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    pkv::DecodeParams p;
    memset(&p, 0, sizeof p);
    p.q = static_cast<const uint16_t *>(q);
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.ws = reinterpret_cast<uint32_t *>(ws);
    p.pieces = reinterpret_cast<int2 *>(ws + pl.off_rec);
    p.ml = reinterpret_cast<float *>(ws + pl.off_ml);
    p.part = reinterpret_cast<float *>(ws + pl.off_part);
    p.trace = trace;
    p.num_blocks = num_blocks;
    p.S = num_seqs;
    p.MB = max_blocks_per_seq;
    p.nq = n_query_per_seq;
    p.Hq = num_q_heads;
    p.Hkv = num_kv_heads;
    p.G = pl.G;
    p.rows = pl.rows;
    p.rows_pad = pl.rows_pad;
    p.HG = pl.HG;
    p.n_hg = pl.n_hg;
    p.out_f32 = out_dtype == PKV_FP32;
    p.stage_bytes = pl.stage_bytes;
    p.nst = pl.nst;
    p.whole_box = whole_box;
    p.ncw = pl.HG * pl.wph;
    p.tickets_max = pl.tickets_max;
    p.ticket_div = pl.tail_div;
    p.ticket_units = 4;
    p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    p.pace = g_opt_pace;
    p.meta_ready = (t_meta_ready && !cc.groups) ? 1 : 0;
    p.pace_margin = float(g_opt_pace_margin) * 1e-4f;
    p.pf_units = g_opt_prefetch == 0 ? 64 : g_opt_prefetch - 1;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.q_start = vl.q_start;
    p.tree_mask = vl.tree_mask;
    p.tree_len = vl.tree_len;
    p.table_row = vl.table_row;
    p.total_q = vl.q_start ? vl.total_q : num_seqs * n_query_per_seq;
    p.table_rows = vl.table_row ? vl.table_rows : num_seqs;
    cudaEvent_t ev_b = g_ev_before;
    if (cc.groups) {
        const int64_t total_q = int64_t(num_seqs) * n_query_per_seq;
        p.prefix_groups = cc.groups;
        p.num_groups = cc.num_groups;
        p.pre_ml = reinterpret_cast<float *>(ws + off_pre);
        p.pre_acc = reinterpret_cast<float *>(
            ws + off_pre +
            (size_t(pkv::kMaxPreChunks) * total_q * num_q_heads * 2 * 4 + 255) / 256 * 256);
        // cut each group's prefix into up to kMaxPreChunks block ranges (one
        // partial each) so the prefix pass keeps about two CTAs per SM busy; more
        // ranges cost each member's seed more partials to fold (measured slower)
        const int64_t base_ctas = int64_t(ppl.grid);
        int chunks = int((2 * int64_t(d.num_sms) + base_ctas - 1) / base_ctas);
        chunks = chunks < 1 ? 1 : (chunks > pkv::kMaxPreChunks ? pkv::kMaxPreChunks : chunks);
        p.pre_chunks = chunks;
        ppl.grid = int(base_ctas * chunks);
        // the prefix pass: one kv head per CTA; its own tensor maps (one head per box)
        CUtensorMap pk, pv;
        int pbox = 0;
        if (g_opt_box != 1 &&
            pool_map(k_cache, num_blocks, num_kv_heads, head_dim, 1, 0, &pk) == cudaSuccess &&
            pool_map(v_cache, num_blocks, num_kv_heads, head_dim, 1, 0, &pv) == cudaSuccess)
            pbox = 1;
        if (!pbox &&
            (pool_map(k_cache, num_blocks, num_kv_heads, head_dim, 0, 0, &pk) != cudaSuccess ||
             pool_map(v_cache, num_blocks, num_kv_heads, head_dim, 0, 0, &pv) != cudaSuccess))
            return PKV_ERR_CUDA;
        pkv::DecodeParams pp = p;
        pp.prefix_pass = 1;
        pp.pre_tiles = pre_tiles;
        pp.pre_chunks = p.pre_chunks;
        pp.pre_qrows = 128 / (num_q_heads / num_kv_heads);
        pp.rows = ppl.rows;
        pp.rows_pad = ppl.rows_pad;
        pp.HG = 1;
        pp.n_hg = num_kv_heads;
        pp.stage_bytes = ppl.stage_bytes;
        pp.nst = ppl.nst;
        pp.whole_box = pbox;
        pp.ncw = 8;
        pp.tickets_max = 0;
        pp.ticket_div = 0;
        pp.pace = 0;
        pp.trace = nullptr;
        cudaError_t e = pkv::launch_decode(ppl, pp, pk, pv, static_cast<cudaStream_t>(stream),
                                           ev_b, nullptr);
        if (e != cudaSuccess)
            return PKV_ERR_CUDA;
        ev_b = nullptr;  // the timing hook spans the prefix pass and the main kernel
    }
    cudaError_t e =
        pl.umma ? pkv::launch_decode_umma(pl, p, kmap, vmap, qmap, static_cast<cudaStream_t>(stream),
                                          ev_b, g_ev_after)
                : pkv::launch_decode(pl, p, kmap, vmap, static_cast<cudaStream_t>(stream), ev_b,
                                     g_ev_after);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                                      int64_t num_blocks, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      int32_t num_seqs, int32_t n_query_per_seq,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      float scale, void *out, int32_t out_dtype, void *workspace,
                                      size_t workspace_bytes, void *stream)
{
    return attention(q, k_cache, v_cache, num_blocks, 0, nullptr, nullptr, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, n_query_per_seq, num_q_heads,
                     num_kv_heads, head_dim, scale, out, out_dtype, workspace, workspace_bytes,
                     stream);
}

pkv_status pkv_paged_decode_attention_fp8(const void *q, const void *k_cache, const void *v_cache,
                                          int64_t num_blocks, const float *k_scale,
                                          const float *v_scale, const int32_t *block_tables,
                                          int32_t max_blocks_per_seq,
                                          const int32_t *context_lens, int32_t num_seqs,
                                          int32_t n_query_per_seq, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim, float scale,
                                          void *out, int32_t out_dtype, void *workspace,
                                          size_t workspace_bytes, void *stream)
{
    return attention(q, k_cache, v_cache, num_blocks, 1, k_scale, v_scale, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, n_query_per_seq, num_q_heads,
                     num_kv_heads, head_dim, scale, out, out_dtype, workspace, workspace_bytes,
                     stream);
}

size_t pkv_workspace_size_cascade(int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim)
{
    const size_t base = pkv_workspace_size(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads,
                                           head_dim);
    if (base == 0)
        return 0;
    return (base + 255) / 256 * 256 +
           prefix_region_bytes(int64_t(num_seqs) * n_query_per_seq, num_q_heads, head_dim);
}

pkv_status pkv_paged_decode_attention_cascade(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
    int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, float scale, const int32_t *prefix_groups, int32_t num_groups,
    int32_t max_group_seqs, void *out, int32_t out_dtype, void *workspace,
    size_t workspace_bytes, void *stream)
{
    if (num_groups < 0 || max_group_seqs < 0)
        return PKV_ERR_SHAPE;
    Cascade cc;
    if (num_seqs > 0 && num_groups > 0 && max_group_seqs > 0) {
        if (!prefix_groups)
            return PKV_ERR_NULL;
        if (!aligned(prefix_groups, 4))
            return PKV_ERR_ALIGN;
        if (int64_t(num_groups) > num_seqs || max_group_seqs > num_seqs)
            return PKV_ERR_RANGE;
        cc.groups = prefix_groups;
        cc.num_groups = num_groups;
        cc.max_group_seqs = max_group_seqs;
    }
    return attention(q, k_cache, v_cache, num_blocks, 0, nullptr, nullptr, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, n_query_per_seq, num_q_heads,
                     num_kv_heads, head_dim, scale, out, out_dtype, workspace, workspace_bytes,
                     stream, Varlen(), cc);
}

pkv_status pkv_paged_decode_attention_varlen(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    const int32_t *block_tables, int32_t max_blocks_per_seq, int32_t num_table_rows,
    const int32_t *table_row, const int32_t *context_lens, const int32_t *q_start,
    const uint32_t *tree_mask, const int32_t *tree_len, int32_t num_seqs, int32_t max_q_len,
    int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
    void *out, int32_t out_dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    if (num_seqs > 0 && !q_start)
        return PKV_ERR_NULL;
    if ((tree_mask == nullptr) != (tree_len == nullptr))
        return PKV_ERR_NULL;  // masks and their windows come together
    if (total_q < 0 || num_table_rows < 0 || (table_row == nullptr && num_table_rows < num_seqs))
        return PKV_ERR_SHAPE;
    if ((q_start && !aligned(q_start, 4)) || (tree_mask && !aligned(tree_mask, 4)) ||
        (tree_len && !aligned(tree_len, 4)) || (table_row && !aligned(table_row, 4)))
        return PKV_ERR_ALIGN;
    Varlen vl;
    vl.q_start = q_start;
    vl.tree_mask = tree_mask;
    vl.tree_len = tree_len;
    vl.table_row = table_row;
    vl.total_q = total_q;
    vl.table_rows = table_row ? num_table_rows : num_seqs;
    return attention(q, k_cache, v_cache, num_blocks, 0, nullptr, nullptr, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, max_q_len, num_q_heads,
                     num_kv_heads, head_dim, scale, out, out_dtype, workspace, workspace_bytes,
                     stream, vl);
}

pkv_status pkv_kv_append_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                             int64_t n_new, void *k_cache, void *v_cache, int64_t num_blocks,
                             int32_t num_kv_heads, int32_t head_dim, const float *k_scale,
                             const float *v_scale, void *stream)
{
    if (n_new < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1)
        return PKV_ERR_SHAPE;
    if (n_new == 0)
        return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
        return PKV_ERR_NULL;
    if (head_dim % 8 != 0)
        return PKV_ERR_UNSUPPORTED;
    if (head_dim > 1024 || num_kv_heads > 1024 || n_new > 0x7fffffffLL ||
        num_blocks > (int64_t(1) << 40))
        return PKV_ERR_RANGE;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 8) ||
        !aligned(v_cache, 8) || !aligned(slot_mapping, 8) || !aligned(k_scale, 4) ||
        !aligned(v_scale, 4))
        return PKV_ERR_ALIGN;
    cudaError_t e = pkv::launch_kv_append_fp8(k_new, v_new, slot_mapping, n_new, k_cache,
                                              v_cache, num_blocks, num_kv_heads, head_dim,
                                              k_scale, v_scale, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"

namespace pkv {

pkv_status attention_need(const void *q, const void *k_cache, const void *v_cache,
                          int64_t num_blocks, const int32_t *block_tables,
                          int32_t max_blocks_per_seq, const int32_t *context_lens,
                          int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, void *out, int32_t out_dtype,
                          size_t *need)
{
    return attention(q, k_cache, v_cache, num_blocks, 0, nullptr, nullptr, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, n_query_per_seq, num_q_heads,
                     num_kv_heads, head_dim, 1.f, out, out_dtype, nullptr, 0, nullptr, Varlen(),
                     Cascade(), need);
}

pkv_status attention_check(const void *q, const void *k_cache, const void *v_cache,
                           int64_t num_blocks, int kv8, const float *k_scale,
                           const float *v_scale, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t n_query_per_seq, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, void *out, int32_t out_dtype,
                           size_t *need)
{
    return attention(q, k_cache, v_cache, num_blocks, kv8, k_scale, v_scale, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, n_query_per_seq, num_q_heads,
                     num_kv_heads, head_dim, 1.f, out, out_dtype, nullptr, 0, nullptr, Varlen(),
                     Cascade(), need);
}

}  // namespace pkv
