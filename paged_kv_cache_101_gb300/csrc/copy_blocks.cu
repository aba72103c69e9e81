// copy_blocks.cu -- copy whole physical blocks of the paged pool (the device
// half of copy-on-write).
//
// "ML Interview Prep, Lesson 13" section 3.5 "Sharing": before a sequence
// writes into a block whose reference count is above 1 it gets a private copy.
// The host block manager picks the (source, destination) pairs; this kernel
// moves the bytes. A block is 16 token rows of [Hkv][D] bf16 in K and the same
// in V: 2 * 16 * Hkv * D * 2 bytes (64 KiB at Hkv = 8, D = 128).
//
// Grid: x = pair, y = 16 KiB chunks of the pair's K-then-V bytes. Each thread
// issues its four 16-byte loads before any store, so a CTA keeps 16 KiB in
// flight and the copy streams at HBM speed once there are a few hundred pairs.
// Pairs naming a block outside the pool, or src == dst, are skipped.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {

namespace {
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int64_t kCopyChunkVecs = int64_t(kCopyThreads) * kCopyUnroll;  // 16 KiB
}  // namespace

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, const int32_t *__restrict__ src,
    const int32_t *__restrict__ dst, int64_t num_blocks, int64_t block_vecs, int64_t chunks)
{
    const int64_t a = __ldg(src + blockIdx.x);
    const int64_t b = __ldg(dst + blockIdx.x);
    if (a < 0 || a >= num_blocks || b < 0 || b >= num_blocks || a == b)
        return;
    const int64_t total = 2 * block_vecs;  // K vectors, then V vectors
    for (int64_t c = blockIdx.y; c < chunks; c += gridDim.y) {
        const int64_t base = c * kCopyChunkVecs + threadIdx.x;
        uint4 r[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t e = base + u * kCopyThreads;
            if (e < total) {
                const uint4 *from = e < block_vecs ? k_cache + a * block_vecs + e
                                                   : v_cache + a * block_vecs + (e - block_vecs);
                r[u] = __ldcs(from);
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t e = base + u * kCopyThreads;
            if (e < total) {
                uint4 *to = e < block_vecs ? k_cache + b * block_vecs + e
                                           : v_cache + b * block_vecs + (e - block_vecs);
                *to = r[u];
            }
        }
    }
}

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, int64_t num_blocks, int num_kv_heads,
                               int head_dim, const int32_t *src, const int32_t *dst,
                               int num_pairs, cudaStream_t stream)
{
    const int64_t block_vecs = int64_t(kBlockSize) * num_kv_heads * head_dim / 8;
    const int64_t chunks = (2 * block_vecs + kCopyChunkVecs - 1) / kCopyChunkVecs;
    const unsigned gy = unsigned(chunks < 65535 ? chunks : 65535);
    copy_blocks_kernel<<<dim3(unsigned(num_pairs), gy), kCopyThreads, 0, stream>>>(
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), src, dst, num_blocks,
        block_vecs, chunks);
    return cudaGetLastError();
}

}  // namespace pkv
