// The two companion kernels of paged decode.
//
// reshape_and_cache: each new token's key and value rows (all KV heads) are
// written into its slot of the block pool -- "PagedAttention, explained.",
// procedure step 4 and "Across GPUs" (the fused write kernels); slot =
// block * block_size + offset, "Paged Attention: Virtual Memory for the KV
// Cache", section "Finding a token: position, block, slot". In the
// [num_blocks, block_size, Hkv, D] layout a slot is one contiguous row of
// Hkv * D elements, so the scatter is a row copy with 16-byte vectors.
//
// copy_blocks: copy-on-write clones whole blocks before a shared block is
// written -- "PagedAttention: KV cache virtual memory", section
// "Copy-on-write"; "How PagedAttention Eliminates KV-Cache Fragmentation",
// section "Advanced Memory Sharing and Copy-on-Write". Each CTA copies one
// 8 KiB chunk of one block of one cache with 16-byte vectors.
//
// swap_blocks: the same whole-block copy between two pools, either of which
// may be page-locked host memory -- preempted sequences' blocks are moved to
// CPU memory and back ("PagedAttention, explained.", procedure steps 7 and 8;
// "What Does PagedAttention Actually Optimize?", section 12). The pages note
// that swapping small blocks is slow because it means many small transfers;
// here one kernel moves every block of the request, each CTA streaming an
// 8 KiB chunk over the CPU-GPU link with 16-byte accesses.
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "internal.h"

namespace pa {

__global__ void __launch_bounds__(128)
reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                         uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const int64_t *__restrict__ slot_mapping, int64_t num_slots, int row_vecs) {
    grid_dependency_wait();
    grid_dependents_launch();
    const int i = blockIdx.x;
    const int64_t slot = slot_mapping[i];
    if (slot < 0 || slot >= num_slots) return;
    const uint4 *ks = key + static_cast<int64_t>(i) * row_vecs;
    const uint4 *vs = value + static_cast<int64_t>(i) * row_vecs;
    uint4 *kd = k_cache + slot * row_vecs;
    uint4 *vd = v_cache + slot * row_vecs;
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) {
        const uint4 a = ks[c];
        const uint4 v = vs[c];
        kd[c] = a;
        vd[c] = v;
    }
}

cudaError_t launch_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                     void *v_cache, const int64_t *slot_mapping, int num_tokens,
                                     int64_t num_slots, int row_bytes, cudaStream_t stream) {
    const int row_vecs = row_bytes / 16;
    const int threads = row_vecs >= 128 ? 128 : ((row_vecs + 31) / 32) * 32;
    return launch_kernel(reshape_and_cache_kernel, dim3(num_tokens), dim3(threads), 0, stream, 1u,
                         static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
                         static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slot_mapping,
                         num_slots, row_vecs);
}

// The step's new token of every sequence, written to position
// context_lens[b] - 1 (its slot taken from the block table): the scatter of
// pa_decode_append where the decode kernel does not write it itself. One CTA
// per sequence; lengths of 0, or past len_cap, write nothing.
__global__ void __launch_bounds__(128)
append_last_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value, uint4 *__restrict__ k_cache,
                   uint4 *__restrict__ v_cache, const int32_t *__restrict__ block_tables,
                   const int32_t *__restrict__ context_lens, int max_blocks, int block_size, int num_blocks,
                   int len_cap, int row_vecs) {
    grid_dependency_wait();
    grid_dependents_launch();
    const int b = blockIdx.x;
    const int len = context_lens[b];
    if (len <= 0 || len > len_cap || len > max_blocks * block_size) return;
    const int pos = len - 1;
    const int blk = block_tables[static_cast<int64_t>(b) * max_blocks + pos / block_size];
    if (blk < 0 || blk >= num_blocks) return;
    const int64_t slot = static_cast<int64_t>(blk) * block_size + pos % block_size;
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) {
        const uint4 a = key[static_cast<int64_t>(b) * row_vecs + c];
        const uint4 v = value[static_cast<int64_t>(b) * row_vecs + c];
        k_cache[slot * row_vecs + c] = a;
        v_cache[slot * row_vecs + c] = v;
    }
}

cudaError_t launch_append_last(const void *key, const void *value, void *k_cache, void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                               int max_blocks, int block_size, int num_blocks, int len_cap, int row_bytes,
                               cudaStream_t stream) {
    const int row_vecs = row_bytes / 16;
    const int threads = row_vecs >= 128 ? 128 : ((row_vecs + 31) / 32) * 32;
    return launch_kernel(append_last_kernel, dim3(num_seqs), dim3(threads), 0, stream, 1u,
                         static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
                         static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), block_tables,
                         context_lens, max_blocks, block_size, num_blocks, len_cap, row_vecs);
}

constexpr int kCopyChunkVecs = 512;  // 8 KiB per CTA

__global__ void __launch_bounds__(256)
transfer_blocks_kernel(uint4 *__restrict__ dst_k, uint4 *__restrict__ dst_v, const uint4 *__restrict__ src_k,
                       const uint4 *__restrict__ src_v, const int64_t *__restrict__ block_mapping,
                       int64_t src_blocks, int64_t dst_blocks, int64_t block_vecs) {
    grid_dependency_wait();
    grid_dependents_launch();
    const int pair = blockIdx.x;
    const int which = blockIdx.y & 1;
    const int64_t chunk = blockIdx.y >> 1;
    const int64_t src = block_mapping[2 * static_cast<int64_t>(pair)];
    const int64_t dst = block_mapping[2 * static_cast<int64_t>(pair) + 1];
    if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) return;
    const uint4 *s = (which ? src_v : src_k) + src * block_vecs;
    uint4 *d = (which ? dst_v : dst_k) + dst * block_vecs;
    const int64_t c0 = chunk * kCopyChunkVecs;
    const int64_t c1 = c0 + kCopyChunkVecs < block_vecs ? c0 + kCopyChunkVecs : block_vecs;
    // all loads of the chunk in flight before the stores (the source may be
    // host memory across the CPU-GPU link)
    constexpr int kPer = kCopyChunkVecs / 256;
    uint4 v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int64_t c = c0 + threadIdx.x + j * 256;
        if (c < c1) v[j] = s[c];
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int64_t c = c0 + threadIdx.x + j * 256;
        if (c < c1) d[c] = v[j];
    }
}

cudaError_t launch_transfer_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                                   const int64_t *block_mapping, int num_pairs, int64_t src_blocks,
                                   int64_t dst_blocks, int64_t block_bytes, cudaStream_t stream) {
    const int64_t block_vecs = block_bytes / 16;
    const int64_t chunks = (block_vecs + kCopyChunkVecs - 1) / kCopyChunkVecs;
    if (chunks * 2 > 65535) return cudaErrorInvalidValue;
    dim3 grid(num_pairs, static_cast<unsigned>(chunks * 2));
    return launch_kernel(transfer_blocks_kernel, grid, dim3(256), 0, stream, 1u, static_cast<uint4 *>(dst_k),
                         static_cast<uint4 *>(dst_v), static_cast<const uint4 *>(src_k),
                         static_cast<const uint4 *>(src_v), block_mapping, src_blocks, dst_blocks, block_vecs);
}

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int64_t *block_mapping,
                               int num_pairs, int64_t num_blocks, int64_t block_bytes,
                               cudaStream_t stream) {
    return launch_transfer_blocks(k_cache, v_cache, k_cache, v_cache, block_mapping, num_pairs, num_blocks,
                                  num_blocks, block_bytes, stream);
}

}  // namespace pa
