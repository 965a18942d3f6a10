// Launchers shared between the translation units of libpa (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

struct DecodeParams;
struct PrefixParams;

bool decode_mma_supported(int head_dim, int block_size);   // D 64/128, blocks of 1..256 (powers of two)
int decode_mma_tile_tokens(int block_size);       // tokens per pipeline stage (16)
int decode_mma_box_tokens(int block_size);        // rows per TMA box: min(block_size, 16)
int decode_mma_heads_per_cta(int num_kv_heads, int max_heads);   // KV heads (consumer warps) per CTA
int decode_mma_stage_bytes(int head_dim, int block_size, int heads_per_cta);
int decode_mma_ring_bytes(int head_dim, int block_size, int heads_per_cta, int budget_bytes);   // whole stages
int decode_mma_cluster_bytes(int head_dim, int heads_per_cta);   // shared memory the cluster merge needs
constexpr int kMaxClusterSplits = 8;                              // portable cluster size
cudaError_t launch_decode_mma(const DecodeParams &p, const CUtensorMap &tmap_k,
                              const CUtensorMap &tmap_v, dim3 grid, cudaStream_t stream);
// Shared-prefix pass (prefix_mma.cu): grid (chunks, Hkv, row groups).
constexpr int kPrefixMaxRingBytes = 128 * 1024;
int prefix_rows_per_cta();
int prefix_stage_bytes(int head_dim);
cudaError_t launch_prefix_mma(const PrefixParams &p, const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                              dim3 grid, cudaStream_t stream);
// Shared-prefix pass on tcgen05 (prefix_tc.cu): grid (chunks, Hkv, cdiv(row groups, groups_per_cta)).
// A row group is floor(128 / G) whole sequences x their G query heads (G <= 128).
constexpr int kTcMaxRingBytes = 192 * 1024;
constexpr int kTcChunkBlocks = 256;   // most block ids one chunk of the tcgen05 pass may span
int prefix_tc_max_rows();             // rows of a row group at most (tensor-memory lanes)
int prefix_tc_tile_tokens();
int prefix_tc_stage_bytes(int head_dim);
int prefix_tc_out_cols();             // fp32 columns per box of the partial-output store map
// ring bytes for a budget, clamped to what the kernel needs and its shared memory allows
int prefix_tc_ring_bytes(int head_dim, int groups_per_cta, int budget_bytes);
// tmap_q: query as (dim, half, head in group, KV head, sequence), box (64, 1, G, 1, seqs_per_group);
// tmap_o: tmp_out as (dim, partition, head, sequence), box (out_cols, 1, G, seqs_per_group), fp32
cudaError_t launch_prefix_tc(const PrefixParams &p, int groups_per_cta, const CUtensorMap &tmap_k,
                             const CUtensorMap &tmap_v, const CUtensorMap &tmap_q, const CUtensorMap &tmap_o,
                             dim3 grid, cudaStream_t stream);
// Balanced decode (decode_balanced.cu): the batch's tiles, concatenated
// sequence after sequence, cut into `ctas` equal ranges per (KV-head group,
// head tile); pieces of a sequence split between CTAs are merged after.
struct BalancedParams {
    int ctas;       // CTAs per (KV-head group, head tile): grid.x
    int len_cap;    // tokens past this are not attended (max_context_len)
    int *prefix;    // [num_seqs + 1] tile prefix sums, written by the decode for the merge
};
constexpr int kBalancedMaxSeqs = 2048;   // the prefix sums live in shared memory
bool decode_balanced_supported(int head_dim, int block_size);
size_t decode_balanced_smem_extra(int num_seqs);
cudaError_t launch_decode_balanced(const DecodeParams &p, const BalancedParams &bp, const CUtensorMap &tmap_k,
                                   const CUtensorMap &tmap_v, dim3 grid, cudaStream_t stream);
cudaError_t launch_balanced_merge(const DecodeParams &p, const BalancedParams &bp, cudaStream_t stream);
cudaError_t launch_append_last(const void *key, const void *value, void *k_cache, void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                               int max_blocks, int block_size, int num_blocks, int len_cap, int row_bytes,
                               cudaStream_t stream);
// kv_type / out_type: 0 fp32, 1 bf16, 2 fp16 (the public dtype codes)
cudaError_t launch_decode_simt(const DecodeParams &p, int kv_type, dim3 grid, cudaStream_t stream);
// The log-sum-exp merge; `sms` (the device's SM count) picks its form: with
// at most kMergeOnlineRowsPerSm (sequence, head) rows per SM, the
// barrier-free online merge (latency-bound), else the shared-weights one.
constexpr int kMergeOnlineRowsPerSm = 4;
cudaError_t launch_lse_merge(void *out, int out_type, const float *tmp_out, const float *max_logits,
                             const float *exp_sums, const int32_t *context_lens, int num_seqs,
                             int num_heads, int head_dim, int max_partitions, int partition_size,
                             int sms, cudaStream_t stream);
cudaError_t launch_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                     void *v_cache, const int64_t *slot_mapping, int num_tokens,
                                     int64_t num_slots, int row_bytes, cudaStream_t stream);
// Arguments of a decode call (mirrors pa_decode, dtypes as pa_dtype values).
struct DecodeCall {
    void *out;
    int out_dtype;
    const void *query;
    int q_dtype;
    const void *k_cache;
    const void *v_cache;
    int kv_dtype;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
        max_context_len;
    float scale;
};

// Decode with pa_decode's plan for a caller with a workspace, the
// ragged-balanced path aside: a split that fits a thread-block cluster is
// merged there; a wider one writes its partials into `scratch` and the merge
// kernel reads them back (every entry it reads is written by the same call).
// Returns a pa_status value; PA_ERR_WORKSPACE (checked before any pointer)
// when a wider split needs more than scratch_bytes.
int decode_into_scratch(const DecodeCall &c, void *scratch, size_t scratch_bytes, void *stream);

// The device status word of the current device (nullptr on a CUDA error).
int *device_status_word();
// Launch the bounded-wait check (health.cu): one CTA waits on an mbarrier
// phase that no copy completes, gives up after limit_ns and records a
// timeout in `status`.
cudaError_t launch_wait_timeout_check(int *status, unsigned long long limit_ns, cudaStream_t stream);

cudaError_t launch_transfer_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                                   const int64_t *block_mapping, int num_pairs, int64_t src_blocks,
                                   int64_t dst_blocks, int64_t block_bytes, cudaStream_t stream);

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int64_t *block_mapping,
                               int num_pairs, int64_t num_blocks, int64_t block_bytes,
                               cudaStream_t stream);

}  // namespace pa
