// Paged decode attention on the CUDA cores (fp32 caches, and bf16 or fp16
// caches whose block size the tensor-core kernel does not take), plus the
// log-sum-exp merge of split-K partitions.
//
// Same work decomposition and epilogue as the tensor-core kernel: one CTA per
// (sequence, KV head, head tile, partition). The four warps take the
// partition's tokens four at a time, round robin; a lane owns head_dim/32
// consecutive dims (one coalesced vector load per K or V row), a warp loads
// its four tokens' K and V rows before using any, dot products are reduced
// with warp shuffles, and the online softmax runs in fp32 in base 2.
// Pages: "What Does PagedAttention Actually Optimize?", sections 8, 14 and
// 17 (read_kv: logical block = t / B, offset = t % B, physical block from the
// table).
#include "device_common.cuh"
#include "internal.h"

namespace pa {

template <int E, typename KV>
struct RowLoad;

template <int E>
struct RowLoad<E, float> {
    __device__ static void load(const float *row, float (&x)[E]) {
        if constexpr (E == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(row);
            x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
        } else if constexpr (E == 2) {
            const float2 v = *reinterpret_cast<const float2 *>(row);
            x[0] = v.x; x[1] = v.y;
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) x[e] = row[e];
        }
    }
};

template <int E>
struct RowLoad<E, __nv_bfloat16> {
    __device__ static void load(const __nv_bfloat16 *row, float (&x)[E]) {
        if constexpr (E == 4) {
            const uint2 v = *reinterpret_cast<const uint2 *>(row);
            x[0] = bf16_bits_to_float(v.x & 0xffffu); x[1] = bf16_bits_to_float(v.x >> 16);
            x[2] = bf16_bits_to_float(v.y & 0xffffu); x[3] = bf16_bits_to_float(v.y >> 16);
        } else if constexpr (E == 2) {
            const uint32_t v = *reinterpret_cast<const uint32_t *>(row);
            x[0] = bf16_bits_to_float(v & 0xffffu); x[1] = bf16_bits_to_float(v >> 16);
        } else {
            const uint16_t *u = reinterpret_cast<const uint16_t *>(row);
#pragma unroll
            for (int e = 0; e < E; ++e) x[e] = bf16_bits_to_float(u[e]);
        }
    }
};

template <int E>
struct RowLoad<E, __half> {
    __device__ static void load(const __half *row, float (&x)[E]) {
        if constexpr (E == 4) {
            const uint2 v = *reinterpret_cast<const uint2 *>(row);
            const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
            const float2 c = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
            x[0] = a.x; x[1] = a.y; x[2] = c.x; x[3] = c.y;
        } else if constexpr (E == 2) {
            const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(row));
            x[0] = a.x; x[1] = a.y;
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) x[e] = __half2float(row[e]);
        }
    }
};

template <int D, int MAXR, typename KV>
__global__ void __launch_bounds__(128)
decode_simt_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int E = D / 32;
    constexpr int kWarps = 4;
    extern __shared__ float smem_f[];

    const int part = blockIdx.x;
    const int g = blockIdx.y / p.ntile;
    const int tile = blockIdx.y % p.ntile;
    const int b = blockIdx.z;
    const int rows = min(kRowsPerTile, p.group - tile * kRowsPerTile);
    grid_dependency_wait();
    const SeqWork w = seq_work(p, b, part);
    if (w.tok_begin >= w.tok_end) {
        write_empty<D>(p, b, g, tile, part, rows, w.nparts);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h0 = g * p.group + tile * kRowsPerTile;

    float q[MAXR][E], o[MAXR][E], m[MAXR], l[MAXR];
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) o[r][e] = q[r][e] = 0.f;
        if (r < rows) {
            const int64_t off = (static_cast<int64_t>(b) * p.num_heads + h0 + r) * D + lane * E;
            RowLoad<E, KV>::load(static_cast<const KV *>(p.query) + off, q[r]);   // the query has the caches' type
        }
    }

    const KV *kc = static_cast<const KV *>(p.k_cache);
    const KV *vc = static_cast<const KV *>(p.v_cache);
    const int32_t *table = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;
    const int t_begin = w.tok_begin;
    const int t_end = w.tok_end;
    // Each warp takes kTok consecutive tokens per iteration and loads all
    // their K and V rows before using any (2 kTok row loads in flight per
    // warp), then folds the kTok scores of each query row into its online
    // softmax at once. A block id outside the pool reads as zeros.
    constexpr int kTok = 4;
    for (int t0 = t_begin + warp * kTok; t0 < t_end; t0 += kWarps * kTok) {
        float kx[kTok][E], vx[kTok][E];
#pragma unroll
        for (int u = 0; u < kTok; ++u) {
            const int t = t0 + u;
            const int64_t phys = t < t_end ? table[t / p.block_size] : -1;
            if (phys >= 0 && phys < p.num_blocks) {
                const int64_t row = ((phys * p.block_size + t % p.block_size) * p.num_kv_heads + g) * D + lane * E;
                RowLoad<E, KV>::load(kc + row, kx[u]);
                RowLoad<E, KV>::load(vc + row, vx[u]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) kx[u][e] = vx[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < MAXR; ++r) {
            if (r >= rows) break;
            float s[kTok];
#pragma unroll
            for (int u = 0; u < kTok; ++u) {
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) acc = fmaf(q[r][e], kx[u][e], acc);
                s[u] = acc;
            }
#pragma unroll
            for (int off = 16; off; off >>= 1)
#pragma unroll
                for (int u = 0; u < kTok; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
            float mn = m[r];
#pragma unroll
            for (int u = 0; u < kTok; ++u) {
                s[u] = t0 + u < t_end ? s[u] * p.scale_log2 : -INFINITY;   // tokens past the partition: weight 0
                mn = fmaxf(mn, s[u]);
            }
            const float a = fast_exp2(m[r] - mn);
            float pr[kTok], ps = 0.f;
#pragma unroll
            for (int u = 0; u < kTok; ++u) {
                pr[u] = fast_exp2(s[u] - mn);
                ps += pr[u];
            }
            l[r] = l[r] * a + ps;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                float acc = o[r][e] * a;
#pragma unroll
                for (int u = 0; u < kTok; ++u) acc = fmaf(pr[u], vx[u][e], acc);
                o[r][e] = acc;
            }
            m[r] = mn;
        }
    }

    using L = MergeLayout<D>;
#pragma unroll
    for (int r = 0; r < kRowsPerTile; ++r) {
        if (r < MAXR) {
#pragma unroll
            for (int e = 0; e < E; ++e) L::o(smem_f, warp)[r * L::kStride + lane * E + e] = o[r][e];
            if (lane == 0) {
                L::m(smem_f, warp)[r] = m[r];
                L::l(smem_f, warp)[r] = l[r];
            }
        } else if (lane == 0) {
            L::m(smem_f, warp)[r] = -INFINITY;
            L::l(smem_f, warp)[r] = 0.f;
        }
    }
    __syncthreads();
    combine_warps<D>(smem_f, kWarps, rows);
    grid_dependents_launch();
    write_result<D>(p, smem_f, kWarps, b, g, tile, part, rows);
}

template <int D, int MAXR, typename KV>
static cudaError_t launch_simt_impl(const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    auto kern = decode_simt_kernel<D, MAXR, KV>;
    const size_t smem = MergeLayout<D>::bytes(4);
    static unsigned long long done = 0;
    cudaError_t e = ensure_smem_limit(kern, smem, done);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, dim3(128), smem, stream, 1u, p);
}

template <int D, typename KV>
static cudaError_t launch_simt_rows(const DecodeParams &p, dim3 grid, cudaStream_t stream) {
    const int rows = p.group < kRowsPerTile ? p.group : kRowsPerTile;
    if (rows <= 1) return launch_simt_impl<D, 1, KV>(p, grid, stream);
    if (rows <= 2) return launch_simt_impl<D, 2, KV>(p, grid, stream);
    if (rows <= 4) return launch_simt_impl<D, 4, KV>(p, grid, stream);
    if (rows <= 8) return launch_simt_impl<D, 8, KV>(p, grid, stream);
    return launch_simt_impl<D, 16, KV>(p, grid, stream);
}

template <int D>
static cudaError_t launch_simt_dim(const DecodeParams &p, int kv_type, dim3 grid, cudaStream_t stream) {
    if (kv_type == 1) return launch_simt_rows<D, __nv_bfloat16>(p, grid, stream);
    if (kv_type == 2) return launch_simt_rows<D, __half>(p, grid, stream);
    return launch_simt_rows<D, float>(p, grid, stream);
}

cudaError_t launch_decode_simt(const DecodeParams &p, int kv_type, dim3 grid, cudaStream_t stream) {
    if (p.head_dim == 128) return launch_simt_dim<128>(p, kv_type, grid, stream);
    if (p.head_dim == 64) return launch_simt_dim<64>(p, kv_type, grid, stream);
    return cudaErrorInvalidValue;
}

__device__ __forceinline__ void store_merged(void *out, int out_type, int64_t idx, float v) {
    if (out_type == 1)
        reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
    else if (out_type == 2)
        reinterpret_cast<__half *>(out)[idx] = __float2half_rn(v);
    else
        reinterpret_cast<float *>(out)[idx] = v;
}

// ---------------------------------------------------------------------------
// log-sum-exp merge of split-K partitions: one CTA per (head, sequence).
// Two forms of the same merge (an empty partition has sum 0 and weight 0):
//  * lse_merge_kernel, for many rows (CTAs) per SM: warp 0 turns every
//    partition's max and sum into a weight in shared memory, once per CTA,
//    then every thread combines its output dim's values; few registers, so
//    many CTAs stay resident and hide each other's latency.
//  * lse_merge_online_kernel, for few rows per SM (long contexts: a handful
//    of CTAs, each latency-bound): no barrier. Partitions are taken eight at a
//    time: every lane issues its column's eight values while lane j < 8 loads
//    partition j's max and sum, so a batch costs one round trip to L2; the
//    warp moves its running max by a shuffle reduction, lane j computes
//    partition j's weight, and the weights are broadcast by shuffles.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128)
lse_merge_kernel(void *out, int out_type, const float *tmp_out, const float *max_logits,
                 const float *exp_sums, const int32_t *context_lens, int num_heads, int head_dim,
                 int max_partitions, int partition_size) {
    extern __shared__ float wgt[];  // [max_partitions]
    __shared__ float s_inv;
    const int h = blockIdx.x, b = blockIdx.y;
    grid_dependency_wait();
    grid_dependents_launch();
    int len = context_lens[b];
    if (len < 0) len = 0;
    // partition_size 0: every partition of the row (empty ones carry a zero sum)
    const int np = partition_size > 0 ? min((len + partition_size - 1) / partition_size, max_partitions)
                                      : max_partitions;
    const int64_t row0 = (static_cast<int64_t>(b) * num_heads + h) * max_partitions;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        float M = -INFINITY;
        for (int q = lane; q < np; q += 32)
            if (exp_sums[row0 + q] > 0.f) M = fmaxf(M, max_logits[row0 + q]);
#pragma unroll
        for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float tot = 0.f;
        for (int q = lane; q < np; q += 32) {
            const float es = exp_sums[row0 + q];
            const float wq = es > 0.f ? es * fast_exp2((max_logits[row0 + q] - M) * kLog2e) : 0.f;
            wgt[q] = wq;
            tot += wq;
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
        if (lane == 0) s_inv = tot > 0.f ? 1.f / tot : 0.f;
    }
    __syncthreads();
    const float inv = s_inv;
    for (int d = threadIdx.x; d < head_dim; d += blockDim.x) {
        // independent loads, unrolled (an empty partition holds zeros, weight 0)
        float acc = 0.f;
        const float *src = tmp_out + row0 * head_dim + d;
#pragma unroll 8
        for (int q = 0; q < np; ++q) acc += wgt[q] * __ldcg(src + static_cast<int64_t>(q) * head_dim);
        store_merged(out, out_type, (static_cast<int64_t>(b) * num_heads + h) * head_dim + d, acc * inv);
    }
}

constexpr int kMergeBatch = 8;

__global__ void __launch_bounds__(128)
lse_merge_online_kernel(void *out, int out_type, const float *tmp_out, const float *max_logits,
                        const float *exp_sums, const int32_t *context_lens, int num_heads, int head_dim,
                        int max_partitions, int partition_size) {
    const int h = blockIdx.x, b = blockIdx.y, lane = threadIdx.x & 31;
    grid_dependency_wait();
    grid_dependents_launch();
    int len = context_lens[b];
    if (len < 0) len = 0;
    const int np = partition_size > 0 ? min((len + partition_size - 1) / partition_size, max_partitions)
                                      : max_partitions;
    const int64_t row0 = (static_cast<int64_t>(b) * num_heads + h) * max_partitions;
    const float *ml = max_logits + row0, *es = exp_sums + row0;
    // (warp-uniform trip counts: every lane of a warp takes part in the shuffles)
    for (int d0 = threadIdx.x & ~31; d0 < head_dim; d0 += blockDim.x) {
        const int d = d0 + lane;
        const bool col = d < head_dim;
        const float *src = tmp_out + row0 * head_dim + d;
        float M = -INFINITY, L = 0.f, acc = 0.f;
        for (int q0 = 0; q0 < np; q0 += kMergeBatch) {
            float o[kMergeBatch];
#pragma unroll
            for (int j = 0; j < kMergeBatch; ++j)
                o[j] = (col && q0 + j < np) ? __ldcg(src + static_cast<int64_t>(q0 + j) * head_dim) : 0.f;
            const bool mine = lane < kMergeBatch && q0 + lane < np;   // lane j: partition q0 + j
            const float lj = mine ? __ldcg(es + q0 + lane) : 0.f;
            const float mj = mine ? __ldcg(ml + q0 + lane) : -INFINITY;
            float Mc = lj > 0.f ? mj : -INFINITY;
#pragma unroll
            for (int off = kMergeBatch / 2; off; off >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, off));
            Mc = fmaxf(__shfl_sync(0xffffffffu, Mc, 0), M);
            if (Mc > M) {   // the running max moves: rescale what is summed so far
                const float sc = fast_exp2((M - Mc) * kLog2e);
                L *= sc;
                acc *= sc;
                M = Mc;
            }
            const float wj = lj > 0.f ? lj * fast_exp2((mj - M) * kLog2e) : 0.f;
#pragma unroll
            for (int j = 0; j < kMergeBatch; ++j) {
                const float w = __shfl_sync(0xffffffffu, wj, j);
                L += w;
                acc += w * o[j];
            }
        }
        if (col) store_merged(out, out_type, (static_cast<int64_t>(b) * num_heads + h) * head_dim + d,
                              L > 0.f ? acc / L : 0.f);
    }
}

cudaError_t launch_lse_merge(void *out, int out_type, const float *tmp_out, const float *max_logits,
                             const float *exp_sums, const int32_t *context_lens, int num_seqs,
                             int num_heads, int head_dim, int max_partitions, int partition_size,
                             int sms, cudaStream_t stream) {
    if (head_dim <= 0) return cudaErrorInvalidValue;
    const unsigned threads = head_dim >= 128 ? 128u : static_cast<unsigned>((head_dim + 31) / 32 * 32);
    dim3 grid(num_heads, num_seqs);
    const int64_t rows = static_cast<int64_t>(num_seqs) * num_heads;
    if (rows <= static_cast<int64_t>(kMergeOnlineRowsPerSm) * sms)
        return launch_kernel(lse_merge_online_kernel, grid, dim3(threads), 0, stream, 1u, out, out_type, tmp_out,
                             max_logits, exp_sums, context_lens, num_heads, head_dim, max_partitions,
                             partition_size);
    const size_t smem = sizeof(float) * static_cast<size_t>(max_partitions);
    if (smem > 48 * 1024) {
        static unsigned long long done = 0;
        cudaError_t e = ensure_smem_limit(lse_merge_kernel, 200 * 1024, done);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(lse_merge_kernel, grid, dim3(threads), smem, stream, 1u, out, out_type, tmp_out,
                         max_logits, exp_sums, context_lens, num_heads, head_dim, max_partitions,
                         partition_size);
}

}  // namespace pa
