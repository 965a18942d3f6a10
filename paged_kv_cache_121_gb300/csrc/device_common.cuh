// Device-side building blocks shared by the decode kernels: parameter block,
// PTX wrappers (mbarrier, TMA and bulk copies, ldmatrix, mma), bounded waits,
// programmatic dependent launch, and the CUDA-core kernel's CTA epilogue,
// which writes either the final output or a split-K partition.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <cstdlib>

namespace pa {

constexpr int kRowsPerTile = 16;     // query heads per CTA (the MMA's M)
constexpr int kMaxSplits = 64;       // most partitions pa_decode's plan cuts one context into
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s: far above any legal wait

enum DecodeMode : int { kModeFinal = 0, kModeSplitK = 1 };
enum StatusCode : int { kStatusTimeout = 5 };

// Everything a decode launch needs; passed by value.
// Two kernels that read nothing of each other's output (the shared-prefix
// pass and the rest-of-context decode) overlap through programmatic
// dependent launch. The first waits for the stream as usual, then lets the
// second launch at once: the second is scheduled as soon as every CTA of the
// first has started, so no CTA ever waits on one that is not resident. The
// second skips the start-of-kernel wait (the first already made it) and
// instead waits for the first before it exits, so that its completion, which
// the next kernel waits for, implies the first's.
enum PairRole : int { kPairNone = 0, kPairFirst = 1, kPairSecond = 2 };

struct DecodeParams {
    const void *query;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    void *out;
    float *tmp_out;      // split-K mode
    float *max_logits;
    float *exp_sums;
    int *status;         // device status word
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size;
    int max_blocks, num_blocks;
    int contig_stride;   // > 0: contiguous cache [num_seqs, contig_stride, Hkv, D] (no
                         // block table; block_size is then the tile length)
    int group;           // num_heads / num_kv_heads
    int ntile;           // cdiv(group, 16)
    int heads_per_cta;   // KV heads one CTA serves (grid.y = Hkv / heads_per_cta * ntile)
    int ring_bytes;      // shared-memory ring of the tensor-core kernel
    int cluster_merge;   // fused split merged through distributed shared memory
                         // (grid.x = nsplit = cluster size)
    int nsplit;          // grid.x: partitions per (sequence, head tile)
    int part_tokens;     // tokens per partition (a multiple of the kernel's tile length)
    int skip_tokens;     // each context's first skip_tokens tokens are not attended here
                         // (a shared prefix attended by the prefix pass)
    int part_stride;     // split-K rows: partitions per (sequence, head) in tmp_out (0: nsplit)
    int part_offset;     //   and the index of this launch's partition 0 there
    int mode;
    int out_bf16;        // output element: bf16, else fp16 if out_f16, else fp32
    int out_f16;
    int q_bf16;
    int kv_f16;          // 16-bit query and caches are fp16 (else bf16)
    const void *append_key;     // [num_seqs, Hkv, D] or null: the step's new token of sequence b,
    const void *append_value;   //   written to position context_lens[b] - 1 before it is read
    int pair_role;              // PairRole: one of two overlapped kernels, or neither
    float scale_log2;    // scale * log2(e): scores are kept in base-2 units
};

// ---------------------------------------------------------------------------
// Programmatic dependent launch: every kernel of the library is launched so
// that it may be scheduled while the previous kernel on the stream finishes;
// it waits (griddepcontrol.wait) for that kernel's completion and memory
// before reading anything, and lets its own dependents be scheduled once its
// main work is done. Hides the launch gap between back-to-back kernels (in a
// CUDA graph too). PA_PDL=0 launches plainly.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

inline bool pdl_enabled() {
    static const bool v = [] {
        const char *e = std::getenv("PA_PDL");
        return !(e && e[0] == '0' && e[1] == 0);
    }();
    return v;
}

// Launch kern<<<grid, block, smem, stream>>>(args...) with programmatic
// stream serialization (unless disabled) and, if cluster_x > 1, a cluster of
// cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Shared-prefix pass: attention of every (sequence, query head) row over the
// shared leading blocks, one chunk per partition, in split-K form.
struct PrefixParams {
    const void *query;            // [B, Hq, D] bf16
    const int32_t *prefix_table;  // the shared leading block ids (a block-table row)
    const int32_t *context_lens;  // [B]
    float *tmp_out;               // [B, Hq, part_stride, D]: chunk c at partition c
    float *max_logits;            // [B, Hq, part_stride]
    float *exp_sums;              // [B, Hq, part_stride]
    int *status;                  // device status word
    int num_seqs, num_heads, num_kv_heads, head_dim, group, block_size;
    int prefix_tokens;            // tokens in the shared blocks attended here (a multiple of 16)
    int chunk_tokens;             // tokens per chunk (a multiple of 16)
    int part_stride;              // partitions per row in tmp_out
    int ring_bytes;
    int kv_f16;                   // query and caches are fp16 (else bf16)
    int seqs_per_group;           // tcgen05 pass: whole sequences per row group (rows = this x group)
    int row_groups;               // tcgen05 pass: row groups of the batch
    int pair_role;                // PairRole: one of two overlapped kernels, or neither
    float scale_log2;
};

// Raise a kernel's dynamic shared-memory limit once per device (host side;
// keeps the call out of CUDA-graph capture after the first launch). Each
// kernel instantiation passes its own `done` mask (bit d: device d set up).
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel kern, size_t bytes, unsigned long long &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess && bit) __atomic_fetch_or(&done, bit, __ATOMIC_ACQ_REL);
    return e;
}

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Two fp32 values into the output element type (out_type: 0 fp32, 1 bf16,
// 2 fp16, as the public dtype codes), at out + idx (idx even).
__device__ __forceinline__ void store_pair_as(void *out, int out_type, int64_t idx, float a, float c) {
    if (out_type == 1)
        *reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(out) + idx) = pack_bf16x2(a, c);
    else if (out_type == 2)
        *reinterpret_cast<uint32_t *>(static_cast<__half *>(out) + idx) = pack_f16x2(a, c);
    else
        *reinterpret_cast<float2 *>(static_cast<float *>(out) + idx) = make_float2(a, c);
}

// The decode's output element type as a dtype code.
__device__ __forceinline__ int out_type_of(const DecodeParams &p) { return p.out_bf16 ? 1 : p.out_f16 ? 2 : 0; }

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void record_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// mbarrier (shared::cta)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Raise the current phase's expected transaction bytes (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; gives up after
// limit_ns and returns false (the caller records a timeout and unwinds).
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u && global_timer_ns() - t0 > limit_ns) return false;
    }
}

// The kernels' wait: bounded by kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// ---------------------------------------------------------------------------
// TMA: 4-D tiled load global -> shared, completion counted on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
        "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, int c4, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar),
        "l"(policy)
        : "memory");
}

// Bulk copy of `bytes` (a multiple of 16) global -> shared, both addresses
// 16-byte aligned; completion is counted as transaction bytes on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------------------
// thread-block cluster: rank, peer shared-memory addresses, barrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_map(uint32_t local_smem_addr, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_smem_addr), "r"(rank));
    return a;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float2 ld_cluster_f32x2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

// All threads of every CTA of the cluster: writes before it are visible to
// reads after it, cluster-wide.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------------------
// warp-level tensor-core MMA (m16n8k16, bf16 in, fp32 accumulate)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The m16n8k16 product for 16-bit inputs of either kind.
template <bool kF16>
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (kF16) mma_f16_16816(c, a, b0, b1);
    else mma_bf16_16816(c, a, b0, b1);
}

// Split-K row of (sequence b, query head h, partition part) in tmp_out /
// max_logits / exp_sums.
__device__ __forceinline__ int64_t split_row(const DecodeParams &p, int b, int h, int part) {
    const int stride = p.part_stride > 0 ? p.part_stride : p.nsplit;
    return (static_cast<int64_t>(b) * p.num_heads + h) * stride + p.part_offset + part;
}

// ---------------------------------------------------------------------------
// Per-sequence bookkeeping shared by every decode kernel
// ---------------------------------------------------------------------------
struct SeqWork {
    int len;        // tokens attended (clamped to the cache's capacity and the grid's reach)
    int nparts;     // partitions with work
    int tok_begin;  // this CTA's first token
    int tok_end;    // one past its last token (<= tok_begin: nothing to do)
};

__device__ __forceinline__ SeqWork seq_work(const DecodeParams &p, int b, int part) {
    SeqWork w;
    int len = p.context_lens[b];
    if (len < 0) len = 0;
    const int cap = p.contig_stride > 0 ? p.contig_stride : p.max_blocks * p.block_size;
    if (len > cap) len = cap;
    const int first = min(p.skip_tokens, len);
    const int64_t reach = first + static_cast<int64_t>(p.nsplit) * p.part_tokens;
    if (len > reach) len = static_cast<int>(reach);
    w.len = len;
    w.nparts = (len - first + p.part_tokens - 1) / p.part_tokens;
    w.tok_begin = first + part * p.part_tokens;
    w.tok_end = min(len, w.tok_begin + p.part_tokens);
    return w;
}

// ---------------------------------------------------------------------------
// CTA result: per-warp partial softmax states combined, then written out.
//
// Shared-memory layout (floats), row stride D + 4:
//   warp region w: m[16], l[16], O[16][D+4]   for w < nwarps
//   cta region:    m[16], l[16], O[16][D+4]
// m is a running max of base-2 scores, l the sum of 2^(s - m), O the
// unnormalised sum of 2^(s - m) * v.
// ---------------------------------------------------------------------------
template <int D>
struct MergeLayout {
    static constexpr int kStride = D + 4;
    static constexpr int kRegion = 32 + kRowsPerTile * kStride;
    __device__ static float *m(float *base, int w) { return base + w * kRegion; }
    __device__ static float *l(float *base, int w) { return base + w * kRegion + 16; }
    __device__ static float *o(float *base, int w) { return base + w * kRegion + 32; }
    static constexpr size_t bytes(int nwarps) {
        return sizeof(float) * static_cast<size_t>(nwarps + 1) * kRegion;
    }
};

// Combine nwarps warp regions into the CTA region (all threads participate).
template <int D>
__device__ void combine_warps(float *base, int nwarps, int rows) {
    using L = MergeLayout<D>;
    float *cm = L::m(base, nwarps), *cl = L::l(base, nwarps), *co = L::o(base, nwarps);
    for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        float M = -INFINITY;
        for (int w = 0; w < nwarps; ++w) M = fmaxf(M, L::m(base, w)[r]);
        float acc = 0.f;
        if (M != -INFINITY)
            for (int w = 0; w < nwarps; ++w)
                acc += fast_exp2(L::m(base, w)[r] - M) * L::o(base, w)[r * L::kStride + d];
        co[r * L::kStride + d] = acc;
    }
    if (threadIdx.x < rows) {
        const int r = threadIdx.x;
        float M = -INFINITY;
        for (int w = 0; w < nwarps; ++w) M = fmaxf(M, L::m(base, w)[r]);
        float s = 0.f;
        if (M != -INFINITY)
            for (int w = 0; w < nwarps; ++w) s += fast_exp2(L::m(base, w)[r] - M) * L::l(base, w)[r];
        cm[r] = M;
        cl[r] = s;
    }
    __syncthreads();
}

__device__ __forceinline__ void store_out(const DecodeParams &p, int64_t idx, float v) {
    if (p.out_bf16)
        reinterpret_cast<__nv_bfloat16 *>(p.out)[idx] = __float2bfloat16_rn(v);
    else if (p.out_f16)
        reinterpret_cast<__half *>(p.out)[idx] = __float2half_rn(v);
    else
        reinterpret_cast<float *>(p.out)[idx] = v;
}

// Write rows [0, rows) of the CTA result for (b, kv head g, head tile, partition).
template <int D>
__device__ void write_result(const DecodeParams &p, float *base, int nwarps, int b, int g,
                             int tile, int part, int rows) {
    using L = MergeLayout<D>;
    float *cm = L::m(base, nwarps), *cl = L::l(base, nwarps), *co = L::o(base, nwarps);
    const int h0 = g * p.group + tile * kRowsPerTile;
    if (p.mode == kModeFinal) {
        for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
            const int r = idx / D, d = idx % D;
            const float l = cl[r];
            const float v = l > 0.f ? co[r * L::kStride + d] / l : 0.f;
            store_out(p, (static_cast<int64_t>(b) * p.num_heads + h0 + r) * D + d, v);
        }
        return;
    }
    // split-K: normalised partial output, its maximum (natural log units) and sum
    for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        const float l = cl[r];
        const int64_t row = split_row(p, b, h0 + r, part);
        p.tmp_out[row * D + d] = l > 0.f ? co[r * L::kStride + d] / l : 0.f;
    }
    if (threadIdx.x < rows) {
        const int r = threadIdx.x;
        const int64_t row = split_row(p, b, h0 + r, part);
        const float l = cl[r];
        p.max_logits[row] = l > 0.f ? cm[r] * kLn2 : -INFINITY;
        p.exp_sums[row] = l;
    }
}

// One warp, one KV head: rows h0 .. h0+rows-1 of a partition holding no tokens.
template <int D>
__device__ void warp_write_empty(const DecodeParams &p, int b, int h0, int part, int rows, int nparts,
                                 int lane) {
    if (p.mode == kModeSplitK) {
        for (int r = 0; r < rows; ++r) {
            const int64_t row = split_row(p, b, h0 + r, part);
            for (int d = lane; d < D; d += 32) p.tmp_out[row * D + d] = 0.f;
            if (lane == 0) {
                p.max_logits[row] = -INFINITY;
                p.exp_sums[row] = 0.f;
            }
        }
        return;
    }
    if (nparts == 0 && part == 0)
        for (int r = 0; r < rows; ++r)
            for (int d = lane; d < D; d += 32)
                store_out(p, (static_cast<int64_t>(b) * p.num_heads + h0 + r) * D + d, 0.f);
}

// A CTA whose partition holds no tokens.
template <int D>
__device__ void write_empty(const DecodeParams &p, int b, int g, int tile, int part, int rows,
                            int nparts) {
    const int h0 = g * p.group + tile * kRowsPerTile;
    if (p.mode == kModeSplitK) {
        for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
            const int r = idx / D, d = idx % D;
            const int64_t row = split_row(p, b, h0 + r, part);
            p.tmp_out[row * D + d] = 0.f;
        }
        if (threadIdx.x < rows) {
            const int64_t row = split_row(p, b, h0 + threadIdx.x, part);
            p.max_logits[row] = -INFINITY;
            p.exp_sums[row] = 0.f;
        }
        return;
    }
    // final: an empty sequence has one all-zero output row, written by partition 0
    if (nparts == 0 && part == 0)
        for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
            const int r = idx / D, d = idx % D;
            store_out(p, (static_cast<int64_t>(b) * p.num_heads + h0 + r) * D + d, 0.f);
        }
}

}  // namespace pa
