// C ABI of libpa: argument checks, work planning, TMA descriptors, launches.
// Declarations and the contract of each entry point are in include/pa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/pa.h"
#include "device_common.cuh"
#include "internal.h"

namespace pa {

// Device status word (one per device that loads the library): kernels record
// a bounded-wait timeout here; read and cleared through pa_device_status.
__device__ int g_device_status;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kCtasPerSmMma = 2;      // CTAs per SM the split plan aims at: tensor-core kernel,
constexpr int kCtasPerSmSimt = 12;    //   CUDA-core kernel (its 4-warp CTAs are latency-bound: more of
                                      //   them hide more; Qwen3 layer 558 -> 238 us from 2 to 12)
constexpr int kMmaHeadsPerCta = 4;    // KV heads per tensor-core CTA (consumer warps)
constexpr int kContiguousTile = 16;   // tokens per tile of a contiguous cache
constexpr int kMmaRingKiB = 96;       // shared-memory ring per tensor-core CTA: three stages when a
                                      // cluster merges the split,
constexpr int kSplitRingKiB = 64;     // two when the split goes through the workspace (measured on
                                      // GB300: 4 x 32 K tokens 87.0-87.5 us against 89.1-89.5 with three)
constexpr int kPrefixTcRingKiB = 192;  // tcgen05 prefix pass: as many stages as fit beside Q and P
constexpr int kBalancedHeadsPerCta = 8;   // ragged-balanced decode: every KV head of a group in one CTA,
constexpr int kBalancedCtasPerSm = 1;     //   one CTA per SM,
constexpr int kBalancedRingKiB = 132;     //   two 64 KiB stages (93.6 us against 94.0 with three)
constexpr int kMinSplitTokens = 256;  // do not split a context finer than this
constexpr int kMinPrefixChunk = 64;   // tokens per chunk of the shared-prefix pass, at least
constexpr int kMinRestSplitTokens = 64;   // partitions of the rest of a shared-prefix context, at least
constexpr int kRestCtasPerSm = 2;         // the rest's split: two CTAs per SM (it runs beside the prefix pass)
// The SM share of a prefix pass that runs first (measured over fourteen
// copy-on-write shapes on GB300): one unit of its work (a 64-token tile of
// one 128-row group and KV head) weighs as much as this many MB of the
// rest-of-context decode's K/V; at this share or above it takes every SM.
constexpr double kPrefixUnitMB = 0.12;
constexpr double kPrefixAllSmsFrac = 0.85;

std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int *> g_status_addr[kMaxDevices];

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int element_bytes(pa_dtype t) { return t == PA_F32 ? 4 : 2; }

bool valid_dtype(pa_dtype t) { return t == PA_F32 || t == PA_BF16 || t == PA_F16; }

// bf16 and fp16 share the tensor-core kernels (one instantiation each)
bool is16(pa_dtype t) { return t == PA_BF16 || t == PA_F16; }

pa_status current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return PA_ERR_CUDA;
    if (*dev < 0 || *dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

int sm_count(int dev) {
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 0;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

int *status_word(int dev) {
    int *p = g_status_addr[dev].load(std::memory_order_acquire);
    if (p) return p;
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return nullptr;
    g_status_addr[dev].store(static_cast<int *>(addr), std::memory_order_release);
    return static_cast<int *>(addr);
}

int env_int(const char *name, int lo, int hi) {
    const char *e = std::getenv(name);
    const int x = e ? std::atoi(e) : 0;
    return (x >= lo && x <= hi) ? x : 0;
}

// Optional tuning knobs, read once (0 = the built-in default):
//   PA_DECODE_CTAS_PER_SM  CTAs per SM the split plan aims at
//   PA_DECODE_HEADS        KV heads per tensor-core CTA (1..8)
//   PA_DECODE_RING_KB      shared-memory ring per tensor-core CTA (KiB)
//   PA_PREFIX_KERNEL       "mma": shared-prefix pass on mma.sync (default: tcgen05)
//   PA_PREFIX_OVERLAP      "0": shared-prefix pass not overlapped with the rest
//   PA_DECODE_KERNEL       "simt": bf16 decode on the CUDA-core kernel
//   PA_DECODE_BALANCE      "0": never the ragged-balanced decode, "1": whenever it applies
int ctas_per_sm_override() {
    static const int v = env_int("PA_DECODE_CTAS_PER_SM", 1, 64);
    return v;
}
int heads_override() {
    static const int v = env_int("PA_DECODE_HEADS", 1, 8);
    return v;
}
int heads_cap() { return heads_override() ? heads_override() : kMmaHeadsPerCta; }
// PA_PREFIX_OVERLAP=0 runs the shared-prefix pass and the rest-of-context
// decode strictly one after the other instead of letting them overlap.
bool prefix_overlap_enabled() {
    static const bool v = [] {
        const char *e = std::getenv("PA_PREFIX_OVERLAP");
        return !(e && std::strcmp(e, "0") == 0);
    }();
    return v;
}

// PA_PREFIX_KERNEL=mma runs the shared-prefix pass on mma.sync instead of tcgen05.
bool prefix_tc_enabled() {
    static const bool v = [] {
        const char *e = std::getenv("PA_PREFIX_KERNEL");
        return !(e && std::strcmp(e, "mma") == 0);
    }();
    return v;
}
// PA_DECODE_BALANCE: -1 automatic (default), 0 never, 1 whenever it applies.
int balance_mode() {
    static const int v = [] {
        const char *e = std::getenv("PA_DECODE_BALANCE");
        if (!e) return -1;
        return std::strcmp(e, "0") == 0 ? 0 : std::strcmp(e, "1") == 0 ? 1 : -1;
    }();
    return v;
}

//   PA_PREFIX_CTAS         CTAs the shared-prefix pass aims at (default: one per SM)
int prefix_ctas_override() {
    static const int v = env_int("PA_PREFIX_CTAS", 1, 65536);
    return v;
}

//   PA_PREFIX_GROUPS       row groups per CTA of the tcgen05 prefix pass (1 or 2)
//   PA_PREFIX_ORDER        "rest": the rest-of-context decode first, the prefix pass
//                          behind it (default: the prefix pass first)
bool prefix_first_enabled() {
    static const bool v = [] {
        const char *e = std::getenv("PA_PREFIX_ORDER");
        return !(e && std::strcmp(e, "rest") == 0);
    }();
    return v;
}
int prefix_groups_override() {
    static const int v = env_int("PA_PREFIX_GROUPS", 1, 2);
    return v;
}

int ring_override_kb() {
    static const int v = env_int("PA_DECODE_RING_KB", 16, 200);
    return v;
}
int ring_kb() { return ring_override_kb() ? ring_override_kb() : kMmaRingKiB; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// 5-D view of a bf16 cache [num_blocks, block_size, Hkv, D], listed innermost
// first as (dim within a 64-dim half, token, half, head, block): the strides
// of the middle three are permuted so that a box of 64 dims x box_tokens
// tokens x every half x box_heads heads lands in shared memory as
// [head][half][token][128 bytes] (box_halves 0: every half). 128-byte
// swizzle; out-of-range coordinates read as zeros.
pa_status make_cache_map(CUtensorMap *map, const void *cache, int64_t num_blocks, int64_t block_size,
                         int num_kv_heads, int head_dim, int box_tokens, int box_heads, int box_halves,
                         bool f16) {
    auto enc = tensor_map_encoder();
    if (!enc) return PA_ERR_CUDA;
    const cuuint64_t halves = static_cast<cuuint64_t>(head_dim / 64);
    const cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(block_size), halves,
                                static_cast<cuuint64_t>(num_kv_heads), static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t row = static_cast<cuuint64_t>(head_dim) * 2;
    const cuuint64_t strides[4] = {row * num_kv_heads, 128, row, row * num_kv_heads * block_size};
    const cuuint32_t box[5] = {64, static_cast<cuuint32_t>(box_tokens),
                               static_cast<cuuint32_t>(box_halves > 0 ? box_halves : static_cast<int>(halves)),
                               static_cast<cuuint32_t>(box_heads), 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(cache), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Query [B, Hkv * G, D] (16-bit) as 5-D, innermost first: (dim within a 64-dim
// half, half, head within the GQA group, KV head, sequence). A box of 64 dims
// x 1 half x G heads x 1 KV head x seqs sequences is one row group's half of
// Q: rows sequence * G + head, 128 bytes each, with the 128-byte swizzle (the
// K-major operand layout of the tensor cores). Sequences past the batch read
// as zeros.
pa_status make_query_group_map(CUtensorMap *map, const void *query, int num_seqs, int num_kv_heads, int group,
                               int head_dim, int seqs, bool f16) {
    auto enc = tensor_map_encoder();
    if (!enc) return PA_ERR_CUDA;
    const cuuint64_t row = static_cast<cuuint64_t>(head_dim) * 2;
    const cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(head_dim / 64), static_cast<cuuint64_t>(group),
                                static_cast<cuuint64_t>(num_kv_heads), static_cast<cuuint64_t>(num_seqs)};
    const cuuint64_t strides[4] = {128, row, row * group, row * group * num_kv_heads};
    const cuuint32_t box[5] = {64, 1, static_cast<cuuint32_t>(group), 1, static_cast<cuuint32_t>(seqs)};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                     const_cast<void *>(query), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Split-K partial outputs tmp_out [B, Hq, part_stride, D] fp32 as 4-D,
// innermost first: (dim, partition, query head, sequence). A box of out_cols
// dims x 1 partition x G heads x seqs sequences is 128-byte rows (sequence *
// G + head) of one row group, with the 128-byte swizzle; the store clips
// sequences past the batch.
pa_status make_partials_store_map(CUtensorMap *map, void *tmp_out, int num_seqs, int num_heads, int part_stride,
                                  int head_dim, int group, int seqs) {
    auto enc = tensor_map_encoder();
    if (!enc) return PA_ERR_CUDA;
    const cuuint64_t row = static_cast<cuuint64_t>(head_dim) * 4;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(part_stride),
                                static_cast<cuuint64_t>(num_heads), static_cast<cuuint64_t>(num_seqs)};
    const cuuint64_t strides[3] = {row, row * part_stride, row * part_stride * num_heads};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(prefix_tc_out_cols()), 1, static_cast<cuuint32_t>(group),
                               static_cast<cuuint32_t>(seqs)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, tmp_out, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

struct DecodeShape {
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks, num_blocks, max_ctx;
};

pa_status check_shape(const DecodeShape &s) {
    if (s.num_seqs < 0 || s.num_heads <= 0 || s.num_kv_heads <= 0 || s.max_blocks <= 0 ||
        s.num_blocks <= 0 || s.max_ctx < 0 || s.block_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (s.num_heads % s.num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(s.max_ctx) > static_cast<int64_t>(s.max_blocks) * s.block_size)
        return PA_ERR_INVALID_ARG;
    if (s.head_dim != 64 && s.head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (s.block_size > 256) return PA_ERR_UNSUPPORTED;
    const int ntile = (s.num_heads / s.num_kv_heads + kRowsPerTile - 1) / kRowsPerTile;
    if (s.num_seqs > 65535 || static_cast<int64_t>(s.num_kv_heads) * ntile > 65535)
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

struct Plan {
    bool mma;           // tensor-core kernel (else CUDA-core)
    bool cluster;       // split merged through distributed shared memory (no workspace)
    int heads_per_cta;
    int ntile;
    int nsplit;
    int part_tokens;    // tokens per partition
    bool balanced = false;   // ragged-balanced decode: the batch's tiles cut into equal ranges
    int bal_ctas = 0;        //   CTAs per (KV-head group, head tile)
};

// PA_DECODE_KERNEL=simt runs bf16 decode on the CUDA-core kernel (for comparison).
bool simt_forced() {
    static const bool v = [] {
        const char *e = std::getenv("PA_DECODE_KERNEL");
        return e && std::strcmp(e, "simt") == 0;
    }();
    return v;
}

bool use_mma(const DecodeShape &s, bool kv16) {
    return kv16 && decode_mma_supported(s.head_dim, s.block_size) && !simt_forced();
}

// Partition granularity: the tensor-core kernel's tile, the CUDA-core
// kernel's block.
int split_granule(const DecodeShape &s, bool mma) { return mma ? decode_mma_tile_tokens(s.block_size) : s.block_size; }

// Split each (sequence, KV-head group, head tile) context so that about
// sm_count * ctas_per_sm CTAs exist, with at least kMinSplitTokens per piece.
// Partitions are whole granules, sized evenly over max_context_len.
Plan plan_split(const DecodeShape &s, int sms, bool mma, int min_split_tokens = kMinSplitTokens,
                int ctas_per_sm = 0) {
    Plan pl;
    pl.mma = mma;
    pl.heads_per_cta = mma ? decode_mma_heads_per_cta(s.num_kv_heads, heads_cap()) : 1;
    const int group = s.num_heads / s.num_kv_heads;
    pl.ntile = (group + kRowsPerTile - 1) / kRowsPerTile;
    const int64_t units =
        static_cast<int64_t>(s.num_seqs) * (s.num_kv_heads / pl.heads_per_cta) * pl.ntile;
    const int gran = split_granule(s, mma);
    const int64_t ngran = std::max<int64_t>(1, cdiv64(s.max_ctx, gran));
    const int per_sm = ctas_per_sm_override() ? ctas_per_sm_override()
                       : ctas_per_sm > 0      ? ctas_per_sm
                                              : (mma ? kCtasPerSmMma : kCtasPerSmSimt);
    const int64_t cap = static_cast<int64_t>(sms) * per_sm;
    int64_t nsplit = 1;
    if (units > 0 && units < cap) {
        nsplit = cap / units;
        const int64_t min_pg = std::max<int64_t>(1, cdiv64(min_split_tokens, gran));
        nsplit = std::min(nsplit, std::max<int64_t>(1, ngran / min_pg));
        nsplit = std::min<int64_t>(nsplit, kMaxSplits);
    }
    // Tensor-core kernel: merge inside a cluster when the split fits one
    // (or when trimming it to one still leaves ~3/4 of the CTA slots busy).
    pl.cluster = false;
    if (mma && nsplit >= 2) {
        if (nsplit > kMaxClusterSplits && units * kMaxClusterSplits * 4 >= cap * 3)
            nsplit = kMaxClusterSplits;
        pl.cluster = nsplit <= kMaxClusterSplits;
    }
    const int64_t pg = cdiv64(ngran, nsplit);
    pl.part_tokens = static_cast<int>(pg * gran);
    pl.nsplit = static_cast<int>(cdiv64(ngran, pg));
    if (pl.nsplit < 2) pl.cluster = false;
    if (pl.cluster) {
        // the cluster must span exactly the partitions of one context
        pl.nsplit = static_cast<int>(nsplit);
    }
    return pl;
}

// The plan pa_decode uses: with no workspace, a split the tensor-core kernel
// cannot keep inside a cluster is trimmed to one (CUDA-core: not split).
// The ragged-balanced decode applies to a paged bf16 cache with blocks of 16
// or more, a workspace, and a batch whose tile count fits an int. By default
// it is taken when the batch has so many sequences that the CTA slots would
// split each context at most twice: there, ragged lengths leave the CTAs of
// long contexts running alone.
bool take_balanced(const DecodeShape &s, const Plan &pl, int sms, bool have_workspace, bool paged) {
    if (!pl.mma || !have_workspace || !paged || s.num_seqs < 1 || s.num_seqs > kBalancedMaxSeqs) return false;
    if (!decode_balanced_supported(s.head_dim, s.block_size)) return false;
    if (static_cast<int64_t>(s.num_seqs) * cdiv64(s.max_ctx, 16) >= (int64_t(1) << 30)) return false;
    const int mode = balance_mode();
    if (mode >= 0) return mode == 1;
    // enough sequences that the CTA slots would split each context at most twice
    const int64_t units = static_cast<int64_t>(s.num_seqs) * (s.num_kv_heads / pl.heads_per_cta) * pl.ntile;
    const int per_sm = ctas_per_sm_override() ? ctas_per_sm_override() : kCtasPerSmMma;
    return s.num_seqs >= 2 && units * 3 > static_cast<int64_t>(sms) * per_sm;
}

Plan plan_decode(const DecodeShape &s, int sms, bool mma, bool have_workspace, bool paged = true) {
    Plan pl = plan_split(s, sms, mma);
    pl.balanced = take_balanced(s, pl, sms, have_workspace, paged);
    pl.bal_ctas = 0;
    if (pl.balanced) {
        // whole head groups per CTA: fewer, larger boxes and one query load per head group
        pl.heads_per_cta = decode_mma_heads_per_cta(
            s.num_kv_heads, heads_override() ? heads_override() : kBalancedHeadsPerCta);
        const int lanes = (s.num_kv_heads / pl.heads_per_cta) * pl.ntile;
        const int per_sm = ctas_per_sm_override() ? ctas_per_sm_override() : kBalancedCtasPerSm;
        pl.bal_ctas = std::max(1, sms * per_sm / lanes);
        pl.cluster = false;
        pl.nsplit = pl.bal_ctas;
        pl.part_tokens = 0;
        return pl;
    }
    if (!have_workspace && !pl.cluster) {
        const int gran = split_granule(s, mma);
        const int64_t ngran = std::max<int64_t>(1, cdiv64(s.max_ctx, gran));
        if (pl.mma && pl.nsplit > 1) {
            const int64_t pg = cdiv64(ngran, std::min(pl.nsplit, kMaxClusterSplits));
            pl.part_tokens = static_cast<int>(pg * gran);
            pl.nsplit = static_cast<int>(cdiv64(ngran, pg));
            pl.cluster = pl.nsplit > 1;
        } else {
            pl.part_tokens = static_cast<int>(ngran * gran);
            pl.nsplit = 1;
        }
    }
    return pl;
}

struct WorkspaceLayout {
    size_t o_off, ml_off, count_off, prefix_off, total;
};

// Wide splits are written in split-K form (normalised partial outputs,
// maxima, sums) and merged by the log-sum-exp merge kernel.
WorkspaceLayout workspace_layout(const DecodeShape &s, const Plan &pl) {
    WorkspaceLayout w{};
    if (pl.balanced) {
        // pieces: rows (c + b) * Hq + h for c < ctas, b < num_seqs; then the tile prefix sums
        const size_t rows = static_cast<size_t>(pl.bal_ctas + s.num_seqs) * s.num_heads;
        w.o_off = 0;
        w.ml_off = align256(rows * s.head_dim * sizeof(float));
        w.count_off = w.ml_off + align256(rows * sizeof(float));
        w.prefix_off = w.count_off + align256(rows * sizeof(float));
        w.total = w.prefix_off + align256(static_cast<size_t>(s.num_seqs + 1) * sizeof(int));
        return w;
    }
    if (pl.nsplit <= 1 || pl.cluster) return w;
    const size_t rows = static_cast<size_t>(s.num_seqs) * s.num_heads * pl.nsplit;
    w.o_off = 0;
    w.ml_off = align256(rows * s.head_dim * sizeof(float));            // maxima
    w.count_off = w.ml_off + align256(rows * sizeof(float));            // sums
    w.total = w.count_off + align256(rows * sizeof(float));
    return w;
}

pa_status launch_decode(const DecodeShape &s, DecodeParams &p, pa_dtype kv_dtype, bool mma, int dev,
                        cudaStream_t stream);

// Decode of a wide split: partitions in split-K form into the workspace, then
// the merge kernel on the same stream.
pa_status launch_split_and_merge(const DecodeShape &s, DecodeParams &p, pa_dtype kv_dtype, bool mma,
                                 int dev, void *workspace, const WorkspaceLayout &wl, void *out, int out_type,
                                 cudaStream_t stream) {
    char *ws = static_cast<char *>(workspace);
    p.tmp_out = reinterpret_cast<float *>(ws + wl.o_off);
    p.max_logits = reinterpret_cast<float *>(ws + wl.ml_off);
    p.exp_sums = reinterpret_cast<float *>(ws + wl.count_off);
    p.mode = kModeSplitK;
    p.cluster_merge = 0;
    pa_status st = launch_decode(s, p, kv_dtype, mma, dev, stream);
    if (st != PA_OK) return st;
    const cudaError_t e = launch_lse_merge(out, out_type, p.tmp_out, p.max_logits, p.exp_sums,
                                           p.context_lens, s.num_seqs, s.num_heads, s.head_dim,
                                           p.nsplit, p.part_tokens, sm_count(dev), stream);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status check_dtypes(pa_dtype q_dtype, pa_dtype kv_dtype) {
    if (!valid_dtype(q_dtype) || !valid_dtype(kv_dtype)) return PA_ERR_INVALID_ARG;
    if (q_dtype != kv_dtype) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// Shared by pa_decode and pa_decode_splitk; `mma` picks the tensor-core
// kernel (bf16, a supported block size, partitions of whole 16-token tiles).
pa_status launch_decode(const DecodeShape &s, DecodeParams &p, pa_dtype kv_dtype, bool mma, int dev,
                        cudaStream_t stream) {
    p.status = status_word(dev);
    if (!p.status) return PA_ERR_CUDA;
    const dim3 grid(static_cast<unsigned>(p.nsplit),
                    static_cast<unsigned>((s.num_kv_heads / p.heads_per_cta) * p.ntile),
                    static_cast<unsigned>(s.num_seqs));
    cudaError_t e;
    if (mma) {
        const int box = decode_mma_box_tokens(s.block_size);
        const int box_heads = p.heads_per_cta;     // one box covers every head of the CTA
        const int stage = decode_mma_stage_bytes(s.head_dim, s.block_size, p.heads_per_cta);
        const int budget_kb = ring_override_kb() ? ring_override_kb() : p.cluster_merge ? kMmaRingKiB : kSplitRingKiB;
        p.ring_bytes = decode_mma_ring_bytes(s.head_dim, s.block_size, p.heads_per_cta, budget_kb * 1024);
        if (p.cluster_merge) {
            const int need = decode_mma_cluster_bytes(s.head_dim, p.heads_per_cta);
            if (p.ring_bytes < need) p.ring_bytes = static_cast<int>(cdiv64(need, stage) * stage);
        }
        // a contiguous cache [B, stride, Hkv, D] is mapped as one block of B * stride tokens
        const bool contig = p.contig_stride > 0;
        const int64_t map_blocks = contig ? 1 : s.num_blocks;
        const int64_t map_tokens = contig ? static_cast<int64_t>(s.num_seqs) * p.contig_stride : s.block_size;
        CUtensorMap tk, tv;
        pa_status st = make_cache_map(&tk, p.k_cache, map_blocks, map_tokens, s.num_kv_heads, s.head_dim, box, box_heads,
                                      0, p.kv_f16 != 0);
        if (st != PA_OK) return st;
        st = make_cache_map(&tv, p.v_cache, map_blocks, map_tokens, s.num_kv_heads, s.head_dim, box, box_heads, 0,
                            p.kv_f16 != 0);
        if (st != PA_OK) return st;
        e = launch_decode_mma(p, tk, tv, grid, stream);
    } else {
        e = launch_decode_simt(p, static_cast<int>(kv_dtype), grid, stream);
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Ragged-balanced decode: equal tile ranges per CTA, then the merge of the
// pieces of sequences split between CTAs (both through the workspace).
pa_status launch_balanced(const DecodeShape &s, DecodeParams &p, const Plan &pl, int dev, void *workspace,
                          const WorkspaceLayout &wl, cudaStream_t stream) {
    p.status = status_word(dev);
    if (!p.status) return PA_ERR_CUDA;
    char *ws = static_cast<char *>(workspace);
    p.tmp_out = reinterpret_cast<float *>(ws + wl.o_off);
    p.max_logits = reinterpret_cast<float *>(ws + wl.ml_off);
    p.exp_sums = reinterpret_cast<float *>(ws + wl.count_off);
    p.mode = kModeSplitK;
    p.cluster_merge = 0;
    BalancedParams bp;
    bp.ctas = pl.bal_ctas;
    bp.len_cap = s.max_ctx;
    bp.prefix = reinterpret_cast<int *>(ws + wl.prefix_off);
    const int stage = decode_mma_stage_bytes(s.head_dim, s.block_size, p.heads_per_cta);
    const int ring_budget = (ring_override_kb() ? ring_override_kb() : kBalancedRingKiB) * 1024;
    p.ring_bytes = decode_mma_ring_bytes(s.head_dim, s.block_size, p.heads_per_cta, ring_budget);
    if (p.ring_bytes < stage) return PA_ERR_UNSUPPORTED;
    const int box = decode_mma_box_tokens(s.block_size);
    CUtensorMap tk, tv;
    pa_status st = make_cache_map(&tk, p.k_cache, s.num_blocks, s.block_size, s.num_kv_heads, s.head_dim, box,
                                  p.heads_per_cta, 0, p.kv_f16 != 0);
    if (st != PA_OK) return st;
    if ((st = make_cache_map(&tv, p.v_cache, s.num_blocks, s.block_size, s.num_kv_heads, s.head_dim, box,
                             p.heads_per_cta, 0, p.kv_f16 != 0)) != PA_OK)
        return st;
    const dim3 grid(static_cast<unsigned>(pl.bal_ctas),
                    static_cast<unsigned>((s.num_kv_heads / p.heads_per_cta) * p.ntile), 1u);
    if (launch_decode_balanced(p, bp, tk, tv, grid, stream) != cudaSuccess) return PA_ERR_CUDA;
    return launch_balanced_merge(p, bp, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

void fill_common(DecodeParams &p, const DecodeShape &s, const void *query, pa_dtype q_dtype,
                 const void *k_cache, const void *v_cache, const int32_t *block_tables,
                 const int32_t *context_lens, float scale) {
    std::memset(&p, 0, sizeof p);
    p.query = query;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.num_seqs = s.num_seqs;
    p.num_heads = s.num_heads;
    p.num_kv_heads = s.num_kv_heads;
    p.head_dim = s.head_dim;
    p.block_size = s.block_size;
    p.max_blocks = s.max_blocks;
    p.num_blocks = s.num_blocks;
    p.group = s.num_heads / s.num_kv_heads;
    p.q_bf16 = q_dtype == PA_BF16;
    p.kv_f16 = q_dtype == PA_F16;   // the caches have the query's type
    p.scale_log2 = scale * kLog2e;
}

// Plan, check the pointers and launch one decode (paged when contig_stride
// is 0, else over a contiguous cache [num_seqs, contig_stride, Hkv, D]).
// The shape and dtypes have been checked by the caller.
pa_status decode_planned(const DecodeShape &s, void *out, pa_dtype out_dtype, const void *query,
                         pa_dtype q_dtype, const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                         const int32_t *block_tables, const int32_t *context_lens, int contig_stride,
                         float scale, void *workspace, size_t workspace_bytes, void *stream,
                         const void *append_key = nullptr, const void *append_value = nullptr) {
    if (!out || !query || !k_cache || !v_cache || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    int dev;
    pa_status st = current_device(&dev);
    if (st != PA_OK) return st;
    const int sms = sm_count(dev);
    if (sms <= 0) return PA_ERR_CUDA;

    const Plan pl = plan_decode(s, sms, use_mma(s, is16(kv_dtype)),
                                workspace != nullptr || workspace_bytes != 0, contig_stride == 0);
    DecodeParams p;
    fill_common(p, s, query, q_dtype, k_cache, v_cache, block_tables, context_lens, scale);
    p.contig_stride = contig_stride;
    p.out = out;
    p.out_bf16 = out_dtype == PA_BF16;
    p.out_f16 = out_dtype == PA_F16;
    p.ntile = pl.ntile;
    p.heads_per_cta = pl.heads_per_cta;
    p.nsplit = pl.nsplit;
    p.part_tokens = pl.part_tokens;
    p.cluster_merge = pl.cluster ? 1 : 0;
    if (pl.balanced || (!pl.cluster && pl.nsplit > 1)) {   // refuse before anything is launched
        const WorkspaceLayout wl = workspace_layout(s, pl);
        if (!workspace || workspace_bytes < wl.total || !aligned16(workspace)) return PA_ERR_WORKSPACE;
    }
    if (append_key) {
        // the step's new tokens: written by the tensor-core kernels themselves (the CTA that
        // reads each one writes it first), else by a scatter launched ahead of the decode
        if (pl.mma && contig_stride == 0) {
            p.append_key = append_key;
            p.append_value = append_value;
        } else if (launch_append_last(append_key, append_value, const_cast<void *>(k_cache),
                                      const_cast<void *>(v_cache), block_tables, context_lens, s.num_seqs,
                                      s.max_blocks, s.block_size, s.num_blocks, s.max_ctx,
                                      s.num_kv_heads * s.head_dim * element_bytes(kv_dtype),
                                      as_stream(stream)) != cudaSuccess) {
            return PA_ERR_CUDA;
        }
    }
    if (pl.balanced) {
        const WorkspaceLayout wl = workspace_layout(s, pl);
        if (!workspace || workspace_bytes < wl.total || !aligned16(workspace)) return PA_ERR_WORKSPACE;
        return launch_balanced(s, p, pl, dev, workspace, wl, as_stream(stream));
    }
    if (pl.cluster) {
        p.mode = kModeFinal;   // the cluster merge writes the output
    } else if (pl.nsplit > 1) {
        const WorkspaceLayout wl = workspace_layout(s, pl);
        if (!workspace || workspace_bytes < wl.total || !aligned16(workspace)) return PA_ERR_WORKSPACE;
        return launch_split_and_merge(s, p, kv_dtype, pl.mma, dev, workspace, wl, out, static_cast<int>(out_dtype),
                                      as_stream(stream));
    } else {
        p.mode = kModeFinal;
    }
    return launch_decode(s, p, kv_dtype, pl.mma, dev, as_stream(stream));
}

// ---------------------------------------------------------------------------
// Shared-prefix decode: the shared leading blocks attended once for every row
// (prefix pass), the rest of each context by the decode kernel in split-K
// form, both merged by the log-sum-exp merge.
// ---------------------------------------------------------------------------
struct PrefixPlan {
    bool tc;             // prefix pass on tcgen05 (else mma.sync)
    int prefix_tokens;   // shared tokens attended by the prefix pass (whole tiles)
    int chunk_tokens;
    int chunks;          // prefix partitions (grid.x of the prefix pass)
    int row_groups;      // grid.z of the prefix pass
    int seqs_per_group;  // tcgen05: whole sequences per row group of at most 128 rows
    int tc_groups;       // tcgen05: row groups of the batch
    int groups_per_cta;  // tcgen05: row groups one CTA serves (they share its K/V tiles)
    Plan suffix;         // the decode kernel's split of the rest (never a cluster)
    int part_stride;     // partitions per (sequence, head): chunks + suffix splits
};

PrefixPlan plan_prefix(const DecodeShape &s, int shared_blocks, int sms, bool tc) {
    PrefixPlan pp{};
    // the tcgen05 pass takes row groups of whole sequences: at most 128 query heads per KV head
    tc = tc && s.num_heads / s.num_kv_heads <= prefix_tc_max_rows();
    pp.tc = tc;
    // the prefix pass takes whole tiles; shared tokens past the last one go with the rest
    const int tile = tc ? prefix_tc_tile_tokens() : 16;
    int64_t P = std::min<int64_t>(static_cast<int64_t>(shared_blocks) * s.block_size, s.max_ctx);
    P = P / tile * tile;
    pp.prefix_tokens = static_cast<int>(P);
    const int group = s.num_heads / s.num_kv_heads;
    if (tc) {
        pp.seqs_per_group = prefix_tc_max_rows() / group;
        pp.tc_groups = static_cast<int>(cdiv64(s.num_seqs, pp.seqs_per_group));
        // head_dim 128: one row group per CTA. For the same number of CTAs that
        // halves the chunks, so the partials written and merged, and each CTA
        // runs twice the tiles through one setup. At head_dim 64, where a CTA
        // with two groups sharing each K/V tile is small, two are faster.
        pp.groups_per_cta = pp.tc_groups >= 2 && s.head_dim == 64 ? 2 : 1;
        if (prefix_groups_override()) pp.groups_per_cta = std::min(pp.tc_groups, prefix_groups_override());
        pp.row_groups = static_cast<int>(cdiv64(pp.tc_groups, pp.groups_per_cta));
    } else {
        pp.row_groups = static_cast<int>(cdiv64(static_cast<int64_t>(s.num_seqs) * group, prefix_rows_per_cta()));
    }
    if (P > 0) {
        const int64_t per_chunk = static_cast<int64_t>(s.num_kv_heads) * pp.row_groups;
        int64_t cap = prefix_ctas_override() ? prefix_ctas_override()
                                             : static_cast<int64_t>(sms) * (tc ? 1 : kCtasPerSmMma);
        int64_t chunks = std::max<int64_t>(1, cap / per_chunk);
        if (tc && !prefix_ctas_override() && prefix_first_enabled()) {
            // The prefix pass goes first and holds its SMs (one CTA each) while
            // the rest-of-context decode runs on the others: give it a share of
            // the SMs in proportion to its work, the rest's bytes at the largest
            // lengths against the pass's (64-token tile x 128-row group x KV
            // head) units, each worth kPrefixUnitMB of rest; all of them when
            // the rest is small. A head_dim 64 unit counts 3/4 of one at 128:
            // half the products and bytes, the same softmax.
            const double units = static_cast<double>(P / tile) * s.num_kv_heads * pp.tc_groups *
                                 (0.5 + 0.5 * s.head_dim / 128.0);
            const double rest_mb = static_cast<double>(s.num_seqs) * std::max<int64_t>(0, s.max_ctx - P) *
                                   s.num_kv_heads * s.head_dim * 4 / 1e6;
            const double frac = units * kPrefixUnitMB / (units * kPrefixUnitMB + rest_mb);
            if (frac < kPrefixAllSmsFrac) {
                const int64_t share = std::max<int64_t>(1, std::llround(sms * frac));
                chunks = std::max<int64_t>(1, std::min<int64_t>((share + per_chunk / 2) / per_chunk,
                                                                std::max<int64_t>(1, sms / per_chunk)));
            }
        }
        chunks = std::min<int64_t>(chunks, std::max<int64_t>(1, P / std::max(kMinPrefixChunk, tile)));
        chunks = std::min<int64_t>(chunks, kMaxSplits);
        const int64_t tiles = P / tile;
        int64_t ct = cdiv64(tiles, chunks);
        if (tc)   // a chunk's block ids must fit the kernel's staging array
            ct = std::min<int64_t>(ct, std::max<int64_t>(1, (static_cast<int64_t>(kTcChunkBlocks - 1) * s.block_size) / tile));
        pp.chunk_tokens = static_cast<int>(ct * tile);
        pp.chunks = static_cast<int>(cdiv64(tiles, ct));
    }
    DecodeShape rest = s;
    rest.max_ctx = static_cast<int>(std::max<int64_t>(0, s.max_ctx - P));
    // the merge kernel runs anyway: the rest may be cut finer than a plain decode's
    pp.suffix = plan_split(rest, sms, true, kMinRestSplitTokens, kRestCtasPerSm);
    pp.suffix.cluster = false;
    if (pp.suffix.nsplit > 1) {   // partitions of the rest, in whole tiles, without the cluster's rounding
        const int64_t ngran = std::max<int64_t>(1, cdiv64(rest.max_ctx, 16));
        pp.suffix.nsplit = static_cast<int>(cdiv64(ngran, cdiv64(pp.suffix.part_tokens, 16)));
    }
    pp.part_stride = pp.chunks + pp.suffix.nsplit;   // the rest's partitions follow the prefix chunks
    return pp;
}

WorkspaceLayout prefix_workspace(const DecodeShape &s, const PrefixPlan &pp) {
    WorkspaceLayout w{};
    const size_t rows = static_cast<size_t>(s.num_seqs) * s.num_heads * pp.part_stride;
    w.o_off = 0;
    w.ml_off = align256(rows * s.head_dim * sizeof(float));
    w.count_off = w.ml_off + align256(rows * sizeof(float));
    w.total = w.count_off + align256(rows * sizeof(float));
    return w;
}

pa_status check_prefix_call(const DecodeShape &s, pa_dtype q_dtype, pa_dtype kv_dtype, int shared_blocks) {
    pa_status st = check_shape(s);
    if (st != PA_OK) return st;
    if ((st = check_dtypes(q_dtype, kv_dtype)) != PA_OK) return st;
    if (shared_blocks < 0 || shared_blocks > s.max_blocks) return PA_ERR_INVALID_ARG;
    // the prefix passes land one block (up to a tile) per TMA box: 8 rows or more
    if (!is16(kv_dtype) || !decode_mma_supported(s.head_dim, s.block_size) || s.block_size < 8)
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

}  // namespace

int *device_status_word() {
    int dev;
    if (current_device(&dev) != PA_OK) return nullptr;
    return status_word(dev);
}

int decode_into_scratch(const DecodeCall &c, void *scratch, size_t scratch_bytes, void *stream) {
    const DecodeShape s{c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim, c.block_size,
                        c.max_blocks_per_seq, c.num_blocks, c.max_context_len};
    const pa_dtype out_dtype = static_cast<pa_dtype>(c.out_dtype);
    const pa_dtype q_dtype = static_cast<pa_dtype>(c.q_dtype);
    const pa_dtype kv_dtype = static_cast<pa_dtype>(c.kv_dtype);
    pa_status st = check_shape(s);
    if (st != PA_OK) return st;
    if (!valid_dtype(out_dtype) || !std::isfinite(c.scale)) return PA_ERR_INVALID_ARG;
    if ((st = check_dtypes(q_dtype, kv_dtype)) != PA_OK) return st;
    if (c.num_seqs == 0) return PA_OK;
    int dev;
    if ((st = current_device(&dev)) != PA_OK) return st;
    const int sms = sm_count(dev);
    if (sms <= 0) return PA_ERR_CUDA;
    // pa_decode's plan for a caller with a workspace, without the ragged-balanced
    // path: a split that fits a thread-block cluster is merged there, in shared
    // memory (no scratch); a wider one goes through the scratch.
    const Plan pl = plan_split(s, sms, use_mma(s, is16(kv_dtype)));
    const bool wide = !pl.cluster && pl.nsplit > 1;
    const WorkspaceLayout wl = workspace_layout(s, pl);
    if (wide && (wl.total > scratch_bytes || !scratch || !aligned16(scratch))) return PA_ERR_WORKSPACE;
    if (!c.out || !c.query || !c.k_cache || !c.v_cache || !c.block_tables || !c.context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(c.out) || !aligned16(c.query) || !aligned16(c.k_cache) || !aligned16(c.v_cache))
        return PA_ERR_INVALID_ARG;
    DecodeParams p;
    fill_common(p, s, c.query, q_dtype, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale);
    p.out = c.out;
    p.out_bf16 = out_dtype == PA_BF16;
    p.out_f16 = out_dtype == PA_F16;
    p.ntile = pl.ntile;
    p.heads_per_cta = pl.heads_per_cta;
    p.nsplit = pl.nsplit;
    p.part_tokens = pl.part_tokens;
    p.cluster_merge = pl.cluster ? 1 : 0;
    if (wide)
        return launch_split_and_merge(s, p, kv_dtype, pl.mma, dev, scratch, wl, c.out, static_cast<int>(out_dtype),
                                      as_stream(stream));
    p.mode = kModeFinal;   // unsplit, or merged by the cluster
    return launch_decode(s, p, kv_dtype, pl.mma, dev, as_stream(stream));
}

}  // namespace pa

using namespace pa;

extern "C" {

PA_API const char *pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_OUT_OF_BLOCKS: return "out of KV blocks";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_TIMEOUT: return "kernel wait timed out";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_NOT_FOUND: return "unknown sequence";
    }
    return "unknown status";
}

PA_API int pa_abi_version(void) { return PA_ABI_VERSION; }

PA_API pa_status pa_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                      void *v_cache, const int64_t *slot_mapping, int num_tokens,
                                      int num_blocks, int block_size, int num_kv_heads,
                                      int head_dim, pa_dtype kv_dtype, void *stream) {
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        !valid_dtype(kv_dtype))
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * element_bytes(kv_dtype);
    if (row_bytes % 16 != 0 || row_bytes / 16 > (1 << 20)) return PA_ERR_UNSUPPORTED;
    const int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
    cudaError_t e = launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                             num_slots, static_cast<int>(row_bytes), as_stream(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_decode_append(void *out, pa_dtype out_dtype, const void *query, pa_dtype q_dtype,
                                  const void *new_key, const void *new_value, void *k_cache, void *v_cache,
                                  pa_dtype kv_dtype, const int32_t *block_tables, const int32_t *context_lens,
                                  int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, int max_context_len, float scale,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    const DecodeShape s{num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                        max_blocks_per_seq, num_blocks, max_context_len};
    pa_status st = check_shape(s);
    if (st != PA_OK) return st;
    if (!valid_dtype(out_dtype) || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if ((st = check_dtypes(q_dtype, kv_dtype)) != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if (!block_tables || !new_key || !new_value || !aligned16(new_key) || !aligned16(new_value))
        return PA_ERR_INVALID_ARG;
    return decode_planned(s, out, out_dtype, query, q_dtype, k_cache, v_cache, kv_dtype, block_tables,
                          context_lens, 0, scale, workspace, workspace_bytes, stream, new_key, new_value);
}

PA_API pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *block_mapping,
                                int num_pairs, int num_blocks, int block_size, int num_kv_heads,
                                int head_dim, pa_dtype kv_dtype, void *stream) {
    if (num_pairs < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        !valid_dtype(kv_dtype))
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !block_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    const int64_t block_bytes =
        static_cast<int64_t>(block_size) * num_kv_heads * head_dim * element_bytes(kv_dtype);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    cudaError_t e = launch_copy_blocks(k_cache, v_cache, block_mapping, num_pairs, num_blocks,
                                       block_bytes, as_stream(stream));
    if (e == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// The address a kernel uses for p: device memory as is; page-locked host
// memory through its device mapping. Pageable host memory gives nullptr.
static const void *device_view(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    return nullptr;
}

PA_API pa_status pa_swap_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                                const int64_t *block_mapping, int num_pairs, int src_num_blocks,
                                int dst_num_blocks, int block_size, int num_kv_heads, int head_dim,
                                pa_dtype kv_dtype, void *stream) {
    if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || !valid_dtype(kv_dtype))
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!dst_k || !dst_v || !src_k || !src_v || !block_mapping) return PA_ERR_INVALID_ARG;
    const int64_t block_bytes =
        static_cast<int64_t>(block_size) * num_kv_heads * head_dim * element_bytes(kv_dtype);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    void *dk = const_cast<void *>(device_view(dst_k)), *dv = const_cast<void *>(device_view(dst_v));
    const void *sk = device_view(src_k), *sv = device_view(src_v), *bm = device_view(block_mapping);
    if (!dk || !dv || !sk || !sv || !bm) return PA_ERR_INVALID_ARG;
    if (!aligned16(dk) || !aligned16(dv) || !aligned16(sk) || !aligned16(sv)) return PA_ERR_INVALID_ARG;
    cudaError_t e = launch_transfer_blocks(dk, dv, sk, sv, static_cast<const int64_t *>(bm), num_pairs,
                                           src_num_blocks, dst_num_blocks, block_bytes, as_stream(stream));
    if (e == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                       int block_size, int max_context_len) {
    const DecodeShape s{num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                        std::max(1, block_size > 0 ? (max_context_len + block_size - 1) / block_size : 1),
                        1, max_context_len};
    if (check_shape(s) != PA_OK) return 0;
    int dev;
    if (current_device(&dev) != PA_OK) return 0;
    const int sms = sm_count(dev);
    if (sms <= 0) return 0;
    return std::max({workspace_layout(s, plan_split(s, sms, true)).total,
                     workspace_layout(s, plan_split(s, sms, false)).total,
                     workspace_layout(s, plan_decode(s, sms, true, true)).total});
}

PA_API pa_status pa_decode_plan(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_context_len, pa_dtype kv_dtype,
                                int with_workspace, pa_decode_plan_t *plan) {
    if (!plan || !valid_dtype(kv_dtype)) return PA_ERR_INVALID_ARG;
    const DecodeShape s{num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                        std::max(1, block_size > 0 ? (max_context_len + block_size - 1) / block_size : 1),
                        1, max_context_len};
    pa_status st = check_shape(s);
    if (st != PA_OK) return st;
    int dev;
    if ((st = current_device(&dev)) != PA_OK) return st;
    const int sms = sm_count(dev);
    if (sms <= 0) return PA_ERR_CUDA;
    const Plan pl = plan_decode(s, sms, use_mma(s, is16(kv_dtype)), with_workspace != 0);
    const bool wide = !pl.cluster && pl.nsplit > 1;
    plan->tensor_cores = pl.mma ? 1 : 0;
    plan->heads_per_cta = pl.heads_per_cta;
    plan->num_splits = pl.nsplit;
    plan->partition_tokens = pl.part_tokens;
    plan->cluster_merge = pl.cluster ? 1 : 0;
    plan->kernel_launches = num_seqs == 0 ? 0 : (wide ? 2 : 1);
    plan->workspace_bytes = wide ? workspace_layout(s, pl).total : 0;
    plan->balanced = pl.balanced ? 1 : 0;
    return PA_OK;
}

PA_API pa_status pa_decode(void *out, pa_dtype out_dtype, const void *query, pa_dtype q_dtype,
                           const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                           const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                           int num_heads, int num_kv_heads, int head_dim, int block_size,
                           int max_blocks_per_seq, int num_blocks, int max_context_len, float scale,
                           void *workspace, size_t workspace_bytes, void *stream) {
    const DecodeShape s{num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                        max_blocks_per_seq, num_blocks, max_context_len};
    pa_status st = check_shape(s);
    if (st != PA_OK) return st;
    if (!valid_dtype(out_dtype) || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if ((st = check_dtypes(q_dtype, kv_dtype)) != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if (!block_tables) return PA_ERR_INVALID_ARG;
    return decode_planned(s, out, out_dtype, query, q_dtype, k_cache, v_cache, kv_dtype, block_tables,
                          context_lens, 0, scale, workspace, workspace_bytes, stream);
}

PA_API size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                                     int head_dim, int block_size, int max_context_len,
                                                     int shared_blocks) {
    const DecodeShape s{num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                        std::max(1, block_size > 0 ? (max_context_len + block_size - 1) / block_size : 1),
                        1, max_context_len};
    if (check_prefix_call(s, PA_BF16, PA_BF16, std::min(shared_blocks, s.max_blocks)) != PA_OK) return 0;
    int dev;
    if (current_device(&dev) != PA_OK) return 0;
    const int sms = sm_count(dev);
    if (sms <= 0) return 0;
    const PrefixPlan pp = plan_prefix(s, shared_blocks, sms, prefix_tc_enabled());
    const size_t plain = std::max(workspace_layout(s, plan_split(s, sms, true)).total,
                                  workspace_layout(s, plan_decode(s, sms, true, true)).total);
    return std::max(prefix_workspace(s, pp).total, plain);
}

PA_API pa_status pa_decode_shared_prefix(void *out, pa_dtype out_dtype, const void *query, pa_dtype q_dtype,
                                         const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                                         const int32_t *block_tables, const int32_t *context_lens,
                                         int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                         int block_size, int max_blocks_per_seq, int num_blocks,
                                         int max_context_len, int shared_blocks, float scale, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    const DecodeShape s{num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                        max_blocks_per_seq, num_blocks, max_context_len};
    pa_status st = check_prefix_call(s, q_dtype, kv_dtype, shared_blocks);
    if (st != PA_OK) return st;
    if (!valid_dtype(out_dtype) || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    int dev;
    if ((st = current_device(&dev)) != PA_OK) return st;
    const int sms = sm_count(dev);
    if (sms <= 0) return PA_ERR_CUDA;
    const PrefixPlan pp = plan_prefix(s, shared_blocks, sms, prefix_tc_enabled());
    if (pp.chunks == 0)   // nothing shared in whole tiles: the plain decode
        return decode_planned(s, out, out_dtype, query, q_dtype, k_cache, v_cache, kv_dtype, block_tables,
                              context_lens, 0, scale, workspace, workspace_bytes, stream);
    const WorkspaceLayout wl = prefix_workspace(s, pp);
    if (!workspace || workspace_bytes < wl.total || !aligned16(workspace)) return PA_ERR_WORKSPACE;
    int *status = status_word(dev);
    if (!status) return PA_ERR_CUDA;
    char *ws = static_cast<char *>(workspace);
    float *tmp_out = reinterpret_cast<float *>(ws + wl.o_off);
    float *max_logits = reinterpret_cast<float *>(ws + wl.ml_off);
    float *exp_sums = reinterpret_cast<float *>(ws + wl.count_off);
    cudaStream_t strm = as_stream(stream);
    // The prefix pass and the rest-of-context decode write disjoint partitions
    // and read nothing of each other's: they overlap as a pair (PairRole) on
    // the caller's stream, then the merge, the second's dependent, sees both.
    // The tcgen05 pass goes first, on the share of SMs its plan gave it, and
    // the decode runs on the others; the mma.sync pass goes second, into SMs
    // the decode frees. Without overlap the two run one after the other.
    const bool overlap = prefix_overlap_enabled();
    const bool prefix_first = prefix_first_enabled() && pp.tc;
    auto launch_prefix = [&]() -> pa_status {   // 1. the shared prefix, once for every row
        PrefixParams pq;
        std::memset(&pq, 0, sizeof pq);
        pq.query = query;
        pq.prefix_table = block_tables;   // row 0 holds the shared ids like every row
        pq.context_lens = context_lens;
        pq.tmp_out = tmp_out;
        pq.max_logits = max_logits;
        pq.exp_sums = exp_sums;
        pq.status = status;
        pq.num_seqs = num_seqs;
        pq.num_heads = num_heads;
        pq.num_kv_heads = num_kv_heads;
        pq.head_dim = head_dim;
        pq.group = num_heads / num_kv_heads;
        pq.block_size = block_size;
        pq.prefix_tokens = pp.prefix_tokens;
        pq.chunk_tokens = pp.chunk_tokens;
        pq.part_stride = pp.part_stride;
        pq.scale_log2 = scale * kLog2e;
        pq.kv_f16 = kv_dtype == PA_F16;
        pq.pair_role = !overlap ? kPairNone : prefix_first ? kPairFirst : kPairSecond;
        const dim3 grid(static_cast<unsigned>(pp.chunks), static_cast<unsigned>(num_kv_heads),
                        static_cast<unsigned>(pp.row_groups));
        CUtensorMap tk, tv;
        pa_status err;
        if (pp.tc) {
            // boxes of one block (up to a 64-token tile), one 64-dim half, one head
            const int box = std::min(block_size, prefix_tc_tile_tokens());
            pq.ring_bytes = prefix_tc_ring_bytes(head_dim, pp.groups_per_cta,
                                                 (ring_override_kb() ? ring_override_kb() : kPrefixTcRingKiB) * 1024);
            pq.seqs_per_group = pp.seqs_per_group;
            pq.row_groups = pp.tc_groups;
            CUtensorMap tq, to;
            if ((err = make_cache_map(&tk, k_cache, num_blocks, block_size, num_kv_heads, head_dim, box, 1, 1,
                                      pq.kv_f16 != 0)) != PA_OK ||
                (err = make_cache_map(&tv, v_cache, num_blocks, block_size, num_kv_heads, head_dim, box, 1, 1,
                                      pq.kv_f16 != 0)) != PA_OK ||
                (err = make_query_group_map(&tq, query, num_seqs, num_kv_heads, pq.group, head_dim,
                                            pp.seqs_per_group, pq.kv_f16 != 0)) != PA_OK ||
                (err = make_partials_store_map(&to, tmp_out, num_seqs, num_heads, pp.part_stride, head_dim,
                                               pq.group, pp.seqs_per_group)) != PA_OK)
                return err;
            return launch_prefix_tc(pq, pp.groups_per_cta, tk, tv, tq, to, grid, strm) == cudaSuccess
                       ? PA_OK : PA_ERR_CUDA;
        }
        const int box = decode_mma_box_tokens(block_size);
        const int stage = prefix_stage_bytes(head_dim);
        pq.ring_bytes = std::max(stage, std::min(kPrefixMaxRingBytes, ring_kb() * 1024) / stage * stage);
        if ((err = make_cache_map(&tk, k_cache, num_blocks, block_size, num_kv_heads, head_dim, box, 1, 0,
                                  pq.kv_f16 != 0)) != PA_OK ||
            (err = make_cache_map(&tv, v_cache, num_blocks, block_size, num_kv_heads, head_dim, box, 1, 0,
                                  pq.kv_f16 != 0)) != PA_OK)
            return err;
        return launch_prefix_mma(pq, tk, tv, grid, strm) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    };
    auto launch_rest = [&]() -> pa_status {   // 2. the rest of every context (the tokens past the shared ones)
        DecodeParams p;
        fill_common(p, s, query, q_dtype, k_cache, v_cache, block_tables, context_lens, scale);
        p.tmp_out = tmp_out;
        p.max_logits = max_logits;
        p.exp_sums = exp_sums;
        p.ntile = pp.suffix.ntile;
        p.heads_per_cta = pp.suffix.heads_per_cta;
        p.nsplit = pp.suffix.nsplit;
        p.part_tokens = pp.suffix.part_tokens;
        p.skip_tokens = pp.prefix_tokens;
        p.part_stride = pp.part_stride;
        // split-K partitions after the prefix chunks, then the merge
        p.part_offset = pp.chunks;
        p.mode = kModeSplitK;
        p.pair_role = !overlap ? kPairNone : prefix_first ? kPairSecond : kPairFirst;
        return launch_decode(s, p, kv_dtype, true, dev, strm);
    };
    if (overlap && !prefix_first) {
        if ((st = launch_rest()) != PA_OK || (st = launch_prefix()) != PA_OK) return st;
    } else {
        if ((st = launch_prefix()) != PA_OK || (st = launch_rest()) != PA_OK) return st;
    }
    // 3. merge all partitions of every row
    const cudaError_t e = launch_lse_merge(out, static_cast<int>(out_dtype), tmp_out, max_logits, exp_sums,
                                           context_lens, num_seqs, num_heads, head_dim, pp.part_stride, 0, sms,
                                           strm);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_decode_contiguous(void *out, pa_dtype out_dtype, const void *query, pa_dtype q_dtype,
                                      const void *k, const void *v, pa_dtype kv_dtype,
                                      const int32_t *context_lens, int num_seqs, int num_heads,
                                      int num_kv_heads, int head_dim, int max_seq_len, int max_context_len,
                                      float scale, void *workspace, size_t workspace_bytes, void *stream) {
    if (max_seq_len <= 0 || max_context_len > max_seq_len) return PA_ERR_INVALID_ARG;
    const DecodeShape s{num_seqs, num_heads, num_kv_heads, head_dim, kContiguousTile,
                        static_cast<int>(cdiv64(max_seq_len, kContiguousTile)), 1, max_context_len};
    pa_status st = check_shape(s);
    if (st != PA_OK) return st;
    if (!valid_dtype(out_dtype) || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if ((st = check_dtypes(q_dtype, kv_dtype)) != PA_OK) return st;
    if (!is16(kv_dtype)) return PA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(num_seqs) * max_seq_len > INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    return decode_planned(s, out, out_dtype, query, q_dtype, k, v, kv_dtype, nullptr, context_lens,
                          max_seq_len, scale, workspace, workspace_bytes, stream);
}

PA_API pa_status pa_decode_splitk(float *tmp_out, float *max_logits, float *exp_sums,
                                  int partition_size, const void *query, pa_dtype q_dtype,
                                  const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                                  const int32_t *block_tables, const int32_t *context_lens,
                                  int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                  int block_size, int max_blocks_per_seq, int num_blocks,
                                  int max_context_len, float scale, void *stream) {
    const DecodeShape s{num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                        max_blocks_per_seq, num_blocks, max_context_len};
    pa_status st = check_shape(s);
    if (st != PA_OK) return st;
    if (partition_size <= 0 || partition_size % block_size != 0 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if ((st = check_dtypes(q_dtype, kv_dtype)) != PA_OK) return st;
    const int64_t P = cdiv64(max_context_len, partition_size);
    if (num_seqs == 0 || P == 0) return PA_OK;
    if (P > 65535) return PA_ERR_UNSUPPORTED;
    if (!tmp_out || !max_logits || !exp_sums || !query || !k_cache || !v_cache || !block_tables ||
        !context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    int dev;
    if ((st = current_device(&dev)) != PA_OK) return st;
    DecodeParams p;
    fill_common(p, s, query, q_dtype, k_cache, v_cache, block_tables, context_lens, scale);
    p.tmp_out = tmp_out;
    p.max_logits = max_logits;
    p.exp_sums = exp_sums;
    // the tensor-core kernel cuts partitions at whole 16-token tiles
    const bool mma = use_mma(s, is16(kv_dtype)) &&
                     partition_size % decode_mma_tile_tokens(block_size) == 0;
    p.ntile = (s.num_heads / s.num_kv_heads + kRowsPerTile - 1) / kRowsPerTile;
    p.heads_per_cta = mma ? decode_mma_heads_per_cta(s.num_kv_heads, heads_cap()) : 1;
    p.nsplit = static_cast<int>(P);
    p.part_tokens = partition_size;
    p.mode = kModeSplitK;
    return launch_decode(s, p, kv_dtype, mma, dev, as_stream(stream));
}

PA_API pa_status pa_lse_merge(void *out, pa_dtype out_dtype, const float *tmp_out,
                              const float *max_logits, const float *exp_sums,
                              const int32_t *context_lens, int num_seqs, int num_heads,
                              int head_dim, int max_partitions, int partition_size, void *stream) {
    if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || max_partitions <= 0 || partition_size <= 0 ||
        !valid_dtype(out_dtype))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (num_seqs > 65535 || static_cast<size_t>(max_partitions) * sizeof(float) > 200 * 1024)
        return PA_ERR_UNSUPPORTED;
    if (!out || !tmp_out || !max_logits || !exp_sums || !context_lens) return PA_ERR_INVALID_ARG;
    int dev;
    pa_status st = current_device(&dev);
    if (st != PA_OK) return st;
    const int sms = sm_count(dev);
    if (sms <= 0) return PA_ERR_CUDA;
    cudaError_t e = launch_lse_merge(out, static_cast<int>(out_dtype), tmp_out, max_logits, exp_sums,
                                     context_lens, num_seqs, num_heads, head_dim, max_partitions,
                                     partition_size, sms, as_stream(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_device_status(int *status, int clear, void *stream) {
    if (!status) return PA_ERR_INVALID_ARG;
    int dev;
    pa_status st = current_device(&dev);
    if (st != PA_OK) return st;
    int *addr = status_word(dev);
    if (!addr) return PA_ERR_CUDA;
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(status, addr, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    if (clear && *status != 0) {
        const int zero = 0;
        if (cudaMemcpyAsync(addr, &zero, sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    return PA_OK;
}

}  // extern "C"
