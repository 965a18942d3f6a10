// Paged decode attention, bf16 or fp16 K/V, tensor-core kernel for sm_103a.
//
// What it computes: for each sequence b and query head h, softmax(scale *
// q_h K^T) V over the sequence's tokens, with K and V fetched block by block
// through the block table ("What Does PagedAttention Actually Optimize?",
// sections 8 and 14; "PagedAttention, explained.", procedure step 5). Query
// head h reads KV head h / (Hq / Hkv).
//
// How. One CTA = one sequence x a group of up to 8 KV heads x up to 16 query
// heads per KV head x one partition of the sequence's tokens (whole tiles of
// 16 tokens; a block of 32 or more tokens may straddle two partitions).
//  * The last warp walks the block table (read 32 tiles' entries at a time, a
//    chunk ahead) and, per 16-token tile (two blocks when blocks are 8 tokens),
//    issues one TMA tiled load (cp.async.bulk.tensor.5d) of the tile's K and
//    one of its V into a stage of a shared-memory ring; completion is counted
//    on the stage's mbarrier. The tensor map views the cache as (dim within a
//    64-dim half, token, half, head, block), so one box covers every KV head
//    of the group and both halves: the block's K (and V) -- contiguous in the
//    [num_blocks, block_size, Hkv, D] layout -- is fetched as one burst, and
//    the producer issues two instructions per tile. Rows land head by head
//    as 64-dim halves with the 128-byte swizzle, which makes the matrix loads
//    below bank-conflict free. Blocks of 1, 2 or 4 tokens are gathered row
//    by row with bulk copies instead (rows mode, below).
//  * Called for a decode step (pa_decode_append), the producer of the CTA
//    whose partition holds a sequence's newest token first stores that
//    token's K and V rows into their slot ("PagedAttention, explained.",
//    procedure step 4), fenced against the async proxy that reads them.
//  * Consumer warp j owns KV head j of the group for the whole CTA and reads
//    every stage. S = Q K^T runs on the tensor cores (mma.m16n8k16, M = the
//    query heads of the GQA group, N = tokens, K = head dims; Q stays in
//    registers). Online softmax in base 2 with a running max and sum per row.
//    P is split into a 16-bit high part and a residual so that P.V (M =
//    heads, N = head dims, K = tokens) keeps ~16 bits of P. Each warp
//    releases the stage with one mbarrier arrive; the stage is refilled once
//    every head's warp has released it.
//  * Tokens past the context in the last tile are masked (score -inf, V rows
//    zeroed in shared memory, so stale or NaN slot contents never leak).
//  * Each warp finishes its own head from registers: the final output or a
//    split-K partition (merged by the log-sum-exp merge kernel); or, when a
//    context's partitions form one thread-block cluster, the partitions are
//    merged through distributed shared memory.
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the device status word, drains its own copies and returns.
#include "device_common.cuh"
#include "internal.h"
#include "mma_tile.cuh"

namespace pa {

template <int D, int TT>
struct MmaCfg {
    static constexpr int kMaxHeads = 8;                 // KV heads per CTA = consumer warps
    static constexpr int kThreads = 32 * (kMaxHeads + 1);   // one producer warp (rows mode: two)
    __host__ __device__ static constexpr int producers(int load_mode) { return load_mode == 2 ? 2 : 1; }
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = TT * 128;         // one 64-dim half of one head's tile
    static constexpr int kHeadBytes = TT * D * 2;       // one head's K (or V) rows of a tile
    // Stage layout, K then V: [head][64-dim half][token][128 bytes], filled by
    // one TMA box (64 dims x TT tokens x every half x every head of the CTA).
    // Blocks of TT / 2 tokens: [block of the pair][head][half][token].
    static constexpr int kMaxRingBytes = 200 * 1024;
    static constexpr int kMaxStages = 32;
    static constexpr size_t kBarrierBytes = 2 * kMaxStages * sizeof(uint64_t);
    static size_t smem_bytes(int ring) { return 1024 + static_cast<size_t>(ring) + kBarrierBytes; }
    static_assert(kHalfBytes % 1024 == 0, "swizzled halves must stay 1024-byte aligned");
    static_assert(TT == 16, "tiles are 16 tokens (two 8-token blocks, or part of a larger block)");
};

__device__ __forceinline__ void store_out2(const DecodeParams &p, int64_t idx, float a, float c) {
    store_pair_as(p.out, out_type_of(p), idx, a, c);
}


// Write a warp's result (final output or split-K partition) for query heads
// h0 .. h0+rows-1.
template <int D>
__device__ __forceinline__ void warp_epilogue(const DecodeParams &p, WarpState<D> &st, int b, int part,
                                              int h0, int rows, int lane) {
    const int r = lane >> 2, q4 = lane & 3;
    const bool v0 = r < rows, v1 = r + 8 < rows;
    if (p.mode == kModeFinal) {
        const float i0 = st.l0 > 0.f ? 1.f / st.l0 : 0.f, i1 = st.l1 > 0.f ? 1.f / st.l1 : 0.f;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            const int d = 8 * dn + 2 * q4;
            if (v0) store_out2(p, (static_cast<int64_t>(b) * p.num_heads + h0 + r) * D + d,
                               st.o[dn][0] * i0, st.o[dn][1] * i0);
            if (v1) store_out2(p, (static_cast<int64_t>(b) * p.num_heads + h0 + r + 8) * D + d,
                               st.o[dn][2] * i1, st.o[dn][3] * i1);
        }
        return;
    }
    const int64_t row0 = split_row(p, b, h0 + r, part);
    const int64_t row1 = split_row(p, b, h0 + r + 8, part);
    const float i0 = st.l0 > 0.f ? 1.f / st.l0 : 0.f, i1 = st.l1 > 0.f ? 1.f / st.l1 : 0.f;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
        const int d = 8 * dn + 2 * q4;
        if (v0) *reinterpret_cast<float2 *>(p.tmp_out + row0 * D + d) = make_float2(st.o[dn][0] * i0, st.o[dn][1] * i0);
        if (v1) *reinterpret_cast<float2 *>(p.tmp_out + row1 * D + d) = make_float2(st.o[dn][2] * i1, st.o[dn][3] * i1);
    }
    if (q4 == 0) {   // report the true max: sum of 2^(s - t) = l * 2^(m - t)
        if (v0) {
            p.max_logits[row0] = st.l0 > 0.f ? st.t0 * kLn2 : -INFINITY;
            p.exp_sums[row0] = st.l0 > 0.f ? st.l0 * fast_exp2(st.m0 - st.t0) : 0.f;
        }
        if (v1) {
            p.max_logits[row1] = st.l1 > 0.f ? st.t1 * kLn2 : -INFINITY;
            p.exp_sums[row1] = st.l1 > 0.f ? st.l1 * fast_exp2(st.m1 - st.t1) : 0.f;
        }
    }
}

// Split merged inside a thread-block cluster: the cluster is the nsplit
// partitions of one (sequence, KV-head group, head tile). Each CTA leaves the
// per-head softmax states of its partition in its own shared memory (m[16],
// l[16], O[16][D + 8] per head: rows padded by 8 floats, so that the 8-byte
// stores of a half-warp's four rows fall in 32 different banks); after a
// cluster barrier every CTA merges a slice of the outputs by reading all
// partitions straight from its peers' shared memory; a second barrier keeps
// each CTA (and its shared memory) alive until every peer is done reading it.
// Its arrive is relaxed: the reads it waits for have been consumed by then,
// and nothing else needs ordering. No global workspace, no atomics.
template <int D>
__device__ __forceinline__ void cluster_exchange_merge(const DecodeParams &p, const WarpState<D> &st, float *sm, int b,
                                       int hgrp, int tile, int rows, int warp, int lane) {
    constexpr int kStride = D + 8;                         // floats per state row
    constexpr int kRegion = 32 + kRowsPerTile * kStride;   // floats per head
    const int hpc = p.heads_per_cta;
    if (warp < hpc) {
        float *reg = sm + warp * kRegion;
        const int r = lane >> 2, q4 = lane & 3;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            const int d = 8 * dn + 2 * q4;
            *reinterpret_cast<float2 *>(reg + 32 + r * kStride + d) = make_float2(st.o[dn][0], st.o[dn][1]);
            *reinterpret_cast<float2 *>(reg + 32 + (r + 8) * kStride + d) = make_float2(st.o[dn][2], st.o[dn][3]);
        }
        if (q4 == 0) {   // (max, sum) pairs, row-major
            *reinterpret_cast<float2 *>(reg + 2 * r) = make_float2(st.m0, st.l0);
            *reinterpret_cast<float2 *>(reg + 2 * (r + 8)) = make_float2(st.m1, st.l1);
        }
    }
    cluster_sync_all();   // every partition's state is now readable cluster-wide

    // Each thread merges 4 consecutive dims of one (head, row): it issues the
    // reads of all partitions (a 16-byte vector of O and the (max, sum) pair
    // each) before using any of them, so the exchange costs one round of
    // distributed-shared-memory reads.
    const int ns = p.nsplit;                 // cluster size
    const int rank = static_cast<int>(cluster_rank());
    constexpr int kD4 = D / 4;
    const int total = hpc * rows * kD4;
    const int chunk = (total + ns - 1) / ns;
    const int begin = rank * chunk;
    const int end = min(total, begin + chunk);
    const uint32_t base = smem_addr(sm);
    for (int idx = begin + static_cast<int>(threadIdx.x); idx < end; idx += blockDim.x) {
        const int j = idx / (rows * kD4);
        const int rem = idx - j * rows * kD4;
        const int rr = rem / kD4, d4 = rem - rr * kD4;
        const uint32_t ml_off = base + 4u * static_cast<uint32_t>(j * kRegion + 2 * rr);
        const uint32_t o_off = base + 4u * static_cast<uint32_t>(j * kRegion + 32 + rr * kStride + 4 * d4);
        float2 ml[8];
        float4 oq[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (q < ns) {
                ml[q] = ld_cluster_f32x2(cluster_map(ml_off, q));
                oq[q] = ld_cluster_f32x4(cluster_map(o_off, q));
            } else {
                ml[q] = make_float2(-INFINITY, 0.f);
                oq[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (ml[q].y > 0.f) M = fmaxf(M, ml[q].x);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (ml[q].y > 0.f) {
                const float wq = fast_exp2(ml[q].x - M);
                L += wq * ml[q].y;
                acc.x += wq * oq[q].x;
                acc.y += wq * oq[q].y;
                acc.z += wq * oq[q].z;
                acc.w += wq * oq[q].w;
            }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const int h = (hgrp * hpc + j) * p.group + tile * kRowsPerTile + rr;
        const int64_t o = (static_cast<int64_t>(b) * p.num_heads + h) * D + 4 * d4;
        store_out2(p, o, acc.x * inv, acc.y * inv);
        store_out2(p, o + 2, acc.z * inv, acc.w * inv);
    }
    // peers have finished reading this CTA's shared memory
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

// How the producer fills a stage: one TMA box per tile (blocks of 16 tokens
// or more), two boxes per tile (blocks of 8), or one bulk copy per token row
// (blocks of 1, 2 or 4 tokens: a box of fewer than 8 rows cannot fill the
// 1024-byte swizzle atom on its own). Rows mode lays a stage out as
// [token][head][dim] with rows padded by 16 bytes instead of swizzled.
enum LoadMode { kLoadBox = 0, kLoadPairs = 1, kLoadRows = 2 };
static_assert(MmaCfg<128, 16>::producers(kLoadRows) == 2 && MmaCfg<128, 16>::producers(kLoadBox) == 1, "");

template <int D, int TT, bool kCluster, int kLoad, bool kF16>
__global__ void __launch_bounds__(32 * (MmaCfg<D, TT>::kMaxHeads + MmaCfg<D, TT>::producers(kLoad)), 1)
decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ DecodeParams p) {
    using C = MmaCfg<D, TT>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.ring_bytes);
    __shared__ int s_abort;
    __shared__ int s_issued;

    const int hpc = p.heads_per_cta;
    const int part = blockIdx.x;
    const int hgrp = blockIdx.y / p.ntile;
    const int tile = blockIdx.y % p.ntile;
    const int b = blockIdx.z;
    const int rows = min(kRowsPerTile, p.group - tile * kRowsPerTile);
    // the previous kernel on the stream (e.g. the scatter) is complete
    if (p.pair_role != kPairSecond) grid_dependency_wait();
    if (p.pair_role == kPairFirst) grid_dependents_launch();
    // second of a pair: one CTA outlives the first kernel (the others need not hold their SMs)
    const bool tie = p.pair_role == kPairSecond && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
    const SeqWork w = seq_work(p, b, part);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // (one instantiation per epilogue keeps the other's registers out of the loop)
    constexpr bool cluster = kCluster;
    if (w.tok_begin >= w.tok_end && !cluster) {
        if (warp < hpc) {
            const int gh = hgrp * hpc + warp;
            warp_write_empty<D>(p, b, gh * p.group + tile * kRowsPerTile, part, rows, w.nparts, lane);
        }
        if (tie) grid_dependency_wait();
        return;
    }
    // (in a cluster every CTA takes part in the exchange, an empty partition included)
    const int tok_begin = w.tok_begin;     // a multiple of TT (partitions are whole tiles)
    const int tok_end = w.tok_end;
    const int ntiles = tok_end > tok_begin ? (tok_end - tok_begin + TT - 1) / TT : 0;
    const int bs = p.block_size;
    // A tile is TT tokens of one block; or (pairs: blocks of TT / 2 tokens)
    // two whole blocks back to back, one TMA box of box_rows rows each; or
    // (copies) TT / bs short blocks, gathered row by row into the one-box
    // layout. (Separate instantiations: the second box's loads, even never
    // taken, slow the single-box loop.)
    constexpr bool kPairs = kLoad == kLoadPairs;
    constexpr bool kRows = kLoad == kLoadRows;
    constexpr int bpt = kPairs ? 2 : 1;
    constexpr int box_rows = TT / bpt;
    // rows mode: one token's K (or V) for the group's heads, plus 16 bytes of
    // padding that puts 8 consecutive rows in 8 different bank groups
    const int row_pitch = hpc * D * 2 + 16;
    const int stage_bytes = kRows ? 2 * TT * row_pitch : 2 * hpc * C::kHeadBytes;
    int nstages = p.ring_bytes / stage_bytes;
    if (nstages > C::kMaxStages) nstages = C::kMaxStages;
    const int v_off = stage_bytes / 2;
    // byte offsets within one stage's K (or V): head, 64-dim half, token row
    constexpr int kHalfStride = kRows ? 128 : box_rows * 128;
    constexpr int kHeadStride = kRows ? D * 2 : C::kHalves * kHalfStride;
    const int pair_stride = hpc * kHeadStride;     // second block of a pair
    auto tok_off = [&](int t) -> int {
        return kRows ? t * row_pitch : kPairs ? (t / box_rows) * pair_stride + (t % box_rows) * 128 : t * 128;
    };

    constexpr int kProducers = C::producers(kLoad);
    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(smem_addr(&bars[s]), kProducers);   // one arrival per producer warp
            mbar_init(smem_addr(&bars[C::kMaxStages + s]), hpc);
        }
        s_abort = 0;
        s_issued = 0;
        mbar_fence_init();
    }
    __syncthreads();

    WarpState<D> st;
    st.init();

    if (kRows && warp >= hpc) {
        // ------------------------ producers (short blocks) --------------------
        // Per tile, lane t < 16 of the first producer warp copies token t's K
        // row, and of the second its V row (the group's heads: hpc * D * 2
        // contiguous bytes of the cache), one bulk copy each, counted in bytes
        // on the stage's mbarrier. (A warp issues bulk copies one at a time:
        // two warps double the rate at which the copies start.) The block ids
        // of 32 blocks are held one per lane and fetched a chunk ahead; a
        // tile's TT / bs blocks never straddle two chunks (bs divides TT
        // divides 32).
        const bool is_v = warp > hpc;
        const int32_t *table = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;
        const int bs_shift = __ffs(bs) - 1;
        const int nb = TT >> bs_shift;                                  // blocks per tile
        const int blk_begin = tok_begin >> bs_shift;                    // tok_begin is whole tiles
        const int nblk = (tok_end - tok_begin + bs - 1) >> bs_shift;    // blocks of this partition
        auto entry = [&](int j) -> int { return j < nblk ? table[blk_begin + j] : 0; };
        int cur = entry(lane), nxt = entry(32 + lane);
        const uint64_t policy = l2_policy_evict_first();
        const int64_t row_bytes = static_cast<int64_t>(p.num_kv_heads) * D * 2;   // one token, all heads
        const int64_t blk_bytes = row_bytes * bs;
        const uint32_t grp_bytes = static_cast<uint32_t>(hpc * D * 2);           // copied per row
        const int t = lane & (TT - 1);
        const unsigned char *src_base = static_cast<const unsigned char *>(is_v ? p.v_cache : p.k_cache) +
                                        hgrp * hpc * D * 2 + (t & (bs - 1)) * row_bytes;
        const uint32_t dst_lane = static_cast<uint32_t>((is_v ? v_off : 0) + t * row_pitch);
        if (p.append_key && tok_begin <= w.len - 1 && w.len - 1 < tok_end &&
            p.context_lens[b] == w.len)   // this CTA reads the new token (a length cut short writes none)
            warp_append_row<D>(p, is_v ? p.append_value : p.append_key, is_v ? p.v_cache : p.k_cache, b,
                               w.len - 1, hgrp * hpc, hpc, lane);
        int issued = 0;
        for (int i = 0; i < ntiles; ++i) {
            const int j0 = i * nb;
            if ((j0 & 31) == 0 && j0 > 0) {
                cur = nxt;
                nxt = entry(j0 + 32 + lane);
            }
            const int blk = __shfl_sync(0xffffffffu, cur, (j0 + (t >> bs_shift)) & 31);
            const bool live = lane < TT && t < min(TT, tok_end - (tok_begin + i * TT));
            // a block id outside the pool is not read: its rows are zeroed
            const bool in_pool = static_cast<unsigned>(blk) < static_cast<unsigned>(p.num_blocks);
            const unsigned ncopy = __popc(__ballot_sync(0xffffffffu, live && in_pool));
            int ok = 1;
            const int s = i % nstages, k = i / nstages;
            const uint32_t full = smem_addr(&bars[s]);
            if (lane == 0) {
                if (k > 0) {
                    if (*reinterpret_cast<volatile int *>(&s_abort)) {
                        ok = 0;
                    } else if (!mbar_wait(smem_addr(&bars[C::kMaxStages + s]), (k - 1) & 1)) {
                        record_status(p.status, kStatusTimeout);
                        s_abort = 1;
                        ok = 0;
                    }
                }
                if (ok) mbar_expect_tx(full, ncopy * grp_bytes);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            const uint32_t dst = smem_addr(smem + s * stage_bytes) + dst_lane;
            if (live && in_pool) {
                bulk_load(dst, src_base + blk * blk_bytes, grp_bytes, full, policy);
            } else if (live) {
                for (uint32_t o = 0; o < grp_bytes; o += 16)
                    *reinterpret_cast<uint4 *>(smem + s * stage_bytes + dst_lane + o) = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(full);   // after the zeroed rows: the phase covers them
            issued = i + 1;
        }
        if (lane == 0 && !is_v) s_issued = issued;
    } else if (!kRows && warp == hpc) {
        // ------------------------------ producer ------------------------------
        // paged: each box's block id from the table; contiguous: token offset only
        const bool contig = p.contig_stride > 0;
        const int32_t *table = contig ? nullptr : p.block_tables + static_cast<int64_t>(b) * p.max_blocks;
        const int contig_tok0 = contig ? b * p.contig_stride + tok_begin : 0;
        uint64_t policy = 0;
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
            policy = l2_policy_evict_first();
        }
        // Block id of box j of tile t; entries for 32 tiles are fetched at a
        // time, one chunk ahead. Boxes past the context are not read (the
        // table holds no entry for them).
        auto entry = [&](int t, int j) -> int {
            const int tok = tok_begin + t * TT + j * box_rows;
            return (!contig && t < ntiles && tok < tok_end) ? table[tok / bs] : 0;
        };
        int cur0 = entry(lane, 0), cur1 = kPairs ? entry(lane, 1) : 0;
        int nxt0 = entry(32 + lane, 0), nxt1 = kPairs ? entry(32 + lane, 1) : 0;
        int issued = 0;
        const int head0 = hgrp * hpc;
        if (p.append_key && tok_begin <= w.len - 1 && w.len - 1 < tok_end &&
            p.context_lens[b] == w.len) {   // this CTA reads the new token (a length cut short writes none)
            warp_append_row<D>(p, p.append_key, p.k_cache, b, w.len - 1, head0, hpc, lane);
            warp_append_row<D>(p, p.append_value, p.v_cache, b, w.len - 1, head0, hpc, lane);
        }
        for (int i = 0; i < ntiles; ++i) {
            if ((i & 31) == 0 && i > 0) {
                cur0 = nxt0;
                cur1 = nxt1;
                nxt0 = entry(i + 32 + lane, 0);
                if (kPairs) nxt1 = entry(i + 32 + lane, 1);
            }
            const int phys0 = __shfl_sync(0xffffffffu, cur0, i & 31);
            const int phys1 = kPairs ? __shfl_sync(0xffffffffu, cur1, i & 31) : 0;
            int ok = 1;
            if (lane == 0) {
                const int s = i % nstages, k = i / nstages;
                if (k > 0) {
                    if (*reinterpret_cast<volatile int *>(&s_abort)) {
                        ok = 0;
                    } else if (!mbar_wait(smem_addr(&bars[C::kMaxStages + s]), (k - 1) & 1)) {
                        record_status(p.status, kStatusTimeout);
                        s_abort = 1;
                        ok = 0;
                    }
                }
                if (ok) {
                    const int t0 = tok_begin + i * TT;
                    // boxes with tokens in them (the last tile may hold fewer blocks)
                    const int nbox = kPairs && t0 + box_rows < tok_end ? 2 : 1;
                    const uint32_t full = smem_addr(&bars[s]);
                    mbar_arrive_expect_tx(full, static_cast<uint32_t>(stage_bytes / bpt * nbox));
                    const uint32_t kdst = smem_addr(smem + s * stage_bytes);
                    const int tok0 = contig ? contig_tok0 + i * TT : t0 % bs;
                    const int blk0 = contig ? 0 : phys0;
                    // tensor-map coordinates, innermost first: (dim, token, half, head, block);
                    // one box of K and one of V per block
                    tma_load_5d(kdst, &tmap_k, 0, tok0, 0, head0, blk0, full, policy);
                    tma_load_5d(kdst + v_off, &tmap_v, 0, tok0, 0, head0, blk0, full, policy);
                    if (kPairs && nbox > 1) {
                        tma_load_5d(kdst + pair_stride, &tmap_k, 0, 0, 0, head0, phys1, full, policy);
                        tma_load_5d(kdst + v_off + pair_stride, &tmap_v, 0, 0, 0, head0, phys1, full, policy);
                    }
                    issued = i + 1;
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        }
        if (lane == 0) s_issued = issued;
    } else if (warp < hpc) {
        // ------------------------------ consumers -----------------------------
        const int gh = hgrp * hpc + warp;                     // this warp's KV head
        const int h0 = gh * p.group + tile * kRowsPerTile;    // its first query head
        const int r = lane >> 2;
        uint32_t qa[D / 16][4];
        {
            const uint32_t *q0 = reinterpret_cast<const uint32_t *>(
                static_cast<const uint16_t *>(p.query) +
                (static_cast<int64_t>(b) * p.num_heads + h0 + r) * D);
            load_query_fragments<D>(qa, q0, q0 + 8 * (D / 2), r < rows, r + 8 < rows, lane);
        }
        const float sl2 = p.scale_log2;

        for (int i = 0; i < ntiles; ++i) {
            if (*reinterpret_cast<volatile int *>(&s_abort)) break;
            const int s = i % nstages, k = i / nstages;
            if (!mbar_wait(smem_addr(&bars[s]), k & 1)) {
                record_status(p.status, kStatusTimeout);
                s_abort = 1;
                break;
            }
            unsigned char *kst = smem + s * stage_bytes + warp * kHeadStride;   // this head (rows: its dims)
            const uint32_t kbase = smem_addr(kst);
            const uint32_t vbase = kbase + v_off;
            const int valid = min(TT, tok_end - (tok_begin + i * TT));
            if (valid < TT) {
                // zero this head's V rows past the context (whole 128-byte rows)
                for (int c = lane; c < C::kHalves * TT * 8; c += 32) {
                    const int hh = c / (TT * 8), row = (c % (TT * 8)) / 8;
                    if (row >= valid)
                        *reinterpret_cast<uint4 *>(kst + v_off + hh * kHalfStride + tok_off(row) + (c % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }

            warp_tile_attention<D, TT, !kRows, kF16>(st, qa, kbase, vbase, kHalfStride, tok_off, valid, valid, sl2,
                                                     lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars[C::kMaxStages + s]));
        }
        st.reduce_sums();
        if (!cluster) warp_epilogue<D>(p, st, b, part, h0, rows, lane);
    }

    // Drain: wait (bounded) for the last phase of every stage this CTA armed,
    // so that no copy is still landing in shared memory when the CTA exits
    // (or when the ring is reused below).
    __syncthreads();
    if (threadIdx.x == 0) {
        const int issued = s_issued;
        for (int s = 0; s < nstages && s < issued; ++s) {
            const int k_last = (issued - 1 - s) / nstages;
            if (!mbar_wait(smem_addr(&bars[s]), k_last & 1)) record_status(p.status, kStatusTimeout);
        }
    }
    if (cluster) {
        __syncthreads();
        cluster_exchange_merge<D>(p, st, reinterpret_cast<float *>(smem), b, hgrp, tile, rows, warp, lane);
    }
    if (tie) grid_dependency_wait();
}

template <int D, int TT, int kLoad, bool kF16>
static cudaError_t launch_impl(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                               dim3 grid, cudaStream_t stream) {
    using C = MmaCfg<D, TT>;
    const size_t smem = C::smem_bytes(p.ring_bytes);
    const dim3 block(32 * (p.heads_per_cta + C::producers(kLoad)));
    if (!p.cluster_merge) {
        auto kern = decode_mma_kernel<D, TT, false, kLoad, kF16>;
        static unsigned long long done = 0;
        cudaError_t e = ensure_smem_limit(kern, C::smem_bytes(C::kMaxRingBytes), done);
        if (e != cudaSuccess) return e;
        return launch_kernel(kern, grid, block, smem, stream, 1u, tk, tv, p);
    }
    auto kern = decode_mma_kernel<D, TT, true, kLoad, kF16>;
    static unsigned long long done = 0;
    cudaError_t e = ensure_smem_limit(kern, C::smem_bytes(C::kMaxRingBytes), done);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, block, smem, stream, grid.x, tk, tv, p);
}

bool decode_mma_supported(int head_dim, int block_size) {
    return (head_dim == 64 || head_dim == 128) && block_size >= 1 && block_size <= 256 &&
           (block_size & (block_size - 1)) == 0;
}

int decode_mma_tile_tokens(int) { return 16; }

int decode_mma_box_tokens(int block_size) { return block_size < 16 ? block_size : 16; }

int decode_mma_heads_per_cta(int num_kv_heads, int max_heads) {
    for (int h = max_heads < MmaCfg<128, 16>::kMaxHeads ? max_heads : MmaCfg<128, 16>::kMaxHeads; h > 1; --h)
        if (num_kv_heads % h == 0) return h;
    return 1;
}

int decode_mma_stage_bytes(int head_dim, int block_size, int heads_per_cta) {
    const int tt = decode_mma_tile_tokens(block_size);
    if (block_size < 8) return 2 * tt * (heads_per_cta * head_dim * 2 + 16);   // padded token rows
    return 2 * heads_per_cta * tt * head_dim * 2;
}

int decode_mma_ring_bytes(int head_dim, int block_size, int heads_per_cta, int budget_bytes) {
    // stages are counted at the unpadded size, so that the padding of rows
    // mode does not cost a stage of the budget
    const int stage = decode_mma_stage_bytes(head_dim, block_size, heads_per_cta);
    const int nominal = 2 * heads_per_cta * decode_mma_tile_tokens(block_size) * head_dim * 2;
    int n = budget_bytes / nominal;
    while (n > 1 && n * stage > MmaCfg<128, 16>::kMaxRingBytes) --n;
    return (n < 1 ? 1 : n) * stage;
}

int decode_mma_cluster_bytes(int head_dim, int heads_per_cta) {
    return heads_per_cta * (32 + kRowsPerTile * (head_dim + 8)) * 4;   // the exchange's state rows, padded
}

int decode_mma_load_mode(int block_size, bool contiguous) {
    if (contiguous || block_size >= 16) return kLoadBox;
    return block_size == 8 ? kLoadPairs : kLoadRows;   // blocks of 8: two per 16-token tile
}

template <int D, bool kF16>
static cudaError_t launch_for_dim(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                                  dim3 grid, cudaStream_t stream) {
    switch (decode_mma_load_mode(p.block_size, p.contig_stride > 0)) {
        case kLoadBox: return launch_impl<D, 16, kLoadBox, kF16>(p, tk, tv, grid, stream);
        case kLoadPairs: return launch_impl<D, 16, kLoadPairs, kF16>(p, tk, tv, grid, stream);
        default: return launch_impl<D, 16, kLoadRows, kF16>(p, tk, tv, grid, stream);
    }
}

cudaError_t launch_decode_mma(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                              dim3 grid, cudaStream_t stream) {
    if (p.head_dim == 128)
        return p.kv_f16 ? launch_for_dim<128, true>(p, tk, tv, grid, stream)
                        : launch_for_dim<128, false>(p, tk, tv, grid, stream);
    if (p.head_dim == 64)
        return p.kv_f16 ? launch_for_dim<64, true>(p, tk, tv, grid, stream)
                        : launch_for_dim<64, false>(p, tk, tv, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
