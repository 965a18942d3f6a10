// Shared-prefix attention pass on the fifth-generation tensor cores
// (tcgen05 + tensor memory), sm_103a.
//
// What it computes: the same as the mma.sync prefix pass -- for every query
// row (sequence, query head) of the batch, attention over one chunk of the
// blocks all sequences share, in split form (normalised partial output,
// maximum score in natural-log units, sum of exp(score - maximum)); the
// decode kernel attends the rest of each context and the log-sum-exp merge
// combines them ("PagedAttention: KV cache virtual memory", "Copy-on-write:
// when two requests share a prefix"; "What Does PagedAttention Actually
// Optimize?", section 8: attention is unchanged by how K and V are stored).
//
// Why tcgen05 here: with up to 128 query rows per KV head against the same
// K/V, the prefix is a real matrix product (M = 128 rows, N = 64 tokens per
// tile, K = head_dim for Q.K^T; M = 128, N = head_dim, K = 64 tokens for
// P.V), unlike per-sequence decode where M is one GQA group.
//
// How. A row group is floor(128 / G) whole sequences x their G query heads
// of one KV head (G = Hq / Hkv), row R = sequence * G + head, at most 128
// rows: one tensor-memory lane each. One CTA = one KV head x one chunk of
// the prefix x kGroups (1 or 2) row groups, which share every K/V tile.
//  * Warp 4 kGroups (TMA) loads the row groups' Q with one tensor-map box
//    per 64-dim half (K-major, 128-byte swizzle, the MMA's A layout), then
//    streams the tiles' K and V (one box per block, 64-dim half and cache)
//    into a ring of stages guarded by mbarriers.
//  * Warp 4 kGroups + 1 owns the tensor memory (per row group: S
//    double-buffered, 2 x 64 columns, and O, head_dim columns) and one of
//    its threads issues the MMAs: per tile, S = Q K^T for each row group,
//    then O += P_hi V + P_lo V for each row group's previous tile (V read
//    MN-major), with tcgen05.commit arriving on the mbarriers that release
//    S to the softmax warps, the P buffer, and the ring stage.
//  * Warps 4 g .. 4 g + 3 run row group g's softmax, one row per thread (its
//    tensor-memory lane): the base-2 online softmax in registers, O rescaled
//    in tensor memory when the running max moves by more than 8 (rare), P
//    written as a 16-bit high part and residual into the group's shared
//    buffer once the previous tile's P.V has read it.
//  * Epilogue: O / l goes through shared memory, laid out as the 128-byte
//    swizzled boxes of a tensor map over the partial outputs, and one
//    thread writes each box with a TMA store (rows are scattered over the
//    partial array: per-thread row stores cost ~32 L1 wavefronts each).
// Every wait is bounded; on expiry the kernel records a timeout, waits for
// its own MMAs and copies (bounded), frees its tensor memory and returns.
#include "device_common.cuh"
#include "internal.h"
#include "mma_tile.cuh"
#include "tcgen05.cuh"

namespace pa {

namespace {

constexpr int kTcLanes = 128;            // tensor-memory lanes: MMA M, rows of a row group at most
constexpr int kTcTile = 64;              // tokens per tile (MMA N of Q.K^T, K of P.V)
constexpr int kTcMaxStages = 8;
constexpr int kTcMaxChunkBlocks = kTcChunkBlocks;   // block ids of one chunk, staged in shared memory
constexpr float kTcSlack = 8.f;          // base-2 headroom before the running max moves
constexpr int kTcOutCols = 32;           // fp32 columns per output box (128 bytes: the swizzle span)

template <int D, int kGroups>
struct TcCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kQBytes = kHalves * kTcLanes * 128;     // one row group's Q, K-major per half
    static constexpr int kPBytes = kTcLanes * 128;               // one P part (hi or lo) of one row group
    static constexpr int kKBytes = kHalves * kTcTile * 128;      // one tile's K (or V)
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kOutBoxBytes = kTcLanes * 128;          // 32 fp32 columns of 128 rows
    static constexpr int kOutBytes = (D / kTcOutCols) * kOutBoxBytes;   // one row group's O, staged
    static constexpr int kSoftmaxWarps = 4 * kGroups;
    static constexpr int kThreads = 32 * (kSoftmaxWarps + 2);
    static constexpr int kTmaWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;
    static constexpr uint32_t kTmemCols = kGroups == 1 ? 256u : 512u;
    // tensor-memory columns of row group g: S buffer b, and O (head_dim <= 128 columns)
    __device__ static constexpr uint32_t s_col(int g, int b) { return g * 128 + b * kTcTile; }
    __device__ static constexpr uint32_t o_col(int g) { return kGroups * 128 + g * 128; }
    // shared memory: Q (every group) | P hi/lo (every group) | ring | barriers.
    // After the last P.V the P buffers and the ring hold the staged output.
    static constexpr int kPOffset = kGroups * kQBytes;
    static constexpr int kRingOffset = kPOffset + 2 * kGroups * kPBytes;
    static size_t smem_bytes(int ring);
    // At least two stages: tile i + 1's Q.K^T is issued before tile i's P.V,
    // which frees tile i's stage, so one stage would wait on itself. And the
    // staged output must fit in P + ring.
    static int min_ring_bytes() {
        const int need = kGroups * kOutBytes - 2 * kGroups * kPBytes;
        return need > 2 * kStageBytes ? need : 2 * kStageBytes;
    }
    static int max_ring_bytes();    // whole stages within the shared memory of one CTA
};

struct TcBars {
    uint64_t full[kTcMaxStages];
    uint64_t empty[kTcMaxStages];
    uint64_t q_full;                       // the row groups' Q has landed
    uint64_t s_full[2][2], s_free[2][2];   // [row group][S buffer]: written by Q.K^T, read by softmax
    uint64_t p_full[2], pv_done[2];        // [row group]: P written by softmax, read by P.V
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int issued;
    int blk[kTcMaxChunkBlocks];            // the chunk's block ids
};

template <int D, int kGroups>
size_t TcCfg<D, kGroups>::smem_bytes(int ring) {
    return 1024 + static_cast<size_t>(kRingOffset) + static_cast<size_t>(ring) + sizeof(TcBars);
}

constexpr int kSmemPerCta = 227 * 1024;   // dynamic shared memory one CTA may have

template <int D, int kGroups>
int TcCfg<D, kGroups>::max_ring_bytes() {
    int room = kSmemPerCta - static_cast<int>(smem_bytes(0));
    if (room > kTcMaxRingBytes) room = kTcMaxRingBytes;
    if (room > kTcMaxStages * kStageBytes) room = kTcMaxStages * kStageBytes;
    return room / kStageBytes * kStageBytes;
}

// A matrix descriptor's start-address field is the byte address / 16 in its
// low 14 bits; shared-memory addresses stay below 2^18, so the descriptor of
// base + bytes is the base's plus bytes / 16 (no carry leaves the field).
// Stepping by constant adds keeps the MMA thread's work per instruction to
// one add: computed in full each time, the descriptors cost more issue time
// than the instructions themselves at N = 64.
__host__ __device__ constexpr uint64_t desc_step(int bytes) { return static_cast<uint64_t>(bytes >> 4); }

__device__ __forceinline__ bool tc_wait(const PrefixParams &p, TcBars *bars, uint64_t *bar, uint32_t parity) {
    if (*reinterpret_cast<volatile int *>(&bars->abort_flag)) return false;
    if (mbar_wait(smem_addr(bar), parity)) return true;
    record_status(p.status, kStatusTimeout);
    bars->abort_flag = 1;
    return false;
}

// Barrier among the softmax warps only (named barrier 1).
__device__ __forceinline__ void softmax_warps_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// TMA tiled store shared -> global (4-D map), tracked as a bulk group.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
// Commit the bulk stores issued so far and wait until they have read their
// shared-memory source (the writes themselves complete with the grid).
__device__ __forceinline__ void bulk_commit_and_wait_read() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

template <int D, int kGroups, bool kF16>
__global__ void __launch_bounds__(TcCfg<D, kGroups>::kThreads, 1)
prefix_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_o,
                 const __grid_constant__ PrefixParams p) {
    using C = TcCfg<D, kGroups>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *q_s = smem;
    unsigned char *pbuf = smem + C::kPOffset;         // [row group][hi, lo]
    unsigned char *ring = smem + C::kRingOffset;
    unsigned char *stage_out = pbuf;                  // the staged output (after the last P.V)
    TcBars *bars = reinterpret_cast<TcBars *>(ring + p.ring_bytes);
    auto p_hi = [&](int g) { return pbuf + (2 * g) * C::kPBytes; };
    auto p_lo = [&](int g) { return pbuf + (2 * g + 1) * C::kPBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == C::kTmaWarp && lane == 0) {   // the maps are kernel parameters: fetch them now
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
        tma_prefetch_desc(&tmap_o);
    }
    if (p.pair_role != kPairSecond) grid_dependency_wait();
    if (p.pair_role == kPairFirst) grid_dependents_launch();
    const int chunk = blockIdx.x, kvh = blockIdx.y;
    const int grp0 = blockIdx.z * kGroups;                      // this CTA's first row group
    const int ngrp = min(kGroups, p.row_groups - grp0);         // row groups with rows (>= 1)
    const int tok_begin = chunk * p.chunk_tokens;
    const int tok_end = min(p.prefix_tokens, tok_begin + p.chunk_tokens);
    const int ntiles = tok_end > tok_begin ? (tok_end - tok_begin) / kTcTile : 0;   // whole tiles
    int nstages = p.ring_bytes / C::kStageBytes;
    if (nstages > kTcMaxStages) nstages = kTcMaxStages;
    const int spg = p.seqs_per_group;                  // sequences per row group
    const int rows = spg * p.group;                    // rows per row group (<= 128)
    const int bs = p.block_size;
    const int R_box = bs < kTcTile ? bs : kTcTile;     // tokens per TMA box
    const int first = tok_begin / bs;

    // TMA producer: one thread; tile i into stage i % nstages
    uint64_t policy = 0;
    auto issue_tile = [&](int i) {
        const int s = i % nstages;
        const uint32_t full = smem_addr(&bars->full[s]);
        mbar_arrive_expect_tx(full, static_cast<uint32_t>(C::kStageBytes));
        const uint32_t kdst = smem_addr(ring + s * C::kStageBytes);
        const uint32_t vdst = kdst + C::kKBytes;
        const int t0 = tok_begin + i * kTcTile;
        for (int j = 0; j < kTcTile / R_box; ++j) {
            const int tok = t0 + j * R_box;
            const int blk = bars->blk[tok / bs - first];
            const int off = tok % bs;
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) {
                const uint32_t o = h * (kTcTile * 128) + j * R_box * 128;
                // coordinates, innermost first: (dim, token, half, head, block)
                tma_load_5d(kdst + o, &tmap_k, 0, off, h, kvh, blk, full, policy);
                tma_load_5d(vdst + o, &tmap_v, 0, off, h, kvh, blk, full, policy);
            }
        }
    };

    // ---- setup: the TMA warp loads Q and starts the first tiles while the
    // MMA warp allocates tensor memory ----
    int preissued = 0;
    if (warp == C::kTmaWarp) {
        const int nblk = tok_end > tok_begin ? (tok_end - 1) / bs - first + 1 : 0;   // <= kTcMaxChunkBlocks
        for (int e = lane; e < nblk; e += 32) bars->blk[e] = p.prefix_table[first + e];
        __syncwarp();
        if (lane == 0) {
            for (int s = 0; s < nstages; ++s) {
                mbar_init(smem_addr(&bars->full[s]), 1);
                mbar_init(smem_addr(&bars->empty[s]), 1);
            }
            mbar_init(smem_addr(&bars->q_full), 1);
            for (int g = 0; g < 2; ++g) {
                for (int b = 0; b < 2; ++b) {
                    mbar_init(smem_addr(&bars->s_full[g][b]), 1);
                    mbar_init(smem_addr(&bars->s_free[g][b]), 4);
                }
                mbar_init(smem_addr(&bars->p_full[g]), 4);
                mbar_init(smem_addr(&bars->pv_done[g]), 1);
            }
            mbar_init(smem_addr(&bars->mma_done), 1);
            bars->abort_flag = 0;
            mbar_fence_init();
            // Q of each row group: (dim, half, head in group, KV head, sequence), one box per half
            const uint32_t qf = smem_addr(&bars->q_full);
            mbar_arrive_expect_tx(qf, static_cast<uint32_t>(ngrp * C::kHalves * rows * 128));
            const uint64_t q_policy = l2_policy_evict_first();
            for (int g = 0; g < ngrp; ++g)
                for (int h = 0; h < C::kHalves; ++h)
                    tma_load_5d(smem_addr(q_s + (g * C::kHalves + h) * (kTcLanes * 128)), &tmap_q, 0, h, 0, kvh,
                                (grp0 + g) * spg, qf, q_policy);
            policy = l2_policy_evict_last();   // every row group reads the prefix
            preissued = min(1, ntiles);   // the producer loop issues the next ones after the sync
            for (int i = 0; i < preissued; ++i) issue_tile(i);
            bars->issued = preissued;
        }
    } else if (warp == C::kMmaWarp) {
        tmem_alloc(smem_addr(&bars->tmem_base), C::kTmemCols);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == C::kTmaWarp) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            int issued = preissued;
            for (int i = preissued; i < ntiles; ++i) {
                const int s = i % nstages, k = i / nstages;
                if (!tc_wait(p, bars, &bars->empty[s], (k - 1) & 1)) break;
                issue_tile(i);
                issued = i + 1;
            }
            bars->issued = issued;
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_16bit_f32(kTcLanes, kTcTile, false, false, kF16);
            constexpr uint32_t id_pv = idesc_16bit_f32(kTcLanes, D, false, true, kF16);
            const uint32_t q_base = smem_addr(q_s);
            // O += P V for tile i, row group g
            auto issue_pv = [&](int i, int g) -> bool {
                if (!tc_wait(p, bars, &bars->p_full[g], i & 1)) return false;
                tc_fence_after();
                // descriptors of the tile's operands, stepped by constant adds
                const uint64_t vd = smem_desc_sw128(smem_addr(ring + (i % nstages) * C::kStageBytes) + C::kKBytes,
                                                    kTcTile * 128, 1024);
                const uint64_t hd = smem_desc_sw128(smem_addr(p_hi(g)), 16, 1024);
                const uint64_t ld = smem_desc_sw128(smem_addr(p_lo(g)), 16, 1024);
                const uint32_t first = i > 0 ? 1u : 0u;
#pragma unroll
                for (int kk = 0; kk < kTcTile / 16; ++kk) {
                    const uint64_t bdesc = vd + desc_step(kk * 16 * 128);
                    tc_mma_16bit(tmem + C::o_col(g), hd + desc_step(kk * 32), bdesc, id_pv, kk > 0 ? 1u : first);
                    tc_mma_16bit(tmem + C::o_col(g), ld + desc_step(kk * 32), bdesc, id_pv, 1u);
                }
                tc_commit(smem_addr(&bars->pv_done[g]));
                return true;
            };
            auto issue_pv_all = [&](int i) -> bool {
                for (int g = 0; g < ngrp; ++g)
                    if (!issue_pv(i, g)) return false;
                tc_commit(smem_addr(&bars->empty[i % nstages]));   // the stage is free once every P.V read it
                return true;
            };
            bool ok = tc_wait(p, bars, &bars->q_full, 0);
            for (int i = 0; i < ntiles && ok; ++i) {
                const int s = i % nstages, b = i & 1;
                if (!tc_wait(p, bars, &bars->full[s], (i / nstages) & 1)) { ok = false; break; }
                tc_fence_after();
                const uint32_t kbase = smem_addr(ring + s * C::kStageBytes);
                for (int g = 0; g < ngrp && ok; ++g) {
                    if (i >= 2 && !tc_wait(p, bars, &bars->s_free[g][b], ((i >> 1) - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t qd = smem_desc_sw128(q_base + g * C::kQBytes, 16, 1024);
                    const uint64_t kd = smem_desc_sw128(kbase, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int half = kk / 4, off = (kk % 4) * 32;
                        tc_mma_16bit(tmem + C::s_col(g, b), qd + desc_step(half * (kTcLanes * 128) + off),
                                    kd + desc_step(half * (kTcTile * 128) + off), id_qk, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(smem_addr(&bars->s_full[g][b]));
                }
                if (ok && i >= 1) ok = issue_pv_all(i - 1);
            }
            if (ok && ntiles > 0) issue_pv_all(ntiles - 1);
            // every MMA this thread issued has completed once mma_done arrives
            tc_commit(smem_addr(&bars->mma_done));
            if (!mbar_wait(smem_addr(&bars->mma_done), 0)) record_status(p.status, kStatusTimeout);
        }
    } else {
        // ------------------------------ softmax warps ------------------------------
        const int g = warp >> 2;                           // row group
        const int R = (warp & 3) * 32 + lane;              // row = tensor-memory lane
        const int seq = (grp0 + g) * spg + R / p.group;
        const bool live = g < ngrp && R < rows && seq < p.num_seqs;
        int len = live ? p.context_lens[seq] : 0;
        len = min(max(len, 0), p.prefix_tokens);
        const float sl2 = p.scale_log2;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        float m = -1e30f, l = 0.f, t = -INFINITY;     // finite reference max (see the mma.sync pass)
        bool ok = g < ngrp;
        for (int i = 0; i < ntiles && ok; ++i) {
            const int b = i & 1;
            if (!tc_wait(p, bars, &bars->s_full[g][b], (i >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            float s[kTcTile];
            tmem_ld64(tmem + lane_off + C::s_col(g, b), s);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars->s_free[g][b]));
            const int t0 = tok_begin + i * kTcTile;
            const int valid = min(kTcTile, max(0, len - t0));
            // Tokens past a live row's length only occur when the shared blocks
            // are shorter than a context (outside the contract): masked then.
            // Rows past the batch read a zero Q, so their scores are finite;
            // their outputs are never stored. The largest scaled score is the
            // scale times the largest raw score (the smallest, for a negative
            // scale); masked scores scale to -inf.
            const bool up = sl2 >= 0.f;
            if (__any_sync(0xffffffffu, live && valid < kTcTile)) {
#pragma unroll
                for (int j = 0; j < kTcTile; ++j) s[j] = j < valid ? s[j] : up ? -INFINITY : INFINITY;
            }
            // (eight partial maxima and four partial sums: short dependency chains)
            float mx8[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) mx8[j] = s[j];
            if (up) {
#pragma unroll
                for (int j = 8; j < kTcTile; ++j) mx8[j & 7] = fmaxf(mx8[j & 7], s[j]);
            } else {
#pragma unroll
                for (int j = 8; j < kTcTile; ++j) mx8[j & 7] = fminf(mx8[j & 7], s[j]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) mx8[j] = up ? fmaxf(mx8[j], mx8[j + 4]) : fminf(mx8[j], mx8[j + 4]);
            const float e01 = up ? fmaxf(mx8[0], mx8[1]) : fminf(mx8[0], mx8[1]);
            const float e23 = up ? fmaxf(mx8[2], mx8[3]) : fminf(mx8[2], mx8[3]);
            const float mx = sl2 * (up ? fmaxf(e01, e23) : fminf(e01, e23));
            t = fmaxf(t, mx);
            const bool need = mx > m + kTcSlack;
            const float m_new = need ? fmaxf(m, mx) : m;
            const float alpha = fast_exp2(m - m_new);
            m = m_new;
            l *= alpha;
            // P in registers first, in the type of V (high part and residual):
            // this overlaps the previous tile's P.V, which still reads the buffer
            uint32_t hi[kTcTile / 2], lo[kTcTile / 2];
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < kTcTile / 2; ++e) {   // 2^(s * scale - m): one fma and one ex2
                const float p0 = fast_exp2(fmaf(s[2 * e], sl2, -m)), p1 = fast_exp2(fmaf(s[2 * e + 1], sl2, -m));
                l4[e & 3] += p0 + p1;
                split_x2<kF16>(p0, p1, hi[e], lo[e]);
            }
            l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
            if (i >= 1) {
                // the previous tile's P.V has read the P buffer and landed in O
                if (!tc_wait(p, bars, &bars->pv_done[g], (i - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (__any_sync(0xffffffffu, need)) {   // rescale O
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        float o[32];
                        tmem_ld32(tmem + lane_off + C::o_col(g) + c, o);
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] *= alpha;
                        tmem_st32(tmem + lane_off + C::o_col(g) + c, o);
                    }
                }
            }
            unsigned char *hi_b = p_hi(g), *lo_b = p_lo(g);
#pragma unroll
            for (int c = 0; c < 8; ++c) {   // 8 tokens per 16-byte chunk, at chunk c ^ (row % 8)
                const int pos = R * 128 + ((c ^ (R & 7)) << 4);
                *reinterpret_cast<uint4 *>(hi_b + pos) = make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
                *reinterpret_cast<uint4 *>(lo_b + pos) = make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars->p_full[g]));
        }
        // ---- epilogue: O / l in split form at partition `chunk` ----
        // every row group's last P.V done: P buffers and ring are free for staging
        if (ok && ntiles > 0 && !tc_wait(p, bars, &bars->pv_done[g], (ntiles - 1) & 1)) ok = false;
        softmax_warps_sync(32 * C::kSoftmaxWarps);
        tc_fence_after();
        if (g < ngrp && !*reinterpret_cast<volatile int *>(&bars->abort_flag)) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            unsigned char *box0 = stage_out + g * C::kOutBytes + R * 128;
#pragma unroll
            for (int c = 0; c < D; c += 64) {
                float o[64];
                if (ntiles > 0) {
                    tmem_ld64(tmem + lane_off + C::o_col(g) + c, o);
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) o[j] = 0.f;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {   // two boxes of 32 columns
                    unsigned char *row = box0 + ((c + 32 * h) / kTcOutCols) * C::kOutBoxBytes;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {   // 16-byte chunk j of the row at chunk j ^ (row % 8)
                        const float *q = o + 32 * h + 4 * j;
                        *reinterpret_cast<float4 *>(row + ((j ^ (R & 7)) << 4)) =
                            make_float4(q[0] * inv, q[1] * inv, q[2] * inv, q[3] * inv);
                    }
                }
            }
            if (live) {
                const int64_t prow = (static_cast<int64_t>(seq) * p.num_heads + kvh * p.group + R % p.group) *
                                         p.part_stride + chunk;
                p.max_logits[prow] = l > 0.f ? t * kLn2 : -INFINITY;
                p.exp_sums[prow] = l > 0.f ? l * fast_exp2(m - t) : 0.f;
            }
            fence_proxy_async_smem();
        }
        softmax_warps_sync(32 * C::kSoftmaxWarps);
        if (threadIdx.x == 0 && !*reinterpret_cast<volatile int *>(&bars->abort_flag)) {
            // (dim, partition, query head, sequence): rows past the batch are not written
            for (int gg = 0; gg < ngrp; ++gg)
                for (int c = 0; c < D / kTcOutCols; ++c)
                    tma_store_4d(&tmap_o, smem_addr(stage_out + gg * C::kOutBytes + c * C::kOutBoxBytes),
                                 c * kTcOutCols, chunk, kvh * p.group, (grp0 + gg) * spg);
            bulk_commit_and_wait_read();
        }
    }

    // ---- drain: copies still landing, then free the tensor memory ----
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait(smem_addr(&bars->q_full), 0)) record_status(p.status, kStatusTimeout);
        const int issued = bars->issued;
        for (int s = 0; s < nstages && s < issued; ++s) {
            const int k_last = (issued - 1 - s) / nstages;
            if (!mbar_wait(smem_addr(&bars->full[s]), k_last & 1)) record_status(p.status, kStatusTimeout);
        }
    }
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if (p.pair_role == kPairSecond) grid_dependency_wait();   // this grid completes after the first
}

template <int D, int kGroups, bool kF16>
cudaError_t launch_tc_impl(const PrefixParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                           const CUtensorMap &tq, const CUtensorMap &to, dim3 grid, cudaStream_t stream) {
    using C = TcCfg<D, kGroups>;
    if (p.ring_bytes < C::min_ring_bytes() || p.ring_bytes > C::max_ring_bytes() || p.ring_bytes % C::kStageBytes)
        return cudaErrorInvalidValue;
    auto kern = prefix_tc_kernel<D, kGroups, kF16>;
    static unsigned long long done = 0;
    cudaError_t e = ensure_smem_limit(kern, C::smem_bytes(C::max_ring_bytes()), done);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, dim3(C::kThreads), C::smem_bytes(p.ring_bytes), stream, 1u, tk, tv, tq, to, p);
}

template <int D, bool kF16>
cudaError_t launch_tc_dim(const PrefixParams &p, int groups_per_cta, const CUtensorMap &tk, const CUtensorMap &tv,
                          const CUtensorMap &tq, const CUtensorMap &to, dim3 grid, cudaStream_t stream) {
    return groups_per_cta == 2 ? launch_tc_impl<D, 2, kF16>(p, tk, tv, tq, to, grid, stream)
                               : launch_tc_impl<D, 1, kF16>(p, tk, tv, tq, to, grid, stream);
}

}  // namespace

int prefix_tc_max_rows() { return kTcLanes; }
int prefix_tc_tile_tokens() { return kTcTile; }
int prefix_tc_stage_bytes(int head_dim) { return 2 * (head_dim / 64) * kTcTile * 128; }
int prefix_tc_out_cols() { return kTcOutCols; }

template <int D, int kGroups>
int ring_for(int budget_bytes) {
    using C = TcCfg<D, kGroups>;
    int ring = budget_bytes / C::kStageBytes * C::kStageBytes;
    if (ring > C::max_ring_bytes()) ring = C::max_ring_bytes();
    if (ring < C::min_ring_bytes()) ring = (C::min_ring_bytes() + C::kStageBytes - 1) / C::kStageBytes * C::kStageBytes;
    return ring;
}

int prefix_tc_ring_bytes(int head_dim, int groups_per_cta, int budget_bytes) {
    if (head_dim == 128) return groups_per_cta == 2 ? ring_for<128, 2>(budget_bytes) : ring_for<128, 1>(budget_bytes);
    return groups_per_cta == 2 ? ring_for<64, 2>(budget_bytes) : ring_for<64, 1>(budget_bytes);
}

cudaError_t launch_prefix_tc(const PrefixParams &p, int groups_per_cta, const CUtensorMap &tk,
                             const CUtensorMap &tv, const CUtensorMap &tq, const CUtensorMap &to, dim3 grid,
                             cudaStream_t stream) {
    if (p.head_dim == 128)
        return p.kv_f16 ? launch_tc_dim<128, true>(p, groups_per_cta, tk, tv, tq, to, grid, stream)
                        : launch_tc_dim<128, false>(p, groups_per_cta, tk, tv, tq, to, grid, stream);
    if (p.head_dim == 64)
        return p.kv_f16 ? launch_tc_dim<64, true>(p, groups_per_cta, tk, tv, tq, to, grid, stream)
                        : launch_tc_dim<64, false>(p, groups_per_cta, tk, tv, tq, to, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
