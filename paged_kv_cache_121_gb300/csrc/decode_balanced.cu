// Paged decode attention with the work of a ragged batch balanced across
// CTAs, bf16 or fp16 K/V, tensor cores, sm_103a.
//
// What it computes: the same softmax(scale * q_h K^T) V per (sequence, query
// head) as the per-partition kernel ("What Does PagedAttention Actually
// Optimize?", section 8; "PagedAttention, explained.", procedure step 5).
//
// How it divides the work. For one (KV-head group, head tile), the batch's
// 16-token tiles are laid end to end, sequence after sequence: W tiles in
// all, sequence b owning tiles [P[b], P[b+1]) with P the prefix sums of
// cdiv(len, 16) computed on the device from the context lengths. CTA c of
// C (C at most W) takes tiles [c W / C, (c+1) W / C): every CTA gets the same number of
// tiles however ragged the lengths, with no length on the host. A CTA walks
// its range as segments, one per sequence it touches. A segment that holds
// a whole sequence writes the final output; a piece of a sequence split
// between CTAs goes to workspace row (c + b) * Hq + h (c + b grows by at
// least one from one piece to the next in tile order, so rows never
// collide), and the merge kernel combines the pieces by log-sum-exp.
//
// The pipeline inside a CTA is the per-partition kernel's: a producer warp
// loads one 5-D TMA box of K and one of V per tile into an mbarrier ring
// (blocks of 16 tokens or more), one consumer warp per KV head runs the
// tile step of mma_tile.cuh, every wait is bounded.
#include "device_common.cuh"
#include "internal.h"
#include "mma_tile.cuh"

namespace pa {
namespace {

constexpr int kTT = 16;           // tokens per tile
constexpr int kMaxHeads = 8;      // consumer warps
constexpr int kMaxStages = 32;
constexpr int kMaxRingBytes = 200 * 1024;
constexpr size_t kBarrierBytes = 2 * kMaxStages * sizeof(uint64_t);

size_t smem_bytes(int ring, int num_seqs) {
    return 1024 + static_cast<size_t>(ring) + kBarrierBytes + static_cast<size_t>(num_seqs + 1) * sizeof(int);
}

// Tokens of sequence b that are attended (clamped like the per-partition
// kernel: to the table's reach and to the host bound).
__device__ __forceinline__ int attended_len(const DecodeParams &p, const BalancedParams &bp, int b) {
    int len = p.context_lens[b];
    if (len < 0) len = 0;
    const int cap = min(p.max_blocks * p.block_size, bp.len_cap);
    return min(len, cap);
}

// P[b] = tiles of sequences 0 .. b-1 for b = 0 .. B (P[B] = W). All threads
// of the CTA take part; `scratch` holds one int per warp.
__device__ void tile_prefix(const DecodeParams &p, const BalancedParams &bp, int *P, int *scratch) {
    const int B = p.num_seqs, nt = blockDim.x;
    const int per = (B + nt - 1) / nt;
    const int b0 = static_cast<int>(threadIdx.x) * per;
    int sum = 0;
    for (int j = 0; j < per; ++j)
        if (b0 + j < B) sum += (attended_len(p, bp, b0 + j) + kTT - 1) / kTT;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += scratch[w];
    for (int j = 0; j < per; ++j)
        if (b0 + j < B) {
            P[b0 + j] = run;
            run += (attended_len(p, bp, b0 + j) + kTT - 1) / kTT;
        }
    if (threadIdx.x == static_cast<unsigned>(nt - 1)) P[B] = run;   // the last thread's running sum is W
    __syncthreads();
}

// The sequence owning tile g (0 <= g < P[B]): the largest b with P[b] <= g,
// which skips empty sequences.
__device__ __forceinline__ int seq_of(const int *P, int B, int g) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P[mid] <= g) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The CTA whose range holds tile t: ranges start at floor(c W / C).
__device__ __forceinline__ int cta_of(int t, int W, int C) {
    return static_cast<int>((static_cast<int64_t>(t + 1) * C - 1) / W);
}

// The step's new token of sequence b (position pos, in block blk: the block
// of the tile being loaded) for heads head0 .. head0+hpc-1, K and V, copied
// by one warp into its slot, then fenced against the async proxy so that the
// TMA reads of the tile that follow see it ("PagedAttention, explained.",
// procedure step 4). The block id comes from the producer's lookup and both
// rows are loaded before either is stored: one round trip to memory instead
// of a table read and a row read for each of K and V, in the middle of the
// pipeline.
template <int D>
__device__ __forceinline__ void append_kv(const DecodeParams &p, int blk, int b, int pos, int head0, int hpc,
                                          int lane) {
    constexpr int kPer = kMaxHeads * D / 8 / 32;   // 16-byte pieces per lane and row, at most
    const int n = hpc * D / 8;
    if (static_cast<unsigned>(blk) < static_cast<unsigned>(p.num_blocks)) {
        const int64_t src_off = (static_cast<int64_t>(b) * p.num_kv_heads + head0) * D;
        const int64_t slot = static_cast<int64_t>(blk) * p.block_size + pos % p.block_size;
        const int64_t dst_off = (slot * p.num_kv_heads + head0) * D;
        const uint4 *ks = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.append_key) + src_off);
        const uint4 *vs = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.append_value) + src_off);
        uint4 *kd = reinterpret_cast<uint4 *>(const_cast<uint16_t *>(static_cast<const uint16_t *>(p.k_cache)) + dst_off);
        uint4 *vd = reinterpret_cast<uint4 *>(const_cast<uint16_t *>(static_cast<const uint16_t *>(p.v_cache)) + dst_off);
        uint4 kr[kPer], vr[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int c = lane + 32 * j;
            if (c < n) {
                kr[j] = ks[c];
                vr[j] = vs[c];
            }
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int c = lane + 32 * j;
            if (c < n) {
                kd[c] = kr[j];
                vd[c] = vr[j];
            }
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
}

__device__ __forceinline__ void prefetch_l1(const void *ptr) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ void store_pair(const DecodeParams &p, int64_t idx, float a, float c) {
    store_pair_as(p.out, out_type_of(p), idx, a, c);
}

// A finished segment of sequence b for query heads h0 .. h0+rows-1: the
// final output (whole sequence), or a piece in workspace row (c + b) * Hq + h.
template <int D>
__device__ __forceinline__ void segment_epilogue(const DecodeParams &p, const WarpState<D> &st, int b, int c,
                                                 bool whole, int h0, int rows, int lane) {
    const int r = lane >> 2, q4 = lane & 3;
    const bool v0 = r < rows, v1 = r + 8 < rows;
    const float i0 = st.l0 > 0.f ? 1.f / st.l0 : 0.f, i1 = st.l1 > 0.f ? 1.f / st.l1 : 0.f;
    if (whole) {
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            const int d = 8 * dn + 2 * q4;
            if (v0) store_pair(p, (static_cast<int64_t>(b) * p.num_heads + h0 + r) * D + d,
                               st.o[dn][0] * i0, st.o[dn][1] * i0);
            if (v1) store_pair(p, (static_cast<int64_t>(b) * p.num_heads + h0 + r + 8) * D + d,
                               st.o[dn][2] * i1, st.o[dn][3] * i1);
        }
        return;
    }
    const int64_t row0 = static_cast<int64_t>(c + b) * p.num_heads + h0 + r;
    const int64_t row1 = row0 + 8;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
        const int d = 8 * dn + 2 * q4;
        if (v0) *reinterpret_cast<float2 *>(p.tmp_out + row0 * D + d) = make_float2(st.o[dn][0] * i0, st.o[dn][1] * i0);
        if (v1) *reinterpret_cast<float2 *>(p.tmp_out + row1 * D + d) = make_float2(st.o[dn][2] * i1, st.o[dn][3] * i1);
    }
    if (q4 == 0) {   // natural-log max and the sum relative to it
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

template <int D, bool kF16>
__global__ void __launch_bounds__(32 * (kMaxHeads + 1), 1)
decode_balanced_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                       const __grid_constant__ DecodeParams p, const __grid_constant__ BalancedParams bp) {
    constexpr int kHalves = D / 64;
    constexpr int kHalfStride = kTT * 128;               // one 64-dim half of one head's tile
    constexpr int kHeadStride = kHalves * kHalfStride;   // one head's K (or V) rows of a tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.ring_bytes);
    int *P = reinterpret_cast<int *>(bars + 2 * kMaxStages);
    __shared__ int s_scratch[32];
    __shared__ int s_abort;
    __shared__ int s_issued;

    const int hpc = p.heads_per_cta;
    const int c = blockIdx.x, B = p.num_seqs;
    const int hgrp = blockIdx.y / p.ntile;
    const int tile = blockIdx.y % p.ntile;
    const int rows = min(kRowsPerTile, p.group - tile * kRowsPerTile);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dependency_wait();   // the previous kernel on the stream (e.g. the scatter) is complete

    tile_prefix(p, bp, P, s_scratch);
    const int W = P[B];
    if (c == 0 && blockIdx.y == 0)   // for the merge kernel
        for (int i = threadIdx.x; i <= B; i += blockDim.x) bp.prefix[i] = P[i];
    const int C = min(bp.ctas, W);   // at most one CTA per tile: no range is empty
    if (c >= C) return;
    const int start = static_cast<int>(static_cast<int64_t>(c) * W / C);
    const int end = static_cast<int>(static_cast<int64_t>(c + 1) * W / C);
    if (start >= end) return;
    const int ntiles = end - start;
    const int bs = p.block_size;   // >= 16: a tile lies inside one block

    const int stage_bytes = 2 * hpc * kTT * D * 2;
    int nstages = p.ring_bytes / stage_bytes;
    if (nstages > kMaxStages) nstages = kMaxStages;
    const int v_off = stage_bytes / 2;
    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(smem_addr(&bars[s]), 1);
            mbar_init(smem_addr(&bars[kMaxStages + s]), hpc);
        }
        s_abort = 0;
        s_issued = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == hpc) {
        // ------------------------------ producer ------------------------------
        // Lane l holds the block id and the in-block token offset of tile
        // start + 32 k + l for the current chunk k, the next chunk fetched
        // ahead, and (when the step's new tokens are written here) the
        // sequence whose last tile it is, else -1. Tiles past the range are
        // not looked up.
        uint64_t policy = 0;
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
            policy = l2_policy_evict_first();
        }
        auto lookup = [&](int i, int &blk, int &off, int &last_of) {
            blk = 0;
            off = 0;
            last_of = -1;
            if (i < ntiles) {
                const int g = start + i;
                const int b = seq_of(P, B, g);
                const int tok = (g - P[b]) * kTT;
                blk = p.block_tables[static_cast<int64_t>(b) * p.max_blocks + tok / bs];
                off = tok % bs;
                if (p.append_key && g == P[b + 1] - 1 && p.context_lens[b] == attended_len(p, bp, b))
                    last_of = b;   // a length cut short writes none
            }
        };
        const int head0 = hgrp * hpc;
        int cur_blk, cur_off, cur_last, nxt_blk, nxt_off, nxt_last;
        lookup(lane, cur_blk, cur_off, cur_last);
        lookup(32 + lane, nxt_blk, nxt_off, nxt_last);
        int issued = 0;
        for (int i = 0; i < ntiles; ++i) {
            if ((i & 31) == 0 && i > 0) {
                cur_blk = nxt_blk;
                cur_off = nxt_off;
                cur_last = nxt_last;
                lookup(i + 32 + lane, nxt_blk, nxt_off, nxt_last);
            }
            const int blk = __shfl_sync(0xffffffffu, cur_blk, i & 31);
            const int off = __shfl_sync(0xffffffffu, cur_off, i & 31);
            const int last_of = __shfl_sync(0xffffffffu, cur_last, i & 31);
            if (last_of >= 0)   // the tile holds a sequence's new token: store it before reading the tile
                append_kv<D>(p, blk, last_of, attended_len(p, bp, last_of) - 1, head0, hpc, lane);
            int ok = 1;
            if (lane == 0) {
                const int s = i % nstages, k = i / nstages;
                if (k > 0) {
                    if (*reinterpret_cast<volatile int *>(&s_abort)) {
                        ok = 0;
                    } else if (!mbar_wait(smem_addr(&bars[kMaxStages + s]), (k - 1) & 1)) {
                        record_status(p.status, kStatusTimeout);
                        s_abort = 1;
                        ok = 0;
                    }
                }
                if (ok) {
                    const uint32_t full = smem_addr(&bars[s]);
                    mbar_arrive_expect_tx(full, static_cast<uint32_t>(stage_bytes));
                    const uint32_t kdst = smem_addr(smem + s * stage_bytes);
                    // (dim, token, half, head, block), innermost first
                    tma_load_5d(kdst, &tmap_k, 0, off, 0, head0, blk, full, policy);
                    tma_load_5d(kdst + v_off, &tmap_v, 0, off, 0, head0, blk, full, policy);
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
        const float sl2 = p.scale_log2;
        auto tok_off = [](int t) -> int { return t * 128; };
        WarpState<D> st;
        uint32_t qa[D / 16][4];
        int b = seq_of(P, B, start);
        int len = 0, seg_end = 0;
        bool open = false;
        for (int i = 0; i < ntiles; ++i) {
            if (*reinterpret_cast<volatile int *>(&s_abort)) break;
            const int g = start + i;
            if (!open || g >= seg_end) {
                if (open) {   // the previous sequence's segment is done
                    st.reduce_sums();
                    segment_epilogue<D>(p, st, b, c, P[b] >= start && seg_end <= end, h0, rows, lane);
                    ++b;
                }
                while (P[b + 1] <= g) ++b;   // skip empty sequences
                len = attended_len(p, bp, b);
                seg_end = P[b + 1];
                const uint16_t *qb = static_cast<const uint16_t *>(p.query);
                const uint32_t *q0 = reinterpret_cast<const uint32_t *>(
                    qb + (static_cast<int64_t>(b) * p.num_heads + h0 + r) * D);
                load_query_fragments<D>(qa, q0, q0 + 8 * (D / 2), r < rows, r + 8 < rows, lane);
                st.init();
                open = true;
                // the next sequence of this range: its query rows into L1 now,
                // so that the switch does not wait on HBM
                int nb = b + 1;
                while (nb < B && P[nb + 1] == P[nb]) ++nb;
                if (nb < B && P[nb] < end) {
                    const uint16_t *n0 = qb + (static_cast<int64_t>(nb) * p.num_heads + h0 + r) * D;
#pragma unroll
                    for (int x = 0; x < D * 2; x += 128) {
                        if (r < rows) prefetch_l1(reinterpret_cast<const char *>(n0) + x);
                        if (r + 8 < rows) prefetch_l1(reinterpret_cast<const char *>(n0 + 8 * D) + x);
                    }
                }
            }
            const int s = i % nstages, k = i / nstages;
            if (!mbar_wait(smem_addr(&bars[s]), k & 1)) {
                record_status(p.status, kStatusTimeout);
                s_abort = 1;
                break;
            }
            unsigned char *kst = smem + s * stage_bytes + warp * kHeadStride;   // this head
            const uint32_t kbase = smem_addr(kst);
            const int valid = min(kTT, len - (g - P[b]) * kTT);
            if (valid < kTT) {
                // zero this head's V rows past the context (whole 128-byte rows)
                for (int e = lane; e < kHalves * kTT * 8; e += 32) {
                    const int hh = e / (kTT * 8), row = (e % (kTT * 8)) / 8;
                    if (row >= valid)
                        *reinterpret_cast<uint4 *>(kst + v_off + hh * kHalfStride + row * 128 + (e % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            warp_tile_attention<D, kTT, true, kF16>(st, qa, kbase, kbase + v_off, kHalfStride, tok_off, valid, valid,
                                                    sl2, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars[kMaxStages + s]));
        }
        if (open) {
            st.reduce_sums();
            segment_epilogue<D>(p, st, b, c, P[b] >= start && seg_end <= end, h0, rows, lane);
        }
    }

    grid_dependents_launch();   // the merge kernel may be scheduled; it waits for this grid's memory
    // Drain: wait (bounded) for the last phase of every stage this CTA armed.
    __syncthreads();
    if (threadIdx.x == 0) {
        const int issued = s_issued;
        for (int s = 0; s < nstages && s < issued; ++s) {
            const int k_last = (issued - 1 - s) / nstages;
            if (!mbar_wait(smem_addr(&bars[s]), k_last & 1)) record_status(p.status, kStatusTimeout);
        }
    }
}

// Merge the pieces of each sequence that was split between CTAs: one warp
// per (sequence, query head), D / 32 dims per lane. Pieces are normalised
// partial outputs with their natural-log max and the sum relative to it.
// A sequence held whole by one CTA was written by the decode kernel and is
// skipped; an empty one gets zeros.
template <int D>
__global__ void __launch_bounds__(128) balanced_merge_kernel(const __grid_constant__ DecodeParams p,
                                                             const __grid_constant__ BalancedParams bp) {
    constexpr int E = D / 32;
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * 4 + warp;
    grid_dependency_wait();   // the decode kernel's pieces and prefix sums are complete
    if (h >= p.num_heads) return;
    const int B = p.num_seqs;
    const int pb = bp.prefix[b], pe = bp.prefix[b + 1], W = bp.prefix[B];
    const int C = min(bp.ctas, W);   // as the decode kernel cut the ranges
    const int64_t o = (static_cast<int64_t>(b) * p.num_heads + h) * D + lane * E;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    if (pe > pb) {
        const int c0 = cta_of(pb, W, C), c1 = cta_of(pe - 1, W, C);
        if (c0 == c1) return;
        // pieces four at a time, every load of a group issued before any use;
        // the running max moves between groups with a rescale
        float M = -INFINITY, L = 0.f;
        for (int base = c0; base <= c1; base += 4) {
            float m[4], l[4], ov[4][E];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                l[j] = 0.f;
                m[j] = -INFINITY;
                if (base + j <= c1) {
                    const int64_t row = static_cast<int64_t>(base + j + b) * p.num_heads + h;
                    m[j] = __ldcg(p.max_logits + row);
                    l[j] = __ldcg(p.exp_sums + row);
                    const float *src = p.tmp_out + row * D + lane * E;
#pragma unroll
                    for (int e = 0; e < E; ++e) ov[j][e] = __ldcg(src + e);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) ov[j][e] = 0.f;
                }
            }
            float Mc = M;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (l[j] > 0.f) Mc = fmaxf(Mc, m[j]);
            if (Mc > M) {
                const float sc = fast_exp2((M - Mc) * kLog2e);
                L *= sc;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] *= sc;
                M = Mc;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (l[j] > 0.f) {
                    const float w = l[j] * fast_exp2((m[j] - M) * kLog2e);
                    L += w;
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[e] += w * ov[j][e];
                }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] *= inv;
    }
#pragma unroll
    for (int e = 0; e < E; e += 2) store_pair(p, o + e, acc[e], acc[e + 1]);
}

template <int D, bool kF16>
cudaError_t launch_balanced_dim(const DecodeParams &p, const BalancedParams &bp, const CUtensorMap &tk,
                                const CUtensorMap &tv, dim3 grid, cudaStream_t stream) {
    auto kern = decode_balanced_kernel<D, kF16>;
    static unsigned long long done = 0;
    cudaError_t e = ensure_smem_limit(kern, smem_bytes(kMaxRingBytes, kBalancedMaxSeqs), done);
    if (e != cudaSuccess) return e;
    const dim3 block(32 * (p.heads_per_cta + 1));
    return launch_kernel(kern, grid, block, smem_bytes(p.ring_bytes, p.num_seqs), stream, 1u, tk, tv, p, bp);
}

}  // namespace

bool decode_balanced_supported(int head_dim, int block_size) {
    return (head_dim == 64 || head_dim == 128) && block_size >= kTT && block_size <= 256 &&
           (block_size & (block_size - 1)) == 0;
}

size_t decode_balanced_smem_extra(int num_seqs) { return static_cast<size_t>(num_seqs + 1) * sizeof(int); }

cudaError_t launch_decode_balanced(const DecodeParams &p, const BalancedParams &bp, const CUtensorMap &tk,
                                   const CUtensorMap &tv, dim3 grid, cudaStream_t stream) {
    if (p.num_seqs < 1 || p.num_seqs > kBalancedMaxSeqs || p.ring_bytes > kMaxRingBytes || bp.ctas < 1 ||
        p.heads_per_cta < 1 || p.heads_per_cta > kMaxHeads)
        return cudaErrorInvalidValue;
    if (p.head_dim == 128)
        return p.kv_f16 ? launch_balanced_dim<128, true>(p, bp, tk, tv, grid, stream)
                        : launch_balanced_dim<128, false>(p, bp, tk, tv, grid, stream);
    if (p.head_dim == 64)
        return p.kv_f16 ? launch_balanced_dim<64, true>(p, bp, tk, tv, grid, stream)
                        : launch_balanced_dim<64, false>(p, bp, tk, tv, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_balanced_merge(const DecodeParams &p, const BalancedParams &bp, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(p.num_seqs), static_cast<unsigned>((p.num_heads + 3) / 4));
    if (p.head_dim == 128) return launch_kernel(balanced_merge_kernel<128>, grid, dim3(128), 0, stream, 1u, p, bp);
    if (p.head_dim == 64) return launch_kernel(balanced_merge_kernel<64>, grid, dim3(128), 0, stream, 1u, p, bp);
    return cudaErrorInvalidValue;
}

}  // namespace pa
