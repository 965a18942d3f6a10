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
// Why tcgen05 here: with 128 query rows per KV head against the same K/V,
// the prefix is a real matrix product (M = 128 rows, N = 64 tokens per tile,
// K = head_dim for Q.K^T; M = 128, N = head_dim, K = 64 tokens for P.V),
// unlike per-sequence decode where M is one GQA group.
//
// How. One CTA = one KV head x one chunk of the prefix x 128 query rows.
//  * Warps 0-3 (128 threads, thread i = row i = TMEM lane i) load Q into
//    shared memory (K-major, 128-byte swizzle), then per 64-token tile read
//    their row of S from tensor memory, run the base-2 online softmax in
//    registers (a row per thread: no shuffles), rescale their row of O in
//    tensor memory when the running max moves by more than 8 (rare), and
//    write P as a 16-bit high part and a residual into one of two shared
//    buffers (tile i + 1's softmax does not wait for tile i's P.V).
//  * Warp 4 streams the tiles' K and V with TMA (one box per block, 64-dim
//    half and cache) into a ring of stages guarded by mbarriers; it fills
//    the ring while the other warps load Q and allocate tensor memory.
//  * Warp 5 owns the tensor memory (S double-buffered: 2 x 64 columns; O:
//    head_dim columns) and one of its threads issues the MMAs: S = Q K^T as
//    head_dim / 16 K-steps, then O += P_hi V + P_lo V (V read MN-major) as
//    4 + 4 K-steps, with tcgen05.commit arriving on the mbarriers that
//    release S to the softmax warps, the P buffer and the ring stage.
// Every wait is bounded; on expiry the kernel records a timeout, waits for
// its own MMAs and copies (bounded), frees its tensor memory and returns.
#include "device_common.cuh"
#include "internal.h"
#include "mma_tile.cuh"
#include "tcgen05.cuh"

namespace pa {

namespace {

constexpr int kTcRows = 128;             // query rows per CTA (MMA M)
constexpr int kTcTile = 64;              // tokens per tile (MMA N of Q.K^T, K of P.V)
constexpr int kTcThreads = 192;          // 4 softmax warps, 1 TMA warp, 1 MMA warp
constexpr int kTcMaxStages = 8;
constexpr int kTcMaxChunkBlocks = kTcChunkBlocks;   // block ids of one chunk, staged in shared memory
constexpr float kTcSlack = 8.f;          // base-2 headroom before the running max moves

template <int D>
struct TcCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kQBytes = kHalves * kTcRows * 128;      // Q, K-major per half
    static constexpr int kPBytes = kTcRows * 128;                // one P buffer (hi or lo)
    static constexpr int kKBytes = kHalves * kTcTile * 128;      // one tile's K (or V)
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kTmemCols = 256;                        // S: 2 x 64, O: D (<= 128)
    static constexpr int kSCol0 = 0, kOCol = 128;
    static size_t smem_bytes(int ring) {
        return 1024 + kQBytes + 4 * kPBytes + static_cast<size_t>(ring) + sizeof(int) * kTcMaxChunkBlocks + 256;
    }
};

struct TcBars {
    uint64_t full[kTcMaxStages];
    uint64_t empty[kTcMaxStages];
    uint64_t s_full[2], s_free[2];   // S buffers: written by Q.K^T, read by the softmax warps
    uint64_t p_full[2], pv_done[2];  // P buffers: written by the softmax warps, read by P.V
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int issued;
    int blk[kTcMaxChunkBlocks];   // the chunk's block ids
};

__device__ __forceinline__ bool tc_wait(const PrefixParams &p, TcBars *bars, uint64_t *bar, uint32_t parity) {
    if (*reinterpret_cast<volatile int *>(&bars->abort_flag)) return false;
    if (mbar_wait(smem_addr(bar), parity)) return true;
    record_status(p.status, kStatusTimeout);
    bars->abort_flag = 1;
    return false;
}

template <int D, bool kF16>
__global__ void __launch_bounds__(kTcThreads, 1)
prefix_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const __grid_constant__ PrefixParams p) {
    using C = TcCfg<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *q_s = smem;
    unsigned char *pbuf = q_s + C::kQBytes;          // [buffer 0..1][hi, lo]
    unsigned char *ring = pbuf + 4 * C::kPBytes;
    TcBars *bars = reinterpret_cast<TcBars *>(ring + p.ring_bytes);
    auto p_hi = [&](int b) { return pbuf + (2 * b) * C::kPBytes; };
    auto p_lo = [&](int b) { return pbuf + (2 * b + 1) * C::kPBytes; };

    grid_dependency_wait();
    const int chunk = blockIdx.x, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tok_begin = chunk * p.chunk_tokens;
    const int tok_end = min(p.prefix_tokens, tok_begin + p.chunk_tokens);
    const int ntiles = tok_end > tok_begin ? (tok_end - tok_begin) / kTcTile : 0;   // whole tiles
    int nstages = p.ring_bytes / C::kStageBytes;
    if (nstages > kTcMaxStages) nstages = kTcMaxStages;
    const int nrows = p.num_seqs * p.group;
    const int row = threadIdx.x;                         // softmax threads: 0..127
    const int R = blockIdx.z * kTcRows + row;
    const int bs = p.block_size;
    const int R_box = bs < kTcTile ? bs : kTcTile;      // tokens per TMA box
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
                tma_load_5d(kdst + o, &tmap_k, 0, off, h, g, blk, full, policy);
                tma_load_5d(vdst + o, &tmap_v, 0, off, h, g, blk, full, policy);
            }
        }
    };

    // ---- setup, overlapped: the producer starts the first tiles while the
    // softmax warps load Q and warp 5 allocates tensor memory ----
    int preissued = 0;
    if (warp == 4) {
        const int nblk = tok_end > tok_begin ? (tok_end - 1) / bs - first + 1 : 0;   // <= kTcMaxChunkBlocks
        for (int e = lane; e < nblk; e += 32) bars->blk[e] = p.prefix_table[first + e];
        __syncwarp();
        if (lane == 0) {
            for (int s = 0; s < nstages; ++s) {
                mbar_init(smem_addr(&bars->full[s]), 1);
                mbar_init(smem_addr(&bars->empty[s]), 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_addr(&bars->s_full[b]), 1);
                mbar_init(smem_addr(&bars->s_free[b]), 4);
                mbar_init(smem_addr(&bars->p_full[b]), 4);
                mbar_init(smem_addr(&bars->pv_done[b]), 1);
            }
            mbar_init(smem_addr(&bars->mma_done), 1);
            bars->abort_flag = 0;
            mbar_fence_init();
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
            policy = l2_policy_evict_last();   // every row group reads the prefix
            preissued = min(nstages, ntiles);
            for (int i = 0; i < preissued; ++i) issue_tile(i);
            bars->issued = preissued;
        }
    } else if (warp < 4) {
        // Q rows into shared memory (K-major, 128-byte swizzle)
        const bool live = R < nrows;
        const int b = live ? R / p.group : 0;
        const int hq = g * p.group + (live ? R % p.group : 0);
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.query) +
                                                           (static_cast<int64_t>(b) * p.num_heads + hq) * D);
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 v = live ? src[h * 8 + j] : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(q_s + h * (kTcRows * 128) + row * 128 + ((j ^ (row & 7)) << 4)) = v;
            }
        fence_proxy_async_smem();
    } else {
        tmem_alloc(smem_addr(&bars->tmem_base), C::kTmemCols);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 4) {
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
    } else if (warp == 5) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_16bit_f32(kTcRows, kTcTile, false, false, kF16);
            constexpr uint32_t id_pv = idesc_16bit_f32(kTcRows, D, false, true, kF16);
            const uint32_t q_base = smem_addr(q_s);
            auto issue_pv = [&](int i) -> bool {   // O += P V for tile i (P buffer i % 2)
                const int pb = i & 1;
                if (!tc_wait(p, bars, &bars->p_full[pb], (i >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t vbase = smem_addr(ring + (i % nstages) * C::kStageBytes) + C::kKBytes;
                const uint32_t hi = smem_addr(p_hi(pb)), lo = smem_addr(p_lo(pb));
#pragma unroll
                for (int kk = 0; kk < kTcTile / 16; ++kk) {
                    const uint64_t bdesc = smem_desc_sw128(vbase + kk * 16 * 128, kTcTile * 128, 1024);
                    tc_mma_16bit(tmem + C::kOCol, smem_desc_sw128(hi + kk * 32, 16, 1024), bdesc, id_pv,
                                (i > 0 || kk > 0) ? 1u : 0u);
                    tc_mma_16bit(tmem + C::kOCol, smem_desc_sw128(lo + kk * 32, 16, 1024), bdesc, id_pv, 1u);
                }
                tc_commit(smem_addr(&bars->pv_done[pb]));
                tc_commit(smem_addr(&bars->empty[i % nstages]));
                return true;
            };
            bool ok = true;
            for (int i = 0; i < ntiles && ok; ++i) {
                const int s = i % nstages, b = i & 1;
                if (!tc_wait(p, bars, &bars->full[s], (i / nstages) & 1)) { ok = false; break; }
                if (i >= 2 && !tc_wait(p, bars, &bars->s_free[b], ((i >> 1) - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                const uint32_t kbase = smem_addr(ring + s * C::kStageBytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t half = kk / 4, off = (kk % 4) * 32;
                    tc_mma_16bit(tmem + C::kSCol0 + b * kTcTile,
                                smem_desc_sw128(q_base + half * (kTcRows * 128) + off, 16, 1024),
                                smem_desc_sw128(kbase + half * (kTcTile * 128) + off, 16, 1024), id_qk,
                                kk > 0 ? 1u : 0u);
                }
                tc_commit(smem_addr(&bars->s_full[b]));
                if (i >= 1) ok = issue_pv(i - 1);
            }
            if (ok && ntiles > 0) issue_pv(ntiles - 1);
            // every MMA this thread issued has completed once mma_done arrives
            tc_commit(smem_addr(&bars->mma_done));
            if (!mbar_wait(smem_addr(&bars->mma_done), 0)) record_status(p.status, kStatusTimeout);
        }
    } else {
        // ------------------------------ softmax warps ------------------------------
        const bool live = R < nrows;
        int len = live ? p.context_lens[R / p.group] : 0;
        len = min(max(len, 0), p.prefix_tokens);
        const float sl2 = p.scale_log2;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        float m = -1e30f, l = 0.f, t = -INFINITY;     // finite reference max (see the mma.sync pass)
        bool ok = true;
        for (int i = 0; i < ntiles; ++i) {
            const int b = i & 1;
            if (!tc_wait(p, bars, &bars->s_full[b], (i >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            float s[kTcTile];
            {
                float part[32];
                tmem_ld32(tmem + lane_off + C::kSCol0 + b * kTcTile, part);
#pragma unroll
                for (int j = 0; j < 32; ++j) s[j] = part[j];
                tmem_ld32(tmem + lane_off + C::kSCol0 + b * kTcTile + 32, part);
#pragma unroll
                for (int j = 0; j < 32; ++j) s[32 + j] = part[j];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars->s_free[b]));
            const int t0 = tok_begin + i * kTcTile;
            const int valid = min(kTcTile, max(0, len - t0));
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < kTcTile; ++j) {
                s[j] = j < valid ? s[j] * sl2 : -INFINITY;
                mx = fmaxf(mx, s[j]);
            }
            t = fmaxf(t, mx);
            const bool need = mx > m + kTcSlack;
            const float m_new = need ? fmaxf(m, mx) : m;
            const float alpha = fast_exp2(m - m_new);
            m = m_new;
            l *= alpha;
            if (i >= 1 && __any_sync(0xffffffffu, need)) {
                // rescale O: the previous tile's P.V must have landed first
                if (!tc_wait(p, bars, &bars->pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    float o[32];
                    tmem_ld32(tmem + lane_off + C::kOCol + c, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= alpha;
                    tmem_st32(tmem + lane_off + C::kOCol + c, o);
                }
            }
            // P buffer b is free once the P.V of tile i - 2 is done
            if (i >= 2 && !tc_wait(p, bars, &bars->pv_done[b], ((i - 2) >> 1) & 1)) { ok = false; break; }
            unsigned char *hi_b = p_hi(b), *lo_b = p_lo(b);
#pragma unroll
            for (int c = 0; c < 8; ++c) {   // 8 tokens per 16-byte chunk
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = fast_exp2(s[8 * c + 2 * e] - m), p1 = fast_exp2(s[8 * c + 2 * e + 1] - m);
                    l += p0 + p1;
                    split_x2<kF16>(p0, p1, hi[e], lo[e]);   // P in the type of V
                }
                const int pos = row * 128 + ((c ^ (row & 7)) << 4);
                *reinterpret_cast<uint4 *>(hi_b + pos) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(lo_b + pos) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars->p_full[b]));
        }
        // ---- epilogue: O / l in split form at partition `chunk` ----
        const int last = ntiles - 1;
        if (ok && ntiles > 0 && tc_wait(p, bars, &bars->pv_done[last & 1], (last >> 1) & 1)) {
            tc_fence_after();
            const int64_t prow = live ? (static_cast<int64_t>(R / p.group) * p.num_heads + g * p.group +
                                         R % p.group) * p.part_stride + chunk
                                      : 0;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                float o[32];
                tmem_ld32(tmem + lane_off + C::kOCol + c, o);
                if (live) {
                    float4 *dst = reinterpret_cast<float4 *>(p.tmp_out + prow * D + c);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j] = make_float4(o[4 * j] * inv, o[4 * j + 1] * inv, o[4 * j + 2] * inv, o[4 * j + 3] * inv);
                }
            }
            if (live) {
                p.max_logits[prow] = l > 0.f ? t * kLn2 : -INFINITY;
                p.exp_sums[prow] = l > 0.f ? l * fast_exp2(m - t) : 0.f;
            }
        }
    }

    // ---- drain: copies still landing, then free the tensor memory ----
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int issued = bars->issued;
        for (int s = 0; s < nstages && s < issued; ++s) {
            const int k_last = (issued - 1 - s) / nstages;
            if (!mbar_wait(smem_addr(&bars->full[s]), k_last & 1)) record_status(p.status, kStatusTimeout);
        }
    }
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool kF16>
cudaError_t launch_tc_impl(const PrefixParams &p, const CUtensorMap &tk, const CUtensorMap &tv, dim3 grid,
                           cudaStream_t stream) {
    using C = TcCfg<D>;
    auto kern = prefix_tc_kernel<D, kF16>;
    static unsigned long long done = 0;
    cudaError_t e = ensure_smem_limit(kern, C::smem_bytes(kTcMaxRingBytes), done);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, dim3(kTcThreads), C::smem_bytes(p.ring_bytes), stream, 1u, tk, tv, p);
}

}  // namespace

int prefix_tc_rows_per_cta() { return kTcRows; }
int prefix_tc_tile_tokens() { return kTcTile; }
int prefix_tc_stage_bytes(int head_dim) { return 2 * (head_dim / 64) * kTcTile * 128; }

cudaError_t launch_prefix_tc(const PrefixParams &p, const CUtensorMap &tk, const CUtensorMap &tv, dim3 grid,
                             cudaStream_t stream) {
    if (p.head_dim == 128)
        return p.kv_f16 ? launch_tc_impl<128, true>(p, tk, tv, grid, stream)
                        : launch_tc_impl<128, false>(p, tk, tv, grid, stream);
    if (p.head_dim == 64)
        return p.kv_f16 ? launch_tc_impl<64, true>(p, tk, tv, grid, stream)
                        : launch_tc_impl<64, false>(p, tk, tv, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
