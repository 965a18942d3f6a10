// Shared-prefix attention pass, bf16 or fp16 K/V, tensor cores, sm_103a.
//
// What it computes. When every sequence of a batch starts with the same
// physical blocks (a prompt prefix shared by reference count: "PagedAttention:
// KV cache virtual memory", "Copy-on-write: when two requests share a
// prefix"; "Paged Attention: Virtual Memory for the KV Cache", "Sharing a
// prefix: one copy for many requests"), attention over those blocks is the
// same key/value set for every sequence. This pass reads each shared block
// once and, for every query row (sequence, query head) of the batch, writes
// the attention over one chunk of the prefix in split form: the normalised
// partial output, the maximum score (natural-log units) and the sum of
// exp(score - maximum). The rest of each context is attended by the decode
// kernel, and the log-sum-exp merge combines both -- the same result as one
// pass over the whole context.
//
// How. One CTA = one KV head x one chunk of the prefix x 64 query rows (4
// consumer warps of 16 rows; a row is (sequence, query head of the group),
// row-major over sequences). The producer warp walks the shared block ids and
// issues one 5-D TMA box of K and one of V per 16-token tile (one head, both
// 64-dim halves) into a shared-memory ring; every consumer warp reads every
// stage, so the CTA reads each prefix byte once for 64 rows. The consumer
// tile step is the decode kernel's (mma.m16n8k16, base-2 online softmax). A
// row's tokens at or past its sequence's length are masked.
#include "device_common.cuh"
#include "internal.h"
#include "mma_tile.cuh"

namespace pa {

namespace {

constexpr int kPrefixWarps = 4;                        // consumer warps per CTA
constexpr int kPrefixThreads = 32 * (kPrefixWarps + 1);
constexpr int kPrefixTile = 16;                        // tokens per stage
constexpr int kPrefixMaxStages = 32;

template <int D>
struct PrefixCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kStageBytes = 2 * kPrefixTile * D * 2;   // K and V of one head
    static constexpr size_t kBarrierBytes = 2 * kPrefixMaxStages * sizeof(uint64_t);
    static size_t smem_bytes(int ring) { return 1024 + static_cast<size_t>(ring) + kBarrierBytes; }
};

template <int D, bool kPairs, bool kF16>
__global__ void __launch_bounds__(kPrefixThreads, 2)
prefix_mma_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ PrefixParams p) {
    using C = PrefixCfg<D>;
    constexpr int TT = kPrefixTile;
    constexpr int box_rows = kPairs ? TT / 2 : TT;
    constexpr int kHalfStride = box_rows * 128;
    constexpr int kPairStride = C::kHalves * kHalfStride;   // second block of a pair
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.ring_bytes);
    __shared__ int s_abort;
    __shared__ int s_issued;

    if (p.pair_role != kPairSecond) grid_dependency_wait();
    if (p.pair_role == kPairFirst) grid_dependents_launch();
    const int chunk = blockIdx.x;
    const int g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tok_begin = chunk * p.chunk_tokens;
    const int tok_end = min(p.prefix_tokens, tok_begin + p.chunk_tokens);
    const int ntiles = tok_end > tok_begin ? (tok_end - tok_begin) / TT : 0;   // whole tiles
    constexpr int stage_bytes = C::kStageBytes;
    int nstages = p.ring_bytes / stage_bytes;
    if (nstages > kPrefixMaxStages) nstages = kPrefixMaxStages;
    constexpr int v_off = TT * D * 2;
    auto tok_off = [&](int t) -> int {
        return kPairs ? (t / box_rows) * kPairStride + (t % box_rows) * 128 : t * 128;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(smem_addr(&bars[s]), 1);
            mbar_init(smem_addr(&bars[kPrefixMaxStages + s]), kPrefixWarps);
        }
        s_abort = 0;
        s_issued = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == kPrefixWarps) {
        // ------------------------------ producer ------------------------------
        uint64_t policy = 0;
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
            policy = l2_policy_evict_last();   // the prefix is read by every row group
        }
        auto entry = [&](int t, int j) -> int {
            const int tok = tok_begin + t * TT + j * box_rows;
            return (t < ntiles && tok < tok_end) ? p.prefix_table[tok / p.block_size] : 0;
        };
        int cur0 = entry(lane, 0), cur1 = kPairs ? entry(lane, 1) : 0;
        int nxt0 = entry(32 + lane, 0), nxt1 = kPairs ? entry(32 + lane, 1) : 0;
        int issued = 0;
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
                    } else if (!mbar_wait(smem_addr(&bars[kPrefixMaxStages + s]), (k - 1) & 1)) {
                        record_status(p.status, kStatusTimeout);
                        s_abort = 1;
                        ok = 0;
                    }
                }
                if (ok) {
                    const uint32_t full = smem_addr(&bars[s]);
                    mbar_arrive_expect_tx(full, static_cast<uint32_t>(stage_bytes));   // tiles are whole
                    const uint32_t kdst = smem_addr(smem + s * stage_bytes);
                    const int t0 = tok_begin + i * TT;
                    // coordinates, innermost first: (dim, token, half, head, block)
                    tma_load_5d(kdst, &tmap_k, 0, kPairs ? 0 : t0 % p.block_size, 0, g, phys0, full, policy);
                    tma_load_5d(kdst + v_off, &tmap_v, 0, kPairs ? 0 : t0 % p.block_size, 0, g, phys0, full,
                                policy);
                    if (kPairs) {
                        tma_load_5d(kdst + kPairStride, &tmap_k, 0, 0, 0, g, phys1, full, policy);
                        tma_load_5d(kdst + v_off + kPairStride, &tmap_v, 0, 0, 0, g, phys1, full, policy);
                    }
                    issued = i + 1;
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        }
        if (lane == 0) s_issued = issued;
    } else {
        // ------------------------------ consumers -----------------------------
        // rows (sequence, query head of group g), 16 per warp: lane r holds
        // rows R and R + 8
        const int nrows = p.num_seqs * p.group;
        const int r = lane >> 2;
        const int R0 = (blockIdx.z * kPrefixWarps + warp) * 16 + r, R1 = R0 + 8;
        const bool live0 = R0 < nrows, live1 = R1 < nrows;
        const int b0 = live0 ? R0 / p.group : 0, b1 = live1 ? R1 / p.group : 0;
        const int hq0 = g * p.group + (live0 ? R0 % p.group : 0);
        const int hq1 = g * p.group + (live1 ? R1 % p.group : 0);
        int len0 = live0 ? p.context_lens[b0] : 0, len1 = live1 ? p.context_lens[b1] : 0;
        len0 = min(max(len0, 0), p.prefix_tokens);
        len1 = min(max(len1, 0), p.prefix_tokens);
        uint32_t qa[D / 16][4];
        {
            const uint16_t *q = static_cast<const uint16_t *>(p.query);
            const uint32_t *q0 = reinterpret_cast<const uint32_t *>(
                q + (static_cast<int64_t>(b0) * p.num_heads + hq0) * D);
            const uint32_t *q1 = reinterpret_cast<const uint32_t *>(
                q + (static_cast<int64_t>(b1) * p.num_heads + hq1) * D);
            load_query_fragments<D>(qa, q0, q1, live0, live1, lane);
        }
        WarpState<D> st;
        st.init();
        // a finite reference max: a row whose first tiles are all masked keeps
        // 2^(-inf - m) = 0 instead of 2^(-inf + inf)
        st.m0 = st.m1 = -1e30f;
        const float sl2 = p.scale_log2;

        for (int i = 0; i < ntiles; ++i) {
            if (*reinterpret_cast<volatile int *>(&s_abort)) break;
            const int s = i % nstages, k = i / nstages;
            if (!mbar_wait(smem_addr(&bars[s]), k & 1)) {
                record_status(p.status, kStatusTimeout);
                s_abort = 1;
                break;
            }
            const uint32_t kbase = smem_addr(smem + s * stage_bytes);
            const int t0 = tok_begin + i * TT;
            const int valid0 = min(TT, max(0, len0 - t0)), valid1 = min(TT, max(0, len1 - t0));
            warp_tile_attention<D, TT, true, kF16>(st, qa, kbase, kbase + v_off, kHalfStride, tok_off, valid0, valid1,
                                       sl2, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars[kPrefixMaxStages + s]));
        }
        st.reduce_sums();

        // split form at partition `chunk` of rows (b, hq)
        const int q4 = lane & 3;
        const int64_t row0 = (static_cast<int64_t>(b0) * p.num_heads + hq0) * p.part_stride + chunk;
        const int64_t row1 = (static_cast<int64_t>(b1) * p.num_heads + hq1) * p.part_stride + chunk;
        const float i0 = st.l0 > 0.f ? 1.f / st.l0 : 0.f, i1 = st.l1 > 0.f ? 1.f / st.l1 : 0.f;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            const int d = 8 * dn + 2 * q4;
            if (live0)
                *reinterpret_cast<float2 *>(p.tmp_out + row0 * D + d) = make_float2(st.o[dn][0] * i0, st.o[dn][1] * i0);
            if (live1)
                *reinterpret_cast<float2 *>(p.tmp_out + row1 * D + d) = make_float2(st.o[dn][2] * i1, st.o[dn][3] * i1);
        }
        if (q4 == 0) {   // the true max: sum of 2^(s - t) = l * 2^(m - t)
            if (live0) {
                p.max_logits[row0] = st.l0 > 0.f ? st.t0 * kLn2 : -INFINITY;
                p.exp_sums[row0] = st.l0 > 0.f ? st.l0 * fast_exp2(st.m0 - st.t0) : 0.f;
            }
            if (live1) {
                p.max_logits[row1] = st.l1 > 0.f ? st.t1 * kLn2 : -INFINITY;
                p.exp_sums[row1] = st.l1 > 0.f ? st.l1 * fast_exp2(st.m1 - st.t1) : 0.f;
            }
        }
    }

    // Drain: wait (bounded) for the last phase of every stage this CTA armed.
    __syncthreads();
    if (threadIdx.x == 0) {
        const int issued = s_issued;
        for (int s = 0; s < nstages && s < issued; ++s) {
            const int k_last = (issued - 1 - s) / nstages;
            if (!mbar_wait(smem_addr(&bars[s]), k_last & 1)) record_status(p.status, kStatusTimeout);
        }
    }
    if (p.pair_role == kPairSecond) grid_dependency_wait();   // this grid completes after the first
}

template <int D, bool kPairs, bool kF16>
cudaError_t launch_prefix_impl(const PrefixParams &p, const CUtensorMap &tk, const CUtensorMap &tv, dim3 grid,
                               cudaStream_t stream) {
    using C = PrefixCfg<D>;
    auto kern = prefix_mma_kernel<D, kPairs, kF16>;
    static unsigned long long done = 0;
    cudaError_t e = ensure_smem_limit(kern, C::smem_bytes(kPrefixMaxRingBytes), done);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, dim3(kPrefixThreads), C::smem_bytes(p.ring_bytes), stream, 1u, tk, tv, p);
}

}  // namespace

int prefix_rows_per_cta() { return 16 * kPrefixWarps; }

int prefix_stage_bytes(int head_dim) { return 2 * kPrefixTile * head_dim * 2; }

cudaError_t launch_prefix_mma(const PrefixParams &p, const CUtensorMap &tk, const CUtensorMap &tv, dim3 grid,
                              cudaStream_t stream) {
    const bool pairs = p.block_size < kPrefixTile;
    if (p.head_dim == 128) {
        if (p.kv_f16)
            return pairs ? launch_prefix_impl<128, true, true>(p, tk, tv, grid, stream)
                         : launch_prefix_impl<128, false, true>(p, tk, tv, grid, stream);
        return pairs ? launch_prefix_impl<128, true, false>(p, tk, tv, grid, stream)
                     : launch_prefix_impl<128, false, false>(p, tk, tv, grid, stream);
    }
    if (p.head_dim == 64) {
        if (p.kv_f16)
            return pairs ? launch_prefix_impl<64, true, true>(p, tk, tv, grid, stream)
                         : launch_prefix_impl<64, false, true>(p, tk, tv, grid, stream);
        return pairs ? launch_prefix_impl<64, true, false>(p, tk, tv, grid, stream)
                     : launch_prefix_impl<64, false, false>(p, tk, tv, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pa
