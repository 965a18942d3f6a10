// Paged decode attention, bf16 K/V, tensor-core kernel for sm_103a.
//
// What it computes: for each sequence b and query head h, softmax(scale *
// q_h K^T) V over the sequence's tokens, with K and V fetched block by block
// through the block table ("What Does PagedAttention Actually Optimize?",
// sections 8 and 14; "PagedAttention, explained.", procedure step 5). Query
// head h reads KV head h / (Hq / Hkv).
//
// How (one CTA = one sequence x one KV head x up to 16 of its query heads x
// one partition of its blocks):
//  * warp 4 (one elected lane) walks the block table and issues TMA tiled
//    loads (cp.async.bulk.tensor) of each physical block's K and V rows for
//    this KV head into a ring of shared-memory stages, completion counted on
//    mbarriers. The tile is the page: block_size rows of head_dim bf16,
//    loaded as 64-dim halves with the 128-byte swizzle so that the matrix
//    loads below are bank-conflict free.
//  * warps 0-3 take the stages round-robin. S = Q K^T runs on the tensor
//    cores with mma.m16n8k16 (M = query heads of the GQA group, N = tokens,
//    K = head dims), Q living in registers for the whole CTA. Online softmax
//    in base 2 (scores pre-multiplied by scale*log2 e) with the running max
//    and sum per row; P is split into a bf16 high part and a bf16 residual
//    so that P.V (mma with M = heads, N = head dims, K = tokens) keeps ~16
//    bits of P. A consumer releases its stage with an mbarrier arrive.
//  * tokens past the context in the last block are masked (score -inf, V
//    rows zeroed in shared memory, so stale or NaN slot contents never leak).
//  * the four warps' softmax states are merged in shared memory and handed to
//    the shared epilogue (final output, split-K partition, or fused
//    last-CTA log-sum-exp merge).
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the device status word, drains its own copies and returns.
#include "device_common.cuh"
#include "internal.h"

namespace pa {

template <int D, int BS>
struct MmaCfg {
    static constexpr int kConsumerWarps = 4;
    static constexpr int kThreads = 32 * (kConsumerWarps + 1);
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = BS * 128;      // one 64-dim half of a K or V tile
    static constexpr int kTileBytes = BS * D * 2;    // K (or V) rows of one block, one head
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRawStages = (64 * 1024) / kStageBytes;
    static constexpr int kStages = kRawStages > 16 ? 16 : kRawStages;
    static constexpr size_t kMergeBytes = MergeLayout<D>::bytes(kConsumerWarps);
    static constexpr size_t kRingBytes = static_cast<size_t>(kStages) * kStageBytes;
    static constexpr size_t kDataBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static constexpr size_t kSmemBytes = 1024 + kDataBytes + 2 * kStages * sizeof(uint64_t);
    static_assert(kStages % kConsumerWarps == 0, "stage ring must be a multiple of the consumer warps");
    static_assert(kHalfBytes % 1024 == 0, "swizzled halves must stay 1024-byte aligned");
    static_assert(BS % 8 == 0 && BS <= 32, "block size must be 8, 16 or 32");
};

__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16x2(x, y);
    const float hx = bf16_bits_to_float(hi & 0xffffu);
    const float hy = bf16_bits_to_float(hi >> 16);
    lo = pack_bf16x2(x - hx, y - hy);
}

template <int D, int BS>
__global__ void __launch_bounds__(MmaCfg<D, BS>::kThreads, 2)
decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ DecodeParams p) {
    using C = MmaCfg<D, BS>;
    constexpr int kStages = C::kStages;
    constexpr int kNT = BS / 8;  // n-tiles of 8 tokens per block
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kDataBytes);
    __shared__ int s_abort;
    __shared__ int s_issued;

    const int part = blockIdx.x;
    const int g = blockIdx.y / p.ntile;
    const int tile = blockIdx.y % p.ntile;
    const int b = blockIdx.z;
    const int rows = min(kRowsPerTile, p.group - tile * kRowsPerTile);
    const SeqWork w = seq_work(p, b, part);
    if (w.blk_begin >= w.blk_end) {
        write_empty<D>(p, b, g, tile, part, rows, w.nparts);
        return;
    }
    const int ntiles = w.blk_end - w.blk_begin;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&bars[s]), 1);
            mbar_init(smem_addr(&bars[kStages + s]), 1);
        }
        s_abort = 0;
        s_issued = 0;
        mbar_fence_init();
    }
    __syncthreads();

    float o[D / 8][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    if (warp == C::kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
            const uint64_t policy = l2_policy_evict_first();
            const int32_t *table = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;
            int issued = 0;
            for (int i = 0; i < ntiles; ++i) {
                const int s = i % kStages, k = i / kStages;
                if (k > 0) {
                    if (*reinterpret_cast<volatile int *>(&s_abort)) break;
                    if (!mbar_wait(smem_addr(&bars[kStages + s]), (k - 1) & 1)) {
                        record_status(p.status, kStatusTimeout);
                        s_abort = 1;
                        break;
                    }
                }
                const int phys = table[w.blk_begin + i];
                const uint32_t full = smem_addr(&bars[s]);
                mbar_arrive_expect_tx(full, C::kStageBytes);
                const uint32_t kdst = smem_addr(smem + s * C::kStageBytes);
                const uint32_t vdst = kdst + C::kTileBytes;
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h) {
                    tma_load_4d(kdst + h * C::kHalfBytes, &tmap_k, h * 64, g, 0, phys, full, policy);
                    tma_load_4d(vdst + h * C::kHalfBytes, &tmap_v, h * 64, g, 0, phys, full, policy);
                }
                issued = i + 1;
            }
            s_issued = issued;
        }
    } else {
        // ------------------------------ consumers -----------------------------
        const int r = lane >> 2, q4 = lane & 3;
        // Q fragments (A operand, rows = query heads of this tile), held for the CTA's lifetime
        uint32_t qa[D / 16][4];
        {
            const int h0 = g * p.group + tile * kRowsPerTile;
            const uint32_t *q0 = reinterpret_cast<const uint32_t *>(
                static_cast<const __nv_bfloat16 *>(p.query) +
                (static_cast<int64_t>(b) * p.num_heads + h0 + r) * D);
            const uint32_t *q1 = q0 + 8 * (D / 2);
            const bool v0 = r < rows, v1 = r + 8 < rows;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int c = (16 * kk + 2 * q4) / 2;
                qa[kk][0] = v0 ? q0[c] : 0u;
                qa[kk][1] = v1 ? q1[c] : 0u;
                qa[kk][2] = v0 ? q0[c + 4] : 0u;
                qa[kk][3] = v1 ? q1[c + 4] : 0u;
            }
        }
        const float sl2 = p.scale_log2;

        for (int i = warp; i < ntiles; i += C::kConsumerWarps) {
            if (*reinterpret_cast<volatile int *>(&s_abort)) break;
            const int s = i % kStages, k = i / kStages;
            if (!mbar_wait(smem_addr(&bars[s]), k & 1)) {
                record_status(p.status, kStatusTimeout);
                s_abort = 1;
                break;
            }
            unsigned char *stage = smem + s * C::kStageBytes;
            const uint32_t kbase = smem_addr(stage);
            const uint32_t vbase = kbase + C::kTileBytes;
            const int t0 = (w.blk_begin + i) * BS;
            const int valid = min(BS, w.len - t0);
            if (valid < BS) {
                // zero V rows past the context (whole 128-byte rows: swizzle is irrelevant)
                uint4 *vz = reinterpret_cast<uint4 *>(stage + C::kTileBytes);
                for (int c = lane; c < C::kHalves * BS * 8; c += 32)
                    if ((c % (BS * 8)) / 8 >= valid) vz[c] = make_uint4(0u, 0u, 0u, 0u);
                __syncwarp();
            }

            // ---- S = Q K^T ----
            float sacc[kNT][4];
#pragma unroll
            for (int j = 0; j < kNT; ++j) {
                sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < D / 16; kk += 2) {
                    const int tok = 8 * j + (lane & 7);
                    const int c = 2 * kk + (lane >> 3);
                    const uint32_t addr = kbase + (c >> 3) * C::kHalfBytes + tok * 128 +
                                          (((c & 7) ^ (tok & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(addr, b0, b1, b2, b3);
                    mma_bf16_16816(sacc[j], qa[kk], b0, b1);
                    mma_bf16_16816(sacc[j], qa[kk + 1], b2, b3);
                }
            }

            // ---- online softmax (base 2) ----
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int j = 0; j < kNT; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const bool live = 8 * j + 2 * q4 + e < valid;
                    const float s0 = live ? sacc[j][e] * sl2 : -INFINITY;
                    const float s1 = live ? sacc[j][2 + e] * sl2 : -INFINITY;
                    sacc[j][e] = s0;
                    sacc[j][2 + e] = s1;
                    mx0 = fmaxf(mx0, s0);
                    mx1 = fmaxf(mx1, s1);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float a0 = fast_exp2(m0 - mn0), a1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            l0 *= a0;
            l1 *= a1;
#pragma unroll
            for (int i2 = 0; i2 < D / 8; ++i2) {
                o[i2][0] *= a0;
                o[i2][1] *= a0;
                o[i2][2] *= a1;
                o[i2][3] *= a1;
            }
            constexpr int kKS = (kNT + 1) / 2;  // 16-token k-steps of P.V
            uint32_t phi[kKS][4], plo[kKS][4];
#pragma unroll
            for (int u = 0; u < kKS; ++u) phi[u][2] = phi[u][3] = plo[u][2] = plo[u][3] = 0u;
#pragma unroll
            for (int j = 0; j < kNT; ++j) {
                const float p0 = fast_exp2(sacc[j][0] - mn0), p1 = fast_exp2(sacc[j][1] - mn0);
                const float p2 = fast_exp2(sacc[j][2] - mn1), p3 = fast_exp2(sacc[j][3] - mn1);
                l0 += p0 + p1;
                l1 += p2 + p3;
                const int u = j >> 1, hh = (j & 1) * 2;
                split_bf16x2(p0, p1, phi[u][hh], plo[u][hh]);
                split_bf16x2(p2, p3, phi[u][hh + 1], plo[u][hh + 1]);
            }

            // ---- O += P V ----
            if constexpr (BS >= 16) {
#pragma unroll
                for (int u = 0; u < kKS; ++u)
#pragma unroll
                    for (int dn = 0; dn < D / 8; dn += 2) {
                        const int mi = lane >> 3;
                        const int tok = 16 * u + (mi & 1) * 8 + (lane & 7);
                        const int c = dn + (mi >> 1);
                        const uint32_t addr = vbase + (c >> 3) * C::kHalfBytes + tok * 128 +
                                              (((c & 7) ^ (tok & 7)) << 4);
                        uint32_t v0, v1, v2, v3;
                        ldmatrix_x4_trans(addr, v0, v1, v2, v3);
                        mma_bf16_16816(o[dn], phi[u], v0, v1);
                        mma_bf16_16816(o[dn + 1], phi[u], v2, v3);
                        mma_bf16_16816(o[dn], plo[u], v0, v1);
                        mma_bf16_16816(o[dn + 1], plo[u], v2, v3);
                    }
            } else {
#pragma unroll
                for (int dn = 0; dn < D / 8; dn += 4) {
                    const int tok = lane & 7;
                    const int c = dn + (lane >> 3);
                    const uint32_t addr = vbase + (c >> 3) * C::kHalfBytes + tok * 128 +
                                          (((c & 7) ^ (tok & 7)) << 4);
                    uint32_t v0, v1, v2, v3;
                    ldmatrix_x4_trans(addr, v0, v1, v2, v3);
                    mma_bf16_16816(o[dn], phi[0], v0, 0u);
                    mma_bf16_16816(o[dn + 1], phi[0], v1, 0u);
                    mma_bf16_16816(o[dn + 2], phi[0], v2, 0u);
                    mma_bf16_16816(o[dn + 3], phi[0], v3, 0u);
                    mma_bf16_16816(o[dn], plo[0], v0, 0u);
                    mma_bf16_16816(o[dn + 1], plo[0], v1, 0u);
                    mma_bf16_16816(o[dn + 2], plo[0], v2, 0u);
                    mma_bf16_16816(o[dn + 3], plo[0], v3, 0u);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars[kStages + s]));
        }
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    }
    __syncthreads();

    // Drain: wait (bounded) for the last phase of every stage this CTA armed,
    // so that no copy is still landing in shared memory we are about to reuse.
    if (threadIdx.x == 0) {
        const int issued = s_issued;
        for (int s = 0; s < kStages && s < issued; ++s) {
            const int k_last = (issued - 1 - s) / kStages;
            if (!mbar_wait(smem_addr(&bars[s]), k_last & 1)) record_status(p.status, kStatusTimeout);
        }
    }
    __syncthreads();

    // Per-warp softmax states -> shared memory, then merged across warps.
    float *mbase = reinterpret_cast<float *>(smem);
    using L = MergeLayout<D>;
    if (warp < C::kConsumerWarps) {
        const int r = lane >> 2, q4 = lane & 3;
        float *wo = L::o(mbase, warp);
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            const int d = 8 * dn + 2 * q4;
            *reinterpret_cast<float2 *>(&wo[r * L::kStride + d]) = make_float2(o[dn][0], o[dn][1]);
            *reinterpret_cast<float2 *>(&wo[(r + 8) * L::kStride + d]) = make_float2(o[dn][2], o[dn][3]);
        }
        if (q4 == 0) {
            L::m(mbase, warp)[r] = m0;
            L::m(mbase, warp)[r + 8] = m1;
            L::l(mbase, warp)[r] = l0;
            L::l(mbase, warp)[r + 8] = l1;
        }
    }
    __syncthreads();
    combine_warps<D>(mbase, C::kConsumerWarps, rows);
    write_result<D>(p, mbase, C::kConsumerWarps, b, g, tile, part, rows, w.nparts);
}

template <int D, int BS>
static cudaError_t launch_impl(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                               dim3 grid, cudaStream_t stream) {
    using C = MmaCfg<D, BS>;
    auto kern = decode_mma_kernel<D, BS>;
    static unsigned long long done = 0;
    cudaError_t e = ensure_smem_limit(kern, C::kSmemBytes, done);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

bool decode_mma_supported(int head_dim, int block_size) {
    return (head_dim == 64 || head_dim == 128) &&
           (block_size == 8 || block_size == 16 || block_size == 32);
}

cudaError_t launch_decode_mma(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                              dim3 grid, cudaStream_t stream) {
    if (p.head_dim == 128) {
        if (p.block_size == 16) return launch_impl<128, 16>(p, tk, tv, grid, stream);
        if (p.block_size == 32) return launch_impl<128, 32>(p, tk, tv, grid, stream);
        if (p.block_size == 8) return launch_impl<128, 8>(p, tk, tv, grid, stream);
    } else if (p.head_dim == 64) {
        if (p.block_size == 16) return launch_impl<64, 16>(p, tk, tv, grid, stream);
        if (p.block_size == 32) return launch_impl<64, 32>(p, tk, tv, grid, stream);
        if (p.block_size == 8) return launch_impl<64, 8>(p, tk, tv, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pa
