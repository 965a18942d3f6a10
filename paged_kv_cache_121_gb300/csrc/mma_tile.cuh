// One warp's share of decode attention on the tensor cores: 16 query rows
// (one m16 tile) against one 16-token tile of K and V in shared memory,
// with a base-2 online softmax ("What Does PagedAttention Actually
// Optimize?", section 8: softmax(scale q K^T) V, computed block by block).
// Shared by the paged decode kernels and the shared-prefix kernel; bf16 or
// fp16 inputs (kF16), fp32 accumulation.
//
// Shared-memory tile layout: for each 64-dim half of the head dimension, 16
// token rows of 128 bytes; row t of half c lives at base + c * half_stride +
// tok_off(t). Swizzled (written by TMA with the 128-byte swizzle): its
// 16-byte chunk j is stored at chunk j ^ (t & 7). Unswizzled: at chunk j,
// with row starts spread over the banks by the caller's tok_off.
#pragma once

#include "device_common.cuh"

namespace pa {

constexpr float kRescaleSlack = 8.f;   // base-2 headroom before the running max is moved

__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16x2(x, y);
    const float hx = bf16_bits_to_float(hi & 0xffffu);
    const float hy = bf16_bits_to_float(hi >> 16);
    lo = pack_bf16x2(x - hx, y - hy);
}

__device__ __forceinline__ void split_f16x2(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x, y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    const float2 hf = __half22float2(h);
    lo = pack_f16x2(x - hf.x, y - hf.y);
}

// P (probabilities in [0, 1]) as a 16-bit high part plus a 16-bit residual,
// in the element type of the products.
template <bool kF16>
__device__ __forceinline__ void split_x2(float x, float y, uint32_t &hi, uint32_t &lo) {
    if constexpr (kF16) split_f16x2(x, y, hi, lo);
    else split_bf16x2(x, y, hi, lo);
}

// One warp's softmax state for 16 query rows of one KV head, in the mma
// accumulator layout: lane (r = lane/4, q = lane%4) holds rows r and r+8,
// dims 8*dn + 2q and +1 of every 8-dim slice dn.
template <int D>
struct WarpState {
    float o[D / 8][4];
    float m0, m1, l0, l1;   // reference max (base 2) and sum of 2^(s - m) per row
    float t0, t1;           // true running max of the scores (base 2)

    __device__ __forceinline__ void init() {
        m0 = m1 = t0 = t1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }

    // The per-lane partial sums become the row sums (after the last tile).
    __device__ __forceinline__ void reduce_sums() {
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    }
};

// The A fragments of the warp's 16 query rows (16-bit, D dims): q0 / q1 point at
// rows r and r + 8 (lane r = lane / 4); a row that is not live reads as zeros.
template <int D>
__device__ __forceinline__ void load_query_fragments(uint32_t (&qa)[D / 16][4], const uint32_t *q0,
                                                     const uint32_t *q1, bool live0, bool live1, int lane) {
    const int q4 = lane & 3;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int c = (16 * kk + 2 * q4) / 2;
        qa[kk][0] = live0 ? q0[c] : 0u;
        qa[kk][1] = live1 ? q1[c] : 0u;
        qa[kk][2] = live0 ? q0[c + 4] : 0u;
        qa[kk][3] = live1 ? q1[c + 4] : 0u;
    }
}

// The step's new token of sequence b (position pos), heads head0 ..
// head0+hpc-1 of K (or V), copied by one warp into its slot of the cache,
// then made visible to this CTA's later TMA / bulk reads of that slot (the
// generic-proxy writes are fenced against the async proxy before the warp
// moves on). "PagedAttention, explained.", procedure step 4.
template <int D>
__device__ __forceinline__ void warp_append_row(const DecodeParams &p, const void *src_rows, const void *cache,
                                                int b, int pos, int head0, int hpc, int lane) {
    const int blk = p.block_tables[static_cast<int64_t>(b) * p.max_blocks + pos / p.block_size];
    if (static_cast<unsigned>(blk) < static_cast<unsigned>(p.num_blocks)) {
        const int64_t slot = static_cast<int64_t>(blk) * p.block_size + pos % p.block_size;
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const uint16_t *>(src_rows) + (static_cast<int64_t>(b) * p.num_kv_heads + head0) * D);
        uint4 *dst = reinterpret_cast<uint4 *>(const_cast<uint16_t *>(static_cast<const uint16_t *>(cache)) +
                                               (slot * p.num_kv_heads + head0) * D);
        for (int c = lane; c < hpc * D / 8; c += 32) dst[c] = src[c];
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
}

// S = Q K^T for the tile, masking, online softmax update, O += P V. Tokens at
// or past valid0 (row r) / valid1 (row r + 8) get score -inf. V rows of tokens
// past the tile's data must already hold zeros (0 * NaN would leak).
template <int D, int TT, bool kSwizzled = true, bool kF16 = false, typename TokOff>
__device__ __forceinline__ void warp_tile_attention(WarpState<D> &st, const uint32_t (&qa)[D / 16][4],
                                                    uint32_t kbase, uint32_t vbase, int half_stride,
                                                    TokOff tok_off, int valid0, int valid1, float sl2,
                                                    int lane) {
    static_assert(TT == 16, "16-token tiles");
    constexpr int kNT = TT / 8;   // n-tiles of 8 tokens
    const int q4 = lane & 3;

    // ---- S = Q K^T (two interleaved accumulator chains per n-tile) ----
    float sacc[kNT][4];
#pragma unroll
    for (int j = 0; j < kNT; ++j) {
        float acc2[4] = {0.f, 0.f, 0.f, 0.f};
        sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; kk += 2) {
            const int tok = 8 * j + (lane & 7);
            const int c = 2 * kk + (lane >> 3);
            const uint32_t addr = kbase + (c >> 3) * half_stride + tok_off(tok) +
                                  (((c & 7) ^ (kSwizzled ? tok & 7 : 0)) << 4);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(addr, b0, b1, b2, b3);
            mma_16816<kF16>(sacc[j], qa[kk], b0, b1);
            mma_16816<kF16>(acc2, qa[kk + 1], b2, b3);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[j][e] = (sacc[j][e] + acc2[e]) * sl2;
    }

    // ---- online softmax (base 2) ----
    if (valid0 < TT || valid1 < TT) {
#pragma unroll
        for (int j = 0; j < kNT; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = 8 * j + 2 * q4 + e;
                if (t >= valid0) sacc[j][e] = -INFINITY;
                if (t >= valid1) sacc[j][2 + e] = -INFINITY;
            }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < kNT; ++j) {
        mx0 = fmaxf(mx0, fmaxf(sacc[j][0], sacc[j][1]));
        mx1 = fmaxf(mx1, fmaxf(sacc[j][2], sacc[j][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    st.t0 = fmaxf(st.t0, mx0);
    st.t1 = fmaxf(st.t1, mx1);
    // Lazy rescale: the reference max only moves when a score exceeds it by
    // more than kRescaleSlack (base 2), so 2^(s - m) stays <= 2^slack and the
    // O rescale is skipped while no row in the warp needs it.
    const bool need0 = mx0 > st.m0 + kRescaleSlack, need1 = mx1 > st.m1 + kRescaleSlack;
    if (__any_sync(0xffffffffu, need0 || need1)) {
        const float mn0 = need0 ? fmaxf(st.m0, mx0) : st.m0;
        const float mn1 = need1 ? fmaxf(st.m1, mx1) : st.m1;
        const float a0 = fast_exp2(st.m0 - mn0), a1 = fast_exp2(st.m1 - mn1);
        st.m0 = mn0;
        st.m1 = mn1;
        st.l0 *= a0;
        st.l1 *= a1;
#pragma unroll
        for (int i2 = 0; i2 < D / 8; ++i2) {
            st.o[i2][0] *= a0;
            st.o[i2][1] *= a0;
            st.o[i2][2] *= a1;
            st.o[i2][3] *= a1;
        }
    }
    const float mn0 = st.m0, mn1 = st.m1;
    uint32_t phi[4], plo[4];
#pragma unroll
    for (int j = 0; j < kNT; ++j) {
        const float p0 = fast_exp2(sacc[j][0] - mn0), p1 = fast_exp2(sacc[j][1] - mn0);
        const float p2 = fast_exp2(sacc[j][2] - mn1), p3 = fast_exp2(sacc[j][3] - mn1);
        st.l0 += p0 + p1;
        st.l1 += p2 + p3;
        split_x2<kF16>(p0, p1, phi[2 * j], plo[2 * j]);
        split_x2<kF16>(p2, p3, phi[2 * j + 1], plo[2 * j + 1]);
    }

    // ---- O += P V (P as a 16-bit high part plus a 16-bit residual) ----
#pragma unroll
    for (int dn = 0; dn < D / 8; dn += 2) {
        const int mi = lane >> 3;
        const int tok = (mi & 1) * 8 + (lane & 7);
        const int c = dn + (mi >> 1);
        const uint32_t addr = vbase + (c >> 3) * half_stride + tok_off(tok) +
                              (((c & 7) ^ (kSwizzled ? tok & 7 : 0)) << 4);
        uint32_t v0, v1, v2, v3;
        ldmatrix_x4_trans(addr, v0, v1, v2, v3);
        mma_16816<kF16>(st.o[dn], phi, v0, v1);
        mma_16816<kF16>(st.o[dn + 1], phi, v2, v3);
        mma_16816<kF16>(st.o[dn], plo, v0, v1);
        mma_16816<kF16>(st.o[dn + 1], plo, v2, v3);
    }
}

}  // namespace pa
