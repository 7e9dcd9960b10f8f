// The rare exact step of the bf16 forward kernels' online softmax, shared so that both
// kernels give the same bits.
//
// Past the first key tile of a query tile, both kernels exponentiate a tile's scores with
// the running maximum m at once, with no maximum pass ahead of the exponentials: m stays
// the first tile's (raised only here), which leaves O_c / l_c and lse unchanged and P as
// precise (bf16 and fp32 carry the same relative precision at any magnitude). Only when a
// row's sum for a tile passes 2^32 (a score far above m, where P could overflow) does the
// warp take the tile again, maximum-first: P has already replaced half of the scores in
// tensor memory, so the scores are recomputed here on the CUDA cores (the thread's query
// row from the shared-memory Q box, the keys' rows from global memory).
#pragma once
#include <cuda_bf16.h>

#include "sm103a_ptx.cuh"

namespace diffattn {

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Score of one query row against one key (d = 64): <q, k> in fp32, the products summed in
// order of the component index. q_row: shared-memory address of the row in a [128 x 64]
// bf16 box with the 128-byte swizzle (16-byte chunk i at chunk i ^ (r % 8)); k_row: the
// key's 64 bf16 in global memory (16-byte aligned). Both are read again for every key, so
// that this rare step holds few registers.
__device__ __forceinline__ float exact_score(uint32_t q_row, int r, const __nv_bfloat16* k_row) {
    const uint4* kp = reinterpret_cast<const uint4*>(k_row);
    float s = 0.f;
#pragma unroll 2
    for (int i = 0; i < 8; ++i) {
        const uint4 qv = lds_u4(q_row + ((uint32_t)(i ^ (r & 7)) << 4));
        const uint4 kv = __ldg(kp + i);
        s = fmaf(bf_lo(qv.x), bf_lo(kv.x), s);
        s = fmaf(bf_hi(qv.x), bf_hi(kv.x), s);
        s = fmaf(bf_lo(qv.y), bf_lo(kv.y), s);
        s = fmaf(bf_hi(qv.y), bf_hi(kv.y), s);
        s = fmaf(bf_lo(qv.z), bf_lo(kv.z), s);
        s = fmaf(bf_hi(qv.z), bf_hi(kv.z), s);
        s = fmaf(bf_lo(qv.w), bf_lo(kv.w), s);
        s = fmaf(bf_hi(qv.w), bf_hi(kv.w), s);
    }
    return s;
}

// The tile maximum-first for this warp's rows. Keys >= lim (tile-relative) are masked;
// k_base points at key 0 of the tile, k_stride elements between keys. m is raised to the
// tile's maximum (times sl2) when that is more than the threshold above it, and alpha is
// the factor for the earlier sums; P_c (bf16 pairs) goes to t_s one column (two keys) at a
// time; the return value is this tile's row sum in the new reference.
template <int BN>
__device__ __forceinline__ float softmax_exact_tile(uint32_t t_s, uint32_t q_row, int r, const __nv_bfloat16* k_base,
                                                    size_t k_stride, int lim, float sl2, float threshold, float& m,
                                                    float& alpha) {
    const int nk = min(max(lim, 0), BN);
    float mx = -INFINITY;
#pragma unroll 1
    for (int k = 0; k < nk; ++k) mx = fmaxf(mx, exact_score(q_row, r, k_base + (size_t)k * k_stride));
    const float m_tile = mx * sl2;
    alpha = 1.f;
    if (m_tile > m + threshold) {
        alpha = ex2_approx(m - m_tile);
        m = m_tile;
    }
    float sum = 0.f;
    tmem_wait_st();  // the fast pass's P is replaced below
    // one column (keys 2i, 2i + 1) at a time: every lane stores every column (the stores
    // are warp-wide), masked keys give 0
#pragma unroll 1
    for (int i = 0; i < BN / 2; ++i) {
        const int k = 2 * i;
        const float p0 = k < nk ? ex2_approx(__fmaf_rn(exact_score(q_row, r, k_base + (size_t)k * k_stride), sl2, -m)) : 0.f;
        const float p1 =
            k + 1 < nk ? ex2_approx(__fmaf_rn(exact_score(q_row, r, k_base + (size_t)(k + 1) * k_stride), sl2, -m)) : 0.f;
        sum = __fadd_rn(__fadd_rn(sum, p0), p1);
        tmem_st1(t_s + (uint32_t)i, pack_bf16x2(p0, p1));
    }
    return sum;
}

}  // namespace diffattn
