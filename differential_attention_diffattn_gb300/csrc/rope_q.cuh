// Rotary embedding of one query tile inside the one-item-per-CTA forward kernel,
// on the Q box in shared memory after its TMA load and before the first score
// MMA reads it, with the tile's cos / sin rows staged in shared memory
// ("LlamaDiffSdpaAttention.py", forward, "Apply RoPE before splitting";
// "Add an isolated implementation of FlashDiffAttention", test script:
// apply_rotary_emb(..., interleaved=True) on the doubled d-wide heads).
//
// The Q box holds 128 query rows of one head as two [128 x 64] bf16 boxes (Q1,
// Q2), 128-byte swizzled: row r's 16-byte chunk j sits at chunk j ^ (r % 8). The
// head row (2d = 128 coordinates, box b holding coordinates 64 b .. 64 b + 63) is
// cut into segments of rot_dim coordinates; in a segment, pair i < rot_dim / 2 is
// (i, i + rot_dim / 2) (half-split) or (2i, 2i + 1) (interleaved), rotated by the
// angle pos * theta^(-2i / rot_dim) whose cos / sin come from the fp32 tables of
// diffattn_rope_tables:  a' = a cos - b sin,  b' = b cos + a sin, in fp32, one
// round to nearest bf16. The separate rotation pass (rope_simt.cu) writes the
// same two expressions with the same explicit roundings, so both give the same
// bits.
#pragma once
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103a_ptx.cuh"

namespace diffattn {

// a' = a c - b s and b' = b c + a s with every rounding spelled out.
__device__ __forceinline__ void rope_pair(float a, float b, float c, float s, float& ra, float& rb) {
    ra = __fmaf_rn(a, c, -__fmul_rn(b, s));
    rb = __fmaf_rn(b, c, __fmul_rn(a, s));
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ uint4 pack_bf16x8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// Rotation units of one row: 16 interleaved (a 16-byte chunk, 4 pairs) or 8
// half-split (two 16-byte chunks rot_dim / 2 apart, 8 pairs).
__device__ __forceinline__ int rope_units(int interleaved) { return interleaved ? 16 : 8; }

// Rotates unit u of row r of the Q box at shared address sq (two boxes of
// box_bytes), the tile's tables in shared memory: cos at tc, sin at ts, the row of
// query r at r x (rot_dim / 2) x 4 bytes.
__device__ __forceinline__ void rope_unit_smem(uint32_t sq, uint32_t box_bytes, int r, int u, uint32_t tc,
                                               uint32_t ts, int rot, int interleaved) {
    const int half = rot >> 1;
    const uint32_t trow = (uint32_t)r * (uint32_t)half * 4u;
    auto chunk_addr = [&](int e) {  // 16-byte chunk holding coordinate e (a multiple of 8)
        const int b = e >> 6, j = (e & 63) >> 3;
        return sq + (uint32_t)b * box_bytes + (uint32_t)r * 128u + ((uint32_t)(j ^ (r & 7)) << 4);
    };
    auto lds_f4 = [&](uint32_t a) {
        const uint4 v = lds_u4(a);
        return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
    };
    if (interleaved) {
        const int e0 = 8 * u, i0 = (e0 % rot) >> 1;  // pairs i0 .. i0 + 3
        const float4 c = lds_f4(tc + trow + 4u * i0), sn = lds_f4(ts + trow + 4u * i0);
        const uint32_t a = chunk_addr(e0);
        float f[8];
        unpack_bf16x8(lds_u4(a), f);
        const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {sn.x, sn.y, sn.z, sn.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) rope_pair(f[2 * m], f[2 * m + 1], cc[m], ss[m], f[2 * m], f[2 * m + 1]);
        sts_u4(a, pack_bf16x8(f));
    } else {
        const int per_seg = half >> 3, seg = u / per_seg, jj = u - seg * per_seg;
        const int c0 = seg * rot + 8 * jj, i0 = 8 * jj;  // pairs (c0 + m, c0 + half + m), m < 8
        const uint32_t a0 = chunk_addr(c0), a1 = chunk_addr(c0 + half);
        float f0[8], f1[8];
        unpack_bf16x8(lds_u4(a0), f0);
        unpack_bf16x8(lds_u4(a1), f1);
#pragma unroll
        for (int h4 = 0; h4 < 2; ++h4) {
            const float4 c = lds_f4(tc + trow + 4u * (i0 + 4 * h4)), sn = lds_f4(ts + trow + 4u * (i0 + 4 * h4));
            const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {sn.x, sn.y, sn.z, sn.w};
#pragma unroll
            for (int m = 0; m < 4; ++m)
                rope_pair(f0[4 * h4 + m], f1[4 * h4 + m], cc[m], ss[m], f0[4 * h4 + m], f1[4 * h4 + m]);
        }
        sts_u4(a0, pack_bf16x8(f0));
        sts_u4(a1, pack_bf16x8(f1));
    }
}

}  // namespace diffattn
