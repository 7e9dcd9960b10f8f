// Rotary position embedding of q and k ahead of the differential attention.
//
// Head rows (2d wide) are split into segments of R coordinates (R = 2d: the
// whole row before the q1 | q2 chunk, "LlamaDiffSdpaAttention.py", forward,
// "Apply RoPE before splitting"; R = d: every component on its own, the doubled
// heads of the FlashDiffAttention test script). In each segment pair i < R/2 is
// (i, i + R/2) or, interleaved, (2i, 2i + 1), rotated by pos * theta^(-2i/R):
//   a' = a cos - b sin,  b' = b cos + a sin.
//
// One streaming pass: K is rotated once here rather than per tile inside the
// attention kernel, where every query tile that loads a key tile would repeat
// the rotation. Each thread owns four pairs of one segment (8 coordinates: one
// 16-byte bf16 chunk interleaved, two 8-byte chunks half-split) of one token,
// reads the four matching cos / sin values once, and rotates that group in
// every head row of q and k.
#include <cuda_bf16.h>

#include "internal.h"

namespace diffattn {
namespace {

__global__ void diffattn_rope_tables_kernel(double theta, int n_pos, int half, float* cos_out, float* sin_out) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)n_pos * half) return;
    const int p = (int)(idx / half), i = (int)(idx % half);
    const double ang = (double)p * pow(theta, -2.0 * (double)i / (double)(2 * half));
    double s, c;
    sincos(ang, &s, &c);
    cos_out[idx] = (float)c;
    sin_out[idx] = (float)s;
}

template <typename T>
struct Vec8;
template <>
struct Vec8<__nv_bfloat16> {
    // 8 coordinates at p (contiguous) or 4 at p and 4 at p + gap
    __device__ static void load(const void* base, size_t off, size_t gap, bool split, float (&f)[8]) {
        const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(base) + off;
        uint32_t w[4];
        if (split) {
            const uint2 a = *reinterpret_cast<const uint2*>(p), b = *reinterpret_cast<const uint2*>(p + gap);
            w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y;
        } else {
            const uint4 a = *reinterpret_cast<const uint4*>(p);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static void store(void* base, size_t off, size_t gap, bool split, const float (&f)[8]) {
        __nv_bfloat16* p = static_cast<__nv_bfloat16*>(base) + off;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        if (split) {
            *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
            *reinterpret_cast<uint2*>(p + gap) = make_uint2(w[2], w[3]);
        } else {
            *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
};
template <>
struct Vec8<float> {
    __device__ static void load(const void* base, size_t off, size_t gap, bool split, float (&f)[8]) {
        const float* p = static_cast<const float*>(base) + off;
        const float4 a = *reinterpret_cast<const float4*>(p);
        const float4 b = *reinterpret_cast<const float4*>(p + (split ? gap : 4));
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
    __device__ static void store(void* base, size_t off, size_t gap, bool split, const float (&f)[8]) {
        float* p = static_cast<float*>(base) + off;
        *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(p + (split ? gap : 4)) = make_float4(f[4], f[5], f[6], f[7]);
    }
};

__device__ __forceinline__ int token_position(const RopeParams& p, long long t) {
    if (p.positions != nullptr) return p.positions[t];
    if (p.cu_seqlens != nullptr) {
        int lo = 0, hi = p.num_seqs;  // last sequence whose start is <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.cu_seqlens[mid] <= t) lo = mid; else hi = mid;
        }
        return (int)(t - p.cu_seqlens[lo]);
    }
    return (int)(t % p.seqlen);
}

// Rotates the 8 coordinates at `off` of rows [0, nrows) of one tensor for one
// token. (Keeping eight rows' loads in flight per thread measured slower: 2.3 to
// 3.3 TB/s against 4.4 for this loop.)
template <typename T, bool INTERLEAVED>
__device__ __forceinline__ void rotate_rows(const void* src, void* dst, size_t row0, int nrows, int width,
                                            size_t off, size_t gap, const float (&cc)[4], const float (&ss)[4],
                                            bool ok) {
#pragma unroll 4
    for (int r = 0; r < nrows; ++r) {
        const size_t o = (row0 + r) * width + off;
        float f[8], g[8];
        Vec8<T>::load(src, o, gap, !INTERLEAVED, f);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            // interleaved: pair m = coordinates (2m, 2m+1); half-split: (m, 4 + m) of the two chunks
            const int ia = INTERLEAVED ? 2 * m : m, ib = INTERLEAVED ? 2 * m + 1 : 4 + m;
            // the roundings spelled out, as in the forward kernels' own rotation of q
            g[ia] = ok ? __fmaf_rn(f[ia], cc[m], -__fmul_rn(f[ib], ss[m])) : f[ia];  // outside the tables:
            g[ib] = ok ? __fmaf_rn(f[ib], cc[m], __fmul_rn(f[ia], ss[m])) : f[ib];   // copied through
        }
        Vec8<T>::store(dst, o, gap, !INTERLEAVED, g);
    }
}

// One thread = one token and one group of four pairs (8 coordinates) of a
// segment; it reads that group's cos / sin once and walks every head row of q
// and k (consecutive threads cover consecutive 16-byte chunks of a row).
template <typename T, bool INTERLEAVED>
__global__ void __launch_bounds__(256) diffattn_rope_qk_kernel(const RopeParams p) {
    const int units_row = p.width / 8;
    const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= p.tokens * units_row) return;
    const long long t = u / units_row;
    const int w = (int)(u % units_row);
    const int per_seg = p.rot_dim / 8;
    const int seg = w / per_seg, j = w % per_seg;            // pairs 4j .. 4j+3 of segment seg
    const size_t off = (size_t)seg * p.rot_dim + (INTERLEAVED ? 8 * j : 4 * j);
    const size_t gap = p.rot_dim / 2;
    const int pos = token_position(p, t);
    const bool ok = pos >= 0 && pos < p.n_pos;
    float cc[4] = {0.f, 0.f, 0.f, 0.f}, ss[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
        const float4 c = *reinterpret_cast<const float4*>(p.cos + (size_t)pos * gap + 4 * j);
        const float4 s = *reinterpret_cast<const float4*>(p.sin + (size_t)pos * gap + 4 * j);
        cc[0] = c.x; cc[1] = c.y; cc[2] = c.z; cc[3] = c.w;
        ss[0] = s.x; ss[1] = s.y; ss[2] = s.z; ss[3] = s.w;
    } else if (w == 0) {
        atomicOr(p.error_word, kErrBadPositions);
    }
    if (p.H > 0) rotate_rows<T, INTERLEAVED>(p.q_in, p.q_out, (size_t)t * p.H, p.H, p.width, off, gap, cc, ss, ok);
    if (p.Hkv > 0)
        rotate_rows<T, INTERLEAVED>(p.k_in, p.k_out, (size_t)t * p.Hkv, p.Hkv, p.width, off, gap, cc, ss, ok);
}

}  // namespace

cudaError_t launch_rope_tables(double theta, int n_pos, int rot_dim, float* cos_out, float* sin_out,
                               cudaStream_t stream) {
    const long long n = (long long)n_pos * (rot_dim / 2);
    const int threads = 256;
    diffattn_rope_tables_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, stream>>>(
        theta, n_pos, rot_dim / 2, cos_out, sin_out);
    return cudaGetLastError();
}

cudaError_t launch_rope_qk(const RopeParams& p, bool bf16, bool interleaved, cudaStream_t stream) {
    const long long n = p.tokens * (long long)(p.width / 8);
    const int threads = 256;
    const unsigned blocks = (unsigned)((n + threads - 1) / threads);
    if (bf16) {
        if (interleaved) diffattn_rope_qk_kernel<__nv_bfloat16, true><<<blocks, threads, 0, stream>>>(p);
        else diffattn_rope_qk_kernel<__nv_bfloat16, false><<<blocks, threads, 0, stream>>>(p);
    } else {
        if (interleaved) diffattn_rope_qk_kernel<float, true><<<blocks, threads, 0, stream>>>(p);
        else diffattn_rope_qk_kernel<float, false><<<blocks, threads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace diffattn
