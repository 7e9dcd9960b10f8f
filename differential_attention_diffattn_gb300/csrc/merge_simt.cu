// Merge of partial differential-attention results over disjoint key blocks
// (context-parallel split of one sequence), then the combine and normalisation
// of the forward.
//
// Part j of a (token, head) row holds, per component c, lse_c^j = log2 of the
// sum of 2^(scaled score) over its visible keys and O_c^j, the attention output
// normalised over those keys (the training forward's saved statistics). Each
// component's softmax over all keys is the combination of the parts weighted by
// their sums of exponentials, so with L = max_j lse_c^j
//   O_c = sum_j 2^(lse_c^j - L) O_c^j / sum_j 2^(lse_c^j - L);
// then D = O_1 - lambda O_2, RMSNorm over dv, weight, (1 - lambda_init)
// ("DiffTransformer.py", MultiHeadDifferentialAttention.forward). The RMSNorm is
// not linear, so it runs only after both merges.
#include <cuda_bf16.h>

#include "internal.h"

namespace diffattn {
namespace {

constexpr int WARPS = 8;
constexpr int MAX_V4 = 4;  // dv <= 4 * 32 * 4 = 512 values per row

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// One warp per (token, head) row; lane l owns the float4 columns l, l + 32, ...
__global__ void __launch_bounds__(32 * WARPS) diffattn_merge_kernel(const MergeParams p) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
    if (row >= p.tokens * p.H) return;
    const int h = (int)(row % p.H);
    const int nv4 = p.dv / 4;
    const size_t part_rows = (size_t)p.tokens * p.H;
    // per component: the largest lse over the parts (lanes stride over the parts)
    float L[2] = {-INFINITY, -INFINITY};
    for (int j = lane; j < p.n_parts; j += 32) {
        const float2 l2 = reinterpret_cast<const float2*>(p.lse)[(size_t)j * part_rows + row];
        L[0] = fmaxf(L[0], l2.x);
        L[1] = fmaxf(L[1], l2.y);
    }
    L[0] = warp_max(L[0]);
    L[1] = warp_max(L[1]);
    float4 acc[2][MAX_V4];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = 0; i < MAX_V4; ++i) acc[c][i] = make_float4(0.f, 0.f, 0.f, 0.f);
    float W[2] = {0.f, 0.f};
    for (int j = 0; j < p.n_parts; ++j) {
        const float2 l2 = reinterpret_cast<const float2*>(p.lse)[(size_t)j * part_rows + row];
        // a part in which the row sees no key has lse = -inf and weight 0
        const float w0 = l2.x == -INFINITY ? 0.f : exp2f(l2.x - L[0]);
        const float w1 = l2.y == -INFINITY ? 0.f : exp2f(l2.y - L[1]);
        W[0] += w0;
        W[1] += w1;
        const float4* a = reinterpret_cast<const float4*>(p.o1) + ((size_t)j * part_rows + row) * nv4;
        const float4* b = reinterpret_cast<const float4*>(p.o2) + ((size_t)j * part_rows + row) * nv4;
#pragma unroll
        for (int i = 0; i < MAX_V4; ++i) {
            const int c4 = lane + 32 * i;
            if (c4 < nv4) {
                if (w0 != 0.f) {
                    const float4 x = a[c4];
                    acc[0][i].x = fmaf(w0, x.x, acc[0][i].x); acc[0][i].y = fmaf(w0, x.y, acc[0][i].y);
                    acc[0][i].z = fmaf(w0, x.z, acc[0][i].z); acc[0][i].w = fmaf(w0, x.w, acc[0][i].w);
                }
                if (w1 != 0.f) {
                    const float4 y = b[c4];
                    acc[1][i].x = fmaf(w1, y.x, acc[1][i].x); acc[1][i].y = fmaf(w1, y.y, acc[1][i].y);
                    acc[1][i].z = fmaf(w1, y.z, acc[1][i].z); acc[1][i].w = fmaf(w1, y.w, acc[1][i].w);
                }
            }
        }
    }
    // no visible key in any part: the component's output is taken as 0
    const float i0 = W[0] > 0.f ? 1.f / W[0] : 0.f, i1 = W[1] > 0.f ? 1.f / W[1] : 0.f;
    const float lam = p.lambda[h * p.lambda_stride];
    float ss = 0.f;
    float4 D[MAX_V4];
#pragma unroll
    for (int i = 0; i < MAX_V4; ++i) {
        D[i].x = acc[0][i].x * i0 - lam * (acc[1][i].x * i1);
        D[i].y = acc[0][i].y * i0 - lam * (acc[1][i].y * i1);
        D[i].z = acc[0][i].z * i0 - lam * (acc[1][i].z * i1);
        D[i].w = acc[0][i].w * i0 - lam * (acc[1][i].w * i1);
        ss += D[i].x * D[i].x + D[i].y * D[i].y + D[i].z * D[i].z + D[i].w * D[i].w;  // zero past dv
    }
    ss = warp_sum(ss);
    const float scale = (1.f - p.lambda_init) / sqrtf(ss / (float)p.dv + p.eps);
#pragma unroll
    for (int i = 0; i < MAX_V4; ++i) {
        const int c4 = lane + 32 * i;
        if (c4 < nv4) {
            const float4 w = reinterpret_cast<const float4*>(p.subln_w)[c4];
            const float y0 = D[i].x * scale * w.x, y1 = D[i].y * scale * w.y;
            const float y2 = D[i].z * scale * w.z, y3 = D[i].w * scale * w.w;
            if (p.out_bf16) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(y0, y1), hi = __floats2bfloat162_rn(y2, y3);
                uint2 u;
                u.x = *reinterpret_cast<uint32_t*>(&lo);
                u.y = *reinterpret_cast<uint32_t*>(&hi);
                reinterpret_cast<uint2*>(p.out)[(size_t)row * nv4 + c4] = u;
            } else {
                reinterpret_cast<float4*>(p.out)[(size_t)row * nv4 + c4] = make_float4(y0, y1, y2, y3);
            }
        }
    }
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
    const long long rows = p.tokens * p.H;
    diffattn_merge_kernel<<<(unsigned)((rows + WARPS - 1) / WARPS), 32 * WARPS, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace diffattn
