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
constexpr int PARTS_PER_ROUND = 4;  // parts whose loads are in flight together

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ void axpy4(float4& acc, float w, const float4& x) {
    acc.x = fmaf(w, x.x, acc.x);
    acc.y = fmaf(w, x.y, acc.y);
    acc.z = fmaf(w, x.z, acc.z);
    acc.w = fmaf(w, x.w, acc.w);
}
__device__ __forceinline__ void scale4(float4& acc, float r) {
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
}

// One warp per (token, head) row; lane l owns the float4 columns l, l + 32, ...
// (V of them: dv <= 128 V). The parts are merged online, PARTS_PER_ROUND at a
// time: their lse and outputs are loaded together, the running maximum of each
// component is raised to the round's largest lse and the running sums rescaled.
// A part in which the row sees no key has lse = -inf (and an undefined output):
// its weight is 0 and its values are dropped by a select, never multiplied.
template <int V>
__global__ void __launch_bounds__(32 * WARPS) diffattn_merge_kernel(const MergeParams p) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
    if (row >= p.tokens * p.H) return;
    const int h = (int)(row % p.H);
    const int nv4 = p.dv / 4;
    const size_t part_rows = (size_t)p.tokens * p.H;
    float M[2] = {-INFINITY, -INFINITY};  // running maxima of lse
    float W[2] = {0.f, 0.f};              // running sums of 2^(lse - M)
    float4 acc[2][V];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[c][i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < p.n_parts; j0 += PARTS_PER_ROUND) {
        float2 l[PARTS_PER_ROUND];
        float4 x[PARTS_PER_ROUND][V], y[PARTS_PER_ROUND][V];
#pragma unroll
        for (int u = 0; u < PARTS_PER_ROUND; ++u) {
            const int j = j0 + u;
            const bool in = j < p.n_parts;
            const size_t prow = (size_t)(in ? j : 0) * part_rows + row;
            l[u] = in ? reinterpret_cast<const float2*>(p.lse)[prow] : make_float2(-INFINITY, -INFINITY);
            const float4* a = reinterpret_cast<const float4*>(p.o1) + prow * nv4;
            const float4* b = reinterpret_cast<const float4*>(p.o2) + prow * nv4;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int c4 = lane + 32 * i;
                const bool ok = in && c4 < nv4;
                x[u][i] = ok ? a[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
                y[u][i] = ok ? b[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float m = M[c];
#pragma unroll
            for (int u = 0; u < PARTS_PER_ROUND; ++u) m = fmaxf(m, c ? l[u].y : l[u].x);
            if (m == -INFINITY) continue;  // no visible key so far
            const float r = M[c] == -INFINITY ? 0.f : exp2f(M[c] - m);
            W[c] *= r;
#pragma unroll
            for (int i = 0; i < V; ++i) scale4(acc[c][i], r);
#pragma unroll
            for (int u = 0; u < PARTS_PER_ROUND; ++u) {
                const float lu = c ? l[u].y : l[u].x;
                const bool vis = lu != -INFINITY;
                const float w = vis ? exp2f(lu - m) : 0.f;
                W[c] += w;
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    float4 v = c ? y[u][i] : x[u][i];
                    v = vis ? v : make_float4(0.f, 0.f, 0.f, 0.f);
                    axpy4(acc[c][i], w, v);
                }
            }
            M[c] = m;
        }
    }
    // no visible key in any part: the component's output is taken as 0
    const float i0 = W[0] > 0.f ? 1.f / W[0] : 0.f, i1 = W[1] > 0.f ? 1.f / W[1] : 0.f;
    const float lam = p.lambda[h * p.lambda_stride];
    float ss = 0.f;
    float4 D[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        D[i].x = acc[0][i].x * i0 - lam * (acc[1][i].x * i1);
        D[i].y = acc[0][i].y * i0 - lam * (acc[1][i].y * i1);
        D[i].z = acc[0][i].z * i0 - lam * (acc[1][i].z * i1);
        D[i].w = acc[0][i].w * i0 - lam * (acc[1][i].w * i1);
        ss += D[i].x * D[i].x + D[i].y * D[i].y + D[i].z * D[i].z + D[i].w * D[i].w;  // zero past dv
    }
    ss = warp_sum(ss);
    const float scale = (1.f - p.lambda_init) / sqrtf(ss / (float)p.dv + p.eps);
#pragma unroll
    for (int i = 0; i < V; ++i) {
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
    const unsigned grid = (unsigned)((rows + WARPS - 1) / WARPS);
    if (p.dv <= 128)
        diffattn_merge_kernel<1><<<grid, 32 * WARPS, 0, stream>>>(p);
    else if (p.dv <= 256)
        diffattn_merge_kernel<2><<<grid, 32 * WARPS, 0, stream>>>(p);
    else
        diffattn_merge_kernel<4><<<grid, 32 * WARPS, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace diffattn
