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
constexpr int P = 2;  // parts whose loads are in flight together

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

// LPR lanes per (token, head) row, 32 / LPR rows per warp; lane s of a row owns
// the float4 columns s, s + LPR, ... (V of them: dv <= 4 LPR V), so each load
// instruction reads LPR x 16 contiguous bytes of a row. The weights of a row are
// worked out by every lane of its group: with fewer lanes per row that fixed
// cost covers more columns. The parts are merged online, two at a time: their lse
// and outputs are loaded together, the running maximum of each component is
// raised to the round's largest lse and the running sums rescaled (not in the
// first round, where they are still empty). A part in which the row sees no key
// has lse = -inf (and an undefined output): its weight is 0 and its values are
// dropped by a select, never multiplied.
template <int LPR, int V>
__global__ void __launch_bounds__(32 * WARPS) diffattn_merge_kernel(const MergeParams p) {
    constexpr int RPW = 32 / LPR;
    const int lane = threadIdx.x & 31, sub = lane % LPR;
    const long long rows = p.tokens * p.H;
    const long long row = ((long long)blockIdx.x * WARPS + (threadIdx.x >> 5)) * RPW + lane / LPR;
    // a row past the end takes the last row's values (every lane of the warp
    // joins the reduction's shuffles) and stores nothing
    const bool live = row < rows;
    const long long r = live ? row : rows - 1;
    const int h = (int)(r % p.H);
    const int nv4 = p.dv / 4;
    const size_t part_rows = (size_t)rows;
    float M[2] = {-INFINITY, -INFINITY};  // running maxima of lse
    float W[2] = {0.f, 0.f};              // running sums of 2^(lse - M)
    float4 acc[2][V];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[c][i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < p.n_parts; j0 += P) {
        float2 l[P];
        float4 x[P][V], y[P][V];
#pragma unroll
        for (int u = 0; u < P; ++u) {
            const int j = j0 + u;
            const bool in = j < p.n_parts;
            const size_t prow = (size_t)(in ? j : 0) * part_rows + (size_t)r;
            l[u] = in ? reinterpret_cast<const float2*>(p.lse)[prow] : make_float2(-INFINITY, -INFINITY);
            const float4* a = reinterpret_cast<const float4*>(p.o1) + prow * nv4;
            const float4* b = reinterpret_cast<const float4*>(p.o2) + prow * nv4;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int c4 = sub + LPR * i;
                const bool ok = in && c4 < nv4;
                x[u][i] = ok ? a[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
                y[u][i] = ok ? b[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float m = M[c];
#pragma unroll
            for (int u = 0; u < P; ++u) m = fmaxf(m, c ? l[u].y : l[u].x);
            if (m == -INFINITY) continue;  // no visible key so far
            if (M[c] != -INFINITY && M[c] != m) {
                const float sc = exp2f(M[c] - m);
                W[c] *= sc;
#pragma unroll
                for (int i = 0; i < V; ++i) scale4(acc[c][i], sc);
            }
#pragma unroll
            for (int u = 0; u < P; ++u) {
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
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (!live) return;
    const float scale = (1.f - p.lambda_init) / sqrtf(ss / (float)p.dv + p.eps);
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int c4 = sub + LPR * i;
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

template <int LPR, int V>
cudaError_t launch_rows(const MergeParams& p, long long rows, cudaStream_t stream) {
    const long long per_block = (long long)WARPS * (32 / LPR);
    const long long grid = (rows + per_block - 1) / per_block;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    diffattn_merge_kernel<LPR, V><<<(unsigned)grid, 32 * WARPS, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
    const long long rows = p.tokens * p.H;
    if (rows == 0) return cudaSuccess;
    // rows of up to 128 values: 16 lanes a row (two rows a warp); wider rows: 32.
    // Measured on 16 heads x dv 128, L2 flushed, against one warp a row with four
    // parts a round: 0.62 -> 0.86 of the HBM copy rate at 2 parts x 16384 tokens,
    // 0.95 either way at 4 parts; four parts a round at 16 lanes (114 registers)
    // was slower at every part count
    if (p.dv <= 64) return launch_rows<16, 1>(p, rows, stream);
    if (p.dv <= 128) return launch_rows<16, 2>(p, rows, stream);
    if (p.dv <= 256) return launch_rows<32, 2>(p, rows, stream);
    return launch_rows<32, 4>(p, rows, stream);
}

}  // namespace diffattn
