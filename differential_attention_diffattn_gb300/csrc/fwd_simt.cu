// CUDA-core kernels: the lambda reparameterisation and the fp32
// differential-attention forward (d in {16, 32, 64}, dv = 2d).
//
// The fp32 forward keeps IEEE fp32 arithmetic throughout (expf, division and
// sqrtf as compiled without fast-math) because its acceptance bound is 1e-5
// max-abs, below what tf32 tensor cores reach.
#include "internal.h"
#include "lambda_warp.cuh"
#include "sm103a_ptx.cuh"

namespace diffattn {
namespace {

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

// lambda_i = exp(lq1_i . lk1_i) - exp(lq2_i . lk2_i) + lambda_init; one warp per set
// ("DiffTransformer.py", MultiHeadDifferentialAttention.forward,
// "Compute lambda using reparameterization").
__global__ void diffattn_lambda_kernel(const float* __restrict__ lq1, const float* __restrict__ lk1,
                                       const float* __restrict__ lq2, const float* __restrict__ lk2, int n_sets,
                                       int d, float lambda_init, float* __restrict__ out) {
    // a forward launched next on the stream as a programmatic dependent may start
    // its setup now; it reads lambda only after this grid has completed
    griddep_launch_dependents();
    const int set = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (set >= n_sets) return;
    const size_t base = (size_t)set * d;
    const float lam = lambda_value_warp(lq1 + base, lk1 + base, lq2 + base, lk2 + base, d, lambda_init, lane);
    if (lane == 0) out[set] = lam;
}

constexpr int ROWS_PER_BLOCK = 4;  // one warp per (query row, head)

// One warp owns one query row of one diff head. Keys are taken 32 at a time:
// lane t scores key (block + t) for both components, the warp updates the two
// online-softmax states, then every lane accumulates its dv/32 value columns.
template <int D>
__global__ void __launch_bounds__(32 * ROWS_PER_BLOCK)
diffattn_fwd_f32_kernel(const FwdParams p) {
    constexpr int DVV = 2 * D;
    constexpr int NV = DVV / 32;  // value columns per lane
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int h = blockIdx.y;
    const int seq = blockIdx.z;
    const int i = blockIdx.x * ROWS_PER_BLOCK + warp;

    int start, len;
    if (p.cu_seqlens != nullptr) {
        start = p.cu_seqlens[seq];
        const int end = p.cu_seqlens[seq + 1];
        const bool bad = start < 0 || end < start || end > p.total_tokens || end - start > p.max_seqlen ||
                         (seq == 0 && start != 0) || (seq == p.num_seqs - 1 && end != p.total_tokens);
        if (bad) {
            if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.error_word, kErrBadSeqlens);
            return;
        }
        len = end - start;
    } else {
        start = seq * p.seqlen;
        len = p.seqlen;
    }
    if (i >= len) return;
    const int g = h / (p.H / p.Hkv);
    const int n_keys = p.causal ? i + 1 : len;
    const float* __restrict__ qrow = static_cast<const float*>(p.q) + ((size_t)(start + i) * p.H + h) * (2 * D);
    const float* __restrict__ kbase = static_cast<const float*>(p.k) + (size_t)g * (2 * D);
    const float* __restrict__ vbase = static_cast<const float*>(p.v) + (size_t)g * DVV;
    const size_t kstride = (size_t)p.Hkv * (2 * D);
    const size_t vstride = (size_t)p.Hkv * DVV;

    float q1[D], q2[D];
#pragma unroll
    for (int e = 0; e < D; ++e) {
        q1[e] = qrow[e];
        q2[e] = qrow[D + e];
    }
    float m1 = -INFINITY, m2 = -INFINITY, l1 = 0.f, l2 = 0.f;
    float acc1[NV], acc2[NV];
#pragma unroll
    for (int t = 0; t < NV; ++t) acc1[t] = acc2[t] = 0.f;

    for (int kb = 0; kb < n_keys; kb += 32) {
        const int j = kb + lane;
        const bool valid = j < n_keys;
        float z1 = -INFINITY, z2 = -INFINITY;
        if (valid) {
            const float* kr = kbase + (size_t)(start + j) * kstride;
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int e = 0; e < D; ++e) {
                a = fmaf(q1[e], kr[e], a);
                b = fmaf(q2[e], kr[D + e], b);
            }
            z1 = a * p.scale;
            z2 = b * p.scale;
        }
        const float n1 = fmaxf(m1, warp_max(z1));
        const float n2 = fmaxf(m2, warp_max(z2));
        const float a1 = expf(m1 - n1);  // 0 on the first block (m = -inf)
        const float a2 = expf(m2 - n2);
        const float p1 = valid ? expf(z1 - n1) : 0.f;
        const float p2 = valid ? expf(z2 - n2) : 0.f;
        l1 = l1 * a1 + warp_sum(p1);
        l2 = l2 * a2 + warp_sum(p2);
        m1 = n1;
        m2 = n2;
#pragma unroll
        for (int t = 0; t < NV; ++t) {
            acc1[t] *= a1;
            acc2[t] *= a2;
        }
        const int nb = min(32, n_keys - kb);
        for (int jj = 0; jj < nb; ++jj) {
            const float w1 = __shfl_sync(0xffffffffu, p1, jj);
            const float w2 = __shfl_sync(0xffffffffu, p2, jj);
            const float* vr = vbase + (size_t)(start + kb + jj) * vstride;
#pragma unroll
            for (int t = 0; t < NV; ++t) {
                const float vv = vr[t * 32 + lane];
                acc1[t] = fmaf(w1, vv, acc1[t]);
                acc2[t] = fmaf(w2, vv, acc2[t]);
            }
        }
    }
    // D = O1/l1 - lambda O2/l2, then RMSNorm over dv, weight and (1 - lambda_init)
    const float lam = p.lambda[h * p.lambda_stride];
    float dd[NV];
    float ss = 0.f;
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        dd[t] = acc1[t] / l1 - lam * (acc2[t] / l2);
        ss = fmaf(dd[t], dd[t], ss);
    }
    ss = warp_sum(ss);
    const float rinv = 1.f / sqrtf(ss / (float)DVV + p.eps);
    float* orow = static_cast<float*>(p.out) + ((size_t)(start + i) * p.H + h) * DVV;
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        const int e = t * 32 + lane;
        orow[e] = dd[t] * rinv * p.subln_w[e] * (1.f - p.lambda_init);
    }
}

}  // namespace

cudaError_t launch_lambda(const float* lq1, const float* lk1, const float* lq2, const float* lk2, int n_sets,
                          int d, float lambda_init, float* out, cudaStream_t stream) {
    const int warps = 4;
    const int blocks = (n_sets + warps - 1) / warps;
    diffattn_lambda_kernel<<<blocks, 32 * warps, 0, stream>>>(lq1, lk1, lq2, lk2, n_sets, d, lambda_init, out);
    return cudaGetLastError();
}

cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream) {
    dim3 grid((unsigned)((p.max_seqlen + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK), (unsigned)p.H,
              (unsigned)p.num_seqs);
    dim3 block(32 * ROWS_PER_BLOCK);
    switch (p.d) {
        case 16: diffattn_fwd_f32_kernel<16><<<grid, block, 0, stream>>>(p); break;
        case 32: diffattn_fwd_f32_kernel<32><<<grid, block, 0, stream>>>(p); break;
        case 64: diffattn_fwd_f32_kernel<64><<<grid, block, 0, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace diffattn
