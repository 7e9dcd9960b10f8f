// Combine step of the cache forward (decode and short query blocks): the split
// kernel (decode_sm103a.cu) leaves, per key split and per (query, head) row and
// component, the online-softmax state (m, l) and the unnormalised output O.
// Per (b, query, head) this kernel merges the splits per component (rescale by
// 2^(m_s - M), sum), forms O1/l1 - lambda O2/l2 ("DiffTransformer.py", forward:
// attn1 - lambda_full * attn2 in the output-difference form), applies the
// per-head RMSNorm over dv, the weight and (1 - lambda_init), and stores bf16.
#include <cuda_bf16.h>

#include "internal.h"

namespace diffattn {
namespace {

constexpr int DVD = 128;        // value dim

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// One CTA (128 threads = 128 value columns) per (batch, query, head). The
// (m, l) of every split are staged in shared memory by parallel loads, the
// split weights 2^(m_s - M) computed once, then every thread sums its column.
constexpr int MAX_COMBINE_SPLITS = 1024;

__global__ void __launch_bounds__(DVD)
diffattn_decode_combine_kernel(const KvParams p) {
    const int row = blockIdx.x;  // ((b * q_len) + t) * H + h
    const int h = row % p.H;
    const int b = row / (p.H * p.q_len);
    const int tid = threadIdx.x;
    const int L = p.cache_seqlens ? p.cache_seqlens[b] : p.capacity;
    if (L < p.q_len || L > p.capacity) return;  // reported by the split kernel
    __shared__ float wgt[2][MAX_COMBINE_SPLITS];  // m_s, then 2^(m_s - M)
    __shared__ float lsm[2][MAX_COMBINE_SPLITS];
    __shared__ float red[2][DVD / 32];
    __shared__ float mmax[2];
    const int n = p.num_splits;
    const float* ml = p.ws_ml + (size_t)row * n * 4;  // [split][component][m, l]
    for (int i = tid; i < 2 * n; i += DVD) {
        const int s_ = i >> 1, c = i & 1;
        wgt[c][s_] = ml[(s_ * 2 + c) * 2];
        lsm[c][s_] = ml[(s_ * 2 + c) * 2 + 1];
    }
    __syncthreads();
    if (tid < 64) {  // warp 0: max of component 0, warp 1: component 1
        const int c = tid >> 5, ln = tid & 31;
        float m = -INFINITY;
        for (int s_ = ln; s_ < n; s_ += 32) m = fmaxf(m, wgt[c][s_]);
        m = warp_max(m);
        if (ln == 0) mmax[c] = m;
    }
    __syncthreads();
    for (int i = tid; i < 2 * n; i += DVD) {
        const int s_ = i >> 1, c = i & 1;
        const float ms = wgt[c][s_];
        wgt[c][s_] = ms == -INFINITY ? 0.f : exp2f(ms - mmax[c]);  // empty splits weigh nothing
    }
    __syncthreads();
    float o[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        float lsum = 0.f, acc = 0.f;
        const float* op = p.ws_o + ((size_t)row * n * 2 + c) * DVD + tid;
#pragma unroll 4
        for (int s_ = 0; s_ < n; ++s_) {
            const float wv = wgt[c][s_];
            lsum = fmaf(lsm[c][s_], wv, lsum);
            acc = fmaf(op[(size_t)s_ * 2 * DVD], wv, acc);
        }
        o[c] = acc / lsum;
    }
    const float lam = p.lambda[h * p.lambda_stride];
    const float dval = o[0] - lam * o[1];
    float ss = warp_sum(dval * dval);
    if ((tid & 31) == 0) red[0][tid >> 5] = ss;
    __syncthreads();
    ss = red[0][0] + red[0][1] + red[0][2] + red[0][3];
    const float rinv = 1.f / sqrtf(ss / (float)DVD + p.eps);
    const float y = dval * rinv * p.subln_w[tid] * (1.f - p.lambda_init);
    static_cast<__nv_bfloat16*>(p.out)[(size_t)row * DVD + tid] = __float2bfloat16_rn(y);
}

}  // namespace

int decode_rows_supported(int rows) { return decode_tc_rows_supported(rows); }

int decode_max_splits() { return MAX_COMBINE_SPLITS; }

int decode_ctas_per_sm() { return decode_tc_ctas_per_sm(); }

cudaError_t launch_decode(const KvParams& p, const KvTensorMaps& maps, cudaStream_t stream) {
    cudaError_t err = launch_decode_tc(p, maps, stream);
    if (err != cudaSuccess) return err;
    diffattn_decode_combine_kernel<<<(unsigned)(p.batch * p.q_len * p.H), DVD, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace diffattn
