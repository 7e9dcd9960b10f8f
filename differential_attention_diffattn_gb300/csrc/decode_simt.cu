// Combine step of the cache forward (decode and short query blocks): the split
// kernel (decode_sm103a.cu) leaves, per key split and per (query, head) row and
// component, the online-softmax state (m, l) and the unnormalised output O.
// Per (b, query, head) this kernel merges the splits per component (rescale by
// 2^(m_s - M), sum), forms O1/l1 - lambda O2/l2 ("DiffTransformer.py", forward:
// attn1 - lambda_full * attn2 in the output-difference form), applies the
// per-head RMSNorm over dv, the weight and (1 - lambda_init), and stores bf16.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103a_ptx.cuh"

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

// One CTA of 256 threads per (batch, query, head). The (m, l) of every split are
// staged in shared memory by parallel loads and the split weights 2^(m_s - M)
// computed once; then warp w sums splits w, w + 8, ... for both components
// (lane = four value columns, float4 loads), the eight warps' sums are added
// through shared memory, and the first 128 threads (one per value column)
// normalise and store.
constexpr int MAX_COMBINE_SPLITS = 1024;
constexpr int CWARPS = 8;

__global__ void __launch_bounds__(32 * CWARPS)
diffattn_decode_combine_kernel(const KvParams p) {
    griddep_wait();  // a programmatic dependent of the split kernel: its partials are complete
    const int row = blockIdx.x;  // ((b * q_len) + t) * H + h
    const int h = row % p.H;
    const int b = row / (p.H * p.q_len);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = p.cache_seqlens ? p.cache_seqlens[b] : p.capacity;
    if (L < p.q_len || L > p.capacity) return;  // reported by the split kernel
    __shared__ float wgt[2][MAX_COMBINE_SPLITS];  // m_s, then 2^(m_s - M)
    __shared__ float lsm[2][MAX_COMBINE_SPLITS];
    __shared__ __align__(16) float part[CWARPS][2][DVD];
    __shared__ float red[DVD / 32];
    __shared__ float mmax[2], lsum[2];
    const int n = p.num_splits;
    const float* ml = p.ws_ml + (size_t)row * n * 4;  // [split][component][m, l]
    for (int i = tid; i < 2 * n; i += 32 * CWARPS) {
        const int s_ = i >> 1, c = i & 1;
        wgt[c][s_] = ml[(s_ * 2 + c) * 2];
        lsm[c][s_] = ml[(s_ * 2 + c) * 2 + 1];
    }
    __syncthreads();
    if (warp < 2) {  // warp 0: max of component 0, warp 1: component 1
        float m = -INFINITY;
        for (int s_ = lane; s_ < n; s_ += 32) m = fmaxf(m, wgt[warp][s_]);
        m = warp_max(m);
        if (lane == 0) mmax[warp] = m;
    }
    __syncthreads();
    for (int i = tid; i < 2 * n; i += 32 * CWARPS) {
        const int s_ = i >> 1, c = i & 1;
        const float ms = wgt[c][s_];
        wgt[c][s_] = ms == -INFINITY ? 0.f : exp2f(ms - mmax[c]);  // empty splits weigh nothing
    }
    __syncthreads();
    if (warp < 2) {
        float ls = 0.f;
        for (int s_ = lane; s_ < n; s_ += 32) ls = fmaf(lsm[warp][s_], wgt[warp][s_], ls);
        ls = warp_sum(ls);
        if (lane == 0) lsum[warp] = ls;
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4* op = reinterpret_cast<const float4*>(p.ws_o + ((size_t)row * n * 2 + c) * DVD) + lane;
#pragma unroll 4
        for (int s_ = warp; s_ < n; s_ += CWARPS) {
            const float wv = wgt[c][s_];
            const float4 o = op[(size_t)s_ * 2 * (DVD / 4)];
            acc.x = fmaf(o.x, wv, acc.x);
            acc.y = fmaf(o.y, wv, acc.y);
            acc.z = fmaf(o.z, wv, acc.z);
            acc.w = fmaf(o.w, wv, acc.w);
        }
        reinterpret_cast<float4*>(part[warp][c])[lane] = acc;
    }
    __syncthreads();
    float dval = 0.f;
    if (tid < DVD) {
        float o[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < CWARPS; ++w) acc += part[w][c][tid];
            o[c] = acc / lsum[c];
        }
        const float lam = p.lambda[h * p.lambda_stride];
        dval = o[0] - lam * o[1];
        const float ss = warp_sum(dval * dval);
        if (lane == 0) red[warp] = ss;
    }
    __syncthreads();
    if (tid < DVD) {
        const float ss = red[0] + red[1] + red[2] + red[3];
        const float rinv = 1.f / sqrtf(ss / (float)DVD + p.eps);
        const float y = dval * rinv * p.subln_w[tid] * (1.f - p.lambda_init);
        static_cast<__nv_bfloat16*>(p.out)[(size_t)row * DVD + tid] = __float2bfloat16_rn(y);
    }
}

}  // namespace

int decode_rows_supported(int rows) { return decode_tc_rows_supported(rows); }

int decode_max_splits() { return MAX_COMBINE_SPLITS; }

int decode_ctas_per_sm() { return decode_tc_ctas_per_sm(); }

cudaError_t launch_decode(const KvParams& p, const KvTensorMaps& maps, cudaStream_t stream) {
    cudaError_t err = launch_decode_tc(p, maps, stream);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.batch * p.q_len * p.H));
    cfg.blockDim = dim3(32 * CWARPS);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, diffattn_decode_combine_kernel, p);
}

}  // namespace diffattn
