// lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init for one parameter set
// ("DiffTransformer.py", MultiHeadDifferentialAttention.forward, "Compute lambda
// using reparameterization"), formed by one warp: lanes stride over the d entries,
// then a butterfly sum over the warp. Every kernel that forms lambda calls this,
// so all of them give the same bits.
#pragma once

namespace diffattn {

__device__ __forceinline__ float lambda_value_warp(const float* lq1, const float* lk1, const float* lq2,
                                                   const float* lk2, int d, float lambda_init, int lane) {
    float a = 0.f, b = 0.f;
    for (int e = lane; e < d; e += 32) {
        a = fmaf(lq1[e], lk1[e], a);
        b = fmaf(lq2[e], lk2[e], b);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    return expf(a) - expf(b) + lambda_init;
}

}  // namespace diffattn
