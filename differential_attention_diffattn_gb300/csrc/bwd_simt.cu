// CUDA-core parts of the backward pass: the per-row preprocessing (gradient of
// the per-head RMSNorm and the output scale, the row deltas of the two
// softmaxes, and the lambda / norm-weight gradients) and the gradient of the
// lambda reparameterisation.
//
// Per (token, head) row, with D = O1 - lambda O2, r = sqrt(mean(D^2) + eps),
// y = D / r * w * (1 - lambda_init) ("DiffTransformer.py",
// MultiHeadDifferentialAttention.forward, "Normalize each head independently
// using RMSNorm", "Scale the normalized output") and u = dy * w * (1 - lambda_init):
//   dD      = u / r - D * <u, D> / (dv r^3)
//   delta_c = <dD, O_c>               (O_c the normalised attention output)
//   dlambda -= <dD, O2>               (D depends on lambda through -lambda O2)
//   dw     += dy * D / r * (1 - lambda_init)
#include <cuda_bf16.h>

#include "internal.h"

namespace diffattn {
namespace {

constexpr int DVD = 128;
constexpr int ROWS_PER_WARP = 8;  // loaded together, so their memory latencies overlap
constexpr int WARPS = 8;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Block (x, h): rows t = x * 64 .. x * 64 + 63 of head h; warp w takes 8 of them,
// lane l owns value columns 4l .. 4l+3. The norm-weight and lambda gradients are
// summed over the block before one set of atomics.
__global__ void __launch_bounds__(32 * WARPS, 2)  // two blocks an SM: 16 warps' loads in flight
diffattn_bwd_pre_kernel(const BwdPreParams p) {
    __shared__ float s_dw[WARPS][DVD];
    __shared__ float s_dl[WARPS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y;
    const int t0 = (blockIdx.x * WARPS + warp) * ROWS_PER_WARP;
    const float lam = p.lambda[h * p.lambda_stride];
    const float post = 1.f - p.lambda_init;
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = p.subln_w[4 * lane + i];
    float dy[ROWS_PER_WARP][4], o1[ROWS_PER_WARP][4], o2[ROWS_PER_WARP][4];
    // lane r < ROWS_PER_WARP fetches row r's (lse_1, lse_2) with the other loads, so
    // no row waits on a load of its own
    float2 lse_r = make_float2(0.f, 0.f);
    if (lane < ROWS_PER_WARP && t0 + lane < p.tokens)
        lse_r = reinterpret_cast<const float2*>(p.lse)[(size_t)(t0 + lane) * p.H + h];
#pragma unroll
    for (int r = 0; r < ROWS_PER_WARP; ++r) {
        const int t = t0 + r;
        if (t < p.tokens) {
            const size_t idx = ((size_t)t * p.H + h) * (DVD / 4) + lane;
            const uint2 u = reinterpret_cast<const uint2*>(p.dout)[idx];
            dy[r][0] = __uint_as_float(u.x << 16);
            dy[r][1] = __uint_as_float(u.x & 0xffff0000u);
            dy[r][2] = __uint_as_float(u.y << 16);
            dy[r][3] = __uint_as_float(u.y & 0xffff0000u);
            const float4 a1 = reinterpret_cast<const float4*>(p.o1)[idx];
            const float4 a2 = reinterpret_cast<const float4*>(p.o2)[idx];
            o1[r][0] = a1.x; o1[r][1] = a1.y; o1[r][2] = a1.z; o1[r][3] = a1.w;
            o2[r][0] = a2.x; o2[r][1] = a2.y; o2[r][2] = a2.z; o2[r][3] = a2.w;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) dy[r][i] = o1[r][i] = o2[r][i] = 0.f;
        }
    }
    float dw[4] = {0.f, 0.f, 0.f, 0.f};
    float dlam = 0.f;
#pragma unroll
    for (int r = 0; r < ROWS_PER_WARP; ++r) {
        const int t = t0 + r;
        float D[4], u[4], ss = 0.f, ud = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            D[i] = o1[r][i] - lam * o2[r][i];
            u[i] = dy[r][i] * w[i] * post;
            ss = fmaf(D[i], D[i], ss);
            ud = fmaf(u[i], D[i], ud);
        }
        ss = warp_sum(ss);
        ud = warp_sum(ud);
        const float rinv = 1.f / sqrtf(ss / (float)DVD + p.eps);
        const float corr = ud * rinv * rinv * rinv / (float)DVD;
        float dd[4], d1 = 0.f, d2 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            dd[i] = u[i] * rinv - D[i] * corr;
            d1 = fmaf(dd[i], o1[r][i], d1);
            d2 = fmaf(dd[i], o2[r][i], d2);
            dw[i] = fmaf(dy[r][i], D[i] * rinv * post, dw[i]);  // zero for rows past the end (dy = 0)
        }
        d1 = warp_sum(d1);
        d2 = warp_sum(d2);
        const float lse1 = __shfl_sync(0xffffffffu, lse_r.x, r), lse2 = __shfl_sync(0xffffffffu, lse_r.y, r);
        if (t < p.tokens) {
            dlam -= d2;
            const size_t row = (size_t)t * p.H + h;
            __nv_bfloat162 lo2 = __floats2bfloat162_rn(dd[0], dd[1]);
            __nv_bfloat162 hi2 = __floats2bfloat162_rn(dd[2], dd[3]);
            uint2 st;
            st.x = *reinterpret_cast<uint32_t*>(&lo2);
            st.y = *reinterpret_cast<uint32_t*>(&hi2);
            reinterpret_cast<uint2*>(p.dd)[row * (DVD / 4) + lane] = st;
            if (lane == 0) {  // negated: the backward kernels add them to products
                reinterpret_cast<float4*>(p.rowstat)[(size_t)h * p.tokens + t] = make_float4(-lse1, -lse2, -d1, -d2);
                // the dK/dV kernel's row operand: values split into bf16 terms whose sum
                // carries about 24 bits (each term rounds the remainder of the ones before)
                const float u1 = -lse1 / p.scale_log2, u2 = -lse2 / p.scale_log2, e1 = -d1, cd = d1 - d2;
                alignas(16) __nv_bfloat16 v[16];
                auto split3 = [&](float x, int at) {
                    const __nv_bfloat16 a = __float2bfloat16_rn(x);
                    const float r1 = x - __bfloat162float(a);
                    const __nv_bfloat16 b = __float2bfloat16_rn(r1);
                    v[at] = a;
                    v[at + 1] = b;
                    v[at + 2] = __float2bfloat16_rn(r1 - __bfloat162float(b));
                };
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __float2bfloat16_rn(0.f);
                split3(u1, 0);
                split3(u2, 3);
                split3(e1, 6);
                // delta_1 - delta_2 as two bf16 terms in slots 12-13 of this row and in slots
                // 14-15 of the row before, so that one 8-byte load gives a row and its successor
                const __nv_bfloat16 ch = __float2bfloat16_rn(cd);
                v[12] = ch;
                v[13] = __float2bfloat16_rn(cd - __bfloat162float(ch));
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.stat_aug) + ((size_t)h * p.tokens + t) * 16;
                *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&v[0]);
                *reinterpret_cast<uint2*>(dst + 8) = *reinterpret_cast<const uint2*>(&v[8]);
                *reinterpret_cast<uint32_t*>(dst + 12) = *reinterpret_cast<const uint32_t*>(&v[12]);
                if (t > 0) *reinterpret_cast<uint32_t*>(dst - 2) = *reinterpret_cast<const uint32_t*>(&v[12]);
                if (t == p.tokens - 1) *reinterpret_cast<uint32_t*>(dst + 14) = 0u;  // no successor: finite zeros
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) s_dw[warp][4 * lane + i] = dw[i];
    if (lane == 0) s_dl[warp] = dlam;
    __syncthreads();
    if (threadIdx.x < DVD) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < WARPS; ++k) acc += s_dw[k][threadIdx.x];
        atomicAdd(p.dsubln_w + threadIdx.x, acc);
    }
    if (threadIdx.x == 0) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < WARPS; ++k) acc += s_dl[k];
        atomicAdd(p.dlambda + h * p.lambda_stride, acc);
    }
}

// One warp per lambda parameter set:
//   dlq1 = dl e^a lk1, dlk1 = dl e^a lq1, dlq2 = -dl e^b lk2, dlk2 = -dl e^b lq2,
//   a = lq1 . lk1, b = lq2 . lk2   (derivative of "Compute lambda using reparameterization").
__global__ void diffattn_lambda_bwd_kernel(const float* __restrict__ lq1, const float* __restrict__ lk1,
                                           const float* __restrict__ lq2, const float* __restrict__ lk2,
                                           const float* __restrict__ dl, int n_sets, int d, float* dlq1,
                                           float* dlk1, float* dlq2, float* dlk2) {
    const int set = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (set >= n_sets) return;
    const size_t base = (size_t)set * d;
    float a = 0.f, b = 0.f;
    for (int e = lane; e < d; e += 32) {
        a = fmaf(lq1[base + e], lk1[base + e], a);
        b = fmaf(lq2[base + e], lk2[base + e], b);
    }
    a = warp_sum(a);
    b = warp_sum(b);
    const float ga = dl[set] * expf(a), gb = -dl[set] * expf(b);
    for (int e = lane; e < d; e += 32) {
        dlq1[base + e] = ga * lk1[base + e];
        dlk1[base + e] = ga * lq1[base + e];
        dlq2[base + e] = gb * lk2[base + e];
        dlk2[base + e] = gb * lq2[base + e];
    }
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream) {
    const int rows_per_block = WARPS * ROWS_PER_WARP;
    dim3 grid((unsigned)((p.tokens + rows_per_block - 1) / rows_per_block), (unsigned)p.H);
    diffattn_bwd_pre_kernel<<<grid, 32 * WARPS, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_lambda_bwd(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                              const float* dlambda, int n_sets, int d, float* dlq1, float* dlk1, float* dlq2,
                              float* dlk2, cudaStream_t stream) {
    const int warps = 4;
    diffattn_lambda_bwd_kernel<<<(n_sets + warps - 1) / warps, 32 * warps, 0, stream>>>(
        lq1, lk1, lq2, lk2, dlambda, n_sets, d, dlq1, dlk1, dlq2, dlk2);
    return cudaGetLastError();
}

}  // namespace diffattn
