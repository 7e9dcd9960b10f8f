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
#include "sm103a_ptx.cuh"

namespace diffattn {
namespace {

constexpr int DVD = 128;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
// Four independent warp sums with their shuffles interleaved (each in the order of warp_sum).
__device__ __forceinline__ void warp_sum4(float& a, float& b, float& c, float& d) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ta = __shfl_xor_sync(0xffffffffu, a, o), tb = __shfl_xor_sync(0xffffffffu, b, o);
        const float tc = __shfl_xor_sync(0xffffffffu, c, o), td = __shfl_xor_sync(0xffffffffu, d, o);
        a += ta, b += tb, c += tc, d += td;
    }
}

// The rows (token, head) are taken in memory order, R = t H + h, in chunks of RC rows: a
// chunk's dout, O1 and O2 rows are three contiguous ranges, staged in shared memory by
// bulk copies (no registers hold data in flight). One CTA per SM; warp w of CTA b takes
// the chunks b + (w + NW i) gridDim.x, i = 0, 1, ..., and keeps the next DEPTH of them
// in flight in stages of its own, issuing a chunk's copies itself once it has read the
// stage's previous chunk.
namespace pre {
constexpr int RC = 4;                              // rows per chunk
constexpr int NW = 16;                             // warps
constexpr int DEPTH = 2;                           // stages per warp
constexpr uint32_t DYB = RC * DVD * 2, OB = RC * DVD * 4;
constexpr uint32_t STB = DYB + 2 * OB;             // 5 KB a chunk
constexpr int MAX_SMEM_HEADS = 1024;               // per-head lambda gradients summed in shared memory
struct Smem {
    uint8_t stage[NW][DEPTH][STB];
    uint64_t full[NW][DEPTH];
    float dw[NW][DVD];
    float dl[MAX_SMEM_HEADS];
    int abort_flag;
};
constexpr uint32_t SMEM = (uint32_t)sizeof(Smem) + 128;
}  // namespace pre

__device__ __forceinline__ uint2 lds_u2(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

// Per row, lane l owns value columns 4l .. 4l+3; lane r < RC then writes row r's
// statistics. The norm-weight gradient is kept per lane over all the warp's rows and the
// lambda gradient per head in shared memory (a register for a shared lambda), each summed
// over the CTA before one set of atomics.
__global__ void __launch_bounds__(32 * pre::NW, 1) diffattn_bwd_pre_kernel(const BwdPreParams p) {
    using namespace pre;
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long nrows = (long long)p.tokens * p.H;
    const long long nchunks = (nrows + RC - 1) / RC;
    // chunks of this warp: c_i = blockIdx.x + (warp + NW i) gridDim.x
    const long long first = blockIdx.x + (long long)warp * gridDim.x, step = (long long)NW * gridDim.x;
    const int nk = nchunks > first ? (int)((nchunks - 1 - first) / step + 1) : 0;
    const bool head_lam = p.lambda_stride != 0;
    const bool smem_heads = head_lam && p.H <= MAX_SMEM_HEADS;
    if (lane == 0) {
        for (int s = 0; s < DEPTH; ++s) mbar_init(smem_u32(&sm.full[warp][s]), 1);
        if (warp == 0) sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (smem_heads)
        for (int i = threadIdx.x; i < p.H; i += blockDim.x) sm.dl[i] = 0.f;
    __syncthreads();
    const AbortState ab{&sm.abort_flag, p.error_word, p.timeout_ns};
    auto issue = [&](int i) {  // lane 0: chunk i of this warp into stage i % DEPTH
        const long long r0 = (first + (long long)i * step) * RC;
        const uint32_t n = (uint32_t)min((long long)RC, nrows - r0);
        const uint32_t bar = smem_u32(&sm.full[warp][i % DEPTH]), st = smem_u32(sm.stage[warp][i % DEPTH]);
        mbar_arrive_expect_tx(bar, n * (DVD * 2 + 2 * DVD * 4));
        bulk_copy_g2s(st, static_cast<const __nv_bfloat16*>(p.dout) + r0 * DVD, n * DVD * 2, bar);
        bulk_copy_g2s(st + DYB, static_cast<const float*>(p.o1) + r0 * DVD, n * DVD * 4, bar);
        bulk_copy_g2s(st + DYB + OB, static_cast<const float*>(p.o2) + r0 * DVD, n * DVD * 4, bar);
    };
    if (lane == 0)
        for (int i = 0; i < min(nk, DEPTH); ++i) issue(i);
    __syncwarp();

    const float post = 1.f - p.lambda_init;
    const float lam0 = p.lambda[0];
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = p.subln_w[4 * lane + i];
    float dw[4] = {0.f, 0.f, 0.f, 0.f};
    float dlam = 0.f;  // shared lambda: this lane's rows
    int done = 0;
    for (int i = 0; i < nk; ++i) {
        const int s = i % DEPTH;
        const long long r0 = (first + (long long)i * step) * RC;
        const int n = (int)min((long long)RC, nrows - r0);
        // lane r < n: row r's (lse_1, lse_2) and lambda, fetched while the chunk lands
        float2 lse_r = make_float2(0.f, 0.f);
        float lam_r = lam0;
        if (lane < n) {
            lse_r = reinterpret_cast<const float2*>(p.lse)[r0 + lane];
            if (head_lam) lam_r = p.lambda[(int)(r0 + lane) % p.H];  // tokens x H < 2^31
        }
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.full[warp][s]), (uint32_t)(i / DEPTH) & 1u, ab))) break;
        done = i + 1;
        const uint32_t st = smem_u32(sm.stage[warp][s]);
        float md1 = 0.f, md2 = 0.f;  // lane r: delta_1, delta_2 of row r
#pragma unroll
        for (int j = 0; j < RC; j += 2) {
            if (j >= n) break;
            // rows j and j + 1 (the second may be past the chunk: its values are unused)
            const bool two = j + 1 < n;
            float dy[2][4], o1[2][4], o2[2][4], D[2][4], u[2][4];
            float ss[2] = {0.f, 0.f}, ud[2] = {0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int jj = two ? j + e : j;
                const uint2 y = lds_u2(st + (uint32_t)jj * (DVD * 2) + 8u * lane);
                const uint4 a1 = lds_u4(st + DYB + (uint32_t)jj * (DVD * 4) + 16u * lane);
                const uint4 a2 = lds_u4(st + DYB + OB + (uint32_t)jj * (DVD * 4) + 16u * lane);
                dy[e][0] = __uint_as_float(y.x << 16);
                dy[e][1] = __uint_as_float(y.x & 0xffff0000u);
                dy[e][2] = __uint_as_float(y.y << 16);
                dy[e][3] = __uint_as_float(y.y & 0xffff0000u);
                o1[e][0] = __uint_as_float(a1.x), o1[e][1] = __uint_as_float(a1.y);
                o1[e][2] = __uint_as_float(a1.z), o1[e][3] = __uint_as_float(a1.w);
                o2[e][0] = __uint_as_float(a2.x), o2[e][1] = __uint_as_float(a2.y);
                o2[e][2] = __uint_as_float(a2.z), o2[e][3] = __uint_as_float(a2.w);
                const float lam = __shfl_sync(0xffffffffu, lam_r, jj);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    D[e][k] = o1[e][k] - lam * o2[e][k];
                    u[e][k] = dy[e][k] * w[k] * post;
                    ss[e] = fmaf(D[e][k], D[e][k], ss[e]);
                    ud[e] = fmaf(u[e][k], D[e][k], ud[e]);
                }
            }
            warp_sum4(ss[0], ud[0], ss[1], ud[1]);
            float d1[2] = {0.f, 0.f}, d2[2] = {0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float rinv = 1.f / sqrtf(ss[e] / (float)DVD + p.eps);
                const float corr = ud[e] * rinv * rinv * rinv / (float)DVD;
                float dd[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    dd[k] = u[e][k] * rinv - D[e][k] * corr;
                    d1[e] = fmaf(dd[k], o1[e][k], d1[e]);
                    d2[e] = fmaf(dd[k], o2[e][k], d2[e]);
                }
                if (e == 0 || two) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) dw[k] = fmaf(dy[e][k], D[e][k] * rinv * post, dw[k]);
                    __nv_bfloat162 lo2 = __floats2bfloat162_rn(dd[0], dd[1]);
                    __nv_bfloat162 hi2 = __floats2bfloat162_rn(dd[2], dd[3]);
                    uint2 o;
                    o.x = *reinterpret_cast<uint32_t*>(&lo2);
                    o.y = *reinterpret_cast<uint32_t*>(&hi2);
                    reinterpret_cast<uint2*>(p.dd)[(r0 + j + e) * (DVD / 4) + lane] = o;
                }
            }
            warp_sum4(d1[0], d2[0], d1[1], d2[1]);
            if (lane == j) md1 = d1[0], md2 = d2[0];
            if (lane == j + 1) md1 = d1[1], md2 = d2[1];
        }
        // the stage has been read: its next chunk may land there
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && i + DEPTH < nk) issue(i + DEPTH);
        if (lane < n) {  // row r0 + lane's statistics
            const int R = (int)(r0 + lane);
            const int t = R / p.H, h = R - t * p.H;
            if (smem_heads)
                atomicAdd(&sm.dl[h], -md2);
            else if (head_lam)
                atomicAdd(p.dlambda + h, -md2);
            else
                dlam -= md2;
            // negated: the backward kernels add them to products
            reinterpret_cast<float4*>(p.rowstat)[(size_t)h * p.tokens + t] = make_float4(-lse_r.x, -lse_r.y, -md1, -md2);
            // the dK/dV kernel's row operand: values split into bf16 terms whose sum
            // carries about 24 bits (each term rounds the remainder of the ones before)
            const float u1 = -lse_r.x / p.scale_log2, u2 = -lse_r.y / p.scale_log2, e1 = -md1, cd = md1 - md2;
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
            for (int k = 0; k < 16; ++k) v[k] = __float2bfloat16_rn(0.f);
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
    // let copies still in flight (after an abort) land before the CTA can exit
    if (lane == 0) {
        const int issued = min(nk, done + DEPTH);
        for (int i = done; i < issued; ++i)
            mbar_wait_drain(smem_u32(&sm.full[warp][i % DEPTH]), (uint32_t)(i / DEPTH) & 1u, p.timeout_ns);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) sm.dw[warp][4 * lane + k] = dw[k];
    if (!head_lam) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dlam += __shfl_xor_sync(0xffffffffu, dlam, o);
        if (lane == 0 && dlam != 0.f) atomicAdd(p.dlambda, dlam);
    }
    __syncthreads();
    if (threadIdx.x < DVD) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < NW; ++k) acc += sm.dw[k][threadIdx.x];
        atomicAdd(p.dsubln_w + threadIdx.x, acc);
    }
    if (smem_heads)
        for (int i = threadIdx.x; i < p.H; i += blockDim.x) atomicAdd(p.dlambda + i, sm.dl[i]);
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
    const long long nchunks = ((long long)p.tokens * p.H + pre::RC - 1) / pre::RC;
    if (nchunks == 0) return cudaSuccess;
    static int sms = 0;
    static bool attr = false;
    if (!attr) {
        int dev = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(diffattn_bwd_pre_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pre::SMEM);
        if (err != cudaSuccess) return err;
        attr = true;
    }
    const unsigned grid = (unsigned)std::min<long long>((nchunks + pre::NW - 1) / pre::NW, sms);
    diffattn_bwd_pre_kernel<<<grid, 32 * pre::NW, pre::SMEM, stream>>>(p);
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
