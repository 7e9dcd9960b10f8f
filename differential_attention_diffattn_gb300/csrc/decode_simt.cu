// Combine step of the cache forward (decode and short query blocks): the split
// kernel (decode_sm103a.cu) leaves, per key split and per (query, head) row and
// component, the online-softmax state (m, l) and the unnormalised output O.
// Per (b, query, head) this kernel merges the splits per component (rescale by
// 2^(m_s - M), sum), forms O1/l1 - lambda O2/l2 ("DiffTransformer.py", forward:
// attn1 - lambda_full * attn2 in the output-difference form), applies the
// per-head RMSNorm over dv, the weight and (1 - lambda_init), and stores bf16.
#include <cuda_bf16.h>

#include "internal.h"
#include "lambda_warp.cuh"
#include "sm103a_ptx.cuh"

namespace diffattn {
namespace {

constexpr int DVD = 128;        // value dim

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// One warp per (batch, query, head) row, eight rows a block; lane l owns value
// columns 4l .. 4l + 3. The splits are merged online, SPLITS_PER_ROUND at a time
// with all their loads in flight together (no block-wide step: the row's whole
// merge is one warp's): per component the running maximum M is raised to the
// round's largest m_s and the running sums rescaled; split s weighs 2^(m_s - M)
// (an empty split, m_s = -inf, weighs 0). Then O_c = acc_c / l_c, D = O_1 -
// lambda O_2, the RMSNorm over dv (a warp reduction), the weight and
// (1 - lambda_init), and four bf16 values per lane.
constexpr int MAX_COMBINE_SPLITS = 1024;
constexpr int CWARPS = 8;
constexpr int SPLITS_PER_ROUND = 4;

__global__ void __launch_bounds__(32 * CWARPS)
diffattn_decode_combine_kernel(const KvParams p) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * CWARPS + (threadIdx.x >> 5);  // ((b * q_len) + t) * H + h
    const bool row_ok = row < (long long)p.batch * p.q_len * p.H;
    const int h = (int)(row % p.H);
    const int b = (int)(row / ((long long)p.H * p.q_len));
    // The inputs of the call (lengths, weight, lambda) are read before the wait for
    // the split kernel: this grid is placed only once every split CTA has passed its
    // own wait for the kernels before it (the lambda kernel among them), so they are
    // complete; only the partials come from the split kernel. In a combined call each
    // row's warp forms its head's lambda from the parameter vectors, and the warps of
    // the first query's rows write it out.
    int L = 0;
    float lam = 0.f;
    float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.lq1 != nullptr) {  // warp-uniform; rows past the end form a valid set's lambda too
        const int set = p.lambda_stride ? h : 0;
        const size_t base = (size_t)set * p.lambda_d;
        lam = lambda_value_warp(p.lq1 + base, p.lk1 + base, p.lq2 + base, p.lk2 + base, p.lambda_d, p.lambda_init,
                                lane);
        if (lane == 0 && row == set) p.lambda_out[set] = lam;  // row (b = 0, t = 0, h = set)
    }
    if (row_ok) {  // from L2 (ld.global.cg): no line an earlier grid left in this SM's L1
        L = p.cache_seqlens ? __ldcg(p.cache_seqlens + b) : p.capacity;
        if (p.lq1 == nullptr) lam = __ldcg(p.lambda + h * p.lambda_stride);
        w = __ldcg(reinterpret_cast<const float4*>(p.subln_w) + lane);
    }
    griddep_wait();  // a programmatic dependent of the split kernel: its partials are complete
    if (!row_ok) return;
    if (L < p.q_len || L > p.capacity) return;  // reported by the split kernel
    const int n = p.num_splits;
    const float* ml = p.ws_ml + (size_t)row * n * 4;              // [split][component][m, l]
    const float4* op = reinterpret_cast<const float4*>(p.ws_o + (size_t)row * n * 2 * DVD) + lane;  // [split][c][dv]
    float M[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int s0 = 0; s0 < n; s0 += SPLITS_PER_ROUND) {
        float4 mlv[SPLITS_PER_ROUND];  // m_1, l_1, m_2, l_2
        float4 ov[SPLITS_PER_ROUND][2];
#pragma unroll
        for (int u = 0; u < SPLITS_PER_ROUND; ++u) {
            const int sp = s0 + u;
            if (sp < n) {
                mlv[u] = reinterpret_cast<const float4*>(ml)[sp];
                ov[u][0] = op[(size_t)sp * 2 * (DVD / 4)];
                ov[u][1] = op[(size_t)sp * 2 * (DVD / 4) + DVD / 4];
            } else {
                mlv[u] = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
                ov[u][0] = ov[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float m = M[c];
#pragma unroll
            for (int u = 0; u < SPLITS_PER_ROUND; ++u) m = fmaxf(m, c ? mlv[u].z : mlv[u].x);
            if (m == -INFINITY) continue;  // no visible key so far
            if (M[c] != -INFINITY && M[c] != m) {
                const float r = exp2f(M[c] - m);
                lsum[c] *= r;
                acc[c].x *= r;
                acc[c].y *= r;
                acc[c].z *= r;
                acc[c].w *= r;
            }
#pragma unroll
            for (int u = 0; u < SPLITS_PER_ROUND; ++u) {
                const float ms = c ? mlv[u].z : mlv[u].x, ls = c ? mlv[u].w : mlv[u].y;
                const float w = ms == -INFINITY ? 0.f : exp2f(ms - m);  // empty splits weigh nothing
                lsum[c] = fmaf(ls, w, lsum[c]);
                acc[c].x = fmaf(ov[u][c].x, w, acc[c].x);
                acc[c].y = fmaf(ov[u][c].y, w, acc[c].y);
                acc[c].z = fmaf(ov[u][c].z, w, acc[c].z);
                acc[c].w = fmaf(ov[u][c].w, w, acc[c].w);
            }
            M[c] = m;
        }
    }
    const float i1 = 1.f / lsum[0], i2 = 1.f / lsum[1];  // every row sees at least one key
    const float4 d = make_float4(acc[0].x * i1 - lam * (acc[1].x * i2), acc[0].y * i1 - lam * (acc[1].y * i2),
                                 acc[0].z * i1 - lam * (acc[1].z * i2), acc[0].w * i1 - lam * (acc[1].w * i2));
    const float ss = warp_sum(d.x * d.x + d.y * d.y + d.z * d.z + d.w * d.w);
    const float post = (1.f - p.lambda_init) / sqrtf(ss / (float)DVD + p.eps);
    __nv_bfloat162 lo = __floats2bfloat162_rn(d.x * post * w.x, d.y * post * w.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(d.z * post * w.z, d.w * post * w.w);
    uint2 u2;
    u2.x = *reinterpret_cast<uint32_t*>(&lo);
    u2.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + (size_t)row * DVD)[lane] = u2;
}

}  // namespace

int decode_rows_supported(int rows) { return decode_tc_rows_supported(rows); }

int decode_max_splits() { return MAX_COMBINE_SPLITS; }

int decode_ctas_per_sm() { return decode_tc_ctas_per_sm(); }

cudaError_t launch_decode(const KvParams& p, const KvTensorMaps& maps, cudaStream_t stream) {
    cudaError_t err = launch_decode_tc(p, maps, stream);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    const long long rows = (long long)p.batch * p.q_len * p.H;
    cfg.gridDim = dim3((unsigned)((rows + CWARPS - 1) / CWARPS));
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
