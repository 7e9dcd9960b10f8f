// Differential-attention forward against a key/value cache (decode and short
// query blocks), split over the keys.
//
// The new queries of a sequence are its last q_len tokens: with L cached keys
// (the new tokens included), query t (0-based among the new ones) sits at
// position L - q_len + t and, when causal, sees keys j <= L - q_len + t -- the
// bottom-right aligned mask triu(-inf, 1 + src_len - tgt_len) of the
// FlashDiffAttention review snippet ("Add an isolated implementation of
// FlashDiffAttention", alternative_forward), on the cache layout of the Llama
// gist ("LlamaDiffSdpaAttention.py", forward: past_key_value.update with k1, k2
// stacked).
//
// This path streams the whole cache once per call and does ~3 fused
// multiply-adds per byte for a single decoded token per kv head, so it is
// bound by HBM bandwidth: it runs on the CUDA cores, in two kernels:
//  1. split kernel: CTA (split s, kv head g, batch b) walks keys
//     [s * chunk, (s + 1) * chunk) in 64-key tiles (cp.async double buffer)
//     for all R = q_len * (H / Hkv) query rows that read kv head g, keeping per
//     row and component an online softmax (m, l) and an unnormalised O, and
//     writes them to the workspace;
//  2. combine kernel: per (b, query, head) merges the splits per component
//     (rescale by 2^(m_s - M), sum), forms O1/l1 - lambda O2/l2, the per-head
//     RMSNorm over dv, the weight and (1 - lambda_init), stores bf16.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103a_ptx.cuh"

namespace diffattn {
namespace {

constexpr int DK = 64;          // component dim d
constexpr int DVD = 128;        // value dim
constexpr int TK = 64;          // keys per tile
constexpr int NT = 128;         // threads per split CTA
constexpr int KROW = 136;       // padded K row (bf16): 272 B, conflict-free 16-byte reads
constexpr float LOG2E = 1.4426950408889634f;

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

// 16-byte async copy; bytes = 0 writes zeros without reading global memory.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int bytes) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

struct DecodeSmemLayout {
    static constexpr size_t k_tile = (size_t)TK * KROW * 2;
    static constexpr size_t v_tile = (size_t)TK * DVD * 2;
};

template <int R>
__global__ void __launch_bounds__(NT)
diffattn_decode_split_kernel(const KvParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    float* qs = reinterpret_cast<float*>(smem);                                     // [R][2 * DK]
    __nv_bfloat16* ks = reinterpret_cast<__nv_bfloat16*>(smem + (size_t)R * 2 * DK * 4);   // [2][TK][KROW]
    __nv_bfloat16* vs = ks + 2 * TK * KROW;                                          // [2][TK][DVD]
    float* ps = reinterpret_cast<float*>(vs + 2 * TK * DVD);                        // [R * 2][TK]
    float* alpha_s = ps + R * 2 * TK;                                                 // [R * 2]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = p.H / p.Hkv;
    const int L = p.cache_seqlens ? p.cache_seqlens[b] : p.capacity;
    // partial-result slots of this CTA's rows: row r = t * G + gh <-> (query t, head g * G + gh)
    auto slot = [&](int r) {
        const int t = r / G, gh = r % G;
        return (((size_t)b * p.q_len + t) * p.H + (g * G + gh)) * p.num_splits + split;
    };
    if (L < p.q_len || L > p.capacity) {
        if (tid == 0 && split == 0 && g == 0) atomicOr(p.error_word, kErrBadSeqlens);
        return;
    }
    const int q_off = L - p.q_len;  // position of the first new query
    const int k0 = split * p.chunk;
    const int k1 = min(k0 + p.chunk, L);
    if (k0 >= k1) {  // empty split: neutral partial (m = -inf, l = 0)
        for (int r = 0; r < R; ++r)
            for (int c = 0; c < 2; ++c) {
                const size_t sl = slot(r) * 2 + c;
                if (tid == 0) {
                    p.ws_ml[sl * 2] = -INFINITY;
                    p.ws_ml[sl * 2 + 1] = 0.f;
                }
                p.ws_o[sl * DVD + tid] = 0.f;
            }
        return;
    }

    // queries of the R rows, fp32 in shared memory
    for (int i = tid; i < R * 2 * DK; i += NT) {
        const int r = i / (2 * DK), e = i % (2 * DK);
        const int t = r / G, gh = r % G;
        const __nv_bfloat16* qrow =
            static_cast<const __nv_bfloat16*>(p.q) + (((size_t)b * p.q_len + t) * p.H + (g * G + gh)) * (2 * DK);
        qs[i] = __bfloat162float(qrow[e]);
    }

    const size_t kv_row = (size_t)p.Hkv;  // stride between keys, in heads
    const __nv_bfloat16* kbase = static_cast<const __nv_bfloat16*>(p.k) + ((size_t)b * p.capacity * kv_row + g) * (2 * DK);
    const __nv_bfloat16* vbase = static_cast<const __nv_bfloat16*>(p.v) + ((size_t)b * p.capacity * kv_row + g) * DVD;
    const int n_tiles = (k1 - k0 + TK - 1) / TK;

    auto load_tile = [&](int it, int buf) {
        const int kt = k0 + it * TK;
        // K: 64 rows x 256 B = 1024 chunks of 16 B; V: 64 rows x 256 B
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int ci = tid + i * NT;           // chunk index
            const int row = ci >> 4, col = (ci & 15) * 8;
            const int key = kt + row;
            const bool ok = key < k1;              // never read past the split (and the cache)
            const size_t src = ok ? (size_t)key * kv_row * (2 * DK) + col : 0;
            cp_async16(ks + (size_t)buf * TK * KROW + row * KROW + col, kbase + src, ok ? 16 : 0);
            const size_t vsrc = ok ? (size_t)key * kv_row * DVD + col : 0;
            cp_async16(vs + (size_t)buf * TK * DVD + row * DVD + col, vbase + vsrc, ok ? 16 : 0);
        }
        cp_async_commit();
    };

    // running state: warp w owns pairs pr = w, w + 4, ... (pair = row * 2 + component)
    constexpr int PAIRS = R * 2;
    constexpr int PPW = (PAIRS + 3) / 4;
    float m_run[PPW], l_run[PPW];
#pragma unroll
    for (int i = 0; i < PPW; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.f;
    }
    // P V: thread owns value columns 2*cp, 2*cp+1 for the keys of half kh of
    // each tile; the two halves are added once, at the end of the split.
    const int cp = tid & 63, kh = tid >> 6;
    float acc[PAIRS][2];
#pragma unroll
    for (int i = 0; i < PAIRS; ++i) acc[i][0] = acc[i][1] = 0.f;
    const float sl2 = p.scale * LOG2E;

    load_tile(0, 0);
    for (int it = 0; it < n_tiles; ++it) {
        const int buf = it & 1;
        if (it + 1 < n_tiles) {
            load_tile(it + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int kt = k0 + it * TK;
        // ---- scores: thread = (key j, component c); all R rows
        {
            const int j = tid & (TK - 1), c = tid >> 6;
            const __nv_bfloat16* krow = ks + (size_t)buf * TK * KROW + j * KROW + c * DK;
            uint64_t kf[DK / 2];  // packed (k[2i], k[2i+1])
#pragma unroll
            for (int e = 0; e < DK; e += 8) {
                const uint4 u = *reinterpret_cast<const uint4*>(krow + e);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    kf[e / 2 + i] = f2_pack(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
            }
            const int key = kt + j;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                // even and odd coordinates summed separately, in one packed multiply-add per pair
                const uint64_t* qr = reinterpret_cast<const uint64_t*>(qs + r * 2 * DK + c * DK);
                uint64_t s2 = f2_pack(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < DK / 2; ++e) s2 = ffma2(qr[e], kf[e], s2);
                const float2 sv = f2_unpack(s2);
                const int t = r / G;
                const bool vis = key < k1 && (!p.causal || key <= q_off + t);
                ps[(r * 2 + c) * TK + j] = vis ? (sv.x + sv.y) * sl2 : -INFINITY;
            }
        }
        __syncthreads();
        // ---- online softmax per pair (warp-wide over the 64 keys of the tile)
#pragma unroll
        for (int i = 0; i < PPW; ++i) {
            const int pr = warp + 4 * i;
            if (pr < PAIRS) {
                float* row = ps + pr * TK;
                const float x0 = row[lane], x1 = row[lane + 32];
                const float mt = warp_max(fmaxf(x0, x1));
                const float mn = fmaxf(m_run[i], mt);
                const float mref = mn == -INFINITY ? 0.f : mn;  // a fully masked tile leaves the state as is
                const float e0 = exp2f(x0 - mref), e1 = exp2f(x1 - mref);
                const float al = exp2f(m_run[i] - mref);
                row[lane] = e0;
                row[lane + 32] = e1;
                l_run[i] = l_run[i] * al + warp_sum(e0 + e1);
                m_run[i] = mn;
                if (lane == 0) alpha_s[pr] = al;
            }
        }
        __syncthreads();
        // ---- O += P V (probabilities as float4 broadcasts, values as bf16 pairs)
        {
            const uint32_t* vrow = reinterpret_cast<const uint32_t*>(vs + (size_t)buf * TK * DVD) + cp;
#pragma unroll
            for (int pr = 0; pr < PAIRS; ++pr) {
                acc[pr][0] *= alpha_s[pr];
                acc[pr][1] *= alpha_s[pr];
            }
            // (Packed fp32 pairs here, with the probabilities stored twice per key, measured
            // slower: the doubled probability traffic cost more than the halved FMA count.)
#pragma unroll 2
            for (int j = kh * (TK / 2); j < kh * (TK / 2) + TK / 2; j += 4) {
                float vx[4], vy[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const uint32_t w2 = vrow[(j + jj) * (DVD / 2)];
                    vx[jj] = __uint_as_float(w2 << 16);
                    vy[jj] = __uint_as_float(w2 & 0xffff0000u);
                }
#pragma unroll
                for (int pr = 0; pr < PAIRS; ++pr) {
                    const float4 pp = *reinterpret_cast<const float4*>(ps + pr * TK + j);
                    acc[pr][0] = fmaf(pp.x, vx[0], fmaf(pp.y, vx[1], fmaf(pp.z, vx[2], fmaf(pp.w, vx[3], acc[pr][0]))));
                    acc[pr][1] = fmaf(pp.x, vy[0], fmaf(pp.y, vy[1], fmaf(pp.z, vy[2], fmaf(pp.w, vy[3], acc[pr][1]))));
                }
            }
        }
        __syncthreads();  // the buffer is refilled by the next iteration's copy
    }
    // ---- partials: add the two key halves (through the K buffers, now idle), write O
    float* red = reinterpret_cast<float*>(ks);  // [PAIRS][DVD] floats <= 2 K buffers
    static_assert((size_t)PAIRS * DVD * 4 <= 2 * DecodeSmemLayout::k_tile, "reduction buffer");
    if (kh == 1) {
#pragma unroll
        for (int pr = 0; pr < PAIRS; ++pr) *reinterpret_cast<float2*>(red + pr * DVD + 2 * cp) = make_float2(acc[pr][0], acc[pr][1]);
    }
    __syncthreads();
    if (kh == 0) {
#pragma unroll
        for (int pr = 0; pr < PAIRS; ++pr) {
            const float2 o = *reinterpret_cast<const float2*>(red + pr * DVD + 2 * cp);
            *reinterpret_cast<float2*>(p.ws_o + (slot(pr >> 1) * 2 + (pr & 1)) * DVD + 2 * cp) =
                make_float2(acc[pr][0] + o.x, acc[pr][1] + o.y);
        }
    }
#pragma unroll
    for (int i = 0; i < PPW; ++i) {
        const int pr = warp + 4 * i;
        if (pr < PAIRS && lane == 0) {
            const size_t sl = slot(pr >> 1) * 2 + (pr & 1);
            p.ws_ml[sl * 2] = m_run[i];
            p.ws_ml[sl * 2 + 1] = l_run[i];
        }
    }
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

size_t split_smem_bytes(int R) {
    return (size_t)R * 2 * DK * 4 + 2 * DecodeSmemLayout::k_tile + 2 * DecodeSmemLayout::v_tile +
           (size_t)R * 2 * TK * 4 + (size_t)R * 2 * 4;
}

template <int R>
cudaError_t launch_split(const KvParams& p, cudaStream_t stream) {
    const size_t smem = split_smem_bytes(R);
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !attr_done[dev]) {
        err = cudaFuncSetAttribute(diffattn_decode_split_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem);
        if (err != cudaSuccess) return err;
        attr_done[dev] = true;
    }
    dim3 grid((unsigned)p.num_splits, (unsigned)p.Hkv, (unsigned)p.batch);
    diffattn_decode_split_kernel<R><<<grid, NT, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

int decode_rows_supported(int rows) { return rows == 1 || rows == 2 || rows == 4 || rows == 8 || rows == 16; }

int decode_max_splits() { return MAX_COMBINE_SPLITS; }

int decode_ctas_per_sm(int rows) {
    // 232448 bytes of shared memory per SM usable by blocks, 1 KB reserved per block
    const size_t per = split_smem_bytes(rows) + 1024;
    const int n = (int)(232448 / per);
    return n < 1 ? 1 : (n > 8 ? 8 : n);
}

cudaError_t launch_decode(const KvParams& p, cudaStream_t stream) {
    const int R = p.q_len * (p.H / p.Hkv);
    cudaError_t err;
    switch (R) {
        case 1: err = launch_split<1>(p, stream); break;
        case 2: err = launch_split<2>(p, stream); break;
        case 4: err = launch_split<4>(p, stream); break;
        case 8: err = launch_split<8>(p, stream); break;
        case 16: err = launch_split<16>(p, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (err != cudaSuccess) return err;
    diffattn_decode_combine_kernel<<<(unsigned)(p.batch * p.q_len * p.H), DVD, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace diffattn
