// Differential-attention forward against a key/value cache on the tensor cores
// (sm_103a): decode and short query blocks, split over the keys.
//
// The new queries of a sequence are its last q_len tokens: with L cached keys
// (the new tokens included), query t sits at position L - q_len + t and, when
// causal, sees keys j <= L - q_len + t -- the bottom-right aligned mask
// triu(-inf, 1 + src_len - tgt_len) of the FlashDiffAttention review snippet
// ("Add an isolated implementation of FlashDiffAttention", alternative_forward),
// on the cache layout of the Llama gist ("LlamaDiffSdpaAttention.py", forward:
// past_key_value.update with k1, k2 stacked).
//
// CTA (split s, kv head g, batch b) walks keys [s * chunk, (s + 1) * chunk) in
// 64-key tiles for the R = q_len * (H / Hkv) query rows that read kv head g
// (1 <= R <= 32), and writes per row and component the online-softmax state
// (m, l) and the unnormalised output O to the workspace; the combine kernel
// (decode_simt.cu) merges the splits and applies lambda and the RMSNorm.
//
// Both components in one pair of MMA chains. The query rows are stacked into
// two zero-padded boxes: box 1 holds Q1 of row r at row r, box 2 holds Q2 of
// row r at row 32 + r. Then
//   S = box1 K1^T + box2 K2^T          (M 128, N 64 keys, K 2 x 64)
// has S_1 of row r in TMEM lane r and S_2 of row r in lane 32 + r (every other
// product is with a zero row), and after the softmax
//   O += P V                           (M 128, N 128, K 64 keys, P from TMEM)
// accumulates O_1 and O_2 in the same lanes: an output row depends only on its
// own P row. The boxes hold rows 0-63 only (8 KB each): rows 64-127 of an
// M = 128 operand are the next 8 KB of shared memory (box 2, then a K box),
// whose products land in TMEM lanes 64-127, which nothing reads. The padding
// costs tensor work only; the path is bound by streaming the cache.
//
// Roles (128 threads):
//   warp 0  softmax of component 1 (TMEM lanes 0-31, rows r < R);
//   warp 1  softmax of component 2 (lanes 32-63);
//   warp 2  TMA producer (K1|K2 and V boxes of [64 keys x 64] per tile, 3 stages);
//   warp 3  TMEM allocator and MMA issuer.
// Tensor memory (256 columns, so two CTAs share an SM): S / P double-buffered
// at [0, 64) and [64, 128), O at [128, 256). S(j + 1) is issued before P(j) V,
// so the softmax of a tile overlaps the MMAs of its neighbours.
// Every wait is bounded; on a timeout the CTA records the error, lets its copies
// and MMAs in flight finish, frees TMEM and returns.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103a_ptx.cuh"

namespace diffattn {
namespace {

constexpr int TK = 64;                 // keys per tile
constexpr int HD = 64;                 // component dim d
constexpr int DV = 128;                // value dim
constexpr int STAGES = 3;
constexpr int MAX_ROWS = 32;
constexpr int NUM_THREADS = 128;
constexpr int SOFTMAX_WARPS = 2, PRODUCER_WARP = 2, MMA_WARP = 3;
constexpr uint32_t QBOX_BYTES = 64 * HD * 2;         // one component's stacked query box: 8 KB
constexpr uint32_t KVBOX_BYTES = TK * 64 * 2;        // [64 keys x 64] bf16: 8 KB
constexpr uint32_t K_BYTES = 2 * KVBOX_BYTES;
constexpr uint32_t V_BYTES = 2 * KVBOX_BYTES;
constexpr uint32_t STAGE_BYTES = K_BYTES + V_BYTES;
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_STAGE0 = 2 * QBOX_BYTES;
constexpr uint32_t OFF_MISC = OFF_STAGE0 + STAGES * STAGE_BYTES;
constexpr uint32_t MISC_BYTES = 256;
// No alignment slack (two CTAs per SM need every byte): the kernel checks that
// the dynamic shared memory starts on a 1024-byte boundary (the swizzle atoms'
// alignment) and reports an error otherwise.
constexpr uint32_t SMEM_BYTES = OFF_MISC + MISC_BYTES;
static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs per SM (228 KB, 1 KB reserved per CTA)");
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t COL_O = 128;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units; P stays below 2^8
constexpr float LOG2E = 1.4426950408889634f;

struct Misc {
    uint64_t k_full[STAGES], v_full[STAGES], kv_empty[STAGES];
    uint64_t s_full[2], p_ready[2];
    uint64_t pv_done, o_full;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Misc) <= MISC_BYTES, "misc area too small");

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) { return smem_desc_sw128(saddr, 16, 1024); }
// MN-major value operand: 64-column halves one box apart, 8-key groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_value(uint32_t saddr) { return smem_desc_sw128(saddr, KVBOX_BYTES, 1024); }
__device__ __forceinline__ bool warp_all(bool p) { return __all_sync(0xffffffffu, p); }

__global__ void __launch_bounds__(NUM_THREADS)
diffattn_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const KvParams p) {
    extern __shared__ uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(p.error_word, kErrLayout);
        return;
    }
    Misc& ms = *reinterpret_cast<Misc*>(smem + OFF_MISC);
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    // Launched as a programmatic dependent of the previous kernel on the stream:
    // nothing is read before that kernel has completed. The combine kernel may
    // then be placed as soon as every split CTA is running (it waits for this
    // grid to complete before it reads a partial).
    griddep_wait();
    griddep_launch_dependents();
    const int G = p.H / p.Hkv;
    const int R = p.q_len * G;
    const int L = p.cache_seqlens ? p.cache_seqlens[b] : p.capacity;
    // partial-result slot of row r = t * G + gh <-> (query t, head g * G + gh)
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
    if (k0 >= k1) {  // empty split: neutral partial (m = -inf, l = 0, O = 0)
        for (int i = tid; i < R * 2; i += NUM_THREADS) {
            const size_t sl = slot(i >> 1) * 2 + (i & 1);
            p.ws_ml[sl * 2] = -INFINITY;
            p.ws_ml[sl * 2 + 1] = 0.f;
        }
        for (int i = tid; i < R * 2 * (DV / 4); i += NUM_THREADS) {
            const int pr = i / (DV / 4), c4 = i % (DV / 4);
            reinterpret_cast<float4*>(p.ws_o + (slot(pr >> 1) * 2 + (pr & 1)) * DV)[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    const int n_tiles = (k1 - k0 + TK - 1) / TK;

    auto bar_k_full = [&](int s) { return smem_u32(&ms.k_full[s]); };
    auto bar_v_full = [&](int s) { return smem_u32(&ms.v_full[s]); };
    auto bar_kv_empty = [&](int s) { return smem_u32(&ms.kv_empty[s]); };
    auto bar_s_full = [&](int bf) { return smem_u32(&ms.s_full[bf]); };
    auto bar_p_ready = [&](int bf) { return smem_u32(&ms.p_ready[bf]); };
    const uint32_t bar_pv_done = smem_u32(&ms.pv_done), bar_o_full = smem_u32(&ms.o_full);
    auto sk = [&](int s) { return sbase + OFF_STAGE0 + (uint32_t)s * STAGE_BYTES; };
    auto sv = [&](int s) { return sbase + OFF_STAGE0 + (uint32_t)s * STAGE_BYTES + K_BYTES; };

    // The producer lane initialises the barriers and at once issues the first
    // STAGES K / V tiles (fresh stages: nothing to wait for), before the query
    // boxes are filled and the CTA meets at its barrier: the cache rows are in
    // flight while the queries are gathered.
    const int row0 = b * p.capacity + k0;
    const int n_pre = min(n_tiles, STAGES);
    auto issue_kv = [&](int j, uint64_t pol) {
        const int s = j % STAGES;
        const int row = row0 + j * TK;  // rows past the split are masked, past the cache read as zero
        mbar_arrive_expect_tx(bar_k_full(s), K_BYTES);
        tma_load_2d(sk(s), &tm_k, bar_k_full(s), g * 2 * HD, row, pol);
        tma_load_2d(sk(s) + KVBOX_BYTES, &tm_k, bar_k_full(s), g * 2 * HD + HD, row, pol);
        mbar_arrive_expect_tx(bar_v_full(s), V_BYTES);
        tma_load_2d(sv(s), &tm_v, bar_v_full(s), g * DV, row, pol);
        tma_load_2d(sv(s) + KVBOX_BYTES, &tm_v, bar_v_full(s), g * DV + 64, row, pol);
    };
    if (warp == PRODUCER_WARP && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_k_full(s), 1);
            mbar_init(bar_v_full(s), 1);
            mbar_init(bar_kv_empty(s), 1);
        }
        for (int bf = 0; bf < 2; ++bf) {
            mbar_init(bar_s_full(bf), 1);
            mbar_init(bar_p_ready(bf), 32 * SOFTMAX_WARPS);
        }
        mbar_init(bar_pv_done, 1);
        mbar_init(bar_o_full, 1);
        ms.abort_flag = 0;
        fence_barrier_init();
        const uint64_t pol = l2_policy_evict_first();  // the cache is streamed once
        for (int j = 0; j < n_pre; ++j) issue_kv(j, pol);
    }

    // ---- stacked query boxes (128-byte swizzle: row x at x * 128 B, 16-byte
    // chunk c of the row at physical chunk c ^ (x % 8)); every other row zero
    {
        const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q);
        for (int i = tid; i < 2 * 64 * 8; i += NUM_THREADS) {
            const int box = i >> 9, x = (i >> 3) & 63, pc = i & 7;
            const int lc = pc ^ (x & 7);
            const int r = x - 32 * box;  // box 1: rows 0..R-1; box 2: rows 32..32+R-1
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r >= 0 && r < R) {
                const int t = r / G, gh = r % G;
                const __nv_bfloat16* qrow = qb + (((size_t)b * p.q_len + t) * p.H + (g * G + gh)) * (2 * HD);
                v = *reinterpret_cast<const uint4*>(qrow + box * HD + lc * 8);
            }
            *reinterpret_cast<uint4*>(smem + OFF_Q + (uint32_t)box * QBOX_BYTES + (uint32_t)x * 128u + (uint32_t)pc * 16u) = v;
        }
        fence_proxy_async_smem();  // the boxes, visible to the tensor cores
    }

    if (warp == MMA_WARP) tmem_alloc(smem_u32(&ms.tmem_base), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;
    const AbortState ab{&ms.abort_flag, p.error_word, p.timeout_ns};

    if (warp == PRODUCER_WARP) {
        // ================================================= TMA producer ===
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();  // the cache is streamed once
            int issued = n_pre;  // issued in the prologue
            for (int j = n_pre; j < n_tiles; ++j) {
                if (!mbar_wait(bar_kv_empty(j % STAGES), ((uint32_t)(j / STAGES) & 1u) ^ 1u, ab)) break;
                issue_kv(j, pol);
                issued = j + 1;
            }
            for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j) {
                const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
                mbar_wait_drain(bar_k_full(j % STAGES), ph, p.timeout_ns);
                mbar_wait_drain(bar_v_full(j % STAGES), ph, p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ==================================================== MMA issuer ===
        constexpr uint32_t idesc_s = idesc_bf16_f32(128, TK, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, DV, true);
        constexpr uint64_t KSTEP = 32 >> 4, VSTEP = (16 * 128) >> 4, STG = STAGE_BYTES >> 4;
        constexpr uint64_t QBOX = QBOX_BYTES >> 4, KBOX = KVBOX_BYTES >> 4;
        const uint64_t qdesc = desc_kmajor(sbase + OFF_Q), kdesc = desc_kmajor(sk(0)), vdesc = desc_value(sv(0));
        auto issue_s = [&](int j) {  // S(j) = box1 K1^T + box2 K2^T into buffer j & 1
            const uint32_t d = tmem + (uint32_t)(j & 1) * TK;
            const uint64_t kb = kdesc + (uint64_t)(j % STAGES) * STG;
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    mma_ss_elect(d, qdesc + c * QBOX + kk * KSTEP, kb + c * KBOX + kk * KSTEP, idesc_s,
                                 (c > 0 || kk > 0) ? 1u : 0u);
            mma_commit_elect(bar_s_full(j & 1));
        };
        bool ok = warp_all(mbar_wait(bar_k_full(0), 0, ab));
        if (ok) {
            tc_fence_after();
            issue_s(0);
        }
        for (int j = 0; ok && j < n_tiles; ++j) {
            const int s = j % STAGES;
            if (j + 1 < n_tiles) {  // the next scores go into the other buffer, whose P was read by P(j-1) V
                if (!(ok = warp_all(mbar_wait(bar_k_full((j + 1) % STAGES), (uint32_t)((j + 1) / STAGES) & 1u, ab))))
                    break;
                tc_fence_after();
                issue_s(j + 1);
            }
            if (!(ok = warp_all(mbar_wait(bar_v_full(s), (uint32_t)(j / STAGES) & 1u, ab)))) break;
            const int kt = k0 + j * TK;
            if (kt + TK > k1) {
                // keys past the split end: P is zero there, but the rows past the
                // sequence may hold anything (0 x NaN is NaN), so they are cleared
                const int first = k1 - kt;
                for (int i = lane; i < 2 * (TK - first) * 8; i += 32) {
                    const int box = i / ((TK - first) * 8), rr = first + (i / 8) % (TK - first), ch = i % 8;
                    *reinterpret_cast<uint4*>(smem + (sv(s) - sbase) + (uint32_t)box * KVBOX_BYTES + (uint32_t)rr * 128u +
                                              (uint32_t)ch * 16u) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (!(ok = warp_all(mbar_wait(bar_p_ready(j & 1), (uint32_t)(j >> 1) & 1u, ab)))) break;
            tc_fence_after();
            const uint32_t a = tmem + (uint32_t)(j & 1) * TK;  // P: bf16 pairs in the first 32 columns
            const uint64_t vb = vdesc + (uint64_t)s * STG;
#pragma unroll
            for (int kk = 0; kk < TK / 16; ++kk)
                mma_ts_elect(tmem + COL_O, a + kk * 8, vb + kk * VSTEP, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit_elect(bar_kv_empty(s));
            mma_commit_elect(bar_pv_done);
        }
        mma_commit_elect(bar_o_full);
        mbar_wait_drain(bar_o_full, 0, p.timeout_ns);
        __syncwarp();
    } else {
        // ======================================== softmax (warps 0, 1) ===
        const int c = warp;                   // component
        const int r = lane;                   // query row of this lane (TMEM lane 32 c + r)
        const bool row_ok = r < R;
        const int t = row_ok ? r / G : 0;
        const uint32_t lane_off = (uint32_t)(32 * c) << 16;
        // keys < lim are visible to this row
        const int lim = row_ok ? (p.causal ? min(k1, q_off + t + 1) : k1) : k0;
        const float sl2 = p.scale * LOG2E;
        const uint64_t sl2p = f2_pack(sl2, sl2);
        float m = -INFINITY;  // running max of scores * scale * log2(e); -inf until a key is visible
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int bf = j & 1;
            if (!(ok = warp_all(mbar_wait(bar_s_full(bf), (uint32_t)(j >> 1) & 1u, ab)))) break;
            tc_fence_after();
            const uint32_t t_s = tmem + lane_off + (uint32_t)bf * TK;
            float x[TK];
            {
                uint32_t sr[2][32];
                tmem_ld32(t_s, sr[0]);
                tmem_ld32(t_s + 32, sr[1]);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < TK; ++e) x[e] = __uint_as_float(sr[e >> 5][e & 31]);
            }
            const int kt = k0 + j * TK;
            if (kt + TK > lim) {
#pragma unroll
                for (int e = 0; e < TK; ++e)
                    if (kt + e >= lim) x[e] = -INFINITY;
            }
            float mx0 = fmaxf(x[0], x[1]), mx1 = fmaxf(x[2], x[3]), mx2 = fmaxf(x[4], x[5]), mx3 = fmaxf(x[6], x[7]);
#pragma unroll
            for (int e = 8; e < TK; e += 8) {
                mx0 = fmax3(mx0, x[e], x[e + 1]);
                mx1 = fmax3(mx1, x[e + 2], x[e + 3]);
                mx2 = fmax3(mx2, x[e + 4], x[e + 5]);
                mx3 = fmax3(mx3, x[e + 6], x[e + 7]);
            }
            const float m_tile = fmax3(fmaxf(mx0, mx1), mx2, mx3) * sl2;
            float alpha = 1.f;
            if (m_tile > m + RESCALE_THRESHOLD) {  // false while nothing is visible (m_tile = -inf)
                alpha = ex2_approx(m - m_tile);    // 0 when m = -inf
                m = m_tile;
            }
            // O holds P V through an earlier tile; rescaling it waits for P(j-1) V
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                if (!(ok = warp_all(mbar_wait(bar_pv_done, (uint32_t)(j - 1) & 1u, ab)))) break;
                tc_fence_after();
#pragma unroll
                for (int ch = 0; ch < DV / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_off + COL_O + ch * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tmem + lane_off + COL_O + ch * 32, o);
                }
            }
            const float mref = m == -INFINITY ? 0.f : m;  // nothing visible yet: every P is 0
            const uint64_t nmp = f2_pack(-mref, -mref);
            uint64_t sa = 0, sb = 0;
#pragma unroll
            for (int ch = 0; ch < TK / 32; ++ch) {
#pragma unroll
                for (int e = ch * 32; e < ch * 32 + 32; e += 4) {
                    const float2 u0 = f2_unpack(ffma2(f2_pack(x[e], x[e + 1]), sl2p, nmp));
                    const float2 u1 = f2_unpack(ffma2(f2_pack(x[e + 2], x[e + 3]), sl2p, nmp));
                    x[e] = ex2_approx(u0.x);
                    x[e + 1] = ex2_approx(u0.y);
                    x[e + 2] = ex2_approx(u1.x);
                    x[e + 3] = ex2_approx(u1.y);
                    sa = fadd2(sa, f2_pack(x[e], x[e + 1]));
                    sb = fadd2(sb, f2_pack(x[e + 2], x[e + 3]));
                }
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(x[ch * 32 + 2 * i], x[ch * 32 + 2 * i + 1]);
                tmem_st16(t_s + ch * 16, pk);
            }
            const float2 sab = f2_unpack(fadd2(sa, sb));
            l = l * alpha + (sab.x + sab.y);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar_p_ready(bf));
        }
        // ---- partials of this component's rows
        ok = warp_all(ok && mbar_wait(bar_o_full, 0, ab));
        if (ok) {
            tc_fence_after();
            const size_t sl = row_ok ? slot(r) * 2 + c : 0;
            if (row_ok) {
                p.ws_ml[sl * 2] = m;
                p.ws_ml[sl * 2 + 1] = l;
            }
#pragma unroll
            for (int ch = 0; ch < DV / 32; ++ch) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + COL_O + ch * 32, o);
                tmem_wait_ld();
                if (row_ok) {
                    float4* dst = reinterpret_cast<float4*>(p.ws_o + sl * DV + ch * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                             __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
                }
            }
        }
    }

    // ---- teardown: all TMEM traffic of this CTA is complete -----------------
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

int decode_tc_rows_supported(int rows) { return rows >= 1 && rows <= MAX_ROWS; }

int decode_tc_ctas_per_sm() { return 2; }

cudaError_t launch_decode_tc(const KvParams& p, const KvTensorMaps& maps, cudaStream_t stream) {
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !attr_done[dev]) {
        err = cudaFuncSetAttribute(diffattn_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)SMEM_BYTES);
        if (err != cudaSuccess) return err;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.num_splits, (unsigned)p.Hkv, (unsigned)p.batch);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, diffattn_decode_tc_kernel, maps.k, maps.v, p);
}

}  // namespace diffattn
