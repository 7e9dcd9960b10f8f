// Backward pass of the differential-attention forward on sm_103a (bf16
// operands, fp32 accumulation in tensor memory), d = 64, dv = 128.
//
// With D = O1 - lambda O2 (O_c = softmax(s Q_c K_c^T) V) and dD the gradient of
// the pre-norm output (from the per-row preprocessing kernel), the two
// components see dO_1 = dD and dO_2 = -lambda dD, so one product dP = dD V^T
// serves both, and per (query row i, key j):
//   P_c  = 2^(s log2(e) <Q_c[i], K_c[j]> - lse_c[i])                (saved by the forward)
//   dS_1 = P_1 (dP - delta_1[i]),  dS_2 = -lambda P_2 (dP - delta_2[i])
//   (the kernels carry dS / s and apply s once to dQ and dK in their epilogues)
//   delta_c[i] = <dD[i], O_c[i] / l_c[i]>                        (preprocessing)
//   dQ_c += s dS_c K_c,  dK_c += s dS_c^T Q_c,  dV += (P_1 - lambda P_2)^T dD
// (the derivative of softmax(...) V through "DiffTransformer.py",
// MultiHeadDifferentialAttention.forward, in the output-difference form of
// "LlamaDiffSdpaAttention.py", forward).
//
// Two kernels, each a TMA producer warp, an MMA warp (elected lane issues) and
// one warpgroup of 128 threads that owns one TMEM lane each:
//   dQ kernel : CTA = 128 query rows of one head; walks the visible 128-key
//               tiles. TMEM: S1 [0,128), S2 [128,256), dP [256,384),
//               dQ1 [384,448), dQ2 [448,512); dS_c (bf16) over S_c.
//   dKV kernel: CTA = 128 keys of one kv head; walks the heads of its group and
//               the 64-row query blocks that see its keys. With keys as the MMA
//               rows: S_c^T [0,64) [64,128), dP^T [128,192), dS_1^T | dS_2^T
//               (bf16 pairs) [192,256), dV [256,384), dK1 [384,448), dK2 [448,512);
//               P_1 - lambda P_2 (bf16) goes through shared memory.
// Every wait is bounded; on a timeout a CTA records the error, lets its copies
// and MMAs land, frees TMEM and returns.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103a_ptx.cuh"

namespace diffattn {
namespace {

constexpr int HD = 64;
constexpr int DV = 128;
constexpr uint32_t ROW = 128;                      // bytes of one swizzled row (64 bf16)
constexpr int NT = 320;                            // 8 compute warps (two warpgroups) + producer + MMA
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;

__device__ __forceinline__ uint64_t desc_k(uint32_t a) { return smem_desc_sw128(a, 16, 1024); }
// MN-major operand whose N extent is split in 64-wide boxes `box` bytes apart.
__device__ __forceinline__ uint64_t desc_mn(uint32_t a, uint32_t box) { return smem_desc_sw128(a, box, 1024); }
__device__ __forceinline__ bool warp_all(bool p) { return __all_sync(0xffffffffu, p); }

// ---- sequence bounds (uniform over the CTA); false: nothing to do / bad lengths
__device__ __forceinline__ bool seq_bounds(const BwdParams& p, int seq, int* start, int* len) {
    if (p.cu_seqlens != nullptr) {
        const int s0 = p.cu_seqlens[seq], s1 = p.cu_seqlens[seq + 1];
        const bool bad = s0 < 0 || s1 < s0 || s1 > p.total_tokens || s1 - s0 > p.max_seqlen ||
                         (seq == 0 && s0 != 0) || (seq == p.num_seqs - 1 && s1 != p.total_tokens);
        if (bad) {
            if (threadIdx.x == 0) atomicOr(p.error_word, kErrBadSeqlens);
            return false;
        }
        *start = s0;
        *len = s1 - s0;
    } else {
        *start = seq * p.seqlen;
        *len = p.seqlen;
    }
    return true;
}

// =============================================================== dQ ===
// One thread (= one query row) and 32 keys: dS_1, dS_2 as bf16 pairs from S_1,
// S_2, dP and the row's (lse_1, lse_2, delta_1, delta_2). MASK zeroes keys at or
// past `nvis` (the number of visible keys in this group of 32, any value).
// Adjacent keys go through packed fp32 pairs (half the multiply/add
// instructions of the scalar form); the second component's factor
// lambda (delta_2 - dP) is one fused multiply-add, -lambda dP + lambda delta_2.
template <bool MASK>
__device__ __forceinline__ void dq_keys32(const uint32_t (&s1)[32], const uint32_t (&s2)[32],
                                          const uint32_t (&dp)[32], const float4 rs, float lam, float sl2, float sc,
                                          int nvis, uint32_t (&d1)[16], uint32_t (&d2)[16]) {
    // rs holds the row's statistics negated: (-lse_1, -lse_2, -delta_1, -delta_2)
    const uint64_t sl2p = f2_pack(sl2, sl2), nl1 = f2_pack(rs.x, rs.x), nl2 = f2_pack(rs.y, rs.y);
    const uint64_t nd1 = f2_pack(rs.z, rs.z), nlam = f2_pack(-lam, -lam), lamd2 = f2_pack(-lam * rs.w, -lam * rs.w);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float2 x1 = f2_unpack(ffma2(f2_pack(__uint_as_float(s1[i]), __uint_as_float(s1[i + 1])), sl2p, nl1));
        const float2 x2 = f2_unpack(ffma2(f2_pack(__uint_as_float(s2[i]), __uint_as_float(s2[i + 1])), sl2p, nl2));
        const uint64_t p1 = f2_pack(ex2_approx(x1.x), ex2_approx(x1.y));
        const uint64_t p2 = f2_pack(ex2_approx(x2.x), ex2_approx(x2.y));
        const uint64_t pp = f2_pack(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1]));
        float2 a = f2_unpack(fmul2(p1, fadd2(pp, nd1)));          // dS_1 / s
        float2 b = f2_unpack(fmul2(p2, ffma2(pp, nlam, lamd2)));  // dS_2 / s
        if (MASK) {
            const bool v0 = i < nvis, v1 = i + 1 < nvis;
            a.x = v0 ? a.x : 0.f;
            a.y = v1 ? a.y : 0.f;
            b.x = v0 ? b.x : 0.f;
            b.y = v1 ? b.y : 0.f;
        }
        d1[i / 2] = pack_bf16x2(a.x, a.y);
        d2[i / 2] = pack_bf16x2(b.x, b.y);
    }
}

// K and V have rings of their own: a tile's V is free once its dP MMAs have run,
// its K only after its dQ steps, so three K stages and two V stages give each
// load about two tiles of lead (one shared two-stage ring left the MMA warp
// waiting ~0.8 us a tile for the next tile's rows).
namespace dq {
constexpr int BM = 128, BN = 128, KSTAGES = 3, VSTAGES = 2;
constexpr uint32_t BOX = 128 * ROW;                // [128 x 64] bf16 box: 16 KB
constexpr uint32_t OFF_Q = 0;                      // Q1 | Q2
constexpr uint32_t OFF_DD = 2 * BOX;               // dD (two 64-column halves)
constexpr uint32_t OFF_K = 4 * BOX;                // K stages: K1 | K2
constexpr uint32_t OFF_V = OFF_K + KSTAGES * 2 * BOX;  // V stages: V lo | V hi
constexpr uint32_t OFF_MISC = OFF_V + VSTAGES * 2 * BOX;
constexpr uint32_t SMEM = 1024 + OFF_MISC + 512;
static_assert(SMEM <= 232448, "smem");
struct Misc {
    uint64_t q_full, k_full[KSTAGES], k_empty[KSTAGES], v_full[VSTAGES], v_empty[VSTAGES], s_ready[2], ds_ready[2],
        dq_done;
    uint32_t tmem;
    int abort_flag;
};
}  // namespace dq

__global__ void __launch_bounds__(NT, 1)
diffattn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dd,
                       const BwdParams p) {
    using namespace dq;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc& ms = *reinterpret_cast<Misc*>(smem + OFF_MISC);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grid (head group x query tile x head in group, 1, sequence), or with the tiles
    // outermost (head, sequence, query tile); either way the longest query tiles of a
    // sequence are scheduled first. A group's K / V (sized by the host) stays in L2
    // while its CTAs stream it.
    const bool outer = p.dq_tiles_outer != 0;
    int h, seq, qt;
    if (outer) {
        h = blockIdx.x, seq = blockIdx.y, qt = gridDim.z - 1 - blockIdx.z;
    } else {
        const int n_qt = (p.max_seqlen + BM - 1) / BM, hg = p.dq_group_heads;
        const int grp = (int)blockIdx.x / (n_qt * hg), rem = (int)blockIdx.x - grp * (n_qt * hg);
        h = grp * hg + rem % hg, seq = blockIdx.z, qt = n_qt - 1 - rem / hg;
    }
    int start = 0, len = 0;
    if (!seq_bounds(p, seq, &start, &len)) return;
    if (qt * BM >= len) return;
    const int n_kv = p.causal ? qt + 1 : (len + BN - 1) / BN;
    const int g = h / (p.H / p.Hkv);

    const uint32_t b_q = smem_u32(&ms.q_full), b_dq = smem_u32(&ms.dq_done);
    auto b_s = [&](int w) { return smem_u32(&ms.s_ready[w]); };
    auto b_ds = [&](int w) { return smem_u32(&ms.ds_ready[w]); };
    auto b_kf = [&](int s) { return smem_u32(&ms.k_full[s]); };
    auto b_ke = [&](int s) { return smem_u32(&ms.k_empty[s]); };
    auto b_vf = [&](int s) { return smem_u32(&ms.v_full[s]); };
    auto b_ve = [&](int s) { return smem_u32(&ms.v_empty[s]); };
    if (warp == PRODUCER_WARP && lane == 0) {
        mbar_init(b_q, 1);
        for (int s = 0; s < KSTAGES; ++s) {
            mbar_init(b_kf(s), 1);
            mbar_init(b_ke(s), 1);
        }
        for (int s = 0; s < VSTAGES; ++s) {
            mbar_init(b_vf(s), 1);
            mbar_init(b_ve(s), 1);
        }
        mbar_init(b_s(0), 1);
        mbar_init(b_s(1), 1);
        mbar_init(b_ds(0), 128);
        mbar_init(b_ds(1), 128);
        mbar_init(b_dq, 1);
        ms.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == MMA_WARP) tmem_alloc(smem_u32(&ms.tmem), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem;
    const AbortState ab{&ms.abort_flag, p.error_word, p.timeout_ns};

    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            const int row_q = start + qt * BM;
            mbar_arrive_expect_tx(b_q, 4 * BOX);
            tma_load_2d(sb + OFF_Q, &tm_q, b_q, h * 2 * HD, row_q, pol);
            tma_load_2d(sb + OFF_Q + BOX, &tm_q, b_q, h * 2 * HD + HD, row_q, pol);
            tma_load_2d(sb + OFF_DD, &tm_dd, b_q, h * DV, row_q, pol);
            tma_load_2d(sb + OFF_DD + BOX, &tm_dd, b_q, h * DV + 64, row_q, pol);
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int sk = j % KSTAGES, sv = j % VSTAGES;
                const int row = start + j * BN;
                if (j + 2 < n_kv) {  // two tiles ahead into L2, so that their loads find them there
                    const int row2 = row + 2 * BN;
                    tma_prefetch_l2_2d(&tm_k, g * 2 * HD, row2);
                    tma_prefetch_l2_2d(&tm_k, g * 2 * HD + HD, row2);
                    tma_prefetch_l2_2d(&tm_v, g * DV, row2);
                    tma_prefetch_l2_2d(&tm_v, g * DV + 64, row2);
                }
                if (!mbar_wait(b_ke(sk), ((uint32_t)(j / KSTAGES) & 1u) ^ 1u, ab)) break;
                const uint32_t kst = sb + OFF_K + (uint32_t)sk * 2 * BOX;
                mbar_arrive_expect_tx(b_kf(sk), 2 * BOX);
                tma_load_2d(kst, &tm_k, b_kf(sk), g * 2 * HD, row, pol);
                tma_load_2d(kst + BOX, &tm_k, b_kf(sk), g * 2 * HD + HD, row, pol);
                k_issued = j + 1;
                if (!mbar_wait(b_ve(sv), ((uint32_t)(j / VSTAGES) & 1u) ^ 1u, ab)) break;
                const uint32_t vst = sb + OFF_V + (uint32_t)sv * 2 * BOX;
                mbar_arrive_expect_tx(b_vf(sv), 2 * BOX);
                tma_load_2d(vst, &tm_v, b_vf(sv), g * DV, row, pol);
                tma_load_2d(vst + BOX, &tm_v, b_vf(sv), g * DV + 64, row, pol);
                v_issued = j + 1;
            }
            mbar_wait_drain(b_q, 0, p.timeout_ns);
            for (int j = k_issued > KSTAGES ? k_issued - KSTAGES : 0; j < k_issued; ++j)
                mbar_wait_drain(b_kf(j % KSTAGES), (uint32_t)(j / KSTAGES) & 1u, p.timeout_ns);
            for (int j = v_issued > VSTAGES ? v_issued - VSTAGES : 0; j < v_issued; ++j)
                mbar_wait_drain(b_vf(j % VSTAGES), (uint32_t)(j / VSTAGES) & 1u, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // Two 64-key halves per tile, pipelined: as soon as warpgroup h has written
        // dS of half h, its dQ steps go out and then the scores of half h of the next
        // tile, which overwrite only half h's columns (the pipe runs in issue order,
        // so the dQ steps have read dS before the new scores land).
        constexpr uint32_t id_s = idesc_bf16_f32(128, 64, false);    // S_c, dP of a half: both operands K-major
        constexpr uint32_t id_dq = idesc_bf16_f32(128, 64, true);    // dQ_c: B = K_c is MN-major (d contiguous)
        const uint64_t dq_q = desc_k(sb + OFF_Q), dq_dd = desc_k(sb + OFF_DD);
        const uint64_t dk0 = desc_k(sb + OFF_K), dkm = desc_mn(sb + OFF_K, BOX), dv0 = desc_k(sb + OFF_V);
        constexpr uint64_t KS = 32 >> 4, BX = BOX >> 4, KR = (16 * ROW) >> 4, SG2 = (2 * BOX) >> 4;
        constexpr uint64_t HK = (64 * ROW) >> 4;  // 64 key rows of a K-major box
        // S_c = Q_c K_c^T and dP = dD V^T for keys [64 h, 64 h + 64) of tile t
        auto issue_sdp = [&](int t, int h) {
            const uint64_t st_k = dk0 + (uint64_t)(t % KSTAGES) * SG2 + (uint64_t)h * HK;
            const uint64_t st_v = dv0 + (uint64_t)(t % VSTAGES) * SG2 + (uint64_t)h * HK;
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss_elect(tmem + c * 128 + 64 * h, dq_q + c * BX + kk * KS, st_k + c * BX + kk * KS, id_s,
                                 kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // K = dv = 128 over the two 64-column halves of dD and of V
                mma_ss_elect(tmem + 256 + 64 * h, dq_dd + (kk >> 2) * BX + (kk & 3) * KS,
                             st_v + (kk >> 2) * BX + (kk & 3) * KS, id_s, kk > 0);
            mma_commit_elect(b_s(h));
            if (h == 1) mma_commit_elect(b_ve(t % VSTAGES));  // both dP halves of tile t issued
        };
        auto kv_ready = [&](int t) {
            return warp_all(mbar_wait(b_kf(t % KSTAGES), (uint32_t)(t / KSTAGES) & 1u, ab)) &&
                   warp_all(mbar_wait(b_vf(t % VSTAGES), (uint32_t)(t / VSTAGES) & 1u, ab));
        };
        bool ok = warp_all(mbar_wait(b_q, 0, ab)) && kv_ready(0);
        if (ok) {
            tc_fence_after();
            issue_sdp(0, 0);
            issue_sdp(0, 1);
        }
        for (int j = 0; ok && j < n_kv; ++j) {
            const bool has_next = j + 1 < n_kv;
            const uint64_t st_km = dkm + (uint64_t)(j % KSTAGES) * SG2;
            for (int h = 0; h < 2; ++h) {
                if (!(ok = warp_all(mbar_wait(b_ds(h), (uint32_t)j & 1u, ab)))) break;
                tc_fence_after();
                // dQ_c += dS_c K_c over keys [64 h, 64 h + 64): A = dS_c (bf16 in TMEM, at column
                // 64 h + 8 (kk % 4) for keys 16 kk..), B = K_c rows (MN-major)
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
                        mma_ts_elect(tmem + 384 + c * 64, tmem + c * 128 + 64 * h + 8 * (kk & 3), st_km + c * BX + kk * KR,
                                     id_dq, (j > 0 || kk > 0) ? 1u : 0u);
                }
                if (has_next) {
                    if (h == 0 && !(ok = kv_ready(j + 1))) break;
                    tc_fence_after();
                    issue_sdp(j + 1, h);
                }
            }
            if (!ok) break;
            mma_commit_elect(b_ke(j % KSTAGES));  // every MMA reading tile j's K has been issued
        }
        mma_commit_elect(b_dq);
        mbar_wait_drain(b_dq, 0, p.timeout_ns);
        __syncwarp();
    } else {
        // ============================================== compute warpgroups ===
        // Warpgroup w handles keys [64 w, 64 w + 64) of every tile; thread = query row.
        const int w = warp >> 2;
        const int r = (warp & 3) * 32 + lane;  // query row in the tile = TMEM lane
        const uint32_t lo = (uint32_t)((warp & 3) * 32) << 16;
        const int qi = qt * BM + r;
        const bool row_ok = qi < len;
        const size_t grow = (size_t)(start + (row_ok ? qi : 0));
        float4 rs = make_float4(0.f, 0.f, 0.f, 0.f);  // -lse1, -lse2, -delta1, -delta2
        if (row_ok) rs = reinterpret_cast<const float4*>(p.rowstat)[(size_t)h * p.total_tokens + grow];
        const float lam = p.lambda[h * p.lambda_stride];
        const float sl2 = p.scale_log2, sc = p.scale;
        const int lim = row_ok ? (p.causal ? min(qi + 1, len) : len) : 0;  // keys < lim are visible
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            if (!(ok = warp_all(mbar_wait(b_s(w), (uint32_t)j & 1u, ab)))) break;
            tc_fence_after();
            const int kb = j * BN;
            // masking only on tiles where some row of the warp has keys past its limit
            const bool need_mask = __any_sync(0xffffffffu, kb + BN > lim);
#pragma unroll 1
            for (int ch = 2 * w; ch < 2 * w + 2; ++ch) {
                uint32_t s1[32], s2[32], dp[32];
                tmem_ld32(tmem + lo + ch * 32, s1);
                tmem_ld32(tmem + lo + 128 + ch * 32, s2);
                tmem_ld32(tmem + lo + 256 + ch * 32, dp);
                tmem_wait_ld();
                uint32_t d1[16], d2[16];
                if (need_mask)
                    dq_keys32<true>(s1, s2, dp, rs, lam, sl2, sc, lim - (kb + ch * 32), d1, d2);
                else
                    dq_keys32<false>(s1, s2, dp, rs, lam, sl2, sc, 0, d1, d2);
                // dS_c of keys [32 ch, 32 ch + 32) -> columns [64 w + 16 (ch - 2 w), + 16) of S_c:
                // already read, and inside this warpgroup's own columns [64 w, 64 w + 64)
                const uint32_t dcol = 64 * w + 16 * (ch - 2 * w);
                tmem_st16(tmem + lo + dcol, d1);
                tmem_st16(tmem + lo + 128 + dcol, d2);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(b_ds(w));
        }
        ok = ok && warp_all(mbar_wait(b_dq, 0, ab));
        // ok is warp-uniform; row_ok is not: every lane takes part in the (warp-wide)
        // TMEM loads and only the global stores depend on the row.
        if (ok) {
            tc_fence_after();
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dq) + (grow * p.H + h) * (2 * HD));
#pragma unroll
            for (int ch = 2 * w; ch < 2 * w + 2; ++ch) {  // dQ1 = columns 0..63 (w = 0), dQ2 = 64..127 (w = 1)
                uint32_t o[32];
                tmem_ld32(tmem + lo + 384 + ch * 32, o);
                tmem_wait_ld();
                uint32_t pk[16];  // the softmax scale s, left out of dS, applied here
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * sc, __uint_as_float(o[2 * i + 1]) * sc);
                if (row_ok) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[ch * 4 + i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ============================================================== dKV ===
// CTA = 128 keys of one kv head; walks the heads of its group and the 64-row
// query blocks that see its keys. Keys are the MMA rows, so S_c^T, dP^T, and the
// dV, dK_1, dK_2 accumulators live in tensor memory with one key per lane.
// Per block:
//   MMA warp : S_c^T = K_c Q_c^T and dP^T = V dD^T (operands in shared memory),
//              N = 64 rows;
//   compute  : warpgroup w takes rows [32 w, 32 w + 32): it loads its columns of
//              S_1^T, S_2^T, dP^T, releases the score buffer (so the next
//              block's scores are issued while it computes), forms
//              P_1 - lambda P_2, dS_1 / s, dS_2 / s as bf16 and writes the first
//              into a [128 keys x 64 rows] K-major tile in shared memory, the
//              other two into tensor memory columns of their own;
//   MMA warp : dV += (P_1 - lambda P_2)^T dD, dK_c += dS_c^T Q_c (B = the
//              block's dD / Q_c rows, MN-major).
// The tensor pipe runs the block's scores while the compute warps work on the
// previous block, and the previous block's dV / dK while they wait. Every MMA has
// N >= 64: below that an MMA with both operands in shared memory is bound by the
// operand bandwidth (measured 40 cycles at N = 32, 48 at N = 64, 64 at N = 128
// for M128 K16), and a 64-row block as two 32-row halves took 44 MMAs instead of 28.
// The row statistics enter the score and dP MMAs as one more 16-wide K step: the
// row operand holds -lse_c / (s log2 e) and -delta_1 split into three bf16 terms
// each (slots 0-2, 3-5, 6-8; written by the preprocessing kernel), the key operand
// is one of three constant tiles with ones in the matching three slots, so
//   S_c^T' = S_c^T - lse_c / (s log2 e)   ->  P_c = 2^(S_c^T' s log2 e),
//   dP^T'  = dP^T - delta_1               ->  dS_1 / s = P_1 dP^T',
// and of the statistics only delta_1 - delta_2 is read, for
// dS_2 / s = -lambda P_2 (dP^T' + delta_1 - delta_2): slots 12-13 of row r hold it as
// two bf16 terms and slots 14-15 hold the next row's, one 8-byte load for two rows.
// The per-row loads of all four statistics (a broadcast 16-byte shared load per row
// and warp, two wavefronts) had been half of this kernel's shared-memory traffic.
// The 16-wide operands use the 32-byte swizzle: 32-byte rows, 16-byte chunk c of row
// r at c ^ ((r / 4) % 2).
namespace dkv {
constexpr int BK = 128, BQ = 64, STAGES = 4;
constexpr uint32_t COL_DS = 192;                   // dS_1^T [192, 224), dS_2^T [224, 256): bf16 pairs
constexpr uint32_t COL_DV = 256, COL_DK = 384;     // dV [256, 384), dK1 [384, 448), dK2 [448, 512)
constexpr uint32_t KBOX = 128 * ROW;               // [128 keys x 64] 16 KB
constexpr uint32_t QBOX = 64 * ROW;                // [64 rows x 64] 8 KB
constexpr uint32_t AUG_ROW = 32;                   // a 16-wide bf16 row of the extra K step
constexpr uint32_t ONES = 8 * AUG_ROW;             // one 8-row group, read for all 128 keys
constexpr uint32_t OFF_K = 0;                      // K1 | K2
constexpr uint32_t OFF_V = 2 * KBOX;               // V lo | V hi
constexpr uint32_t OFF_ONES = 4 * KBOX;            // three key-side tiles of the extra K step
constexpr uint32_t OFF_ST = OFF_ONES + 1024;       // stages: Q1 | Q2 | dD lo | dD hi | row operand
constexpr uint32_t ST_AUG = 4 * QBOX;              // the stage's row operand, [64 rows x 16]
constexpr uint32_t STAGE = 4 * QBOX + 2048;        // 2 KB of row operand
constexpr uint32_t OFF_P = OFF_ST + STAGES * STAGE;  // (P_1 - lambda P_2)^T: [128 keys x 64 rows] bf16, K-major
constexpr uint32_t OFF_MISC = OFF_P + 128 * ROW;
constexpr uint32_t SMEM = 1024 + OFF_MISC + 512;
static_assert(SMEM <= 232448, "smem");
static_assert(STAGE % 1024 == 0 && OFF_ST % 1024 == 0 && OFF_P % 1024 == 0, "swizzle atoms are 1024-byte aligned");
// K-major operand of one 16-wide K step in the 32-byte swizzle: 8-row groups sbo bytes apart
// (256 for a dense tile; 0 repeats one group, every row of the key-side tiles being the same).
__device__ __forceinline__ uint64_t desc_sw32(uint32_t saddr, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;   // leading byte offset: unused (one atom along K)
    d |= (uint64_t)(sbo >> 4) << 32;   // stride byte offset
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)6u << 61;           // layout: 32-byte swizzle
    return d;
}
struct Misc {
    uint64_t kv_full, st_full[STAGES], st_empty[STAGES], acc_done;
    uint64_t s_ready, sdp_free, ops_ready, ops_free;
    uint32_t tmem;
    int abort_flag;
};
}  // namespace dkv

// delta_1 - delta_2 of block rows r and r + 1 from the stage's row operand: slots 12-15 of
// row r (two bf16 terms for each of the two rows, chunk 1 of the row under the 32-byte
// swizzle).
__device__ __forceinline__ float2 aug_c2(uint32_t aug, int r) {
    uint32_t a, b;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                 : "=r"(a), "=r"(b)
                 : "r"(aug + (uint32_t)r * 32u + ((uint32_t)(1 ^ ((r >> 2) & 1)) << 4) + 8u));
    return make_float2(__uint_as_float(a << 16) + __uint_as_float(a & 0xffff0000u),
                       __uint_as_float(b << 16) + __uint_as_float(b & 0xffff0000u));
}

// One thread (= one key) and N query rows r0 + i: P_1 - lambda P_2, dS_1, dS_2 as
// bf16 pairs from S_1^T', S_2^T', dP^T' (the statistics already subtracted by the
// extra K step) and delta_1 - delta_2, on packed fp32 pairs of adjacent rows:
//   P_c = 2^(S_c^T' s log2(e)),  -lambda P_2,  P_1 - lambda P_2,
//   dS_1 / s = P_1 dP^T',  dS_2 / s = -lambda P_2 (dP^T' + delta_1 - delta_2).
// MASK zeroes rows outside [q_min, q_end); without it every row is visible.
// The exponentials run on every element and masking is a select after the
// products, so the operands of rows past the end never reach the results.
template <bool MASK, int N>
__device__ __forceinline__ void dkv_rows(const uint32_t (&s1)[N], const uint32_t (&s2)[N], const uint32_t (&dp)[N],
                                         uint32_t aug, int r0, float lam, float sl2, int q0, int q_end, int q_min,
                                         uint32_t (&pc)[N / 2], uint32_t (&d1)[N / 2], uint32_t (&d2)[N / 2]) {
    const uint64_t sl2p = f2_pack(sl2, sl2), nlam = f2_pack(-lam, -lam);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const float2 cc = aug_c2(aug, r0 + i);
        const float2 x1 = f2_unpack(fmul2(f2_pack(__uint_as_float(s1[i]), __uint_as_float(s1[i + 1])), sl2p));
        const float2 x2 = f2_unpack(fmul2(f2_pack(__uint_as_float(s2[i]), __uint_as_float(s2[i + 1])), sl2p));
        const uint64_t p1 = f2_pack(ex2_approx(x1.x), ex2_approx(x1.y));
        const uint64_t q2 = fmul2(f2_pack(ex2_approx(x2.x), ex2_approx(x2.y)), nlam);  // -lambda P_2
        const uint64_t pp = f2_pack(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1]));
        float2 a = f2_unpack(fadd2(p1, q2));
        float2 b1 = f2_unpack(fmul2(p1, pp));
        float2 b2 = f2_unpack(fmul2(q2, fadd2(pp, f2_pack(cc.x, cc.y))));
        if (MASK) {
            const int qi = q0 + i;
            const bool v0 = (qi < q_end) & (qi >= q_min), v1 = (qi + 1 < q_end) & (qi + 1 >= q_min);
            a.x = v0 ? a.x : 0.f;
            b1.x = v0 ? b1.x : 0.f;
            b2.x = v0 ? b2.x : 0.f;
            a.y = v1 ? a.y : 0.f;
            b1.y = v1 ? b1.y : 0.f;
            b2.y = v1 ? b2.y : 0.f;
        }
        pc[i / 2] = pack_bf16x2(a.x, a.y);
        d1[i / 2] = pack_bf16x2(b1.x, b1.y);
        d2[i / 2] = pack_bf16x2(b2.x, b2.y);
    }
}

// Rows [32 w, 32 w + 32) of key k's row in a [128 keys x 64 rows] K-major tile
// (128-byte swizzle: 16-byte chunk c of row k at physical chunk c ^ (k % 8)).
__device__ __forceinline__ void store_op_row(uint32_t tile, int k, int w, const uint32_t (&v)[16]) {
    const uint32_t row = tile + (uint32_t)k * ROW;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        sts_u4(row + ((uint32_t)((4 * w + j) ^ (k & 7)) << 4), make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
}

__global__ void __launch_bounds__(NT, 1)
diffattn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dd,
                        const __grid_constant__ CUtensorMap tm_aug, const BwdParams p) {
    using namespace dkv;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc& ms = *reinterpret_cast<Misc*>(smem + OFF_MISC);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grid (kv head, key tile, sequence), or with the tiles outermost (kv head,
    // sequence, key tile). Causal: key tile kt is seen by the query blocks from kt on,
    // so the first tiles carry the most work and are scheduled first
    // (kv head group x key tile x kv head in group, 1, sequence): a group's Q / dD
    // (sized by the host) stays in L2 while its CTAs stream it
    const bool outer = p.dkv_tiles_outer != 0;
    int g, seq, kt;
    if (outer) {
        g = blockIdx.x, seq = blockIdx.y, kt = blockIdx.z;
    } else {
        const int n_kt = (p.max_seqlen + BK - 1) / BK, kg = p.dkv_group_kv;
        const int grp = (int)blockIdx.x / (n_kt * kg), rem = (int)blockIdx.x - grp * (n_kt * kg);
        g = grp * kg + rem % kg, seq = blockIdx.z, kt = rem / kg;
    }
    int start = 0, len = 0;
    if (!seq_bounds(p, seq, &start, &len)) return;
    if (kt * BK >= len) return;
    const int G = p.H / p.Hkv;
    const int qb0 = p.causal ? (kt * BK) / BQ : 0;          // first query block that sees these keys
    const int nqb = (len + BQ - 1) / BQ - qb0;             // query blocks per head
    const int n_items = G * nqb;                            // (head, query block) items

    const uint32_t b_kv = smem_u32(&ms.kv_full), b_acc = smem_u32(&ms.acc_done);
    const uint32_t b_s = smem_u32(&ms.s_ready), b_free = smem_u32(&ms.sdp_free);
    const uint32_t b_ops = smem_u32(&ms.ops_ready), b_opf = smem_u32(&ms.ops_free);
    auto b_sf = [&](int s) { return smem_u32(&ms.st_full[s]); };
    auto b_se = [&](int s) { return smem_u32(&ms.st_empty[s]); };
    auto item_head = [&](int it) { return g * G + it / nqb; };
    auto item_row0 = [&](int it) { return (qb0 + it % nqb) * BQ; };  // first query position of the block
    if (warp == PRODUCER_WARP && lane == 0) {
        mbar_init(b_kv, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(b_sf(s), 1);
            mbar_init(b_se(s), 1);
        }
        mbar_init(b_s, 1);
        mbar_init(b_free, 8);  // one arrive per compute warp
        mbar_init(b_ops, 8);
        mbar_init(b_opf, 1);
        mbar_init(b_acc, 1);
        ms.abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x < 8) {
        // the key-side tiles of the extra K step: tile j holds bf16 ones in slots 3j..3j+2
        // of each of its 8 rows (the MMAs read the group for every 8 keys)
        const int k = threadIdx.x;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            uint32_t wd[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t lo = (2 * i >= 3 * j && 2 * i < 3 * j + 3) ? 0x3F80u : 0u;
                const uint32_t hi = (2 * i + 1 >= 3 * j && 2 * i + 1 < 3 * j + 3) ? 0x3F80u : 0u;
                wd[i] = lo | (hi << 16);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c)
                sts_u4(sb + OFF_ONES + (uint32_t)j * ONES + (uint32_t)k * AUG_ROW + ((uint32_t)(c ^ ((k >> 2) & 1)) << 4),
                       make_uint4(wd[4 * c], wd[4 * c + 1], wd[4 * c + 2], wd[4 * c + 3]));
        }
        fence_proxy_async_smem();  // visible to the tensor cores (ordered by the barrier below)
    }
    if (warp == MMA_WARP) tmem_alloc(smem_u32(&ms.tmem), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem;
    const AbortState ab{&ms.abort_flag, p.error_word, p.timeout_ns};

    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            const int row_k = start + kt * BK;
            mbar_arrive_expect_tx(b_kv, 4 * KBOX);
            tma_load_2d(sb + OFF_K, &tm_k, b_kv, g * 2 * HD, row_k, pol);
            tma_load_2d(sb + OFF_K + KBOX, &tm_k, b_kv, g * 2 * HD + HD, row_k, pol);
            tma_load_2d(sb + OFF_V, &tm_v, b_kv, g * DV, row_k, pol);
            tma_load_2d(sb + OFF_V + KBOX, &tm_v, b_kv, g * DV + 64, row_k, pol);
            int issued = 0;
            for (int it = 0; it < n_items; ++it) {
                const int s = it % STAGES;
                if (!mbar_wait(b_se(s), ((uint32_t)(it / STAGES) & 1u) ^ 1u, ab)) break;
                const uint32_t st = sb + OFF_ST + (uint32_t)s * STAGE;
                const int hh = item_head(it);
                const int t0 = start + item_row0(it);
                mbar_arrive_expect_tx(b_sf(s), 4 * QBOX + BQ * AUG_ROW);
                tma_load_2d(st, &tm_q, b_sf(s), hh * 2 * HD, t0, pol);
                tma_load_2d(st + QBOX, &tm_q, b_sf(s), hh * 2 * HD + HD, t0, pol);
                tma_load_2d(st + 2 * QBOX, &tm_dd, b_sf(s), hh * DV, t0, pol);
                tma_load_2d(st + 3 * QBOX, &tm_dd, b_sf(s), hh * DV + 64, t0, pol);
                // the rows' operand of the extra K step (rows past the tokens read as zero)
                tma_load_2d(st + ST_AUG, &tm_aug, b_sf(s), 0, hh * p.total_tokens + t0, pol);
                issued = it + 1;
            }
            mbar_wait_drain(b_kv, 0, p.timeout_ns);
            for (int it = issued > STAGES ? issued - STAGES : 0; it < issued; ++it)
                mbar_wait_drain(b_sf(it % STAGES), (uint32_t)(it / STAGES) & 1u, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // Per block it: the scores of block it (once its rows have landed and the
        // compute warps have read block it - 1's scores out of the buffer), then dV / dK
        // of block it - 1 (once its operand tiles are written). The pipe runs in issue
        // order, so block it's scores fill the tensor pipe while the compute warps work
        // on block it - 1.
        constexpr uint32_t id_s = idesc_bf16_f32(128, 64, false);    // S_c^T, dP^T: N = 64 rows, both K-major
        constexpr uint32_t id_v = idesc_bf16_f32(128, 128, true);    // dV: B = dD rows, MN-major (dv)
        constexpr uint32_t id_k = idesc_bf16_f32(128, 64, true);     // dK_c: B = Q_c rows, MN-major (d)
        constexpr uint64_t KS = 32 >> 4, KB = KBOX >> 4, QB = QBOX >> 4, SG = STAGE >> 4, KR = (16 * ROW) >> 4;
        const uint64_t d_k = desc_k(sb + OFF_K), d_v = desc_k(sb + OFF_V), d_p = desc_k(sb + OFF_P);
        const uint64_t d_q = desc_k(sb + OFF_ST), d_qm = desc_mn(sb + OFF_ST, QBOX);
        // S_c^T = K_c Q_c^T (A = the K_c box, B = the block's Q_c rows) and dP^T = V dD^T (K = dv
        // = 128 over the two 64-column halves of V and of dD).
        auto issue_sdp = [&](int it) {
            const uint64_t sq = d_q + (uint64_t)(it % STAGES) * SG;
            const uint64_t sa = desc_sw32(sb + OFF_ST + (uint32_t)(it % STAGES) * STAGE + ST_AUG, 256u);
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss_elect(tmem + c * 64, d_k + c * KB + kk * KS, sq + c * QB + kk * KS, id_s, kk > 0);
                mma_ss_elect(tmem + c * 64, desc_sw32(sb + OFF_ONES + (uint32_t)c * ONES, 0u), sa, id_s, 1u);  // - lse_c
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ss_elect(tmem + 128, d_v + (kk >> 2) * KB + (kk & 3) * KS,
                             sq + 2 * QB + (kk >> 2) * QB + (kk & 3) * KS, id_s, kk > 0);
            mma_ss_elect(tmem + 128, desc_sw32(sb + OFF_ONES + 2 * ONES, 0u), sa, id_s, 1u);  // - delta_1
            mma_commit_elect(b_s);
        };
        // dV += (P_1 - lambda P_2)^T dD and dK_c += dS_c^T Q_c over the block's 64 rows, 16 a
        // step: A = the P tile (shared memory, K-major) or dS_c^T (tensor memory, 8 columns a
        // step), B = the rows of dD / Q_c in the stage (MN-major).
        auto issue_dvdk = [&](int it) {
            const int s = it % STAGES;
            const uint64_t sqm = d_qm + (uint64_t)s * SG;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                mma_ss_elect(tmem + COL_DV, d_p + kk * KS, sqm + 2 * QB + kk * KR, id_v, acc);
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    mma_ts_elect(tmem + COL_DK + c * 64, tmem + COL_DS + 32 * c + 8 * kk, sqm + c * QB + kk * KR, id_k,
                                 acc);
            }
            mma_commit_elect(b_opf);    // the operands may be rewritten once these have run
            mma_commit_elect(b_se(s));  // every MMA reading stage s has been issued
        };
        bool ok = warp_all(mbar_wait(b_kv, 0, ab));
        for (int it = 0; ok && it < n_items; ++it) {
            if (!(ok = warp_all(mbar_wait(b_sf(it % STAGES), (uint32_t)(it / STAGES) & 1u, ab)))) break;
            if (it > 0 && !(ok = warp_all(mbar_wait(b_free, (uint32_t)(it - 1) & 1u, ab)))) break;
            tc_fence_after();
            issue_sdp(it);
            if (it > 0) {
                if (!(ok = warp_all(mbar_wait(b_ops, (uint32_t)(it - 1) & 1u, ab)))) break;
                tc_fence_after();
                issue_dvdk(it - 1);
            }
        }
        if (ok && n_items > 0 && (ok = warp_all(mbar_wait(b_ops, (uint32_t)(n_items - 1) & 1u, ab)))) {
            tc_fence_after();
            issue_dvdk(n_items - 1);
        }
        mma_commit_elect(b_acc);
        mbar_wait_drain(b_acc, 0, p.timeout_ns);
        __syncwarp();
    } else {
        // ============================================== compute warpgroups ===
        // Warpgroup w handles query rows [32 w, 32 w + 32) of every block; thread = key.
        const int w = warp >> 2;
        const int k = (warp & 3) * 32 + lane;  // key in the tile = TMEM lane
        const uint32_t lo = (uint32_t)((warp & 3) * 32) << 16;
        const int kj = kt * BK + k;      // key position in the sequence
        const bool key_ok = kj < len;
        const int q_end = key_ok ? len : 0;       // visible query rows of this key: [q_min, q_end)
        const int q_min = p.causal ? kj : 0;
        const float sl2 = p.scale_log2, sc = p.scale;
        bool ok = true;
        for (int it = 0; ok && it < n_items; ++it) {
            if (!(ok = warp_all(mbar_wait(b_s, (uint32_t)it & 1u, ab)))) break;
            tc_fence_after();
            uint32_t s1[32], s2[32], dp[32];
            tmem_ld32(tmem + lo + 32 * w, s1);
            tmem_ld32(tmem + lo + 64 + 32 * w, s2);
            tmem_ld32(tmem + lo + 128 + 32 * w, dp);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_free);  // the next block's scores may overwrite the buffer
            const int s = it % STAGES;
            // the block's row operand (delta_1 - delta_2 per row; shared-window address)
            const uint32_t aug = sb + OFF_ST + (uint32_t)s * STAGE + ST_AUG;
            const int hh = item_head(it);
            const float lam = p.lambda[hh * p.lambda_stride];
            const int row0 = item_row0(it);
            // masking only where a row or key passes the sequence end or (causal) a row
            // precedes a key of the tile: the first two blocks and the last one
            const bool need_mask = row0 + BQ > len || kt * BK + BK > len || (p.causal && row0 < kt * BK + BK - 1);
            uint32_t pc[16], d1[16], d2[16];
            if (need_mask)
                dkv_rows<true, 32>(s1, s2, dp, aug, 32 * w, lam, sl2, row0 + 32 * w, q_end, q_min, pc, d1, d2);
            else
                dkv_rows<false, 32>(s1, s2, dp, aug, 32 * w, lam, sl2, 0, 0, 0, pc, d1, d2);
            // the previous block's operands have been read by its dV / dK MMAs
            if (it > 0 && !(ok = warp_all(mbar_wait(b_opf, (uint32_t)(it - 1) & 1u, ab)))) break;
            store_op_row(sb + OFF_P, k, w, pc);
            tmem_st16(tmem + lo + COL_DS + 16 * w, d1);
            tmem_st16(tmem + lo + COL_DS + 32 + 16 * w, d2);
            fence_proxy_async_smem();  // the P tile, visible to the tensor cores
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_ops);
        }
        ok = ok && warp_all(mbar_wait(b_acc, 0, ab));
        // ok is warp-uniform; key_ok is not: every lane takes part in the (warp-wide)
        // TMEM loads and only the global stores depend on the key.
        if (ok) {
            tc_fence_after();
            const size_t grow = (size_t)(start + (key_ok ? kj : 0));
            uint4* dvp = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dv) + (grow * p.Hkv + g) * DV);
            uint4* dkp = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dk) + (grow * p.Hkv + g) * (2 * HD));
            // warpgroup 0 stores dV (columns 192..319), warpgroup 1 dK1 | dK2 (320..447)
            uint4* dst = w == 0 ? dvp : dkp;
            const float f = w == 0 ? 1.f : sc;  // dK: the softmax scale s, left out of dS, applied here
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t o[32];
                tmem_ld32(tmem + lo + COL_DV + 128 * w + ch * 32, o);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * f, __uint_as_float(o[2 * i + 1]) * f);
                if (key_ok) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[ch * 4 + i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <typename K>
cudaError_t set_smem(K kernel, uint32_t bytes, bool* done) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !done[dev]) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (err != cudaSuccess) return err;
        done[dev] = true;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_sm103a(const BwdParams& p, const BwdTensorMaps& m, cudaStream_t stream) {
    static bool dq_done[64] = {false}, dkv_done[64] = {false};
    cudaError_t err = set_smem(diffattn_bwd_dq_kernel, dq::SMEM, dq_done);
    if (err != cudaSuccess) return err;
    err = set_smem(diffattn_bwd_dkv_kernel, dkv::SMEM, dkv_done);
    if (err != cudaSuccess) return err;
    const int n_qt = (p.max_seqlen + dq::BM - 1) / dq::BM;
    if (p.dq_group_heads < 1 || p.H % p.dq_group_heads != 0 || p.dkv_group_kv < 1 || p.Hkv % p.dkv_group_kv != 0)
        return cudaErrorInvalidValue;
    const dim3 dq_grid = p.dq_tiles_outer ? dim3((unsigned)p.H, (unsigned)p.num_seqs, (unsigned)n_qt)
                                          : dim3((unsigned)(p.H * n_qt), 1u, (unsigned)p.num_seqs);
    diffattn_bwd_dq_kernel<<<dq_grid, NT, dq::SMEM, stream>>>(
        m.q128, m.k128, m.v128, m.dd128, p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    const int n_kt = (p.max_seqlen + dkv::BK - 1) / dkv::BK;
    const dim3 dkv_grid = p.dkv_tiles_outer ? dim3((unsigned)p.Hkv, (unsigned)p.num_seqs, (unsigned)n_kt)
                                            : dim3((unsigned)(p.Hkv * n_kt), 1u, (unsigned)p.num_seqs);
    diffattn_bwd_dkv_kernel<<<dkv_grid, NT, dkv::SMEM, stream>>>(
        m.q64, m.k128, m.v128, m.dd64, m.aug64, p);
    return cudaGetLastError();
}

}  // namespace diffattn
