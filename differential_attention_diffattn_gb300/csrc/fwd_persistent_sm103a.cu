// Persistent form of the fused differential-attention forward for sm_103a
// (bf16 in, fp32 accumulate, bf16 out), d = 64, dv = 128, used when the (query
// tile, sequence, head) items have few key tiles each: one CTA per SM walks the
// non-empty items in a static snake order over the items sorted longest first
// (every CTA gets about the same number of key tiles), and the next item's Q and
// K / V loads, its first scores and its softmax run while the epilogue
// warpgroup finishes the current item. That hides the per-CTA setup, the
// epilogue and the gap between CTAs, which weigh most when each item has few
// key tiles. The producer warp enumerates the items (for packed sequences from
// their tile counts, staged in shared memory; at most MAX_PACKED_SEQS
// sequences) and hands each to the other roles through a four-slot ring.
//
// Per item the arithmetic is that of the one-item-per-CTA kernel (fwd_sm103a.cu):
// S_c = Q_c K_c^T, two online softmaxes, O_c += P_c V on the tensor cores, then
// O1/l1 - lambda O2/l2, RMSNorm over dv, weight, (1 - lambda_init)
// ("DiffTransformer.py", forward; "LlamaDiffSdpaAttention.py", forward).
//
// Roles (512 threads, four warpgroups): warps 0-3 / 4-7 softmax of component
// 1 / 2; warps 8-11 the epilogue (warp 8 + q reads TMEM lanes 32q..32q+31); warp
// 12 TMA producer; warp 13 TMEM allocator and MMA issuer; warps 14-15 idle. With
// the epilogue in its own warpgroup the softmax warps go on to the next item as
// soon as their last P is stored, and the epilogue of one item runs under the
// next item's key tiles. Sixteen warps leave 128 registers a thread at launch;
// the warpgroups then move registers with setmaxnreg: softmax 168, epilogue 80,
// producer / MMA 96 (8 x 32 x 168 + 4 x 32 x (80 + 96) = the 65,536 the launch
// holds; each SM sub-partition runs two softmax warps, one epilogue warp and one
// of warps 12-15: 2 x 168 + 80 + 96 = 512 registers a lane, its whole share; the
// MMA warp's one-item lookahead spilled at 88).
//
// Shared memory: two Q boxes (Q1 | Q2 of two items, so the next item's Q loads
// while the current one runs), two K stages (K1 | K2) and two V stages with
// their own barriers (a K stage is free once both score MMAs of its tile have
// run, a V stage once both P V MMAs have: two stages each give the loads the
// slack of a three-stage ring shared by K and V), and 32 KB where the epilogue
// keeps half of each row's D. The epilogue reads O from tensor memory once: it
// forms D = O1/l1 - lambda O2/l2, keeps it in shared memory in fp32 (columns
// 0-63 in the 32 KB area, 64-127 in the item's own Q box, whose score MMAs have
// all run), sums D^2, and releases O to the next item's first P V; a second
// pass over the kept D normalises and stores. The item's Q box is released to
// the producer after that pass.
//
// Barriers that advance once per item: item_full / item_empty (a four-slot ring
// of items), q_full / q_empty per Q box, stats_full[item parity] (1/l_c per row
// from the softmax warps), o_full / o_empty (the O accumulators: an item's first
// P V waits until the epilogue of the previous one has read them); once per key
// tile over all items: k_full / k_empty and v_full / v_empty per stage, s_full,
// p_ready. The MMA warp looks one item ahead: the next item's first scores of
// component 1 are issued right after the current item's last P V of component 1
// (when that item's Q and keys have landed), as within an item, and the two
// softmax warpgroups cross item boundaries each at its own pace (component 1 at
// most one item and one tile ahead), keeping their stagger on the tensor pipe.
// Every wait is an mbarrier wait, bounded and watching the CTA's abort flag, so
// a role that gives up never leaves another waiting at a barrier it has left.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103a_ptx.cuh"
#include "softmax_exact.cuh"

namespace diffattn {
namespace {

constexpr int BM = 128, BN = 128, HD = 64, DV = 128, STAGES = 2, QBUF = 2;
constexpr int NUM_THREADS = 512, EPI_WARP0 = 8, PRODUCER_WARP = 12, MMA_WARP = 13;
constexpr int NSLOT = 4;  // item ring
// registers a thread: at launch (65,536 / 512) and after the split
constexpr int REG_LAUNCH = 128, REG_SOFTMAX = 168, REG_EPI = 80, REG_COPY = 96;
constexpr int REG_NEED = 8 * 32 * REG_SOFTMAX + 4 * 32 * REG_EPI + 4 * 32 * REG_COPY;
static_assert(REG_NEED <= NUM_THREADS * REG_LAUNCH, "the register split exceeds the launch's registers");
static_assert(2 * REG_SOFTMAX + REG_EPI + REG_COPY <= 4 * REG_LAUNCH, "the split exceeds one sub-partition's share");
constexpr uint32_t BOX_BYTES = BM * HD * 2;
constexpr uint32_t Q_BYTES = 2 * BOX_BYTES, K_BYTES = 2 * BOX_BYTES, V_BYTES = 2 * BOX_BYTES;
constexpr uint32_t D_HALF_BYTES = BM * 64 * 4;  // 64 fp32 values of D per row
static_assert(D_HALF_BYTES == Q_BYTES, "the second half of D fills one Q box");
constexpr uint32_t OFF_Q0 = 0;
constexpr uint32_t OFF_K0 = OFF_Q0 + QBUF * Q_BYTES;
constexpr uint32_t OFF_V0 = OFF_K0 + STAGES * K_BYTES;
constexpr uint32_t OFF_D = OFF_V0 + STAGES * V_BYTES;
constexpr uint32_t OFF_MISC = OFF_D + D_HALF_BYTES;
constexpr uint32_t MISC_BYTES = 3072;
// No alignment slack: every byte up to the per-block limit is in use; the
// kernel checks that its dynamic shared memory starts on a 1024-byte boundary.
constexpr uint32_t SMEM_BYTES = OFF_MISC + MISC_BYTES;
static_assert(SMEM_BYTES <= 232448, "exceeds the per-block shared memory limit");
constexpr uint32_t TMEM_COLS = 512;
__device__ __forceinline__ uint32_t col_s(int c) { return (uint32_t)c * 128u; }
__device__ __forceinline__ uint32_t col_o(int c) { return 256u + (uint32_t)c * 128u; }
constexpr float RESCALE_THRESHOLD = 8.0f;
// Past an item's first tile, the row sum of a tile above which the warp takes it
// maximum-first (the steps of the one-item-per-CTA kernel).
constexpr float EXACT_SUM = 4294967296.0f;  // 2^32
constexpr int MAX_PACKED_SEQS = 64;

// One work item: 128 query rows of one diff head of one sequence (n_kv < 0: no
// more items).
struct Item {
    int h, qt, start, len, n_kv;
    int pad[3];
};

struct Misc {
    uint64_t item_full[NSLOT], item_empty[NSLOT];
    uint64_t q_full[QBUF], q_empty[QBUF];
    uint64_t k_full[STAGES], k_empty[STAGES], v_full[STAGES], v_empty[STAGES];
    uint64_t s_full[2], p_ready[2];
    uint64_t o_full, o_empty, stats_full[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    float il[2][2][BM];                 // 1/l_c per row, by item parity and component
    float w[DV];
    Item work[NSLOT];                   // the item ring
    uint16_t tiles[MAX_PACKED_SEQS];    // 128-row tiles of each packed sequence (0: none or bad bounds)
};
static_assert(sizeof(Misc) <= MISC_BYTES, "misc area too small");

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) { return smem_desc_sw128(saddr, 16, 1024); }
__device__ __forceinline__ uint64_t desc_value(uint32_t saddr) { return smem_desc_sw128(saddr, BOX_BYTES, 1024); }
__device__ __forceinline__ bool warp_all(bool pred) { return __all_sync(0xffffffffu, pred); }
__global__ void __launch_bounds__(NUM_THREADS, 1)
diffattn_fwd_bf16_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p, int n_qt) {
    extern __shared__ uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(p.error_word, kErrLayout);
        return;
    }
    // A programmatic dependent of the previous kernel on the stream: nothing is
    // read before it has completed, except with lambda_pending (that kernel writes
    // lambda alone), where only the epilogue's reads of lambda wait.
    if (!p.lambda_pending) griddep_wait();
    griddep_launch_dependents();
    Misc& ms = *reinterpret_cast<Misc*>(smem + OFF_MISC);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar_item_full = [&](int i) { return smem_u32(&ms.item_full[i]); };
    auto bar_item_empty = [&](int i) { return smem_u32(&ms.item_empty[i]); };

    auto bar_q_full = [&](int b) { return smem_u32(&ms.q_full[b]); };
    auto bar_q_empty = [&](int b) { return smem_u32(&ms.q_empty[b]); };
    auto bar_k_full = [&](int s) { return smem_u32(&ms.k_full[s]); };
    auto bar_k_empty = [&](int s) { return smem_u32(&ms.k_empty[s]); };
    auto bar_v_full = [&](int s) { return smem_u32(&ms.v_full[s]); };
    auto bar_v_empty = [&](int s) { return smem_u32(&ms.v_empty[s]); };
    auto bar_s_full = [&](int c) { return smem_u32(&ms.s_full[c]); };
    auto bar_p_ready = [&](int c) { return smem_u32(&ms.p_ready[c]); };
    const uint32_t bar_o_full = smem_u32(&ms.o_full), bar_o_empty = smem_u32(&ms.o_empty);
    const uint32_t bar_mma_done = smem_u32(&ms.mma_done);
    auto bar_stats_full = [&](int i) { return smem_u32(&ms.stats_full[i]); };
    auto sq = [&](int b) { return sbase + OFF_Q0 + (uint32_t)b * Q_BYTES; };
    auto sk = [&](int s) { return sbase + OFF_K0 + (uint32_t)s * K_BYTES; };
    auto sv = [&](int s) { return sbase + OFF_V0 + (uint32_t)s * V_BYTES; };

    if (warp == PRODUCER_WARP && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(bar_item_full(i), 1);
            mbar_init(bar_item_empty(i), 13);  // the MMA warp, the eight softmax and four epilogue warps
        }
        for (int b = 0; b < QBUF; ++b) {
            mbar_init(bar_q_full(b), 1);
            mbar_init(bar_q_empty(b), 4);  // one arrive per epilogue warp, after its second pass
        }
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_k_full(s), 1);
            mbar_init(bar_k_empty(s), 1);
            mbar_init(bar_v_full(s), 1);
            mbar_init(bar_v_empty(s), 1);
        }
        for (int c = 0; c < 2; ++c) {
            mbar_init(bar_s_full(c), 1);
            mbar_init(bar_p_ready(c), 128);
        }
        mbar_init(bar_o_full, 1);
        mbar_init(bar_o_empty, 128);     // every epilogue thread
        mbar_init(bar_stats_full(0), 256);  // every softmax thread, items of even / odd index
        mbar_init(bar_stats_full(1), 256);
        mbar_init(bar_mma_done, 1);
        ms.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == PRODUCER_WARP) {
        for (int i = lane; i < DV; i += 32) ms.w[i] = p.subln_w[i];
        // packed sequences: tile counts, and the bounds checked once
        if (p.cu_seqlens != nullptr) {
            for (int sq_i = lane; sq_i < p.num_seqs; sq_i += 32) {
                const int s0 = p.cu_seqlens[sq_i], s1 = p.cu_seqlens[sq_i + 1];
                const bool bad = s0 < 0 || s1 < s0 || s1 > p.total_tokens || s1 - s0 > p.max_seqlen ||
                                 (sq_i == 0 && s0 != 0) || (sq_i == p.num_seqs - 1 && s1 != p.total_tokens);
                if (bad && blockIdx.x == 0) atomicOr(p.error_word, kErrBadSeqlens);
                ms.tiles[sq_i] = (uint16_t)(bad ? 0 : (s1 - s0 + BM - 1) / BM);
            }
        }
    }
    if (warp == MMA_WARP) tmem_alloc(smem_u32(&ms.tmem_base), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;
    const AbortState ab{&ms.abort_flag, p.error_word, p.timeout_ns};

    // Each warpgroup moves to its register count first (setmaxnreg applies to the
    // whole warpgroup, so warps 12-15 share one branch).
    if (warp < EPI_WARP0) {
        setmaxnreg_inc<REG_SOFTMAX>();
        // ====================================================== softmax (warps 0-7) ===
        const int c = warp >> 2;
        const int r = (warp & 3) * 32 + lane;  // query row in the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t t_s = tmem + lane_off + col_s(c);
        const uint32_t t_o = tmem + lane_off + col_o(c);
        const float sl2 = p.scale_log2;
        const uint64_t sl2p = f2_pack(sl2, sl2);
        int tile = 0, items = 0;
        bool ok = true;
        for (;;) {
            const int slot = items % NSLOT;
            ok = warp_all(ok && mbar_wait(bar_item_full(slot), (uint32_t)(items / NSLOT) & 1u, ab));
            if (!ok) break;
            const Item it = ms.work[slot];
            if (it.n_kv < 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_item_empty(slot));
                break;
            }
            const int qi = it.qt * BM + r;
            // the softmax steps of the one-item-per-CTA kernel: the item's first tile
            // maximum-first, later ones exponentiated with that reference at once, the
            // rare tile whose row sum passes 2^32 taken again maximum-first (softmax_exact.cuh)
            float m = -INFINITY, l = 0.f;
            for (int j = 0; ok && j < it.n_kv; ++j, ++tile) {
                if (!(ok = warp_all(mbar_wait(bar_s_full(c), (uint32_t)tile & 1u, ab)))) break;
                tc_fence_after();
                float x[BN];
                {
                    // two 64-column loads: one 128-column load needs more registers than
                    // the kernel's launch count, against which every instruction is checked
                    uint32_t sr[2][64];
                    tmem_ld64(t_s, sr[0]);
                    tmem_ld64(t_s + 64, sr[1]);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < BN; ++e) x[e] = __uint_as_float(sr[e >> 6][e & 63]);
                }
                // keys < lim(j) of tile j are visible (all of them off the diagonal and the sequence end)
                auto lim_of = [&](int jj) {
                    const bool masked = (p.causal && jj == it.qt) || jj * BN + BN > it.len;
                    return masked ? (p.causal ? min(qi + 1, it.len) : it.len) - jj * BN : BN;
                };
                if ((p.causal && j == it.qt) || j * BN + BN > it.len) {
                    const int lim = lim_of(j);
#pragma unroll
                    for (int e = 0; e < BN; ++e)
                        if (e >= lim) x[e] = -INFINITY;
                }
                float alpha = 1.f;
                if (j == 0) {
                    float mx0 = fmaxf(x[0], x[1]), mx1 = fmaxf(x[2], x[3]), mx2 = fmaxf(x[4], x[5]),
                          mx3 = fmaxf(x[6], x[7]);
#pragma unroll
                    for (int e = 8; e < BN; e += 8) {
                        mx0 = fmax3(mx0, x[e], x[e + 1]);
                        mx1 = fmax3(mx1, x[e + 2], x[e + 3]);
                        mx2 = fmax3(mx2, x[e + 4], x[e + 5]);
                        mx3 = fmax3(mx3, x[e + 6], x[e + 7]);
                    }
                    const float m_tile = fmax3(fmaxf(mx0, mx1), mx2, mx3) * sl2;
                    if (m_tile > m + RESCALE_THRESHOLD) {
                        alpha = ex2_approx(m - m_tile);
                        m = m_tile;
                    }
                }
                const uint64_t nmp = f2_pack(-m, -m);
                uint64_t sa = 0, sb = 0;
#pragma unroll
                for (int ch = 0; ch < BN / 32; ++ch) {
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
                float sum = __fadd_rn(sab.x, sab.y);
                // A row sum above 2^32 (or not finite): the warp takes the tile maximum-first
                // and O_c (this item's sum through tile j-1) moves to the new reference. Rows
                // past the sequence end take no part in the choice.
                if (j > 0 && __any_sync(0xffffffffu, qi < it.len && !(sum <= EXACT_SUM))) {
                    const volatile Item* iv = &ms.work[slot];
                    const int hv = iv->h, g = hv / (p.H / p.Hkv);
                    sum = softmax_exact_tile<BN>(
                        t_s, sq(items & 1) + (uint32_t)c * BOX_BYTES + (uint32_t)r * 128u, r,
                        reinterpret_cast<const __nv_bfloat16*>(p.k) + ((size_t)(iv->start + j * BN) * p.Hkv + g) * (2 * HD) +
                            c * HD,
                        (size_t)p.Hkv * (2 * HD), lim_of(j), sl2, RESCALE_THRESHOLD, m, alpha);
                    if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                        for (int ch = 0; ch < DV / 32; ++ch) {
                            uint32_t o[32];
                            tmem_ld32(t_o + ch * 32, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(t_o + ch * 32, o);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar_p_ready(c));
                l = __fmaf_rn(l, alpha, sum);
            }
            if (!ok) break;
            // Training outputs: lse_c = m_c + log2(l_c), so that P_c = 2^(S_c scale log2(e) - lse_c).
            // The item's start and head are read again from its slot (the softmax warps
            // release the slot only below): held across the tile loop they pushed the
            // softmax warps past their registers.
            if (p.lse != nullptr && qi < it.len) {
                const volatile Item* iv = &ms.work[slot];
                p.lse[((size_t)(iv->start + qi) * p.H + iv->h) * 2 + c] = m + __log2f(l);
            }
            // 1/l_c for the epilogue, in the buffer and on the barrier of this item's
            // parity: the epilogue of item - 2 read that buffer and waited on that
            // barrier before it released O for item - 1, whose first P V precedes every
            // score of this item. (One barrier for all items could run two phases ahead
            // of the epilogue: an item of one key tile needs no P V before its scores,
            // so its stats can follow the previous item's while the epilogue is still on
            // the one before, and a parity wait cannot tell those phases apart.)
            ms.il[items & 1][c][r] = 1.f / l;
            mbar_arrive(bar_stats_full(items & 1));
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_item_empty(slot));
            ++items;
        }
    } else if (warp < PRODUCER_WARP) {
        setmaxnreg_dec<REG_EPI>();
        // =================================================== epilogue (warps 8-11) ===
        // One thread per row, all dv values: D = O1/l1 - lambda O2/l2, RMSNorm over dv,
        // weight, (1 - lambda_init), bf16. O is read once: D goes to shared memory in
        // fp32 (values 0-63 in the D area, 64-127 in the item's Q box) while the sums
        // of squares build up, and O is released to the next item's first P V before
        // the second pass normalises the kept D. Each half of the row is summed on its
        // own and the halves added, the order of the one-item-per-CTA kernel's two
        // warpgroups, so the two kernels give the same bits. Row r of a half is 256
        // bytes at r x 256, its 16-byte chunk i at chunk i ^ (r % 8) (no bank
        // conflicts: the 8 rows of a store phase hit 8 different chunks).
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t t_o1 = tmem + lane_off + col_o(0), t_o2 = tmem + lane_off + col_o(1);
        auto d_chunk = [&](int half, int buf, int i) {  // i: 16-byte chunk 0..15 of the half row
            uint8_t* base = smem + (half == 0 ? OFF_D : OFF_Q0 + (uint32_t)buf * Q_BYTES);
            return reinterpret_cast<float4*>(base + (uint32_t)r * 256u + (uint32_t)((i & 8) | ((i ^ r) & 7)) * 16u);
        };
        if (p.lambda_pending) griddep_wait();  // lambda comes from the preceding grid
        int items = 0;
        for (;;) {
            const int slot = items % NSLOT;
            if (!warp_all(mbar_wait(bar_item_full(slot), (uint32_t)(items / NSLOT) & 1u, ab))) break;
            const Item it = ms.work[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_item_empty(slot));
            if (it.n_kv < 0) break;
            if (p.inject == 2) {  // test hook: hold the epilogue back so the softmax warps run ahead
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 20000ull) {
                }
            }
            const int par = items & 1, qb = items & 1;
            if (!warp_all(mbar_wait(bar_stats_full(par), (uint32_t)(items >> 1) & 1u, ab))) break;
            if (!warp_all(mbar_wait(bar_o_full, (uint32_t)par, ab))) break;
            tc_fence_after();
            const int qi = it.qt * BM + r;
            const bool store = qi < it.len;
            const float lam = p.lambda[it.h * p.lambda_stride];
            const float il1 = ms.il[par][0][r], il2 = ms.il[par][1][r];
            float ss_half[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float ssp = 0.f;
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {  // 16 values at a time
                    const int col = hf * 64 + c4 * 16;
                    uint32_t o1[16], o2[16];
                    tmem_ld16(t_o1 + col, o1);
                    tmem_ld16(t_o2 + col, o2);
                    tmem_wait_ld();
                    if (col == DV - 16) {  // O has been read: the next item's first P V may overwrite it
                        tc_fence_before();
                        mbar_arrive(bar_o_empty);
                    }
                    // Training outputs: the normalised attention output of each component,
                    // kept in fp32 (the lambda gradient sums many cancelling terms of them).
                    if (store && p.o1 != nullptr) {
                        const size_t base = (((size_t)(it.start + qi) * p.H + it.h) * DV + col) / 4;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            reinterpret_cast<float4*>(p.o1)[base + i] =
                                make_float4(__uint_as_float(o1[4 * i]) * il1, __uint_as_float(o1[4 * i + 1]) * il1,
                                            __uint_as_float(o1[4 * i + 2]) * il1, __uint_as_float(o1[4 * i + 3]) * il1);
                            reinterpret_cast<float4*>(p.o2)[base + i] =
                                make_float4(__uint_as_float(o2[4 * i]) * il2, __uint_as_float(o2[4 * i + 1]) * il2,
                                            __uint_as_float(o2[4 * i + 2]) * il2, __uint_as_float(o2[4 * i + 3]) * il2);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float dq[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            dq[e] = diff_combine(__uint_as_float(o1[4 * i + e]), il1, __uint_as_float(o2[4 * i + e]), il2,
                                                 lam);
                            ssp = fmaf(dq[e], dq[e], ssp);
                        }
                        *d_chunk(hf, qb, c4 * 4 + i) = make_float4(dq[0], dq[1], dq[2], dq[3]);
                    }
                }
                ss_half[hf] = ssp;
            }
            const float ss = ss_half[0] + ss_half[1];
            const float post = (1.f - p.lambda_init) / sqrtf(ss / (float)DV + p.eps);
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                                  ((size_t)(it.start + (store ? qi : 0)) * p.H + it.h) * DV);
#pragma unroll 1
            for (int ch = 0; ch < DV / 32; ++ch) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 dq = *d_chunk(ch >> 1, qb, (ch & 1) * 8 + i);
                    const int e = ch * 32 + 4 * i;
                    pk[2 * i] = pack_bf16x2(dq.x * post * ms.w[e], dq.y * post * ms.w[e + 1]);
                    pk[2 * i + 1] = pack_bf16x2(dq.z * post * ms.w[e + 2], dq.w * post * ms.w[e + 3]);
                }
                if (store) {
#pragma unroll
                    for (int g4 = 0; g4 < 4; ++g4)
                        dst[ch * 4 + g4] = make_uint4(pk[4 * g4], pk[4 * g4 + 1], pk[4 * g4 + 2], pk[4 * g4 + 3]);
                }
            }
            // The item's Q box (the second half of D) goes back to the producer.
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_q_empty(qb));
            ++items;
        }
    } else {
        setmaxnreg_dec<REG_COPY>();
        if (warp == PRODUCER_WARP) {
            // ================================================= TMA producer ===
            // Item k of the longest-first order (query tile descending, then sequence,
            // then head, empty (tile, sequence) pairs left out): rank q = n_qt - 1 - qt
            // holds the sequences with at least n_qt - q tiles; a cursor walks the ranks
            // as k grows. This CTA takes k = r G + c on even rounds r, r G + G - 1 - c
            // on odd ones.
            if (lane == 0) {
                const uint64_t pol_q = l2_policy_evict_first(), pol_kv = l2_policy_evict_last();
                const bool packed = p.cu_seqlens != nullptr;
                auto tiles_of = [&](int sq_i) { return packed ? (int)ms.tiles[sq_i] : n_qt; };
                auto count_rank = [&](int q) {  // sequences with at least n_qt - q tiles
                    if (!packed) return p.num_seqs;
                    int n = 0;
                    for (int sq_i = 0; sq_i < p.num_seqs; ++sq_i) n += tiles_of(sq_i) >= n_qt - q;
                    return n;
                };
                long long total = 0;
                for (int sq_i = 0; sq_i < p.num_seqs; ++sq_i) total += tiles_of(sq_i);
                const long long n_valid = total * p.H;
                const long long G = gridDim.x;
                int q = 0, cq = count_rank(0);
                long long P = 0;
                int tile = 0, items = 0;
                int q_issued = 0, k_issued = 0, v_issued = 0;  // loads issued, for the drain below
                bool ok = true;
                for (long long r = 0; ok && r * G < n_valid; ++r) {
                    const long long k = r * G + ((r & 1) ? G - 1 - blockIdx.x : blockIdx.x);
                    if (k >= n_valid) continue;
                    while (k >= P + (long long)cq * p.H) {
                        P += (long long)cq * p.H;
                        cq = count_rank(++q);
                    }
                    const int j = (int)((k - P) / p.H), h = (int)((k - P) % p.H);
                    int sq_i = j;
                    if (packed) {
                        int cnt = -1;
                        for (sq_i = 0; sq_i < p.num_seqs; ++sq_i)
                            if (tiles_of(sq_i) >= n_qt - q && ++cnt == j) break;
                    }
                    Item it{};
                    it.h = h;
                    it.qt = n_qt - 1 - q;
                    it.start = packed ? p.cu_seqlens[sq_i] : sq_i * p.seqlen;
                    it.len = packed ? p.cu_seqlens[sq_i + 1] - it.start : p.seqlen;
                    it.n_kv = p.causal ? it.qt + 1 : (it.len + BN - 1) / BN;
                    const int slot = items % NSLOT;
                    if (!(ok = mbar_wait(bar_item_empty(slot), ((uint32_t)(items / NSLOT) & 1u) ^ 1u, ab))) break;
                    ms.work[slot] = it;
                    mbar_arrive(bar_item_full(slot));
                    if (p.inject == 1) {  // test hook: no loads, so the other roles' waits run out
                        ++items;
                        continue;
                    }
                    const int g = h / (p.H / p.Hkv);
                    const int qb = items % QBUF;
                    if (!(ok = mbar_wait(bar_q_empty(qb), ((uint32_t)(items / QBUF) & 1u) ^ 1u, ab))) break;
                    const int row_q = it.start + it.qt * BM;
                    mbar_arrive_expect_tx(bar_q_full(qb), Q_BYTES);
                    tma_load_2d(sq(qb), &tm_q, bar_q_full(qb), h * 2 * HD, row_q, pol_q);
                    tma_load_2d(sq(qb) + BOX_BYTES, &tm_q, bar_q_full(qb), h * 2 * HD + HD, row_q, pol_q);
                    ++q_issued;
                    for (int jj = 0; jj < it.n_kv; ++jj, ++tile) {
                        const int s = tile % STAGES;
                        const uint32_t ph = ((uint32_t)(tile / STAGES) & 1u) ^ 1u;
                        const int row = it.start + jj * BN;
                        if (!(ok = mbar_wait(bar_k_empty(s), ph, ab))) break;
                        mbar_arrive_expect_tx(bar_k_full(s), K_BYTES);
                        tma_load_2d(sk(s), &tm_k, bar_k_full(s), g * 2 * HD, row, pol_kv);
                        tma_load_2d(sk(s) + BOX_BYTES, &tm_k, bar_k_full(s), g * 2 * HD + HD, row, pol_kv);
                        ++k_issued;
                        if (!(ok = mbar_wait(bar_v_empty(s), ph, ab))) break;
                        mbar_arrive_expect_tx(bar_v_full(s), V_BYTES);
                        tma_load_2d(sv(s), &tm_v, bar_v_full(s), g * DV, row, pol_kv);
                        tma_load_2d(sv(s) + BOX_BYTES, &tm_v, bar_v_full(s), g * DV + 64, row, pol_kv);
                        ++v_issued;
                    }
                    ++items;
                }
                // end of the items: a sentinel in the next slot
                const int slot = items % NSLOT;
                if (ok && mbar_wait(bar_item_empty(slot), ((uint32_t)(items / NSLOT) & 1u) ^ 1u, ab)) {
                    Item end{};
                    end.n_kv = -1;
                    ms.work[slot] = end;
                    mbar_arrive(bar_item_full(slot));
                }
                // Let every copy this CTA started land before shared memory goes away:
                // the last Q load of each box and the last K and V load of each stage.
                for (int k = q_issued > QBUF ? q_issued - QBUF : 0; k < q_issued; ++k)
                    mbar_wait_drain(bar_q_full(k % QBUF), (uint32_t)(k / QBUF) & 1u, p.timeout_ns);
                for (int jj = k_issued > STAGES ? k_issued - STAGES : 0; jj < k_issued; ++jj)
                    mbar_wait_drain(bar_k_full(jj % STAGES), (uint32_t)(jj / STAGES) & 1u, p.timeout_ns);
                for (int jj = v_issued > STAGES ? v_issued - STAGES : 0; jj < v_issued; ++jj)
                    mbar_wait_drain(bar_v_full(jj % STAGES), (uint32_t)(jj / STAGES) & 1u, p.timeout_ns);
            }
            __syncwarp();
        } else if (warp == MMA_WARP) {
            // ==================================================== MMA issuer ===
            // Items are fetched one ahead: at an item's last tile the next item's first
            // score MMAs of component 1 follow this item's last P V of component 1 when
            // that item's Q box and keys have already landed (otherwise they follow the
            // item's last P V of component 2, so that its O is not held back).
            constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, DV, true);
            constexpr uint64_t KSTEP = 32 >> 4, VSTEP = (16 * 128) >> 4, BOX = BOX_BYTES >> 4;
            constexpr uint64_t QSTG = Q_BYTES >> 4, KSTG = K_BYTES >> 4, VSTG = V_BYTES >> 4;
            const uint64_t qdesc = desc_kmajor(sq(0)), kdesc = desc_kmajor(sk(0)), vdesc = desc_value(sv(0));
            auto issue_s = [&](int c, int qb, int tile) {
                const uint64_t a0 = qdesc + (uint64_t)qb * QSTG + (uint64_t)c * BOX;
                const uint64_t b0 = kdesc + (uint64_t)(tile % STAGES) * KSTG + (uint64_t)c * BOX;
                const uint32_t d = tmem + col_s(c);
    #pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) mma_ss_elect(d, a0 + kk * KSTEP, b0 + kk * KSTEP, idesc_s, kk > 0 ? 1u : 0u);
                mma_commit_elect(bar_s_full(c));
                if (c == 1) mma_commit_elect(bar_k_empty(tile % STAGES));  // both score MMAs of the tile issued
            };
            auto issue_pv = [&](int c, int tile, bool first) {
                const uint64_t b0 = vdesc + (uint64_t)(tile % STAGES) * VSTG;
                const uint32_t d = tmem + col_o(c), a = tmem + col_s(c);
    #pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts_elect(d, a + kk * 8, b0 + kk * VSTEP, idesc_pv, (kk > 0 || !first) ? 1u : 0u);
            };
            auto fetch = [&](int k, int& n_kv) {  // the MMA warp needs only the item's key tile count
                const int slot = k % NSLOT;
                if (!warp_all(mbar_wait(bar_item_full(slot), (uint32_t)(k / NSLOT) & 1u, ab))) return false;
                n_kv = ms.work[slot].n_kv;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_item_empty(slot));
                return true;
            };
            // Q box of item k and the keys of `tile` landed: waiting, or only probing.
            auto s_ready = [&](int k, int tile) {
                return warp_all(mbar_wait(bar_q_full(k % QBUF), (uint32_t)(k / QBUF) & 1u, ab)) &&
                       warp_all(mbar_wait(bar_k_full(tile % STAGES), (uint32_t)(tile / STAGES) & 1u, ab));
            };
            auto s_ready_now = [&](int k, int tile) {
                return warp_all(mbar_try_wait(bar_q_full(k % QBUF), (uint32_t)(k / QBUF) & 1u)) &&
                       warp_all(mbar_try_wait(bar_k_full(tile % STAGES), (uint32_t)(tile / STAGES) & 1u));
            };
            int tile = 0, items = 0, cur_n = -1;
            bool ok = fetch(0, cur_n);
            if (ok && cur_n >= 0 && (ok = s_ready(0, 0))) {
                tc_fence_after();
                issue_s(0, 0, 0);
                issue_s(1, 0, 0);
            }
            while (ok && cur_n >= 0) {
                const int qb = items % QBUF;
                int nxt_n = -1;
                bool next_s1 = false;  // the next item's first component-1 scores are issued
                for (int j = 0; j < cur_n; ++j, ++tile) {
                    const int s = tile % STAGES;
                    const bool last = j + 1 == cur_n;
                    const int t1 = tile + 1;
                    if (!(ok = warp_all(mbar_wait(bar_v_full(s), (uint32_t)(tile / STAGES) & 1u, ab)))) break;
                    if (j == 0 && !(ok = warp_all(mbar_wait(bar_o_empty, ((uint32_t)items & 1u) ^ 1u, ab)))) break;
                    if (!(ok = warp_all(mbar_wait(bar_p_ready(0), (uint32_t)tile & 1u, ab)))) break;
                    tc_fence_after();
                    issue_pv(0, tile, j == 0);
                    if (!last) {
                        if (!(ok = warp_all(mbar_wait(bar_k_full(t1 % STAGES), (uint32_t)(t1 / STAGES) & 1u, ab)))) break;
                        issue_s(0, qb, t1);
                    } else {
                        if (!(ok = fetch(items + 1, nxt_n))) break;
                        if (nxt_n >= 0 && s_ready_now(items + 1, t1)) {
                            tc_fence_after();
                            issue_s(0, (items + 1) % QBUF, t1);
                            next_s1 = true;
                        }
                    }
                    if (!(ok = warp_all(mbar_wait(bar_p_ready(1), (uint32_t)tile & 1u, ab)))) break;
                    tc_fence_after();
                    issue_pv(1, tile, j == 0);
                    mma_commit_elect(bar_v_empty(s));
                    if (!last) issue_s(1, qb, t1);
                }
                if (!ok) break;
                mma_commit_elect(bar_o_full);  // every P V of this item issued
                ++items;
                cur_n = nxt_n;
                if (cur_n < 0) break;
                if (!next_s1) {
                    if (!(ok = s_ready(items, tile))) break;
                    tc_fence_after();
                    issue_s(0, items % QBUF, tile);
                }
                issue_s(1, items % QBUF, tile);
            }
            // every MMA issued has completed before TMEM is released
            mma_commit_elect(bar_mma_done);
            mbar_wait_drain(bar_mma_done, 0, p.timeout_ns);
            __syncwarp();
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

cudaError_t launch_fwd_bf16_persistent(const FwdParams& p, const FwdTensorMaps& maps, cudaStream_t stream) {
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !attr_done[dev]) {
        err = cudaFuncSetAttribute(diffattn_fwd_bf16_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)SMEM_BYTES);
        if (err != cudaSuccess) return err;
        attr_done[dev] = true;
    }
    // the register split needs the launch to hold REG_LAUNCH registers a thread
    static int launch_regs = 0;
    if (launch_regs == 0) {
        cudaFuncAttributes fa{};
        err = cudaFuncGetAttributes(&fa, diffattn_fwd_bf16_persistent_kernel);
        if (err != cudaSuccess) return err;
        launch_regs = fa.numRegs;
    }
    if (launch_regs * NUM_THREADS < REG_NEED || launch_regs < REG_LAUNCH) return cudaErrorInvalidConfiguration;
    int sms = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const int n_qt = (p.max_seqlen + BM - 1) / BM;
    if (p.cu_seqlens != nullptr && p.num_seqs > MAX_PACKED_SEQS) return cudaErrorInvalidValue;
    const long long n_items = (long long)n_qt * p.H * p.num_seqs;  // upper bound (packed: some are empty)
    if (n_items <= 0 || n_items > INT32_MAX) return cudaErrorInvalidValue;
    const int grid = (int)(n_items < sms ? n_items : sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, diffattn_fwd_bf16_persistent_kernel, maps.q, maps.k, maps.v, p, n_qt);
}

}  // namespace diffattn
