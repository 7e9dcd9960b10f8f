// Fused differential-attention forward for sm_103a (bf16 in, fp32 accumulate,
// bf16 out), d = 64, dv = 128.
//
// One CTA owns 128 query rows of one diff head of one sequence and walks the
// visible 128-key tiles. Per tile it computes, on the tensor cores,
//   S1 = Q1 K1^T, S2 = Q2 K2^T           ("DiffTransformer.py", forward,
//                                          "Compute attention scores")
// keeps two online-softmax states (running max m_c, running sum l_c), writes
// the unnormalised probabilities P_c back to tensor memory as bf16 and
// accumulates O_c += P_c V with the SAME value tile for both components
// ("LlamaDiffSdpaAttention.py", forward: two attention calls over one
// value_states). The epilogue forms O1/l1 - lambda O2/l2 (the output-difference
// form attn1 - lambda_full * attn2), applies the per-head RMSNorm over dv, the
// weight and (1 - lambda_init) ("DiffTransformer.py", forward, "Normalize each
// head independently using RMSNorm", "Scale the normalized output") and stores
// bf16.
//
// Roles (320 threads):
//   warps 0-3  softmax of component 1 (TMEM lanes 0-127 = query rows), then
//              the epilogue for values 0-63 of every row;
//   warps 4-7  softmax of component 2, then the epilogue for values 64-127;
//   warp  8    TMA producer (Q once, K1|K2 and V per tile into a STAGES ring);
//   warp  9    TMEM allocator and single-thread tcgen05.mma issuer.
// Tensor memory (512 columns of 128 lanes x 32 bit):
//   [0,128) S1 / P1 (bf16 pairs in the first 64 columns), [128,256) S2 / P2,
//   [256,384) O1, [384,512) O2.
// Shared memory: Q1|Q2 (32 KB) + STAGES x (K1|K2 32 KB + V 32 KB), all
// 128-byte swizzled boxes of [128 rows x 64 bf16] as written by TMA.
//
// Every wait is bounded (see sm103a_ptx.cuh); on a timeout the CTA records the
// error, lets its copies and MMAs in flight finish, frees TMEM and returns.
//
// Per component the tile loop is a chain: softmax(j) -> P_c(j) V and S_c(j+1)
// on the tensor pipe -> softmax(j+1); the two components' chains interleave on
// the tensor pipe. (A variant with two 64-key S buffers per component, which
// breaks the chain, measured slower on GB300: it doubles the MMA instruction
// and barrier count per key.)
#include <cuda_bf16.h>

#include "internal.h"
#include "rope_q.cuh"
#include "lambda_warp.cuh"
#include "sm103a_ptx.cuh"
#include "softmax_exact.cuh"

namespace diffattn {
namespace {

constexpr int BM = 128;                 // query rows per CTA
constexpr int BN = 128;                 // keys per tile
constexpr int HD = 64;                  // component dim d
constexpr int DV = 128;                 // value dim
constexpr int STAGES = 3;               // K/V ring depth
constexpr int NUM_THREADS = 320;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr uint32_t BOX_BYTES = BM * HD * 2;          // one [128 x 64] bf16 box: 16 KB
constexpr uint32_t Q_BYTES = 2 * BOX_BYTES;
constexpr uint32_t K_BYTES = 2 * BOX_BYTES;
constexpr uint32_t V_BYTES = 2 * BOX_BYTES;
constexpr uint32_t STAGE_BYTES = K_BYTES + V_BYTES;
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_STAGE0 = Q_BYTES;
constexpr uint32_t OFF_MISC = OFF_STAGE0 + STAGES * STAGE_BYTES;
// Epilogue staging in the K / V stages (every load consumed by then): the bf16 output
// in the first 32 KB, the training outputs O1 / l1 and O2 / l2 (fp32) after it, each as
// four [128 rows x 32] boxes of 16 KB with the 128-byte swizzle.
constexpr uint32_t O_BOX = BM * 32 * 4;
constexpr uint32_t OFF_OSTAGE = OFF_STAGE0 + 2 * BOX_BYTES;
static_assert(OFF_OSTAGE + 8 * O_BOX <= OFF_MISC, "training-output staging fits the stages");
constexpr uint32_t MISC_BYTES = 1024;
constexpr uint32_t SMEM_BYTES = 1024 /* alignment slack */ + OFF_MISC + MISC_BYTES;
static_assert(SMEM_BYTES <= 232448, "exceeds the per-block shared memory limit");

constexpr uint32_t TMEM_COLS = 512;
__device__ __forceinline__ uint32_t col_s(int c) { return (uint32_t)c * 128u; }        // S_c / P_c
__device__ __forceinline__ uint32_t col_o(int c) { return 256u + (uint32_t)c * 128u; } // O_c

// A maximum-first tile (the first, or the rare exact step) moves the reference maximum
// only when its own maximum is more than 2^8 above it (in log2 units).
constexpr float RESCALE_THRESHOLD = 8.0f;
// Past the first tile, the row sum of a tile above which the warp takes it maximum-first.
constexpr float EXACT_SUM = 4294967296.0f;  // 2^32

struct Misc {  // lives at OFF_MISC
    uint64_t q_full;
    uint64_t k_full[STAGES];
    uint64_t v_full[STAGES];
    uint64_t kv_empty[STAGES];
    uint64_t s_full[2];
    uint64_t p_ready[2];
    uint64_t o_full;
    uint64_t w_full;  // the norm weight and lambda have landed in shared memory
    uint64_t q_rot;   // with the rotary embedding: Q rotated in shared memory
    uint64_t tab_full;  // with the rotary embedding: the tile's cos / sin rows in shared memory
    uint32_t tmem_base;
    int abort_flag;
    float lam;        // lambda of this head, and the norm weight, staged at setup
    float w[DV];
};
static_assert(sizeof(Misc) <= MISC_BYTES, "misc area too small");

// K-major operand (rows of 64 bf16 = 128 B, 8-row groups 1024 B apart).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) { return smem_desc_sw128(saddr, 16, 1024); }
// MN-major value operand: 64-column halves 16 KB apart, 8-key groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_value(uint32_t saddr) { return smem_desc_sw128(saddr, BOX_BYTES, 1024); }

// True on every lane iff `pred` holds on every lane of the warp.
__device__ __forceinline__ bool warp_all(bool pred) { return __all_sync(0xffffffffu, pred); }

// The kernel body; TRAIN: the training form (O1 / l1 and O2 / l2 of full tiles staged in
// shared memory for bulk tensor stores); LAMBDA: lambda formed from its parameter vectors
// by the producer warp once its copies have landed (only the epilogue reads it). Each
// form is a kernel of its own, so that the plain inference form keeps its code.
template <bool TRAIN, bool LAMBDA>
__device__ __forceinline__ void fwd_bf16_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                              const CUtensorMap& tm_out, const CUtensorMap& tm_o1,
                                              const CUtensorMap& tm_o2, const FwdParams& p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc& ms = *reinterpret_cast<Misc*>(smem + OFF_MISC);
    const uint32_t sbase = smem_u32(smem);

    // Launched as a programmatic dependent of the previous kernel on the stream
    // (typically the lambda kernel): nothing is read before it has completed,
    // except with lambda_pending, where that kernel writes lambda alone and only
    // the producer's read of lambda waits (below).
    if (!p.lambda_pending) griddep_wait();
    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Launch order within a sequence: groups of group_heads heads one after another,
    // and within a group the query tiles longest first, the group's heads fastest.
    // The CTAs in flight then stream the K / V of one group, which the host sizes
    // to stay in L2.
    const int n_qt = (p.max_seqlen + BM - 1) / BM;
    const int hg = p.group_heads;
    const int grp = (int)blockIdx.x / (n_qt * hg), rem = (int)blockIdx.x - grp * (n_qt * hg);
    const int h = grp * hg + rem % hg;
    const int qt = n_qt - 1 - rem / hg;  // longest query tiles are scheduled first
    const int seq = blockIdx.z;

    // ---- sequence bounds; uniform over the CTA -----------------------------
    int start, len;
    if (p.cu_seqlens != nullptr) {
        start = p.cu_seqlens[seq];
        const int end = p.cu_seqlens[seq + 1];
        const bool bad = start < 0 || end < start || end > p.total_tokens || end - start > p.max_seqlen ||
                         (seq == 0 && start != 0) || (seq == p.num_seqs - 1 && end != p.total_tokens);
        if (bad) {
            if (threadIdx.x == 0) atomicOr(p.error_word, kErrBadSeqlens);
            return;
        }
        len = end - start;
    } else {
        start = seq * p.seqlen;
        len = p.seqlen;
    }
    if (qt * BM >= len) return;
    const int n_kv = p.causal ? qt + 1 : (len + BN - 1) / BN;
    const int g = h / (p.H / p.Hkv);

    const uint32_t bar_q_full = smem_u32(&ms.q_full);
    auto bar_k_full = [&](int s) { return smem_u32(&ms.k_full[s]); };
    auto bar_v_full = [&](int s) { return smem_u32(&ms.v_full[s]); };
    auto bar_kv_empty = [&](int s) { return smem_u32(&ms.kv_empty[s]); };
    auto bar_s_full = [&](int c) { return smem_u32(&ms.s_full[c]); };
    auto bar_p_ready = [&](int c) { return smem_u32(&ms.p_ready[c]); };
    const uint32_t bar_o_full = smem_u32(&ms.o_full);
    const uint32_t bar_w_full = smem_u32(&ms.w_full);
    const uint32_t bar_q_rot = smem_u32(&ms.q_rot);
    const uint32_t bar_tab_full = smem_u32(&ms.tab_full);
    const bool rope = p.rope_cos != nullptr;
    // With the rotary embedding the tile's cos / sin rows (one contiguous block per
    // table) come by bulk copy into the last K/V stage, whose first load waits until
    // Q has been rotated: read from shared memory, the 64 KB of table entries a
    // tile needs do not queue ahead of the Q and K loads (as 4096 plain loads a CTA
    // they had delayed Q by ~4.6 us).
    const int rope_rows = rope ? max(0, min(BM, p.rope_npos - qt * BM)) : 0;
    const uint32_t rope_row_bytes = rope ? (uint32_t)(p.rope_dim / 2) * 4u : 0u;
    const uint32_t sq = sbase + OFF_Q;
    auto sk = [&](int s) { return sbase + OFF_STAGE0 + (uint32_t)s * STAGE_BYTES; };
    auto sv = [&](int s) { return sbase + OFF_STAGE0 + (uint32_t)s * STAGE_BYTES + K_BYTES; };

    // ---- setup --------------------------------------------------------------
    // The producer issues Q and the first STAGES key / value tiles as soon as its
    // barriers exist, before the CTA-wide barrier, and the norm weight and lambda
    // come by cp.async on their own barrier (waited for only by the epilogue): on a
    // cold L2 the plain loads of those had held the first TMA loads back ~2 us.
    const uint64_t pol_q = l2_policy_evict_first();
    const uint64_t pol_kv = l2_policy_evict_last();
    auto load_kv = [&](int j) {
        const int s = j % STAGES;
        const int row = start + j * BN;
        mbar_arrive_expect_tx(bar_k_full(s), K_BYTES);
        tma_load_2d(sk(s), &tm_k, bar_k_full(s), g * 2 * HD, row, pol_kv);
        tma_load_2d(sk(s) + BOX_BYTES, &tm_k, bar_k_full(s), g * 2 * HD + HD, row, pol_kv);
        mbar_arrive_expect_tx(bar_v_full(s), V_BYTES);
        tma_load_2d(sv(s), &tm_v, bar_v_full(s), g * DV, row, pol_kv);
        tma_load_2d(sv(s) + BOX_BYTES, &tm_v, bar_v_full(s), g * DV + 64, row, pol_kv);
    };
    // With the test hook set, no load is issued: the barriers the other roles
    // wait on are never armed, so their bounded waits run out.
    // tiles loaded before the CTA barrier (with the rotary embedding the last stage
    // holds the tables until Q is rotated)
    const int early = p.inject == 1 ? 0 : min(n_kv, rope ? STAGES - 1 : STAGES);
    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_init(bar_q_full, 1);
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(bar_k_full(s), 1);
                mbar_init(bar_v_full(s), 1);
                mbar_init(bar_kv_empty(s), 1);
            }
            for (int c = 0; c < 2; ++c) {
                mbar_init(bar_s_full(c), 1);
                mbar_init(bar_p_ready(c), 128);
            }
            mbar_init(bar_o_full, 1);
            mbar_init(bar_w_full, LAMBDA ? 33 : 32);  // one cp.async arrive per lane, and lambda's
            mbar_init(bar_q_rot, 256);  // every softmax thread, after rotating its part of Q
            mbar_init(bar_tab_full, 1);
            ms.abort_flag = 0;
            fence_barrier_init();
            if (p.inject != 1) {
                const int row_q = start + qt * BM;
                mbar_arrive_expect_tx(bar_q_full, Q_BYTES);
                tma_load_2d(sq, &tm_q, bar_q_full, h * 2 * HD, row_q, pol_q);
                tma_load_2d(sq + BOX_BYTES, &tm_q, bar_q_full, h * 2 * HD + HD, row_q, pol_q);
                for (int j = 0; j < early; ++j) load_kv(j);  // fresh stages: nothing to wait for
                if (rope) {
                    const uint32_t tab = sk(STAGES - 1), bytes = (uint32_t)rope_rows * rope_row_bytes;
                    mbar_arrive_expect_tx(bar_tab_full, 2u * bytes);
                    if (bytes > 0) {
                        const size_t off = (size_t)qt * BM * (p.rope_dim / 2);
                        bulk_copy_g2s(tab, p.rope_cos + off, bytes, bar_tab_full);
                        bulk_copy_g2s(tab + 32768u, p.rope_sin + off, bytes, bar_tab_full);
                    }
                }
            }
        }
        __syncwarp();  // the barriers exist before any lane arrives on them
        if (p.lambda_pending) griddep_wait();  // lambda comes from the preceding grid
        for (int i = lane; i < DV; i += 32) cp_async4(smem_u32(&ms.w[i]), p.subln_w + i);
        if (lane == 0 && !LAMBDA) cp_async4(smem_u32(&ms.lam), p.lambda + h * p.lambda_stride);
        cp_async_arrive_noinc(bar_w_full);
    }
    if (warp == MMA_WARP) tmem_alloc(smem_u32(&ms.tmem_base), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;
    const AbortState ab{&ms.abort_flag, p.error_word, p.timeout_ns};

    if (warp == PRODUCER_WARP) {
        // ================================================= TMA producer ===
        if (lane == 0 && p.inject != 1) {
            int issued = early;
            for (int j = early; j < n_kv; ++j) {
                const int s = j % STAGES;
                const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
                if (rope && j == STAGES - 1 && !mbar_wait(bar_q_rot, 0, ab)) break;  // the tables are read
                if (!mbar_wait(bar_kv_empty(s), ph ^ 1u, ab)) break;
                load_kv(j);
                issued = j + 1;
            }
            // Let every copy this CTA started land before shared memory goes away.
            mbar_wait_drain(bar_q_full, 0, p.timeout_ns);
            if (rope) mbar_wait_drain(bar_tab_full, 0, p.timeout_ns);
            for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j) {
                const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
                mbar_wait_drain(bar_k_full(j % STAGES), ph, p.timeout_ns);
                mbar_wait_drain(bar_v_full(j % STAGES), ph, p.timeout_ns);
            }
        }
        cp_async_wait_all();  // the weight copies have landed, whatever the epilogue did
        __syncwarp();
        if (LAMBDA) {
            // the CTAs of the first query tile write lambda out (all of them, for a shared one)
            const int set = p.lambda_stride ? h : 0;
            const size_t base = (size_t)set * p.lambda_d;
            const float lam = lambda_value_warp(p.lq1 + base, p.lk1 + base, p.lq2 + base, p.lk2 + base, p.lambda_d,
                                                p.lambda_init, lane);
            if (lane == 0) {
                ms.lam = lam;
                if (qt == 0) atomicExch(p.lambda_out + set, lam);
                mbar_arrive(bar_w_full);  // releases the store above to the epilogue's wait
            }
        }
    } else if (warp == MMA_WARP) {
        // ==================================================== MMA issuer ===
        // The whole warp walks the loop with warp-uniform values; one elected
        // lane issues each tcgen05 instruction. Descriptors are built once and
        // advanced by constant offsets of their start-address field (16-byte
        // units): with per-instruction descriptor arithmetic, issue rather than
        // the tensor pipe limited the MMA rate.
        constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, DV, true);
        constexpr uint64_t KSTEP = 32 >> 4, VSTEP = (16 * 128) >> 4, STG = STAGE_BYTES >> 4, BOX = BOX_BYTES >> 4;
        const uint64_t qdesc = desc_kmajor(sq), kdesc = desc_kmajor(sk(0)), vdesc = desc_value(sv(0));
        auto issue_s = [&](int c, int j) {
            const uint64_t a0 = qdesc + (uint64_t)c * BOX;
            const uint64_t b0 = kdesc + (uint64_t)(j % STAGES) * STG + (uint64_t)c * BOX;
            const uint32_t d = tmem + col_s(c);
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) mma_ss_elect(d, a0 + kk * KSTEP, b0 + kk * KSTEP, idesc_s, kk > 0 ? 1u : 0u);
            mma_commit_elect(bar_s_full(c));
        };
        auto issue_pv = [&](int c, int j) {
            const uint64_t b0 = vdesc + (uint64_t)(j % STAGES) * STG;
            const uint32_t d = tmem + col_o(c), a = tmem + col_s(c);
            const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) mma_ts_elect(d, a + kk * 8, b0 + kk * VSTEP, idesc_pv, kk > 0 ? 1u : acc0);
        };
        bool ok = warp_all(mbar_wait(rope ? bar_q_rot : bar_q_full, 0, ab)) && warp_all(mbar_wait(bar_k_full(0), 0, ab));
        if (ok) { tc_fence_after(); issue_s(0, 0); issue_s(1, 0); }
        for (int j = 0; ok && j < n_kv; ++j) {
            const int s = j % STAGES;
            const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
            const bool has_next = j + 1 < n_kv;
            const int s1 = (j + 1) % STAGES;
            const uint32_t ph1 = (uint32_t)((j + 1) / STAGES) & 1u;
            if (!(ok = warp_all(mbar_wait(bar_v_full(s), ph, ab)))) break;
            if (!(ok = warp_all(mbar_wait(bar_p_ready(0), (uint32_t)j & 1u, ab)))) break;
            tc_fence_after();
            issue_pv(0, j);
            if (has_next) {
                if (!(ok = warp_all(mbar_wait(bar_k_full(s1), ph1, ab)))) break;
                issue_s(0, j + 1);
            }
            if (!(ok = warp_all(mbar_wait(bar_p_ready(1), (uint32_t)j & 1u, ab)))) break;
            tc_fence_after();
            issue_pv(1, j);
            mma_commit_elect(bar_kv_empty(s));
            if (has_next) issue_s(1, j + 1);
        }
        mma_commit_elect(bar_o_full);
        mbar_wait_drain(bar_o_full, 0, p.timeout_ns);
        __syncwarp();
    } else {
        // ======================================== softmax (warps 0-7) ===
        const int c = warp >> 2;
        const int r = (warp & 3) * 32 + lane;  // query row in the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t t_s = tmem + lane_off + col_s(c);
        const uint32_t t_o = tmem + lane_off + col_o(c);
        const int qi = qt * BM + r;
        const float sl2 = p.scale_log2;
        const uint64_t sl2p = f2_pack(sl2, sl2);
        float m = -INFINITY;  // running max of scores * scale * log2(e)
        float l = 0.f;        // running sum of 2^(x - m)
        bool ok = true;
        if (rope) {
            // Rotary embedding of the tile's queries before the first score MMA. Thread t
            // takes unit t % U of rows t / U + (256 / U) m: consecutive threads read
            // consecutive table entries and distinct Q chunks (no bank conflicts).
            const int t = threadIdx.x, U = rope_units(p.rope_interleaved), step = 256 / U, u = t % U;
            ok = warp_all(mbar_wait(bar_q_full, 0, ab)) && warp_all(mbar_wait(bar_tab_full, 0, ab));
            bool bad = false;
            if (ok) {
                const uint32_t tab = sk(STAGES - 1);
                for (int rr = t / U; rr < BM; rr += step) {
                    if (rr >= rope_rows) {  // position past the tables: left unrotated
                        bad |= qt * BM + rr < len;
                        continue;
                    }
                    rope_unit_smem(sq, BOX_BYTES, rr, u, tab, tab + 32768u, p.rope_dim, p.rope_interleaved);
                }
            }
            if (bad) atomicOr(p.error_word, kErrBadPositions);
            fence_proxy_async_smem();  // the rotated rows, visible to the MMAs
            mbar_arrive(bar_q_rot);
        }
        // The reference maximum m is the first tile's: later tiles are exponentiated with it
        // at once (no maximum pass ahead of the exponentials), P staying below 2^32 unless
        // a tile's scores rise that far above it; then the warp takes that tile
        // maximum-first (softmax_exact.cuh). O_c / l_c and lse do not depend on the
        // reference, and relative precision does not depend on the magnitude.
        for (int j = 0; j < n_kv; ++j) {
            if (!(ok = warp_all(mbar_wait(bar_s_full(c), (uint32_t)j & 1u, ab)))) break;
            tc_fence_after();
            float x[BN];
            {
                // one wide load (measured faster than four 32-column loads)
                uint32_t sr[BN];
                tmem_ld128(t_s, sr);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < BN; ++e) x[e] = __uint_as_float(sr[e]);
            }
            const int kbase = j * BN;
            const bool masked = (p.causal && j == qt) || kbase + BN > len;
            // keys < lim of this tile are visible
            const int lim = masked ? (p.causal ? min(qi + 1, len) : len) - kbase : BN;
            if (masked) {
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
                    alpha = ex2_approx(m - m_tile);  // 0 on the first tile (m = -inf)
                    m = m_tile;
                }
            }
            // x * scale * log2(e) - m and the row sum as packed fp32 pairs (half the
            // instructions of the scalar forms)
            const uint64_t nmp = f2_pack(-m, -m);
            uint64_t sa = 0, sb = 0;
            // P_c (bf16 pairs: column i holds keys 2i (low half) and 2i+1) over S_c, stored
            // 32 keys at a time so the TMEM stores overlap the next chunk's exponentials.
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
            // A row sum above 2^32 (or not finite) means a maximum far above m: the warp takes
            // the tile maximum-first, and O_c (the sum through tile j-1: S_c(j) was issued after
            // PV_c(j-1)) moves to the new reference. Rows past the sequence end (never stored)
            // take no part in the choice, so that it depends on the item's own rows alone.
            if (j > 0 && __any_sync(0xffffffffu, qi < len && !(sum <= EXACT_SUM))) {
                sum = softmax_exact_tile<BN>(
                    t_s, sq + (uint32_t)c * BOX_BYTES + (uint32_t)r * 128u, r,
                    reinterpret_cast<const __nv_bfloat16*>(p.k) + ((size_t)(start + kbase) * p.Hkv + g) * (2 * HD) +
                        c * HD,
                    (size_t)p.Hkv * (2 * HD), lim, sl2, RESCALE_THRESHOLD, m, alpha);
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

        // Training outputs: log2-sum-exp of the scaled scores per component,
        // lse_c = m_c + log2(l_c), so that P_c = 2^(S_c * scale * log2(e) - lse_c).
        if (ok && p.lse != nullptr && qi < len) p.lse[((size_t)(start + qi) * p.H + h) * 2 + c] = m + __log2f(l);
        // ---- epilogue, split by columns: warpgroup c handles values [64c, 64c + 64)
        // of every row. 1/l_c and the partial sums of squares cross between the two
        // warpgroups through the Q1 box (2 KB of it), once every softmax warp has left
        // its loop: every MMA reading Q has retired then (the tensor pipe completes in
        // issue order), and so has every maximum-first step, which reads Q rows.
        float* xch = reinterpret_cast<float*>(smem + OFF_Q);  // [0,256): 1/l_c, [256,512): sum D^2
        named_barrier_sync(1, 256);
        xch[c * BM + r] = 1.f / l;
        named_barrier_sync(1, 256);
        ok = warp_all(ok && mbar_wait(bar_o_full, 0, ab));
        ok = warp_all(ok && mbar_wait(bar_w_full, 0, ab));
        const bool store = qi < len;
        // training outputs of a tile wholly inside its sequence: staged for bulk tensor stores
        const bool stage_o = TRAIN && qt * BM + BM <= len;
        float D[64];
        float ssp = 0.f;
        if (ok) {
            tc_fence_after();
            const float lam = ms.lam;
            const float il1 = xch[r], il2 = xch[BM + r];
            const uint32_t t_o1 = tmem + lane_off + col_o(0) + 64 * c;
            const uint32_t t_o2 = tmem + lane_off + col_o(1) + 64 * c;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t o1[32], o2[32];
                tmem_ld32(t_o1 + ch * 32, o1);
                tmem_ld32(t_o2 + ch * 32, o2);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    D[ch * 32 + i] = diff_combine(__uint_as_float(o1[i]), il1, __uint_as_float(o2[i]), il2, lam);
                    ssp = fmaf(D[ch * 32 + i], D[ch * 32 + i], ssp);
                }
                // Training outputs: the normalised attention output of each component,
                // kept in fp32 (the lambda gradient sums many cancelling terms of them).
                if (stage_o && p.o1 != nullptr) {
                    // box 2c + ch of each: row r at r * 128 bytes, 16-byte chunk i at (i ^ (r % 8))
                    uint8_t* row1 = smem + OFF_OSTAGE + (uint32_t)(2 * c + ch) * O_BOX + (uint32_t)r * 128u;
                    uint8_t* row2 = row1 + 4 * O_BOX;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t off = (uint32_t)((i ^ (r & 7)) << 4);
                        *reinterpret_cast<float4*>(row1 + off) =
                            make_float4(__uint_as_float(o1[4 * i]) * il1, __uint_as_float(o1[4 * i + 1]) * il1,
                                        __uint_as_float(o1[4 * i + 2]) * il1, __uint_as_float(o1[4 * i + 3]) * il1);
                        *reinterpret_cast<float4*>(row2 + off) =
                            make_float4(__uint_as_float(o2[4 * i]) * il2, __uint_as_float(o2[4 * i + 1]) * il2,
                                        __uint_as_float(o2[4 * i + 2]) * il2, __uint_as_float(o2[4 * i + 3]) * il2);
                    }
                } else if (store && p.o1 != nullptr) {
                    const size_t base = ((size_t)(start + qi) * p.H + h) * DV / 4 + c * 16 + ch * 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        reinterpret_cast<float4*>(p.o1)[base + i] =
                            make_float4(__uint_as_float(o1[4 * i]) * il1, __uint_as_float(o1[4 * i + 1]) * il1,
                                        __uint_as_float(o1[4 * i + 2]) * il1, __uint_as_float(o1[4 * i + 3]) * il1);
                        reinterpret_cast<float4*>(p.o2)[base + i] =
                            make_float4(__uint_as_float(o2[4 * i]) * il2, __uint_as_float(o2[4 * i + 1]) * il2,
                                        __uint_as_float(o2[4 * i + 2]) * il2, __uint_as_float(o2[4 * i + 3]) * il2);
                    }
                }
            }
        }
        xch[2 * BM + c * BM + r] = ssp;
        named_barrier_sync(1, 256);
        // A tile wholly inside its sequence leaves through a bulk tensor store of the
        // 128 x 128 bf16 block, staged in the first K box (free: every load of this CTA
        // has been consumed); a tile past the sequence end (whose rows beyond it may
        // belong to the next packed sequence) is stored row by row.
        const bool full_tile = qt * BM + BM <= len;
        if (ok) {
            // RMSNorm over the dv values of the row, weight, (1 - lambda_init), bf16
            const float ss = xch[2 * BM + r] + xch[3 * BM + r];
            const float post = (1.f - p.lambda_init) / sqrtf(ss / (float)DV + p.eps);
            const float* wv = ms.w + 64 * c;
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                                  ((size_t)(start + (store ? qi : 0)) * p.H + h) * DV + 64 * c);
            // box c of the staging area: row r at r * 128 bytes, 16-byte chunk g at (g ^ (r % 8))
            uint8_t* stage_row = smem + OFF_STAGE0 + (uint32_t)c * BOX_BYTES + (uint32_t)r * 128u;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                uint32_t pk[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = g * 8 + 2 * i;
                    pk[i] = pack_bf16x2(D[e] * post * wv[e], D[e + 1] * post * wv[e + 1]);
                }
                const uint4 v4 = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                if (full_tile)
                    *reinterpret_cast<uint4*>(stage_row + ((g ^ (r & 7)) << 4)) = v4;
                else if (store)
                    dst[g] = v4;
            }
        }
        if (full_tile) {
            fence_proxy_async_smem();  // the staged rows, visible to the bulk copy
            named_barrier_sync(1, 256);
            if (warp == 0 && lane == 0 && ok) {
                const uint32_t src = sbase + OFF_STAGE0;
                tma_store_2d(&tm_out, src, h * DV, start + qt * BM);
                tma_store_2d(&tm_out, src + BOX_BYTES, h * DV + 64, start + qt * BM);
                if (TRAIN && p.o1 != nullptr) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        tma_store_2d(&tm_o1, sbase + OFF_OSTAGE + (uint32_t)b * O_BOX, h * DV + 32 * b, start + qt * BM);
                        tma_store_2d(&tm_o2, sbase + OFF_OSTAGE + (uint32_t)(4 + b) * O_BOX, h * DV + 32 * b,
                                     start + qt * BM);
                    }
                }
                bulk_commit_group();
                bulk_wait_group_read0();  // shared memory stays until the copy has read it
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

__global__ void __launch_bounds__(NUM_THREADS, 1)
diffattn_fwd_bf16_sm103a_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
                                const FwdParams p) {
    fwd_bf16_body<false, false>(tm_q, tm_k, tm_v, tm_out, tm_out, tm_out, p);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
diffattn_fwd_bf16_sm103a_lambda_kernel(const __grid_constant__ CUtensorMap tm_q,
                                       const __grid_constant__ CUtensorMap tm_k,
                                       const __grid_constant__ CUtensorMap tm_v,
                                       const __grid_constant__ CUtensorMap tm_out, const FwdParams p) {
    fwd_bf16_body<false, true>(tm_q, tm_k, tm_v, tm_out, tm_out, tm_out, p);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
diffattn_fwd_bf16_sm103a_train_kernel(const __grid_constant__ CUtensorMap tm_q,
                                      const __grid_constant__ CUtensorMap tm_k,
                                      const __grid_constant__ CUtensorMap tm_v,
                                      const __grid_constant__ CUtensorMap tm_out,
                                      const __grid_constant__ CUtensorMap tm_o1,
                                      const __grid_constant__ CUtensorMap tm_o2, const FwdParams p) {
    fwd_bf16_body<true, false>(tm_q, tm_k, tm_v, tm_out, tm_o1, tm_o2, p);
}

}  // namespace

cudaError_t launch_fwd_bf16_sm103a(const FwdParams& p, const FwdTensorMaps& maps, cudaStream_t stream) {
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !attr_done[dev]) {
        err = cudaFuncSetAttribute(diffattn_fwd_bf16_sm103a_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)SMEM_BYTES);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(diffattn_fwd_bf16_sm103a_train_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(diffattn_fwd_bf16_sm103a_lambda_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (err != cudaSuccess) return err;
        attr_done[dev] = true;
    }
    const int n_qt = (p.max_seqlen + BM - 1) / BM;
    if (p.group_heads < 1 || p.H % p.group_heads != 0 || (long long)n_qt * p.H > INT32_MAX) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_qt * p.H), 1u, (unsigned)p.num_seqs);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.o1 != nullptr)
        return cudaLaunchKernelEx(&cfg, diffattn_fwd_bf16_sm103a_train_kernel, maps.q, maps.k, maps.v, maps.out,
                                  maps.o1, maps.o2, p);
    if (p.lq1 != nullptr)
        return cudaLaunchKernelEx(&cfg, diffattn_fwd_bf16_sm103a_lambda_kernel, maps.q, maps.k, maps.v, maps.out, p);
    return cudaLaunchKernelEx(&cfg, diffattn_fwd_bf16_sm103a_kernel, maps.q, maps.k, maps.v, maps.out, p);
}

}  // namespace diffattn
