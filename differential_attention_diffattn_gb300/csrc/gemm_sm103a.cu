// Output projection after the differential attention on sm_103a:
//   y[M][N] = x[M][K] W[N][K]^T   (bf16 in, fp32 accumulate in tensor memory, bf16 out)
// ("LlamaDiffSdpaAttention.py", forward: o_proj = nn.Linear(H * dv, hidden,
// bias=False) on the attention output reshaped to [tokens, H * dv]).
//
// Persistent kernel, one CTA per SM walking 128 x 256 output tiles (column tile
// fastest, so CTAs running at the same time share the rows of x they read).
// Roles (192 threads):
//   warps 0-3  epilogue: tensor memory -> registers -> bf16 -> global, one
//              output row per thread (TMEM lane = row);
//   warp  4    TMA producer: per 64-wide K block a [128 x 64] box of x and a
//              [256 x 64] box of W (128-byte swizzle) into a 4-stage ring;
//   warp  5    TMEM allocator and MMA issuer (elected lane, warp-uniform loop):
//              four tcgen05.mma M128 N256 K16 per K block.
// Tensor memory: two 256-column fp32 accumulators, so the epilogue of one tile
// overlaps the MMAs of the next.
// Every wait is bounded; on a timeout the CTA records the error, lets its copies
// and MMAs in flight finish, frees TMEM and returns.
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103a_ptx.cuh"

namespace diffattn {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int NUM_THREADS = 192;
constexpr int PRODUCER_WARP = 4, MMA_WARP = 5;
constexpr uint32_t A_BYTES = BM * BK * 2;                 // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;                 // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t OFF_MISC = STAGES * STAGE_BYTES;
constexpr uint32_t SMEM_BYTES = 1024 + OFF_MISC + 256;
static_assert(SMEM_BYTES <= 232448, "exceeds the per-block shared memory limit");

struct Misc {
    uint64_t full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], done;
    uint32_t tmem;
    int abort_flag;
};
static_assert(sizeof(Misc) <= 256, "misc area too small");

__device__ __forceinline__ bool warp_all(bool p) { return __all_sync(0xffffffffu, p); }
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) { return smem_desc_sw128(saddr, 16, 1024); }

__global__ void __launch_bounds__(NUM_THREADS, 1)
diffattn_out_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                         const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc& ms = *reinterpret_cast<Misc*>(smem + OFF_MISC);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (p.M + BM - 1) / BM, n_tiles = (p.N + BN - 1) / BN, k_blocks = (p.K + BK - 1) / BK;
    const int tiles = m_tiles * n_tiles;
    auto b_full = [&](int s) { return smem_u32(&ms.full[s]); };
    auto b_empty = [&](int s) { return smem_u32(&ms.empty[s]); };
    auto b_accf = [&](int b) { return smem_u32(&ms.acc_full[b]); };
    auto b_acce = [&](int b) { return smem_u32(&ms.acc_empty[b]); };

    if (warp == PRODUCER_WARP && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(b_full(s), 1);
            mbar_init(b_empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(b_accf(b), 1);
            mbar_init(b_acce(b), 128);
        }
        mbar_init(smem_u32(&ms.done), 1);
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
            const uint64_t pol_x = l2_policy_evict_first(), pol_w = l2_policy_evict_last();
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
                const int m = t / n_tiles, n = t % n_tiles;
                for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!(ok = mbar_wait(b_empty(s), ((uint32_t)(it / STAGES) & 1u) ^ 1u, ab))) break;
                    const uint32_t st = sb + (uint32_t)s * STAGE_BYTES;
                    // boxes past M, N or K are zero-filled and still count their full bytes
                    mbar_arrive_expect_tx(b_full(s), STAGE_BYTES);
                    tma_load_2d(st, &tm_x, b_full(s), kb * BK, m * BM, pol_x);
                    tma_load_2d(st + A_BYTES, &tm_w, b_full(s), kb * BK, n * BN, pol_w);
                }
            }
            for (int j = it > STAGES ? it - STAGES : 0; j < it; ++j)
                mbar_wait_drain(b_full(j % STAGES), (uint32_t)(j / STAGES) & 1u, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false);
        constexpr uint64_t KS = 32 >> 4, SG = STAGE_BYTES >> 4, AB = A_BYTES >> 4;
        const uint64_t d0 = desc_kmajor(sb);
        int it = 0, tc = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++tc) {
            const int buf = tc & 1;
            if (!(ok = warp_all(mbar_wait(b_acce(buf), ((uint32_t)(tc >> 1) & 1u) ^ 1u, ab)))) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)buf * BN;
            for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                const int s = it % STAGES;
                if (!(ok = warp_all(mbar_wait(b_full(s), (uint32_t)(it / STAGES) & 1u, ab)))) break;
                tc_fence_after();
                const uint64_t a = d0 + (uint64_t)s * SG, b = a + AB;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_ss_elect(d, a + kk * KS, b + kk * KS, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                mma_commit_elect(b_empty(s));
            }
            if (!ok) break;
            mma_commit_elect(b_accf(buf));
        }
        // everything this warp issued (also the MMAs of a tile left by an abort)
        // has completed before TMEM is released
        mma_commit_elect(smem_u32(&ms.done));
        mbar_wait_drain(smem_u32(&ms.done), 0, p.timeout_ns);
        __syncwarp();
    } else {
        // ================================================ epilogue warps 0-3 ===
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        int tc = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tc) {
            const int buf = tc & 1;
            if (!warp_all(mbar_wait(b_accf(buf), (uint32_t)(tc >> 1) & 1u, ab))) break;
            tc_fence_after();
            const int m = t / n_tiles, n = t % n_tiles;
            const int row = m * BM + warp * 32 + lane;
            __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(p.y) + (size_t)(row < p.M ? row : 0) * p.N;
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + (uint32_t)buf * BN + ch * 32, r);
                tmem_wait_ld();
                const int col0 = n * BN + ch * 32;
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                if (row < p.M) {
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        if (col0 + 8 * g + 8 <= p.N)
                            *reinterpret_cast<uint4*>(yrow + col0 + 8 * g) =
                                make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(b_acce(buf));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_out_proj(const GemmParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                            cudaStream_t stream) {
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !attr_done[dev]) {
        err = cudaFuncSetAttribute(diffattn_out_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)SMEM_BYTES);
        if (err != cudaSuccess) return err;
        attr_done[dev] = true;
    }
    int sms = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const long long tiles = (long long)((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    const int grid = (int)(tiles < sms ? tiles : sms);
    diffattn_out_proj_kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(tm_x, tm_w, p);
    return cudaGetLastError();
}

}  // namespace diffattn
