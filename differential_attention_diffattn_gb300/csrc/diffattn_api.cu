// Host side of the C ABI declared in include/diffattn.h: argument validation,
// the per-device error word, TMA descriptor encoding and kernel dispatch.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/diffattn.h"
#include "internal.h"

namespace diffattn {
namespace {

// An NVTX range over one call of the ABI, so that a profiler's timeline shows each
// call (and the launches it makes) under the entry point's name; with no tool
// attached a push or pop is a check of one function pointer.
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

// Error bits written by kernels; one word per device (a module variable of
// this library, so nothing is allocated for it).
__device__ unsigned int g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_error_ptr[kMaxDevices] = {nullptr};
unsigned long long g_timeout_ns = kDefaultWaitTimeoutNs;
int g_inject = 0;

cudaError_t error_word_ptr(unsigned int** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_error_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        err = cudaGetSymbolAddress(&ptr, g_error_word);
        if (err != cudaSuccess) return err;
        g_error_ptr[dev] = static_cast<unsigned int*>(ptr);
    }
    *out = g_error_ptr[dev];
    return cudaSuccess;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 map over a [rows][row_elems] row-major tensor; box = 64 elements
// (128 bytes, 128-byte swizzle) x 128 rows. Rows past the end read as zero.
bool encode_bf16_rows(CUtensorMap* map, const void* base, uint64_t row_elems, uint64_t rows,
                      uint32_t box_rows = 128) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {row_elems, rows};
    const cuuint64_t strides[1] = {row_elems * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 map over a [rows][row_elems] row-major tensor; box = 32 elements (128 bytes,
// 128-byte swizzle) x 128 rows.
bool encode_f32_rows(CUtensorMap* map, const void* base, uint64_t row_elems, uint64_t rows) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {row_elems, rows};
    const cuuint64_t strides[1] = {row_elems * 4};
    const cuuint32_t box[2] = {32, 128};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 map over [rows][16] (32-byte rows): boxes of 16 x 64 rows with the
// 32-byte swizzle, as K-major MMA operands of one 16-wide K step.
bool encode_bf16_aug(CUtensorMap* map, const void* base, uint64_t rows) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {16, rows};
    const cuuint64_t strides[1] = {32};
    const cuuint32_t box[2] = {16, 64};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device (looked up once per device).
int sm_count() {
    static int counts[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    if (counts[dev] == 0) {
        int n = 0;
        counts[dev] = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0 ? n : 152;
    }
    return counts[dev];
}

// Which bf16 forward kernel runs. Items of at most 64 key tiles (sequences of
// at most 8192 tokens), at least two (query tile, head, sequence) items per SM
// and at most 64 packed sequences go to the persistent kernel: it hides the
// per-CTA setup, the epilogue and the gap between CTAs, a large share when items
// are short (measured against the one-item-per-CTA kernel: x1.13 at B = 4,
// T = 2048, 16 / 4 heads; x1.14 on 32768 tokens packed in 14 sequences of
// 128..4096; x1.01-1.03 at T = 8192). Longer sequences stay on the
// one-item-per-CTA kernel (T = 16384: a tie; T = 32768: x0.975 for the
// persistent one), and so do grids of about one item per SM.
bool fwd_use_persistent(bool packed, int max_seqlen, int heads, int num_seqs) {
    const long long n_qt = (max_seqlen + 127) / 128;
    if (n_qt > 64 || (packed && num_seqs > 64)) return false;
    return n_qt * heads * num_seqs >= 2LL * sm_count();
}

// Heads per launch group of the one-item-per-CTA bf16 forward: a whole number of
// kv-head groups whose K and V (max_seqlen rows of 2d + dv bf16 per kv head) fit in
// 32 MB, a quarter of the L2. The CTAs in flight (one per SM) then walk the K / V
// tiles of those heads only, and re-read them from L2 rather than HBM; with every
// head in one group, 16 heads of T = 16384 keep 128 MB of K / V in flight and the
// launch read 3.4x its algorithmic bytes from DRAM.
int fwd_group_heads(int H, int Hkv, int max_seqlen) {
    const int G = H / Hkv;
    const double kv_head_bytes = (double)max_seqlen * (2 * 64 + 128) * 2;
    int kv = (int)((32.0 * (1 << 20)) / (kv_head_bytes > 1.0 ? kv_head_bytes : 1.0));
    if (kv < 1) kv = 1;
    if (kv > Hkv) kv = Hkv;
    while (Hkv % kv != 0) --kv;  // a divisor of Hkv, so that groups tile the heads
    return kv * G;
}

// Launch order of a causal backward kernel, whose CTA for tile t of a sequence of n
// 128-row tiles visits t + 1 (dQ) or n - t (dK/dV) tiles. Sequence-major order keeps
// the CTAs in flight on one or two sequences, so the operands they stream are shared
// in L2; but the last sequence's longest CTA is then handed out only after the rest of
// the grid and can end well after the average SM. Estimate that end (one CTA per SM,
// each costing the tiles it visits plus half a tile of setup, the sequences taken as
// max_seqlen long) and go tiles-outermost, the longest tiles of every sequence first,
// when it is more than 10 % past the average. Measured on 16 / 4 heads, T = 2048:
// backward x1.18 at B = 4 (dK/dV grid of 256 CTAs); at B = 8, T = 4096 with 16 kv heads
// the tiles-outermost order was 6 % slower (no tail, less L2 reuse) and is not chosen.
bool bwd_tiles_outermost(int num_seqs, int heads, int max_seqlen) {
    if (num_seqs < 2) return false;
    const double n = (double)((max_seqlen + 127) / 128);
    const double per_seq = heads * (n * (n + 1) / 2 + 0.5 * n);
    const double slots = (double)sm_count();
    const double avg_end = per_seq * num_seqs / slots;
    const double last_end = per_seq * (num_seqs - 1) / slots + n + 0.5;
    return last_end > 1.1 * avg_end;
}

// Key-split count of a cache forward from the sequences' actual key counts (a
// host copy of cache_seqlens): the count whose modelled time is least, fewer
// splits on a tie. A split CTA streams its keys (512 bytes per key and kv head at
// d = 64) at t(A) = sqrt(t1^2 + (A * 512 B / BW)^2) per key while A split CTAs
// stream together: t1 = 10.4 ns is one CTA's own rate (its two-stage pipeline),
// BW = 5.8 TB/s the device's; the CTAs run in waves of the resident slots, each
// wave's longest chunk setting its time, plus 2.5 us a wave and the combine's
// reads (1040 bytes per row and split at ~3 TB/s). Fitted on GB300 to forced
// split sweeps: 16 ragged caches of 1016..7005 keys (capacity 8192, 4 kv heads,
// 4 new tokens) measured best at 6-7 splits (34.4 us; the shape-only plan took 4,
// 38.4 us), 8 full 16k caches at 8-9 (46.8 us).
template <typename RoundPlan>
long long kv_plan_from_lengths(const diffattn_kv_desc& d, RoundPlan round_plan) {
    const long long cap = d.cache_capacity;
    const int rows = d.q_len * (d.num_heads / d.num_kv_heads);
    const double slots = (double)sm_count() * (decode_rows_supported(rows) ? decode_ctas_per_sm() : 1);
    const double t1 = 10.4, per_cta = 512.0 / 5.8e3;  // ns per key; ns per key per streaming CTA
    auto rate = [&](double a) { return std::sqrt(t1 * t1 + (a * per_cta) * (a * per_cta)); };
    const double comb_per_split = (double)d.batch * d.q_len * d.num_heads * 1040.0 / 3.0e3;  // ns
    const long long max_n = std::min<long long>((cap + 255) / 256, decode_max_splits());
    long long best_n = 1;
    double best_t = -1.0;
    for (long long cand = 1; cand <= max_n; ++cand) {
        long long cc = 0;
        const long long n = round_plan(cand, &cc);
        double active = 0.0;
        for (int b = 0; b < d.batch; ++b) {
            const long long L = std::min<long long>(std::max(d.host_seqlens[b], 1), cap);
            active += (double)((L + cc - 1) / cc);
        }
        active *= d.num_kv_heads;
        const double full = std::floor(active / slots), rest = active - full * slots;
        const double waves = full + (rest > 0.0 ? 1.0 : 0.0);
        const double t = (double)cc * (full * rate(slots) + (rest > 0.0 ? rate(rest) : 0.0)) + 2500.0 * waves +
                         (double)n * comb_per_split;
        if (best_t < 0.0 || t < best_t * 0.995) {
            best_t = t;
            best_n = n;
        }
    }
    return best_n;
}

// Key-split plan of a cache forward: (number of splits, keys per split), with
// splits of at least 256 keys (64-key multiples). Without a requested count it
// takes the fewest waves of resident split CTAs on the device's SMs (1 to 4) whose
// last wave is at least 80 % full, else the fullest: every wave repeats the
// per-CTA setup and pipeline ramp, which measured costlier than a few idle
// slots (decode_b8_c16384: 9 splits in one wave 5221 GB/s, 19 in two 5009).
// Deterministic in the shape.
bool kv_plan(const diffattn_kv_desc& d, int* n_splits, int* chunk) {
    if (d.batch < 0 || d.q_len < 1 || d.cache_capacity < d.q_len || d.num_heads <= 0 || d.num_kv_heads <= 0 ||
        d.num_heads % d.num_kv_heads != 0 || d.num_splits < 0)
        return false;
    const long long cap = d.cache_capacity;
    auto round_plan = [&](long long n, long long* c_out) {
        long long c = (cap + n - 1) / n;
        c = (c + 63) / 64 * 64;
        *c_out = c;
        return (cap + c - 1) / c;
    };
    long long n = d.num_splits, c = 0;
    if (n == 0 && d.host_seqlens != nullptr && d.batch > 0) {
        n = kv_plan_from_lengths(d, round_plan);
    } else if (n == 0) {
        const long long ctas = (long long)d.batch * d.num_kv_heads;
        const int rows = d.q_len * (d.num_heads / d.num_kv_heads);
        const long long slots = (long long)sm_count() * (decode_rows_supported(rows) ? decode_ctas_per_sm() : 1);
        const long long max_n = (cap + 255) / 256;
        double best = -1.0;
        n = 1;
        for (long long waves = 1; waves <= 4 && ctas > 0; ++waves) {
            long long cand = waves * slots / ctas;
            if (cand < 1) cand = 1;
            if (cand > max_n) cand = max_n;
            long long cc;
            cand = round_plan(cand, &cc);
            const long long total = cand * ctas;
            const double fill = (double)total / (double)(((total + slots - 1) / slots) * slots);
            if (fill > best + 1e-9) {
                best = fill;
                n = cand;
            }
            if (fill >= 0.8) break;
        }
    }
    n = round_plan(n, &c);
    if (n > decode_max_splits()) return false;
    *n_splits = (int)n;
    *chunk = (int)c;
    return true;
}

unsigned long long kv_workspace_bytes(const diffattn_kv_desc& d, int n_splits) {
    const unsigned long long rows = (unsigned long long)d.batch * d.q_len * d.num_heads * n_splits * 2;
    const unsigned long long o = rows * (unsigned long long)d.dv * 4;
    return o + rows * 2 * 4;
}

// The cache forward's checks of the descriptor alone (no pointers): the split
// plan, sizes and limits (INVALID_ARG), then what the kernels support
// (UNSUPPORTED). On success the split count and chunk are set.
diffattn_status kv_check_desc(const diffattn_kv_desc& ds, float lambda_init, int* n_splits, int* chunk) {
    if (!kv_plan(ds, n_splits, chunk)) return DIFFATTN_ERR_INVALID_ARG;
    if (ds.d <= 0 || ds.dv != 2 * ds.d) return DIFFATTN_ERR_INVALID_ARG;
    if (!(ds.eps >= 0.f) || !std::isfinite(ds.eps) || !std::isfinite(lambda_init)) return DIFFATTN_ERR_INVALID_ARG;
    if (ds.dtype != DIFFATTN_DTYPE_F32 && ds.dtype != DIFFATTN_DTYPE_BF16) return DIFFATTN_ERR_INVALID_ARG;
    if ((long long)ds.batch * ds.cache_capacity * ds.num_kv_heads * ds.dv >= (1LL << 40) ||
        (long long)ds.batch * ds.cache_capacity > INT32_MAX - 64 ||
        (long long)ds.batch * ds.q_len * ds.num_heads > INT32_MAX || ds.batch > 65535 || ds.num_kv_heads > 65535)
        return DIFFATTN_ERR_INVALID_ARG;
    const int rows = ds.q_len * (ds.num_heads / ds.num_kv_heads);
    if (ds.dtype != DIFFATTN_DTYPE_BF16 || ds.d != 64 || !decode_rows_supported(rows))
        return DIFFATTN_ERR_UNSUPPORTED;
    return DIFFATTN_OK;
}

}  // namespace
}  // namespace diffattn

using namespace diffattn;

extern "C" {

float diffattn_lambda_init(int depth) {
    if (depth < 1) return NAN;
    return (float)(0.8 - 0.6 * std::exp(-0.3 * (double)(depth - 1)));
}

diffattn_status diffattn_lambda(const float* lq1, const float* lk1, const float* lq2, const float* lk2, int n_sets,
                                int d, float lambda_init, float* lambda_out, void* stream) {
    const CallRange nvtx_range("diffattn_lambda");
    if (!lq1 || !lk1 || !lq2 || !lk2 || !lambda_out) return DIFFATTN_ERR_INVALID_ARG;
    if (n_sets < 1 || d < 1 || d > 1024) return DIFFATTN_ERR_INVALID_ARG;
    if (launch_lambda(lq1, lk1, lq2, lk2, n_sets, d, lambda_init, lambda_out,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;
    return DIFFATTN_OK;
}

}  // extern "C"

namespace {
// Shared body of diffattn_fwd and diffattn_fwd_train; lse, o1, o2 are all null
// (inference) or all set (training outputs, bf16 tcgen05 kernel only).
// The lambda kernel a combined call launches just before its forward, writing
// the `lambda` the forward reads.
struct LambdaCall {
    const float *lq1, *lk1, *lq2, *lk2;
    int n_sets, d;
};

diffattn_status fwd_common(const diffattn_desc* desc, const void* q, const void* k, const void* v,
                           const float* lambda, int lambda_per_head, float lambda_init, const float* subln_w,
                           int causal, const int* cu_seqlens, void* out, float* lse, void* o1, void* o2,
                           void* stream, const diffattn_rope_q* rope = nullptr,
                           const LambdaCall* lam_call = nullptr) {
    if (!desc) return DIFFATTN_ERR_INVALID_ARG;
    const bool train = lse != nullptr || o1 != nullptr || o2 != nullptr;
    if (train && (!lse || !o1 || !o2 || !aligned16(o1) || !aligned16(o2) ||
                  (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return DIFFATTN_ERR_INVALID_ARG;
    const diffattn_desc& ds = *desc;
    if (ds.num_heads <= 0 || ds.num_kv_heads <= 0 || ds.num_heads % ds.num_kv_heads != 0 || ds.num_heads > 65535)
        return DIFFATTN_ERR_INVALID_ARG;
    if (ds.d <= 0 || ds.dv != 2 * ds.d) return DIFFATTN_ERR_INVALID_ARG;
    if (!(ds.eps >= 0.f) || !std::isfinite(ds.eps) || !std::isfinite(lambda_init)) return DIFFATTN_ERR_INVALID_ARG;
    if (ds.dtype != DIFFATTN_DTYPE_F32 && ds.dtype != DIFFATTN_DTYPE_BF16) return DIFFATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return DIFFATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(lambda) & 3u) || (reinterpret_cast<uintptr_t>(subln_w) & 3u))
        return DIFFATTN_ERR_INVALID_ARG;

    FwdParams p{};
    if (cu_seqlens == nullptr) {
        if (ds.batch < 0 || ds.seqlen < 0) return DIFFATTN_ERR_INVALID_ARG;
        const long long tokens = (long long)ds.batch * ds.seqlen;
        if (tokens > INT32_MAX) return DIFFATTN_ERR_INVALID_ARG;
        p.num_seqs = ds.batch;
        p.seqlen = ds.seqlen;
        p.max_seqlen = ds.seqlen;
        p.total_tokens = (int)tokens;
    } else {
        if (ds.num_seqs < 0 || ds.max_seqlen < 0 || ds.total_tokens < 0) return DIFFATTN_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return DIFFATTN_ERR_INVALID_ARG;
        p.num_seqs = ds.num_seqs;
        p.seqlen = 0;
        p.max_seqlen = ds.max_seqlen;
        p.total_tokens = ds.total_tokens;
    }
    if (p.num_seqs > 65535) return DIFFATTN_ERR_INVALID_ARG;
    // rows of q / out as 32-bit TMA coordinates and element offsets
    if ((long long)p.total_tokens * ds.num_heads * ds.dv >= (1LL << 40)) return DIFFATTN_ERR_INVALID_ARG;

    const bool bf16_tc = ds.dtype == DIFFATTN_DTYPE_BF16 && ds.d == 64;
    const bool f32_simt = ds.dtype == DIFFATTN_DTYPE_F32 && (ds.d == 16 || ds.d == 32 || ds.d == 64);
    if (rope != nullptr) {  // the rotary embedding of q inside the kernels
        if ((rope->rot_dim != ds.d && rope->rot_dim != 2 * ds.d) || (rope->rot_dim % 8) != 0 || rope->n_pos < 1 ||
            (rope->interleaved != 0 && rope->interleaved != 1) || !rope->cos || !rope->sin ||
            !aligned16(rope->cos) || !aligned16(rope->sin))
            return DIFFATTN_ERR_INVALID_ARG;
        if (!bf16_tc) return DIFFATTN_ERR_UNSUPPORTED;
    }
    if (!bf16_tc && !f32_simt) return DIFFATTN_ERR_UNSUPPORTED;
    if (train && !bf16_tc) return DIFFATTN_ERR_UNSUPPORTED;

    // An empty problem launches nothing; its tensor pointers may be NULL.
    if (p.total_tokens == 0 || p.num_seqs == 0 || p.max_seqlen == 0) return DIFFATTN_OK;
    if (!q || !k || !v || !lambda || !subln_w || !out) return DIFFATTN_ERR_INVALID_ARG;

    unsigned int* err_word = nullptr;
    if (error_word_ptr(&err_word) != cudaSuccess) return DIFFATTN_ERR_CUDA;

    p.q = q;
    p.k = k;
    p.v = v;
    p.out = out;
    p.lambda = lambda;
    p.subln_w = subln_w;
    p.cu_seqlens = cu_seqlens;
    p.error_word = err_word;
    p.H = ds.num_heads;
    p.Hkv = ds.num_kv_heads;
    p.d = ds.d;
    p.dv = ds.dv;
    p.lambda_stride = lambda_per_head ? 1 : 0;
    p.causal = causal ? 1 : 0;
    p.lambda_init = lambda_init;
    p.eps = ds.eps;
    p.scale = (float)(1.0 / std::sqrt((double)ds.d));
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)ds.d));
    p.timeout_ns = g_timeout_ns;
    p.inject = g_inject;
    p.lse = lse;
    p.o1 = o1;
    p.o2 = o2;
    p.group_heads = fwd_group_heads(p.H, p.Hkv, p.max_seqlen);
    if (rope != nullptr) {
        p.rope_cos = rope->cos;
        p.rope_sin = rope->sin;
        p.rope_npos = rope->n_pos;
        p.rope_dim = rope->rot_dim;
        p.rope_interleaved = rope->interleaved;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the combined call's lambda kernel goes first, once nothing can fail on the host
    auto launch_lambda_first = [&]() {
        return launch_lambda(lam_call->lq1, lam_call->lk1, lam_call->lq2, lam_call->lk2, lam_call->n_sets,
                             lam_call->d, lambda_init, const_cast<float*>(lambda), st);
    };

    if (f32_simt) {
        if (lam_call && launch_lambda_first() != cudaSuccess) return DIFFATTN_ERR_CUDA;
        return launch_fwd_f32(p, st) == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
    }

    FwdTensorMaps maps;
    if (!encode_bf16_rows(&maps.q, q, (uint64_t)ds.num_heads * 2 * ds.d, (uint64_t)p.total_tokens) ||
        !encode_bf16_rows(&maps.k, k, (uint64_t)ds.num_kv_heads * 2 * ds.d, (uint64_t)p.total_tokens) ||
        !encode_bf16_rows(&maps.v, v, (uint64_t)ds.num_kv_heads * ds.dv, (uint64_t)p.total_tokens) ||
        !encode_bf16_rows(&maps.out, out, (uint64_t)ds.num_heads * ds.dv, (uint64_t)p.total_tokens))
        return DIFFATTN_ERR_CUDA;
    if (train) {
        if (!encode_f32_rows(&maps.o1, o1, (uint64_t)ds.num_heads * ds.dv, (uint64_t)p.total_tokens) ||
            !encode_f32_rows(&maps.o2, o2, (uint64_t)ds.num_heads * ds.dv, (uint64_t)p.total_tokens))
            return DIFFATTN_ERR_CUDA;
    } else {
        maps.o1 = maps.out;  // not read without training outputs
        maps.o2 = maps.out;
    }
    // The rotary embedding of q is applied by the one-item-per-CTA kernel only: it
    // stages each tile's cos / sin rows in its last K/V stage, which the persistent
    // kernel does not have (its shared memory is all in use).
    const bool persistent = rope == nullptr && fwd_use_persistent(cu_seqlens != nullptr, p.max_seqlen, p.H, p.num_seqs);
    // A combined call whose one-item-per-CTA grid fits one wave forms lambda in that
    // kernel (one launch: the step is a latency chain, 2 x 512 tokens 19.0 -> 16.9 us a
    // flushed step); longer grids launch the lambda kernel first, which runs under the
    // forward's start (in-kernel there measured 0.3 % slower at 16384 tokens).
    const long long grid_ctas = (long long)((p.max_seqlen + 127) / 128) * p.H * p.num_seqs;
    if (lam_call && (persistent || grid_ctas > sm_count())) {
        if (launch_lambda_first() != cudaSuccess) return DIFFATTN_ERR_CUDA;
        p.lambda_pending = 1;  // the forward's reads of lambda alone wait for that kernel
    } else if (lam_call) {
        p.lq1 = lam_call->lq1;
        p.lk1 = lam_call->lk1;
        p.lq2 = lam_call->lq2;
        p.lk2 = lam_call->lk2;
        p.lambda_d = lam_call->d;
        p.lambda_out = const_cast<float*>(lambda);
    }
    const cudaError_t err = persistent ? launch_fwd_bf16_persistent(p, maps, st) : launch_fwd_bf16_sm103a(p, maps, st);
    return err == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}
}  // namespace

extern "C" {

const char* diffattn_fwd_kernel(const diffattn_desc* desc, int packed) {
    if (!desc || desc->num_heads <= 0) return nullptr;
    const diffattn_desc& ds = *desc;
    if (ds.dtype == DIFFATTN_DTYPE_F32 && (ds.d == 16 || ds.d == 32 || ds.d == 64)) return "diffattn_fwd_f32_kernel";
    if (ds.dtype != DIFFATTN_DTYPE_BF16 || ds.d != 64) return nullptr;
    const int max_seqlen = packed ? ds.max_seqlen : ds.seqlen;
    const int num_seqs = packed ? ds.num_seqs : ds.batch;
    return fwd_use_persistent(packed != 0, max_seqlen, ds.num_heads, num_seqs) ? "diffattn_fwd_bf16_persistent_kernel"
                                                                               : "diffattn_fwd_bf16_sm103a_kernel";
}

diffattn_status diffattn_fwd(const diffattn_desc* desc, const void* q, const void* k, const void* v,
                             const float* lambda, int lambda_per_head, float lambda_init, const float* subln_w,
                             int causal, const int* cu_seqlens, void* out, void* stream) {
    const CallRange nvtx_range("diffattn_fwd");
    return fwd_common(desc, q, k, v, lambda, lambda_per_head, lambda_init, subln_w, causal, cu_seqlens, out,
                      nullptr, nullptr, nullptr, stream);
}

diffattn_status diffattn_fwd_lambda(const diffattn_desc* desc, const void* q, const void* k, const void* v,
                                    const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                                    int lambda_per_head, int lambda_d, float lambda_init, float* lambda_out,
                                    const float* subln_w, int causal, const int* cu_seqlens, void* out,
                                    void* stream) {
    const CallRange nvtx_range("diffattn_fwd_lambda");
    if (!desc || !lq1 || !lk1 || !lq2 || !lk2 || !lambda_out) return DIFFATTN_ERR_INVALID_ARG;
    if (lambda_d < 1 || lambda_d > 1024 || (reinterpret_cast<uintptr_t>(lambda_out) & 3u)) return DIFFATTN_ERR_INVALID_ARG;
    const LambdaCall lc{lq1, lk1, lq2, lk2, lambda_per_head ? desc->num_heads : 1, lambda_d};
    if (lc.n_sets < 1) return DIFFATTN_ERR_INVALID_ARG;
    return fwd_common(desc, q, k, v, lambda_out, lambda_per_head, lambda_init, subln_w, causal, cu_seqlens, out,
                      nullptr, nullptr, nullptr, stream, nullptr, &lc);
}

diffattn_status diffattn_fwd_rope_q(const diffattn_desc* desc, const void* q, const void* k, const void* v,
                                    const float* lambda, int lambda_per_head, float lambda_init,
                                    const float* subln_w, int causal, const int* cu_seqlens,
                                    const diffattn_rope_q* rope, void* out, void* stream) {
    const CallRange nvtx_range("diffattn_fwd_rope_q");
    if (!rope) return DIFFATTN_ERR_INVALID_ARG;
    return fwd_common(desc, q, k, v, lambda, lambda_per_head, lambda_init, subln_w, causal, cu_seqlens, out,
                      nullptr, nullptr, nullptr, stream, rope);
}

diffattn_status diffattn_fwd_train(const diffattn_desc* desc, const void* q, const void* k, const void* v,
                                   const float* lambda, int lambda_per_head, float lambda_init,
                                   const float* subln_w, int causal, const int* cu_seqlens, void* out, float* lse,
                                   void* o1, void* o2, void* stream) {
    const CallRange nvtx_range("diffattn_fwd_train");
    if (!lse || !o1 || !o2) return DIFFATTN_ERR_INVALID_ARG;
    return fwd_common(desc, q, k, v, lambda, lambda_per_head, lambda_init, subln_w, causal, cu_seqlens, out, lse,
                      o1, o2, stream);
}

unsigned long long diffattn_fwd_kvcache_workspace_size(const diffattn_kv_desc* desc) {
    int n = 0, c = 0;
    if (!desc || !kv_plan(*desc, &n, &c)) return 0;
    return kv_workspace_bytes(*desc, n);
}

}  // extern "C"

namespace {
// Shared body of diffattn_fwd_kvcache and diffattn_fwd_kvcache_lambda (which
// passes the lambda parameter vectors: the combine kernel forms lambda from them
// and writes it to `lambda`).
diffattn_status kv_common(const diffattn_kv_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                          const int* cache_seqlens, const float* lambda, int lambda_per_head, float lambda_init,
                          const float* subln_w, int causal, void* workspace, unsigned long long workspace_bytes,
                          void* out, void* stream, const LambdaCall* lam_call) {
    if (!desc) return DIFFATTN_ERR_INVALID_ARG;
    const diffattn_kv_desc& ds = *desc;
    int n_splits = 0, chunk = 0;
    const diffattn_status desc_st = kv_check_desc(ds, lambda_init, &n_splits, &chunk);
    if (desc_st != DIFFATTN_OK) return desc_st;
    if (ds.batch == 0) return DIFFATTN_OK;
    if (!q || !k_cache || !v_cache || !lambda || !subln_w || !out || !workspace) return DIFFATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace))
        return DIFFATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(lambda) & 3u) || (reinterpret_cast<uintptr_t>(subln_w) & 3u) ||
        (reinterpret_cast<uintptr_t>(cache_seqlens) & 3u))
        return DIFFATTN_ERR_INVALID_ARG;
    if (workspace_bytes < kv_workspace_bytes(ds, n_splits)) return DIFFATTN_ERR_INVALID_ARG;

    unsigned int* err_word = nullptr;
    if (error_word_ptr(&err_word) != cudaSuccess) return DIFFATTN_ERR_CUDA;
    KvParams p{};
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.out = out;
    p.lambda = lambda;
    p.subln_w = subln_w;
    p.cache_seqlens = cache_seqlens;
    p.error_word = err_word;
    const unsigned long long rows_total = (unsigned long long)ds.batch * ds.q_len * ds.num_heads * n_splits * 2;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = p.ws_o + rows_total * ds.dv;
    p.batch = ds.batch;
    p.q_len = ds.q_len;
    p.capacity = ds.cache_capacity;
    p.H = ds.num_heads;
    p.Hkv = ds.num_kv_heads;
    p.lambda_stride = lambda_per_head ? 1 : 0;
    p.causal = causal ? 1 : 0;
    p.num_splits = n_splits;
    p.chunk = chunk;
    p.lambda_init = lambda_init;
    p.eps = ds.eps;
    p.scale = (float)(1.0 / std::sqrt((double)ds.d));
    p.timeout_ns = g_timeout_ns;
    KvTensorMaps maps;
    const uint64_t cache_rows = (uint64_t)ds.batch * ds.cache_capacity;
    if (!encode_bf16_rows(&maps.k, k_cache, (uint64_t)ds.num_kv_heads * 2 * ds.d, cache_rows, 64) ||
        !encode_bf16_rows(&maps.v, v_cache, (uint64_t)ds.num_kv_heads * ds.dv, cache_rows, 64))
        return DIFFATTN_ERR_CUDA;
    if (lam_call) {  // the combine kernel forms lambda itself
        p.lq1 = lam_call->lq1;
        p.lk1 = lam_call->lk1;
        p.lq2 = lam_call->lq2;
        p.lk2 = lam_call->lk2;
        p.lambda_d = lam_call->d;
        p.lambda_out = const_cast<float*>(lambda);
    }
    return launch_decode(p, maps, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}
}  // namespace

extern "C" {

diffattn_status diffattn_fwd_kvcache(const diffattn_kv_desc* desc, const void* q, const void* k_cache,
                                     const void* v_cache, const int* cache_seqlens, const float* lambda,
                                     int lambda_per_head, float lambda_init, const float* subln_w, int causal,
                                     void* workspace, unsigned long long workspace_bytes, void* out,
                                     void* stream) {
    const CallRange nvtx_range("diffattn_fwd_kvcache");
    return kv_common(desc, q, k_cache, v_cache, cache_seqlens, lambda, lambda_per_head, lambda_init, subln_w, causal,
                     workspace, workspace_bytes, out, stream, nullptr);
}

diffattn_status diffattn_fwd_kvcache_lambda(const diffattn_kv_desc* desc, const void* q, const void* k_cache,
                                            const void* v_cache, const int* cache_seqlens, const float* lq1,
                                            const float* lk1, const float* lq2, const float* lk2,
                                            int lambda_per_head, int lambda_d, float lambda_init, float* lambda_out,
                                            const float* subln_w, int causal, void* workspace,
                                            unsigned long long workspace_bytes, void* out, void* stream) {
    const CallRange nvtx_range("diffattn_fwd_kvcache_lambda");
    if (!desc || !lq1 || !lk1 || !lq2 || !lk2 || !lambda_out) return DIFFATTN_ERR_INVALID_ARG;
    if (lambda_d < 1 || lambda_d > 1024 || (reinterpret_cast<uintptr_t>(lambda_out) & 3u)) return DIFFATTN_ERR_INVALID_ARG;
    const LambdaCall lc{lq1, lk1, lq2, lk2, lambda_per_head ? desc->num_heads : 1, lambda_d};
    if (lc.n_sets < 1) return DIFFATTN_ERR_INVALID_ARG;
    return kv_common(desc, q, k_cache, v_cache, cache_seqlens, lambda_out, lambda_per_head, lambda_init, subln_w,
                     causal, workspace, workspace_bytes, out, stream, &lc);
}

}  // extern "C"

// ---- allocation-free cache forward -------------------------------------------
// The key-split partials of diffattn_fwd_kvcache_noalloc live in this array
// (one per device, for the life of the process). Host code must not use the
// array's name as an address: on the host it is only a stand-in, so the device
// address is looked up once per device and cached.
namespace diffattn {
namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[DIFFATTN_NOALLOC_SCRATCH_BYTES];
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_scratch on the current device (looked up on the
// first call per device, with that device current).
cudaError_t noalloc_scratch_ptr(void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}
}  // namespace
}  // namespace diffattn

extern "C" {

diffattn_status diffattn_fwd_kvcache_noalloc(const diffattn_kv_desc* desc, const void* q, const void* k_cache,
                                             const void* v_cache, const int* cache_seqlens, const float* lambda,
                                             int lambda_per_head, float lambda_init, const float* subln_w,
                                             int causal, void* out, void* stream) {
    const CallRange nvtx_range("diffattn_fwd_kvcache_noalloc");
    if (!desc) return DIFFATTN_ERR_INVALID_ARG;
    // The descriptor is checked first, so that a bad one gives the same status as
    // diffattn_fwd_kvcache rather than a size rejection.
    diffattn_kv_desc ds = *desc;
    int n_splits = 0, chunk = 0;
    const diffattn_status desc_st = kv_check_desc(ds, lambda_init, &n_splits, &chunk);
    if (desc_st != DIFFATTN_OK) return desc_st;
    // With the automatic plan, fewer key splits are taken when the planned ones'
    // partials would not fit the array; a forced split count is kept as given.
    if (ds.num_splits == 0) {
        for (int n = n_splits; n >= 1 && kv_workspace_bytes(ds, n_splits) > DIFFATTN_NOALLOC_SCRATCH_BYTES; --n) {
            ds.num_splits = n;
            if (kv_check_desc(ds, lambda_init, &n_splits, &chunk) != DIFFATTN_OK) return DIFFATTN_ERR_INVALID_ARG;
        }
    }
    if (kv_workspace_bytes(ds, n_splits) > DIFFATTN_NOALLOC_SCRATCH_BYTES) return DIFFATTN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (ds.batch > 0) {
        if (noalloc_scratch_ptr(&scratch) != cudaSuccess) return DIFFATTN_ERR_CUDA;
    }
    return diffattn_fwd_kvcache(&ds, q, k_cache, v_cache, cache_seqlens, lambda, lambda_per_head, lambda_init,
                                subln_w, causal, scratch, DIFFATTN_NOALLOC_SCRATCH_BYTES, out, stream);
}

// Backward workspace: dD (bf16 [tokens][H][dv]), the row statistics (16 bytes a row)
// and the dK/dV kernel's row operand (16 bf16 a row).
unsigned long long diffattn_bwd_workspace_size(const diffattn_desc* desc) {
    if (!desc || desc->num_heads <= 0 || desc->dv <= 0) return 0;
    long long tokens = desc->batch > 0 && desc->seqlen > 0 ? (long long)desc->batch * desc->seqlen : 0;
    if (desc->total_tokens > 0) tokens = desc->total_tokens > tokens ? desc->total_tokens : tokens;
    return (unsigned long long)tokens * desc->num_heads * ((unsigned long long)desc->dv * 2 + 16 + 32);
}

diffattn_status diffattn_bwd(const diffattn_desc* desc, const void* q, const void* k, const void* v,
                             const float* lambda, int lambda_per_head, float lambda_init, const float* subln_w,
                             int causal, const int* cu_seqlens, const void* dout, const float* lse, const void* o1,
                             const void* o2, void* dq, void* dk, void* dv, float* dlambda, float* dsubln_w,
                             void* workspace, unsigned long long workspace_bytes, void* stream) {
    const CallRange nvtx_range("diffattn_bwd");
    if (!desc) return DIFFATTN_ERR_INVALID_ARG;
    const diffattn_desc& ds = *desc;
    if (ds.num_heads <= 0 || ds.num_kv_heads <= 0 || ds.num_heads % ds.num_kv_heads != 0 || ds.num_heads > 65535)
        return DIFFATTN_ERR_INVALID_ARG;
    if (ds.d <= 0 || ds.dv != 2 * ds.d) return DIFFATTN_ERR_INVALID_ARG;
    if (!(ds.eps >= 0.f) || !std::isfinite(ds.eps) || !std::isfinite(lambda_init)) return DIFFATTN_ERR_INVALID_ARG;
    if (ds.dtype != DIFFATTN_DTYPE_BF16 || ds.d != 64) return DIFFATTN_ERR_UNSUPPORTED;
    int num_seqs, seqlen, max_seqlen, tokens;
    if (cu_seqlens == nullptr) {
        if (ds.batch < 0 || ds.seqlen < 0 || (long long)ds.batch * ds.seqlen > INT32_MAX) return DIFFATTN_ERR_INVALID_ARG;
        num_seqs = ds.batch;
        seqlen = ds.seqlen;
        max_seqlen = ds.seqlen;
        tokens = ds.batch * ds.seqlen;
    } else {
        if (ds.num_seqs < 0 || ds.max_seqlen < 0 || ds.total_tokens < 0) return DIFFATTN_ERR_INVALID_ARG;
        num_seqs = ds.num_seqs;
        seqlen = 0;
        max_seqlen = ds.max_seqlen;
        tokens = ds.total_tokens;
    }
    // (the rows of the dK/dV kernel's row operand, H x tokens, are 32-bit TMA coordinates)
    if (num_seqs > 65535 || (long long)tokens * ds.num_heads * ds.dv >= (1LL << 40) ||
        (long long)tokens * ds.num_heads > INT32_MAX - 64)
        return DIFFATTN_ERR_INVALID_ARG;
    if (tokens == 0 || num_seqs == 0 || max_seqlen == 0) return DIFFATTN_OK;
    const void* b16[] = {q, k, v, dout, o1, o2, dq, dk, dv, workspace};
    for (const void* ptr : b16)
        if (!ptr || !aligned16(ptr)) return DIFFATTN_ERR_INVALID_ARG;
    const void* f32[] = {lambda, subln_w, lse, dlambda, dsubln_w};
    for (const void* ptr : f32)
        if (!ptr || (reinterpret_cast<uintptr_t>(ptr) & 3u)) return DIFFATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return DIFFATTN_ERR_INVALID_ARG;
    const unsigned long long dd_bytes = (unsigned long long)tokens * ds.num_heads * ds.dv * 2;
    if (workspace_bytes < dd_bytes + (unsigned long long)tokens * ds.num_heads * (16 + 32)) return DIFFATTN_ERR_INVALID_ARG;

    unsigned int* err_word = nullptr;
    if (error_word_ptr(&err_word) != cudaSuccess) return DIFFATTN_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int n_lambda = lambda_per_head ? ds.num_heads : 1;
    if (cudaMemsetAsync(dlambda, 0, sizeof(float) * n_lambda, st) != cudaSuccess ||
        cudaMemsetAsync(dsubln_w, 0, sizeof(float) * ds.dv, st) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;

    void* dd = workspace;
    float* rowstat = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + dd_bytes);
    void* stat_aug = static_cast<uint8_t*>(workspace) + dd_bytes + (unsigned long long)tokens * ds.num_heads * 16;
    BwdPreParams pre{};
    pre.dout = dout;
    pre.o1 = o1;
    pre.o2 = o2;
    pre.lse = lse;
    pre.lambda = lambda;
    pre.lambda_stride = lambda_per_head ? 1 : 0;
    pre.lambda_init = lambda_init;
    pre.subln_w = subln_w;
    pre.eps = ds.eps;
    pre.tokens = tokens;
    pre.H = ds.num_heads;
    pre.dd = dd;
    pre.rowstat = rowstat;
    pre.stat_aug = stat_aug;
    pre.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)ds.d));
    pre.dlambda = dlambda;
    pre.dsubln_w = dsubln_w;
    pre.error_word = err_word;
    pre.timeout_ns = g_timeout_ns;
    if (launch_bwd_pre(pre, st) != cudaSuccess) return DIFFATTN_ERR_CUDA;

    BwdParams p{};
    p.lambda = lambda;
    p.lambda_stride = pre.lambda_stride;
    p.causal = causal ? 1 : 0;
    p.cu_seqlens = cu_seqlens;
    p.num_seqs = num_seqs;
    p.seqlen = seqlen;
    p.max_seqlen = max_seqlen;
    p.total_tokens = tokens;
    p.H = ds.num_heads;
    p.Hkv = ds.num_kv_heads;
    p.scale = (float)(1.0 / std::sqrt((double)ds.d));
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)ds.d));
    p.rowstat = rowstat;
    p.stat_aug = stat_aug;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.error_word = err_word;
    p.timeout_ns = g_timeout_ns;
    p.dq_tiles_outer = causal && bwd_tiles_outermost(num_seqs, p.H, max_seqlen) ? 1 : 0;
    p.dkv_tiles_outer = causal && bwd_tiles_outermost(num_seqs, p.Hkv, max_seqlen) ? 1 : 0;
    // launch groups whose streamed operands fit in 32 MB of L2: for the dQ kernel the
    // K / V of its heads (as the forward), for the dK/dV kernel the Q and dD of every
    // head of its kv heads (2d + dv bf16 and the 32-byte row operand per token)
    p.dq_group_heads = fwd_group_heads(p.H, p.Hkv, max_seqlen);
    {
        const int G = p.H / p.Hkv;
        const double kv_group_bytes = (double)max_seqlen * G * ((2 * 64 + 128) * 2 + 32);
        int kg = (int)((32.0 * (1 << 20)) / (kv_group_bytes > 1.0 ? kv_group_bytes : 1.0));
        kg = kg < 1 ? 1 : (kg > p.Hkv ? p.Hkv : kg);
        while (p.Hkv % kg != 0) --kg;
        p.dkv_group_kv = kg;
    }
    BwdTensorMaps m;
    const uint64_t qw = (uint64_t)ds.num_heads * 2 * ds.d, kw = (uint64_t)ds.num_kv_heads * 2 * ds.d;
    const uint64_t vw = (uint64_t)ds.num_kv_heads * ds.dv, dw = (uint64_t)ds.num_heads * ds.dv;
    if (!encode_bf16_rows(&m.q128, q, qw, tokens, 128) || !encode_bf16_rows(&m.q64, q, qw, tokens, 64) ||
        !encode_bf16_rows(&m.k128, k, kw, tokens, 128) || !encode_bf16_rows(&m.v128, v, vw, tokens, 128) ||
        !encode_bf16_rows(&m.dd128, dd, dw, tokens, 128) || !encode_bf16_rows(&m.dd64, dd, dw, tokens, 64) ||
        !encode_bf16_aug(&m.aug64, stat_aug, (uint64_t)tokens * ds.num_heads))
        return DIFFATTN_ERR_CUDA;
    return launch_bwd_sm103a(p, m, st) == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

diffattn_status diffattn_lambda_bwd(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                                    const float* dlambda, int n_sets, int d, float* dlq1, float* dlk1,
                                    float* dlq2, float* dlk2, void* stream) {
    const CallRange nvtx_range("diffattn_lambda_bwd");
    if (!lq1 || !lk1 || !lq2 || !lk2 || !dlambda || !dlq1 || !dlk1 || !dlq2 || !dlk2) return DIFFATTN_ERR_INVALID_ARG;
    if (n_sets < 1 || d < 1 || d > 1024) return DIFFATTN_ERR_INVALID_ARG;
    return launch_lambda_bwd(lq1, lk1, lq2, lk2, dlambda, n_sets, d, dlq1, dlk1, dlq2, dlk2,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DIFFATTN_OK
               : DIFFATTN_ERR_CUDA;
}

// --------------------------------------------------------------- rotary ---

diffattn_status diffattn_rope_tables(double theta, int n_pos, int rot_dim, float* cos_out, float* sin_out,
                                     void* stream) {
    const CallRange nvtx_range("diffattn_rope_tables");
    if (!cos_out || !sin_out || n_pos < 1 || rot_dim < 2 || (rot_dim & 1) || !(theta > 0.0) || !std::isfinite(theta))
        return DIFFATTN_ERR_INVALID_ARG;
    return launch_rope_tables(theta, n_pos, rot_dim, cos_out, sin_out, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? DIFFATTN_OK
               : DIFFATTN_ERR_CUDA;
}

diffattn_status diffattn_rope_qk(const diffattn_rope_desc* desc, const int* positions, const int* cu_seqlens,
                                 const float* cos_table, const float* sin_table, const void* q_in, void* q_out,
                                 const void* k_in, void* k_out, void* stream) {
    const CallRange nvtx_range("diffattn_rope_qk");
    if (!desc) return DIFFATTN_ERR_INVALID_ARG;
    const diffattn_rope_desc& ds = *desc;
    if (ds.tokens < 0 || ds.num_heads < 0 || ds.num_kv_heads < 0 || ds.num_heads + ds.num_kv_heads < 1 || ds.d < 4 ||
        (ds.d % 4) != 0 || ds.n_pos < 1)
        return DIFFATTN_ERR_INVALID_ARG;
    if (ds.dtype != DIFFATTN_DTYPE_F32 && ds.dtype != DIFFATTN_DTYPE_BF16) return DIFFATTN_ERR_INVALID_ARG;
    if ((ds.rot_dim != ds.d && ds.rot_dim != 2 * ds.d) || (ds.rot_dim % 8) != 0) return DIFFATTN_ERR_INVALID_ARG;
    if (ds.tokens == 0) return DIFFATTN_OK;
    if (!cos_table || !sin_table || !aligned16(cos_table) || !aligned16(sin_table)) return DIFFATTN_ERR_INVALID_ARG;
    if (ds.num_heads > 0 && (!q_in || !q_out || !aligned16(q_in) || !aligned16(q_out)))
        return DIFFATTN_ERR_INVALID_ARG;
    if (ds.num_kv_heads > 0 && (!k_in || !k_out || !aligned16(k_in) || !aligned16(k_out)))
        return DIFFATTN_ERR_INVALID_ARG;
    if (!positions) {
        if (cu_seqlens) {
            if (ds.num_seqs < 1 || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return DIFFATTN_ERR_INVALID_ARG;
        } else if (ds.seqlen < 1) {
            return DIFFATTN_ERR_INVALID_ARG;
        }
    } else if ((reinterpret_cast<uintptr_t>(positions) & 3u) != 0) {
        return DIFFATTN_ERR_INVALID_ARG;
    }
    if (ds.tokens * (long long)(ds.num_heads + ds.num_kv_heads) * (2 * ds.d) >= (1LL << 40))
        return DIFFATTN_ERR_INVALID_ARG;
    unsigned int* err_word = nullptr;
    if (error_word_ptr(&err_word) != cudaSuccess) return DIFFATTN_ERR_CUDA;
    RopeParams p{};
    p.q_in = ds.num_heads > 0 ? q_in : nullptr;
    p.q_out = ds.num_heads > 0 ? q_out : nullptr;
    p.k_in = ds.num_kv_heads > 0 ? k_in : nullptr;
    p.k_out = ds.num_kv_heads > 0 ? k_out : nullptr;
    p.positions = positions;
    p.cu_seqlens = positions ? nullptr : cu_seqlens;
    p.cos = cos_table;
    p.sin = sin_table;
    p.error_word = err_word;
    p.tokens = ds.tokens;
    p.H = ds.num_heads;
    p.Hkv = ds.num_kv_heads;
    p.width = 2 * ds.d;
    p.rot_dim = ds.rot_dim;
    p.n_pos = ds.n_pos;
    p.num_seqs = ds.num_seqs;
    p.seqlen = ds.seqlen;
    return launch_rope_qk(p, ds.dtype == DIFFATTN_DTYPE_BF16, ds.interleaved != 0, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? DIFFATTN_OK
               : DIFFATTN_ERR_CUDA;
}

// ------------------------------------------------------------- out_proj ---

diffattn_status diffattn_out_proj(const diffattn_out_proj_desc* desc, const void* x, const void* w, void* y,
                                  void* stream) {
    const CallRange nvtx_range("diffattn_out_proj");
    if (!desc) return DIFFATTN_ERR_INVALID_ARG;
    const diffattn_out_proj_desc& ds = *desc;
    if (ds.tokens < 0 || ds.in_features < 8 || ds.out_features < 8 || (ds.in_features % 8) != 0 ||
        (ds.out_features % 8) != 0)
        return DIFFATTN_ERR_INVALID_ARG;
    if (ds.tokens == 0) return DIFFATTN_OK;
    if (!x || !w || !y || !aligned16(x) || !aligned16(w) || !aligned16(y)) return DIFFATTN_ERR_INVALID_ARG;
    unsigned int* err_word = nullptr;
    if (error_word_ptr(&err_word) != cudaSuccess) return DIFFATTN_ERR_CUDA;
    CUtensorMap tm_x, tm_w;
    if (!encode_bf16_rows(&tm_x, x, (uint64_t)ds.in_features, (uint64_t)ds.tokens, 128) ||
        !encode_bf16_rows(&tm_w, w, (uint64_t)ds.in_features, (uint64_t)ds.out_features, 256))
        return DIFFATTN_ERR_CUDA;
    GemmParams p{};
    p.M = ds.tokens;
    p.N = ds.out_features;
    p.K = ds.in_features;
    p.y = y;
    p.error_word = err_word;
    p.timeout_ns = g_timeout_ns;
    return launch_out_proj(p, tm_x, tm_w, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DIFFATTN_OK
                                                                                             : DIFFATTN_ERR_CUDA;
}

// ---------------------------------------------------------------- merge ---

diffattn_status diffattn_merge_partials(const diffattn_merge_desc* desc, const float* lse, const float* o1,
                                        const float* o2, const float* lambda, int lambda_per_head,
                                        float lambda_init, const float* subln_w, void* out, void* stream) {
    const CallRange nvtx_range("diffattn_merge_partials");
    if (!desc) return DIFFATTN_ERR_INVALID_ARG;
    const diffattn_merge_desc& ds = *desc;
    if (ds.tokens < 0 || ds.num_heads < 1 || ds.dv < 4 || ds.dv > 512 || (ds.dv % 4) != 0 || ds.n_parts < 1)
        return DIFFATTN_ERR_INVALID_ARG;
    if (ds.out_dtype != DIFFATTN_DTYPE_F32 && ds.out_dtype != DIFFATTN_DTYPE_BF16) return DIFFATTN_ERR_INVALID_ARG;
    if (!(ds.eps >= 0.f) || !std::isfinite(ds.eps) || !std::isfinite(lambda_init)) return DIFFATTN_ERR_INVALID_ARG;
    if (ds.tokens == 0) return DIFFATTN_OK;
    if (!lse || !o1 || !o2 || !lambda || !subln_w || !out) return DIFFATTN_ERR_INVALID_ARG;
    if (!aligned16(lse) || !aligned16(o1) || !aligned16(o2) || !aligned16(subln_w) || !aligned16(out))
        return DIFFATTN_ERR_INVALID_ARG;
    if ((long long)ds.n_parts * ds.tokens * ds.num_heads * ds.dv >= (1LL << 40)) return DIFFATTN_ERR_INVALID_ARG;
    MergeParams p{};
    p.lse = lse;
    p.o1 = o1;
    p.o2 = o2;
    p.lambda = lambda;
    p.lambda_stride = lambda_per_head ? 1 : 0;
    p.lambda_init = lambda_init;
    p.subln_w = subln_w;
    p.eps = ds.eps;
    p.out = out;
    p.out_bf16 = ds.out_dtype == DIFFATTN_DTYPE_BF16;
    p.tokens = ds.tokens;
    p.H = ds.num_heads;
    p.dv = ds.dv;
    p.n_parts = ds.n_parts;
    return launch_merge(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

diffattn_status diffattn_get_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DIFFATTN_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess) return DIFFATTN_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return DIFFATTN_ERR_CUDA;
    }
    if (word & kErrBadSeqlens) return DIFFATTN_ERR_BAD_SEQLENS;
    if (word & kErrBadPositions) return DIFFATTN_ERR_BAD_POSITIONS;
    if (word & kErrTimeout) return DIFFATTN_ERR_TIMEOUT;
    if (word & kErrLayout) return DIFFATTN_ERR_CUDA;  // a kernel found its shared memory misaligned
    return DIFFATTN_OK;
}

const char* diffattn_status_string(diffattn_status s) {
    switch (s) {
        case DIFFATTN_OK: return "ok";
        case DIFFATTN_ERR_INVALID_ARG: return "invalid argument";
        case DIFFATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case DIFFATTN_ERR_CUDA: return "CUDA error";
        case DIFFATTN_ERR_TIMEOUT: return "kernel pipeline wait timed out";
        case DIFFATTN_ERR_BAD_SEQLENS: return "invalid cu_seqlens";
        case DIFFATTN_ERR_BAD_POSITIONS: return "rotary position outside the tables";
    }
    return "unknown status";
}

void diffattn_set_wait_timeout_ns(unsigned long long ns) { g_timeout_ns = ns ? ns : kDefaultWaitTimeoutNs; }

diffattn_status diffattn_set_fault_injection(int mode) {
    // A test hook: it takes effect only in a process that asks for test hooks.
    const char* on = std::getenv("DIFFATTN_TEST_HOOKS");
    if (on == nullptr || std::strcmp(on, "1") != 0) {
        g_inject = 0;
        return DIFFATTN_ERR_UNSUPPORTED;
    }
    if (mode < 0 || mode > 2) return DIFFATTN_ERR_INVALID_ARG;
    g_inject = mode;
    return DIFFATTN_OK;
}

}  // extern "C"
