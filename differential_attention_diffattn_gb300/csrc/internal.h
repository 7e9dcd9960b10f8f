// Launch parameters shared by the host C-ABI layer and the kernel translation
// units of the library. Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace diffattn {

// Bits of the per-device error word written by kernels.
enum : uint32_t { kErrTimeout = 1u, kErrBadSeqlens = 2u, kErrBadPositions = 4u, kErrLayout = 8u };

// Default limit of every bounded pipeline wait inside a kernel.
constexpr unsigned long long kDefaultWaitTimeoutNs = 2000000000ull;

// One forward problem after host validation. Sequence s covers tokens
// [seq_start(s), seq_start(s) + seq_len(s)): dense mode (cu_seqlens == nullptr)
// uses s * seqlen and seqlen; packed mode reads cu_seqlens on the device.
struct FwdParams {
    const void* q;            // [tokens][H][2d]
    const void* k;            // [tokens][Hkv][2d]
    const void* v;            // [tokens][Hkv][dv]
    void* out;                // [tokens][H][dv]
    const float* lambda;      // [H] or [1]
    const float* subln_w;     // [dv]
    const int* cu_seqlens;    // nullptr (dense) or [num_seqs + 1]
    unsigned int* error_word; // per-device error bits
    int num_seqs;             // dense: batch
    int seqlen;               // dense: tokens per sequence
    int max_seqlen;           // sizes the grid; packed sequences longer are errors
    int total_tokens;
    int H, Hkv, d, dv;
    int lambda_stride;        // 1: per head, 0: shared
    int causal;
    float lambda_init;
    float eps;
    float scale_log2;         // d^-0.5 * log2(e)
    float scale;              // d^-0.5
    unsigned long long timeout_ns;
    int inject;               // test hook: 1 = the copy producer issues no loads; 2 = the persistent
                              // kernel's epilogue pauses ~20 us before each item
    int group_heads;          // one-item-per-CTA bf16 kernel: heads per launch group (divides H)
    const float* rope_cos;    // rotary embedding of q inside the bf16 kernels (null: q is used as given):
    const float* rope_sin;    //   fp32 [rope_npos][rope_dim / 2] tables; position = index in the sequence
    int rope_npos, rope_dim, rope_interleaved;
    int lambda_pending;       // bf16 kernels: 1 when the kernel launched just before this one on the stream
                              // (by the same call) is the lambda kernel, which writes `lambda` and nothing
                              // else: every other input is complete at launch, so only the reads of lambda
                              // wait for that grid (the loads and the first tiles run under it); 0: every
                              // read waits for the preceding grid
    float* lse;               // training outputs (all null, or all set; bf16 kernel only):
    void* o1;                 //   lse [tokens][H][2] fp32 (log2 domain of the scaled scores),
    void* o2;                 //   o1, o2 [tokens][H][dv] fp32 = O_c / l_c
    // set (one-item-per-CTA bf16 kernel): lambda is formed in the kernel from these
    // [sets][lambda_d] vectors (the `lambda` read is skipped) and written to lambda_out
    const float *lq1, *lk1, *lq2, *lk2;
    int lambda_d;
    float* lambda_out;
};

// TMA descriptors of the bf16 operands, built on the host per call.
struct FwdTensorMaps {
    CUtensorMap q, k, v, out;  // out: [tokens][H * dv] bf16, 64 x 128 boxes (bulk tensor stores)
    CUtensorMap o1, o2;        // training outputs: [tokens][H * dv] fp32, 32 x 128 boxes (bulk tensor stores)
};

// One forward against a key/value cache (decode / short query blocks).
struct KvParams {
    const void* q;             // [batch][q_len][H][2d]
    const void* k;             // [batch][capacity][Hkv][2d]
    const void* v;             // [batch][capacity][Hkv][dv]
    void* out;                 // [batch][q_len][H][dv]
    const float* lambda;       // [H] or [1]
    const float* subln_w;      // [dv]
    const int* cache_seqlens;  // nullptr (all = capacity) or [batch]
    unsigned int* error_word;
    float* ws_o;               // [batch*q_len*H][num_splits][2][dv]   partial O per split
    float* ws_ml;              // [batch*q_len*H][num_splits][2][2]    (m, l) per split
    int batch, q_len, capacity;
    int H, Hkv;
    int lambda_stride;
    int causal;
    int num_splits;            // key splits per (batch, kv head)
    int chunk;                 // keys per split (multiple of 64)
    float lambda_init;
    float eps;
    float scale;               // d^-0.5
    unsigned long long timeout_ns;
    // set: the combine kernel forms lambda from these [sets][lambda_d] vectors
    // (lambda unused) and writes it to lambda_out
    const float *lq1, *lk1, *lq2, *lk2;
    int lambda_d;
    float* lambda_out;
};

// TMA descriptors of the caches: [batch * capacity][Hkv * 2d] and
// [batch * capacity][Hkv * dv], boxes of 64 columns x 64 rows.
struct KvTensorMaps {
    CUtensorMap k, v;
};

// Backward pass (bf16, d = 64, dv = 128).
struct BwdParams {
    const float* lambda;       // [H] or [1]
    int lambda_stride;
    int causal;
    const int* cu_seqlens;     // nullptr (dense) or [num_seqs + 1]
    int num_seqs, seqlen, max_seqlen, total_tokens;
    int H, Hkv;
    float scale, scale_log2;
    const float* rowstat;      // [H][tokens][4]: -lse1, -lse2, -delta1, -delta2 (workspace)
    // [H][tokens][16] bf16 (workspace), the row operand of the dK/dV kernel's extra K step:
    // slots 0-2 and 3-5 split -lse_c / scale_log2 into three bf16 terms (c = 1, 2), 6-8 split
    // -delta_1, 10-11 hold delta_1 - delta_2 as two terms, the rest zero
    const void* stat_aug;
    void* dq;                  // [tokens][H][2d]
    void* dk;                  // [tokens][Hkv][2d]
    void* dv;                  // [tokens][Hkv][dv]
    unsigned int* error_word;
    unsigned long long timeout_ns;
    int dq_tiles_outer;        // grid order of the dQ kernel: 1 (head, sequence, tile), 0 (head, tile, sequence)
    int dkv_tiles_outer;       // the same for the dK/dV kernel (kv heads)
    int dq_group_heads;        // (head, tile) order: heads per launch group of the dQ kernel (divides H)
    int dkv_group_kv;          // kv heads per launch group of the dK/dV kernel (divides Hkv)
};

// TMA descriptors of the backward kernels: q and dD with 128- and 64-row boxes,
// k and v with 128-row boxes.
struct BwdTensorMaps {
    CUtensorMap q128, q64, k128, v128, dd128, dd64;
    CUtensorMap aug64;  // stat_aug as [H * tokens][16], 64-row boxes, 32-byte swizzle
};

// Per-row preprocessing of the backward (CUDA cores).
struct BwdPreParams {
    const void* dout;          // [tokens][H][dv] bf16
    const void* o1;            // [tokens][H][dv] fp32, normalised O1 (forward)
    const void* o2;
    const float* lse;          // [tokens][H][2]
    const float* lambda;
    int lambda_stride;
    float lambda_init;
    const float* subln_w;      // [dv]
    float eps;
    int tokens, H;
    void* dd;                  // out: [tokens][H][dv] bf16, gradient of the pre-norm output
    float* rowstat;            // out: [H][tokens][4], negated
    void* stat_aug;            // out: [H][tokens][16] bf16 (BwdParams::stat_aug)
    float scale_log2;          // d^-0.5 * log2(e)
    float* dlambda;            // out (accumulated): [H] or [1]
    float* dsubln_w;           // out (accumulated): [dv]
    unsigned int* error_word;  // device error bits (a wait that timed out)
    uint64_t timeout_ns;       // bound of every wait
};

// Rotary embedding of q [tokens][H][width] and k [tokens][Hkv][width] (width = 2d).
struct RopeParams {
    const void* q_in;
    void* q_out;
    const void* k_in;          // may be null with Hkv = 0
    void* k_out;
    const int* positions;      // [tokens] or null
    const int* cu_seqlens;     // [num_seqs + 1] or null
    const float* cos;          // [n_pos][rot_dim / 2]
    const float* sin;
    unsigned int* error_word;
    long long tokens;
    int H, Hkv, width, rot_dim, n_pos, num_seqs, seqlen;
};

// Merge of partials over key blocks (context-parallel split).
struct MergeParams {
    const float* lse;          // [n_parts][tokens][H][2]
    const float* o1;           // [n_parts][tokens][H][dv]
    const float* o2;
    const float* lambda;       // [H] or [1]
    int lambda_stride;
    float lambda_init;
    const float* subln_w;      // [dv]
    float eps;
    void* out;                 // [tokens][H][dv], bf16 or fp32
    int out_bf16;
    long long tokens;
    int H, dv, n_parts;
};

// Output projection y[M][N] = x[M][K] W[N][K]^T (bf16).
struct GemmParams {
    int M, N, K;
    void* y;
    unsigned int* error_word;
    unsigned long long timeout_ns;
};

// Kernel launchers (each defined in its own translation unit). They return the
// cudaError_t of the launch.
cudaError_t launch_lambda(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                          int n_sets, int d, float lambda_init, float* out, cudaStream_t stream);
cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd_bf16_sm103a(const FwdParams& p, const FwdTensorMaps& maps, cudaStream_t stream);
cudaError_t launch_fwd_bf16_persistent(const FwdParams& p, const FwdTensorMaps& maps, cudaStream_t stream);
cudaError_t launch_decode(const KvParams& p, const KvTensorMaps& maps, cudaStream_t stream);
cudaError_t launch_decode_tc(const KvParams& p, const KvTensorMaps& maps, cudaStream_t stream);
cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream);
cudaError_t launch_bwd_sm103a(const BwdParams& p, const BwdTensorMaps& maps, cudaStream_t stream);
cudaError_t launch_lambda_bwd(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                              const float* dlambda, int n_sets, int d, float* dlq1, float* dlk1, float* dlq2,
                              float* dlk2, cudaStream_t stream);
cudaError_t launch_rope_tables(double theta, int n_pos, int rot_dim, float* cos_out, float* sin_out,
                               cudaStream_t stream);
cudaError_t launch_rope_qk(const RopeParams& p, bool bf16, bool interleaved, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
cudaError_t launch_out_proj(const GemmParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                            cudaStream_t stream);
int decode_rows_supported(int rows);  // R = q_len * (H / Hkv) the cache forward takes
int decode_ctas_per_sm();             // resident split CTAs per SM
int decode_max_splits();              // most key splits the combine kernel merges
int decode_tc_rows_supported(int rows);
int decode_tc_ctas_per_sm();

}  // namespace diffattn
