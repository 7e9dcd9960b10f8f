/*
 * diffattn.h -- C ABI of the GB300 (sm_103a) differential-attention forward.
 *
 * Per diff head h, for query row i of a sequence (positions from 0), the
 * library computes
 *
 *   out[i] = RMSNorm( softmax(s Q1 K1^T)[i] V  -  lambda_h softmax(s Q2 K2^T)[i] V ) * w
 *            * (1 - lambda_init)
 *
 * with s = d^-0.5 on the component dim d, keys j <= i when causal, RMSNorm
 * over the dv = 2d values of one (token, head) with eps, and
 *   lambda = exp(lambda_q1 . lambda_k1) - exp(lambda_q2 . lambda_k2) + lambda_init,
 *   lambda_init(l) = 0.8 - 0.6 exp(-0.3 (l - 1)).
 * Sources: "DiffTransformer.py" (MultiHeadDifferentialAttention.forward: the
 * lambda reparameterisation, the causal mask, the two softmax maps and their
 * difference, the per-head RMSNorm and the (1 - lambda_init) scale;
 * DiffTransformer.__init__: the lambda_init schedule) and
 * "LlamaDiffSdpaAttention.py" (forward: the two attention calls combined as
 * attn1 - lambda_full * attn2, grouped key/value heads via repeat_kv on k1, k2
 * and v, the component-dim scale).
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller; the library never
 *    frees or retains them past the call's completion on `stream`.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Work is enqueued asynchronously; nothing synchronises except
 *    diffattn_get_device_status().
 *  - Argument errors are detected on the host and returned synchronously; in
 *    that case NOTHING is launched. Problems only a kernel can see (bad
 *    cu_seqlens contents, a pipeline wait that ran out of time) are recorded
 *    in a per-device error word read by diffattn_get_device_status(); kernels
 *    never trap or assert.
 *  - The library owns, per device, one small error word and cached launch
 *    state; it allocates nothing per call.
 */
#ifndef DIFFATTN_H_
#define DIFFATTN_H_

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DIFFATTN_OK = 0,
    DIFFATTN_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer      */
    DIFFATTN_ERR_UNSUPPORTED = 2,   /* valid request outside the built kernels' shapes */
    DIFFATTN_ERR_CUDA = 3,          /* a CUDA runtime / driver call failed             */
    DIFFATTN_ERR_TIMEOUT = 4,       /* a kernel pipeline wait gave up (device status)  */
    DIFFATTN_ERR_BAD_SEQLENS = 5,   /* cu_seqlens not monotone / out of range (device) */
    DIFFATTN_ERR_BAD_POSITIONS = 6  /* a rotary position outside the tables (device)  */
} diffattn_status;

typedef enum {
    DIFFATTN_DTYPE_F32 = 0,         /* q, k, v, out in fp32 (CUDA-core kernel)          */
    DIFFATTN_DTYPE_BF16 = 1         /* q, k, v, out in bf16 (tcgen05 tensor-core kernel) */
} diffattn_dtype;

/*
 * Problem shape.
 *  Dense mode (cu_seqlens == NULL): `batch` sequences of `seqlen` tokens each,
 *    packed back to back (token index = b * seqlen + position).
 *  Packed mode (cu_seqlens != NULL): `num_seqs` sequences; sequence s holds
 *    tokens cu_seqlens[s] .. cu_seqlens[s+1]-1 of `total_tokens`; `max_seqlen`
 *    must be >= every length (it sizes the launch; longer sequences are
 *    reported as DIFFATTN_ERR_BAD_SEQLENS by the kernel, not processed).
 *  num_heads = H diff heads; num_kv_heads = Hkv key/value diff heads, H % Hkv == 0;
 *    diff head h reads key/value head h / (H / Hkv) for both components.
 *  d = component dim (Q1, Q2, K1, K2); dv = value dim per diff head (must be 2d).
 *  eps = RMSNorm epsilon (1e-5 on the pages).
 */
typedef struct {
    int batch;
    int seqlen;
    int num_seqs;
    int max_seqlen;
    int total_tokens;
    int num_heads;
    int num_kv_heads;
    int d;
    int dv;
    diffattn_dtype dtype;
    float eps;
} diffattn_desc;

/*
 * lambda_init for layer `depth` (counted from 1): 0.8 - 0.6 * exp(-0.3 * (depth - 1)).
 * Source: "DiffTransformer.py", DiffTransformer.__init__ (decaying lambda_init).
 * Host-only, pure; returns NaN for depth < 1.
 */
float diffattn_lambda_init(int depth);

/*
 * lambda reparameterisation, one value per parameter set:
 *   lambda_out[i] = exp(sum_e lq1[i*d+e] * lk1[i*d+e]) - exp(sum_e lq2[i*d+e] * lk2[i*d+e])
 *                   + lambda_init
 * Source: "DiffTransformer.py", MultiHeadDifferentialAttention.forward,
 * "Compute lambda using reparameterization" (the Llama gist computes the same).
 *  lq1, lk1, lq2, lk2: device fp32 [n_sets][d], contiguous.
 *  lambda_out: device fp32 [n_sets]. n_sets = 1 for lambdas shared by all
 *  heads, H for per-head lambdas. Computed in fp32, not rounded further.
 * Errors: INVALID_ARG for null pointers, n_sets < 1, d < 1 or d > 1024.
 */
diffattn_status diffattn_lambda(const float* lq1, const float* lk1, const float* lq2,
                                const float* lk2, int n_sets, int d, float lambda_init,
                                float* lambda_out, void* stream);

/*
 * Name of the kernel diffattn_fwd / diffattn_fwd_train launch for `desc`
 * (packed nonzero: with cu_seqlens), or NULL for an unsupported dtype / d.
 * bf16 inputs run "diffattn_fwd_bf16_sm103a_kernel" (one CTA per 128 query rows
 * of one head of one sequence) or, when those items have at most 64 key tiles
 * (max_seqlen <= 8192), number at least two per SM and come from at most 64
 * packed sequences, "diffattn_fwd_bf16_persistent_kernel" (one CTA per SM
 * walking the items). The two give the same bits for the same rows. fp32
 * inputs run "diffattn_fwd_f32_kernel".
 * Host-only: no launch; the returned string is static.
 */
const char* diffattn_fwd_kernel(const diffattn_desc* desc, int packed);

/*
 * Differential-attention forward (one launch of the fused kernel).
 * Source: as in the file header; the output-difference form
 * O1/l1 - lambda O2/l2 of "LlamaDiffSdpaAttention.py", forward, with the
 * per-head RMSNorm of "DiffTransformer.py", forward.
 *  q   : [tokens][H][2d]   Q1 = q[..., :d], Q2 = q[..., d:]     (dtype of desc)
 *  k   : [tokens][Hkv][2d] K1 = k[..., :d], K2 = k[..., d:]
 *  v   : [tokens][Hkv][dv]
 *  out : [tokens][H][dv]   written for every token of every sequence
 *  lambda : device fp32, lambda_per_head ? [H] : [1] (e.g. from diffattn_lambda)
 *  lambda_init : the scalar of the (1 - lambda_init) output scale
 *  subln_w : device fp32 [dv], the RMSNorm weight shared by all heads
 *  causal : nonzero -> key j takes part in row i iff j <= i (same sequence)
 *  cu_seqlens : NULL (dense mode) or device int32 [num_seqs + 1], cu[0] = 0,
 *               nondecreasing, cu[num_seqs] = total_tokens
 *  All tensors contiguous; q, k, v, out 16-byte aligned. For bf16 the
 *  output is rounded to nearest even.
 * Supported: bf16 with d = 64, dv = 128 (tcgen05 kernel); fp32 with
 *  d in {16, 32, 64}, dv = 2d (CUDA-core kernel). Otherwise UNSUPPORTED.
 * Errors: INVALID_ARG (null pointer, non-positive sizes, H % Hkv != 0,
 *  dv != 2d, misalignment, tokens or indices beyond 2^31); UNSUPPORTED;
 *  CUDA (launch failure). An empty problem (no tokens, no sequences or
 *  max_seqlen 0) returns OK with nothing launched; its tensor pointers may
 *  then be NULL.
 */
diffattn_status diffattn_fwd(const diffattn_desc* desc, const void* q, const void* k,
                             const void* v, const float* lambda, int lambda_per_head,
                             float lambda_init, const float* subln_w, int causal,
                             const int* cu_seqlens, void* out, void* stream);

/*
 * The lambda reparameterisation and the forward in one call: diffattn_lambda
 * into lambda_out, then diffattn_fwd reading it, on the same stream. The two
 * formulas and their sources are those of the two entry points; the results
 * are theirs bit for bit. Because this call launches the lambda kernel itself,
 * right before the forward, the forward's loads, scores and softmax run while
 * the lambda kernel finishes, and only its epilogue waits for lambda (through
 * two separate calls every read of the forward waits for the kernel before it).
 *  lq1, lk1, lq2, lk2: device fp32 [n_sets][lambda_d], n_sets = H when
 *  lambda_per_head, else 1.
 *  lambda_out: device fp32 [n_sets], written by this call (4-byte aligned).
 *  Every other argument as in diffattn_fwd; the inputs must be complete when
 *  the call is made on the stream, as for any stream-ordered call.
 * Errors: those of diffattn_lambda (null vectors, lambda_d outside 1..1024)
 *  and of diffattn_fwd, all checked before anything is launched. An empty
 *  problem launches nothing (lambda_out is not written).
 */
diffattn_status diffattn_fwd_lambda(const diffattn_desc* desc, const void* q, const void* k,
                                    const void* v, const float* lq1, const float* lk1,
                                    const float* lq2, const float* lk2, int lambda_per_head,
                                    int lambda_d, float lambda_init, float* lambda_out,
                                    const float* subln_w, int causal, const int* cu_seqlens,
                                    void* out, void* stream);

/*
 * Forward for training: diffattn_fwd (bf16 tcgen05 kernel only) that also
 * saves what the backward pass needs, per (token, head):
 *  lse : device fp32 [tokens][H][2]: for component c, log2 of the softmax
 *        denominator in the log2 domain of the scaled scores, so that the
 *        probabilities are 2^(s * log2(e) * <Q_c, K_c[j]> - lse[..][c]);
 *  o1, o2 : device fp32 [tokens][H][dv]: the normalised attention outputs
 *        softmax(s Q1 K1^T) V and softmax(s Q2 K2^T) V, 16-byte aligned (fp32:
 *        the lambda gradient is a sum of many cancelling terms of these).
 * Errors: as diffattn_fwd; INVALID_ARG if any of lse, o1, o2 is NULL or
 * misaligned; UNSUPPORTED for fp32.
 */
diffattn_status diffattn_fwd_train(const diffattn_desc* desc, const void* q, const void* k,
                                   const void* v, const float* lambda, int lambda_per_head,
                                   float lambda_init, const float* subln_w, int causal,
                                   const int* cu_seqlens, void* out, float* lse, void* o1, void* o2,
                                   void* stream);

/*
 * Bytes of device workspace diffattn_bwd needs for `desc`: tokens x H x
 * (2 dv + 48) (the gradient of the pre-norm output in bf16, four fp32 row
 * statistics and 16 bf16 of the dK/dV kernel's row operand per (token, head)).
 */
unsigned long long diffattn_bwd_workspace_size(const diffattn_desc* desc);

/*
 * Backward pass of diffattn_fwd_train (bf16, d = 64, dv = 128): given dout, the
 * gradient of the loss with respect to out, and the forward's saved lse, o1,
 * o2, writes the gradients with respect to q, k, v (bf16, layouts of q, k, v),
 * lambda (fp32, [H] or [1] like `lambda`; for shared lambda the heads' sum) and
 * subln_w (fp32 [dv]). The pages define the forward only; these are its plain
 * derivatives (the modules on "DiffTransformer.py" and "LlamaDiffSdpaAttention.py"
 * train lambda_q1 ... lambda_k2 and the norm weight). Launches, on `stream`:
 * two memsets, a per-row kernel (the RMSNorm and output-scale gradient, the row
 * statistics of both softmaxes, the lambda and weight gradients), a dQ kernel
 * and a dK/dV kernel (tcgen05; grouped kv heads summed inside the CTA).
 * workspace: device, 16-byte aligned, >= diffattn_bwd_workspace_size(desc).
 * Errors: as diffattn_fwd (and INVALID_ARG for tokens x H beyond 2^31 - 64);
 * UNSUPPORTED for anything but bf16 with d = 64.
 * Use diffattn_lambda_bwd to turn the lambda gradient into the gradients of the
 * four lambda vectors.
 */
diffattn_status diffattn_bwd(const diffattn_desc* desc, const void* q, const void* k, const void* v,
                             const float* lambda, int lambda_per_head, float lambda_init,
                             const float* subln_w, int causal, const int* cu_seqlens, const void* dout,
                             const float* lse, const void* o1, const void* o2, void* dq, void* dk,
                             void* dv, float* dlambda, float* dsubln_w, void* workspace,
                             unsigned long long workspace_bytes, void* stream);

/*
 * Gradient of the lambda reparameterisation ("DiffTransformer.py",
 * MultiHeadDifferentialAttention.forward, "Compute lambda using
 * reparameterization"): with a = lq1 . lk1, b = lq2 . lk2 per set,
 *   dlq1 = dlambda e^a lk1, dlk1 = dlambda e^a lq1,
 *   dlq2 = -dlambda e^b lk2, dlk2 = -dlambda e^b lq2.
 * All device fp32; vectors [n_sets][d], dlambda [n_sets]. Outputs overwritten.
 */
diffattn_status diffattn_lambda_bwd(const float* lq1, const float* lk1, const float* lq2,
                                    const float* lk2, const float* dlambda, int n_sets, int d,
                                    float* dlq1, float* dlk1, float* dlq2, float* dlk2, void* stream);

/*
 * Shape of a forward against a key/value cache (decode, or a short block of new
 * queries appended to a cached sequence).
 *  batch sequences; each has q_len new query tokens and a cache of
 *  cache_capacity key/value rows, of which cache_seqlens[b] are valid (the new
 *  tokens included: they are the last q_len valid rows).
 *  num_heads, num_kv_heads, d, dv, dtype, eps as in diffattn_desc.
 *  num_splits: key splits per (sequence, kv head), at most 1024; 0 lets the
 *  library choose (the workspace size depends on it).
 *  host_seqlens: NULL, or a HOST copy of cache_seqlens (int32 [batch]) for
 *  callers that have one. With num_splits == 0 the library then plans the
 *  splits from the sequences' actual key counts (a ragged batch wants more
 *  splits than its capacity suggests); without it the plan sees only the
 *  shape. Read during the call, not retained; pass the same descriptor to
 *  diffattn_fwd_kvcache_workspace_size and to the forward, since the split
 *  count sizes the workspace. The device cache_seqlens remain the ones the
 *  kernels use and check.
 */
typedef struct {
    int batch;
    int q_len;
    int cache_capacity;
    int num_heads;
    int num_kv_heads;
    int d;
    int dv;
    diffattn_dtype dtype;
    float eps;
    int num_splits;
    const int* host_seqlens;
} diffattn_kv_desc;

/*
 * Bytes of device workspace diffattn_fwd_kvcache needs for `desc` (partial
 * softmax states of every key split); 0 for an invalid or empty shape.
 */
unsigned long long diffattn_fwd_kvcache_workspace_size(const diffattn_kv_desc* desc);

/*
 * Differential-attention forward of new queries against a key/value cache.
 * Query t of sequence b sits at position cache_seqlens[b] - q_len + t and, when
 * causal, sees cached keys j <= that position: the bottom-right aligned mask
 * triu(-inf, 1 + src_len - tgt_len) of "Add an isolated implementation of
 * FlashDiffAttention" (review snippet, alternative_forward), on the cache of
 * "LlamaDiffSdpaAttention.py" (forward, past_key_value.update with k1, k2
 * stacked). The per-row arithmetic is that of diffattn_fwd.
 *  q       : [batch][q_len][H][2d]            bf16
 *  k_cache : [batch][cache_capacity][Hkv][2d] bf16 (K1 | K2 per kv head)
 *  v_cache : [batch][cache_capacity][Hkv][dv] bf16
 *  cache_seqlens : NULL (every sequence holds cache_capacity keys) or device
 *                  int32 [batch], q_len <= cache_seqlens[b] <= cache_capacity
 *  workspace : device, >= diffattn_fwd_kvcache_workspace_size(desc) bytes,
 *              16-byte aligned, owned by the caller; its contents are scratch
 *  out     : [batch][q_len][H][dv] bf16
 * Two launches on `stream`: a key-split kernel (tensor cores; the cache read
 * through TMA) writing partial (max, sum, O) of both components to the
 * workspace, and a combine kernel (per-component log-sum-exp merge,
 * O1/l1 - lambda O2/l2, RMSNorm, weight, (1 - lambda_init)). Cache rows past
 * cache_seqlens[b] are read but never used: they may hold any bits.
 * Supported: bf16, d = 64, dv = 128, 1 <= q_len * (H / Hkv) <= 32, and
 * batch * cache_capacity below 2^31 - 64.
 * Errors: INVALID_ARG (null / misaligned pointers, bad sizes, workspace too
 * small), UNSUPPORTED, CUDA; cache_seqlens out of range -> BAD_SEQLENS through
 * diffattn_get_device_status (those sequences are not written).
 */
diffattn_status diffattn_fwd_kvcache(const diffattn_kv_desc* desc, const void* q, const void* k_cache,
                                     const void* v_cache, const int* cache_seqlens, const float* lambda,
                                     int lambda_per_head, float lambda_init, const float* subln_w,
                                     int causal, void* workspace, unsigned long long workspace_bytes,
                                     void* out, void* stream);

/*
 * The lambda reparameterisation and the cache forward in one call: the results
 * of diffattn_lambda into lambda_out and of diffattn_fwd_kvcache reading it, bit
 * for bit, from two launches instead of three. Only the combine kernel uses
 * lambda, so it forms lambda itself (each row's warp for its head, with the
 * lambda kernel's arithmetic) and the warps of the first query of the first
 * sequence write lambda_out.
 *  lq1, lk1, lq2, lk2: device fp32 [n_sets][lambda_d], n_sets = H when
 *  lambda_per_head, else 1.
 *  lambda_out: device fp32 [n_sets], written by this call (4-byte aligned).
 *  Every other argument as in diffattn_fwd_kvcache; the inputs must be
 *  complete when the call is made on the stream, as for any stream-ordered call.
 * Errors: those of diffattn_lambda (null vectors, lambda_d outside 1..1024)
 *  and of diffattn_fwd_kvcache, all checked before anything is launched. An
 *  empty batch launches nothing (lambda_out is not written).
 */
diffattn_status diffattn_fwd_kvcache_lambda(const diffattn_kv_desc* desc, const void* q, const void* k_cache,
                                            const void* v_cache, const int* cache_seqlens, const float* lq1,
                                            const float* lk1, const float* lq2, const float* lk2,
                                            int lambda_per_head, int lambda_d, float lambda_init,
                                            float* lambda_out, const float* subln_w, int causal,
                                            void* workspace, unsigned long long workspace_bytes, void* out,
                                            void* stream);

/*
 * Size of the scratch array behind diffattn_fwd_kvcache_noalloc: 16 MiB of
 * device memory per GPU that loads the library, held until the process exits.
 */
#define DIFFATTN_NOALLOC_SCRATCH_BYTES (16ull << 20)

/*
 * diffattn_fwd_kvcache without a workspace argument, for callers that cannot
 * allocate device memory themselves: code embedded in a host program that owns
 * every device allocation (a serving runtime with a fixed memory arena, a
 * plugin interface that hands the library no allocator), or a caller on a
 * latency-critical path where a device allocation, which may synchronise the
 * device, is not acceptable. No counterpart on the pages: this is a calling
 * convention of this library, not part of the method.
 * The key-split partials go to one static device array of
 * DIFFATTN_NOALLOC_SCRATCH_BYTES instead of a caller workspace; the function
 * itself allocates nothing. Arguments and results are those of
 * diffattn_fwd_kvcache. The first call on a device looks up the array's device
 * address (once per device, with that device current); make that first call
 * before any stream capture. Every call on a device shares the one array:
 * calls that overlap on the GPU (different streams, or different host threads)
 * race on it and must be serialised by the caller. Nothing in the array has to
 * start at zero: each call writes every partial it later reads.
 * With desc->num_splits == 0 the automatic split plan is lowered, one split at
 * a time, until the partials fit the array; a caller-forced count is kept.
 * Errors: the descriptor is checked first and gives the statuses of
 * diffattn_fwd_kvcache; then DIFFATTN_ERR_UNSUPPORTED when even the lowest
 * split count (or the forced one) needs more than DIFFATTN_NOALLOC_SCRATCH_BYTES
 * of partials (see diffattn_fwd_kvcache_workspace_size), and DIFFATTN_ERR_CUDA
 * if the address lookup fails.
 */
diffattn_status diffattn_fwd_kvcache_noalloc(const diffattn_kv_desc* desc, const void* q, const void* k_cache,
                                             const void* v_cache, const int* cache_seqlens, const float* lambda,
                                             int lambda_per_head, float lambda_init, const float* subln_w,
                                             int causal, void* out, void* stream);

/*
 * Rotary position embedding ahead of the attention.
 *
 * Passages: "LlamaDiffSdpaAttention.py", forward ("Apply RoPE before splitting":
 * apply_rotary_pos_emb on the whole 2d-wide head row, half-split pairs, then the
 * q1 | q2 chunk) and "Add an isolated implementation of FlashDiffAttention"
 * (test script: apply_rotary_emb(..., interleaved=True) on the doubled d-wide
 * heads). Both are this rule: each head row of width 2d is split into segments
 * of rot_dim coordinates; in a segment, pair i < rot_dim/2 is (i, i + rot_dim/2)
 * (interleaved = 0) or (2i, 2i+1) (interleaved = 1), rotated by the angle
 * pos * theta^(-2i/rot_dim):  a' = a cos - b sin,  b' = b cos + a sin.
 * rot_dim = 2d gives the Llama placement, rot_dim = d the doubled-head one.
 */
typedef struct diffattn_rope_desc {
    long long tokens;   /* rows of q (and of k)                                         */
    int num_heads;      /* H: q is [tokens][H][2d]                                      */
    int num_kv_heads;   /* Hkv: k is [tokens][Hkv][2d]; 0 rotates q only                */
                        /* (num_heads 0 rotates k only; q_in / q_out are then ignored)  */
    int d;              /* component dim; head rows are 2d wide; d % 4 == 0             */
    int dtype;          /* diffattn_dtype of q and k                                     */
    int rot_dim;        /* d or 2d                                                       */
    int interleaved;    /* 0: pairs (i, i + rot_dim/2); 1: pairs (2i, 2i+1)              */
    int n_pos;          /* rows of the cos / sin tables                                  */
    int num_seqs;       /* > 0 with cu_seqlens: positions restart at every sequence      */
    int seqlen;         /* dense batches (no positions, no cu_seqlens): pos = t % seqlen */
} diffattn_rope_desc;

/*
 * Fills cos_out, sin_out (device fp32 [n_pos][rot_dim/2], caller-owned) with
 * cos / sin of p * theta^(-2i/rot_dim), computed in fp64 on the device and
 * rounded once (the pages' modules cache these tables and cast them to bf16).
 * Errors: INVALID_ARG for null pointers, n_pos < 1, odd or non-positive rot_dim,
 * theta <= 0; CUDA if the launch fails. Asynchronous on `stream`.
 */
diffattn_status diffattn_rope_tables(double theta, int n_pos, int rot_dim, float* cos_out, float* sin_out,
                                     void* stream);

/*
 * Rotates q (and k) with the tables of diffattn_rope_tables. Positions come
 * from `positions` (device int32 [tokens], e.g. a decode step's cache offsets)
 * if given, else from `cu_seqlens` (device int32 [num_seqs + 1]: position = token
 * index inside its sequence), else from the dense layout (t % seqlen).
 * q_out may equal q_in and k_out k_in (in place); all device pointers are
 * caller-owned and 16-byte aligned; k_in / k_out are ignored when num_kv_heads
 * is 0. A position outside [0, n_pos) leaves that row unrotated (copied through)
 * and makes diffattn_get_device_status return DIFFATTN_ERR_BAD_POSITIONS.
 * Errors: INVALID_ARG for null or misaligned pointers, rot_dim not d or 2d,
 * rot_dim % 8 != 0, a missing position source; CUDA if the launch fails.
 */
diffattn_status diffattn_rope_qk(const diffattn_rope_desc* desc, const int* positions, const int* cu_seqlens,
                                 const float* cos_table, const float* sin_table, const void* q_in, void* q_out,
                                 const void* k_in, void* k_out, void* stream);

/*
 * The rotary embedding of q, applied by the forward kernels themselves: each
 * query tile is rotated in shared memory once its TMA load lands, before the
 * first score MMA reads it, so q goes through the forward unrotated and is not
 * written back. Same rule, tables and rounding as diffattn_rope_qk (the two give
 * the same bits), positions = the query's index inside its sequence (dense
 * batches and cu_seqlens alike).
 *  cos, sin   : device fp32 [n_pos][rot_dim / 2] from diffattn_rope_tables,
 *               16-byte aligned, caller-owned
 *  rot_dim    : d or 2d, a multiple of 8; interleaved: 0 or 1
 */
typedef struct diffattn_rope_q {
    const float* cos;
    const float* sin;
    int n_pos;
    int rot_dim;
    int interleaved;
} diffattn_rope_q;

/*
 * diffattn_fwd on q before its rotary embedding: the kernels rotate each query
 * tile as it arrives ("LlamaDiffSdpaAttention.py", forward, "Apply RoPE before
 * splitting"; "Add an isolated implementation of FlashDiffAttention", test
 * script, apply_rotary_emb(..., interleaved=True) on the doubled heads). k must
 * already be rotated, e.g. by diffattn_rope_qk with num_heads = 0 (k only): every
 * query tile reads every key tile it sees, so keys are rotated once, apart.
 * Arguments, layouts and results otherwise as diffattn_fwd (the same bits as
 * diffattn_rope_qk then diffattn_fwd). It runs on the one-item-per-CTA forward
 * kernel, which stages each tile's cos / sin rows in shared memory: measured on
 * GB300 it beats the separate q pass on small or launch-bound calls (B = 2,
 * T = 512: 22.0 against 29.7 us with k's pass) and ties it on long sequences
 * (T = 16384), but on batches of short sequences, where diffattn_fwd takes the
 * persistent kernel, diffattn_rope_qk on q and k then diffattn_fwd is faster
 * (B = 4, T = 2048: 121 against 136 us).
 * Supported: bf16, d = 64 (UNSUPPORTED otherwise).
 * Errors: as diffattn_fwd; INVALID_ARG for a null `rope`, null or misaligned
 * tables, rot_dim not d or 2d or not a multiple of 8, n_pos < 1. A query whose
 * position is outside [0, n_pos) is left unrotated and
 * diffattn_get_device_status returns DIFFATTN_ERR_BAD_POSITIONS.
 */
diffattn_status diffattn_fwd_rope_q(const diffattn_desc* desc, const void* q, const void* k, const void* v,
                                    const float* lambda, int lambda_per_head, float lambda_init,
                                    const float* subln_w, int causal, const int* cu_seqlens,
                                    const diffattn_rope_q* rope, void* out, void* stream);

/*
 * Context-parallel merge. The pages give no context-parallel scheme; it
 * follows from the forward ("DiffTransformer.py",
 * MultiHeadDifferentialAttention.forward): each component's softmax over all
 * visible keys combines its softmaxes over disjoint key blocks, weighted by
 * their sums of exponentials, and the combine with lambda and the RMSNorm (not
 * linear) run after both merges. A part is what diffattn_fwd_train saves for
 * one block of keys: lse_c (log2 of the sum of 2^(scaled score)) and O_c
 * normalised over that block. Per (token, head) row and component, with
 * L = max_j lse_c^j:  O_c = sum_j 2^(lse_c^j - L) O_c^j / sum_j 2^(lse_c^j - L);
 * then out = RMSNorm(O_1 - lambda O_2) * w * (1 - lambda_init).
 */
typedef struct diffattn_merge_desc {
    long long tokens;   /* query rows                                           */
    int num_heads;      /* H                                                    */
    int dv;             /* value width, a multiple of 4, at most 512            */
    int n_parts;        /* key blocks, >= 1                                     */
    int out_dtype;      /* diffattn_dtype of out                                */
    float eps;          /* RMSNorm epsilon                                      */
} diffattn_merge_desc;

/*
 * lse: device fp32 [n_parts][tokens][H][2]; o1, o2: device fp32
 * [n_parts][tokens][H][dv] (parts stacked; a part in which a row sees no key
 * has lse = -inf there and its O is not read); lambda fp32 [1] or [H]
 * (lambda_per_head); subln_w fp32 [dv]; out [tokens][H][dv] in out_dtype. All
 * device pointers caller-owned and 16-byte aligned. A row with no visible key
 * in any part gets 0 for that component. Errors: INVALID_ARG for null or
 * misaligned pointers and sizes outside the above; CUDA if the launch fails.
 * Asynchronous on `stream`.
 */
diffattn_status diffattn_merge_partials(const diffattn_merge_desc* desc, const float* lse, const float* o1,
                                        const float* o2, const float* lambda, int lambda_per_head,
                                        float lambda_init, const float* subln_w, void* out, void* stream);

/*
 * Output projection after the attention. Passages: "LlamaDiffSdpaAttention.py",
 * forward (the attention output reshaped to [tokens, H * dv] and passed through
 * o_proj = nn.Linear(H * dv, hidden, bias=False)); "DiffTransformer.py" (W_o,
 * no bias). nn.Linear stores W as [out_features][in_features]:
 *   y[t][n] = sum_k x[t][k] W[n][k]        (bf16 in, fp32 accumulate, bf16 out)
 */
typedef struct diffattn_out_proj_desc {
    int tokens;         /* M: rows of x and y                                   */
    int in_features;    /* K = H * dv; a multiple of 8                          */
    int out_features;   /* N; a multiple of 8                                   */
} diffattn_out_proj_desc;

/*
 * x: device bf16 [tokens][in_features] (e.g. diffattn_fwd's output viewed as
 * [tokens][H * dv]); w: device bf16 [out_features][in_features]; y: device bf16
 * [tokens][out_features]. All caller-owned, 16-byte aligned. Errors:
 * INVALID_ARG for null or misaligned pointers and sizes outside the above; CUDA
 * if a tensor map or the launch fails. Asynchronous on `stream`; a pipeline wait
 * that gives up is reported by diffattn_get_device_status as TIMEOUT.
 */
diffattn_status diffattn_out_proj(const diffattn_out_proj_desc* desc, const void* x, const void* w, void* y,
                                  void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error word.
 * Returns OK, TIMEOUT, BAD_SEQLENS, BAD_POSITIONS (the first error recorded since
 * the last read), or CUDA if the synchronisation itself failed.
 */
diffattn_status diffattn_get_device_status(void* stream);

/* Static, human-readable name of a status code. */
const char* diffattn_status_string(diffattn_status status);

/*
 * Library setting (no paper counterpart): the limit, in nanoseconds, after
 * which a kernel pipeline wait gives up and records DIFFATTN_ERR_TIMEOUT.
 * 0 restores the default (2 s). Affects launches made after the call.
 */
void diffattn_set_wait_timeout_ns(unsigned long long ns);

/*
 * TEST ONLY: not part of the library's interface for callers, and off unless
 * the process environment holds DIFFATTN_TEST_HOOKS=1 when it is called.
 * Hook (no paper counterpart) for the failure-detection tests. mode 1: the copy
 * producer of the bf16 forward kernel issues no loads, so the barriers every
 * other role waits on are never armed; each wait runs out after the wait limit,
 * the kernel records DIFFATTN_ERR_TIMEOUT, frees its tensor memory and returns,
 * and diffattn_get_device_status reports it. mode 2: the epilogue warpgroup of
 * the persistent bf16 forward pauses about 20 us (a bounded spin) before each
 * item, so that the softmax warps run ahead of it; the results and the status
 * must not change. mode 0 (the default) turns it off. Affects launches made
 * after the call; nothing faults, traps or hangs.
 * Returns DIFFATTN_OK; DIFFATTN_ERR_UNSUPPORTED (injection left off) when
 * DIFFATTN_TEST_HOOKS=1 is not set; DIFFATTN_ERR_INVALID_ARG for another mode.
 */
diffattn_status diffattn_set_fault_injection(int mode);

#ifdef __cplusplus
}
#endif

#endif /* DIFFATTN_H_ */
