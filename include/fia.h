/*
 * fia.h -- C ABI of the fused inference attention library (sm_103a).
 *
 * The operator, as the FusedInferAttentionScore pages define it
 * (torch_npu.npu_fused_infer_attention_score_v2, "计算公式";
 * torch_npu.npu_prompt_flash_attention, "功能说明"):
 *
 *     attention_out = softmax(scale_value * query . key^T + atten_mask) . value
 *     softmax_lse   = log(sum(exp(s - max(s)))) + max(s)     (fp32, optional)
 *
 * Three entry points cover the pages' cases:
 *   fia_prefill  -- full attention, Q_S >= 1 (PromptFlashAttention)
 *   fia_decode   -- incremental attention, Q_S = 1 (or up to 16 new tokens),
 *                   paged or contiguous KV cache, optionally MLA (query_rope /
 *                   key_rope) (IncreFlashAttention)
 *   bsa_forward  -- block-sparse attention selected by blockSparseMask
 *                   (aclnnBlockSparseAttentionV2)
 * Each has a first phase that validates the arguments and reports the scratch
 * ("workspace") size, mirroring aclnn's two-phase GetWorkspaceSize + execute
 * calls (aclnnFusedInferAttentionScoreV5, "函数原型").
 *
 * Conventions shared by every call:
 *   - Tensors are described by fia_tensor: a data pointer, an element type and a
 *     row-major, contiguous shape (the pages accept contiguous tensors only).
 *     Data pointers of execute calls are DEVICE pointers, 16-byte aligned.
 *   - Host arrays (actual_seq_qlen / actual_seq_kvlen) are read during the call
 *     and not kept.
 *   - Ownership: the caller owns every buffer (inputs, outputs, workspace).  The
 *     library allocates no device memory, keeps no pointer after returning, and
 *     launches its kernels asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).
 *   - The return value covers argument validation and kernel launch only.  Errors
 *     found on the device (a bounded wait that ran out) are recorded in the
 *     workspace and read with fia_device_status().
 *   - Rows with no key to attend to (K/V with S2 = 0, a fully masked row, a
 *     padding row past a batch's actual query length) give attention_out = 0 and
 *     softmax_lse = +inf, extending the pages' empty-tensor rule
 *     (npu_fused_infer_attention_score_v2, "入参为空的处理").
 *   - A query with zero elements returns FIA_OK without launching anything.
 */
#ifndef FIA_H_
#define FIA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FIA_API __attribute__((visibility("default")))
#else
#define FIA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fia_status {
  FIA_OK = 0,
  FIA_ERR_NULL = 1,          /* a required pointer is NULL                                  */
  FIA_ERR_DTYPE = 2,         /* element types disagree or are not supported                 */
  FIA_ERR_SHAPE = 3,         /* ranks/dims inconsistent (e.g. key != value shape)           */
  FIA_ERR_LAYOUT = 4,        /* unknown input_layout                                        */
  FIA_ERR_UNSUPPORTED = 5,   /* valid on the pages but not implemented by this library     */
  FIA_ERR_SEQLEN = 6,        /* actual_seq_* list length or values invalid                  */
  FIA_ERR_BLOCK_TABLE = 7,   /* block_table / block_size invalid                            */
  FIA_ERR_WORKSPACE = 8,     /* workspace NULL or smaller than the reported size            */
  FIA_ERR_CUDA = 9,          /* a CUDA runtime call or kernel launch failed                 */
  FIA_ERR_TIMEOUT = 10,      /* device: a bounded wait inside a kernel ran out              */
  FIA_ERR_HEADS = 11,        /* num_heads / num_key_value_heads invalid (GQA rules)         */
  FIA_ERR_SPARSE_MODE = 12,  /* sparse_mode outside 0..4 or its mask requirements unmet     */
  FIA_ERR_ALIGNMENT = 13     /* a device pointer is not 16-byte aligned                     */
} fia_status;

typedef enum fia_dtype {
  FIA_DTYPE_F16 = 0,
  FIA_DTYPE_BF16 = 1,
  FIA_DTYPE_F32 = 2,
  FIA_DTYPE_I32 = 3,
  FIA_DTYPE_I64 = 4,
  FIA_DTYPE_U8 = 5,
  FIA_DTYPE_BOOL = 6,
  FIA_DTYPE_I8 = 7,
  FIA_DTYPE_F8E4M3 = 8   /* float8 e4m3 (FN: no infinities), the FP8 block-sparse inputs */
} fia_dtype;

/* A contiguous row-major tensor.  ndim == 0 or data == NULL means "absent"
 * for optional arguments. */
typedef struct fia_tensor {
  void* data;
  int32_t dtype;       /* fia_dtype */
  int32_t ndim;        /* 0..5 */
  int64_t shape[5];
} fia_tensor;

/* Keyword arguments of the pages' Python API (npu_fused_infer_attention_score_v2
 * parameter list; npu_prompt_flash_attention prototype).  Fill with
 * fia_params_init() and override what is needed. */
typedef struct fia_params {
  int64_t num_heads;              /* Q_N (num_query_heads / num_heads)                         */
  int64_t num_key_value_heads;    /* KV_N; 0 means equal to num_heads; Q_N % KV_N == 0,
                                     Q_N / KV_N <= 64                                          */
  double scale_value;             /* softmax_scale / scale_value; default 1.0; must be > 0     */
  const char* input_layout;       /* "BSH", "BSND", "BNSD" or "TND"; default "BSH"             */
  int64_t sparse_mode;            /* 0..4; 2 = leftUpCausal, 3 = rightDownCausal, 4 = band     */
  int64_t pre_tokens;             /* band (mode 4) width before the diagonal; default 2^31-1   */
  int64_t next_tokens;            /* band (mode 4) width after the diagonal; default 2^31-1    */
  const int64_t* actual_seq_qlen;   /* host array or NULL; TND: cumulative, no leading 0       */
  int64_t n_actual_seq_qlen;
  const int64_t* actual_seq_kvlen;  /* host array or NULL; TND: cumulative, no leading 0       */
  int64_t n_actual_seq_kvlen;
  int64_t block_size;             /* PageAttention tokens per block (0 = no paging)           */
  int32_t softmax_lse_flag;       /* return_softmax_lse: 1 = write softmax_lse                 */
  int32_t inner_precise;          /* accepted (0..3); the kernels always keep fp32 softmax    */
} fia_params;

/* Fills *p with the pages' defaults. */
FIA_API void fia_params_init(fia_params* p);

/* ------------------------------------------------------------------------
 * fia_prefill: full attention with Q_S >= 1 over contiguous key/value.
 *   query  (B,S1,H) BSH | (B,S1,N1,D) BSND | (B,N1,S1,D) BNSD | (T1,N1,D) TND;
 *          f16 or bf16.  D is 64 or 128.
 *   key, value: same layout and element type, N2 heads, identical shapes.
 *   atten_mask: optional.  sparse_mode 2/3/4 compute their pattern from
 *          indices; a mask given there must be (2048,2048) / (1,2048,2048) /
 *          (1,1,2048,2048) and is not read.  Mode 4 (band): query row i sees
 *          keys i + d - pre_tokens .. i + d + next_tokens, d = S2 - S1 of the
 *          batch (npu_fused_infer_attention_score_v2, sparse_mode; pre/next
 *          clamped to +-2^30).  Mode 0 with a mask, and mode 1 (allMask,
 *          mask required): bool/int8/uint8, device memory, contiguous, shape
 *          (S1m,S2m), (B|1,S1m,S2m) or (B|1,1,S1m,S2m) with S1m / S2m at least
 *          every batch's query / key length; byte [b][i][j] != 0 masks key j of
 *          the batch's query row i (batch-local indices, also for TND).  Mode 0
 *          also keeps only i - pre_tokens <= j <= i + next_tokens.  A mask
 *          whose address and S2m are multiples of 16 bytes is read fastest
 *          (8 and 4 next; otherwise byte by byte).  A row with every key
 *          masked gives out 0 and lse +inf.
 *   attention_out: the query's shape and element type.
 *   softmax_lse: fp32 (B,N1,S1,1), or (T1,N1,1) for TND; used when
 *          params->softmax_lse_flag != 0 (may be absent otherwise).
 * ------------------------------------------------------------------------ */
FIA_API fia_status fia_prefill_get_workspace_size(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                          const fia_tensor* atten_mask, const fia_params* params,
                                          const fia_tensor* attention_out, const fia_tensor* softmax_lse,
                                          size_t* workspace_bytes);
FIA_API fia_status fia_prefill(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                       const fia_tensor* atten_mask, const fia_params* params, const fia_tensor* attention_out,
                       const fia_tensor* softmax_lse, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * fia_prefill_mla: MLA prefill (npu_fused_infer_attention_score_v2, query D
 * not 512: "query, key, value D 128 with query_rope / key_rope D 64", or
 * "query, key D 192, value D 128").  The score of a pair is
 * scale_value * (q . k + q_rope . k_rope), the product over the 192-column
 * concatenation; value and attention_out have D 128.
 *   query / key: D 192 with query_rope = key_rope = NULL, or D 128 with both
 *          rope tensors given (the query's / key's shape with D 64, same type).
 *   value: key's shape with D 128.  attention_out: query's shape with D 128.
 *   Layouts BSH/BSND/BNSD/TND (the pages list TND), f16 or bf16, GQA allowed.
 *   sparse_mode 0 (with or without atten_mask), 1, 2, 3, 4 and atten_mask as
 *   fia_prefill.  softmax_lse as fia_prefill.
 * ------------------------------------------------------------------------ */
FIA_API fia_status fia_prefill_mla_get_workspace_size(const fia_tensor* query, const fia_tensor* key,
                                              const fia_tensor* value, const fia_tensor* query_rope,
                                              const fia_tensor* key_rope, const fia_tensor* atten_mask,
                                              const fia_params* params, const fia_tensor* attention_out,
                                              const fia_tensor* softmax_lse, size_t* workspace_bytes);
FIA_API fia_status fia_prefill_mla(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                           const fia_tensor* query_rope, const fia_tensor* key_rope, const fia_tensor* atten_mask,
                           const fia_params* params, const fia_tensor* attention_out, const fia_tensor* softmax_lse,
                           void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * fia_prefill_paged: fia_prefill with key/value in a paged cache (chunked
 * prefill: a chunk of new query tokens against a sequence's cached keys).
 *   npu_fused_infer_attention_score_v2, page attention: key j of batch b is
 *   row j % block_size of block block_table[b][j / block_size].
 *   query, atten_mask, sparse_mode (0..4), pre/next tokens, attention_out and
 *          softmax_lse as in fia_prefill (BSH/BSND/BNSD/TND query).
 *   key_cache, value_cache: device, same shape, the query's element type,
 *          (blocknum, KV_N, block_size, D) or (blocknum, block_size, KV_N*D).
 *   block_table: device int32 (B, >= maxBlockNumPerSeq); B = the query's batch
 *          (the number of sequences for TND).  Entries are not range-checked
 *          (the pages leave them to the caller); an id outside the pool reads
 *          as zeros.  NULL block_table = fia_prefill.
 *   params->block_size: 128..512, a multiple of 128; params->actual_seq_kvlen
 *          is required and holds each batch's key count (not cumulative,
 *          also for a TND query: the cache is not TND).
 *   blocknum must cover the blocks the lengths need (FIA_ERR_BLOCK_TABLE).
 * ------------------------------------------------------------------------ */
FIA_API fia_status fia_prefill_paged_get_workspace_size(const fia_tensor* query, const fia_tensor* key_cache,
                                                const fia_tensor* value_cache, const fia_tensor* block_table,
                                                const fia_tensor* atten_mask, const fia_params* params,
                                                const fia_tensor* attention_out, const fia_tensor* softmax_lse,
                                                size_t* workspace_bytes);
FIA_API fia_status fia_prefill_paged(const fia_tensor* query, const fia_tensor* key_cache, const fia_tensor* value_cache,
                             const fia_tensor* block_table, const fia_tensor* atten_mask, const fia_params* params,
                             const fia_tensor* attention_out, const fia_tensor* softmax_lse, void* workspace,
                             size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * fia_decode: incremental attention, Q_S new query tokens per batch.
 *   query  (B,N1,Q_S,D) BNSD | (B,Q_S,N1,D) BSND | (B,Q_S,H) BSH; f16 or bf16.
 *          Q_S = 1, or 2..16 with (N1 / N2) * Q_S <= 64 (not with MLA); then
 *          sparse_mode masks the Q_S x S_kv block as in the formula
 *          (npu_fused_infer_attention_score_v2, sparse_mode): 0 none, 2 key j
 *          <= token i, 3 key j <= i + S_kv - Q_S (the last token sees the whole
 *          cache); other modes return FIA_ERR_UNSUPPORTED.  With Q_S = 1
 *          sparse_mode is ignored, as on the pages.
 *   key/value, contiguous (block_table absent): the query's layout with N2 heads.
 *   key/value, paged (block_table present, PageAttention):
 *          (blocknum, N2, block_size, D)  or  (blocknum, block_size, N2*D);
 *          block_table int32 (B, >= max blocks per sequence); block ids are not
 *          validated (as on the pages); actual_seq_kvlen is required.
 *          block_size: a multiple of 16 that divides 128 or a multiple of 128.
 *   query_rope / key_rope (MLA): both or neither.  Then D = 512, D_rope = 64,
 *          N2 = 1, N1 in {1..128}, key = value = the 512-d latent cache
 *          (blocknum, block_size, 512), key_rope (blocknum, block_size, 64).
 *          scores = scale * (q . k + q_rope . k_rope).
 *   atten_mask: with Q_S = 1 (not MLA), bool / int8 / uint8 of shape (B, KV_S),
 *          (B, 1, KV_S) or (B, 1, 1, KV_S), batch dim B or 1 (broadcast),
 *          KV_S >= every actual_seq_kvlen, contiguous, device memory; a
 *          nonzero byte masks its key.  A row whose keys are all masked gets
 *          0 and softmax_lse +inf.  With Q_S > 1 or MLA it returns
 *          FIA_ERR_UNSUPPORTED.
 *   attention_out: the query's shape; softmax_lse fp32 (B,N1,Q_S,1) if flagged.
 * ------------------------------------------------------------------------ */
FIA_API fia_status fia_decode_get_workspace_size(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                         const fia_tensor* query_rope, const fia_tensor* key_rope,
                                         const fia_tensor* block_table, const fia_tensor* atten_mask,
                                         const fia_params* params, const fia_tensor* attention_out,
                                         const fia_tensor* softmax_lse, size_t* workspace_bytes);
FIA_API fia_status fia_decode(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                      const fia_tensor* query_rope, const fia_tensor* key_rope, const fia_tensor* block_table,
                      const fia_tensor* atten_mask, const fia_params* params, const fia_tensor* attention_out,
                      const fia_tensor* softmax_lse, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * fia_decode_no_alloc: fia_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart: it exists because some callers only
 * hold the input and output buffers they were given (plugin hosts, inference
 * servers that own the memory budget, code where a device allocation is not
 * allowed) and cannot create the workspace fia_decode takes.
 *   Arguments: as fia_decode, without the workspace.
 *   Scratch: a 16 MiB array built into the library (one per GPU that loads it,
 *          held until the process exits).  A call whose workspace need
 *          (fia_decode_get_workspace_size) exceeds 16 MiB returns
 *          FIA_ERR_WORKSPACE before touching the device.
 *   Set-up: every call looks up the array's device address in the calling
 *          thread's current CUDA context (the address belongs to a context:
 *          another context made current through the driver API, or a device
 *          reset, gives another one).  The first call in a context also loads
 *          the library's kernels there; make that first call before any
 *          stream capture.
 *   Sharing: every call uses the same array and leaves its contents behind.
 *          Calls that overlap on the GPU (other streams, other host threads)
 *          race on it; serialise them.  The device status word lives in the
 *          array and is not exposed: a device-side timeout of a call made
 *          through this entry point cannot be read back.
 *   Limit: MLA decode keeps two 256-wide partial outputs per query head and
 *          plan slot, so MLA calls with many query heads do not fit (128 heads
 *          never do, whatever the batch); they return FIA_ERR_WORKSPACE.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 * ------------------------------------------------------------------------ */
FIA_API fia_status fia_decode_no_alloc(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                       const fia_tensor* query_rope, const fia_tensor* key_rope,
                                       const fia_tensor* block_table, const fia_tensor* atten_mask,
                                       const fia_params* params, const fia_tensor* attention_out,
                                       const fia_tensor* softmax_lse, void* stream);

/* ------------------------------------------------------------------------
 * bsa_forward: block-sparse attention (aclnnBlockSparseAttentionV2).
 *   query/key/value: BNSD, BSND or TND (one layout for all three); f16/bf16;
 *          D in {64, 128}; N1 % N2 == 0.
 *   block_sparse_mask: u8/bool (B, N1, ceil(maxQS/X), ceil(maxKVS/Y));
 *          nonzero keeps the X x Y block.
 *   block_shape: {X, Y}; X > 0, Y a multiple of 128 (this library: X also a
 *          multiple of 128).
 *   actual_seq_qlen / actual_seq_kvlen: both or neither (TND: both).
 *   attention_out, softmax_lse: as for fia_prefill.
 * ------------------------------------------------------------------------ */
FIA_API fia_status bsa_get_workspace_size(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                  const fia_tensor* block_sparse_mask, const int64_t* block_shape,
                                  const fia_params* params, const fia_tensor* attention_out,
                                  const fia_tensor* softmax_lse, size_t* workspace_bytes);
FIA_API fia_status bsa_forward(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                       const fia_tensor* block_sparse_mask, const int64_t* block_shape, const fia_params* params,
                       const fia_tensor* attention_out, const fia_tensor* softmax_lse, void* workspace,
                       size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * bsa_forward_fp8: FP8 block-sparse attention (aclnnBlockSparseAttentionV2,
 * "FP8特性说明").  Row i of query head h is worth query[i] *
 * q_dequant_scale[b][h][i / 128]; key / value row j of kv head n is worth
 * key[j] * k_dequant_scale[b][n][j / Y] (value likewise).
 *   query/key/value: float8 e4m3 (FIA_DTYPE_F8E4M3), D = 128, layouts as
 *          bsa_forward.
 *   block_shape: {128, 256} or {128, 512} (the quantisation blocks).
 *   block_sparse_mask: as bsa_forward, or NULL: every block kept, which is
 *          dense (sparse_mode 0) FP8 prefill attention with the same scales.
 *   q_dequant_scale: fp32 (B, N1, ceil(maxQS/128), 1); k_dequant_scale and
 *          v_dequant_scale: fp32 (B, N2, ceil(maxKVS/Y), 1); device memory;
 *          every scale must be positive.  The scales are read on the device
 *          only: a scale <= 0 (or NaN) makes the kernel record
 *          FIA_ERR_UNSUPPORTED in the call's status word (fia_device_status),
 *          and the output of that call is unspecified.
 *   attention_out: bf16, the query's shape.  softmax_lse as bsa_forward.
 *   The scores run on the fp8 tensor cores (e4m3 x e4m3, fp32 accumulate).
 *   V is first rewritten into the workspace as f16 by a separate pass (one
 *   extra read of V and a write of twice its bytes); P V then runs on the
 *   f16 tensor-core path, with P scaled by the tile's value scale.
 * ------------------------------------------------------------------------ */
FIA_API fia_status bsa_fp8_get_workspace_size(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                      const fia_tensor* block_sparse_mask, const int64_t* block_shape,
                                      const fia_tensor* q_dequant_scale, const fia_tensor* k_dequant_scale,
                                      const fia_tensor* v_dequant_scale, const fia_params* params,
                                      const fia_tensor* attention_out, const fia_tensor* softmax_lse,
                                      size_t* workspace_bytes);
FIA_API fia_status bsa_forward_fp8(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                           const fia_tensor* block_sparse_mask, const int64_t* block_shape,
                           const fia_tensor* q_dequant_scale, const fia_tensor* k_dequant_scale,
                           const fia_tensor* v_dequant_scale, const fia_params* params,
                           const fia_tensor* attention_out, const fia_tensor* softmax_lse, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Waits for `stream`, then returns the device-side status recorded in a
 * workspace by the last call that used it (FIA_OK or FIA_ERR_TIMEOUT). */
FIA_API fia_status fia_device_status(const void* workspace, void* stream);

/* Static description of a status code. */
FIA_API const char* fia_status_string(fia_status s);

/* Human-readable detail of the last error returned on the calling thread. */
FIA_API const char* fia_last_error(void);

/* Profiling aid: the next fia_prefill / fia_decode / bsa_forward call made on
 * this thread records `start_event` just before its main attention kernel and
 * `stop_event` just after it, on that call's stream, so the caller can time the
 * kernel alone with cudaEventElapsedTime.  Both are cudaEvent_t created by the
 * caller (either may be NULL); the request is consumed by that one call. */
FIA_API void fia_profile_next_call(void* start_event, void* stop_event);

/* Testing aid for the device-side failure path (FIA-v2 / FIA-V5 constraints
 * list "aicore timeout or trap" among the operator's failures): every kernel
 * wait that can give up does so after `ns` nanoseconds instead of the default
 * 2 s, records FIA_ERR_TIMEOUT in the call's status word (fia_device_status),
 * lets its in-flight copies and products finish, frees its tensor memory and
 * returns.  Applies to calls launched afterwards from any thread; 0 restores
 * the default.  A limit far below a kernel's run time makes its calls fail:
 * meant only for tests of that path. */
FIA_API void fia_debug_set_wait_limit_ns(uint64_t ns);

/* Selects the decode kernel for units (batch, kv head) of at most 16 query
 * rows with head_dim 128: 0 (the default) the warp-level kernel (mma.sync per
 * warp), 1 the tcgen05 kernel that serves larger units.  Both compute the
 * same operation; applies to calls launched afterwards from any thread.
 * Meant for tests that compare the two. */
FIA_API void fia_debug_set_decode_path(int path);

/* Test hook, host only (no device work): the plan fia_decode deals for
 * per-batch lengths kv_len[0..B) (host memory) and N2 kv heads over at most
 * n_cta_max CTAs, with the same per-segment charge as fia_decode.  Writes
 * cta_seg[0..n_cta] (the first segment of each CTA, then the total),
 * segs[4 i .. 4 i + 3] = (unit, first 128-key stage, end stage, part) for each
 * segment in CTA order, unit_parts[2 u .. 2 u + 1] = (first part, parts) for
 * each unit u = b * N2 + kv head, and the counts.  Returns FIA_ERR_SHAPE if a
 * capacity is too small, FIA_ERR_NULL for a NULL pointer. */
FIA_API fia_status fia_debug_plan_decode(const int32_t* kv_len, int B, int N2, int n_cta_max, int32_t* cta_seg,
                                         int cta_seg_cap, int32_t* segs, int segs_cap, int32_t* unit_parts,
                                         int unit_parts_cap, int* n_cta, int* n_segs);

#ifdef __cplusplus
}
#endif

#endif /* FIA_H_ */
