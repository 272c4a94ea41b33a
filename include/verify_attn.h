/*
 * verify_attn.h - C ABI of the GB300 (sm_103a) target-verify attention library.
 *
 * The operation (sglang PR 36330 digest, "Motivation" and "Key code excerpts"):
 * speculative decoding's target-verify step runs a short multi-token query
 * (1-4 draft tokens per sequence, a GQA group of query heads per KV head,
 * head_dim 256) causally over a long paged KV cache (page size 16, FP8 E4M3
 * with per-tensor k/v descale, or BF16). The work of each (sequence, KV head)
 * is split across KV segments and the per-segment partial results are merged
 * by a log-sum-exp segment reduction (same digest, "Implementation breakdown"
 * item 1: the main kernel plus its "reduce segments" kernel).
 *
 * For sequence b with L = cu_seqlens_q[b+1] - cu_seqlens_q[b] draft tokens and
 * S = seqused_k[b] cached tokens (S counts the draft tokens too: the digest's
 * call passes seq_lens + max_q_len), query head h of draft token t reads KV
 * head h / (Hq/Hkv) and sees keys [0, S - L + t]:
 *
 *   out[cu[b]+t, h, :] = softmax(softmax_scale * k_descale * q . K^T) (v_descale * V)
 *
 * A row whose token sees no key (S - L + t < 0) is written as 0.
 *
 * Conventions shared by every entry point
 *  - Every tensor argument is a va_tensor: a DEVICE pointer plus shape and
 *    strides counted in elements. The library never keeps a pointer after the
 *    call returns and never frees caller memory.
 *  - Launches are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream). No entry point synchronises, reads device memory from
 *    the host, or depends on device values for its launch shape: only the
 *    host integers max_seqlen_q / max_seqlen_k (upper bounds) size the grid.
 *  - Errors are returned as va_status before anything is launched; nothing
 *    aborts or throws across the ABI. VA_ERR_CUDA reports a failed launch or
 *    allocation (the CUDA error is left for cudaGetLastError to inspect).
 *  - Device-side preconditions (seqused_k[b] <= block_table width * 16,
 *    0 <= cu_seqlens_q deltas <= max_seqlen_q, cu_seqlens_q[B] <= total_q,
 *    block-table entries < num_blocks) are the caller's. Violations never
 *    cause an out-of-bounds access (lengths are clamped, bad page ids read as
 *    zeros) but the affected output rows are unspecified.
 */
#ifndef VERIFY_ATTN_H
#define VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. FP8_E4M3 is OCP E4M3 "FN" (torch.float8_e4m3fn). */
typedef enum va_dtype {
  VA_BF16 = 0,
  VA_FP8_E4M3 = 1,
  VA_INT32 = 2,
  VA_FP32 = 3
} va_dtype;

/* A strided view of device memory. Strides are in elements. */
typedef struct va_tensor {
  void* data;
  int32_t dtype;      /* va_dtype */
  int32_t ndim;       /* 1..4 */
  int64_t shape[4];
  int64_t stride[4];
} va_tensor;

typedef enum va_status {
  VA_OK = 0,
  VA_ERR_NULL = 1,         /* a required pointer or descriptor is NULL */
  VA_ERR_SHAPE = 2,        /* shapes disagree with each other */
  VA_ERR_DTYPE = 3,        /* an element type is not the one required */
  VA_ERR_UNSUPPORTED = 4,  /* well-formed but outside what the kernels cover */
  VA_ERR_WORKSPACE = 5,    /* caller workspace missing or too small */
  VA_ERR_CUDA = 6,         /* a CUDA runtime call or launch failed */
  VA_ERR_LAYOUT = 7        /* a stride or alignment the kernels cannot read */
} va_status;

/* Launch plan chosen by the host heuristic (pure host arithmetic). */
typedef struct va_plan {
  int32_t tile_keys;       /* keys per pipeline tile of the main kernel */
  int32_t num_splits;      /* CTAs of the main kernel; each takes an equal share
                              of the batch's key tiles (its KV segments) */
  int32_t max_rows;        /* packed rows per (sequence, KV head) = G * max_seqlen_q */
  int32_t num_work;        /* B * Hkv (sequence, KV head) pairs */
  int32_t kernel;          /* main-kernel layout the launch will use: 1 = Q in
                              shared memory (BF16; FP8 batches of fewer than 16
                              tiles per CTA; any variant option), 2 = FP8 with
                              Q and P in tensor memory and a deeper K ring */
  int32_t reserved;
  int64_t workspace_bytes; /* scratch the split-KV partials need */
} va_plan;

/*
 * verify_attn - the operation described above.
 *
 * q            [total_q, Hq, 256] BF16; innermost stride 1, rows 16-byte aligned.
 * k_cache      [num_blocks, 16, Hkv, 256] FP8_E4M3 or BF16; innermost stride 1,
 * v_cache      the other strides multiples of 16 bytes. Same dtype and shape.
 *              Token-major pages with the heads of a token interleaved
 *              (sglang PR 36330 digest, unit test: key/value shape
 *              (num_blocks, block_size, num_kv_heads, head_size)).
 * block_table  [B, W] INT32, logical page -> physical page, W*16 >= max_seqlen_k.
 *              Only the first ceil(seqused_k[b]/16) entries of row b are read.
 * cu_seqlens_q [B+1] INT32 contiguous, prefix sums of the draft-token counts.
 * seqused_k    [B] INT32 contiguous, cached tokens per sequence incl. drafts.
 * max_seqlen_q host upper bound of the draft-token counts; 1 <= max_seqlen_q
 *              and (Hq/Hkv) * max_seqlen_q <= 64.
 * max_seqlen_k host upper bound of seqused_k (the digest passes
 *              page_table.shape[1] * page_size; sglang PR 30105 digest,
 *              "Key code excerpts").
 * softmax_scale  multiplies the logits (head_dim ** -0.5 in the pages).
 * k_descale, v_descale  [1] FP32 device scalars or NULL (= 1.0): the
 *              dequantised value is stored value * descale (sglang PR 34517
 *              digest, "Key code excerpts": qk *= sm_scale * k_scale).
 * out          [total_q, Hq, 256] BF16, written in place (round to nearest
 *              even from fp32); may not alias any input.
 * stream       cudaStream_t.
 *
 * Scratch: a per-device workspace owned by the library, grown (cudaMalloc) on
 * demand and kept until process exit. Because growing allocates, make the
 * first call with the largest shape before capturing a CUDA graph, or use
 * verify_attn_ex with a caller workspace. Calls that share the library
 * workspace must be ordered on one stream (concurrent streams race on it).
 * verify_attn_last_device_error(NULL, ...) reports a bounded wait that ran
 * out in a call made with it.
 */
va_status verify_attn(const va_tensor* q, const va_tensor* k_cache, const va_tensor* v_cache,
                      const va_tensor* block_table, const va_tensor* cu_seqlens_q,
                      const va_tensor* seqused_k, int32_t max_seqlen_q, int32_t max_seqlen_k,
                      float softmax_scale, const va_tensor* k_descale,
                      const va_tensor* v_descale, va_tensor* out, void* stream);

/*
 * verify_attn_ex - verify_attn with a caller-owned workspace and an optional
 * forced split count. Not on the pages: it exists so a caller can own all
 * memory (graph capture, allocator integration) and so tests can force the
 * number of KV segments.
 *
 * workspace        device pointer, 256-byte aligned, at least
 *                  verify_attn_workspace_size(...) bytes for the same shapes
 *                  and num_splits; NULL with workspace_bytes == 0 is valid only
 *                  when that size is 0.
 * num_splits       0 = the heuristic's choice; > 0 forces the main kernel's
 *                  CTA count (clamped to the number of key tiles it could have).
 * event_after_main NULL, or a cudaEvent_t recorded on `stream` between the
 *                  main and the merge kernel (lets a caller time the main
 *                  kernel alone with CUDA events on the launching stream).
 * The workspace holds no state between calls, except its status word (the
 * first 4 bytes; zero it before first use), which a bounded wait that runs out
 * sets and verify_attn_last_device_error reads and clears.
 */
va_status verify_attn_ex(const va_tensor* q, const va_tensor* k_cache, const va_tensor* v_cache,
                         const va_tensor* block_table, const va_tensor* cu_seqlens_q,
                         const va_tensor* seqused_k, int32_t max_seqlen_q, int32_t max_seqlen_k,
                         float softmax_scale, const va_tensor* k_descale,
                         const va_tensor* v_descale, va_tensor* out, void* workspace,
                         size_t workspace_bytes, int32_t num_splits, void* event_after_main,
                         void* stream);

/*
 * verify_attn_check - validation only: the same checks verify_attn runs before
 * launching, as a pure host function (no CUDA call; device pointers are only
 * tested for NULL and alignment). Turns the shape gate of sglang PR 36330
 * digest ("Key code excerpts", aiter_backend.py) and the rejections of sglang
 * PR 34517 digest ("Implementation breakdown": can_handle) into status codes.
 */
va_status verify_attn_check(const va_tensor* q, const va_tensor* k_cache, const va_tensor* v_cache,
                            const va_tensor* block_table, const va_tensor* cu_seqlens_q,
                            const va_tensor* seqused_k, int32_t max_seqlen_q,
                            int32_t max_seqlen_k, const va_tensor* k_descale,
                            const va_tensor* v_descale, const va_tensor* out);

/*
 * verify_attn_plan - the host launch heuristic as a pure function (no CUDA
 * call). Picks the tile size and the number of KV segments (main-kernel CTAs)
 * from the batch, the KV-length bound and the SM count, so that short-query
 * batches fill every SM (sglang PR 36330 digest, "Implementation breakdown"
 * item 1: 8-64 segments for CU parallelism; sglang PR 30105 digest,
 * "Implementation breakdown" item 3: split-KV restores occupancy for short
 * queries).
 *
 * num_sms        SMs of the target device (> 0).
 * force_splits   0 = heuristic; > 0 = this many (clamped as in verify_attn_ex).
 * Returns VA_ERR_NULL if plan is NULL, VA_ERR_UNSUPPORTED for arguments out
 * of range.
 */
va_status verify_attn_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads,
                           int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t kv_dtype,
                           int32_t num_sms, int32_t force_splits, va_plan* plan);

/*
 * verify_attn_workspace_size - bytes of workspace verify_attn_ex needs for
 * these shapes on the current device with num_splits (0 = heuristic). Queries
 * the current device's SM count (a CUDA call); returns 0 on error.
 */
size_t verify_attn_workspace_size(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads,
                                  int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t kv_dtype,
                                  int32_t num_splits);

/*
 * va_options - variants of the generic attention that the pages pass through
 * (sglang PR 30105 digest, "Key code excerpts": unified_attention(...,
 * window_size, softcap, sinks)). All off is window_left = -1, softcap = 0,
 * sinks = NULL.
 *  window_left  sliding window: the draft token at position i = S - L + t
 *               sees keys [i - window_left, i] (the pages' window_size =
 *               (sliding_window_size - 1, 0)); -1 = no window. Block-table
 *               pages holding only keys before every token's window are never
 *               read, so a sliding-window page table need not map them.
 *  softcap      > 0: each logit s = softmax_scale * k_descale * q.k becomes
 *               softcap * tanh(s / softcap) before masking; 0 = off.
 *  sinks        [Hq] fp32, contiguous, or NULL: a per-query-head logit
 *               (natural-log units) that joins that head's softmax normaliser
 *               with a zero value vector. A row that sees no key is still 0.
 */
typedef struct va_options {
  int32_t window_left;
  float softcap;
  const va_tensor* sinks;
} va_options;

/*
 * verify_attn_opt - verify_attn with the variants above.
 *  opts       NULL means all variants off (then this is verify_attn_ex).
 *  workspace  a caller workspace as for verify_attn_ex, or NULL to use the
 *             library's own per-device workspace as verify_attn does (which
 *             may then allocate, so not during stream capture).
 * Other arguments, layouts and results are those of verify_attn_ex; num_splits
 * 0 lets the heuristic pick (with a window it counts only the window's tiles).
 * Returns VA_ERR_SHAPE / VA_ERR_DTYPE / VA_ERR_NULL / VA_ERR_UNSUPPORTED for
 * bad options before launching (window_left < -1, softcap negative or not
 * finite, sinks not fp32 [Hq] contiguous).
 */
va_status verify_attn_opt(const va_tensor* q, const va_tensor* k_cache, const va_tensor* v_cache,
                          const va_tensor* block_table, const va_tensor* cu_seqlens_q,
                          const va_tensor* seqused_k, int32_t max_seqlen_q, int32_t max_seqlen_k,
                          float softmax_scale, const va_tensor* k_descale,
                          const va_tensor* v_descale, va_tensor* out, const va_options* opts,
                          void* workspace, size_t workspace_bytes, int32_t num_splits,
                          void* stream);

/*
 * verify_attn_noalloc - verify_attn for callers that cannot allocate device
 * memory. The pages have no counterpart; this is a library addition.
 *
 * Who needs it: code that must not call cudaMalloc when it runs attention,
 * e.g. a serving runtime that sized its GPU memory pool at start-up and
 * forbids later allocations (cudaMalloc synchronises the device and
 * fragments the pool), or an allocator callback that must not re-enter the
 * allocator. verify_attn would grow its workspace with cudaMalloc;
 * verify_attn_ex needs the caller to allocate one.
 *
 * Arguments, layouts, results and errors are those of verify_attn. The
 * split-KV partials go to a fixed array of VERIFY_ATTN_NOALLOC_SCRATCH_BYTES
 * compiled into the library; every GPU that loads the library holds that
 * array until the process exits. Nothing is allocated or freed by this call.
 *  - Returns VA_ERR_WORKSPACE, before launching anything, when the shapes
 *    need more partial storage than the array holds (it needs about
 *    (B*Hkv + SMs) * (Hq/Hkv) * max_seqlen_q KiB).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and keeps it; make
 *    that first call before any stream capture.
 *  - Every call on a device shares the one array and leaves its contents
 *    behind. Nothing in it needs to start at zero, but calls that overlap on
 *    the GPU (different streams, or different host threads) race on it:
 *    order them on one stream.
 *  - The array's first word is the status word of the kernels' bounded
 *    waits, shared by every call on the device. This call never clears it;
 *    verify_attn_last_device_error(NULL, ...) reads and clears it (and
 *    synchronises the stream it is given, so call it between batches).
 */
#define VERIFY_ATTN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

va_status verify_attn_noalloc(const va_tensor* q, const va_tensor* k_cache,
                              const va_tensor* v_cache, const va_tensor* block_table,
                              const va_tensor* cu_seqlens_q, const va_tensor* seqused_k,
                              int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                              const va_tensor* k_descale, const va_tensor* v_descale,
                              va_tensor* out, void* stream);

/*
 * verify_attn_block_table_from_indptr - the block table and KV lengths of a
 * batch given in flat token-slot form. This is the draft-extend pass of the
 * sglang PR 30105 digest ("Fix 2: draft_extend_v2 re-routed to
 * unified_attention"): it builds a 2D page table from its flat metadata, takes
 * each sequence's KV length as the difference of consecutive kv_indptr
 * entries, and then runs the same split-KV attention as target verify. After
 * this call, verify_attn on (block_table, seqused_k) with
 * max_seqlen_k = width * 16 is that attention.
 *
 * Arguments (all device memory, all int32):
 *  kv_indptr    [B+1], contiguous. Sequence b's tokens are kv_indices
 *               [kv_indptr[b], kv_indptr[b+1]).
 *  kv_indices   [nnz], contiguous. The KV-cache token slot of every token,
 *               slot = page * 16 + position in the page.
 *  block_table  [B, width], any non-negative strides; written. Entry p of
 *               row b is the page holding sequence b's tokens [16p, 16p + 16),
 *               i.e. the page of the first of those slots. Entries past the
 *               sequence's last page are set to pad_page.
 *  seqused_k    [B], any stride; written with kv_indptr[b+1] - kv_indptr[b].
 *  status       optional (NULL: not reported), one int32. The kernel ORs in:
 *                 1  a page's slots are not one page in order: the first slot
 *                    is not a multiple of 16, or the next ones are not
 *                    consecutive. The entry still names the first slot's page.
 *                 2  a sequence has more than width pages; its row keeps the
 *                    first width pages.
 *                 4  kv_indptr[b] is negative, decreases, or passes nnz; that
 *                    row is all pad_page and its length 0.
 *               The kernel never clears it.
 *
 * Behaviour:
 *  - One launch, asynchronous on stream.
 *  - Returns before launching: VA_ERR_NULL, VA_ERR_DTYPE, VA_ERR_SHAPE; VA_ERR_LAYOUT
 *    for a strided kv_indptr / kv_indices; VA_ERR_UNSUPPORTED for more than 65535
 *    sequences.
 *  - Returns VA_ERR_CUDA if the launch fails.
 */
va_status verify_attn_block_table_from_indptr(const va_tensor* kv_indptr,
                                              const va_tensor* kv_indices, va_tensor* block_table,
                                              va_tensor* seqused_k, int32_t pad_page,
                                              int32_t* status, void* stream);

/*
 * verify_attn_mla - target-verify attention over an absorbed-MLA latent cache.
 *
 * The grouped-head shared-KV verify kernel of the sglang PR 34517 digest
 * ("Implementation breakdown" item 1, the verify_mla.py excerpt) also serves
 * an absorbed-MLA layout: the single TP-local KV head is the MLA latent,
 * NOPE_DIM latent columns plus PE_DIM = 64 RoPE columns, and the logits are
 * (q_nope . k_nope + q_pe . k_pe) * softmax_scale * k_scale. The values are
 * the latent columns of the same cache rows. The latent width is not on the
 * pages; this library takes NOPE_DIM = 512 (the DeepSeek-V3 / Kimi-K2 MLA
 * family). For sequence b (L draft tokens, S = seqused_k[b]) and query head h
 * of draft token t, with cache row j = [c_j | r_j] (decoded e4m3 or bf16):
 *
 *   out[cu[b]+t, h, :] = sum_j softmax_j(softmax_scale * k_descale *
 *                          (q[.., :512] . c_j + q[.., 512:] . r_j)) * v_descale * c_j
 *
 * over keys j in [0, S - L + t]; a row that sees no key is 0.
 *
 * Arguments (device memory unless stated):
 *  q            [total_q, Hq, 576] bf16: [q_nope (absorbed, 512) | q_pe (64)].
 *  kv_cache     [num_blocks, 16, 1, 576] FP8 E4M3 (OCP FN) or BF16: [latent |
 *               rope key] (the digest's tests cover both cache types, same
 *               digest, "Implementation breakdown" item 4).
 *  block_table, cu_seqlens_q, seqused_k, max_seqlen_q, max_seqlen_k,
 *  softmax_scale, k_descale, v_descale: as for verify_attn (Hkv = 1, so the
 *               group is Hq and Hq * max_seqlen_q <= 64). A cache with one
 *               scale passes it as both descales.
 *  out          [total_q, Hq, 512] bf16, written.
 *  workspace    device memory of at least verify_attn_mla_workspace_size()
 *               bytes, 256-byte aligned; NULL uses the library's per-device
 *               workspace (grown with cudaMalloc as needed).
 *  num_splits   0 = the library's choice (one CTA per SM, fewer for small
 *               batches); > 0 forces that many CTAs.
 *  event_after_main  optional cudaEvent_t (NULL: none) recorded on stream
 *               between the main kernel and the merge kernel, as in
 *               verify_attn_ex.
 *
 * Layout: innermost strides 1 and every other stride a multiple of 16 bytes;
 * q, out, kv_cache 16-byte aligned.
 * Errors (before any launch): VA_ERR_NULL, VA_ERR_SHAPE, VA_ERR_DTYPE,
 * VA_ERR_LAYOUT as for verify_attn (VA_ERR_DTYPE for a cache that is neither
 * FP8 E4M3 nor BF16); VA_ERR_UNSUPPORTED for more than one KV head, other row
 * widths or Hq * max_seqlen_q > 64;
 * VA_ERR_WORKSPACE for a short or misaligned workspace; VA_ERR_CUDA for a
 * failed launch or allocation. Device-side timeouts set the workspace
 * status word as for verify_attn_ex.
 */
va_status verify_attn_mla(const va_tensor* q, const va_tensor* kv_cache, const va_tensor* block_table,
                          const va_tensor* cu_seqlens_q, const va_tensor* seqused_k,
                          int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                          const va_tensor* k_descale, const va_tensor* v_descale, va_tensor* out,
                          void* workspace, size_t workspace_bytes, int32_t num_splits,
                          void* event_after_main, void* stream);

/* Workspace bytes verify_attn_mla needs for these shapes on the current
 * device, for either cache type (0 if they are unsupported). */
size_t verify_attn_mla_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t max_seqlen_q,
                                      int32_t max_seqlen_k, int32_t num_splits);

/*
 * verify_attn_partial - verify attention over one shard of each sequence's
 * keys, for splitting a sequence's KV over several parts (context
 * parallelism across ranks; a shared prefix in one cache and per-sequence
 * suffixes in another). The pages name a decode-context-parallel degree
 * (sglang PR 34517 digest, attn_dcp_size) and merge split-KV segments by log-sum-exp
 * (sglang PR 36330 digest, "reduce segments"); this entry computes one
 * shard's result and verify_attn_merge_partials combines shards. The
 * exchange of shard results between GPUs is the caller's.
 *
 * A shard holds the keys of global positions [o_b, o_b + S_b) of sequence b,
 * reached through its own block_table row (S_b = seqused_k[b]). With
 * E_b = kv_extent[b] = (the sequence's total keys) - o_b, draft token t of L
 * sees the shard's local keys j <= E_b - L + t (and j < S_b). NULL kv_extent
 * means E_b = S_b, the last shard (or the whole sequence).
 *
 * Arguments as verify_attn_ex, except:
 *  kv_extent  [B] int32 (nullable), contiguous; values below S_b count as S_b.
 *  o          [total_q, Hq, 256] fp32, written: the shard's attention output,
 *             normalised over the shard's visible keys, times v_descale.
 *  lse        [total_q, Hq] fp32, written: ln(sum over the visible keys of
 *             exp(softmax_scale * k_descale * q . k)); -inf (and o = 0) for a
 *             row that sees no key of the shard.
 *  workspace  as verify_attn_ex; NULL uses the library's per-device workspace.
 * The variants of verify_attn_opt are not available here. Errors as
 * verify_attn_ex (o and lse: VA_ERR_DTYPE unless fp32, VA_ERR_SHAPE, and
 * VA_ERR_LAYOUT for o rows that are not 16-byte aligned).
 */
va_status verify_attn_partial(const va_tensor* q, const va_tensor* k_cache, const va_tensor* v_cache,
                              const va_tensor* block_table, const va_tensor* cu_seqlens_q,
                              const va_tensor* seqused_k, const va_tensor* kv_extent,
                              int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                              const va_tensor* k_descale, const va_tensor* v_descale, va_tensor* o,
                              va_tensor* lse, void* workspace, size_t workspace_bytes,
                              int32_t num_splits, void* stream);

/*
 * verify_attn_merge_partials - combines n (1..16) shard results of
 * verify_attn_partial: out = sum_i exp(lse_i - LSE) o_i with
 * LSE = ln sum_i exp(lse_i), rounded to bf16; a row whose lse are all -inf
 * is 0. o_parts and lse_parts are HOST arrays of n descriptors (fp32
 * [total_q, Hq, 256] and [total_q, Hq], device memory); out is bf16
 * [total_q, Hq, 256]. One launch on stream. Returns VA_ERR_UNSUPPORTED for n
 * outside 1..16, and the usual shape / dtype / layout errors.
 */
va_status verify_attn_merge_partials(int32_t n, const va_tensor* o_parts, const va_tensor* lse_parts,
                                     va_tensor* out, void* stream);

/*
 * verify_attn_last_device_error - reads and clears the device status word of
 * a workspace. This turns the pages' gates and asserts (sglang PR 36330 digest,
 * "Key code excerpts") into something a caller can check after launch: a
 * condition found on the device, when no host check could see it.
 *
 * Every wait of the main kernels (a ring slot, a TMA copy landing, an MMA
 * finishing) is bounded in time (2 s unless verify_attn_set_wait_limit says
 * otherwise). A wait that runs out makes the kernel stop issuing work, let
 * its copies and MMAs in flight finish, free its tensor memory and return;
 * it ORs a nonzero code into the status word of the call's workspace. The
 * outputs of that call are then unspecified. The status word is sticky:
 * kernels only ever set bits in it.
 *
 *  workspace  the 256-byte-aligned workspace pointer that was passed to
 *             verify_attn_ex, verify_attn_opt, verify_attn_mla or
 *             verify_attn_partial; or NULL for the library's own scratch on
 *             the current device: the workspace of calls made without one
 *             (verify_attn, and the others with a NULL workspace) and the
 *             built-in array of verify_attn_noalloc. The library's workspace
 *             is replaced when it grows; its word then starts at 0 again.
 *  bits       host int32, written: the OR of the words read (0 = no bounded
 *             wait ran out since the last read and clear). Nonzero bits name
 *             the wait that gave up; they are diagnostic, not an API.
 *  stream     the words are read after the work queued on `stream` (this
 *             call synchronises it), then cleared on it. Calls on other
 *             streams that use the same scratch must be ordered by the caller.
 * Returns VA_ERR_NULL for a NULL bits, VA_ERR_WORKSPACE for a misaligned
 * workspace, VA_ERR_CUDA if a copy or the synchronisation fails.
 */
va_status verify_attn_last_device_error(const void* workspace, int32_t* bits, void* stream);

/*
 * verify_attn_set_wait_limit - the time limit, in nanoseconds, of the main
 * kernels' bounded waits for launches made after this call, process-wide; 0
 * restores the default of 2 s. A hook for tests of the timeout path: a limit
 * of a few nanoseconds makes waits run out on any input, so that a test can
 * check that the call still returns, the status word is set and the next
 * call is correct. Not for production use (any limit shorter than the
 * kernels' normal waits makes every call fail). Always returns VA_OK.
 */
va_status verify_attn_set_wait_limit(uint64_t limit_ns);

/* Static, NUL-terminated name of a status code. */
const char* verify_attn_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_H */
