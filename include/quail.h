/*
 * quail.h - C ABI of libquail, the GB300 (sm_103a) hot path of Quail's prefill-only
 * AI_JOIN / AI.IF forward step: simplified cascade attention and the 8-column restricted
 * head.
 *
 * Sources (page titles and sections; the pages print no equations):
 *   [P1] "Motor de inferência Quail atinge 1 bilhão de tokens por minuto por GPU",
 *        section "Como funciona": zero-decode bullet and simplified-cascade-attention
 *        bullet.
 *   [P2] "Quail: یک میلیارد توکن در دقیقه روی یک GPU": the AI.IF join example and the
 *        key-points list (qwen3-4b-fp8 on one GPU; head limited to 8 output tokens).
 *
 * Conventions for every call:
 *   - Every pointer is DEVICE memory owned by the caller; the library never allocates or
 *     frees memory in these calls and keeps no pointer after a call returns.
 *   - Work is enqueued asynchronously on `stream` (NULL = the legacy default stream).
 *   - Argument errors are found on the host and returned synchronously; nothing is
 *     launched then. They cover NULL pointers, head counts, head_dim, dtypes and scales,
 *     16-byte alignment, and element counts that overflow 64-bit offsets.
 *   - Offset arrays are read on the device. A scheduling kernel checks that they are
 *     monotone and agree with the totals and maxima of the descriptor; if not, no
 *     attention work runs and quail_get_device_error() reports QUAIL_ERR_DEVICE_BOUNDS.
 *   - Every wait inside a kernel is bounded; a wait that runs out sets a device error
 *     word (QUAIL_ERR_TIMEOUT) and the kernel returns cleanly.
 *   - No C++ exception or device trap crosses this boundary.
 *   - The library runs on compute capability 10.3 (GB300) only; elsewhere calls return
 *     QUAIL_ERR_UNSUPPORTED.
 */
#ifndef QUAIL_H_
#define QUAIL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* quail_stream_t;

typedef enum {
  QUAIL_OK = 0,
  QUAIL_ERR_INVALID_ARG = 1,   /* bad argument, found on the host */
  QUAIL_ERR_UNSUPPORTED = 2,   /* valid but not supported (head_dim, GQA ratio, device) */
  QUAIL_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  QUAIL_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out */
  QUAIL_ERR_DEVICE_BOUNDS = 5  /* offsets on the device disagree with the descriptor */
} quail_status;

typedef enum { QUAIL_BF16 = 0, QUAIL_FP8_E4M3 = 1 } quail_dtype;

/*
 * Shape of one ragged cascade-attention batch. A = anchors, S = suffixes, T_A / T_S =
 * total anchor / suffix tokens; query head h reads KV head h / (Hq / Hkv).
 */
typedef struct {
  int32_t num_anchors;           /* A >= 0 */
  int32_t num_suffixes;          /* S >= 0 */
  int64_t total_anchor_tokens;   /* T_A = anchor_offsets[A], known on the host (no sync) */
  int64_t total_suffix_tokens;   /* T_S = suffix_offsets[S] */
  int32_t max_anchor_len;        /* >= every anchor length */
  int32_t max_suffix_len;        /* >= every suffix length */
  int32_t num_q_heads;           /* Hq, a multiple of Hkv */
  int32_t num_kv_heads;          /* Hkv */
  int32_t head_dim;              /* d: 64 or 128 */
  float softmax_scale;           /* 0 => 1/sqrt(d) */
  int32_t kv_anchor_dtype;       /* quail_dtype of k_anc/v_anc */
} quail_cascade_desc;

/*
 * Simplified cascade attention ([P1] "Como funciona", cascade-attention bullet): every
 * token of a suffix attends non-causally to all tokens of its anchor (cross-attention)
 * and causally to its own suffix's tokens up to itself; the two softmax partials are
 * combined by LSE rescaling. The result equals softmax attention over the concatenated
 * prompt [anchor ; suffix] of [P2]'s AI.IF example, restricted to the suffix rows.
 *
 *   q_suf   [T_S, Hq, d]   bf16, post-RoPE suffix queries
 *   k_anc, v_anc [T_A, Hkv, d]  bf16, or e4m3 codes when kv_anchor_dtype = FP8_E4M3
 *   k_suf, v_suf [T_S, Hkv, d]  bf16
 *   anchor_offsets    [A+1] int32 token prefix sums into k_anc/v_anc
 *   anchor_suffix_ptr [A+1] int32: the suffixes of anchor a are
 *                     anchor_suffix_ptr[a] .. anchor_suffix_ptr[a+1]-1 (contiguous)
 *   suffix_offsets    [S+1] int32 token prefix sums into q_suf/k_suf/v_suf/out/lse
 *   k_scale, v_scale  [A, Hkv] fp32 dequantisation scales (value = e4m3(code) * scale);
 *                     required for FP8_E4M3, must be NULL for BF16
 *   out     [T_S, Hq, d] bf16 (round to nearest even from fp32), 32-byte aligned
 *   lse     [T_S, Hq] fp32 natural log of the sum of exp(scaled scores); may be NULL
 *   workspace: device scratch of at least quail_cascade_workspace_size(desc) bytes,
 *              16-byte aligned; its contents are overwritten. Calls that share one
 *              workspace must not overlap on the GPU. With FP8_E4M3 it also holds the
 *              anchor codes widened to bf16 (exact), 4 * T_A * Hkv * d bytes, which
 *              the attention reads in place of the codes.
 * Empty inputs are legal (S = 0, anchors without suffixes, L_a = 0 where lse of the
 * anchor part is -inf). Supported: d in {64, 128}, Hq/Hkv in {1, 2, 4, 8, 16}.
 */
quail_status quail_cascade_attn(const quail_cascade_desc* desc, const void* q_suf,
                                const void* k_anc, const void* v_anc, const void* k_suf,
                                const void* v_suf, const int32_t* anchor_offsets,
                                const int32_t* anchor_suffix_ptr,
                                const int32_t* suffix_offsets, const float* k_scale,
                                const float* v_scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes,
                                quail_stream_t stream);

/* Workspace bytes that quail_cascade_attn needs for `desc` (0 when desc is NULL). */
size_t quail_cascade_workspace_size(const quail_cascade_desc* desc);

/*
 * The same result as quail_cascade_attn computed as two passes and a merge, the three
 * steps of [P1]'s cascade-attention bullet run apart: (A2) an anchor pass - every suffix
 * token against its anchor's keys only - writes the normalised fp32 partial O_a and its
 * lse_a into the workspace; (A3) a suffix pass attends causally over the suffix's own
 * keys; (A4) the LSE merge lse = log(e^lse_a + e^lse_s), out = e^(lse_a - lse) O_a +
 * e^(lse_s - lse) O_s, done in the suffix pass's epilogue (merge_in_suffix_pass = 1) or by
 * a separate merge kernel over out in place (0; the suffix pass then writes O_s to out in
 * bf16 and lse_s to the workspace). It exists to compare with the fused kernel by
 * measurement; results agree with quail_cascade_attn within the bf16 bounds, not bit for
 * bit (O_s or the merge add a rounding).
 *
 * Arguments, layouts, limits and errors as quail_cascade_attn, plus merge_in_suffix_pass
 * (0 or 1) and a workspace of at least quail_cascade_two_pass_workspace_size(desc) bytes
 * (the cascade's workspace + 4 * T_S * Hq * (d + 2) bytes), 16-byte aligned.
 */
quail_status quail_cascade_attn_two_pass(const quail_cascade_desc* desc, const void* q_suf,
                                         const void* k_anc, const void* v_anc,
                                         const void* k_suf, const void* v_suf,
                                         const int32_t* anchor_offsets,
                                         const int32_t* anchor_suffix_ptr,
                                         const int32_t* suffix_offsets, const float* k_scale,
                                         const float* v_scale, int32_t merge_in_suffix_pass,
                                         void* out, float* lse, void* workspace,
                                         size_t workspace_bytes, quail_stream_t stream);

/* Workspace bytes that quail_cascade_attn_two_pass needs for `desc` (0 when invalid). */
size_t quail_cascade_two_pass_workspace_size(const quail_cascade_desc* desc);

/*
 * Causal self-attention over packed sequences: the anchors' own prefill, the step before
 * the cascade ([P1] "Como funciona", cascade-attention bullet: the shared anchor is
 * processed once and its KV reused by every suffix). For sequence s, token i and q-head h
 * (KV head h / (Hq/Hkv)): softmax attention over keys 0..i of the same sequence, i.e.
 * quail_cascade_attn with one anchor of length 0 whose suffixes are the sequences; the
 * same kernels run.
 *
 *   q [T, Hq, d], k, v [T, Hkv, d]  bf16 (post-RoPE)
 *   seq_offsets [S+1] int32 token prefix sums (monotone, seq_offsets[S] == T, every
 *                    length <= max_seq_len; checked on the device as for the cascade)
 *   out [T, Hq, d] bf16, 32-byte aligned; lse [T, Hq] fp32 natural log, may be NULL
 *   k_amax, v_amax [S, Hkv] fp32 out, both NULL or both given: max |k| and max |v| over
 *                    each sequence's tokens and all d, per KV head - the inputs of
 *                    quail_quantize_kv_fp8_with_scales. They come from the K/V tiles the
 *                    attention already loads (no extra read of k and v).
 *   softmax_scale: 0 => 1/sqrt(d)
 *   workspace: at least quail_causal_prefill_workspace_size(...) bytes, 256-byte aligned;
 *              overwritten (the call writes two 2-entry index arrays at its start).
 * Errors and limits as quail_cascade_attn (d in {64, 128}, Hq/Hkv in {1, 2, 4, 8, 16}).
 */
quail_status quail_causal_prefill_attn(int32_t num_seqs, int64_t total_tokens,
                                       int32_t max_seq_len, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim,
                                       float softmax_scale, const void* q, const void* k,
                                       const void* v, const int32_t* seq_offsets, void* out,
                                       float* lse, float* k_amax, float* v_amax,
                                       void* workspace, size_t workspace_bytes,
                                       quail_stream_t stream);

/* Workspace bytes for quail_causal_prefill_attn (0 if the sizes are invalid). */
size_t quail_causal_prefill_workspace_size(int32_t num_seqs, int64_t total_tokens,
                                           int32_t max_seq_len, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim);

/*
 * Query-aware anchor-KV cache plan ([P1] "Como funciona", first bullet: the whole query
 * plan is known in advance, so KV can be evicted without regret; the KV-regret paragraph of
 * "Quail, il motore di inferenza che supera il miliardo di token al minuto su una H100").
 * HOST call on HOST memory (the one exception to the device-pointer rule; no GPU work).
 *
 *   anchor_tokens [num_anchors] KV size of each anchor in tokens (>= 0)
 *   access_anchor [num_accesses] the plan's anchor accesses in execution order (0..A-1)
 *   capacity_tokens  tokens of anchor KV the GPU may hold
 *   policy       QUAIL_KV_LRU (oldest last access is evicted; always inserts) or
 *                QUAIL_KV_FURTHEST_NEXT_USE (the resident - or the incoming anchor, which
 *                is then bypassed - whose next access is furthest; ties: larger size, then
 *                larger id)
 *   hit          [num_accesses] out: 1 = the anchor's KV was resident; may be NULL
 *   stats        out: hits, misses, compulsory tokens (first prefill of each anchor),
 *                regret tokens (prefilled again after an eviction or bypass), peak
 *                resident tokens. An anchor larger than the capacity is never resident.
 * Errors: QUAIL_ERR_INVALID_ARG for negative counts or sizes, ids out of range, NULL
 * inputs with nonzero counts, NULL stats or an unknown policy.
 */
typedef enum { QUAIL_KV_LRU = 0, QUAIL_KV_FURTHEST_NEXT_USE = 1 } quail_kv_policy;
typedef struct {
  int64_t hits, misses;
  int64_t compulsory_tokens, regret_tokens;
  int64_t peak_resident_tokens;
} quail_kv_plan_stats;
quail_status quail_kv_plan(int32_t num_anchors, const int64_t* anchor_tokens,
                           int64_t num_accesses, const int32_t* access_anchor,
                           int64_t capacity_tokens, int32_t policy, uint8_t* hit,
                           quail_kv_plan_stats* stats);

/*
 * Join verdicts from the head's argmax ([P1] "Como funciona": a boolean AI.IF needs only
 * the one token of the last prefill pass, one of 8 options; [P2]'s AI_JOIN keeps the
 * pairs for which it holds). Suffix s (one anchor-candidate pair) passes when
 * argmax[s] == true_index. Device memory, asynchronous on `stream`.
 *
 *   anchor_suffix_ptr [A+1] int32: suffixes of anchor a are [ptr[a], ptr[a+1]); needed
 *                     only with anchor_count
 *   argmax    [S] int32, the restricted head's output for the last token of each suffix
 *   true_index        the option (0..7) that stands for "true"
 *   verdict   [S] uint8 out (1 = passes); may be NULL
 *   selected  [S] int32 out: the passing suffix ids in increasing order (anchor-major);
 *             entries past *num_selected are left as they were
 *   num_selected [1] int32 out (device)
 *   anchor_count [A] int32 out: passing suffixes per anchor; may be NULL
 *   workspace  >= quail_join_select_workspace_size(S) bytes, 16-byte aligned
 * Errors: QUAIL_ERR_INVALID_ARG for negative counts, true_index outside 0..7, NULL or
 * misaligned (4-byte) arrays that the call needs, or a short workspace.
 */
size_t quail_join_select_workspace_size(int32_t num_suffixes);
quail_status quail_join_select(int32_t num_anchors, int32_t num_suffixes,
                               const int32_t* anchor_suffix_ptr, const int32_t* argmax,
                               int32_t true_index, uint8_t* verdict, int32_t* selected,
                               int32_t* num_selected, int32_t* anchor_count, void* workspace,
                               size_t workspace_bytes, quail_stream_t stream);

/*
 * Sharding one batch over ranks by anchor ([P1] "Como funciona", cascade-attention
 * bullet: a suffix attends only to its own anchor and to itself, so an anchor with its
 * suffixes is an independent unit and ranks exchange no data). HOST call on HOST memory
 * (no GPU work).
 *
 *   anchor_offsets [A+1], anchor_suffix_ptr [A+1] (anchor_suffix_ptr[0] == 0),
 *   suffix_offsets [S+1] (S = anchor_suffix_ptr[A]): int32, as for quail_cascade_attn;
 *                  only differences are used, each must be >= 0
 *   num_ranks      >= 1
 *   rank_of_anchor [A] out: the rank that computes anchor a and all its suffixes
 *   rank_pairs     [num_ranks] out (may be NULL): visible (query, key) pairs per rank
 * Work of an anchor = sum over its suffixes of l_s L_a + l_s (l_s + 1) / 2 (attention
 * FLOPs / (4 d Hq)). Assignment: longest processing time first - anchors by decreasing
 * work (ties: lower index), each to the least-loaded rank (ties: lower rank); its largest
 * rank load is at most (4/3 - 1/(3 num_ranks)) times the best possible.
 * Errors: QUAIL_ERR_INVALID_ARG for negative counts or lengths, num_ranks < 1, NULL
 * arrays, or anchor_suffix_ptr[0] != 0.
 */
quail_status quail_shard_anchors(int32_t num_anchors, const int32_t* anchor_offsets,
                                 const int32_t* anchor_suffix_ptr,
                                 const int32_t* suffix_offsets, int32_t num_ranks,
                                 int32_t* rank_of_anchor, int64_t* rank_pairs);

/*
 * One rank's sub-batch of a batch split by quail_shard_anchors. HOST call on HOST memory
 * (no GPU work). The rank's anchors, in their original order, each with all of its
 * suffixes, as a batch that quail_cascade_attn takes, plus the rows of the full batch's
 * tensors that the sub-batch reads and writes.
 *
 *   anchor_offsets [A+1], anchor_suffix_ptr [A+1] (anchor_suffix_ptr[0] == 0),
 *   suffix_offsets [S+1]: int32, as for quail_cascade_attn (lengths >= 0)
 *   rank_of_anchor [A] int32, e.g. from quail_shard_anchors; rank >= 0
 *   sizes     out (always written): the sub-batch's anchors, suffixes, anchor tokens and
 *             suffix tokens
 *   The six arrays below are either all NULL (size query) or all given, sized from
 *   `sizes`:
 *   sub_anchor_offsets [A_r+1], sub_anchor_suffix_ptr [A_r+1], sub_suffix_offsets [S_r+1]
 *             int32 out: the sub-batch's offsets (prefix sums from 0)
 *   anchors     [A_r] int32 out: full-batch index of each kept anchor
 *   anchor_rows [T_A,r] int64 out: rows of k_anc / v_anc, in sub-batch order
 *   suffix_rows [T_S,r] int64 out: rows of q_suf / k_suf / v_suf (and of out / lse)
 * Errors: QUAIL_ERR_INVALID_ARG for negative counts or lengths, NULL inputs or sizes, some
 * but not all output arrays, or anchor_suffix_ptr[0] != 0; QUAIL_ERR_UNSUPPORTED when a
 * sub-batch token count exceeds int32 offsets.
 */
typedef struct {
  int32_t num_anchors, num_suffixes;
  int64_t anchor_tokens, suffix_tokens;
} quail_shard_sizes;
quail_status quail_shard_batch(int32_t num_anchors, const int32_t* anchor_offsets,
                               const int32_t* anchor_suffix_ptr, const int32_t* suffix_offsets,
                               const int32_t* rank_of_anchor, int32_t rank,
                               quail_shard_sizes* sizes, int32_t* sub_anchor_offsets,
                               int32_t* sub_anchor_suffix_ptr, int32_t* sub_suffix_offsets,
                               int32_t* anchors, int64_t* anchor_rows, int64_t* suffix_rows);

/* Size of the library's fixed device scratch array used by quail_cascade_attn_noalloc. */
#define QUAIL_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * quail_cascade_attn without a caller workspace (no counterpart on the pages: it exists
 * for callers that must not allocate device memory - e.g. an engine whose device memory
 * is fixed at start-up, or a plugin host that only passes input and output buffers).
 * Same arguments, meaning, layouts and checks as quail_cascade_attn, minus `workspace`.
 * The scratch lives in one file-scope device array of QUAIL_NOALLOC_SCRATCH_BYTES, held
 * on every GPU that loads the library until the process exits. This call allocates
 * nothing (no cudaMalloc/cudaFree, no allocating library routine).
 *   - Returns QUAIL_ERR_UNSUPPORTED when quail_cascade_workspace_size(desc) exceeds
 *     QUAIL_NOALLOC_SCRATCH_BYTES.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   - Every call uses the same array. Calls whose GPU work overlaps (unordered streams or
 *     threads) race on it and produce wrong results; order them on one stream.
 */
quail_status quail_cascade_attn_noalloc(const quail_cascade_desc* desc, const void* q_suf,
                                        const void* k_anc, const void* v_anc,
                                        const void* k_suf, const void* v_suf,
                                        const int32_t* anchor_offsets,
                                        const int32_t* anchor_suffix_ptr,
                                        const int32_t* suffix_offsets, const float* k_scale,
                                        const float* v_scale, void* out, float* lse,
                                        quail_stream_t stream);

/*
 * Restricted head of the zero-decode step ([P1] "Como funciona": the final prefill pass
 * emits one token and the output vocabulary is cut to 8 options, shrinking the final
 * unembedding matrix; [P2] key points: the head is limited to 8 output tokens). For
 * each output row n with source row r = row_index ? row_index[n] : n:
 *   y = h[r] * rsqrt(mean(h[r]^2) + eps) * gamma          (RMSNorm, fp32 accumulation)
 *   logits[n, j] = sum_k y_k * w8[j, k], j < 8;  argmax[n] = lowest j with the max logit
 *
 *   h        bf16 rows of `hidden` elements, row r at h + r * h_row_stride elements;
 *            h_row_stride >= hidden, (h_row_stride * 2) % 16 == 0
 *   h_rows   number of rows of h (>= 0); without row_index, n_rows <= h_rows
 *   row_index int32 [n_rows] source rows (e.g. the last token of each suffix), or NULL.
 *            Checked on the device: an index outside [0, h_rows) reads nothing, its row
 *            gets NaN logits and argmax -1, and quail_get_device_error() then reports
 *            QUAIL_ERR_DEVICE_BOUNDS.
 *   gamma    bf16 [hidden]; w8 bf16 [8, hidden] row-major
 *   logits   fp32 [n_rows, 8]; argmax int32 [n_rows]
 * hidden must be a positive multiple of 32 and at most 6144. n_rows may be 0.
 */
quail_status quail_restricted_head(int64_t n_rows, int32_t hidden, float eps, const void* h,
                                   int64_t h_rows, int64_t h_row_stride,
                                   const int32_t* row_index, const void* gamma, const void* w8,
                                   float* logits, int32_t* argmax, quail_stream_t stream);

/*
 * Per-(anchor, KV head) E4M3 quantisation of anchor K or V (the FP8 KV of the
 * qwen3-4b-fp8 model named in [P2]'s key points). For anchor a and KV head g:
 *   scale[a, g] = amax / 448 in fp32 (1 when amax == 0), amax over the anchor's tokens
 *   and all d; code = e4m3(x / scale), x / scale rounded to fp32 first, then rounded to
 *   nearest even with saturation at +-448 (sign kept).
 *   kv_bf16 [T_A, Hkv, d] bf16 in; kv_e4m3 [T_A, Hkv, d] codes out; scale [A, Hkv] fp32
 *   out. d in {64, 128}, Hkv * d <= 4096. One kernel on `stream` (clusters of 8 CTAs
 *   holding each (anchor, KV head) slab on chip: one read of kv_bf16 for anchors up to
 *   4,096 tokens at 256-byte token rows per slab, two reads above). Offsets are clamped into
 *   [0, T_A] on the device, so inconsistent ones cannot address outside the tensors.
 */
quail_status quail_quantize_kv_fp8(int32_t num_anchors, const int32_t* anchor_offsets,
                                   int64_t total_anchor_tokens, int32_t num_kv_heads,
                                   int32_t head_dim, const void* kv_bf16, void* kv_e4m3,
                                   float* scale, quail_stream_t stream);

/*
 * The same codes and scales as quail_quantize_kv_fp8 when the max |x| of every (anchor,
 * KV head) is already known - e.g. the k_amax / v_amax that quail_causal_prefill_attn
 * emits while it streams the anchors' K/V ([P1] "Como funciona": the anchor is prefilled
 * once and its KV reused), so quantising costs one read of kv_bf16 and one write.
 *   amax [A, Hkv] fp32 (device); scale[a, g] = amax[a, g] / 448 (1 when 0) is written.
 * Other arguments, limits and errors as quail_quantize_kv_fp8 (plus NULL or misaligned
 * amax -> QUAIL_ERR_INVALID_ARG). The anchors' offsets must be monotone (each token row
 * takes the scale of the anchor holding it).
 */
quail_status quail_quantize_kv_fp8_with_scales(int32_t num_anchors,
                                               const int32_t* anchor_offsets,
                                               int64_t total_anchor_tokens,
                                               int32_t num_kv_heads, int32_t head_dim,
                                               const void* kv_bf16, const float* amax,
                                               void* kv_e4m3, float* scale,
                                               quail_stream_t stream);

/* Static, NUL-terminated name of a status code. */
const char* quail_status_string(quail_status status);

/*
 * Synchronises `stream`, then reads and clears the library's device error word for the
 * current device: QUAIL_OK, QUAIL_ERR_TIMEOUT or QUAIL_ERR_DEVICE_BOUNDS (or
 * QUAIL_ERR_CUDA if the synchronisation itself failed).
 */
quail_status quail_get_device_error(quail_stream_t stream);

/*
 * Limit of every bounded device-side wait, in nanoseconds of GPU global time (default
 * 2e9). Applies to launches made after the call. 0 restores the default.
 */
void quail_set_wait_timeout_ns(uint64_t ns);

/*
 * Host-side fault injection for the timeout tests: with `skip_first_kv_load` != 0 the
 * next cascade launches never issue the load of their first KV tile, so the consumer's
 * bounded wait runs out and the launch reports QUAIL_ERR_TIMEOUT. Nothing faults.
 */
void quail_debug_inject(int32_t skip_first_kv_load);

/*
 * Kernel choice for head_dim 128 cascade calls (fused, without K/V amax). The CTA-pair
 * kernel runs four 128-row query tiles of one (anchor, KV head) on a pair of SMs: each
 * S = Q K^T and O += P V is one 256-row tcgen05 MMA over the pair, each SM holding its
 * own query rows and half of every K/V tile (half the tile loads per SM). The single-SM
 * kernel runs two query tiles on one SM, and loads a suffix window of at most 64 keys as
 * one 64-key tile where the pair always uses 128-key tiles.
 *   QUAIL_CTA_PAIRS_OFF     always the single-SM kernel
 *   QUAIL_CTA_PAIRS_AUTO    (default) the pair kernel (measured faster on every shape
 *                           tried, short suffix windows included), except with the
 *                           fault-injection switch on
 *   QUAIL_CTA_PAIRS_ALWAYS  always the pair kernel
 * Both give the same results within rounding. Process-wide; set it between calls, not
 * while another thread is launching. Returns QUAIL_ERR_INVALID_ARG for another `mode`.
 */
#define QUAIL_CTA_PAIRS_OFF 0
#define QUAIL_CTA_PAIRS_AUTO 1
#define QUAIL_CTA_PAIRS_ALWAYS 2
quail_status quail_set_cta_pairs(int32_t mode);

/* Library version, e.g. "quail-gb300 0.1". */
const char* quail_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QUAIL_H_ */
