/*
 * paq8 -- paged attention over a q8 KV cache, for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  All tensors are caller-owned device buffers passed as plain
 * pointers; the library never allocates or frees device memory and never
 * synchronizes a stream (except pa_check_status).  Each call's work is
 * ordered on the stream given: its kernels run there, or -- the prefill
 * kernel of a batch that mixes prefill and decode (not in
 * pa_paged_attention_noalloc), the values of a fused store of 4096 tokens or
 * more -- on an internal high-priority stream of the device that is forked
 * from it and joined back to it inside the call (the pattern stream capture
 * accepts).  `stream` is a cudaStream_t (NULL = the
 * legacy default stream).  bf16 and fp16 buffers are passed as raw 16-bit
 * words.
 *
 * The q8 format (page "shared/attention_kit.py", `quantize_q8` and the
 * `KVPrefix` docstring): int8 codes, one fp16 scale per (token, kv head,
 * group of 32 consecutive channels):
 *     s     = max(max|x| / 127, 1e-8)                 (fp32)
 *     code  = clamp(round_half_away(x / s), -127, 127) (fp32 divide)
 *     scale = fp16(s), round to nearest even
 * Rounding half away from zero follows "shared/kernels/qk_quant_triton.py"
 * (`_norm_rope_quant`).  -128 is never produced.
 *
 * Cache layout (head-major pages, "HND"; the page "attention_impl.py" allows
 * NHD or HND per layer).  One (block, kv head) page of codes and of scales is
 * contiguous; K pages are token-major, V pages channel-major (a V page is the
 * transpose of its token rows, so that 4 consecutive keys of one channel are
 * one 32-bit word for the PV product):
 *     k_cache : int8 [num_blocks][num_kv_heads][block_size][head_dim]
 *     k_scale : fp16 [num_blocks][num_kv_heads][block_size][head_dim/32]
 *     v_cache : int8 [num_blocks][num_kv_heads][head_dim][block_size]
 *     v_scale : fp16 [num_blocks][num_kv_heads][head_dim/32][block_size]
 * Every base pointer must be 16-byte aligned;
 * num_blocks * num_kv_heads * head_dim must be below 2^31.
 *
 * Supported shapes: head_dim in {64, 128, 256}; block_size in {16, 32};
 * num_q_heads % num_kv_heads == 0 with num_q_heads / num_kv_heads <= 16.
 *
 * Device-side checks: bad metadata found by a kernel (a slot beyond the cache,
 * a block-table entry outside [0, num_blocks), seq_len < q_len, a
 * cu_seqlens_q entry beyond num_tokens) never faults; the kernel skips the
 * access and ORs a bit into a 32-bit status word in device memory, which
 * pa_check_status reads.  The status word must start zeroed.
 */
#ifndef PAQ8_H
#define PAQ8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or workspace */
    PA_ERR_UNSUPPORTED = 2,   /* shape outside the supported list */
    PA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
    PA_ERR_DEVICE_CHECK = 4,  /* a kernel found bad metadata (status bits 0x1-0x4) */
    PA_ERR_TIMEOUT = 5        /* a bounded device-side wait expired (status bit 0x8) */
} pa_status;

/* Bits of the device status word. */
#define PA_DEV_BAD_SLOT  0x1u  /* kv_store: slot >= num_blocks * block_size */
#define PA_DEV_BAD_BLOCK 0x2u  /* block_table entry outside [0, num_blocks) or past its row */
#define PA_DEV_BAD_SEQ   0x4u  /* seq_len < q_len, or cu_seqlens_q inconsistent */
#define PA_DEV_TIMEOUT   0x8u  /* a pipeline wait gave up after its time limit */
#define PA_DEV_BAD_Q     0x10u /* a q value outside the fp16 range (|q| >= 65520 or NaN) */
#define PA_DEV_BAD_POS   0x20u /* kv_store_norm_rope: a position outside the rotation table */

/* Flags of pa_paged_attention / pa_paged_attention_ex. */
#define PA_ATTN_NON_CAUSAL   0x1u  /* every query of a sequence sees all of its seq_len keys */
#define PA_ATTN_TEST_TIMEOUT 0x80000000u /* test hook, see pa_paged_attention_ex */

/*
 * kv_store -- quantize new K/V rows to q8 and scatter them into the paged
 * cache by slot.
 * Passage: "attention_impl.py" (fastkernels-b200), `_store_kvcache_nhd` /
 * `StoreKVCache.forward(key, value, k_cache, v_cache, slot_mapping)`: token n
 * goes to block slot / block_size, offset slot % block_size; slot < 0 (a
 * padding row) is skipped.  Quantization as in the format note above.
 *
 *   key, value        bf16 [num_tokens][num_kv_heads][head_dim]; the head and
 *                     channel dims contiguous, token stride given in elements
 *                     (a multiple of 8, so each row is 16-byte aligned).
 *   slot_mapping      int64 [num_tokens], 8-byte aligned.
 *   k_cache .. v_scale the HND caches (written).
 *   status            device uint32 status word (may be NULL: no reporting).
 * Slots >= num_blocks * block_size are skipped and flagged PA_DEV_BAD_SLOT.
 * Two tokens with the same non-negative slot in one call: undefined.
 * num_tokens == 0 is a no-op.  Returns PA_OK or an error; asynchronous.
 */
pa_status pa_kv_store(const void *key, int64_t key_token_stride,
                      const void *value, int64_t value_token_stride,
                      const int64_t *slot_mapping, int32_t num_tokens,
                      int32_t num_kv_heads, int32_t head_dim,
                      void *k_cache, void *k_scale, void *v_cache, void *v_scale,
                      int32_t num_blocks, int32_t block_size,
                      uint32_t *status, void *stream);

/*
 * kv_store_norm_rope -- kv_store with each key row normalized and rotated
 * first, in one pass from the projection output to the q8 cache.
 * Passage: "shared/kernels/qk_quant_triton.py" (`_norm_rope_quant`, `_rows`):
 * the weighted RMSNorm with fp32 statistics, its output rounded to the
 * activation dtype (bf16), then the fp32 rotation of channel pairs, and the
 * quantization reading the fp32 rotated values (no second bf16 rounding).
 * Here the quantization is the q8 format above and the scatter is kv_store's.
 *
 *   key, value, slot_mapping, caches, status: as pa_kv_store.
 *   positions     int64 [num_tokens]: the row of `rope` of each token (may be
 *                 NULL when rope is NULL).  A position outside
 *                 [0, max_position) skips the token and is flagged
 *                 PA_DEV_BAD_POS.
 *   norm_weight   bf16 [head_dim] (2-byte aligned), or NULL: no norm.  Per key
 *                 row x: total = sum of x_c^2 (lane l of 32 adds channels l,
 *                 l + 32, ... with fused multiply-adds, the 32 lane sums by an
 *                 xor butterfly 16, 8, 4, 2, 1), inv = 1 / sqrt(total /
 *                 head_dim + eps) (sqrt and divide rounded once each),
 *                 y_c = bf16((x_c * inv) * w_c).
 *   rope          fp32 [max_position][rotary_dim / 2][2] (cos, sin of each
 *                 pair), 8-byte aligned, or NULL: no rotation.  Pairs
 *                 (p, p + rotary_dim / 2), or (2p, 2p + 1) when interleaved;
 *                 lead = fma(cos, y_lead, (-sin) * y_trail), trail =
 *                 fma(sin, y_lead, cos * y_trail) in fp32; channels at and
 *                 past rotary_dim keep y.  rotary_dim even, in
 *                 [2, head_dim].
 * Values are stored unchanged, as pa_kv_store stores them.  Every step is
 * rounded as written, so the codes and scales equal those of a CPU
 * implementation of the same steps bit for bit.  Asynchronous.
 */
pa_status pa_kv_store_norm_rope(const void *key, int64_t key_token_stride,
                                const void *value, int64_t value_token_stride,
                                const int64_t *slot_mapping, const int64_t *positions,
                                int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                const void *norm_weight, float eps, const float *rope,
                                int32_t max_position, int32_t rotary_dim, int32_t interleaved,
                                void *k_cache, void *k_scale, void *v_cache, void *v_scale,
                                int32_t num_blocks, int32_t block_size, uint32_t *status,
                                void *stream);

/*
 * Split-KV segments chosen when pa_paged_attention gets num_splits == 0, for
 * these host-side hints (no device access).  Result in [1, 16].
 * Passage: "triton_turboquant_unified_attention.py" launcher (16 segments by
 * default, capped by the KV length); this library targets ~1024 keys per
 * segment and at most ~8192 (sequence, kv head, segment) units in all.
 */
int32_t pa_auto_num_splits(int32_t num_seqs, int32_t num_kv_heads,
                           int32_t max_query_len, int32_t max_seq_len);

/*
 * Bytes of workspace pa_paged_attention needs: 256 bytes of header (the
 * status word at offset 0) plus, when num_splits > 1, fp32 partial triples
 * [num_seqs][num_q_heads][num_splits][head_dim + 2].
 * num_splits == 0 sizes for the largest automatic choice (16).
 */
size_t pa_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                         int32_t num_splits);

/*
 * paged_attention -- unified causal prefill + decode over the q8 cache.
 * Passages: "triton_turboquant_unified_attention.py" (vLLM unified kernel
 * and launcher: query_start_loc / seq_lens / block_table, GQA heads stacked
 * into the row tile, in-tile dequantization, online softmax, 3D split-KV
 * segments merged by `reduce_segments`); "attention_impl.py" torch reference
 * paths for the causal alignment (key_offset = k_len - q_len).
 *
 *   q             bf16 [num_tokens][num_q_heads][head_dim], contiguous.
 *   k_cache..     HND caches (read only).
 *   cu_seqlens_q  int32 [num_seqs + 1]; sequence s owns query tokens
 *                 [cu[s], cu[s+1]); cu[0] = 0, non-decreasing, cu[S] <= num_tokens.
 *   seq_lens      int32 [num_seqs]; the KV length of sequence s INCLUDING its
 *                 new tokens (they must already be stored).  Query i of s sees
 *                 keys 0 .. seq_len - q_len + i (bottom-right causal).
 *   block_table   int32 [num_seqs][block_table_stride]; logical page p of s
 *                 lives in physical block block_table[s][p].
 *   max_query_len host upper bound on every q_len (never synced).  With 1 the
 *                 call takes the decode-only path; a sequence with more query
 *                 tokens is then left unprocessed and flagged PA_DEV_BAD_SEQ.
 *   max_seq_len   host hint for the segment length only; any positive value
 *                 gives correct results (a sequence longer than the hint just
 *                 gets a longer last segment).
 *   softmax_scale applied to q.k before the softmax (1/sqrt(D) typically).
 *   num_splits    0 = automatic, 1 = none, k in [2, 16] = k segments.
 *                 Segments apply to sequences with exactly one query token
 *                 (decode rows); longer query chunks are never split.
 *   out           bf16 [num_tokens][num_q_heads][head_dim] (written).
 *   lse           fp32 [num_tokens][num_q_heads] natural-log LSE of
 *                 softmax_scale * q.k over the visible keys, or NULL.
 *   workspace     device buffer of workspace_bytes >= pa_workspace_size(...);
 *                 its first 4 bytes are the status word (zero it once).
 *   flags         0 (causal) or PA_ATTN_NON_CAUSAL: every query of sequence s
 *                 sees keys 0 .. seq_len - 1, and seq_len may be below q_len
 *                 (even 0: such rows get out = 0, lse = -inf).  This is the
 *                 first pass of attention over a cached prefix plus new keys
 *                 ("shared/attention_kit.py", `_attend_with_prefix`): attend
 *                 the prefix non-causally, the new keys causally, and merge
 *                 the two with pa_merge_attn_states.
 * Rows of tokens no sequence owns are not written.  Asynchronous.
 * Numerics: K codes enter the QK^T product exactly (fp16 integers), each
 * 32-channel group accumulated in fp32 and then scaled; q is rounded to fp16
 * (exact for |q| in [2^-14, 65504]; below 2^-14 the error is under 2^-25;
 * |q| >= 65520 becomes inf and is flagged PA_DEV_BAD_Q); V is dequantized to
 * fp16 (code * scale); softmax and accumulation in fp32; the output rounded
 * to bf16.
 */
pa_status pa_paged_attention(const void *q, const void *k_cache, const void *k_scale,
                             const void *v_cache, const void *v_scale,
                             const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                             const int32_t *block_table, int32_t block_table_stride,
                             int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                             int32_t block_size, int32_t max_query_len, int32_t max_seq_len,
                             float softmax_scale, int32_t num_splits,
                             void *out, float *lse, void *workspace, size_t workspace_bytes,
                             uint32_t flags, void *stream);

/*
 * paged_attention with attention sinks and a sliding window.
 * Passages: "triton_turboquant_unified_attention.py", USE_SINKS (a per-q-head
 * sink logit starts the online softmax as M = sink, L = 1 -- one term of the
 * denominator with no value -- in segment 0 only when the keys are split);
 * "attention_impl.py", `window_size = (sliding_window - 1, 0)` (a query sees
 * only the last sliding_window keys up to its causal limit).
 *
 *   sinks           fp32 [num_q_heads] sink logits, in the units of the
 *                   scaled scores softmax_scale * q.k (natural log), finite
 *                   or -inf (no sink); NULL = none.  The LSE then includes the
 *                   sink: lse = ln(exp(sink) + sum_j exp(s_j)).
 *   sliding_window  0 = none; W > 0: query i of sequence s sees keys
 *                   max(0, p - W + 1) .. p, p = seq_len - q_len + i.  Needs
 *                   causal attention (PA_ERR_INVALID_ARG with
 *                   PA_ATTN_NON_CAUSAL).  Pages wholly before a q-block's
 *                   first visible key are never read, so their block-table
 *                   entries may be stale.
 *   flags           PA_ATTN_NON_CAUSAL as for pa_paged_attention, and
 *                   PA_ATTN_TEST_TIMEOUT, a test hook: the decode kernel's
 *                   producer stages nothing and its waits give up after about
 *                   1 ms, so that the call ends with PA_DEV_TIMEOUT in the
 *                   status word (pa_check_status: PA_ERR_TIMEOUT) and
 *                   garbage rows; the context stays usable.  Only on the
 *                   decode path (max_query_len == 1, at most 8 q heads per kv
 *                   head); never in production.
 * Other arguments, errors and numerics as pa_paged_attention, which is this
 * call with sinks = NULL and sliding_window = 0.
 */
pa_status pa_paged_attention_ex(const void *q, const void *k_cache, const void *k_scale,
                                const void *v_cache, const void *v_scale,
                                const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                const int32_t *block_table, int32_t block_table_stride,
                                int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                                int32_t block_size, int32_t max_query_len, int32_t max_seq_len,
                                float softmax_scale, int32_t num_splits, const float *sinks,
                                int32_t sliding_window, void *out, float *lse, void *workspace,
                                size_t workspace_bytes, uint32_t flags, void *stream);

/*
 * The alternative cache format: fp8 keys and 4-bit values.
 * Passage: "triton_turboquant_unified_attention.py", the FP8-key and 4-bit
 * value load sites of the unified kernel (`_tq_load_k_tile`: an FP8 key is
 * read as its e4m3 value, no scale; `_tq_load_v_tile`: V = idx * scale +
 * zero with one fp16 scale and zero per token).  The page shows only the
 * load sites; the store used here (a reading):
 *     K     = e4m3(x), round to nearest even, saturating at +-448
 *     lo, hi = min, max of the token's D values (fp32)
 *     s     = max((hi - lo) / 15, 1e-8)                        (fp32)
 *     idx   = clamp(round_half_away((x - lo) / s), 0, 15)      (fp32 divide)
 *     scale = fp16(s), zero = fp16(lo)
 * Caches (head-major pages; per (key, kv head) D + D/2 + 4 bytes instead of
 * q8's 2 * (D + D/16)):
 *     k_cache : uint8 [num_blocks][num_kv_heads][block_size][head_dim]   e4m3
 *     v_cache : uint8 [num_blocks][num_kv_heads][head_dim][block_size/2] byte j
 *               of a channel row: keys 2j (low nibble) and 2j + 1 (high)
 *     v_scale, v_zero : fp16 [num_blocks][num_kv_heads][block_size]
 * All base pointers 16-byte aligned.
 */

/*
 * kv_store in the fp8 / 4-bit format.  Arguments as pa_kv_store.  Two tokens
 * of one call whose slots share a nibble byte are both written; a token whose
 * byte mate is not in the call keeps the mate's nibble (it updates its own
 * with 32-bit atomics).  Asynchronous.
 */
pa_status pa_kv_store_f8v4(const void *key, int64_t key_token_stride,
                           const void *value, int64_t value_token_stride,
                           const int64_t *slot_mapping, int32_t num_tokens,
                           int32_t num_kv_heads, int32_t head_dim,
                           void *k_cache, void *v_cache, void *v_scale, void *v_zero,
                           int32_t num_blocks, int32_t block_size,
                           uint32_t *status, void *stream);

/*
 * paged_attention over the fp8 / 4-bit format: as pa_paged_attention_ex
 * (decode and prefill rows in one batch, split-KV segments, non-causal
 * mode, sinks, sliding window, flags).  Numerics: K is exact in fp16 (every
 * e4m3 value is an fp16 value), QK^T accumulates in fp32; V' = idx * scale
 * + zero in one fp16 FMA; softmax and accumulation in fp32; output bf16.
 */
pa_status pa_paged_attention_f8v4(const void *q, const void *k_cache, const void *v_cache,
                                  const void *v_scale, const void *v_zero,
                                  const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                  const int32_t *block_table, int32_t block_table_stride,
                                  int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                                  int32_t block_size, int32_t max_query_len, int32_t max_seq_len,
                                  float softmax_scale, int32_t num_splits, const float *sinks,
                                  int32_t sliding_window, void *out, float *lse, void *workspace,
                                  size_t workspace_bytes, uint32_t flags, void *stream);

/*
 * merge_attn_states -- the attention of queries over the union of two
 * disjoint key sets, from their attention over each set (e.g. a cached
 * prefix attended in one pass and the new keys in another, or two calls'
 * split-KV results).
 * Passage: "shared/attention_kit.py", `_merge_lse_(out, lse, other,
 * other_lse)`: log-sum-exp weights of the two partial results (the page
 * keeps base-2 LSEs; here, as for pa_paged_attention, they are natural-log).
 *
 *   out_a, out_b  bf16 [num_rows][head_dim], 16-byte aligned: the
 *                 normalized attention output of each part (a row = one
 *                 query token and q head, e.g. pa_paged_attention's out
 *                 viewed as [num_tokens * num_q_heads][head_dim]).
 *   lse_a, lse_b  fp32 [num_rows], 4-byte aligned: natural-log LSE of each
 *                 part; -inf marks a part with no key for that row.  +inf
 *                 and NaN are not supported.
 *   out           bf16 [num_rows][head_dim] (written); may be out_a or out_b.
 *   lse           fp32 [num_rows] merged LSE (written), or NULL; may be
 *                 lse_a or lse_b.
 * Per row: M = max(lse_a, lse_b), e_x = exp(lse_x - M),
 *   out = (e_a * out_a + e_b * out_b) / (e_a + e_b)   (fp32, rounded to bf16)
 *   lse = M + ln(e_a + e_b).
 * A row whose two LSEs are both -inf gets out = 0 and lse = -inf.
 * Supported head_dim: 64, 128, 256.  num_rows == 0 is a no-op.
 * Returns PA_OK or an error; asynchronous on `stream`.
 */
pa_status pa_merge_attn_states(const void *out_a, const float *lse_a, const void *out_b,
                               const float *lse_b, void *out, float *lse, int64_t num_rows,
                               int32_t head_dim, void *stream);

/*
 * Synchronizes `stream`, reads the device status word at `status` (a kv_store
 * status word, or the start of an attention workspace), clears it, and maps
 * it to PA_OK / PA_ERR_TIMEOUT (bit 0x8 set) / PA_ERR_DEVICE_CHECK (other
 * bits).  The raw bits go to *bits_out when it is not NULL.  The only call of
 * this library that blocks the host.
 */
pa_status pa_check_status(uint32_t *status, uint32_t *bits_out, void *stream);

/*
 * Allocation-free variant of pa_paged_attention.  The paper has no
 * counterpart to this call; it is an integration convenience.  For callers
 * that cannot call cudaMalloc: plugins run inside another framework's executor where
 * allocation is forbidden, serving loops that must never wait on the
 * allocator, fixed-budget embeddings.  Arguments as pa_paged_attention,
 * except that there is no workspace: the split-KV partials live in a
 * file-scope device array of 8 MiB that every GPU loading the library holds
 * until exit.  The caller still passes inputs and outputs.
 *   status  optional device uint32: receives this call's status bits
 *           (overwritten, not OR-ed); NULL = no reporting.
 * A num_splits > 1 whose partials exceed 8 MiB is rejected
 * (PA_ERR_INVALID_ARG); num_splits == 0 picks the largest automatic count that
 * fits.  Every call looks up the array's device address with the current
 * device (cheap; it follows the module if a context is recreated); the first
 * call on a device may load the module, so make it before any stream capture.
 * Arguments are checked before the array or the stream is touched.
 * Every call shares the one array: calls that overlap on the GPU (other
 * streams, other threads) race and give wrong results; serialize them.
 * Allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 */
pa_status pa_paged_attention_noalloc(const void *q, const void *k_cache, const void *k_scale,
                                     const void *v_cache, const void *v_scale,
                                     const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                     const int32_t *block_table, int32_t block_table_stride,
                                     int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                                     int32_t block_size, int32_t max_query_len,
                                     int32_t max_seq_len, float softmax_scale,
                                     int32_t num_splits, void *out, float *lse,
                                     uint32_t *status, void *stream);

/* Static description of a status code. */
const char *pa_status_string(pa_status s);

/* Description of the last argument error on the calling thread ("" if none). */
const char *pa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PAQ8_H */
