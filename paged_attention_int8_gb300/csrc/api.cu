// C ABI of libpaq8: argument validation and dispatch.  Every entry point is
// declared, with its contract, in include/paq8.h.
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "launch.h"
#include "merge.h"


namespace {

thread_local char g_last_error[256] = "";

pa_status fail(pa_status s, const char *msg) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s", msg);
  return s;
}

pa_status cuda_fail(cudaError_t e) {
  std::snprintf(g_last_error, sizeof g_last_error, "CUDA: %s", cudaGetErrorString(e));
  return PA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dim(int32_t d) { return d == 64 || d == 128 || d == 256; }
bool supported_bs(int32_t bs) { return bs == 16 || bs == 32; }

}  // namespace

extern "C" {

pa_status pa_kv_store(const void *key, int64_t key_token_stride, const void *value,
                      int64_t value_token_stride, const int64_t *slot_mapping,
                      int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                      void *k_cache, void *k_scale, void *v_cache, void *v_scale,
                      int32_t num_blocks, int32_t block_size, uint32_t *status, void *stream) {
  g_last_error[0] = '\0';
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping || !k_cache || !k_scale || !v_cache || !v_scale)
    return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (num_kv_heads <= 0 || num_blocks <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_kv_heads and num_blocks must be positive");
  if (!supported_dim(head_dim)) return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (!supported_bs(block_size)) return fail(PA_ERR_UNSUPPORTED, "block_size must be 16 or 32");
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (key_token_stride < row || value_token_stride < row)
    return fail(PA_ERR_INVALID_ARG, "token stride smaller than num_kv_heads * head_dim");
  if (key_token_stride % 8 || value_token_stride % 8 || !aligned16(key) || !aligned16(value))
    return fail(PA_ERR_INVALID_ARG, "key/value rows must be 16-byte aligned");
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_scale) || !aligned16(v_scale))
    return fail(PA_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)
    return fail(PA_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
  if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size >= (int64_t{1} << 31))
    return fail(PA_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * block_size must be < 2^31");
  cudaError_t e = paq8::launch_kv_store(
      static_cast<const uint16_t *>(key), key_token_stride, static_cast<const uint16_t *>(value),
      value_token_stride, slot_mapping, num_tokens, num_kv_heads, head_dim,
      static_cast<int8_t *>(k_cache), static_cast<uint16_t *>(k_scale),
      static_cast<int8_t *>(v_cache), static_cast<uint16_t *>(v_scale), num_blocks, block_size,
      status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_kv_store_norm_rope(const void *key, int64_t key_token_stride, const void *value,
                                int64_t value_token_stride, const int64_t *slot_mapping,
                                const int64_t *positions, int32_t num_tokens,
                                int32_t num_kv_heads, int32_t head_dim, const void *norm_weight,
                                float eps, const float *rope, int32_t max_position,
                                int32_t rotary_dim, int32_t interleaved, void *k_cache,
                                void *k_scale, void *v_cache, void *v_scale, int32_t num_blocks,
                                int32_t block_size, uint32_t *status, void *stream) {
  g_last_error[0] = '\0';
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping || !k_cache || !k_scale || !v_cache || !v_scale)
    return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (num_kv_heads <= 0 || num_blocks <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_kv_heads and num_blocks must be positive");
  if (!supported_dim(head_dim)) return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (!supported_bs(block_size)) return fail(PA_ERR_UNSUPPORTED, "block_size must be 16 or 32");
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (key_token_stride < row || value_token_stride < row)
    return fail(PA_ERR_INVALID_ARG, "token stride smaller than num_kv_heads * head_dim");
  if (value_token_stride % 8 || !aligned16(value))
    return fail(PA_ERR_INVALID_ARG, "value rows must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(key) & 1u)
    return fail(PA_ERR_INVALID_ARG, "key must be 2-byte aligned");
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_scale) || !aligned16(v_scale))
    return fail(PA_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
      (positions && (reinterpret_cast<uintptr_t>(positions) & 7u)))
    return fail(PA_ERR_INVALID_ARG, "slot_mapping and positions must be 8-byte aligned");
  if (norm_weight && (reinterpret_cast<uintptr_t>(norm_weight) & 1u))
    return fail(PA_ERR_INVALID_ARG, "norm_weight must be 2-byte aligned");
  if (rope) {
    if (!positions) return fail(PA_ERR_INVALID_ARG, "a rotation needs positions");
    if (reinterpret_cast<uintptr_t>(rope) & 7u)
      return fail(PA_ERR_INVALID_ARG, "rope must be 8-byte aligned");
    if (rotary_dim < 2 || rotary_dim > head_dim || rotary_dim % 2)
      return fail(PA_ERR_INVALID_ARG, "rotary_dim must be even, in [2, head_dim]");
    if (max_position <= 0) return fail(PA_ERR_INVALID_ARG, "max_position must be positive");
  }
  if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size >= (int64_t{1} << 31))
    return fail(PA_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * block_size must be < 2^31");
  paq8::KvNormRope p;
  p.key = static_cast<const uint16_t *>(key);
  p.value = static_cast<const uint16_t *>(value);
  p.key_stride = key_token_stride;
  p.value_stride = value_token_stride;
  p.slot_mapping = slot_mapping;
  p.positions = positions;
  p.num_tokens = num_tokens;
  p.hk = num_kv_heads;
  p.d = head_dim;
  p.norm_weight = static_cast<const uint16_t *>(norm_weight);
  p.eps = eps;
  p.rope = rope;
  p.max_position = rope ? max_position : 0;
  p.rotary_dim = rope ? rotary_dim : 0;
  p.interleaved = interleaved != 0;
  p.k_cache = static_cast<int8_t *>(k_cache);
  p.k_scale = static_cast<uint16_t *>(k_scale);
  p.v_cache = static_cast<int8_t *>(v_cache);
  p.v_scale = static_cast<uint16_t *>(v_scale);
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.status = status;
  cudaError_t e = paq8::launch_kv_store_norm_rope(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int32_t pa_auto_num_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t max_query_len,
                           int32_t max_seq_len) {
  return paq8::auto_num_splits(num_seqs, num_kv_heads, max_query_len, max_seq_len);
}

size_t pa_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                         int32_t num_splits) {
  if (num_seqs < 0 || num_q_heads < 0 || head_dim < 0 || num_splits < 0) return 0;
  const int32_t ns = num_splits == 0 ? 16 : num_splits;
  size_t bytes = 256;
  if (ns > 1)
    bytes += static_cast<size_t>(num_seqs) * num_q_heads * ns * (head_dim + 2) * sizeof(float);
  return bytes;
}

}  // extern "C"

namespace {

// Validation of a paged-attention call and its launch description.  Shared by
// every attention entry point, so that the allocation-free one checks its
// arguments before it touches its scratch.
pa_status attention_args(const void *q, const void *k_cache, const void *k_scale,
                         const void *v_cache, const void *v_scale, const int32_t *cu_seqlens_q,
                         const int32_t *seq_lens, const int32_t *block_table,
                         int32_t block_table_stride, int32_t num_seqs, int32_t num_tokens,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t num_blocks, int32_t block_size, int32_t max_query_len,
                         int32_t max_seq_len, float softmax_scale, int32_t num_splits,
                         const float *sinks, int32_t sliding_window, void *out, float *lse,
                         void *workspace, size_t workspace_bytes, uint32_t flags,
                         paq8::AttnLaunch *L, bool *nothing_to_do,
                         const void *v_zero = nullptr) {
  *nothing_to_do = false;
  const bool f8v4 = v_zero != nullptr;
  if (f8v4) k_scale = v_zero;  // the fp8 / 4-bit format has no key scales
  if (flags & ~(PA_ATTN_NON_CAUSAL | PA_ATTN_TEST_TIMEOUT))
    return fail(PA_ERR_INVALID_ARG, "unknown flag bits");
  const bool causal = !(flags & PA_ATTN_NON_CAUSAL);
  if (num_seqs < 0 || num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "null workspace");
  if (sliding_window < 0) return fail(PA_ERR_INVALID_ARG, "sliding_window < 0");
  if (sliding_window > 0 && !causal)
    return fail(PA_ERR_INVALID_ARG, "a sliding window needs causal attention");
  if (num_seqs == 0 || num_tokens == 0) {
    *nothing_to_do = true;
    return PA_OK;
  }
  if (!q || !k_cache || !k_scale || !v_cache || !v_scale || !cu_seqlens_q || !seq_lens ||
      !block_table || !out)
    return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
  if (num_q_heads / num_kv_heads > 16)
    return fail(PA_ERR_UNSUPPORTED, "more than 16 q heads per kv head");
  if (!supported_dim(head_dim)) return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (!supported_bs(block_size)) return fail(PA_ERR_UNSUPPORTED, "block_size must be 16 or 32");
  if (num_blocks <= 0 || block_table_stride <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_blocks and block_table_stride must be positive");
  if (static_cast<int64_t>(num_blocks) * num_kv_heads * head_dim >= (int64_t{1} << 31))
    return fail(PA_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * head_dim must be < 2^31");
  if (max_query_len <= 0 || max_seq_len <= 0)
    return fail(PA_ERR_INVALID_ARG, "max_query_len and max_seq_len must be positive");
  if (num_splits < 0 || num_splits > 16) return fail(PA_ERR_INVALID_ARG, "num_splits in [0, 16]");
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(k_scale) || !aligned16(v_scale) || !aligned16(workspace))
    return fail(PA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if ((lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
      (sinks && (reinterpret_cast<uintptr_t>(sinks) & 3u)))
    return fail(PA_ERR_INVALID_ARG, "lse and sinks must be 4-byte aligned");
  if ((flags & PA_ATTN_TEST_TIMEOUT) &&
      (max_query_len != 1 || num_q_heads / num_kv_heads > 8))
    return fail(PA_ERR_INVALID_ARG,
                "PA_ATTN_TEST_TIMEOUT needs the decode path (max_query_len 1, <= 8 q heads per kv head)");
  // a window bounds the keys a row sees: size the automatic split count for it
  const int32_t seen = sliding_window > 0 && sliding_window < max_seq_len ? sliding_window
                                                                          : max_seq_len;
  int32_t ns = num_splits == 0
                   ? paq8::auto_num_splits(num_seqs, num_kv_heads, max_query_len, seen)
                   : num_splits;
  if (workspace_bytes < pa_workspace_size(num_seqs, num_q_heads, head_dim, ns)) {
    if (num_splits != 0) return fail(PA_ERR_INVALID_ARG, "workspace too small for num_splits");
    while (ns > 1 && workspace_bytes < pa_workspace_size(num_seqs, num_q_heads, head_dim, ns))
      --ns;
    if (workspace_bytes < pa_workspace_size(num_seqs, num_q_heads, head_dim, ns))
      return fail(PA_ERR_INVALID_ARG, "workspace smaller than 256 bytes");
  }
  paq8::AttnLaunch &a = *L;
  a.q = q;
  a.k_cache = k_cache;
  a.k_scale = k_scale;
  a.v_cache = v_cache;
  a.v_scale = v_scale;
  a.cu = cu_seqlens_q;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.bt_stride = block_table_stride;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.hq = num_q_heads;
  a.hk = num_kv_heads;
  a.d = head_dim;
  a.num_blocks = num_blocks;
  a.bs = block_size;
  a.max_query_len = max_query_len;
  a.max_seq_len = max_seq_len;
  a.num_splits = ns;
  a.softmax_scale = softmax_scale;
  a.out = out;
  a.lse = lse;
  a.workspace = static_cast<uint8_t *>(workspace);
  a.causal = causal;
  a.window = sliding_window;
  a.sinks = sinks;
  a.test_timeout = (flags & PA_ATTN_TEST_TIMEOUT) != 0;
  a.f8v4 = f8v4;
  a.v_zero = v_zero;
  return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_paged_attention_ex(const void *q, const void *k_cache, const void *k_scale,
                                const void *v_cache, const void *v_scale,
                                const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                const int32_t *block_table, int32_t block_table_stride,
                                int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                                int32_t block_size, int32_t max_query_len, int32_t max_seq_len,
                                float softmax_scale, int32_t num_splits, const float *sinks,
                                int32_t sliding_window, void *out, float *lse, void *workspace,
                                size_t workspace_bytes, uint32_t flags, void *stream) {
  g_last_error[0] = '\0';
  paq8::AttnLaunch L;
  bool nothing = false;
  pa_status st = attention_args(
      q, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens, block_table,
      block_table_stride, num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, num_blocks,
      block_size, max_query_len, max_seq_len, softmax_scale, num_splits, sinks, sliding_window,
      out, lse, workspace, workspace_bytes, flags, &L, &nothing);
  if (st != PA_OK || nothing) return st;
  cudaError_t e = paq8::launch_paged_attention(L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_paged_attention_f8v4(const void *q, const void *k_cache, const void *v_cache,
                                  const void *v_scale, const void *v_zero,
                                  const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                  const int32_t *block_table, int32_t block_table_stride,
                                  int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                                  int32_t block_size, int32_t max_query_len, int32_t max_seq_len,
                                  float softmax_scale, int32_t num_splits, const float *sinks,
                                  int32_t sliding_window, void *out, float *lse, void *workspace,
                                  size_t workspace_bytes, uint32_t flags, void *stream) {
  g_last_error[0] = '\0';
  if (!v_zero) return fail(PA_ERR_INVALID_ARG, "null v_zero");
  paq8::AttnLaunch L;
  bool nothing = false;
  pa_status st = attention_args(
      q, k_cache, nullptr, v_cache, v_scale, cu_seqlens_q, seq_lens, block_table,
      block_table_stride, num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, num_blocks,
      block_size, max_query_len, max_seq_len, softmax_scale, num_splits, sinks, sliding_window,
      out, lse, workspace, workspace_bytes, flags, &L, &nothing, v_zero);
  if (st != PA_OK || nothing) return st;
  cudaError_t e = paq8::launch_paged_attention(L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_kv_store_f8v4(const void *key, int64_t key_token_stride, const void *value,
                           int64_t value_token_stride, const int64_t *slot_mapping,
                           int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                           void *k_cache, void *v_cache, void *v_scale, void *v_zero,
                           int32_t num_blocks, int32_t block_size, uint32_t *status,
                           void *stream) {
  g_last_error[0] = '\0';
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping || !k_cache || !v_cache || !v_scale || !v_zero)
    return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (num_kv_heads <= 0 || num_blocks <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_kv_heads and num_blocks must be positive");
  if (!supported_dim(head_dim)) return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (!supported_bs(block_size)) return fail(PA_ERR_UNSUPPORTED, "block_size must be 16 or 32");
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (key_token_stride < row || value_token_stride < row)
    return fail(PA_ERR_INVALID_ARG, "token stride smaller than num_kv_heads * head_dim");
  if (key_token_stride % 8 || value_token_stride % 8 || !aligned16(key) || !aligned16(value))
    return fail(PA_ERR_INVALID_ARG, "key/value rows must be 16-byte aligned");
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(v_scale) || !aligned16(v_zero))
    return fail(PA_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)
    return fail(PA_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
  if (static_cast<int64_t>(num_blocks) * num_kv_heads * head_dim >= (int64_t{1} << 31))
    return fail(PA_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * head_dim must be < 2^31");
  cudaError_t e = paq8::launch_kv_store_f8v4(
      static_cast<const uint16_t *>(key), key_token_stride, static_cast<const uint16_t *>(value),
      value_token_stride, slot_mapping, num_tokens, num_kv_heads, head_dim,
      static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache),
      static_cast<uint16_t *>(v_scale), static_cast<uint16_t *>(v_zero), num_blocks, block_size,
      status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_paged_attention(const void *q, const void *k_cache, const void *k_scale,
                             const void *v_cache, const void *v_scale,
                             const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                             const int32_t *block_table, int32_t block_table_stride,
                             int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                             int32_t block_size, int32_t max_query_len, int32_t max_seq_len,
                             float softmax_scale, int32_t num_splits, void *out, float *lse,
                             void *workspace, size_t workspace_bytes, uint32_t flags,
                             void *stream) {
  return pa_paged_attention_ex(q, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens,
                               block_table, block_table_stride, num_seqs, num_tokens,
                               num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                               max_query_len, max_seq_len, softmax_scale, num_splits, nullptr, 0,
                               out, lse, workspace, workspace_bytes, flags, stream);
}

pa_status pa_merge_attn_states(const void *out_a, const float *lse_a, const void *out_b,
                               const float *lse_b, void *out, float *lse, int64_t num_rows,
                               int32_t head_dim, void *stream) {
  g_last_error[0] = '\0';
  if (num_rows < 0) return fail(PA_ERR_INVALID_ARG, "num_rows < 0");
  if (num_rows == 0) return PA_OK;
  if (!out_a || !lse_a || !out_b || !lse_b || !out) return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!supported_dim(head_dim)) return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (!aligned16(out_a) || !aligned16(out_b) || !aligned16(out))
    return fail(PA_ERR_INVALID_ARG, "out_a, out_b and out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse_a) | reinterpret_cast<uintptr_t>(lse_b) |
       reinterpret_cast<uintptr_t>(lse)) & 3u)
    return fail(PA_ERR_INVALID_ARG, "lse arrays must be 4-byte aligned");
  if (num_rows > (int64_t{1} << 40)) return fail(PA_ERR_INVALID_ARG, "num_rows too large");
  cudaError_t e = paq8::launch_merge_states(
      static_cast<const uint16_t *>(out_a), lse_a, static_cast<const uint16_t *>(out_b), lse_b,
      static_cast<uint16_t *>(out), lse, num_rows, head_dim, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_check_status(uint32_t *status, uint32_t *bits_out, void *stream) {
  if (!status) return fail(PA_ERR_INVALID_ARG, "null status pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  cudaError_t e = cudaMemcpyAsync(&bits, status, sizeof bits, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && bits) e = cudaMemsetAsync(status, 0, sizeof bits, s);
  if (e == cudaSuccess && bits) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (bits_out) *bits_out = bits;
  if (bits & PA_DEV_TIMEOUT) return PA_ERR_TIMEOUT;
  if (bits) return PA_ERR_DEVICE_CHECK;
  return PA_OK;
}

const char *pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_DEVICE_CHECK: return "device-side metadata check failed";
    case PA_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char *pa_last_error(void) { return g_last_error; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free paged attention.
//
// Some callers cannot call cudaMalloc: a plugin run inside another
// framework's executor that forbids allocation on its hot path, a serving
// loop that must never wait on the allocator (cudaMalloc can synchronize the
// device), or an embedding with a fixed memory budget.  For them the split-KV
// scratch comes from this file-scope device array instead of a caller
// workspace.  Every GPU that loads the library holds it until the process
// exits.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t{8} << 20;  // 8 MiB per device
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with the device current -- on every call: the lookup is cheap, allocates
// nothing, and stays right if the device's context is torn down and the
// module reloaded (the array may then move).
pa_status noalloc_scratch(void **out) {
  void *p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
  *out = p;
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_paged_attention_noalloc(
    const void *q, const void *k_cache, const void *k_scale, const void *v_cache,
    const void *v_scale, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
    const int32_t *block_table, int32_t block_table_stride, int32_t num_seqs,
    int32_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t num_blocks, int32_t block_size, int32_t max_query_len, int32_t max_seq_len,
    float softmax_scale, int32_t num_splits, void *out, float *lse, uint32_t *status,
    void *stream) {
  g_last_error[0] = '\0';
  if (num_splits > 1 &&
      pa_workspace_size(num_seqs, num_q_heads, head_dim, num_splits) > kNoAllocScratchBytes) {
    char msg[160];
    std::snprintf(msg, sizeof msg,
                  "num_splits=%d needs %zu bytes of split scratch; the static scratch holds %zu",
                  num_splits, pa_workspace_size(num_seqs, num_q_heads, head_dim, num_splits),
                  kNoAllocScratchBytes);
    return fail(PA_ERR_INVALID_ARG, msg);
  }
  void *scratch = nullptr;
  pa_status st = noalloc_scratch(&scratch);
  if (st != PA_OK) return st;
  // every argument is checked before the shared scratch or the stream is touched
  paq8::AttnLaunch L;
  bool nothing = false;
  st = attention_args(q, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens, block_table,
                      block_table_stride, num_seqs, num_tokens, num_q_heads, num_kv_heads,
                      head_dim, num_blocks, block_size, max_query_len, max_seq_len,
                      softmax_scale, num_splits, nullptr, 0, out, lse, scratch,
                      kNoAllocScratchBytes, 0, &L, &nothing);
  if (st != PA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (nothing) {
    if (status) {
      cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return PA_OK;
  }
  // The scratch keeps the previous call's contents: its status word must
  // start at zero; the split partials are always written before they are read.
  cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return cuda_fail(e);
  // no side stream: creating one would create driver resources
  L.side_stream_ok = false;
  e = paq8::launch_paged_attention(L, s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (status) {
    e = cudaMemcpyAsync(status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return PA_OK;
}
