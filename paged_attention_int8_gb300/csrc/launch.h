// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace paq8 {

cudaError_t launch_kv_store(const uint16_t *key, int64_t key_stride, const uint16_t *value,
                            int64_t value_stride, const int64_t *slot_mapping,
                            int32_t num_tokens, int32_t hk, int32_t d, int8_t *k_cache,
                            uint16_t *k_scale, int8_t *v_cache, uint16_t *v_scale,
                            int32_t num_blocks, int32_t block_size, uint32_t *status,
                            cudaStream_t stream);

int32_t auto_num_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t max_query_len,
                        int32_t max_seq_len);

struct AttnLaunch {
  const void *q, *k_cache, *k_scale, *v_cache, *v_scale;
  const int32_t *cu, *seq_lens, *block_table;
  int32_t bt_stride, num_seqs, num_tokens, hq, hk, d, num_blocks, bs, max_query_len,
      max_seq_len, num_splits;
  float softmax_scale;
  void *out;
  float *lse;
  uint8_t *workspace;
  bool side_stream_ok = true;  // a mixed batch may run prefill on the side stream
};

cudaError_t launch_paged_attention(const AttnLaunch &L, cudaStream_t stream);

}  // namespace paq8
