// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace paq8 {

constexpr int kMaxDevices = 64;

// One-time set-up per device (a kernel's shared-memory attribute, an SM
// count), safe when several host threads launch on several devices: init(dev,
// &value) runs once for each device, with that device current, and later
// calls return its value.
class DeviceOnce {
 public:
  template <class F>
  cudaError_t get(int *value, F &&init) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (!done_[dev]) {
      int v = 0;
      e = init(dev, &v);
      if (e != cudaSuccess) return e;
      value_[dev] = v;
      done_[dev] = true;
    }
    if (value) *value = value_[dev];
    return cudaSuccess;
  }

 private:
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
  int value_[kMaxDevices] = {};
};

cudaError_t launch_kv_store(const uint16_t *key, int64_t key_stride, const uint16_t *value,
                            int64_t value_stride, const int64_t *slot_mapping,
                            int32_t num_tokens, int32_t hk, int32_t d, int8_t *k_cache,
                            uint16_t *k_scale, int8_t *v_cache, uint16_t *v_scale,
                            int32_t num_blocks, int32_t block_size, uint32_t *status,
                            cudaStream_t stream);

// The fused store: keys normalized (norm_weight, or none) and rotated (rope,
// or none), then stored with the values as launch_kv_store stores them.
struct KvNormRope {
  const uint16_t *key, *value;
  int64_t key_stride, value_stride;
  const int64_t *slot_mapping, *positions;
  int32_t num_tokens, hk, d;
  const uint16_t *norm_weight;
  float eps;
  const float *rope;  // [max_position][rotary_dim / 2][2] (cos, sin)
  int32_t max_position, rotary_dim;
  bool interleaved;
  int8_t *k_cache, *v_cache;
  uint16_t *k_scale, *v_scale;
  int32_t num_blocks, block_size;
  uint32_t *status;
};

cudaError_t launch_kv_store_norm_rope(const KvNormRope &p, cudaStream_t stream);

// The values of a store whose keys another kernel writes (the fused norm and
// rotation store): kv_store's kernel, value warps only; with `positions`, a
// token whose position is outside [0, max_position) is skipped.
// blocks_per_sm > 0 caps its persistent grid at that many blocks per SM
// (0: as many as are resident).
cudaError_t launch_kv_store_values(const uint16_t *value, int64_t value_stride,
                                   const int64_t *slot_mapping, int32_t num_tokens, int32_t hk,
                                   int32_t d, int8_t *v_cache, uint16_t *v_scale,
                                   int32_t num_blocks, int32_t block_size, uint32_t *status,
                                   const int64_t *positions, int32_t max_position,
                                   cudaStream_t stream, int32_t blocks_per_sm);

// A high-priority side stream of the current device, with fork / join
// events, for work that runs beside the caller's stream.  Created once per
// device; calls from several host threads share it: each holds `mu` from its
// fork record to its join wait, so that another caller's record cannot come
// between its record and its wait (their side work then queues behind one
// another).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
};
cudaError_t side_stream(SideStream **out);

cudaError_t launch_kv_store_f8v4(const uint16_t *key, int64_t key_stride, const uint16_t *value,
                                 int64_t value_stride, const int64_t *slot_mapping,
                                 int32_t num_tokens, int32_t hk, int32_t d, uint8_t *k_cache,
                                 uint8_t *v_cache, uint16_t *v_scale, uint16_t *v_zero,
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
  bool causal = true;          // false: every query sees all seq_len keys
  int32_t window = 0;          // sliding window in keys, 0 = none (causal only)
  const float *sinks = nullptr;  // [hq] sink logits or null
  bool test_timeout = false;   // test hook: decode waits run out after ~1 ms
  // cache format: false = q8; true = fp8 keys and 4-bit values (k_scale
  // unused, v_scale / v_zero one fp16 per key), decode rows only
  bool f8v4 = false;
  const void *v_zero = nullptr;
};

cudaError_t launch_paged_attention(const AttnLaunch &L, cudaStream_t stream);

}  // namespace paq8
