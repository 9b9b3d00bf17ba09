// kv_store with the keys normalized and rotated on the way into the cache:
// the fusion of "shared/kernels/qk_quant_triton.py" (`_norm_rope_quant`,
// `_rows`: weighted RMSNorm with fp32 statistics and its output rounded to
// the activation dtype, then the fp32 rotation of channel pairs, quantized
// from the fp32 rotated values) applied to the q8 cache format.  The values
// are stored as kv_store stores them (kv_store.cu, values-only mode).
//
// Keys: one warp per (token, kv head); lane l holds channels l, l + 32, ...
// (register j = channel l + 32 j), which is also the q8 group layout: group j
// is register j across the 32 lanes.
//  * norm: each lane squares its first channel and adds the next ones with
//    fused multiply-adds (the page's lane sums), the 32 lane sums are added
//    by an xor butterfly (16, 8, 4, 2, 1); inv = 1 / sqrt(total / D + eps)
//    with the square root and the division each rounded once in fp32;
//    y = bf16((x * inv) * w);
//  * rotation: the row goes through shared memory so that every lane reads
//    its pair partner (p with p + rot / 2, or 2p with 2p + 1); lead =
//    fma(cos, y_lead, (-sin) * y_trail), trail = fma(sin, y_lead, cos *
//    y_trail), fp32;
//  * q8: the group max by a warp max-reduction, the code of each lane's value
//    as in kv_store (the product with 1/s, exact near rounding ties).
// Every floating-point step uses an explicitly rounded intrinsic, so that no
// contraction changes a bit: the codes are those of the CPU oracle.
#include "common.cuh"
#include "launch.h"
#include "q8_quant.cuh"

namespace paq8 {

constexpr int kRopeWarps = 8;

template <int D>
__global__ void __launch_bounds__(32 * kRopeWarps) kv_store_norm_rope_kernel(
    const uint16_t *__restrict__ key, int64_t key_stride, const int64_t *__restrict__ slot_mapping,
    const int64_t *__restrict__ positions, int32_t num_tokens, int32_t hk,
    const uint16_t *__restrict__ norm_weight, float eps, const float *__restrict__ rope,
    int32_t max_position, int32_t rot, int32_t interleaved, int8_t *__restrict__ k_cache,
    uint16_t *__restrict__ k_scale, int64_t num_slots, int32_t block_size, uint32_t *status) {
  constexpr int J = D / 32;  // channels per lane, and q8 groups per row
  __shared__ float rowbuf[kRopeWarps][D];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  float *row_s = rowbuf[warp];
  const int64_t units = static_cast<int64_t>(num_tokens) * hk;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kRopeWarps;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * kRopeWarps + warp; u < units; u += stride) {
    const int64_t n = u / hk;
    const int h = static_cast<int>(u % hk);
    const int64_t slot = slot_mapping[n];
    if (slot < 0) continue;  // padding row
    if (slot >= num_slots) {
      if (h == 0 && lane == 0) flag_status(status, PA_DEV_BAD_SLOT);
      continue;
    }
    int64_t pos = 0;
    if (rope) {
      pos = positions[n];
      if (pos < 0 || pos >= max_position) {
        if (h == 0 && lane == 0) flag_status(status, PA_DEV_BAD_POS);
        continue;
      }
    }
    const uint16_t *src = key + n * key_stride + static_cast<int64_t>(h) * D;
    float y[J];
#pragma unroll
    for (int j = 0; j < J; ++j) y[j] = __uint_as_float(static_cast<uint32_t>(src[lane + 32 * j]) << 16);

    // ---- weighted RMSNorm, output rounded to bf16
    if (norm_weight) {
      float acc = __fmul_rn(y[0], y[0]);
#pragma unroll
      for (int j = 1; j < J; ++j) acc = __fmaf_rn(y[j], y[j], acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
      const float inv =
          __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc, static_cast<float>(D)), eps)));
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const float w = __uint_as_float(static_cast<uint32_t>(norm_weight[lane + 32 * j]) << 16);
        const float t = __fmul_rn(__fmul_rn(y[j], inv), w);
        y[j] = __bfloat162float(__float2bfloat16_rn(t));
      }
    }

    // ---- rotation of the first `rot` channels (pairs through shared memory)
    if (rope) {
#pragma unroll
      for (int j = 0; j < J; ++j) row_s[lane + 32 * j] = y[j];
      __syncwarp();
      const float *cs_row = rope + pos * rot;  // [rot / 2][2]: cos, sin
      const int pairs = rot >> 1;
      float out[J];
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int c = lane + 32 * j;
        out[j] = y[j];
        if (c < rot) {
          const bool lead = interleaved ? (c & 1) == 0 : c < pairs;
          const int partner = interleaved ? (c ^ 1) : (lead ? c + pairs : c - pairs);
          const int p = interleaved ? (c >> 1) : (lead ? c : c - pairs);
          const float2 cs = *reinterpret_cast<const float2 *>(cs_row + 2 * p);
          const float other = row_s[partner];
          // lead:  fma(cos, y_lead, (-sin) * y_trail)
          // trail: fma(sin, y_lead, cos * y_trail)
          out[j] = lead ? __fmaf_rn(cs.x, y[j], __fmul_rn(-cs.y, other))
                        : __fmaf_rn(cs.y, other, __fmul_rn(cs.x, y[j]));
        }
      }
      __syncwarp();  // row_s is rewritten for the warp's next unit
#pragma unroll
      for (int j = 0; j < J; ++j) y[j] = out[j];
    }

    // ---- q8 of each group j (register j across the lanes)
    const int64_t blk = slot / block_size, off = slot % block_size;
    const int64_t krow = (blk * hk + h) * block_size + off;
    constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
    constexpr float kFar = 0.5f - 0x1p-15f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      float amax = fabsf(y[j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float sc = group_scale(amax);
      const float rs = __frcp_rn(sc);
      const float q = __fmul_rn(y[j], rs);
      const float t = __fadd_rn(q, kShift);
      int32_t code = static_cast<int32_t>(__float_as_uint(t) & 0xffu);
      // within 2^-15 of a rounding tie: the IEEE quotient's code, exactly
      if (fabsf(__fsub_rn(q, __fsub_rn(t, kShift))) >= kFar) code = tie_code(y[j], sc, rs);
      k_cache[krow * D + 32 * j + lane] = static_cast<int8_t>(code);
      if (lane == 0) k_scale[krow * J + j] = __half_as_ushort(__float2half_rn(sc));
    }
  }
}

cudaError_t launch_kv_store_values(const uint16_t *value, int64_t value_stride,
                                   const int64_t *slot_mapping, int32_t num_tokens, int32_t hk,
                                   int32_t d, int8_t *v_cache, uint16_t *v_scale,
                                   int32_t num_blocks, int32_t block_size, uint32_t *status,
                                   const int64_t *positions, int32_t max_position,
                                   cudaStream_t stream);

template <int D>
static cudaError_t launch_keys(const KvNormRope &p, cudaStream_t stream) {
  static DeviceOnce sm_count;
  int sms = 0;
  cudaError_t e = sm_count.get(&sms, [](int dev, int *v) {
    return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
  });
  if (e != cudaSuccess) return e;
  const int64_t units = static_cast<int64_t>(p.num_tokens) * p.hk;
  const int64_t want = (units + kRopeWarps - 1) / kRopeWarps;
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 8;  // 8 blocks of 256 per SM
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  kv_store_norm_rope_kernel<D><<<grid, 32 * kRopeWarps, 0, stream>>>(
      p.key, p.key_stride, p.slot_mapping, p.positions, p.num_tokens, p.hk, p.norm_weight, p.eps,
      p.rope, p.max_position, p.rotary_dim, p.interleaved ? 1 : 0, p.k_cache, p.k_scale,
      static_cast<int64_t>(p.num_blocks) * p.block_size, p.block_size, p.status);
  return cudaGetLastError();
}

cudaError_t launch_kv_store_norm_rope(const KvNormRope &p, cudaStream_t stream) {
  cudaError_t e = cudaErrorInvalidValue;
  switch (p.d) {
    case 64: e = launch_keys<64>(p, stream); break;
    case 128: e = launch_keys<128>(p, stream); break;
    case 256: e = launch_keys<256>(p, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_kv_store_values(p.value, p.value_stride, p.slot_mapping, p.num_tokens, p.hk, p.d,
                                p.v_cache, p.v_scale, p.num_blocks, p.block_size, p.status,
                                p.rope ? p.positions : nullptr, p.max_position, stream);
}

}  // namespace paq8
