// kv_store: quantize K/V rows to q8 and scatter them into the paged cache
// (K pages token-major, V pages channel-major).
//
// q8 ("shared/attention_kit.py", quantize_q8): per (token, kv head, group of
// 32 channels) s = max(max|x| / 127, 1e-8) in fp32, code =
// clamp(round_half_away(x / s), -127, 127), stored scale = fp16_rne(s).
// Rounding half away from zero as in "shared/kernels/qk_quant_triton.py"
// (_norm_rope_quant), computed exactly (roundf of the IEEE fp32 quotient).
// Scatter ("attention_impl.py", _store_kvcache_nhd): slot < 0 skipped,
// block = slot / block_size, offset = slot % block_size.
//
// One thread per 8 channels of one (token, kv head) row of K and the same 8
// of V: 16-byte loads of bf16, the group max over the 4 threads of a group by
// warp shuffle, 8-byte K code stores and byte stores into the V page rows.
// Memory bound: per (token, kv head) it reads 4*D bytes and writes
// 2*(D + D/16) bytes.
#include "common.cuh"
#include "launch.h"

namespace paq8 {

__device__ __forceinline__ void unpack8(const uint4 v, float (&x)[8]) {
  x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
  x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
  x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

// Codes of 8 values for the group scale s (fp32, IEEE divide, no fast math).
__device__ __forceinline__ uint2 quantize8(const float (&x)[8], float s) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float r = roundf(__fdiv_rn(x[i], s));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    const uint32_t byte = static_cast<uint32_t>(static_cast<int32_t>(r)) & 0xffu;
    w[i >> 2] |= byte << (8 * (i & 3));
  }
  return make_uint2(w[0], w[1]);
}

// fp32 group scale from the group's max |x|: max(amax / 127, 1e-8).
__device__ __forceinline__ float group_scale(float amax) {
  const float s = __fdiv_rn(amax, 127.0f);
  return s < 1e-8f ? 1e-8f : s;
}

template <int D>
__global__ void __launch_bounds__(256) kv_store_kernel(
    const uint16_t *__restrict__ key, int64_t key_stride, const uint16_t *__restrict__ value,
    int64_t value_stride, const int64_t *__restrict__ slot_mapping, int32_t num_tokens,
    int32_t hk, int8_t *__restrict__ k_cache, uint16_t *__restrict__ k_scale,
    int8_t *__restrict__ v_cache, uint16_t *__restrict__ v_scale, int64_t num_slots,
    int32_t block_size, uint32_t *status) {
  constexpr int kChunks = D / 8;   // 8-channel chunks per head row
  constexpr int kGroups = D / 32;
  const int64_t chunks_per_token = static_cast<int64_t>(hk) * kChunks;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = static_cast<int64_t>(num_tokens) * chunks_per_token;
  // Every lane stays to the end: the group max uses full-warp shuffles.  A
  // group's 4 lanes always share one token (kChunks is a multiple of 4).
  const bool in_range = i < total;
  const int64_t n = in_range ? i / chunks_per_token : 0;
  const int32_t c = in_range ? static_cast<int32_t>(i % chunks_per_token) : 0;
  const int32_t h = c / kChunks;
  const int32_t cc = c % kChunks;

  int64_t slot = -1;
  float xk[8], xv[8];
  if (in_range) {
    slot = slot_mapping[n];
    const uint4 k4 = *reinterpret_cast<const uint4 *>(key + n * key_stride + h * D + cc * 8);
    const uint4 v4 = *reinterpret_cast<const uint4 *>(value + n * value_stride + h * D + cc * 8);
    unpack8(k4, xk);
    unpack8(v4, xv);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) xk[e] = xv[e] = 0.0f;
  }
  float ak = 0.0f, av = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ak = fmaxf(ak, fabsf(xk[e]));
    av = fmaxf(av, fabsf(xv[e]));
  }
  ak = fmaxf(ak, __shfl_xor_sync(0xffffffffu, ak, 1));
  ak = fmaxf(ak, __shfl_xor_sync(0xffffffffu, ak, 2));
  av = fmaxf(av, __shfl_xor_sync(0xffffffffu, av, 1));
  av = fmaxf(av, __shfl_xor_sync(0xffffffffu, av, 2));
  if (!in_range || slot < 0) return;
  if (slot >= num_slots) {
    flag_status(status, PA_DEV_BAD_SLOT);
    return;
  }
  const float sk = group_scale(ak);
  const float sv = group_scale(av);
  const int64_t blk = slot / block_size;
  const int64_t off = slot % block_size;
  const int64_t page = blk * hk + h;
  const int64_t row = page * block_size + off;  // K: token-major page row
  *reinterpret_cast<uint2 *>(k_cache + row * D + cc * 8) = quantize8(xk, sk);
  // V: channel-major page, channel c of this token at (page * D + c) * bs + off
  const uint2 vq = quantize8(xv, sv);
  int8_t *vdst = v_cache + (page * D + cc * 8) * block_size + off;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    vdst[e * block_size] = static_cast<int8_t>(((e < 4 ? vq.x : vq.y) >> (8 * (e & 3))) & 0xffu);
  if ((cc & 3) == 0) {
    k_scale[row * kGroups + (cc >> 2)] = __half_as_ushort(__float2half_rn(sk));
    v_scale[(page * kGroups + (cc >> 2)) * block_size + off] =
        __half_as_ushort(__float2half_rn(sv));
  }
}

cudaError_t launch_kv_store(const uint16_t *key, int64_t key_stride, const uint16_t *value,
                            int64_t value_stride, const int64_t *slot_mapping,
                            int32_t num_tokens, int32_t hk, int32_t d, int8_t *k_cache,
                            uint16_t *k_scale, int8_t *v_cache, uint16_t *v_scale,
                            int32_t num_blocks, int32_t block_size, uint32_t *status,
                            cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(num_tokens) * hk * (d / 8);
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
  switch (d) {
#define PAQ8_STORE_CASE(DD)                                                                   \
  case DD:                                                                                    \
    kv_store_kernel<DD><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(               \
        key, key_stride, value, value_stride, slot_mapping, num_tokens, hk, k_cache, k_scale, \
        v_cache, v_scale, num_slots, block_size, status);                                     \
    break;
    PAQ8_STORE_CASE(64)
    PAQ8_STORE_CASE(128)
    PAQ8_STORE_CASE(256)
#undef PAQ8_STORE_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace paq8
