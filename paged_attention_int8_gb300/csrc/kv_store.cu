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
// One thread per (token, kv head, 32-channel group) of K or of V -- one q8
// scale -- with the 32 lanes of a warp on 32 consecutive tokens: the
// group max is a per-thread reduction, K rows go out as 16-byte stores, and
// the byte stores into the channel-major V pages (and the V scale stores)
// coalesce across lanes whenever consecutive tokens fill consecutive slots
// of a page (prefill chunks, cache population).  The quotient x / s is
// formed as x * (1/s) and rounded there unless it lies within 2^-12 of a
// rounding tie, where the IEEE quotient decides (the two differ by less than
// 2.3e-5 for |x / s| <= 127.00001).
// Memory bound: per (token, kv head) it reads 4*D bytes and writes
// 2*(D + D/16) bytes.
#include "common.cuh"
#include "launch.h"

namespace paq8 {

// fp32 group scale from the group's max |x|: max(amax / 127, 1e-8).
__device__ __forceinline__ float group_scale(float amax) {
  const float s = __fdiv_rn(amax, 127.0f);
  return s < 1e-8f ? 1e-8f : s;
}

// Exact q8 code of x for the group scale s: clamp(round_half_away(x / s)).
__device__ __forceinline__ int32_t code_exact(float x, float s) {
  const float r = fminf(fmaxf(roundf(__fdiv_rn(x, s)), -127.0f), 127.0f);
  return static_cast<int32_t>(r);
}

// Codes of 32 values (4-byte words, little-endian) for scale s and its
// correctly rounded reciprocal rs.
__device__ __forceinline__ void quantize32(const float (&x)[32], float s, float rs,
                                           uint32_t (&w)[8]) {
  uint32_t near = 0u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float q = x[i] * rs;
    const float a = fabsf(q);
    const float fl = floorf(a);
    const float f = a - fl;
    // |frac - 1/2| < 2^-12, or a non-finite quotient: let the IEEE divide decide
    if (!(fabsf(f - 0.5f) >= 0x1p-12f)) near |= 1u << i;
    const float m = fminf(fl + (f >= 0.5f ? 1.0f : 0.0f), 127.0f);
    const int32_t c = static_cast<int32_t>(copysignf(m, q));
    if ((i & 3) == 0) w[i >> 2] = 0u;
    w[i >> 2] |= (static_cast<uint32_t>(c) & 0xffu) << (8 * (i & 3));
  }
  if (near) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((near >> i) & 1u) {
        const uint32_t c = static_cast<uint32_t>(code_exact(x[i], s)) & 0xffu;
        const int sh = 8 * (i & 3);
        w[i >> 2] = (w[i >> 2] & ~(0xffu << sh)) | (c << sh);
      }
    }
  }
}

__device__ __forceinline__ void load32(const uint16_t *p, float (&x)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = *reinterpret_cast<const uint4 *>(p + 8 * j);
    x[8 * j + 0] = bf16_lo(v.x); x[8 * j + 1] = bf16_hi(v.x);
    x[8 * j + 2] = bf16_lo(v.y); x[8 * j + 3] = bf16_hi(v.y);
    x[8 * j + 4] = bf16_lo(v.z); x[8 * j + 5] = bf16_hi(v.z);
    x[8 * j + 6] = bf16_lo(v.w); x[8 * j + 7] = bf16_hi(v.w);
  }
}

constexpr int kStoreWarps = 8;

// grid: (ceil(num_tokens / 32), ceil(2 * hk * D/32 / kStoreWarps)); block: 32 x
// kStoreWarps.  Warp (blockIdx.y * kStoreWarps + w) takes one (kv head, group)
// of K (even) or of V (odd) for 32 consecutive tokens.
template <int D>
__global__ void __launch_bounds__(32 * kStoreWarps) kv_store_kernel(
    const uint16_t *__restrict__ key, int64_t key_stride, const uint16_t *__restrict__ value,
    int64_t value_stride, const int64_t *__restrict__ slot_mapping, int32_t num_tokens,
    int32_t hk, int8_t *__restrict__ k_cache, uint16_t *__restrict__ k_scale,
    int8_t *__restrict__ v_cache, uint16_t *__restrict__ v_scale, int64_t num_slots,
    int32_t block_size, uint32_t *status) {
  constexpr int G = D / 32;
  const int lane = threadIdx.x & 31;
  const int combo = blockIdx.y * kStoreWarps + (threadIdx.x >> 5);
  const int64_t n = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  if (combo >= 2 * hk * G || n >= num_tokens) return;
  const bool is_v = combo & 1;
  const int h = (combo >> 1) / G, g = (combo >> 1) % G;
  const int64_t slot = slot_mapping[n];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (combo == 0) flag_status(status, PA_DEV_BAD_SLOT);
    return;
  }
  float x[32];
  uint32_t w[8];
  const int64_t blk = slot / block_size;
  const int64_t off = slot % block_size;
  const int64_t page = blk * hk + h;
  if (!is_v) {
    // K: token-major page row, 32 codes of group g; scale [page][bs][G]
    load32(key + n * key_stride + h * D + g * 32, x);
  } else {
    load32(value + n * value_stride + h * D + g * 32, x);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float sc = group_scale(amax);
  quantize32(x, sc, __frcp_rn(sc), w);
  const uint16_t sbits = __half_as_ushort(__float2half_rn(sc));
  if (!is_v) {
    const int64_t row = page * block_size + off;
    uint4 *kdst = reinterpret_cast<uint4 *>(k_cache + row * D + g * 32);
    kdst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    kdst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    k_scale[row * G + g] = sbits;
  } else {
    // V: channel-major page, channel c of this token at (page * D + c) * bs + off;
    // scale [page][G][bs]
    int8_t *vdst = v_cache + (page * D + g * 32) * block_size + off;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      vdst[static_cast<int64_t>(i) * block_size] =
          static_cast<int8_t>((w[i >> 2] >> (8 * (i & 3))) & 0xffu);
    v_scale[(page * G + g) * block_size + off] = sbits;
  }
}

cudaError_t launch_kv_store(const uint16_t *key, int64_t key_stride, const uint16_t *value,
                            int64_t value_stride, const int64_t *slot_mapping,
                            int32_t num_tokens, int32_t hk, int32_t d, int8_t *k_cache,
                            uint16_t *k_scale, int8_t *v_cache, uint16_t *v_scale,
                            int32_t num_blocks, int32_t block_size, uint32_t *status,
                            cudaStream_t stream) {
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
  const dim3 block(32 * kStoreWarps);
  const dim3 grid(static_cast<unsigned>((num_tokens + 31) / 32),
                  static_cast<unsigned>((2 * hk * (d / 32) + kStoreWarps - 1) / kStoreWarps));
  switch (d) {
#define PAQ8_STORE_CASE(DD)                                                                   \
  case DD:                                                                                    \
    kv_store_kernel<DD><<<grid, block, 0, stream>>>(                                          \
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
