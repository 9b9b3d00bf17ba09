// kv_store for the alternative cache format of the TurboQuant unified kernel
// ("triton_turboquant_unified_attention.py": FP8 keys read as their e4m3
// values; 4-bit values read as idx * scale + zero with one fp16 scale and zero
// per token).  The page shows only the load sites; the store is:
//   K: e4m3 of each bf16 value, round to nearest even, saturating at +-448;
//   V: per (token, kv head) lo = min, hi = max over the D channels (fp32),
//      s = max((hi - lo) / 15, 1e-8), idx = clamp(round_half_away((x - lo) / s),
//      0, 15) of the IEEE fp32 quotient, scale = fp16(s), zero = fp16(lo).
// Caches (head-major pages):
//   k_cache uint8 [num_blocks][hk][bs][D]       e4m3, token-major
//   v_cache uint8 [num_blocks][hk][D][bs / 2]   channel-major nibbles: byte j
//                                               of a channel row holds keys 2j
//                                               (low nibble) and 2j + 1
//   v_scale, v_zero fp16 [num_blocks][hk][bs]
//
// Work units: (32 consecutive tokens, kv head), once for the keys and once
// for the values, one warp each (even warps keys, odd warps values).  Keys:
// token by token, the lanes on consecutive D/32-channel pieces of the row
// (one coalesced load and store per row, eight rows in flight).  Values:
// lane = token.  Two tokens whose slots share a nibble byte (offsets 2j,
// 2j + 1 of one page) and sit in the same warp -- consecutive tokens of a
// prefill chunk -- are written together by the even one; a token whose byte
// mate is not in the warp updates its nibbles with 32-bit atomics (so a mate
// in another warp or from an earlier call is never overwritten).
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "q8_quant.cuh"

namespace paq8 {

constexpr int kF8v4Warps = 8;
constexpr int kNibStride = 34;  // nibble words per row of the staging area: 32 lanes + 2 outside mates

// two fp32 -> e4m3x2 (x0 in byte 0), round to nearest even, saturating
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float x0, float x1) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(x1), "f"(x0));
  return d;
}

// The 4-bit code of x in a row with minimum lo and step s (rs = 1/s):
// round_half_away((x - lo) / s) of the IEEE quotient (the product with 1/s,
// exact near ties), clamped to [0, 15].
// (the rare near-tie decision is a call, so that the unrolled code of a row
// stays small)
__device__ __noinline__ int32_t v4_tie(float v, float s, float rs) { return tie_code(v, s, rs); }

__device__ __forceinline__ uint32_t v4_code(float x, float lo, float s, float rs) {
  constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
  constexpr float kFar = 0.5f - 0x1p-15f;
  const float v = __fsub_rn(x, lo);
  const float q = __fmul_rn(v, rs);
  const float t = __fadd_rn(q, kShift);
  int32_t code = static_cast<int32_t>(__float_as_uint(t) & 0xffu);
  if (fabsf(__fsub_rn(q, __fsub_rn(t, kShift))) >= kFar) code = v4_tie(v, s, rs);
  return static_cast<uint32_t>(min(max(code, 0), 15));
}

// The step of a row from its extremes: max((hi - lo) / 15, 1e-8).
__device__ __forceinline__ float v4_step(float lo, float hi) {
  const float s = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
  return s < 1e-8f ? 1e-8f : s;
}

// The nibbles of value row `row` (one token, one kv head), computed by the
// whole warp (lane l: channels l * D/32 ...) and written as D / 8 words to
// col[0], col[stride], ... (shared memory): the nibbles of a token just
// outside the warp's 32 whose byte mate is a lane of this warp.  The same
// arithmetic as a lane's own row, so the same codes.
template <int D>
__device__ __forceinline__ void v4_row_by_warp(const uint16_t *__restrict__ row, int lane,
                                               uint32_t *col, int stride) {
  constexpr int C = D / 32;  // channels per lane
  float x[C];
  if constexpr (C == 2) {
    const uint32_t a = *reinterpret_cast<const uint32_t *>(row + lane * C);
    x[0] = bf16_lo(a);
    x[1] = bf16_hi(a);
  } else if constexpr (C == 4) {
    const uint2 a = *reinterpret_cast<const uint2 *>(row + lane * C);
    x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
  } else {
    const uint4 a = *reinterpret_cast<const uint4 *>(row + lane * C);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_lo(w[i]);
      x[2 * i + 1] = bf16_hi(w[i]);
    }
  }
  float lo = x[0], hi = x[0];
#pragma unroll
  for (int i = 1; i < C; ++i) {
    lo = fminf(lo, x[i]);
    hi = fmaxf(hi, x[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  const float s = v4_step(lo, hi);
  const float rs = __frcp_rn(s);
  uint32_t chunk = 0u;  // 4C bits: this lane's channels
#pragma unroll
  for (int i = 0; i < C; ++i) chunk |= v4_code(x[i], lo, s, rs) << (4 * i);
  // lane l's chunk is the (l % (8 / C))-th C/2-byte piece of word l / (8 / C)
  constexpr int kLanesPerWord = 8 / C;
  uint8_t *dst = reinterpret_cast<uint8_t *>(col + (lane / kLanesPerWord) * stride) +
                 (lane % kLanesPerWord) * (C / 2);
  if constexpr (C == 2) *dst = static_cast<uint8_t>(chunk);
  else if constexpr (C == 4) *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(chunk);
  else *reinterpret_cast<uint32_t *>(dst) = chunk;
}

template <int D>
__global__ void __launch_bounds__(32 * kF8v4Warps) kv_store_f8v4_kernel(
    const uint16_t *__restrict__ key, int64_t key_stride, const uint16_t *__restrict__ value,
    int64_t value_stride, const int64_t *__restrict__ slot_mapping, int32_t num_tokens,
    int32_t hk, uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
    uint16_t *__restrict__ v_scale, uint16_t *__restrict__ v_zero, int64_t num_slots,
    int32_t block_size, uint32_t *status) {
  constexpr int W = D / 8;  // nibble words of a row (8 channels each)
  __shared__ uint32_t nib_s[kF8v4Warps][W][kNibStride];
  const int lane = threadIdx.x & 31;
  const int n_tblocks = (num_tokens + 31) / 32;
  const int64_t units = static_cast<int64_t>(n_tblocks) * hk * 2;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kF8v4Warps;
  const int bs_log2 = block_size == 32 ? 5 : 4;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * kF8v4Warps + (threadIdx.x >> 5); u < units;
       u += stride) {
    const bool keys = (u & 1) == 0;
    const int h = static_cast<int>((u >> 1) % hk);
    const int64_t tb = (u >> 1) / hk;
    const int64_t n = tb * 32 + lane;
    int64_t slot = n < num_tokens ? slot_mapping[n] : -1;
    if (slot >= num_slots) {
      if (h == 0 && !keys) flag_status(status, PA_DEV_BAD_SLOT);
      slot = -1;
    }
    const bool active = slot >= 0;

    if (keys) {
      // ---- keys: e4m3 of each value; token t of the block at a time, lane l
      // on channels l * KC .. l * KC + KC - 1 (eight rows in flight)
      constexpr int KC = D / 32;
      using Piece = std::conditional_t<KC == 2, uint32_t, std::conditional_t<KC == 4, uint2, uint4>>;
#pragma unroll 1
      for (int t0 = 0; t0 < 32; t0 += 8) {
        Piece a[8];
        int64_t row[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int64_t st = __shfl_sync(0xffffffffu, slot, t0 + i);
          row[i] = -1;
          if (st >= 0) {
            const int64_t nt = tb * 32 + t0 + i;
            a[i] = *reinterpret_cast<const Piece *>(key + nt * key_stride +
                                                     static_cast<int64_t>(h) * D + lane * KC);
            row[i] = (((st >> bs_log2) * hk + h) << bs_log2) + (st & (block_size - 1));
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (row[i] < 0) continue;
          uint8_t *kd = k_cache + row[i] * D + lane * KC;
          if constexpr (KC == 2) {
            *reinterpret_cast<uint16_t *>(kd) =
                static_cast<uint16_t>(f32x2_to_e4m3x2(bf16_lo(a[i]), bf16_hi(a[i])));
          } else if constexpr (KC == 4) {
            *reinterpret_cast<uint32_t *>(kd) =
                f32x2_to_e4m3x2(bf16_lo(a[i].x), bf16_hi(a[i].x)) |
                (f32x2_to_e4m3x2(bf16_lo(a[i].y), bf16_hi(a[i].y)) << 16);
          } else {
            *reinterpret_cast<uint2 *>(kd) =
                make_uint2(f32x2_to_e4m3x2(bf16_lo(a[i].x), bf16_hi(a[i].x)) |
                               (f32x2_to_e4m3x2(bf16_lo(a[i].y), bf16_hi(a[i].y)) << 16),
                           f32x2_to_e4m3x2(bf16_lo(a[i].z), bf16_hi(a[i].z)) |
                               (f32x2_to_e4m3x2(bf16_lo(a[i].w), bf16_hi(a[i].w)) << 16));
          }
        }
      }
      continue;
    }
    const int64_t blk = active ? slot / block_size : 0, off = active ? slot % block_size : 0;
    const int64_t page = blk * hk + h;

    // ---- values: 4-bit codes with the row's scale and zero.  The nibble
    // words go through shared memory (word i of lane l at nib[i][l]), so that
    // the loops below stay rolled (small code) and a byte mate's words are a
    // plain load.
    uint32_t(*nib)[kNibStride] = nib_s[threadIdx.x >> 5];
    if (active) {
      const uint16_t *vs = value + n * value_stride + static_cast<int64_t>(h) * D;
      float lo = INFINITY, hi = -INFINITY;
#pragma unroll 4
      for (int c = 0; c < D; c += 8) {
        const uint4 a = *reinterpret_cast<const uint4 *>(vs + c);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          lo = fmin3(lo, bf16_lo(w[i]), bf16_hi(w[i]));
          hi = fmax3(hi, bf16_lo(w[i]), bf16_hi(w[i]));
        }
      }
      const float s = v4_step(lo, hi);
      const float rs = __frcp_rn(s);
      // The code of v = x - lo: c, the integer nearest to v * (1/s), from one
      // fused multiply-add of 1.5 * 2^23 (its low nibble), and d = v * (1/s)
      // - c from a second, two values at a time; values within 2^-15 of a
      // tie take the IEEE quotient's code exactly (as v4_code).  No clamp is
      // needed: 0 <= v <= RN(hi - lo), so 0 <= v * (1/s) < 15.00001.
      constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
      constexpr float kFar = 0.5f - 0x1p-15f;
      const uint64_t nlo2 = f32x2_pack(-lo, -lo), rs2 = f32x2_pack(rs, rs);
      const uint64_t shift2 = f32x2_pack(kShift, kShift), minus1 = f32x2_pack(-1.0f, -1.0f);
#pragma unroll 1
      for (int c = 0; c < D; c += 8) {
        const uint4 a = *reinterpret_cast<const uint4 *>(vs + c);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
        uint32_t word = 0u;
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // channels 4 half .. 4 half + 3
          uint32_t tb[4];
          float v[4], d[4], nc[4];
          bool near = false;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint32_t ww = w[2 * half + i];
            const uint64_t v2 = f32x2_add(f32x2_pack(bf16_lo(ww), bf16_hi(ww)), nlo2);  // x - lo
            const uint64_t t2 = f32x2_fma(v2, rs2, shift2);      // 1.5 * 2^23 + c
            const uint64_t nc2 = f32x2_fma(t2, minus1, shift2);  // -c, exact
            const uint64_t d2 = f32x2_fma(v2, rs2, nc2);         // v * rs - c
            float t0, t1;
            f32x2_unpack(t2, t0, t1);
            tb[2 * i] = __float_as_uint(t0);
            tb[2 * i + 1] = __float_as_uint(t1);
            f32x2_unpack(v2, v[2 * i], v[2 * i + 1]);
            f32x2_unpack(d2, d[2 * i], d[2 * i + 1]);
            f32x2_unpack(nc2, nc[2 * i], nc[2 * i + 1]);
            near = near || fabsf(d[2 * i]) >= kFar || fabsf(d[2 * i + 1]) >= kFar;
          }
          if (near) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (fabsf(d[i]) >= kFar)
                tb[i] = tie_code_bits(v[i], s, __fsub_rn(copysignf(0.5f, d[i]), nc[i]));
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) word |= (tb[i] & 0xfu) << (16 * half + 4 * i);
        }
        nib[c / 8][lane] = word;
      }
      v_scale[page * block_size + off] = __half_as_ushort(__float2half_rn(s));
      v_zero[page * block_size + off] = __half_as_ushort(__float2half_rn(lo));
    }

    // ---- nibble bytes: pair the two tokens of a byte when both are here
    const uint32_t pair_mask = __match_any_sync(0xffffffffu, active ? (slot >> 1) : -1 - lane);
    const bool paired = __popc(pair_mask) == 2;
    int mate = paired ? __ffs(pair_mask & ~(1u << lane)) - 1 : lane;
    // A stretch of consecutive slots that crosses the warp's first or last
    // token (a chunk starting mid-pair) leaves lane 0 or 31 without its mate
    // in the warp, while the mate is the token just outside: the warp then
    // computes that token's nibbles into column 32 + side, and the lane
    // writes the whole byte -- as does the warp that owns the mate, with the
    // same value.
    bool outer = false;
#pragma unroll
    for (int side = 0; side < 2; ++side) {
      const int src = side == 0 ? 0 : 31;
      const int64_t nm = n + (side == 0 ? -1 : 1);  // the mate token (lane src)
      bool want = false;
      if (lane == src && active && !paired && ((off & 1) != 0) == (side == 0) && nm >= 0 &&
          nm < num_tokens)
        want = slot_mapping[nm] == (side == 0 ? slot - 1 : slot + 1);
      if (!__shfl_sync(0xffffffffu, want, src)) continue;  // warp-uniform
      const int64_t row_m = __shfl_sync(0xffffffffu, nm, src);
      v4_row_by_warp<D>(value + row_m * value_stride + static_cast<int64_t>(h) * D, lane,
                        &nib[0][32 + side], kNibStride);
      if (lane == src) {
        outer = true;
        mate = 32 + side;
      }
    }
    __syncwarp();  // every lane's words (and the outer columns) are in place
    if (active && (outer || paired)) {
      // the even-offset token of an in-warp pair writes the byte; an edge
      // lane writes it with the outside mate's nibbles
      if (outer || !(off & 1)) {
        const bool odd = off & 1;  // the low nibble is the even-offset token's
        uint8_t *vrow = v_cache + page * D * (block_size / 2) + off / 2;  // channel 0's byte
#pragma unroll 1
        for (int i = 0; i < W; ++i) {
          const uint32_t own = nib[i][lane], other = nib[i][mate];
          const uint32_t lo_w = odd ? other : own, hi_w = odd ? own : other;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            vrow[static_cast<int64_t>(8 * i + j) * (block_size / 2)] = static_cast<uint8_t>(
                ((lo_w >> (4 * j)) & 0xfu) | (((hi_w >> (4 * j)) & 0xfu) << 4));
        }
      }
    } else if (active) {
      // the byte mate is not in this call: update this token's nibbles alone
      uint8_t *vrow = v_cache + page * D * (block_size / 2) + off / 2;
#pragma unroll 1
      for (int c = 0; c < D; ++c) {
        const uint32_t v4 = (nib[c / 8][lane] >> (4 * (c % 8))) & 0xfu;
        uint8_t *byte = vrow + static_cast<int64_t>(c) * (block_size / 2);
        unsigned int *word = reinterpret_cast<unsigned int *>(
            reinterpret_cast<uintptr_t>(byte) & ~static_cast<uintptr_t>(3));
        const uint32_t shift = 8u * static_cast<uint32_t>(reinterpret_cast<uintptr_t>(byte) & 3u) +
                               4u * static_cast<uint32_t>(off & 1);
        atomicAnd(word, ~(0xfu << shift));
        atomicOr(word, v4 << shift);
      }
    }
    __syncwarp();  // the words are rewritten for the warp's next unit
  }
}

cudaError_t launch_kv_store_f8v4(const uint16_t *key, int64_t key_stride, const uint16_t *value,
                                 int64_t value_stride, const int64_t *slot_mapping,
                                 int32_t num_tokens, int32_t hk, int32_t d, uint8_t *k_cache,
                                 uint8_t *v_cache, uint16_t *v_scale, uint16_t *v_zero,
                                 int32_t num_blocks, int32_t block_size, uint32_t *status,
                                 cudaStream_t stream) {
  static DeviceOnce sm_count;
  int sms = 0;
  cudaError_t e = sm_count.get(&sms, [](int dev, int *v) {
    return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
  });
  if (e != cudaSuccess) return e;
  const int64_t units = static_cast<int64_t>((num_tokens + 31) / 32) * hk * 2;
  const int64_t want = (units + kF8v4Warps - 1) / kF8v4Warps;
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
#define PAQ8_F8V4_STORE(DD)                                                                       \
  case DD:                                                                                        \
    kv_store_f8v4_kernel<DD><<<grid, 32 * kF8v4Warps, 0, stream>>>(                               \
        key, key_stride, value, value_stride, slot_mapping, num_tokens, hk, k_cache, v_cache,     \
        v_scale, v_zero, num_slots, block_size, status);                                          \
    break;
  switch (d) {
    PAQ8_F8V4_STORE(64)
    PAQ8_F8V4_STORE(128)
    PAQ8_F8V4_STORE(256)
    default:
      return cudaErrorInvalidValue;
  }
#undef PAQ8_F8V4_STORE
  return cudaGetLastError();
}

}  // namespace paq8
