// kv_store with the keys normalized and rotated on the way into the cache:
// the fusion of "shared/kernels/qk_quant_triton.py" (`_norm_rope_quant`,
// `_rows`: weighted RMSNorm with fp32 statistics and its output rounded to
// the activation dtype, then the fp32 rotation of channel pairs, quantized
// from the fp32 rotated values) applied to the q8 cache format.  The values
// are stored as kv_store stores them (kv_store.cu, values-only mode).
//
// Keys: one warp per unit = (token, run of its kv heads): all heads of a
// token when they fit 2 KB of bf16 (fewer per unit otherwise), and as many
// as one warp holds at once for a batch too small to fill the GPU that way;
// one block per 8 units, so that the block scheduler balances the work.  A
// warp holds two rows at once (head size up to 128: 16 lanes per row, lane
// l' of a row holding channels l' + 16 j) or one (256: lane l holding
// l + 32 j); the unit's slot, position and cos / sin values are read once
// for all of its heads, the next rows are in flight while some are worked.
//  * norm: the page's 32 lane sums (lane l: channel l squared, then the
//    channels l + 32, l + 64, ... added by fused multiply-adds; with 16
//    lanes per row each lane forms two of them), added by an xor butterfly
//    (16, 8, 4, 2, 1); inv = 1 / sqrt(total / D + eps) with the square root
//    and the reciprocal each rounded once in fp32 (total / D is exact
//    scaling by a power of two); y = bf16((x * inv) * w), two channels at a
//    time in packed fp32 arithmetic;
//  * rotation: lead = fma(cos, y_lead, (-sin) * y_trail), trail = fma(sin,
//    y_lead, cos * y_trail), fp32.  With split-half pairs over the whole row
//    the partner of register j is register j +- J/2 of the same lane; with
//    interleaved pairs it is the neighbouring lane (one shuffle); other
//    split-half rotary dims go through shared memory;
//  * q8: the group maxima by a reduce-scatter over the row's lanes (each
//    lane ends with one group's), one scale and reciprocal per lane,
//    broadcast back; the code of each value as in kv_store (the product with
//    1/s, exact near rounding ties).
// Every floating-point step uses an explicitly rounded intrinsic, so that no
// contraction changes a bit: the codes are those of the CPU oracle.
#include "common.cuh"
#include "launch.h"
#include "q8_quant.cuh"

namespace paq8 {

constexpr int kRopeWarps = 8;
constexpr int kRopeMaxBytes = 2048;          // bf16 keys of one unit, at most
constexpr int64_t kRopeWideUnits = 16384;    // fewer wide units: one warp's rows per unit
constexpr int32_t kRopeOverlapTokens = 4096;  // fewer tokens: keys, then values

enum RopeMode : int {
  kRopeNone = 0,         // norm only
  kRopeHalfFull = 1,     // split-half pairs (p, p + D/2) over the whole row
  kRopeInterleaved = 2,  // pairs (2p, 2p + 1), any rotary dim
  kRopeHalfPart = 3,     // split-half pairs (p, p + rot/2), rot < D
};

// How a warp holds key rows of D channels: R rows at once, LR lanes per
// row, lane l' (of the row's lanes) holding channels l' + LR j, j < J.  The
// 32 per-lane sums of the norm (lane l: channels l, l + 32, ...) are then
// the chains of registers j = k, k + R, k + 2R, ... of lane l' = l % LR for
// k = l / LR, and q8 group g is registers R g .. R g + R - 1 across the
// row's lanes.
template <int D>
struct RowLayout {
  static constexpr int R = D <= 128 ? 2 : 1;  // rows per warp
  static constexpr int LR = 32 / R;           // lanes per row
  static constexpr int J = D / LR;            // channels per lane
  static constexpr int G = D / 32;            // q8 groups per row
  static constexpr int LG = LR / G;           // lanes per group after the reduce-scatter
};

// Max of each of the G values m[g] over the LR lanes of a row,
// reduce-scattered: returns the max of group l' / (LR / G), i.e. the row's
// lanes g * LR/G .. (g+1) * LR/G - 1 hold group g's.  At each of the first
// log2 G steps a lane keeps half of its groups and sends the other half to
// its partner; the remaining steps are a plain butterfly.
template <int G, int LR>
__device__ __forceinline__ float group_max_scatter(float (&m)[G], int lane) {
#pragma unroll
  for (int width = G, bit = LR / 2; width > 1; width >>= 1, bit >>= 1) {
    const bool hi = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < width / 2; ++i) {
      const float send = hi ? m[i] : m[i + width / 2];
      const float keep = hi ? m[i + width / 2] : m[i];
      m[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, bit));
    }
  }
  float r = m[0];
#pragma unroll
  for (int bit = LR / (2 * G); bit > 0; bit >>= 1)
    r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, bit));
  return r;
}

// The rotation constants of one unit (token) for this lane.
template <int J>
struct TokenRope {
  float2 cs[J];  // cos, sin of the pair of register j (split-half: j < J/2)
  uint64_t cos2[J / 4 > 0 ? J / 4 : 1], sin2[J / 4 > 0 ? J / 4 : 1], nsin2[J / 4 > 0 ? J / 4 : 1];
  const float *row;  // the token's [rot / 2][2] table row
};

template <int D, int MODE>
__device__ __forceinline__ void token_rope(TokenRope<RowLayout<D>::J> &tr, const float *rope,
                                           int64_t pos, int rot, int lr) {
  using L = RowLayout<D>;
  constexpr int J = L::J;
  if constexpr (MODE != kRopeNone) {
    tr.row = rope + pos * rot;
    if constexpr (MODE == kRopeHalfFull) {
#pragma unroll
      for (int j = 0; j < J / 2; ++j)
        tr.cs[j] = *reinterpret_cast<const float2 *>(tr.row + 2 * (lr + L::LR * j));
#pragma unroll
      for (int i = 0; i < J / 4; ++i) {
        tr.cos2[i] = f32x2_pack(tr.cs[2 * i].x, tr.cs[2 * i + 1].x);
        tr.sin2[i] = f32x2_pack(tr.cs[2 * i].y, tr.cs[2 * i + 1].y);
        tr.nsin2[i] = f32x2_pack(-tr.cs[2 * i].y, -tr.cs[2 * i + 1].y);
      }
    } else if constexpr (MODE == kRopeInterleaved) {
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int c = lr + L::LR * j;
        tr.cs[j] = c < rot ? *reinterpret_cast<const float2 *>(tr.row + 2 * (c >> 1))
                           : make_float2(1.0f, 0.0f);
      }
    }
  }
}

// Whether the unit's token is stored; flags a bad slot or position once per
// token (by the unit holding head 0).
__device__ __forceinline__ bool token_ok(int64_t slot, int64_t pos, bool has_rope, int h0,
                                         int lane, int64_t num_slots, int32_t max_position,
                                         uint32_t *status) {
  if (slot < 0) return false;  // padding row
  if (slot >= num_slots) {
    if (h0 == 0 && lane == 0) flag_status(status, PA_DEV_BAD_SLOT);
    return false;
  }
  if (has_rope && (pos < 0 || pos >= max_position)) {
    if (h0 == 0 && lane == 0) flag_status(status, PA_DEV_BAD_POS);
    return false;
  }
  return true;
}

// Norm, rotation and q8 of the warp's R key rows (this lane: y, register j =
// channel lr + LR j of its row), the row stored at cache row krow when live.
template <int D, int MODE>
__device__ __forceinline__ void norm_rope_rows(float (&y)[RowLayout<D>::J],
                                               const uint64_t (&wt2)[RowLayout<D>::J / 2],
                                               bool norm, float eps,
                                               const TokenRope<RowLayout<D>::J> &tr, int rot,
                                               float *row_s, int lane, bool live,
                                               int8_t *__restrict__ k_cache,
                                               uint16_t *__restrict__ k_scale, int64_t krow) {
  using L = RowLayout<D>;
  constexpr int J = L::J, R = L::R, LR = L::LR, G = L::G, LG = L::LG;
  const int lr = lane % LR;
  // ---- weighted RMSNorm, output rounded to bf16
  if (norm) {
    float acc[R];  // the per-lane sums of lanes lr + LR k
#pragma unroll
    for (int k = 0; k < R; ++k) {
      acc[k] = __fmul_rn(y[k], y[k]);
#pragma unroll
      for (int j = k + R; j < J; j += R) acc[k] = __fmaf_rn(y[j], y[j], acc[k]);
    }
    // butterfly 16, 8, ..., 1 over the 32 sums: the steps of at least LR
    // combine sums of one lane, the others go across the row's lanes
    float t = acc[0];
    if constexpr (R == 2) t = __fadd_rn(acc[0], acc[1]);
#pragma unroll
    for (int o = LR / 2; o > 0; o >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, o));
    const float inv =
        __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(t, 1.0f / static_cast<float>(D)), eps)));
    const uint64_t inv2 = f32x2_pack(inv, inv);
#pragma unroll
    for (int i = 0; i < J / 2; ++i) {  // two channels at a time
      const uint64_t t2 = f32x2_mul(f32x2_mul(f32x2_pack(y[2 * i], y[2 * i + 1]), inv2), wt2[i]);
      float t0, t1;
      f32x2_unpack(t2, t0, t1);
      const __nv_bfloat162 r = __floats2bfloat162_rn(t0, t1);
      const uint32_t rb = *reinterpret_cast<const uint32_t *>(&r);
      y[2 * i] = bf16_lo(rb);
      y[2 * i + 1] = bf16_hi(rb);
    }
  }

  // ---- rotation
  if constexpr (MODE == kRopeHalfFull) {
#pragma unroll
    for (int i = 0; i < J / 4; ++i) {  // leads 2i, 2i+1 with trails 2i + J/2, 2i+1 + J/2
      const uint64_t lead = f32x2_pack(y[2 * i], y[2 * i + 1]);
      const uint64_t trail = f32x2_pack(y[2 * i + J / 2], y[2 * i + 1 + J / 2]);
      const uint64_t ol = f32x2_fma(tr.cos2[i], lead, f32x2_mul(tr.nsin2[i], trail));
      const uint64_t ot = f32x2_fma(tr.sin2[i], lead, f32x2_mul(tr.cos2[i], trail));
      f32x2_unpack(ol, y[2 * i], y[2 * i + 1]);
      f32x2_unpack(ot, y[2 * i + J / 2], y[2 * i + 1 + J / 2]);
    }
  } else if constexpr (MODE == kRopeInterleaved) {
    const bool is_lead = (lane & 1) == 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const float other = __shfl_xor_sync(0xffffffffu, y[j], 1);
      if (lr + LR * j < rot)
        y[j] = is_lead ? __fmaf_rn(tr.cs[j].x, y[j], __fmul_rn(-tr.cs[j].y, other))
                       : __fmaf_rn(tr.cs[j].y, other, __fmul_rn(tr.cs[j].x, y[j]));
    }
  } else if constexpr (MODE == kRopeHalfPart) {
    float *rs_row = row_s + (lane / LR) * D;
#pragma unroll
    for (int j = 0; j < J; ++j) rs_row[lr + LR * j] = y[j];
    __syncwarp();
    const int pairs = rot >> 1;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = lr + LR * j;
      if (c < rot) {
        const bool is_lead = c < pairs;
        const int p = is_lead ? c : c - pairs;
        const float2 c2 = *reinterpret_cast<const float2 *>(tr.row + 2 * p);
        const float other = rs_row[is_lead ? c + pairs : c - pairs];
        y[j] = is_lead ? __fmaf_rn(c2.x, y[j], __fmul_rn(-c2.y, other))
                       : __fmaf_rn(c2.y, other, __fmul_rn(c2.x, y[j]));
      }
    }
    __syncwarp();  // row_s is rewritten for the next rows
  }

  // ---- q8 of each group g (registers R g .. R g + R - 1 across the row's lanes)
  float m[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = fabsf(y[R * g]);
#pragma unroll
    for (int r = 1; r < R; ++r) m[g] = fmaxf(m[g], fabsf(y[R * g + r]));
  }
  const float my_sc = group_scale(group_max_scatter<G, LR>(m, lane));
  const float my_rs = __frcp_rn(my_sc);
  const int base = lane & ~(LR - 1);  // first lane of the row
  // c = the integer nearest to q = y * (1/s), taken exactly from one fused
  // multiply-add of 1.5 * 2^23 (its low byte is the code); d = q - c from a
  // second one.  Where |d| < 1/2 - 2^-15 the IEEE quotient y / s rounds to c
  // as well (they differ by under 1.6e-5 for |y / s| <= 127.00002); values
  // closer to a tie are decided exactly below.
  constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
  constexpr float kFar = 0.5f - 0x1p-15f;
  const uint64_t shift2 = f32x2_pack(kShift, kShift);
  const uint64_t minus1 = f32x2_pack(-1.0f, -1.0f);
  uint32_t tb[J];
  float d[J], nc[J];
  bool near = false;
#pragma unroll
  for (int i = 0; i < J / 2; ++i) {  // registers 2i, 2i+1: groups (2i) / R, (2i+1) / R
    const float rs_a = __shfl_sync(0xffffffffu, my_rs, base + (2 * i / R) * LG);
    const float rs_b =
        R == 2 ? rs_a : __shfl_sync(0xffffffffu, my_rs, base + ((2 * i + 1) / R) * LG);
    const uint64_t rs2 = f32x2_pack(rs_a, rs_b);
    const uint64_t y2 = f32x2_pack(y[2 * i], y[2 * i + 1]);
    const uint64_t t2 = f32x2_fma(y2, rs2, shift2);      // 1.5 * 2^23 + c
    const uint64_t nc2 = f32x2_fma(t2, minus1, shift2);  // -c, exact
    const uint64_t d2 = f32x2_fma(y2, rs2, nc2);         // y * rs - c
    float t0, t1;
    f32x2_unpack(t2, t0, t1);
    tb[2 * i] = __float_as_uint(t0);
    tb[2 * i + 1] = __float_as_uint(t1);
    f32x2_unpack(d2, d[2 * i], d[2 * i + 1]);
    f32x2_unpack(nc2, nc[2 * i], nc[2 * i + 1]);
    near = near || fabsf(d[2 * i]) >= kFar || fabsf(d[2 * i + 1]) >= kFar;
  }
  // Values within 2^-15 of a tie take the code of the IEEE quotient, decided
  // without a divide from the half-integer h = c + sign(d) / 2 they lie next
  // to (rare: the whole warp takes this branch together).
  if (__any_sync(0xffffffffu, near)) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float sc = __shfl_sync(0xffffffffu, my_sc, base + g * LG);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int j = R * g + r;
        if (fabsf(d[j]) >= kFar) {
          const float hh = __fsub_rn(copysignf(0.5f, d[j]), nc[j]);
          tb[j] = tie_code_bits(y[j], sc, hh);
        }
      }
    }
  }
  if (live) {
    int8_t *dst = k_cache + krow * D + lr;
#pragma unroll
    for (int j = 0; j < J; ++j) dst[LR * j] = static_cast<int8_t>(tb[j] & 0xffu);
    // each group's first lane stores its scale
    if (lr % LG == 0) k_scale[krow * G + lr / LG] = __half_as_ushort(__float2half_rn(my_sc));
  }
}

// grid: one warp per unit (ceil(units / kRopeWarps) blocks, capped; the
// warps then stride on); block: 32 x kRopeWarps; dynamic shared memory:
// kRopeHalfPart, [kRopeWarps][R][D] fp32.  A warp works its unit's heads R
// at a time, head h0 + R i + lane / LR in lanes LR (lane / LR) ...
template <int D, int BS, int MODE>
__global__ void __launch_bounds__(32 * kRopeWarps) kv_store_norm_rope_kernel(
    const uint16_t *__restrict__ key, int64_t key_stride, const int64_t *__restrict__ slot_mapping,
    const int64_t *__restrict__ positions, int32_t num_tokens, int32_t hk, int32_t head_split,
    const uint16_t *__restrict__ norm_weight, float eps, const float *__restrict__ rope,
    int32_t max_position, int32_t rot, int8_t *__restrict__ k_cache,
    uint16_t *__restrict__ k_scale, int64_t num_slots, uint32_t *status) {
  using L = RowLayout<D>;
  constexpr int J = L::J, R = L::R, LR = L::LR;
  extern __shared__ __align__(16) float rope_rows[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int lr = lane % LR;
  const int my_row = lane / LR;
  float *row_s = rope_rows + warp * R * D;
  const bool norm = norm_weight != nullptr;
  constexpr bool kHasRope = MODE != kRopeNone;

  uint64_t wt2[J / 2];  // norm weights of the lane's channel pairs (registers 2i, 2i + 1)
  if (norm) {
#pragma unroll
    for (int i = 0; i < J / 2; ++i)
      wt2[i] = f32x2_pack(bf16_lo(norm_weight[lr + LR * (2 * i)]),
                          bf16_lo(norm_weight[lr + LR * (2 * i + 1)]));
  }
  const int heads_per = (hk + head_split - 1) / head_split;
  const int64_t units = static_cast<int64_t>(num_tokens) * head_split;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kRopeWarps;
  TokenRope<J> tr;
#pragma unroll 1
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * kRopeWarps + warp; u < units; u += stride) {
    // token and first head of unit u
    int64_t n = u;
    int h0 = 0;
    if (head_split > 1) {
      n = u / head_split;
      h0 = static_cast<int>(u - n * head_split) * heads_per;
    }
    const int h1 = min(h0 + heads_per, hk);
    const int64_t slot = slot_mapping[n];
    const int64_t pos = kHasRope && slot >= 0 && slot < num_slots ? positions[n] : 0;
    if (h0 >= h1 || !token_ok(slot, pos, kHasRope, h0, lane, num_slots, max_position, status))
      continue;
    token_rope<D, MODE>(tr, rope, pos, rot, lr);
    const uint64_t us = static_cast<uint64_t>(slot);
    const int64_t blk = static_cast<int64_t>(us / BS), off = static_cast<int64_t>(us % BS);
    const uint16_t *src = key + n * key_stride + lr;
    uint16_t nxt[J];
    {
      const int h = h0 + my_row;
#pragma unroll
      for (int j = 0; j < J; ++j) nxt[j] = h < h1 ? src[static_cast<int64_t>(h) * D + LR * j] : 0;
    }
#pragma unroll 1
    for (int hb = h0; hb < h1; hb += R) {
      const int h = hb + my_row;
      float y[J];
#pragma unroll
      for (int j = 0; j < J; ++j) y[j] = bf16_lo(nxt[j]);
      const int hn = h + R;
      if (hb + R < h1) {  // the next rows, in flight while these are worked
#pragma unroll
        for (int j = 0; j < J; ++j)
          nxt[j] = hn < h1 ? src[static_cast<int64_t>(hn) * D + LR * j] : 0;
      }
      norm_rope_rows<D, MODE>(y, wt2, norm, eps, tr, rot, row_s, lane, h < h1, k_cache, k_scale,
                              (blk * hk + h) * BS + off);
    }
  }
}

template <int D, int BS, int MODE>
static cudaError_t launch_keys(const KvNormRope &p, cudaStream_t stream) {
  constexpr int smem = MODE == kRopeHalfPart ? kRopeWarps * RowLayout<D>::R * D * 4 : 0;
  // the shared-memory carveout of the values kernel, so that the blocks of
  // both can be resident on one SM together
  static DeviceOnce carveout;
  int unused = 0;
  cudaError_t e = carveout.get(&unused, [](int, int *v) {
    *v = 0;
    return cudaFuncSetAttribute(kv_store_norm_rope_kernel<D, BS, MODE>,
                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
  });
  if (e != cudaSuccess) return e;
  // units of a token's heads (as many as fit kRopeMaxBytes) when that makes
  // enough units to fill the GPU; otherwise one warp's rows (R heads) per unit
  constexpr int kMaxHeads = kRopeMaxBytes / (2 * D);
  const int wide_split = (p.hk + kMaxHeads - 1) / kMaxHeads;
  const int64_t wide_units = static_cast<int64_t>(p.num_tokens) * wide_split;
  constexpr int R = RowLayout<D>::R;
  const int head_split = wide_units >= kRopeWideUnits ? wide_split : (p.hk + R - 1) / R;
  const int64_t units = static_cast<int64_t>(p.num_tokens) * head_split;
  const int64_t want = (units + kRopeWarps - 1) / kRopeWarps;
  const unsigned grid = static_cast<unsigned>(want < (1 << 30) ? want : (1 << 30));
  kv_store_norm_rope_kernel<D, BS, MODE><<<grid, 32 * kRopeWarps, smem, stream>>>(
      p.key, p.key_stride, p.slot_mapping, p.positions, p.num_tokens, p.hk, head_split,
      p.norm_weight, p.eps, p.rope, p.max_position, p.rotary_dim, p.k_cache, p.k_scale,
      static_cast<int64_t>(p.num_blocks) * p.block_size, p.status);
  return cudaGetLastError();
}

template <int D, int BS>
static cudaError_t launch_keys_mode(const KvNormRope &p, cudaStream_t stream) {
  if (!p.rope) return launch_keys<D, BS, kRopeNone>(p, stream);
  if (p.interleaved) return launch_keys<D, BS, kRopeInterleaved>(p, stream);
  if (p.rotary_dim == D) return launch_keys<D, BS, kRopeHalfFull>(p, stream);
  return launch_keys<D, BS, kRopeHalfPart>(p, stream);
}

static cudaError_t launch_keys_any(const KvNormRope &p, cudaStream_t stream) {
#define PAQ8_ROPE_CASE(DD, BB) \
  if (p.d == DD && p.block_size == BB) return launch_keys_mode<DD, BB>(p, stream);
  PAQ8_ROPE_CASE(64, 16)
  PAQ8_ROPE_CASE(64, 32)
  PAQ8_ROPE_CASE(128, 16)
  PAQ8_ROPE_CASE(128, 32)
  PAQ8_ROPE_CASE(256, 16)
  PAQ8_ROPE_CASE(256, 32)
#undef PAQ8_ROPE_CASE
  return cudaErrorInvalidValue;
}

// The values (kv_store's kernel, light on instructions and bound by memory)
// run on the high-priority side stream beside the keys (bound by
// instruction issue), one block per SM, so that the two overlap: their
// blocks are resident together and the keys' many short blocks take what the
// values leave.  A small batch (or a side stream that cannot be had) runs
// the two one after the other on `stream`.
cudaError_t launch_kv_store_norm_rope(const KvNormRope &p, cudaStream_t stream) {
  if (p.num_tokens == 0) return cudaSuccess;
  const int32_t max_pos = p.max_position;
  const int64_t *vpos = p.rope ? p.positions : nullptr;
  SideStream *ss = nullptr;
  if (p.num_tokens >= kRopeOverlapTokens && side_stream(&ss) == cudaSuccess) {
    std::lock_guard<std::mutex> lock(ss->mu);  // fork record .. join wait
    cudaError_t e;
    if ((e = cudaEventRecord(ss->fork, stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss->s, ss->fork, 0)) != cudaSuccess) return e;
    if ((e = launch_kv_store_values(p.value, p.value_stride, p.slot_mapping, p.num_tokens, p.hk,
                                    p.d, p.v_cache, p.v_scale, p.num_blocks, p.block_size,
                                    p.status, vpos, max_pos, ss->s, 1)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(ss->join, ss->s)) != cudaSuccess) return e;
    const cudaError_t ek = launch_keys_any(p, stream);
    // the join is waited for even when the keys failed to launch
    if ((e = cudaStreamWaitEvent(stream, ss->join, 0)) != cudaSuccess) return e;
    return ek;
  }
  cudaError_t e = launch_keys_any(p, stream);
  if (e != cudaSuccess) return e;
  return launch_kv_store_values(p.value, p.value_stride, p.slot_mapping, p.num_tokens, p.hk, p.d,
                                p.v_cache, p.v_scale, p.num_blocks, p.block_size, p.status, vpos,
                                max_pos, stream, 0);
}

}  // namespace paq8
