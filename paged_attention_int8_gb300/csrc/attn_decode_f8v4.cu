// Decode kernel for the alternative cache format: fp8 (e4m3) keys and 4-bit
// values with one fp16 scale and zero per key -- the K and V load sites of
// the TurboQuant unified kernel ("triton_turboquant_unified_attention.py":
// `_tq_load_k_tile` reads FP8 keys as their e4m3 values, `_tq_load_v_tile`
// dequantizes V = idx * scale + zero with per-token scale and zero).
//
// The skeleton is the q8 decode kernel's (attn_decode.cu): single-token rows,
// swap-AB warp MMAs (keys in M, the kv head's q heads in N), 4 consumer
// warps on the 16-key blocks of each 64-key tile (32-key tiles at D = 256),
// a producer warp copying whole pages with 16-byte cp.async, split-KV
// segments merged by the segment reduce.  The load site differs:
//  * K: every e4m3 value is exact in fp16 (cvt.rn.f16x2.e4m3x2), so QK^T is
//    one fp32 accumulation over all channels, with no group scales;
//  * V: a channel's 4 consecutive keys are 16 bits of the channel-major
//    nibble page; the nibbles become exact fp16 integers and V' = idx * scale
//    + zero is one fp16 FMA with the keys' own scale and zero.
// Bytes per (key, kv head): D (K) + D / 2 (V) + 4 (scale, zero).
#include "attn_common.cuh"
#include "attn_f8v4.cuh"
#include "launch.h"

namespace paq8 {

template <int D>
struct F8V4Cfg {
  static constexpr int kTile = D == 256 ? 32 : 64;
  static constexpr int kMt = kTile / 16;
  static constexpr int kWpt = kMt < kConsumerWarps ? kMt : kConsumerWarps;
  static constexpr int kKg = kConsumerWarps / kWpt;
  static constexpr int kCm = D / 16;
  static constexpr int G = D / 32;
  static constexpr int kSt = D == 256 ? 4 : 3;
  static constexpr int kMinBlocks = D == 256 ? 2 : 4;
};

template <int D, int BS>
__global__ void __launch_bounds__(kThreads, F8V4Cfg<D>::kMinBlocks)
    decode_f8v4_kernel(const __grid_constant__ AttnArgs a) {
  using Cfg = F8V4Cfg<D>;
  using L = StageF8V4<D, BS, Cfg::kTile>;
  constexpr int G = Cfg::G;
  constexpr int kTile = Cfg::kTile;
  constexpr int kWpt = Cfg::kWpt;
  constexpr int kKg = Cfg::kKg;
  constexpr int kStages = Cfg::kSt;
  static_assert(kStages % kKg == 0, "a stage always feeds the same tile group");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  float *smem_f = reinterpret_cast<float *>(smem_raw + (smem_base - smem_u32(smem_raw)));

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.hk));
  const int rest = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.hk));
  const int seq = rest % a.num_seqs;
  const int sigma = rest / a.num_seqs;

  const int q_start = a.cu_seqlens_q[seq];
  const int q_len = a.cu_seqlens_q[seq + 1] - q_start;
  if (q_len != 1) {  // not a single-token sequence: the generic kernel's, if it runs
    if (q_len > 1 && !a.multi_token_ok && sigma == 0 && h == 0 && threadIdx.x == 0)
      flag_status(a.status, PA_DEV_BAD_SEQ);  // max_query_len hint was below a q_len
    return;
  }
  if (q_start < 0 || q_start >= a.num_tokens) {
    if (threadIdx.x == 0 && sigma == 0) flag_status(a.status, PA_DEV_BAD_SEQ);
    return;
  }
  const int seq_len = a.seq_lens[seq];
  if (seq_len < (a.causal ? 1 : 0)) {
    if (threadIdx.x == 0 && sigma == 0) flag_status(a.status, PA_DEV_BAD_SEQ);
    return;
  }
  if (seq_len == 0) {  // non-causal, no key: out = 0, lse = sink or -inf
    if (sigma == 0 && threadIdx.x < 32)
      write_empty_rows<D>(a, q_start, h * a.qpk, a.qpk, threadIdx.x);
    return;
  }
  const bool split = a.num_splits > 1;
  const int kv_end = seq_len;
  const int kv_begin = first_key(a, seq_len - 1);
  const int first_tile = kv_begin / kTile;
  const int num_tiles = (kv_end + kTile - 1) / kTile;
  int tile_lo = first_tile, tile_hi = num_tiles;
  if (split) {
    if (sigma >= segments_of(kv_begin, kv_end, kTile, a.seg_tiles, a.num_splits)) return;
    tile_lo = first_tile + sigma * a.seg_tiles;
    tile_hi = sigma == a.num_splits - 1 ? num_tiles : min(num_tiles, tile_lo + a.seg_tiles);
  }
  const int n_iter = tile_hi - tile_lo;
  if (n_iter <= 0) return;

  constexpr int kMergeBytes = 3 * 32 * (4 + 4 * Cfg::kCm) * 4;
  constexpr int kRingBytes = kStages * L::kBytes;
  static_assert(kMergeBytes <= kRingBytes, "merge area fits in the ring");
  const uint32_t bar_full = smem_base + kRingBytes;
  const uint32_t bar_empty = bar_full + kStages * 8;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 32);
      mbar_init(bar_empty + 8 * s, kWpt);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    if (!a.test_timeout)
      produce_f8v4<L, BS, kStages>(a, smem_base, bar_full, bar_empty, seq, h, tile_lo, n_iter,
                                   kv_begin, kv_end, lane);
    return;
  }

  const int g = lane >> 2;
  const int t = lane & 3;
  uint32_t qb[G][2][2];
  {
    const bool hv = g < a.qpk;
    const uint16_t *src =
        a.q + (static_cast<int64_t>(q_start) * a.hq + h * a.qpk + (hv ? g : 0)) * D + t * 8;
    bool bad_q = false;
#pragma unroll
    for (int gq = 0; gq < G; ++gq) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (hv) v = *reinterpret_cast<const uint4 *>(src + gq * 32);
      qb[gq][0][0] = pack_half2(bf16_lo(v.x), bf16_hi(v.x));
      qb[gq][0][1] = pack_half2(bf16_lo(v.y), bf16_hi(v.y));
      qb[gq][1][0] = pack_half2(bf16_lo(v.z), bf16_hi(v.z));
      qb[gq][1][1] = pack_half2(bf16_lo(v.w), bf16_hi(v.w));
      bad_q |= half2_nonfinite(qb[gq][0][0]) || half2_nonfinite(qb[gq][0][1]) ||
               half2_nonfinite(qb[gq][1][0]) || half2_nonfinite(qb[gq][1][1]);
    }
    if (__any_sync(0xffffffffu, bad_q) && warp == 0 && lane == 0 && sigma == 0)
      flag_status(a.status, PA_DEV_BAD_Q);
  }
  const int r0 = perm16(g);
  const int r1 = perm16(g + 8);

  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.0f, 0.0f};
  float o[Cfg::kCm][4];
#pragma unroll
  for (int i = 0; i < Cfg::kCm; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.0f;

  const int my_mt = warp % kWpt;
  const int kg = warp / kWpt;
  bool timed_out = false;
  for (int it = kg; it < n_iter; it += kKg) {
    const int stage = it % kStages;
    if (!mbar_wait(bar_full + 8 * stage, (it / kStages) & 1, a.wait_limit_ns)) {
      timed_out = true;
      break;
    }
    const uint32_t st = smem_base + stage * L::kBytes;
    const int key0 = (tile_lo + it) * kTile + my_mt * 16;
    const bool tail = key0 + 16 > kv_end || key0 < kv_begin;
    bool ok0 = true, ok1 = true;  // score rows r0, r1 inside [kv_begin, kv_end)
    if (tail) {
      ok0 = key0 + r0 >= kv_begin && key0 + r0 < kv_end;
      ok1 = key0 + r1 >= kv_begin && key0 + r1 < kv_end;
    }

    // ---------------- S^T = K Q^T, K exact in fp16, one accumulator
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    {
      const int k0 = my_mt * 16 + r0, k1 = my_mt * 16 + r1;
#pragma unroll
      for (int gq = 0; gq < G; ++gq) {
        const uint2 c0 = lds64(st + L::k_off(k0, gq * 32 + t * 8));
        const uint2 c1 = lds64(st + L::k_off(k1, gq * 32 + t * 8));
        // bytes (0,1) -> k 2t, 2t+1; (2,3) -> k 2t+8, 2t+9, as codes4_to_half2
        const uint32_t a00 = e4m3x2_to_half2(c0.x), a02 = e4m3x2_to_half2(c0.x >> 16);
        const uint32_t a01 = e4m3x2_to_half2(c1.x), a03 = e4m3x2_to_half2(c1.x >> 16);
        const uint32_t a10 = e4m3x2_to_half2(c0.y), a12 = e4m3x2_to_half2(c0.y >> 16);
        const uint32_t a11 = e4m3x2_to_half2(c1.y), a13 = e4m3x2_to_half2(c1.y >> 16);
        mma_f16_16816(s, a00, a01, a02, a03, qb[gq][0][0], qb[gq][0][1]);
        mma_f16_16816(s, a10, a11, a12, a13, qb[gq][1][0], qb[gq][1][1]);
      }
    }

    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float v = (e < 2 ? ok0 : ok1) ? s[e] * a.scale_log2 : -INFINITY;
      s[e] = v;
      mx[e & 1] = fmaxf(mx[e & 1], v);
    }
    float alpha[2], mu[2];
    bool grew = false;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
        mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], off));
      const float mn = fmaxf(m_run[c], mx[c]);
      grew |= mn != m_run[c];
      mu[c] = mn == -INFINITY ? 0.0f : mn;
      alpha[c] = fast_exp2(m_run[c] - mu[c]);
      m_run[c] = mn;
    }
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = fast_exp2(s[e] - mu[e & 1]);
    const uint32_t pb0 = movmatrix_trans(pack_half2(p[0], p[1]));
    const uint32_t pb1 = movmatrix_trans(pack_half2(p[2], p[3]));
    if (__any_sync(0xffffffffu, grew)) {
      l_run[0] *= alpha[0];
      l_run[1] *= alpha[1];
#pragma unroll
      for (int i = 0; i < Cfg::kCm; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[1];
        o[i][2] *= alpha[0];
        o[i][3] *= alpha[1];
      }
    }
    l_run[0] += p[0] + p[2];
    l_run[1] += p[1] + p[3];

    // ---------------- O^T += V'^T P^T, V' = idx * scale + zero (fp16), keys 4t..4t+3
    uint2 vsc = lds64(st + L::vs_off(my_mt * 16 + 4 * t));
    uint2 vzr = lds64(st + L::vz_off(my_mt * 16 + 4 * t));
    if (tail) {  // keys outside [kv_begin, kv_end): V' = 0 (stale bytes may sit there)
      const int k = key0 - my_mt * 16 + my_mt * 16 + 4 * t;
      const uint32_t m0 = (k + 0 >= kv_end || k + 0 < kv_begin) ? 0xffff0000u : 0xffffffffu;
      const uint32_t m1 = (k + 1 >= kv_end || k + 1 < kv_begin) ? 0x0000ffffu : 0xffffffffu;
      const uint32_t m2 = (k + 2 >= kv_end || k + 2 < kv_begin) ? 0xffff0000u : 0xffffffffu;
      const uint32_t m3 = (k + 3 >= kv_end || k + 3 < kv_begin) ? 0x0000ffffu : 0xffffffffu;
      vsc.x &= m0 & m1;
      vsc.y &= m2 & m3;
      vzr.x &= m0 & m1;
      vzr.y &= m2 & m3;
    }
#pragma unroll
    for (int cm = 0; cm < Cfg::kCm; ++cm) {
      const uint32_t w0 = lds16(st + L::v_off(cm * 16 + g, my_mt * 16 + 4 * t));
      const uint32_t w1 = lds16(st + L::v_off(cm * 16 + g + 8, my_mt * 16 + 4 * t));
      uint32_t a0, a2, a1, a3;
      nibbles4_to_half2(w0, a0, a2);  // channel g: keys 4t, 4t+1 | 4t+2, 4t+3
      nibbles4_to_half2(w1, a1, a3);  // channel g + 8
      a0 = hfma2_u32(a0, vsc.x, vzr.x);
      a2 = hfma2_u32(a2, vsc.y, vzr.y);
      a1 = hfma2_u32(a1, vsc.x, vzr.x);
      a3 = hfma2_u32(a3, vsc.y, vzr.y);
      mma_f16_16816(o[cm], a0, a1, a2, a3, pb0, pb1);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * stage);
  }
  if (timed_out && lane == 0) flag_status(a.status, PA_DEV_TIMEOUT);

#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l_run[c] += __shfl_xor_sync(0xffffffffu, l_run[c], off);

  constexpr int kFields = 4 + 4 * Cfg::kCm;
  named_barrier(1, kConsumerWarps * 32);
  if (warp > 0) {
    float *dst = smem_f + (warp - 1) * kFields * 32 + lane;
    dst[0] = m_run[0];
    dst[32] = m_run[1];
    dst[64] = l_run[0];
    dst[96] = l_run[1];
#pragma unroll
    for (int i = 0; i < Cfg::kCm; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[(4 + i * 4 + e) * 32] = o[i][e];
  }
  named_barrier(1, kConsumerWarps * 32);
  if (warp > 0) return;
#pragma unroll 1
  for (int k = 0; k < kConsumerWarps - 1; ++k) {
    const float *src = smem_f + k * kFields * 32 + lane;
    float wa[2], wb[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float mo = src[c * 32];
      const float mn = fmaxf(m_run[c], mo);
      const float muv = mn == -INFINITY ? 0.0f : mn;
      wa[c] = fast_exp2(m_run[c] - muv);
      wb[c] = fast_exp2(mo - muv);
      m_run[c] = mn;
      l_run[c] = l_run[c] * wa[c] + src[(2 + c) * 32] * wb[c];
    }
#pragma unroll
    for (int i = 0; i < Cfg::kCm; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o[i][e] = o[i][e] * wa[e & 1] + src[(4 + i * 4 + e) * 32] * wb[e & 1];
  }

  if (a.sinks && sigma == 0) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int hh = min(2 * t + c, a.qpk - 1);
      const float sk = sink_log2(a, h * a.qpk + hh);
      const float mn = fmaxf(m_run[c], sk);
      if (mn == -INFINITY) continue;
      const float wa = fast_exp2(m_run[c] - mn);
      l_run[c] = l_run[c] * wa + fast_exp2(sk - mn);
      m_run[c] = mn;
#pragma unroll
      for (int i = 0; i < Cfg::kCm; ++i) {
        o[i][c] *= wa;
        o[i][2 + c] *= wa;
      }
    }
  }

#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int hh = 2 * t + c;
    if (hh >= a.qpk) continue;
    const int qh = h * a.qpk + hh;
    if (split) {
      const int64_t prow = (static_cast<int64_t>(seq) * a.hq + qh) * a.num_splits + sigma;
      float *dst = a.part_acc + prow * D;
#pragma unroll
      for (int cm = 0; cm < Cfg::kCm; ++cm) {
        dst[cm * 16 + g] = o[cm][c];
        dst[cm * 16 + g + 8] = o[cm][2 + c];
      }
      if (g == 0)
        *reinterpret_cast<float2 *>(a.part_ml + prow * 2) = make_float2(m_run[c], l_run[c]);
    } else {
      const float inv = 1.0f / l_run[c];
      uint16_t *dst = a.out + (static_cast<int64_t>(q_start) * a.hq + qh) * D;
#pragma unroll
      for (int cm = 0; cm < Cfg::kCm; ++cm) {
        dst[cm * 16 + g] = __bfloat16_as_ushort(__float2bfloat16_rn(o[cm][c] * inv));
        dst[cm * 16 + g + 8] = __bfloat16_as_ushort(__float2bfloat16_rn(o[cm][2 + c] * inv));
      }
      if (g == 0 && a.lse)
        a.lse[static_cast<int64_t>(q_start) * a.hq + qh] = (m_run[c] + log2f(l_run[c])) * kLn2;
    }
  }
}

template <int D, int BS>
static cudaError_t launch_f8v4_t(const AttnArgs &a, cudaStream_t stream) {
  using L = StageF8V4<D, BS, F8V4Cfg<D>::kTile>;
  constexpr int kSmem = F8V4Cfg<D>::kSt * L::kBytes + 2 * F8V4Cfg<D>::kSt * 8 + 1024;
  static DeviceOnce configured;
  cudaError_t e = configured.get(nullptr, [](int, int *) {
    return cudaFuncSetAttribute(decode_f8v4_kernel<D, BS>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.num_seqs) * a.num_splits * a.hk, 1);
  decode_f8v4_kernel<D, BS><<<grid, kThreads, kSmem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_f8v4(const AttnArgs &a, int d, int bs, cudaStream_t stream) {
#define PAQ8_F8V4_CASE(DD, BB) \
  if (d == DD && bs == BB) return launch_f8v4_t<DD, BB>(a, stream);
  PAQ8_F8V4_CASE(64, 16)
  PAQ8_F8V4_CASE(64, 32)
  PAQ8_F8V4_CASE(128, 16)
  PAQ8_F8V4_CASE(128, 32)
  PAQ8_F8V4_CASE(256, 16)
  PAQ8_F8V4_CASE(256, 32)
#undef PAQ8_F8V4_CASE
  return cudaErrorInvalidValue;
}

}  // namespace paq8
