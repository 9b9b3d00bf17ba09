// Decode kernel: sequences with a single query token, their q heads (up to
// 8 per kv head) attending one KV segment each.
//
// Computes, for the token's q heads h of kv head hk (GQA: h / qpk == hk),
// the online-softmax triple of "triton_turboquant_unified_attention.py"
// (3D split-KV kernel): m = max_j s_j, l = sum_j exp(s_j - m),
// acc = sum_j exp(s_j - m) v_j over the segment's keys, s_j = scale * q.k_j.
// Unsplit, it writes out = acc / l and lse = m + ln l directly.
// The visible keys are [kv_begin, seq_len): kv_begin = seq_len - window with
// a sliding window ("attention_impl.py", window_size = (window - 1, 0)),
// else 0.  A sink logit (the USE_SINKS rule of the same Triton page) joins
// the denominator of segment 0 only, as one term with no value.
//
// Swap-AB form: with one token the GQA group has only qpk <= 8 rows, so the
// keys take the MMA's M dimension and the heads its N dimension:
//   S^T[16 keys x 8 heads]  = K[16 keys x 16 ch] . Q^T[16 ch x 8 heads]
//   O^T[16 ch x 8 heads]   += V^T[16 ch x 16 keys] . P^T[16 keys x 8 heads]
// K codes are exact fp16 integers; each 32-channel group's partial scores are
// scaled by the group's fp16 K scale in fp32.  V^T comes straight from the
// channel-major V pages (4 consecutive keys per 32-bit load) and is scaled to
// fp16.  P^T reaches the B-operand layout with one movmatrix per 8x8 block.
//
// CTA = 4 consumer warps, each taking one 16-key block of every 64-key tile
// (D = 256: 32-key tiles, two warps per tile, pairs alternate tiles), with
// private softmax states merged at the end, plus one producer warp whose 32
// lanes copy each tile's pages with 16-byte cp.async (a small page would
// otherwise cost four TMA requests, and the per-request cost, not bandwidth,
// limited the stream).
// Grid: num_splits * num_seqs * num_kv_heads CTAs, segment-major (then
// sequence, then kv head).
#include "attn_common.cuh"
#include "launch.h"

namespace paq8 {

// The G fp16 K scales of one key row (contiguous) as floats.
template <int G>
__device__ __forceinline__ void load_scales_row(uint32_t addr, float (&f)[G]) {
  uint32_t w[G / 2];
  if constexpr (G == 2) {
    w[0] = lds32(addr);
  } else if constexpr (G == 4) {
    const uint2 v = lds64(addr);
    w[0] = v.x;
    w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < G / 8; ++i) {
      const uint4 v = lds128(addr + 16 * i);
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
  }
#pragma unroll
  for (int i = 0; i < G / 2; ++i) {
    const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}

template <int D>
struct DecodeCfg {
  static constexpr int kTile = D == 256 ? 32 : 64;
  static constexpr int kMt = kTile / 16;   // 16-key blocks per tile
  static constexpr int kWpt = kMt < kConsumerWarps ? kMt : kConsumerWarps;  // warps per tile
  static constexpr int kKg = kConsumerWarps / kWpt;  // tile groups (alternate tiles)
  static constexpr int kCm = D / 16;       // 16-channel blocks of the output
  static constexpr int G = D / 32;
  static constexpr int kSt = D == 256 ? 4 : 3;          // ring stages
  static constexpr int kMinBlocks = D == 256 ? 2 : 4;   // CTAs per SM
};

template <int D, int BS>
__global__ void __launch_bounds__(kThreads, DecodeCfg<D>::kMinBlocks)
    decode_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v) {
  using Cfg = DecodeCfg<D>;
  using L = StageLayout<D, BS, Cfg::kTile>;
  constexpr int G = Cfg::G;
  constexpr int kTile = Cfg::kTile;
  constexpr int kWpt = Cfg::kWpt;
  constexpr int kKg = Cfg::kKg;
  constexpr int kStages = Cfg::kSt;
  static_assert(kStages % kKg == 0, "a stage always feeds the same tile group");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  float *smem_f = reinterpret_cast<float *>(smem_raw + (smem_base - smem_u32(smem_raw)));

  // a dependent launched with programmatic serialization (the segment
  // reduce) may be scheduled once every CTA of this grid has started; it
  // still waits for this grid to finish before reading what it wrote
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // segment-major order: every sequence's first segment (and all kv heads)
  // launches before any second segment, so the partial last segments of the
  // longest sequences, not full ones, are what the final wave holds
  const int h = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.hk));
  const int rest = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.hk));
  const int seq = rest % a.num_seqs;
  const int sigma = rest / a.num_seqs;

  const int q_start = a.cu_seqlens_q[seq];
  const int q_len = a.cu_seqlens_q[seq + 1] - q_start;
  if (q_len != 1) {  // not a single-token sequence: the prefill kernel's, if it runs
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
      mbar_init(bar_full + 8 * s, 32);  // one arrival per producer lane
      mbar_init(bar_empty + 8 * s, kWpt);  // every warp of the tile group reads it
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // test hook: stage nothing, so that every consumer wait runs out
    if (!a.test_timeout)
      produce_tiles_lsu<L, BS, kStages>(a, smem_base, bar_full, bar_empty, seq, h, tile_lo,
                                        n_iter, kv_begin, kv_end, lane);
    return;
  }

  const int g = lane >> 2;
  const int t = lane & 3;

  // Q^T as the B operand: lane (g, t) holds head g, channels 32gq + 8t + 4s +
  // {0,1} (k = 2t, 2t+1) and + {2,3} (k = 2t+8, 2t+9) for k-step s.
  uint32_t qb[G][2][2];
  {
    const bool hv = g < a.qpk;
    const uint16_t *src =
        a.q + (static_cast<int64_t>(q_start) * a.hq + h * a.qpk + (hv ? g : 0)) * D + t * 8;
#pragma unroll
    bool bad_q = false;
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
    // q values beyond the fp16 range (|q| >= 65520) would give inf scores
    if (__any_sync(0xffffffffu, bad_q) && warp == 0 && lane == 0 && sigma == 0)
      flag_status(a.status, PA_DEV_BAD_Q);
  }
  const int r0 = perm16(g);      // key (within a 16-key block) of score row g
  const int r1 = perm16(g + 8);  // ... of score row g + 8

  float m_run[2] = {-INFINITY, -INFINITY};  // heads 2t, 2t+1 (log2 units)
  float l_run[2] = {0.0f, 0.0f};            // this lane's share of the expsum
  float o[Cfg::kCm][4];                     // O^T: channels (g, g+8) x heads (2t, 2t+1)
#pragma unroll
  for (int i = 0; i < Cfg::kCm; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.0f;

  // Warp w takes the 16-key block mt = w % kWpt of every tile of its tile
  // group (w / kWpt): all warps read every stage, so the whole ring is in
  // flight for each of them.
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
    const int key0 = (tile_lo + it) * kTile + my_mt * 16;  // first key of this warp's block
    // keys outside [kv_begin, kv_end) in this block: masked, V scales zeroed
    // (stale bytes may sit there).  The lane's validity masks -- score rows
    // r0, r1 and V keys 4t .. 4t+3 -- are formed once per tile, on edge
    // tiles only, and applied without compares elsewhere.
    const bool tail = key0 + 16 > kv_end || key0 < kv_begin;
    bool ok0 = true, ok1 = true;
    uint2 vmask = make_uint2(0xffffffffu, 0xffffffffu);
    if (tail) {
      const auto in = [&](int k) { return k >= kv_begin && k < kv_end; };
      ok0 = in(key0 + r0);
      ok1 = in(key0 + r1);
      const int kv = key0 + 4 * t;
      vmask.x = (in(kv) ? 0x0000ffffu : 0u) | (in(kv + 1) ? 0xffff0000u : 0u);
      vmask.y = (in(kv + 2) ? 0x0000ffffu : 0u) | (in(kv + 3) ? 0xffff0000u : 0u);
    }

    // ---------------- S^T = K Q^T with exact codes, scaled per group
    float s[4];
    {
      const int k0 = my_mt * 16 + r0, k1 = my_mt * 16 + r1;
      float ks0[G], ks1[G];
      load_scales_row<G>(st + L::ks_off(k0, 0), ks0);
      load_scales_row<G>(st + L::ks_off(k1, 0), ks1);
#pragma unroll
      for (int e = 0; e < 4; ++e) s[e] = 0.0f;
#pragma unroll
      for (int gq = 0; gq < G; ++gq) {
        const uint2 c0 = lds64(st + L::k_off(k0, gq * 32 + t * 8));
        const uint2 c1 = lds64(st + L::k_off(k1, gq * 32 + t * 8));
        uint32_t a00, a02, a01, a03, a10, a12, a11, a13;
        codes4_to_half2(c0.x, a00, a02);  // row g, k-step 0: (k 2t,2t+1), (k 2t+8,2t+9)
        codes4_to_half2(c1.x, a01, a03);  // row g+8
        codes4_to_half2(c0.y, a10, a12);  // k-step 1
        codes4_to_half2(c1.y, a11, a13);
        float sg[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_f16_16816(sg, a00, a01, a02, a03, qb[gq][0][0], qb[gq][0][1]);
        mma_f16_16816(sg, a10, a11, a12, a13, qb[gq][1][0], qb[gq][1][1]);
        s[0] = fmaf(sg[0], ks0[gq], s[0]);
        s[1] = fmaf(sg[1], ks0[gq], s[1]);
        s[2] = fmaf(sg[2], ks1[gq], s[2]);
        s[3] = fmaf(sg[3], ks1[gq], s[3]);
      }
    }

    // ---------------- mask the tail, online softmax over keys (rows)
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
    const uint32_t pb0 = movmatrix_trans(pack_half2(p[0], p[1]));  // keys 0..7 -> k 2t, 2t+1
    const uint32_t pb1 = movmatrix_trans(pack_half2(p[2], p[3]));  // keys 8..15 -> k 2t+8, 2t+9
    // rescale only when some head's running max moved (alpha == 1 otherwise)
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

    // ---------------- O^T += V'^T P^T, V' = code * scale in fp16
#pragma unroll
    for (int gv = 0; gv < G; ++gv) {
      uint2 vsc = lds64(st + L::vs_off(my_mt * 16 + 4 * t, gv));
      vsc.x &= vmask.x;
      vsc.y &= vmask.y;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int cm = gv * 2 + half;
        const uint32_t w0 = lds32(st + L::v_off(cm * 16 + g, my_mt * 16 + 4 * t));
        const uint32_t w1 = lds32(st + L::v_off(cm * 16 + g + 8, my_mt * 16 + 4 * t));
        uint32_t a0, a2, a1, a3;
        codes4_to_half2(w0, a0, a2);  // channel g: keys 4t..4t+1 | 4t+2..4t+3
        codes4_to_half2(w1, a1, a3);  // channel g + 8
        a0 = hmul2_u32(a0, vsc.x);
        a2 = hmul2_u32(a2, vsc.y);
        a1 = hmul2_u32(a1, vsc.x);
        a3 = hmul2_u32(a3, vsc.y);
        mma_f16_16816(o[cm], a0, a1, a2, a3, pb0, pb1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * stage);
  }
  if (timed_out && lane == 0) flag_status(a.status, PA_DEV_TIMEOUT);

  // expsum of each head: sum over the 8 lanes that share t
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l_run[c] += __shfl_xor_sync(0xffffffffu, l_run[c], off);

  // ---------------- merge the 4 warps (field-major through shared memory)
  constexpr int kFields = 4 + 4 * Cfg::kCm;
  named_barrier(1, kConsumerWarps * 32);  // every stage consumed: reuse the ring
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

  // ---------------- the sink joins segment 0 as one term (m = sink, l = 1, no value)
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

  // ---------------- write: lane (g, t) holds channels cm*16 + g (+8) of heads 2t, 2t+1
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
cudaError_t launch_decode_t(const AttnArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                            cudaStream_t stream) {
  using L = StageLayout<D, BS, DecodeCfg<D>::kTile>;
  constexpr int kSmem = DecodeCfg<D>::kSt * L::kBytes + 2 * DecodeCfg<D>::kSt * 8 + 1024;
  static DeviceOnce configured;
  cudaError_t e = configured.get(nullptr, [](int, int *) {
    return cudaFuncSetAttribute(decode_kernel<D, BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmem);
  });
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.num_seqs) * a.num_splits * a.hk, 1);
  decode_kernel<D, BS><<<grid, kThreads, kSmem, stream>>>(a, tk, tv);
  return cudaGetLastError();
}

int decode_tile(int d) { return d == 256 ? 32 : 64; }

cudaError_t launch_decode(const AttnArgs &a, const CUtensorMap &tk, const CUtensorMap &tv, int d,
                          int bs, cudaStream_t stream) {
#define PAQ8_DECODE_CASE(DD, BB) \
  if (d == DD && bs == BB) return launch_decode_t<DD, BB>(a, tk, tv, stream);
  PAQ8_DECODE_CASE(64, 16)
  PAQ8_DECODE_CASE(64, 32)
  PAQ8_DECODE_CASE(128, 16)
  PAQ8_DECODE_CASE(128, 32)
  PAQ8_DECODE_CASE(256, 16)
  PAQ8_DECODE_CASE(256, 32)
#undef PAQ8_DECODE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace paq8
