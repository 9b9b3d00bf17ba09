// Generic (prefill) kernel: unified causal attention for q-blocks of
// BLOCK_Q tokens x the q heads of one kv head, stacked as the GQA row tile of
// "triton_turboquant_unified_attention.py" (unified 2D kernel): row m is token
// m / qpk, q head kv * qpk + m % qpk.  For query token i of a sequence
//   out = softmax_j(scale * q . k_j) v_j over keys j <= seq_len - q_len + i,
//   lse = ln sum_j exp(scale * q . k_j),
// with the dequantized q8 rows of the kv head read page by page.  In
// non-causal mode every query sees keys j < seq_len; a sliding window keeps
// the last `window` of a query's keys; a sink logit joins the denominator
// (the options of the AttnArgs visibility fields).
//
// CTA = one q-block x one kv head (x one segment for split single-token
// rows), 5 warps: warp 4 stages each 64-key tile's pages through a 4-deep
// mbarrier ring (16-byte cp.async copies from all 32 lanes); warps 0-3 take the
// rows in groups of 16 (R groups; the 4/R warps sharing a group alternate
// tiles with private softmax states, merged at the end).  QK^T runs on the
// exact integer codes (fp16) per 32-channel group, scaled by the group's K
// scale in fp32; PV multiplies P (fp16) by V' = code * scale (fp16), read
// from the channel-major V pages 4 keys per 32-bit load.
// The same kernel reads the fp8-key / 4-bit-value format (F8): QK^T in one
// accumulation over all channels (e4m3 keys are exact in fp16, no group
// scales), V' = idx * scale + zero per key, pages copied by that format's
// producer.
#include <type_traits>

#include "attn_common.cuh"
#include "attn_f8v4.cuh"
#include "launch.h"

namespace paq8 {

constexpr int kTile = 64;  // keys per pipeline stage

template <int D, int BS, bool F8>
struct AttnCfg {
  using L = std::conditional_t<F8, StageF8V4<D, BS, kTile>, StageLayout<D, BS, kTile>>;
  static constexpr int G = D / 32;
  static constexpr int kQBytes = 4 * G * 2 * 32 * 16;  // fragment-ordered q, 4 row groups
  static constexpr int kQOff = kStages * L::kBytes;
  static constexpr int kBarOff = kQOff + kQBytes;
  static constexpr int kSmemBytes = kBarOff + 2 * kStages * 8 + 1024;  // + alignment slack
  // merge area (inside the stages) per partner warp: m0 m1 l0 l1 + O
  static constexpr int kMergeFields = 4 + 4 * 4 * G;
  static_assert(3 * kMergeFields * 32 * 4 <= kStages * L::kBytes, "merge area");
};

template <int D, int BS, bool F8>
__global__ void __launch_bounds__(kThreads) prefill_kernel(const __grid_constant__ AttnArgs a,
                                                           const __grid_constant__ CUtensorMap tmap_k,
                                                           const __grid_constant__ CUtensorMap tmap_v) {
  using C = AttnCfg<D, BS, F8>;
  using L = typename C::L;
  constexpr int G = C::G;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (smem_base - smem_u32(smem_raw));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y;  // kv head

  // ---- which sequence, which tokens, which keys
  int seq, tok0, sigma;
  const int bx = blockIdx.x;
  if (bx < a.n_qblocks) {
    seq = find_seq(a.cu_seqlens_q, a.num_seqs, a.block_q, bx, lane);
    const int c0 = a.cu_seqlens_q[seq];
    const int first = a.block_q == 1 ? c0 : c0 / a.block_q + seq;
    tok0 = (bx - first) * a.block_q;
    sigma = 0;
  } else {  // continuation segments of single-token sequences
    const int r = bx - a.n_qblocks;
    seq = r / (a.num_splits - 1);
    sigma = 1 + r % (a.num_splits - 1);
    tok0 = 0;
  }
  const int q_start = a.cu_seqlens_q[seq];
  const int q_end = a.cu_seqlens_q[seq + 1];
  const int q_len = q_end - q_start;
  if (tok0 >= q_len) return;
  if (q_len == 1 && a.skip_single) return;  // the decode kernel owns these rows
  if (q_end > a.num_tokens || q_start < 0) {
    if (threadIdx.x == 0 && sigma == 0) flag_status(a.status, PA_DEV_BAD_SEQ);
    return;
  }
  const int seq_len = a.seq_lens[seq];
  const int ctx = seq_len - q_len;
  if (a.causal ? ctx < 0 : seq_len < 0) {
    if (threadIdx.x == 0 && sigma == 0 && tok0 == 0) flag_status(a.status, PA_DEV_BAD_SEQ);
    return;
  }
  const bool split = a.num_splits > 1 && q_len == 1;
  if (!split && sigma > 0) return;
  const int n_tok = min(a.block_q, q_len - tok0);
  const int n_rows = n_tok * a.qpk;
  // keys visible to some row of the block: [kv_begin, kv_end)
  const int kv_end = last_key(a, seq_len, q_len, tok0 + n_tok - 1) + 1;
  const int kv_begin = first_key(a, last_key(a, seq_len, q_len, tok0));
  if (kv_end == 0) {  // non-causal, seq_len == 0: no row sees a key
    if (sigma == 0 && warp < 4)
      for (int idx = warp; idx < n_tok; idx += 4)
        write_empty_rows<D>(a, q_start + tok0 + idx, h * a.qpk, a.qpk, lane);
    return;
  }
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
  const int R = n_rows <= 16 ? 1 : (n_rows <= 32 ? 2 : 4);
  const int KG = kConsumerWarps / R;

  const uint32_t bar_full = smem_base + C::kBarOff;
  const uint32_t bar_empty = bar_full + kStages * 8;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 32);  // one arrival per producer lane
      mbar_init(bar_empty + 8 * s, R);  // a tile is consumed by the R warps of one kv group
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    if constexpr (F8)
      produce_f8v4<L, BS, kStages>(a, smem_base, bar_full, bar_empty, seq, h, tile_lo, n_iter,
                                   kv_begin, kv_end, lane);
    else
      produce_tiles_lsu<L, BS>(a, smem_base, bar_full, bar_empty, seq, h, tile_lo, n_iter,
                               kv_begin, kv_end, lane);
    return;
  }

  // ================================================================== consumers
  const int rg = warp % R;
  const int kg = warp / R;
  const int g = lane >> 2;
  const int t = lane & 3;
  const uint32_t q_frag = smem_base + C::kQOff;

  // q -> fp16 A fragments in MMA order: [row group][group][k-step][lane] x 16 B.
  // Channel order inside a k-step: cols 2t, 2t+1 <- 32gq + 8t + 4s + {0,1},
  // cols 2t+8, 2t+9 <- 32gq + 8t + 4s + {2,3}; K rows use the same order.
  if (warp < R) {
    bool bad_q = false;
#pragma unroll
    for (int gq = 0; gq < G; ++gq) {
      uint32_t f[2][4];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int idx = warp * 16 + g + 8 * half;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (idx < n_rows) {
          const int tq = idx / a.qpk;
          const int hh = h * a.qpk + idx % a.qpk;
          const uint16_t *src = a.q + (static_cast<int64_t>(q_start + tok0 + tq) * a.hq + hh) * D +
                                gq * 32 + t * 8;
          v = *reinterpret_cast<const uint4 *>(src);
        }
        f[0][half] = pack_half2(bf16_lo(v.x), bf16_hi(v.x));
        f[0][2 + half] = pack_half2(bf16_lo(v.y), bf16_hi(v.y));
        f[1][half] = pack_half2(bf16_lo(v.z), bf16_hi(v.z));
        f[1][2 + half] = pack_half2(bf16_lo(v.w), bf16_hi(v.w));
        bad_q |= half2_nonfinite(f[0][half]) || half2_nonfinite(f[0][2 + half]) ||
                 half2_nonfinite(f[1][half]) || half2_nonfinite(f[1][2 + half]);
      }
#pragma unroll
      for (int s = 0; s < 2; ++s)
        sts128(q_frag + (((warp * G + gq) * 2 + s) * 32 + lane) * 16,
               make_uint4(f[s][0], f[s][1], f[s][2], f[s][3]));
    }
    // q values beyond the fp16 range (|q| >= 65520) would give inf scores
    if (__any_sync(0xffffffffu, bad_q) && lane == 0 && sigma == 0)
      flag_status(a.status, PA_DEV_BAD_Q);
  }
  named_barrier(1, kConsumerWarps * 32);

  // visible keys [lo, lim] of rows g and g + 8; padding rows copy the
  // block's last row so their arithmetic stays finite
  int lim[2], lo[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int idx = rg * 16 + g + 8 * half;
    lim[half] = idx < n_rows ? last_key(a, seq_len, q_len, tok0 + idx / a.qpk) : kv_end - 1;
    lo[half] = first_key(a, lim[half]);
  }
  int min_lim = min(lim[0], lim[1]);
  int max_lo = max(lo[0], lo[1]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    min_lim = min(min_lim, __shfl_xor_sync(0xffffffffu, min_lim, o));
    max_lo = max(max_lo, __shfl_xor_sync(0xffffffffu, max_lo, o));
  }

  // key (within its 16-key block) of score column n of an even / odd n-tile
  const int kc0 = perm16(2 * t), kc1 = perm16(2 * t + 1);  // even n-tile, cols 2t, 2t+1
  const int kr_even = perm16(g), kr_odd = perm16(8 + g);    // K rows this lane loads

  float m_run[2] = {-INFINITY, -INFINITY};  // running max, log2 units
  float l_run[2] = {0.0f, 0.0f};            // this lane's share of the expsum
  float o_acc[4 * G][4];                    // n-tile (gq, j): channels 32gq + 8j + 2t + {0,1}
#pragma unroll
  for (int i = 0; i < 4 * G; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o_acc[i][e] = 0.0f;

  bool timed_out = false;
  for (int it = kg; it < n_iter; it += KG) {
    const int stage = it % kStages;
    if (!mbar_wait(bar_full + 8 * stage, (it / kStages) & 1, a.wait_limit_ns)) {
      timed_out = true;
      break;
    }
    const uint32_t st = smem_base + stage * L::kBytes;
    const int key0 = (tile_lo + it) * kTile;

    // ---------------- S = q k^T, exact codes, per-group scale
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] = 0.0f;
#pragma unroll
    for (int gq = 0; gq < G; ++gq) {
      const uint4 qa0 = lds128(q_frag + (((rg * G + gq) * 2 + 0) * 32 + lane) * 16);
      const uint4 qa1 = lds128(q_frag + (((rg * G + gq) * 2 + 1) * 32 + lane) * 16);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int kb16 = (nt >> 1) * 16;
        const uint2 kw = lds64(st + L::k_off(kb16 + ((nt & 1) ? kr_odd : kr_even), gq * 32 + t * 8));
        if constexpr (F8) {  // e4m3 bytes (0,1) -> k 2t, 2t+1; (2,3) -> k 2t+8, 2t+9
          mma_f16_16816(sc[nt], qa0.x, qa0.y, qa0.z, qa0.w, e4m3x2_to_half2(kw.x),
                        e4m3x2_to_half2(kw.x >> 16));
          mma_f16_16816(sc[nt], qa1.x, qa1.y, qa1.z, qa1.w, e4m3x2_to_half2(kw.y),
                        e4m3x2_to_half2(kw.y >> 16));
        } else {
          uint32_t b0, b1, b2, b3;
          codes4_to_half2(kw.x, b0, b1);
          codes4_to_half2(kw.y, b2, b3);
          float sg[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          mma_f16_16816(sg, qa0.x, qa0.y, qa0.z, qa0.w, b0, b1);
          mma_f16_16816(sg, qa1.x, qa1.y, qa1.z, qa1.w, b2, b3);
          const int off = (nt & 1) ? 2 : 0;  // odd n-tiles hold keys 4t+2, 4t+3
          const float s0 = __half2float(__ushort_as_half(lds16(st + L::ks_off(kb16 + kc0 + off, gq))));
          const float s1 = __half2float(__ushort_as_half(lds16(st + L::ks_off(kb16 + kc1 + off, gq))));
          sc[nt][0] = fmaf(sg[0], s0, sc[nt][0]);
          sc[nt][1] = fmaf(sg[1], s1, sc[nt][1]);
          sc[nt][2] = fmaf(sg[2], s0, sc[nt][2]);
          sc[nt][3] = fmaf(sg[3], s1, sc[nt][3]);
        }
      }
    }

    // ---------------- mask, online softmax (log2 domain)
    const bool need_mask = key0 + kTile - 1 > min_lim || key0 < max_lo;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sc[nt][e] * a.scale_log2;
        if (need_mask) {
          const int key = key0 + (nt >> 1) * 16 + ((e & 1) ? kc1 : kc0) + ((nt & 1) ? 2 : 0);
          if (key > lim[e >> 1] || key < lo[e >> 1]) v = -INFINITY;
        }
        sc[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    float alpha[2], mu[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mn = fmaxf(m_run[r], mx[r]);
      mu[r] = mn == -INFINITY ? 0.0f : mn;
      alpha[r] = fast_exp2(m_run[r] - mu[r]);
      m_run[r] = mn;
      l_run[r] *= alpha[r];
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = fast_exp2(sc[nt][e] - mu[e >> 1]);
        sc[nt][e] = p;
        l_run[e >> 1] += p;
      }
#pragma unroll
    for (int i = 0; i < 4 * G; ++i) {
      o_acc[i][0] *= alpha[0];
      o_acc[i][1] *= alpha[0];
      o_acc[i][2] *= alpha[1];
      o_acc[i][3] *= alpha[1];
    }

    // ---------------- O += P V', V' = code * scale in fp16 from channel-major pages
    const bool tail = key0 + kTile > kv_end || key0 < kv_begin;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t pa0 = pack_half2(sc[2 * kk][0], sc[2 * kk][1]);
      const uint32_t pa1 = pack_half2(sc[2 * kk][2], sc[2 * kk][3]);
      const uint32_t pa2 = pack_half2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      const uint32_t pa3 = pack_half2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
      if constexpr (F8) {
        // the 4 keys 4t .. 4t+3 of this 16-key block: their scales and zeros
        // (zeroed outside [kv_begin, kv_end): stale bytes may sit there)
        uint2 vsc = lds64(st + L::vs_off(kk * 16 + 4 * t));
        uint2 vzr = lds64(st + L::vz_off(kk * 16 + 4 * t));
        if (tail) {
          const int k = key0 + kk * 16 + 4 * t;
          const auto in = [&](int x) { return x >= kv_begin && x < kv_end; };
          const uint32_t mx = (in(k) ? 0x0000ffffu : 0u) | (in(k + 1) ? 0xffff0000u : 0u);
          const uint32_t my = (in(k + 2) ? 0x0000ffffu : 0u) | (in(k + 3) ? 0xffff0000u : 0u);
          vsc.x &= mx;
          vzr.x &= mx;
          vsc.y &= my;
          vzr.y &= my;
        }
#pragma unroll
        for (int c8 = 0; c8 < D / 8; ++c8) {
          const uint32_t w = lds16(st + L::v_off(c8 * 8 + g, kk * 16 + 4 * t));
          uint32_t b0, b1;
          nibbles4_to_half2(w, b0, b1);  // keys 4t, 4t+1 | 4t+2, 4t+3
          mma_f16_16816(o_acc[c8], pa0, pa1, pa2, pa3, hfma2_u32(b0, vsc.x, vzr.x),
                        hfma2_u32(b1, vsc.y, vzr.y));
        }
      } else {
#pragma unroll
        for (int gq = 0; gq < G; ++gq) {
          const uint2 vsc = v_scales4<L>(st, kk * 16 + 4 * t, gq, tail, key0, kv_begin, kv_end);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint32_t w = lds32(st + L::v_off(gq * 32 + jj * 8 + g, kk * 16 + 4 * t));
            uint32_t b0, b1;
            codes4_to_half2(w, b0, b1);  // keys 4t, 4t+1 -> k 2t, 2t+1; 4t+2, 4t+3 -> k 2t+8, 2t+9
            mma_f16_16816(o_acc[gq * 4 + jj], pa0, pa1, pa2, pa3, hmul2_u32(b0, vsc.x),
                          hmul2_u32(b1, vsc.y));
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * stage);
  }
  if (timed_out && lane == 0) flag_status(a.status, PA_DEV_TIMEOUT);

  // row expsums: sum the 4 lanes of a row
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
  }

  // ---------------- merge the KG warps of a row group (field-major, no conflicts)
  if (KG > 1) {
    named_barrier(1, kConsumerWarps * 32);  // every stage consumed: reuse them
    float *mbuf = reinterpret_cast<float *>(smem);
    if (kg > 0) {
      float *dst = mbuf + (warp - R) * C::kMergeFields * 32 + lane;
      dst[0 * 32] = m_run[0];
      dst[1 * 32] = m_run[1];
      dst[2 * 32] = l_run[0];
      dst[3 * 32] = l_run[1];
#pragma unroll
      for (int i = 0; i < 4 * G; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[(4 + i * 4 + e) * 32] = o_acc[i][e];
    }
    named_barrier(1, kConsumerWarps * 32);
    if (kg > 0) return;
    for (int k = 1; k < KG; ++k) {
      const float *src = mbuf + (rg + k * R - R) * C::kMergeFields * 32 + lane;
      float wa[2], wb[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float mo = src[r * 32];
        const float lo = src[(2 + r) * 32];
        const float mn = fmaxf(m_run[r], mo);
        const float muv = mn == -INFINITY ? 0.0f : mn;
        wa[r] = fast_exp2(m_run[r] - muv);
        wb[r] = fast_exp2(mo - muv);
        m_run[r] = mn;
        l_run[r] = l_run[r] * wa[r] + lo * wb[r];
      }
#pragma unroll
      for (int i = 0; i < 4 * G; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o_acc[i][e] = o_acc[i][e] * wa[e >> 1] + src[(4 + i * 4 + e) * 32] * wb[e >> 1];
    }
  }

  // ---------------- the sink joins segment 0 as one term (m = sink, l = 1, no value)
  if (a.sinks && sigma == 0) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int idx = min(rg * 16 + g + 8 * half, n_rows - 1);
      const float sk = sink_log2(a, h * a.qpk + idx % a.qpk);
      const float mn = fmaxf(m_run[half], sk);
      if (mn == -INFINITY) continue;
      const float wa = fast_exp2(m_run[half] - mn);
      l_run[half] = l_run[half] * wa + fast_exp2(sk - mn);
      m_run[half] = mn;
#pragma unroll
      for (int i = 0; i < 4 * G; ++i) {
        o_acc[i][2 * half] *= wa;
        o_acc[i][2 * half + 1] *= wa;
      }
    }
  }

  // ---------------- write: final output, or this segment's partial triple
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int idx = rg * 16 + g + 8 * half;
    if (idx >= n_rows) continue;
    const int tok = q_start + tok0 + idx / a.qpk;
    const int hh = h * a.qpk + idx % a.qpk;
    if (split) {
      const int64_t prow = (static_cast<int64_t>(seq) * a.hq + hh) * a.num_splits + sigma;
      float *dst = a.part_acc + prow * D;
#pragma unroll
      for (int i = 0; i < 4 * G; ++i)
        *reinterpret_cast<float2 *>(dst + (i >> 2) * 32 + (i & 3) * 8 + 2 * t) =
            make_float2(o_acc[i][2 * half], o_acc[i][2 * half + 1]);
      if (t == 0)
        *reinterpret_cast<float2 *>(a.part_ml + prow * 2) = make_float2(m_run[half], l_run[half]);
    } else {
      const float inv = 1.0f / l_run[half];
      uint16_t *dst = a.out + (static_cast<int64_t>(tok) * a.hq + hh) * D;
#pragma unroll
      for (int i = 0; i < 4 * G; ++i)
        *reinterpret_cast<uint32_t *>(dst + (i >> 2) * 32 + (i & 3) * 8 + 2 * t) =
            pack_bf162(o_acc[i][2 * half] * inv, o_acc[i][2 * half + 1] * inv);
      if (t == 0 && a.lse)
        a.lse[static_cast<int64_t>(tok) * a.hq + hh] = (m_run[half] + log2f(l_run[half])) * kLn2;
    }
  }
}

template <int D, int BS, bool F8>
static cudaError_t launch_prefill_t(const AttnArgs &args, const CUtensorMap &tk,
                                    const CUtensorMap &tv, dim3 grid, cudaStream_t stream) {
  using C = AttnCfg<D, BS, F8>;
  static DeviceOnce configured;  // the attribute is per device
  cudaError_t e = configured.get(nullptr, [](int, int *) {
    return cudaFuncSetAttribute(prefill_kernel<D, BS, F8>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  prefill_kernel<D, BS, F8><<<grid, kThreads, C::kSmemBytes, stream>>>(args, tk, tv);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const AttnArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                           int d, int bs, bool f8v4, cudaStream_t stream) {
  const int64_t gx = static_cast<int64_t>(a.n_qblocks) +
                     (a.skip_single ? 0 : static_cast<int64_t>(a.num_splits - 1) * a.num_seqs);
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(a.hk), 1);
#define PAQ8_PREFILL_CASE(DD, BB)                                                   \
  if (d == DD && bs == BB)                                                          \
    return f8v4 ? launch_prefill_t<DD, BB, true>(a, tk, tv, grid, stream)           \
                : launch_prefill_t<DD, BB, false>(a, tk, tv, grid, stream);
  PAQ8_PREFILL_CASE(64, 16)
  PAQ8_PREFILL_CASE(64, 32)
  PAQ8_PREFILL_CASE(128, 16)
  PAQ8_PREFILL_CASE(128, 32)
  PAQ8_PREFILL_CASE(256, 16)
  PAQ8_PREFILL_CASE(256, 32)
#undef PAQ8_PREFILL_CASE
  return cudaErrorInvalidValue;
}

}  // namespace paq8
