// paged_attention: unified causal prefill + decode over the q8 HND cache.
//
// What it computes ("triton_turboquant_unified_attention.py", the unified 2D
// and split-KV 3D kernels, and the torch reference paths of
// "attention_impl.py"): for query token i of sequence s and q head h,
//   out = softmax_j(scale * q . k_j) v_j over keys j <= seq_len - q_len + i,
//   lse = ln sum_j exp(scale * q . k_j),
// with k_j, v_j the dequantized q8 rows of kv head h / (Hq / Hk), read page by
// page through the block table.
//
// Structure of one CTA (q-block x kv head x segment), 5 warps:
//  * warp 4 is the producer: it walks the CTA's KV tiles (64 keys), reads the
//    block-table entries 32 pages at a time, and stages each page's int8 K/V
//    codes (2-D TMA, 128-byte swizzle) and fp16 scales (1-D bulk copies) into
//    a ring of shared-memory stages guarded by mbarriers.
//  * warps 0-3 consume.  The q-block's rows (BLOCK_Q tokens x the Hq/Hk q
//    heads of this kv head, stacked as in the pages' GQA row tile) are split
//    into R row groups of 16; the 4/R warps that share a row group take
//    alternate KV tiles, each with its own online-softmax state, and merge at
//    the end.  Decode rows (one token) therefore spread one sequence's KV
//    stream over 4 warps.
//  * QK^T: the int8 K codes become exact fp16 integers in registers and meet
//    q (fp16) in m16n8k16 MMAs, one fp32 accumulator per 32-channel group,
//    scaled by that group's fp16 scale afterwards: the scores carry no
//    dequantization rounding.  Channels are permuted consistently between q
//    and k so that each lane reads 8 contiguous code bytes.
//  * PV: V codes are dequantized to fp16 (code * scale, one rounding),
//    transposed into the B operand with movmatrix, and multiplied by P (fp16).
//  * Split-KV (3D kernel of the pages): sequences with a single query token
//    may be cut into segments; each segment writes its (max, expsum, acc)
//    triple and `reduce_kernel` merges them by log-sum-exp.
#include "common.cuh"
#include "launch.h"

namespace paq8 {

constexpr int kTile = 64;  // keys per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxSplits = 16;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnArgs {
  const uint16_t *q;            // [T, Hq, D] bf16
  const int32_t *cu_seqlens_q;  // [S+1]
  const int32_t *seq_lens;      // [S]
  const int32_t *block_table;   // [S, bt_stride]
  const uint16_t *k_scale;      // [nb, Hk, bs, G] fp16
  const uint16_t *v_scale;
  uint16_t *out;                // [T, Hq, D] bf16
  float *lse;                   // [T, Hq] or null
  float *part_acc;              // [S, Hq, NS, D]
  float *part_ml;               // [S, Hq, NS, 2]  (max in log2 units, expsum)
  uint32_t *status;
  int32_t num_seqs, num_tokens, hq, hk, qpk, num_blocks, bt_stride;
  int32_t block_q;              // tokens per q-block
  int32_t n_qblocks;            // grid.x entries that are q-blocks
  int32_t num_splits;           // segments of single-token sequences
  int32_t seg_tiles;            // tiles per segment
  float scale_log2;             // softmax_scale * log2(e)
};

template <int D, int BS>
struct AttnCfg {
  static constexpr int G = D / 32;
  static constexpr int kPages = kTile / BS;
  static constexpr int kRowBytes = D >= 128 ? 128 : D;  // bytes per row of one TMA box
  static constexpr int kSub = D / kRowBytes;             // boxes per row (2 for D = 256)
  // A stage is always consumed by the same group of warps (stage = tile % 4,
  // group = tile % (4 / R)), so no waiter can run two phases ahead of a
  // stage's barrier.
  static constexpr int kStages = 4;
  static constexpr int kCodeBytes = kTile * D;
  static constexpr int kScaleBytes = kTile * G * 2;
  static constexpr int kStageBytes = 2 * kCodeBytes + 2 * kScaleBytes;
  static constexpr int kQBytes = 4 * G * 2 * 32 * 16;  // fragment-ordered q, 4 row groups
  static constexpr int kQOff = kStages * kStageBytes;
  static constexpr int kBarOff = kQOff + kQBytes;
  static constexpr int kSmemBytes = kBarOff + 2 * kStages * 8 + 1024;  // + alignment slack
  static constexpr uint32_t kPageTx = 2u * BS * D + 2u * BS * G * 2;
  // merge area (inside the stages) per partner warp: m0 m1 l0 l1 + O
  static constexpr int kMergeFields = 4 + 4 * 4 * G;
  static_assert(3 * kMergeFields * 32 * 4 <= kStages * kStageBytes, "merge area");
  static_assert(kStageBytes % 512 == 0, "stage alignment");
  static_assert(kStages % kConsumerWarps == 0, "stages must be a multiple of the kv groups");
};

// Byte offset of (row r, byte b) of a staged code tile, as the TMA swizzle
// lays it out (128-byte swizzle: 16-byte chunk index XOR row % 8; 64-byte
// swizzle for D = 64: chunk XOR (row / 2) % 4).
template <int D>
__device__ __forceinline__ uint32_t code_off(int r, int b) {
  if constexpr (D >= 128) {
    const int off = r * 128 + (b & 127);
    return (b >> 7) * (kTile * 128) + (off ^ (((off >> 7) & 7) << 4));
  } else {
    const int off = r * 64 + b;
    return off ^ (((off >> 7) & 3) << 4);
  }
}

// Warp-cooperative search for the sequence owning q-block `target`: the last
// s with key(s) <= target, key(s) = cu[s] / block_q + s (cu[s] when
// block_q == 1).  The pages use a binary search over the same keys
// (_find_seq_idx); here each round samples 32 candidates at once.
__device__ __forceinline__ int find_seq(const int32_t *cu, int num_seqs, int block_q,
                                        int target, int lane) {
  int lo = 0, hi = num_seqs;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    bool le = false;
    if (idx < hi) {
      const int v = cu[idx];
      const int key = block_q == 1 ? v : v / block_q + idx;
      le = key <= target;
    }
    const unsigned ball = __ballot_sync(0xffffffffu, le);
    const int k = ball ? 31 - __clz(ball) : 0;
    lo = lo + k * step;
    hi = min(hi, lo + step);
  }
  return lo;
}

template <int D, int BS>
__global__ void __launch_bounds__(kThreads) attention_kernel(const __grid_constant__ AttnArgs a,
                                                             const __grid_constant__ CUtensorMap tmap_k,
                                                             const __grid_constant__ CUtensorMap tmap_v) {
  using C = AttnCfg<D, BS>;
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
  if (q_end > a.num_tokens || q_start < 0) {
    if (threadIdx.x == 0 && sigma == 0) flag_status(a.status, PA_DEV_BAD_SEQ);
    return;
  }
  const int seq_len = a.seq_lens[seq];
  const int ctx = seq_len - q_len;
  if (ctx < 0) {
    if (threadIdx.x == 0 && sigma == 0 && tok0 == 0) flag_status(a.status, PA_DEV_BAD_SEQ);
    return;
  }
  const bool split = a.num_splits > 1 && q_len == 1;
  if (!split && sigma > 0) return;
  const int n_tok = min(a.block_q, q_len - tok0);
  const int n_rows = n_tok * a.qpk;
  const int kv_end = ctx + tok0 + n_tok;  // keys visible to the last row
  const int num_tiles = (kv_end + kTile - 1) / kTile;
  int tile_lo = 0, tile_hi = num_tiles;
  if (split) {
    if (static_cast<int64_t>(sigma) * a.seg_tiles * kTile >= seq_len) return;
    tile_lo = sigma * a.seg_tiles;
    tile_hi = sigma == a.num_splits - 1 ? num_tiles : min(num_tiles, tile_lo + a.seg_tiles);
  }
  const int n_iter = tile_hi - tile_lo;
  if (n_iter <= 0) return;
  const int R = n_rows <= 16 ? 1 : (n_rows <= 32 ? 2 : 4);
  const int KG = kConsumerWarps / R;

  const uint32_t bar_full = smem_base + C::kBarOff;
  const uint32_t bar_empty = bar_full + C::kStages * 8;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, R);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ================================================================ producer
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    const int n_pages = (kv_end + BS - 1) / BS;
    const int32_t *bt_row = a.block_table + static_cast<int64_t>(seq) * a.bt_stride;
    int page_base = -(1 << 30);
    int my_blk = -1;
    for (int it = 0; it < n_iter; ++it) {
      const int stage = it % C::kStages;
      if (it >= C::kStages) {
        int ok = 1;
        if (lane == 0) ok = mbar_wait(bar_empty + 8 * stage, ((it / C::kStages) - 1) & 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) flag_status(a.status, PA_DEV_TIMEOUT);
          break;
        }
      }
      const int lp0 = (tile_lo + it) * C::kPages;
      if (lp0 - page_base >= 32) {
        page_base = lp0;
        const int lp = page_base + lane;
        my_blk = -1;
        if (lp < n_pages) {
          const int b = lp < a.bt_stride ? bt_row[lp] : -1;
          if (b >= 0 && b < a.num_blocks) my_blk = b;
          else flag_status(a.status, PA_DEV_BAD_BLOCK);
        }
      }
      int blk[C::kPages];
      int nvalid = 0;
#pragma unroll
      for (int p = 0; p < C::kPages; ++p) {
        blk[p] = __shfl_sync(0xffffffffu, my_blk, lp0 + p - page_base);
        nvalid += blk[p] >= 0;
      }
      if (lane == 0) {
        const uint32_t full = bar_full + 8 * stage;
        const uint32_t st = smem_base + stage * C::kStageBytes;
        mbar_arrive_expect_tx(full, nvalid * C::kPageTx);
#pragma unroll
        for (int p = 0; p < C::kPages; ++p) {
          if (blk[p] < 0) continue;
          const int64_t row0 = (static_cast<int64_t>(blk[p]) * a.hk + h) * BS;
#pragma unroll
          for (int sub = 0; sub < C::kSub; ++sub) {
            const uint32_t dst = sub * (kTile * C::kRowBytes) + p * (BS * C::kRowBytes);
            tma_load_2d(st + dst, &tmap_k, sub * C::kRowBytes, static_cast<int32_t>(row0), full);
            tma_load_2d(st + C::kCodeBytes + dst, &tmap_v, sub * C::kRowBytes,
                        static_cast<int32_t>(row0), full);
          }
          const uint32_t sdst = p * (BS * G * 2);
          bulk_load(st + 2 * C::kCodeBytes + sdst, a.k_scale + row0 * G, BS * G * 2, full);
          bulk_load(st + 2 * C::kCodeBytes + C::kScaleBytes + sdst, a.v_scale + row0 * G,
                    BS * G * 2, full);
        }
      }
      __syncwarp();
    }
    return;
  }

  // ================================================================== consumers
  const int rg = warp % R;
  const int kg = warp / R;
  const int g = lane >> 2;
  const int t = lane & 3;
  const uint32_t q_frag = smem_base + C::kQOff;

  // q -> fp16 fragments in MMA order: [row group][group][k-step][lane] x 16 B.
  if (warp < R) {
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
        // channels 8t + {0..7}; k-step s takes 4s + {0,1} (cols 2t, 2t+1)
        // and 4s + {2,3} (cols 2t+8, 2t+9)
        f[0][half] = pack_half2(bf16_lo(v.x), bf16_hi(v.x));
        f[0][2 + half] = pack_half2(bf16_lo(v.y), bf16_hi(v.y));
        f[1][half] = pack_half2(bf16_lo(v.z), bf16_hi(v.z));
        f[1][2 + half] = pack_half2(bf16_lo(v.w), bf16_hi(v.w));
      }
#pragma unroll
      for (int s = 0; s < 2; ++s)
        sts128(q_frag + (((warp * G + gq) * 2 + s) * 32 + lane) * 16,
               make_uint4(f[s][0], f[s][1], f[s][2], f[s][3]));
    }
  }
  named_barrier(1, kConsumerWarps * 32);

  // causal limits (last visible key) of rows g and g + 8; padding rows copy
  // the block's last row so their arithmetic stays finite
  int lim[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int idx = rg * 16 + g + 8 * half;
    lim[half] = idx < n_rows ? ctx + tok0 + idx / a.qpk : kv_end - 1;
  }
  int min_lim = min(lim[0], lim[1]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) min_lim = min(min_lim, __shfl_xor_sync(0xffffffffu, min_lim, o));

  float m_run[2] = {-INFINITY, -INFINITY};  // running max, log2 units
  float l_run[2] = {0.0f, 0.0f};            // this lane's share of the expsum
  float o_acc[4 * G][4];
#pragma unroll
  for (int i = 0; i < 4 * G; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o_acc[i][e] = 0.0f;

  bool timed_out = false;
  for (int it = kg; it < n_iter; it += KG) {
    const int stage = it % C::kStages;
    if (!mbar_wait(bar_full + 8 * stage, (it / C::kStages) & 1)) {
      timed_out = true;
      break;
    }
    const uint32_t kb = smem_base + stage * C::kStageBytes;
    const uint32_t vb = kb + C::kCodeBytes;
    const uint32_t ksb = kb + 2 * C::kCodeBytes;
    const uint32_t vsb = ksb + C::kScaleBytes;
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
        const uint2 kw = lds64(kb + code_off<D>(nt * 8 + g, gq * 32 + t * 8));
        uint32_t b0, b1, b2, b3;
        codes4_to_half2(kw.x, b0, b1);
        codes4_to_half2(kw.y, b2, b3);
        float sg[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_f16_16816(sg, qa0.x, qa0.y, qa0.z, qa0.w, b0, b1);
        mma_f16_16816(sg, qa1.x, qa1.y, qa1.z, qa1.w, b2, b3);
        const int kr = nt * 8 + 2 * t;
        const float s0 = __half2float(__ushort_as_half(lds16(ksb + (kr * G + gq) * 2)));
        const float s1 = __half2float(__ushort_as_half(lds16(ksb + ((kr + 1) * G + gq) * 2)));
        sc[nt][0] = fmaf(sg[0], s0, sc[nt][0]);
        sc[nt][1] = fmaf(sg[1], s1, sc[nt][1]);
        sc[nt][2] = fmaf(sg[2], s0, sc[nt][2]);
        sc[nt][3] = fmaf(sg[3], s1, sc[nt][3]);
      }
    }

    // ---------------- mask, online softmax (log2 domain)
    const bool need_mask = key0 + kTile - 1 > min_lim;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sc[nt][e] * a.scale_log2;
        if (need_mask) {
          const int key = key0 + nt * 8 + 2 * t + (e & 1);
          if (key > lim[e >> 1]) v = -INFINITY;
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

    // ---------------- O += P V', V' = code * scale in fp16
    const bool tail = key0 + kTile > kv_end;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t pa0 = pack_half2(sc[2 * kk][0], sc[2 * kk][1]);
      const uint32_t pa1 = pack_half2(sc[2 * kk][2], sc[2 * kk][3]);
      const uint32_t pa2 = pack_half2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      const uint32_t pa3 = pack_half2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
      const int ra = kk * 16 + g;
      const int rb = ra + 8;
#pragma unroll
      for (int gq = 0; gq < G; ++gq) {
        const uint2 va = lds64(vb + code_off<D>(ra, gq * 32 + t * 8));
        const uint2 vv = lds64(vb + code_off<D>(rb, gq * 32 + t * 8));
        uint32_t sa = lds16(vsb + (ra * G + gq) * 2);
        uint32_t sb = lds16(vsb + (rb * G + gq) * 2);
        if (tail) {  // keys past the visible range may hold stale bytes
          if (key0 + ra >= kv_end) sa = 0u;
          if (key0 + rb >= kv_end) sb = 0u;
        }
        sa |= sa << 16;
        sb |= sb << 16;
        uint32_t ma[4], mb[4];
        codes4_to_half2(va.x, ma[0], ma[1]);
        codes4_to_half2(va.y, ma[2], ma[3]);
        codes4_to_half2(vv.x, mb[0], mb[1]);
        codes4_to_half2(vv.y, mb[2], mb[3]);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint32_t b0 = movmatrix_trans(hmul2_u32(ma[jj], sa));
          const uint32_t b1 = movmatrix_trans(hmul2_u32(mb[jj], sb));
          mma_f16_16816(o_acc[gq * 4 + jj], pa0, pa1, pa2, pa3, b0, b1);
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
      for (int gq = 0; gq < G; ++gq) {
        float4 lo4 = make_float4(o_acc[gq * 4 + 0][2 * half], o_acc[gq * 4 + 0][2 * half + 1],
                                 o_acc[gq * 4 + 1][2 * half], o_acc[gq * 4 + 1][2 * half + 1]);
        float4 hi4 = make_float4(o_acc[gq * 4 + 2][2 * half], o_acc[gq * 4 + 2][2 * half + 1],
                                 o_acc[gq * 4 + 3][2 * half], o_acc[gq * 4 + 3][2 * half + 1]);
        *reinterpret_cast<float4 *>(dst + gq * 32 + t * 8) = lo4;
        *reinterpret_cast<float4 *>(dst + gq * 32 + t * 8 + 4) = hi4;
      }
      if (t == 0)
        *reinterpret_cast<float2 *>(a.part_ml + prow * 2) = make_float2(m_run[half], l_run[half]);
    } else {
      const float inv = 1.0f / l_run[half];
      uint16_t *dst = a.out + (static_cast<int64_t>(tok) * a.hq + hh) * D;
#pragma unroll
      for (int gq = 0; gq < G; ++gq) {
        uint4 w;
        w.x = pack_bf162(o_acc[gq * 4 + 0][2 * half] * inv, o_acc[gq * 4 + 0][2 * half + 1] * inv);
        w.y = pack_bf162(o_acc[gq * 4 + 1][2 * half] * inv, o_acc[gq * 4 + 1][2 * half + 1] * inv);
        w.z = pack_bf162(o_acc[gq * 4 + 2][2 * half] * inv, o_acc[gq * 4 + 2][2 * half + 1] * inv);
        w.w = pack_bf162(o_acc[gq * 4 + 3][2 * half] * inv, o_acc[gq * 4 + 3][2 * half + 1] * inv);
        *reinterpret_cast<uint4 *>(dst + gq * 32 + t * 8) = w;
      }
      if (t == 0 && a.lse)
        a.lse[static_cast<int64_t>(tok) * a.hq + hh] = (m_run[half] + log2f(l_run[half])) * kLn2;
    }
  }
}

// Merge of the segment triples of single-token sequences (the pages'
// reduce_segments, written from the online-softmax merge rule):
//   M = max m_k;  w_k = 2^(m_k - M);  out = sum w_k acc_k / sum w_k l_k;
//   lse = (M + log2 sum w_k l_k) * ln 2.
// One warp per (sequence, q head); segment k exists when k * seg_keys < seq_len.
template <int D>
__global__ void __launch_bounds__(128) reduce_kernel(const float *__restrict__ part_acc,
                                                     const float *__restrict__ part_ml,
                                                     const int32_t *__restrict__ cu,
                                                     const int32_t *__restrict__ seq_lens,
                                                     int32_t num_seqs, int32_t num_tokens,
                                                     int32_t hq, int32_t num_splits,
                                                     int32_t seg_keys, uint16_t *__restrict__ out,
                                                     float *__restrict__ lse) {
  constexpr int V = D / 32;  // channels per lane
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (gw >= static_cast<int64_t>(num_seqs) * hq) return;
  const int seq = static_cast<int>(gw / hq);
  const int hh = static_cast<int>(gw % hq);
  const int q0 = cu[seq];
  if (cu[seq + 1] - q0 != 1 || q0 < 0 || q0 >= num_tokens) return;
  const int L = seq_lens[seq];
  if (L < 1) return;
  const int nseg = min(num_splits, static_cast<int>((L + seg_keys - 1) / seg_keys));
  const int64_t prow = gw * num_splits;
  float m = -INFINITY, l = 0.0f;
  if (lane < nseg) {
    const float2 ml = *reinterpret_cast<const float2 *>(part_ml + (prow + lane) * 2);
    m = ml.x;
    l = ml.y;
  }
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float mu = M == -INFINITY ? 0.0f : M;
  const float w = lane < nseg ? fast_exp2(m - mu) : 0.0f;
  float lw = w * l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.0f;
  for (int k = 0; k < nseg; ++k) {
    const float wk = __shfl_sync(0xffffffffu, w, k);
    const float *src = part_acc + (prow + k) * D + lane * V;
#pragma unroll
    for (int v = 0; v < V; v += 2) {
      const float2 x = *reinterpret_cast<const float2 *>(src + v);
      acc[v] = fmaf(wk, x.x, acc[v]);
      acc[v + 1] = fmaf(wk, x.y, acc[v + 1]);
    }
  }
  const float inv = 1.0f / lw;
  uint16_t *dst = out + (static_cast<int64_t>(q0) * hq + hh) * D + lane * V;
#pragma unroll
  for (int v = 0; v < V; v += 2)
    *reinterpret_cast<uint32_t *>(dst + v) = pack_bf162(acc[v] * inv, acc[v + 1] * inv);
  if (lane == 0 && lse) lse[static_cast<int64_t>(q0) * hq + hh] = (M + log2f(lw)) * kLn2;
}

// ---------------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2-D map over an HND code cache viewed as rows of D bytes.
static bool encode_code_map(CUtensorMap *map, const void *base, int64_t rows, int d, int bs) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int row_bytes = d >= 128 ? 128 : d;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes), static_cast<cuuint32_t>(bs)};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int BS>
static cudaError_t launch_attention_t(const AttnArgs &args, const CUtensorMap &tk,
                                      const CUtensorMap &tv, dim3 grid, cudaStream_t stream) {
  using C = AttnCfg<D, BS>;
  static int configured_device = -1;  // the attribute is per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel<D, BS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  attention_kernel<D, BS><<<grid, kThreads, C::kSmemBytes, stream>>>(args, tk, tv);
  return cudaGetLastError();
}

int32_t auto_num_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t max_query_len,
                        int32_t max_seq_len) {
  (void)num_seqs;
  (void)num_kv_heads;
  (void)max_query_len;
  // ~512 keys per segment, at most 16 segments (the pages' default count)
  int32_t ns = (max_seq_len + 511) / 512;
  return ns < 1 ? 1 : (ns > kMaxSplits ? kMaxSplits : ns);
}


cudaError_t launch_paged_attention(const AttnLaunch &L, cudaStream_t stream) {
  AttnArgs a;
  a.q = static_cast<const uint16_t *>(L.q);
  a.cu_seqlens_q = L.cu;
  a.seq_lens = L.seq_lens;
  a.block_table = L.block_table;
  a.k_scale = static_cast<const uint16_t *>(L.k_scale);
  a.v_scale = static_cast<const uint16_t *>(L.v_scale);
  a.out = static_cast<uint16_t *>(L.out);
  a.lse = L.lse;
  a.status = reinterpret_cast<uint32_t *>(L.workspace);
  a.num_seqs = L.num_seqs;
  a.num_tokens = L.num_tokens;
  a.hq = L.hq;
  a.hk = L.hk;
  a.qpk = L.hq / L.hk;
  a.num_blocks = L.num_blocks;
  a.bt_stride = L.bt_stride;
  a.block_q = L.max_query_len <= 1 ? 1 : (64 / a.qpk > 0 ? 64 / a.qpk : 1);
  a.n_qblocks = a.block_q == 1 ? L.num_tokens : L.num_tokens / a.block_q + L.num_seqs;
  a.num_splits = L.num_splits;
  const int tiles = (L.max_seq_len + kTile - 1) / kTile;
  a.seg_tiles = (tiles + L.num_splits - 1) / L.num_splits;
  if (a.seg_tiles < 1) a.seg_tiles = 1;
  a.scale_log2 = L.softmax_scale * 1.4426950408889634f;
  a.part_acc = reinterpret_cast<float *>(L.workspace + 256);
  a.part_ml = a.part_acc + static_cast<int64_t>(L.num_seqs) * L.hq * L.num_splits * L.d;
  if (a.n_qblocks <= 0) return cudaSuccess;

  const int64_t rows = static_cast<int64_t>(L.num_blocks) * L.hk * L.bs;
  CUtensorMap tk, tv;
  if (!encode_code_map(&tk, L.k_cache, rows, L.d, L.bs) ||
      !encode_code_map(&tv, L.v_cache, rows, L.d, L.bs))
    return cudaErrorInvalidValue;
  const int64_t gx = static_cast<int64_t>(a.n_qblocks) +
                     static_cast<int64_t>(L.num_splits - 1) * L.num_seqs;
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(L.hk), 1);
  cudaError_t e = cudaErrorInvalidValue;
#define PAQ8_ATTN_CASE(DD, BB)                                        \
  if (L.d == DD && L.bs == BB) e = launch_attention_t<DD, BB>(a, tk, tv, grid, stream);
  PAQ8_ATTN_CASE(64, 16)
  PAQ8_ATTN_CASE(64, 32)
  PAQ8_ATTN_CASE(128, 16)
  PAQ8_ATTN_CASE(128, 32)
  PAQ8_ATTN_CASE(256, 16)
  PAQ8_ATTN_CASE(256, 32)
#undef PAQ8_ATTN_CASE
  if (e != cudaSuccess || L.num_splits <= 1) return e;

  const int64_t warps = static_cast<int64_t>(L.num_seqs) * L.hq;
  const unsigned blocks = static_cast<unsigned>((warps + 3) / 4);
  const int seg_keys = a.seg_tiles * kTile;
  switch (L.d) {
    case 64:
      reduce_kernel<64><<<blocks, 128, 0, stream>>>(a.part_acc, a.part_ml, L.cu, L.seq_lens,
                                                     L.num_seqs, L.num_tokens, L.hq,
                                                     L.num_splits, seg_keys, a.out, L.lse);
      break;
    case 128:
      reduce_kernel<128><<<blocks, 128, 0, stream>>>(a.part_acc, a.part_ml, L.cu, L.seq_lens,
                                                      L.num_seqs, L.num_tokens, L.hq,
                                                      L.num_splits, seg_keys, a.out, L.lse);
      break;
    case 256:
      reduce_kernel<256><<<blocks, 128, 0, stream>>>(a.part_acc, a.part_ml, L.cu, L.seq_lens,
                                                      L.num_seqs, L.num_tokens, L.hq,
                                                      L.num_splits, seg_keys, a.out, L.lse);
      break;
  }
  return cudaGetLastError();
}

}  // namespace paq8
