// Pieces shared by the paged-attention kernels: arguments, the staged page
// layouts in shared memory, the TMA producer loop and the key permutation
// that lets a lane read its MMA fragments with plain vector loads.
#pragma once

#include "common.cuh"

namespace paq8 {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;  // pipeline depth; a multiple of the kv groups (1, 2, 4)
constexpr int kMaxSplits = 16;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnArgs {
  const uint16_t *q;            // [T, Hq, D] bf16
  const int32_t *cu_seqlens_q;  // [S+1]
  const int32_t *seq_lens;      // [S]
  const int32_t *block_table;   // [S, bt_stride]
  const int8_t *k_cache;        // [nb, Hk, bs, D] int8
  const int8_t *v_cache;        // [nb, Hk, D, bs] int8
  const uint16_t *k_scale;      // [nb, Hk, bs, G] fp16
  const uint16_t *v_scale;      // [nb, Hk, G, bs] fp16 (fp8/4-bit format: [nb, Hk, bs])
  const uint16_t *v_zero;       // fp8/4-bit format only: [nb, Hk, bs] fp16
  uint16_t *out;                // [T, Hq, D] bf16
  float *lse;                   // [T, Hq] or null
  float *part_acc;              // [S, Hq, NS, D]
  float *part_ml;               // [S, Hq, NS, 2]  (max in log2 units, expsum)
  uint32_t *status;
  int32_t num_seqs, num_tokens, hq, hk, qpk, num_blocks, bt_stride;
  int32_t block_q;              // tokens per q-block (prefill kernel)
  int32_t n_qblocks;            // grid.x entries that are q-blocks (prefill kernel)
  int32_t num_splits;           // segments of single-token sequences
  int32_t seg_tiles;            // tiles per segment
  int32_t skip_single;          // prefill kernel: leave single-token sequences alone
  int32_t multi_token_ok;       // decode kernel: a prefill kernel runs for q_len > 1
  float scale_log2;             // softmax_scale * log2(e)
  // Visibility.  causal: query i of a sequence sees keys up to
  // seq_len - q_len + i; otherwise every key of the sequence (seq_len may then
  // be below q_len, even 0).  window > 0: a query whose last visible key is p
  // sees keys p - window + 1 .. p only (causal only).
  int32_t causal;
  int32_t window;
  const float *sinks;           // [Hq] sink logits (units of the scaled scores) or null
  int32_t test_timeout;         // test hook: the decode producer stages nothing
  uint64_t wait_limit_ns;       // bound of every pipeline wait of the decode kernel
};

constexpr float kLog2e = 1.4426950408889634f;

// Last visible key of local query token i of a sequence (-1: none).
__device__ __forceinline__ int last_key(const AttnArgs &a, int seq_len, int q_len, int i) {
  return a.causal ? seq_len - q_len + i : seq_len - 1;
}

// First visible key of a query whose last visible key is `last`.
__device__ __forceinline__ int first_key(const AttnArgs &a, int last) {
  return a.window > 0 ? max(0, last - a.window + 1) : 0;
}

// Sink logit of q head hh in log2 units, -inf without sinks.
__device__ __forceinline__ float sink_log2(const AttnArgs &a, int hh) {
  return a.sinks ? a.sinks[hh] * kLog2e : -INFINITY;
}

// Tiles of `tile` keys holding the visible keys [kv_begin, kv_end) of a
// single-token row, and how many of them each split segment takes: the
// decode kernel, the generic kernel and the segment reduce all use this
// rule, so they agree on which segments exist.
__device__ __forceinline__ int segments_of(int kv_begin, int kv_end, int tile, int seg_tiles,
                                           int num_splits) {
  const int vis_tiles = (kv_end + tile - 1) / tile - kv_begin / tile;
  return min(num_splits, (vis_tiles + seg_tiles - 1) / seg_tiles);
}

// out = 0 and lse = sink (or -inf) for the q heads [hh0, hh0 + n) of token
// `tok`: a row that sees no key (only in non-causal mode, seq_len == 0).
// Called by one warp.
template <int D>
__device__ __forceinline__ void write_empty_rows(const AttnArgs &a, int tok, int hh0, int n,
                                                 int lane) {
  for (int r = 0; r < n; ++r) {
    uint16_t *dst = a.out + (static_cast<int64_t>(tok) * a.hq + hh0 + r) * D;
    for (int c = lane * 8; c < D; c += 256)
      *reinterpret_cast<uint4 *>(dst + c) = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0 && a.lse) {
      const float s = a.sinks ? a.sinks[hh0 + r] : -INFINITY;
      a.lse[static_cast<int64_t>(tok) * a.hq + hh0 + r] = s;
    }
  }
}

// Layout of one pipeline stage of TILE keys (a whole number of pages):
//   K codes  [TILE][D]    token-major pages in the 128-byte swizzle pattern
//                         (64-byte for D = 64); D = 256 rows are two halves
//   V codes  [pages][D][BS] channel-major pages (32-byte swizzle for BS = 32)
//   K scales [TILE][G]    fp16
//   V scales [pages][G][BS] fp16
// Filled either by the TMA unit (produce_tiles: a 2-D box per page for the
// codes, a bulk copy per page for each scale array) or by 16-byte cp.async
// chunks written at the same swizzled places (produce_tiles_lsu).
template <int D, int BS, int TILE>
struct StageLayout {
  static constexpr int kD = D;
  static constexpr int G = D / 32;
  static constexpr int kPages = TILE / BS;
  static constexpr int kRowBytes = D >= 128 ? 128 : D;  // K box row bytes
  static constexpr int kSub = D / kRowBytes;             // K boxes per row
  static constexpr int kCodeBytes = TILE * D;
  static constexpr int kScaleBytes = TILE * G * 2;
  static constexpr int kVOff = kCodeBytes;
  static constexpr int kKsOff = 2 * kCodeBytes;
  static constexpr int kVsOff = 2 * kCodeBytes + kScaleBytes;
  static constexpr int kBytes = 2 * kCodeBytes + 2 * kScaleBytes;
  static constexpr uint32_t kPageTx = 2u * BS * D + 2u * BS * G * 2;
  static_assert(TILE % BS == 0 && TILE % 16 == 0, "tile");
  static_assert(kBytes % 512 == 0, "stage alignment for the swizzled boxes");

  // K: byte b of key row r (swizzle as laid out by the TMA unit)
  __device__ static __forceinline__ uint32_t k_off(int r, int b) {
    if constexpr (D >= 128) {
      const int off = r * 128 + (b & 127);
      return (b >> 7) * (TILE * 128) + (off ^ (((off >> 7) & 7) << 4));
    } else {
      const int off = r * 64 + b;
      return off ^ (((off >> 7) & 3) << 4);
    }
  }
  // V: byte of key `key` (0..TILE-1) of channel c
  __device__ static __forceinline__ uint32_t v_off(int c, int key) {
    const int page = key / BS;
    const int off = c * BS + (key % BS);
    if constexpr (BS == 32) {
      return kVOff + page * (D * BS) + (off ^ (((off >> 7) & 1) << 4));
    } else {
      return kVOff + page * (D * BS) + off;
    }
  }
  // K scales: group g of key `key`
  __device__ static __forceinline__ uint32_t ks_off(int key, int g) {
    return kKsOff + (key * G + g) * 2;
  }
  // V scales: group g of key `key`
  __device__ static __forceinline__ uint32_t vs_off(int key, int g) {
    return kVsOff + ((key / BS) * (G * BS) + g * BS + key % BS) * 2;
  }
};

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

// MMA k index -> key within a 16-key block.  A lane reads 4 consecutive keys
// of one V channel (a 32-bit word): keys 4t..4t+1 serve k = 2t, 2t+1 and keys
// 4t+2..4t+3 serve k = 2t+8, 2t+9.  K rows and scores follow the same order.
__device__ __forceinline__ int perm16(int k) {
  return ((k & 7) >> 1) * 4 + (k >> 3) * 2 + (k & 1);
}

// The producer warp: walks tiles [tile_lo, tile_lo + n_iter) of sequence
// `seq`, kv head h, staging each tile's pages through an NST-stage mbarrier
// ring (stage s at smem_base + s * L::kBytes).
// Block-table entries are read 32 pages at a time, one per lane.
// Pages wholly before kv_begin (keys no query of the tile range sees) or at or
// past kv_end are not staged; the consumers mask their keys.
template <class L, int BS, int NST = kStages>
__device__ __forceinline__ void produce_tiles(const AttnArgs &a, const CUtensorMap *tmap_k,
                                              const CUtensorMap *tmap_v, uint32_t smem_base,
                                              uint32_t bar_full, uint32_t bar_empty, int seq,
                                              int h, int tile_lo, int n_iter, int kv_begin,
                                              int kv_end, int lane) {
  const int n_pages = (kv_end + BS - 1) / BS;
  const int32_t *bt_row = a.block_table + static_cast<int64_t>(seq) * a.bt_stride;
  int page_base = -(1 << 30);
  int my_blk = -1;
  for (int it = 0; it < n_iter; ++it) {
    const int stage = it % NST;
    if (it >= NST) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(bar_empty + 8 * stage, ((it / NST) - 1) & 1, a.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) flag_status(a.status, PA_DEV_TIMEOUT);
        return;
      }
    }
    const int lp0 = (tile_lo + it) * L::kPages;
    if (lp0 - page_base >= 32) {
      page_base = lp0;
      const int lp = page_base + lane;
      my_blk = -1;
      if (lp < n_pages && (lp + 1) * BS > kv_begin) {
        const int b = lp < a.bt_stride ? bt_row[lp] : -1;
        if (b >= 0 && b < a.num_blocks) my_blk = b;
        else flag_status(a.status, PA_DEV_BAD_BLOCK);
      }
    }
    int blk[L::kPages];
    int nvalid = 0;
#pragma unroll
    for (int p = 0; p < L::kPages; ++p) {
      blk[p] = __shfl_sync(0xffffffffu, my_blk, lp0 + p - page_base);
      nvalid += blk[p] >= 0;
    }
    if (lane == 0) {
      const uint32_t full = bar_full + 8 * stage;
      const uint32_t st = smem_base + stage * L::kBytes;
      mbar_arrive_expect_tx(full, nvalid * L::kPageTx);
#pragma unroll
      for (int p = 0; p < L::kPages; ++p) {
        if (blk[p] < 0) continue;
        const int64_t page = static_cast<int64_t>(blk[p]) * a.hk + h;
#pragma unroll
        for (int sub = 0; sub < L::kSub; ++sub)
          tma_load_2d(st + sub * (L::kCodeBytes / L::kSub) + p * (BS * L::kRowBytes), tmap_k,
                      sub * L::kRowBytes, static_cast<int32_t>(page * BS), full);
        // V page: D channel rows of BS key bytes; row index page * D in the map
        tma_load_2d(st + L::kVOff + p * (L::kD * BS), tmap_v, 0,
                    static_cast<int32_t>(page * L::kD), full);
        bulk_load(st + L::kKsOff + p * (BS * L::G * 2), a.k_scale + page * BS * L::G,
                  BS * L::G * 2, full);
        bulk_load(st + L::kVsOff + p * (BS * L::G * 2), a.v_scale + page * BS * L::G,
                  BS * L::G * 2, full);
      }
    }
    __syncwarp();
  }
}

// 16-byte LSU copy global -> shared (L2 only), completion tracked per thread.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// The mbarrier receives one arrival from this thread once all its earlier
// cp.async copies have landed (counted against the expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Producer warp with LSU copies: the same tiles and stage layout as
// produce_tiles, but every lane copies 16-byte chunks of the tile's pages
// (K and V codes and both scale arrays) with cp.async, writing each chunk
// at its swizzled place, and arrives on the stage's full barrier (which
// expects 32 arrivals) when its copies land.  A page costs 2 * BS * (D +
// D/16) / 16 chunks spread over the 32 lanes, instead of four TMA requests:
// the TMA unit's per-request cost, not bandwidth, limited small pages.
// it0: ring position of the first tile (a persistent kernel keeps one ring
// position across its work items).  Returns false when a wait gave up.
template <class L, int BS, int NST = kStages>
__device__ __forceinline__ bool produce_tiles_lsu(const AttnArgs &a, uint32_t smem_base,
                                                  uint32_t bar_full, uint32_t bar_empty, int seq,
                                                  int h, int tile_lo, int n_iter, int kv_begin,
                                                  int kv_end, int lane, int it0 = 0) {
  constexpr int D = L::kD;
  constexpr int kKChunks = BS * D / 16;        // K (or V) code chunks of a page
  constexpr int kPer = kKChunks / 32;          // ... per lane
  constexpr int kSChunks = BS * L::G * 2 / 16;  // K (or V) scale chunks of a page
  constexpr int kSPer = (2 * kSChunks + 31) / 32;
  constexpr int kRowChunks = D / 16;           // chunks of one K row
  constexpr int kVRowChunks = BS / 16;         // chunks of one V channel row
  static_assert(kSChunks >= 1 && kKChunks % 32 == 0, "page pieces are whole chunks");
  // Stage offsets of this lane's chunks within page 0; page p adds p times the
  // page's share of each array (the swizzle pattern repeats every page).
  uint32_t koff[kPer], voff[kPer], soff[kSPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int c = lane + 32 * i;
    koff[i] = L::k_off(c / kRowChunks, (c % kRowChunks) * 16);
    voff[i] = L::v_off(c / kVRowChunks, (c % kVRowChunks) * 16);
  }
#pragma unroll
  for (int i = 0; i < kSPer; ++i) {
    const int c = lane + 32 * i;
    soff[i] = c < kSChunks ? L::kKsOff + c * 16 : L::kVsOff + (c - kSChunks) * 16;
  }
  constexpr uint32_t kKPage = BS * L::kRowBytes;  // K bytes of a page within one row block
  constexpr uint32_t kVPage = D * BS;
  constexpr uint32_t kSPage = BS * L::G * 2;
  const int n_pages = (kv_end + BS - 1) / BS;
  const int32_t *bt_row = a.block_table + static_cast<int64_t>(seq) * a.bt_stride;
  int page_base = -(1 << 30);
  int my_blk = -1;
  for (int it = 0; it < n_iter; ++it) {
    const int g = it0 + it;  // ring position
    const int stage = g % NST;
    if (g >= NST) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(bar_empty + 8 * stage, ((g / NST) - 1) & 1, a.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) flag_status(a.status, PA_DEV_TIMEOUT);
        return false;
      }
    }
    const int lp0 = (tile_lo + it) * L::kPages;
    if (lp0 - page_base >= 32) {
      page_base = lp0;
      const int lp = page_base + lane;
      my_blk = -1;
      if (lp < n_pages && (lp + 1) * BS > kv_begin) {
        const int b = lp < a.bt_stride ? bt_row[lp] : -1;
        if (b >= 0 && b < a.num_blocks) my_blk = b;
        else flag_status(a.status, PA_DEV_BAD_BLOCK);
      }
    }
    const uint32_t st = smem_base + stage * L::kBytes;
#pragma unroll
    for (int p = 0; p < L::kPages; ++p) {
      const int blk = __shfl_sync(0xffffffffu, my_blk, lp0 + p - page_base);
      if (blk < 0) continue;  // past the sequence (or a bad entry): the consumers mask it
      const int64_t page = static_cast<int64_t>(blk) * a.hk + h;
      const int8_t *ksrc = a.k_cache + page * (BS * D) + lane * 16;
      const int8_t *vsrc = a.v_cache + page * (BS * D) + lane * 16;
#pragma unroll
      for (int i = 0; i < kPer; ++i) cp_async16(st + p * kKPage + koff[i], ksrc + i * 512);
#pragma unroll
      for (int i = 0; i < kPer; ++i) cp_async16(st + p * kVPage + voff[i], vsrc + i * 512);
      const uint8_t *kss = reinterpret_cast<const uint8_t *>(a.k_scale + page * BS * L::G);
      const uint8_t *vss = reinterpret_cast<const uint8_t *>(a.v_scale + page * BS * L::G);
#pragma unroll
      for (int i = 0; i < kSPer; ++i) {
        const int c = lane + 32 * i;
        if (c < 2 * kSChunks)
          cp_async16(st + p * kSPage + soff[i],
                     c < kSChunks ? kss + c * 16 : vss + (c - kSChunks) * 16);
      }
    }
    cp_async_arrive(bar_full + 8 * stage);
  }
  return true;
}

// Load 4 consecutive fp16 V scales (keys 4t..4t+3 of group g) as two half2
// words, zeroing keys outside [kv_begin, kv_end) (stale bytes may sit there).
template <class L>
__device__ __forceinline__ uint2 v_scales4(uint32_t st, int key, int g, bool edge, int key0,
                                           int kv_begin, int kv_end) {
  uint2 s = lds64(st + L::vs_off(key, g));
  if (edge) {
    const int k = key0 + key;
    if (k + 0 >= kv_end || k + 0 < kv_begin) s.x &= 0xffff0000u;
    if (k + 1 >= kv_end || k + 1 < kv_begin) s.x &= 0x0000ffffu;
    if (k + 2 >= kv_end || k + 2 < kv_begin) s.y &= 0xffff0000u;
    if (k + 3 >= kv_end || k + 3 < kv_begin) s.y &= 0x0000ffffu;
  }
  return s;
}

}  // namespace paq8
