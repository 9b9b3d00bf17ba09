// The fp8-key / 4-bit-value cache format at the attention load site: the
// staged page layout, the producer warp that fills it, and the conversions
// of its codes to fp16 operands.  Shared by the decode kernel of that format
// (attn_decode_f8v4.cu) and the generic kernel (attn_prefill.cu).
//   K: e4m3 codes, every value exact in fp16 (cvt.rn.f16x2.e4m3x2);
//   V: 4-bit indices, V' = idx * scale + zero with the key's fp16 scale and
//      zero, one fp16 FMA ("triton_turboquant_unified_attention.py", the
//      4-bit value load site).
#pragma once

#include "attn_common.cuh"

namespace paq8 {

// One pipeline stage of TILE keys:
//   K  [TILE][D] e4m3, token-major pages in the 128-byte swizzle pattern of
//      StageLayout (64-byte for D = 64); D = 256 rows are two halves
//   V  [pages][D][BS / 2] nibbles, channel-major pages (byte j of a channel
//      row: keys 2j (low nibble) and 2j + 1)
//   Vs [TILE] fp16 scales, Vz [TILE] fp16 zeros (pages in order)
template <int D, int BS, int TILE>
struct StageF8V4 {
  static constexpr int kD = D;
  static constexpr int kPages = TILE / BS;
  static constexpr int kRowBytes = D >= 128 ? 128 : D;
  static constexpr int kKBytes = TILE * D;
  static constexpr int kVOff = kKBytes;
  static constexpr int kVsOff = kVOff + TILE * D / 2;
  static constexpr int kVzOff = kVsOff + TILE * 2;
  static constexpr int kBytes = (kVzOff + TILE * 2 + 1023) / 1024 * 1024;
  static_assert(TILE % BS == 0 && TILE % 16 == 0, "tile");

  __device__ static __forceinline__ uint32_t k_off(int r, int b) {
    return StageLayout<D, BS, TILE>::k_off(r, b);
  }
  // byte holding keys (key, key + 1) of channel c (key even)
  __device__ static __forceinline__ uint32_t v_off(int c, int key) {
    return kVOff + (key / BS) * (D * BS / 2) + c * (BS / 2) + (key % BS) / 2;
  }
  __device__ static __forceinline__ uint32_t vs_off(int key) { return kVsOff + key * 2; }
  __device__ static __forceinline__ uint32_t vz_off(int key) { return kVzOff + key * 2; }
};

// The producer warp: the same walk as produce_tiles_lsu, copying per page its
// K rows (BS * D bytes), its V nibble page (D * BS / 2 bytes) and its BS
// scales and zeros.
template <class L, int BS, int NST>
__device__ __forceinline__ void produce_f8v4(const AttnArgs &a, uint32_t smem_base,
                                             uint32_t bar_full, uint32_t bar_empty, int seq,
                                             int h, int tile_lo, int n_iter, int kv_begin,
                                             int kv_end, int lane) {
  constexpr int D = L::kD;
  constexpr int kKChunks = BS * D / 16;
  constexpr int kKPer = kKChunks / 32;
  constexpr int kVChunks = D * BS / 32;  // (D * BS / 2) / 16
  constexpr int kVPer = kVChunks / 32;
  constexpr int kSChunks = BS * 2 / 16;  // scales (and as many zeros) of a page
  constexpr int kRowChunks = D / 16;
  static_assert(kKChunks % 32 == 0 && kVChunks % 32 == 0 && 2 * kSChunks <= 32, "chunks");
  uint32_t koff[kKPer];
#pragma unroll
  for (int i = 0; i < kKPer; ++i) {
    const int c = lane + 32 * i;
    koff[i] = L::k_off(c / kRowChunks, (c % kRowChunks) * 16);
  }
  constexpr uint32_t kKPage = BS * L::kRowBytes;
  constexpr uint32_t kVPage = D * BS / 2;
  const int n_pages = (kv_end + BS - 1) / BS;
  const int32_t *bt_row = a.block_table + static_cast<int64_t>(seq) * a.bt_stride;
  const uint8_t *kc = reinterpret_cast<const uint8_t *>(a.k_cache);
  const uint8_t *vc = reinterpret_cast<const uint8_t *>(a.v_cache);
  const uint8_t *vs = reinterpret_cast<const uint8_t *>(a.v_scale);
  const uint8_t *vz = reinterpret_cast<const uint8_t *>(a.v_zero);
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
    const uint32_t st = smem_base + stage * L::kBytes;
#pragma unroll
    for (int p = 0; p < L::kPages; ++p) {
      const int blk = __shfl_sync(0xffffffffu, my_blk, lp0 + p - page_base);
      if (blk < 0) continue;  // past the sequence (or a bad entry): the consumers mask it
      const int64_t page = static_cast<int64_t>(blk) * a.hk + h;
      const uint8_t *ksrc = kc + page * (BS * D) + lane * 16;
      const uint8_t *vsrc = vc + page * (BS * D / 2) + lane * 16;
#pragma unroll
      for (int i = 0; i < kKPer; ++i) cp_async16(st + p * kKPage + koff[i], ksrc + i * 512);
#pragma unroll
      for (int i = 0; i < kVPer; ++i)
        cp_async16(st + L::kVOff + p * kVPage + (lane + 32 * i) * 16, vsrc + i * 512);
      if (lane < 2 * kSChunks) {
        const bool zero = lane >= kSChunks;
        const int c = zero ? lane - kSChunks : lane;
        cp_async16(st + (zero ? L::kVzOff : L::kVsOff) + p * (BS * 2) + c * 16,
                   (zero ? vz : vs) + page * (BS * 2) + c * 16);
      }
    }
    cp_async_arrive(bar_full + 8 * stage);
  }
}

// The producer of the tcgen05 prefill kernel in this format: the same walk
// as produce_tiles, per page one 2-D TMA box for the K rows (the q8 K map:
// the pages have the same [BS][D] byte shape) and bulk copies of the V
// nibble page and of the scales and zeros, all completing on the stage's
// full barrier (D <= 128: one K box per page).
template <class L, int BS, int NST>
__device__ __forceinline__ void produce_tiles_f8v4_tma(const AttnArgs &a, const CUtensorMap *tmap_k,
                                                       uint32_t smem_base, uint32_t bar_full,
                                                       uint32_t bar_empty, int seq, int h,
                                                       int tile_lo, int n_iter, int kv_begin,
                                                       int kv_end, int lane) {
  constexpr int D = L::kD;
  static_assert(D <= 128, "one K box per page");
  constexpr uint32_t kKPage = BS * L::kRowBytes;
  constexpr uint32_t kVPage = D * BS / 2;
  constexpr uint32_t kPageTx = BS * D + kVPage + 4 * BS;
  const int n_pages = (kv_end + BS - 1) / BS;
  const int32_t *bt_row = a.block_table + static_cast<int64_t>(seq) * a.bt_stride;
  const uint8_t *vc = reinterpret_cast<const uint8_t *>(a.v_cache);
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
      mbar_arrive_expect_tx(full, nvalid * kPageTx);
#pragma unroll
      for (int p = 0; p < L::kPages; ++p) {
        if (blk[p] < 0) continue;
        const int64_t page = static_cast<int64_t>(blk[p]) * a.hk + h;
        tma_load_2d(st + p * kKPage, tmap_k, 0, static_cast<int32_t>(page * BS), full);
        bulk_load(st + L::kVOff + p * kVPage, vc + page * kVPage, kVPage, full);
        bulk_load(st + L::kVsOff + p * (BS * 2), a.v_scale + page * BS, BS * 2, full);
        bulk_load(st + L::kVzOff + p * (BS * 2), a.v_zero + page * BS, BS * 2, full);
      }
    }
    __syncwarp();
  }
}

// Two e4m3 values (byte 0 -> low half) -> fp16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint32_t v16) {
  uint32_t d;
  asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(d)
      : "r"(v16));
  return d;
}

// Four nibbles (keys k, k+1, k+2, k+3 of one channel: bits 0-3, 4-7, 8-11,
// 12-15 of w) -> two fp16x2 words of exact integers 0..15.
__device__ __forceinline__ void nibbles4_to_half2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t bias = 0x64006400u;  // (1024, 1024) in fp16
  const uint32_t a = (w & 0xfu) | ((w << 12) & 0xf0000u) | bias;          // keys k, k+1
  const uint32_t b = ((w >> 8) & 0xfu) | ((w << 4) & 0xf0000u) | bias;    // keys k+2, k+3
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

}  // namespace paq8
