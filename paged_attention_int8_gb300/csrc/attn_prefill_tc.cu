// Prefill kernel on the 5th-generation tensor cores (tcgen05, TMEM).
//
// Computes, for a q-block of 256 rows (BLOCK_Q = 256 / qpk tokens x the qpk
// q heads of one kv head, the GQA row tile of
// "triton_turboquant_unified_attention.py"):
//   out = softmax_j(scale * q . k_j) v_j over keys j <= seq_len - q_len + i,
//   lse = ln sum_j exp(scale * q . k_j),
// over the dequantized q8 pages, in 64-key tiles with an online softmax.
// In non-causal mode every query sees keys j < seq_len (seq_len may be below
// q_len); a sliding window keeps the last `window` keys of each query; a sink
// logit starts each row's softmax as one term with no value (the options of
// the AttnArgs visibility fields).  Tiles before the block's first visible
// key are not visited.
//
// Exact scores with one accumulator: each dequantized key value
// k = code * scale (exact in fp32, 7 x 11 significant bits) is split into two
// fp16 parts, hi = fp16(k) and lo = fp16(k - hi) (one fp16 FMA, exact while
// |k| >= 2^-7; below that the error is under 2^-25), and
// S = Q K_hi^T + Q K_lo^T accumulates both in the same TMEM columns.  q is
// rounded to fp16 (exact in the normal range).  V is dequantized to fp16
// (one rounding); P is fp16; the accumulators are fp32 in TMEM.
//
// The 256 rows are two 128-row halves (the MMA's M) that share every
// converted K/V tile, so the int8 -> fp16 work per FLOP is halved.  Both MMA
// A operands live in TMEM (q for QK, P for PV): shared memory then carries
// only the K/V tiles (B operands), not a re-read of q for every MMA.
// Warp roles (512 threads; warp w runs on SM sub-partition w % 4, and the
// MMA warp shares its sub-partition only with the producer and two softmax
// warps, so the ALU-heavy dequant warps never delay MMA issue; the others
// each hold two dequant and two softmax warps):
//   warp 5      TMA producer: int8 K/V pages + fp16 scales -> 4-stage ring
//   warp 1      MMA issuer and owner of the TMEM allocation.  The converged
//               warp issues through one elected lane, per tile j,
//               PV(j-1, half 0), QK(j, half 0), PV(j-1, half 1), QK(j, half 1):
//               while one half's softmax runs, the tensor core works on the
//               other half
//   warps 0, 2, 3, 14  K dequant: ring stage -> fp16 K_hi/K_lo (2-slot K
//               ring, a slot freed when both halves' QK MMAs complete)
//   warps 4, 15 V dequant: ring stage -> fp16 V' (2-slot V ring, freed when
//               both halves' PV MMAs complete); both in the canonical
//               128-byte-swizzle K-major layout
//   warps 6-9   softmax of half 0, warps 10-13 of half 1: one q row per
//               thread (its TMEM lane); write q (fp16) into TMEM; per tile read
//               S from TMEM, online softmax, write P (fp16) back into the same
//               TMEM columns as the PV MMA's A operand.  P is taken against
//               the max O is currently scaled to; only when a tile's P
//               sum would pass 2^15 (every P stays inside fp16) does the
//               lane raise that max to the row max, rescale O in TMEM and
//               redo the tile (exact: the final division uses the same
//               max); the epilogue reads O
// TMEM (512 columns): per half, the S/P buffer (64 columns), q (D/2
// columns: two fp16 per column) and O (D columns).  A half's next QK is
// issued after its PV of the previous tile, and tcgen05 MMAs from one thread
// execute in issue order, so the single S/P buffer is never overwritten
// early; the commit of QK(j) also implies PV(j-1) is done, so the softmax may
// rescale O as soon as S(j) is ready.
//
// The same kernel reads the fp8-key / 4-bit-value format (F8): the K
// dequant warps turn e4m3 keys into fp16 exactly (one part, so QK^T is one
// MMA pass with no K_lo), the V dequant warps form V' = idx * scale + zero
// per key, and the producer stages the K rows by TMA and the nibble pages,
// scales and zeros by bulk copies.
#include <type_traits>

#include "attn_common.cuh"
#include "attn_f8v4.cuh"
#include "tcgen05.cuh"
#include "launch.h"

namespace paq8 {

template <int D, int BS, bool F8>
struct TcCfg {
  static constexpr int kTile = 64;
  static constexpr int kHalves = 2;
  static constexpr int kRows = 128 * kHalves;
  static constexpr int kSt = 4;  // int8 staging stages (TMA)
  static constexpr int kWarps = 16;
  using L = std::conditional_t<F8, StageF8V4<D, BS, kTile>, StageLayout<D, BS, kTile>>;
  static constexpr int kKBytes = kTile * D * 2;  // one of K_hi, K_lo: [D/64][64 keys][128 B]
  static constexpr int kKSlot = 2 * kKBytes;     // K ring slot: hi then lo
  static constexpr int kVBytes = D * kTile * 2;  // V' ring slot: [D rows][64 keys]
  static constexpr int align1k(int x) { return (x + 1023) / 1024 * 1024; }
  static constexpr int kKOff = align1k(kSt * L::kBytes);
  static constexpr int kVOff = kKOff + 2 * kKSlot;
  static constexpr int kBarOff = kVOff + 2 * kVBytes;
  static constexpr int kSmem = kBarOff + 256 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kHalfCols = 256;  // per half: S/P at +0, q at +64, O at +128
  static constexpr uint32_t kQCol = 64;
  static constexpr uint32_t kOCol = 128;
  static constexpr float kMaxTileSum = 32768.0f;  // bound on a tile's P sum (so on every P)
  static_assert(D == 64 || D == 128, "tcgen05 prefill handles D = 64, 128");
  static_assert(kSmem <= 232448, "shared memory");
  static_assert(kSt <= 4, "staging barriers");
};

// barrier indices (8 bytes each, from kBarOff)
enum : int {
  kBarStFull = 0,    // [4] producer -> dequant (tx bytes)
  kBarStEmpty = 4,   // [4] dequant -> producer (6 warps)
  kBarKFull = 8,     // [2] K dequant -> MMA (4 warps)
  kBarKEmpty = 10,   // [2] commit after both halves' QK -> K dequant
  kBarVFull = 12,    // [2] V dequant -> MMA (2 warps)
  kBarVEmpty = 14,   // [2] commit after both halves' PV -> V dequant
  kBarSFull = 16,    // [half] commit after QK -> softmax of the half
  kBarPFull = 18,    // [half] softmax (P in TMEM) -> MMA (4 warps)
  kBarPvDone = 20,   // [half] commit after the last PV -> epilogue
  kBarQFull = 22,    // softmax (q written to TMEM) -> MMA (8 warps)
  kNumBars = 23
};

template <int D, int BS, bool F8>
__global__ void __launch_bounds__(512, 1)
    prefill_tc_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
  using C = TcCfg<D, BS, F8>;
  using L = typename C::L;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (smem_base - smem_u32(smem_raw));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y;

  // ---- q-block (heaviest first: later q-blocks see more keys)
  const int bx = a.n_qblocks - 1 - static_cast<int>(blockIdx.x);
  const int seq = find_seq(a.cu_seqlens_q, a.num_seqs, a.block_q, bx, lane);
  const int q_start = a.cu_seqlens_q[seq];
  const int q_end = a.cu_seqlens_q[seq + 1];
  const int q_len = q_end - q_start;
  const int tok0 = (bx - (q_start / a.block_q + seq)) * a.block_q;
  if (tok0 >= q_len) return;
  if (q_len == 1 && a.skip_single) return;
  if (q_end > a.num_tokens || q_start < 0) {
    if (threadIdx.x == 0) flag_status(a.status, PA_DEV_BAD_SEQ);
    return;
  }
  const int seq_len = a.seq_lens[seq];
  const int ctx = seq_len - q_len;
  if (a.causal ? ctx < 0 : seq_len < 0) {
    if (threadIdx.x == 0 && tok0 == 0) flag_status(a.status, PA_DEV_BAD_SEQ);
    return;
  }
  const int n_tok = min(a.block_q, q_len - tok0);
  const int n_rows = n_tok * a.qpk;
  // keys visible to some row of the block: [kv_begin, kv_end)
  const int kv_end = last_key(a, seq_len, q_len, tok0 + n_tok - 1) + 1;
  const int kv_begin = first_key(a, last_key(a, seq_len, q_len, tok0));
  if (kv_end == 0) {  // non-causal, seq_len == 0: no row sees a key
    for (int idx = warp; idx < n_tok; idx += C::kWarps)
      write_empty_rows<D>(a, q_start + tok0 + idx, h * a.qpk, a.qpk, lane);
    return;
  }
  // the block visits tiles t0 .. t0 + nt - 1; iteration j works on tile t0 + j
  const int t0 = kv_begin / C::kTile;
  const int nt = (kv_end + C::kTile - 1) / C::kTile - t0;
  // half 1 holds no valid row when the block is short: it is then skipped
  const int halves = n_rows > 128 ? 2 : 1;

  const uint32_t bars = smem_base + C::kBarOff;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const uint32_t tmem_slot = bars + 8 * kNumBars;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kSt; ++s) {
      mbar_init(bar(kBarStFull + s), 1);
      mbar_init(bar(kBarStEmpty + s), 6);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarKFull + s), 4);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 2);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarPFull + s), 4);
      mbar_init(bar(kBarPvDone + s), 1);
    }
    mbar_init(bar(kBarQFull), 8);
    fence_barrier_init();
  }
  if (warp == 1) tc::alloc(tmem_slot, C::kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::kBarOff + 8 * kNumBars);
  bool ok = true;

  if (warp == 5) {
    // ============================================================ producer
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      if constexpr (!F8) prefetch_tensormap(&tmap_v);
    }
    if constexpr (F8)
      produce_tiles_f8v4_tma<L, BS, C::kSt>(a, &tmap_k, smem_base, bar(kBarStFull),
                                            bar(kBarStEmpty), seq, h, t0, nt, kv_begin, kv_end,
                                            lane);
    else
      produce_tiles<L, BS, C::kSt>(a, &tmap_k, &tmap_v, smem_base, bar(kBarStFull),
                                   bar(kBarStEmpty), seq, h, t0, nt, kv_begin, kv_end, lane);
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    // The whole warp runs this loop (uniform values, no divergence); the
    // elected lane issues every MMA and commit.
    const uint32_t leader = tc::elect_one();
    constexpr uint32_t id_qk = tc::idesc_f16(128, 64);
    constexpr uint32_t id_qk_neg = id_qk | (1u << 14);  // negate B: K_lo is stored as -lo
    constexpr uint32_t id_pv = tc::idesc_f16(128, D);
    auto wait = [&](int i, uint32_t parity) { return __all_sync(0xffffffffu, mbar_wait(bar(i), parity)); };
    // O(half) += P(i, half) V'(i): A = P from the half's S/P columns
    auto issue_pv = [&](int i, int hf) -> bool {
      const int b = i & 1;
      if (hf == 0 && !wait(kBarVFull + b, (i >> 1) & 1)) return false;
      if (!wait(kBarPFull + hf, i & 1)) return false;
      tc::fence_after();
      const uint64_t v_desc = tc::desc_sw128(smem_base + C::kVOff + b * C::kVBytes);
      const uint32_t base = tmem + hf * C::kHalfCols;
#pragma unroll
      for (int ks = 0; ks < C::kTile / 16; ++ks)  // +32 bytes of K per step
        tc::mma_f16_ts_by(leader, base + C::kOCol, base + ks * 8, v_desc + 2 * ks, id_pv,
                          (i > 0 || ks > 0) ? 1u : 0u);
      return true;
    };
    // S(half) = q K_hi(j)^T - q (-K_lo(j))^T: A = q from the half's TMEM columns
    auto issue_qk = [&](int j, int hf) {
      const uint64_t k_desc = tc::desc_sw128(smem_base + C::kKOff + (j & 1) * C::kKSlot);
      const uint32_t base = tmem + hf * C::kHalfCols;
#pragma unroll
      for (int part = 0; part < (F8 ? 1 : 2); ++part)  // F8: exact keys, no K_lo part
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t koff = part * C::kKBytes + (ks >> 2) * (64 * 128) + (ks & 3) * 32;
          tc::mma_f16_ts_by(leader, base, base + C::kQCol + ks * 8, k_desc + (koff >> 4),
                            part ? id_qk_neg : id_qk, (part > 0 || ks > 0) ? 1u : 0u);
        }
      tc::commit_by(leader, bar(kBarSFull + hf));
    };
    ok = wait(kBarQFull, 0);
    tc::fence_after();
    for (int j = 0; ok && j < nt; ++j) {
      const int b = j & 1;
      for (int hf = 0; hf < halves; ++hf) {
        // the half's S/P buffer is free once PV(j - 1) is issued: MMAs from
        // this warp execute in order
        if (j >= 1 && !issue_pv(j - 1, hf)) { ok = false; break; }
        if (hf == 0 && !wait(kBarKFull + b, (j >> 1) & 1)) { ok = false; break; }
        tc::fence_after();
        issue_qk(j, hf);
      }
      if (!ok) break;
      tc::commit_by(leader, bar(kBarKEmpty + b));
      if (j >= 1) tc::commit_by(leader, bar(kBarVEmpty + (b ^ 1)));
    }
    for (int hf = 0; ok && hf < halves; ++hf) {
      if (!issue_pv(nt - 1, hf)) { ok = false; break; }
      tc::commit_by(leader, bar(kBarPvDone + hf));
    }
    __syncwarp();
  } else if (warp < 6 || warp >= 14) {
    // ============================================================ dequant
    // warps 0, 2, 3, 14: K (hi and lo parts), thread = one key row, D/2 channels
    // warps 4, 15: V', thread = D / 64 channel rows of one scale group, all 64 keys
    const bool k_side = warp != 4 && warp != 15;
    const int t = (k_side ? (warp == 14 ? 3 : warp == 0 ? 0 : warp - 1) : (warp == 4 ? 0 : 1)) * 32 +
                  lane;  // K: 0..127, V: 0..63
#pragma unroll 1
    for (int j = 0; j < nt; ++j) {
      const int sb = j % C::kSt, b = j & 1;
      if (!mbar_wait(bar(kBarStFull + sb), (j / C::kSt) & 1)) { ok = false; break; }
      const uint32_t st = smem_base + sb * L::kBytes;
      const int key0 = (t0 + j) * C::kTile;
      // keys outside [kv_begin, kv_end) may hold stale bytes: converted as zeros
      const bool tail = key0 + C::kTile > kv_end || key0 < kv_begin;
      if (k_side) {
        if (j >= 2 && !mbar_wait(bar(kBarKEmpty + b), ((j - 2) >> 1) & 1)) { ok = false; break; }
        const uint32_t kdst = smem_base + C::kKOff + b * C::kKSlot;
        const int r = t & 63;
        const int c0 = (t >> 6) * (D / 2);
        const bool dead = tail && (key0 + r >= kv_end || key0 + r < kv_begin);
        if constexpr (F8) {
          // e4m3 -> fp16 exactly; a row outside the visible keys becomes zeros
#pragma unroll
          for (int c = c0; c < c0 + D / 2; c += 16) {
            const uint4 codes = dead ? make_uint4(0u, 0u, 0u, 0u) : lds128(st + L::k_off(r, c));
            const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
            uint32_t hw[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              hw[2 * i] = e4m3x2_to_half2(cw[i]);
              hw[2 * i + 1] = e4m3x2_to_half2(cw[i] >> 16);
            }
            const int c16 = c / 8;
            sts128(kdst + tc::sw128_chunk(r, c16, 64), make_uint4(hw[0], hw[1], hw[2], hw[3]));
            sts128(kdst + tc::sw128_chunk(r, c16 + 1, 64), make_uint4(hw[4], hw[5], hw[6], hw[7]));
          }
        } else {
#pragma unroll
        for (int c = c0; c < c0 + D / 2; c += 16) {
          const uint4 codes = lds128(st + L::k_off(r, c));
          const uint32_t sbits = lds16(st + L::ks_off(r, c / 32));
          const uint32_t s2 = dead ? 0u : (sbits | (sbits << 16));
          const uint32_t ns2 = s2 ^ 0x80008000u;  // -scale
          uint32_t hw[8], lw[8];
          const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t lo, hi;
            codes4_to_half2(cw[i], lo, hi);
            // hi = fp16(code * s); lw = code * (-s) + hi = -lo (one rounding, exact);
            // the QK MMA of the lo part negates B, so it adds q . lo
            hw[2 * i] = hmul2_u32(lo, s2);
            hw[2 * i + 1] = hmul2_u32(hi, s2);
            asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(lw[2 * i]) : "r"(lo), "r"(ns2), "r"(hw[2 * i]));
            asm("fma.rn.f16x2 %0, %1, %2, %3;"
                : "=r"(lw[2 * i + 1])
                : "r"(hi), "r"(ns2), "r"(hw[2 * i + 1]));
          }
          const int c16 = c / 8;
          sts128(kdst + tc::sw128_chunk(r, c16, 64), make_uint4(hw[0], hw[1], hw[2], hw[3]));
          sts128(kdst + tc::sw128_chunk(r, c16 + 1, 64), make_uint4(hw[4], hw[5], hw[6], hw[7]));
          sts128(kdst + C::kKBytes + tc::sw128_chunk(r, c16, 64),
                 make_uint4(lw[0], lw[1], lw[2], lw[3]));
          sts128(kdst + C::kKBytes + tc::sw128_chunk(r, c16 + 1, 64),
                 make_uint4(lw[4], lw[5], lw[6], lw[7]));
        }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(kBarKFull + b));
          mbar_arrive(bar(kBarStEmpty + sb));
        }
      } else {
        if (j >= 2 && !mbar_wait(bar(kBarVEmpty + b), ((j - 2) >> 1) & 1)) { ok = false; break; }
        const uint32_t vrow = smem_base + C::kVOff + b * C::kVBytes;
        // D / 64 channel rows per thread, all in one scale group (for D = 128:
        // lanes 0-15 take channels 32w + lane and 32w + lane + 16), so the
        // per-key scales are loaded once for both rows
        constexpr int R = D / 64;
        int ch[R];
        if constexpr (R == 2) {
          ch[0] = (t >> 4) * 32 + (t & 15);
          ch[1] = ch[0] + 16;
        } else {
          ch[0] = t;
        }
        if constexpr (F8) {
#pragma unroll
          for (int key = 0; key < C::kTile; key += 16) {  // 16 keys: 8 bytes per channel row
            // the keys' scales and zeros, fp16 pairs (keys 2i, 2i+1); zero
            // outside the visible keys (stale bytes may sit there)
            const uint4 s01 = lds128(st + L::vs_off(key)), s23 = lds128(st + L::vs_off(key + 8));
            const uint4 z01 = lds128(st + L::vz_off(key)), z23 = lds128(st + L::vz_off(key + 8));
            uint32_t sc[8] = {s01.x, s01.y, s01.z, s01.w, s23.x, s23.y, s23.z, s23.w};
            uint32_t zr[8] = {z01.x, z01.y, z01.z, z01.w, z23.x, z23.y, z23.z, z23.w};
            if (tail) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int k0 = key0 + key + 2 * i;
                const uint32_t m = (k0 >= kv_end || k0 < kv_begin ? 0u : 0x0000ffffu) |
                                   (k0 + 1 >= kv_end || k0 + 1 < kv_begin ? 0u : 0xffff0000u);
                sc[i] &= m;
                zr[i] &= m;
              }
            }
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
              const uint2 nb = lds64(st + L::v_off(ch[rr], key));  // keys key .. key+15
              const uint32_t nw[4] = {nb.x, nb.x >> 16, nb.y, nb.y >> 16};
              uint32_t o[8];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t lo, hi;
                nibbles4_to_half2(nw[i], lo, hi);  // keys 4i, 4i+1 | 4i+2, 4i+3
                o[2 * i] = hfma2_u32(lo, sc[2 * i], zr[2 * i]);
                o[2 * i + 1] = hfma2_u32(hi, sc[2 * i + 1], zr[2 * i + 1]);
              }
              sts128(vrow + tc::sw128_chunk(ch[rr], key / 8, D), make_uint4(o[0], o[1], o[2], o[3]));
              sts128(vrow + tc::sw128_chunk(ch[rr], key / 8 + 1, D),
                     make_uint4(o[4], o[5], o[6], o[7]));
            }
          }
        } else {
        const int g = ch[0] / 32;
#pragma unroll
        for (int key = 0; key < C::kTile; key += 16) {  // 16 keys: one 16-byte load
          const uint4 s01 = lds128(st + L::vs_off(key, g));
          const uint4 s23 = lds128(st + L::vs_off(key + 8, g));
          uint32_t sc[8] = {s01.x, s01.y, s01.z, s01.w, s23.x, s23.y, s23.z, s23.w};
          if (tail) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int k0 = key0 + key + 2 * i;
              if (k0 >= kv_end || k0 < kv_begin) sc[i] &= 0xffff0000u;
              if (k0 + 1 >= kv_end || k0 + 1 < kv_begin) sc[i] &= 0x0000ffffu;
            }
          }
#pragma unroll
          for (int rr = 0; rr < R; ++rr) {
            const uint4 codes = lds128(st + L::v_off(ch[rr], key));
            uint32_t o[8];
            const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t lo, hi;
              codes4_to_half2(cw[i], lo, hi);
              o[2 * i] = hmul2_u32(lo, sc[2 * i]);
              o[2 * i + 1] = hmul2_u32(hi, sc[2 * i + 1]);
            }
            sts128(vrow + tc::sw128_chunk(ch[rr], key / 8, D), make_uint4(o[0], o[1], o[2], o[3]));
            sts128(vrow + tc::sw128_chunk(ch[rr], key / 8 + 1, D),
                   make_uint4(o[4], o[5], o[6], o[7]));
          }
        }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(kBarVFull + b));
          mbar_arrive(bar(kBarStEmpty + sb));
        }
      }
    }
  } else {
    // ============================================================ softmax
    const int hf = (warp - 6) >> 2;  // which 128-row half
    const int quarter = warp & 3;    // TMEM lanes this warp may access
    const int lrow = quarter * 32 + lane;
    const int row = hf * 128 + lrow;
    const uint32_t t_lane = tmem + hf * C::kHalfCols + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool valid = row < n_rows;
    const int tq = valid ? row / a.qpk : 0;
    const int hh = h * a.qpk + (valid ? row % a.qpk : 0);
    // visible keys of this row: [lo, limit]
    const int limit = valid ? last_key(a, seq_len, q_len, tok0 + tq) : kv_end - 1;
    const int lo = first_key(a, limit);
    const float sl2 = a.scale_log2;
    // q row -> fp16 pairs in this lane's q columns (the QK MMA's A operand)
    {
      const uint16_t *src = a.q + (static_cast<int64_t>(q_start + tok0 + tq) * a.hq + hh) * D;
      bool bad_q = false;
#pragma unroll 1
      for (int cb = 0; cb < D / 64; ++cb) {
        uint32_t qw[32];
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (valid) v = *reinterpret_cast<const uint4 *>(src + cb * 64 + c16 * 8);
          qw[4 * c16 + 0] = pack_half2(bf16_lo(v.x), bf16_hi(v.x));
          qw[4 * c16 + 1] = pack_half2(bf16_lo(v.y), bf16_hi(v.y));
          qw[4 * c16 + 2] = pack_half2(bf16_lo(v.z), bf16_hi(v.z));
          qw[4 * c16 + 3] = pack_half2(bf16_lo(v.w), bf16_hi(v.w));
          bad_q |= half2_nonfinite(qw[4 * c16]) || half2_nonfinite(qw[4 * c16 + 1]) ||
                   half2_nonfinite(qw[4 * c16 + 2]) || half2_nonfinite(qw[4 * c16 + 3]);
        }
        tc::st32(t_lane + C::kQCol + cb * 32, qw);
      }
      // q values beyond the fp16 range (|q| >= 65520) would give inf scores
      if (__any_sync(0xffffffffu, bad_q) && lane == 0) flag_status(a.status, PA_DEV_BAD_Q);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarQFull));
    }
    float m_used = -INFINITY;  // max the accumulator is scaled to (log2 units)
    float l = 0.0f;
    if (hf < halves) {
#pragma unroll 1
      for (int j = 0; j < nt; ++j) {
        if (!mbar_wait(bar(kBarSFull + hf), j & 1)) { ok = false; break; }
        tc::fence_after();
        const int key0 = (t0 + j) * C::kTile;
        const bool need_mask = key0 + C::kTile - 1 > limit || key0 < lo;
        uint32_t sr[64];
        // S from TMEM; masked columns -> -inf, the rest pre-scaled (only on
        // tiles that cross this row's causal limit)
        auto load_s = [&]() {
          tc::ld32(t_lane, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
          tc::ld32(t_lane + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
          tc::wait_ld();
          if (need_mask) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              sr[c] = __float_as_uint(key0 + c > limit || key0 + c < lo ? -INFINITY
                                                                         : __uint_as_float(sr[c]) * sl2);
          }
        };
        load_s();
        const float mul = need_mask ? 1.0f : sl2;
        // P = 2^(s * scale - m_used) as fp16 pairs and their fp32 sum; pairs
        // of columns go through the packed fp32 FMA and add
        uint32_t pw[32];
        float ts;
        auto exp_tile = [&]() {
          // no visible key yet (m_used = -inf): every column of this tile is
          // masked or the slow path below takes it, so any finite offset works
          const float neg_m = m_used == -INFINITY ? 0.0f : -m_used;
          const uint64_t mul2 = f32x2_pack(mul, mul), neg_m2 = f32x2_pack(neg_m, neg_m);
          uint64_t ls2[4] = {0, 0, 0, 0};  // +0.0f pairs
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float t0, t1;
            f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), mul2,
                                   neg_m2),
                         t0, t1);
            const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
            ls2[(c >> 1) & 3] = f32x2_add(ls2[(c >> 1) & 3], f32x2_pack(p0, p1));
            pw[c >> 1] = pack_half2(p0, p1);
          }
          float ls[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) f32x2_unpack(ls2[k], ls[2 * k], ls[2 * k + 1]);
          ts = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        };
        // The max the accumulator is scaled to moves only when this tile's
        // P would exceed C::kMaxTileSum (2^15, inside fp16): no row max is
        // taken on the common path.  A row with no max yet (m_used = -inf)
        // always takes the slow path, which sets it once a key is visible.
        exp_tile();
        const bool grow = !(ts <= C::kMaxTileSum) || m_used == -INFINITY;
        if (__any_sync(0xffffffffu, grow)) {
          float f = 1.0f;  // factor for what O and l hold
          load_s();        // S is still in TMEM (P not yet written)
          if (grow) {
            float e[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 64; ++c) e[c & 3] = fmaxf(e[c & 3], __uint_as_float(sr[c]) * mul);
            const float m_new = fmaxf(m_used, fmaxf(fmaxf(e[0], e[1]), fmaxf(e[2], e[3])));
            if (m_new > -INFINITY) {  // else nothing visible yet: P stays 0
              f = fast_exp2(m_used - m_new);  // 0 when the row had no max
              l *= f;
              m_used = m_new;
            }
          }
          exp_tile();
          if (j > 0) {
            // O holds tiles < j (PV(j - 1) completed before S(j) was
            // committed): scale it in TMEM
#pragma unroll 1
            for (int cb = 0; cb < D / 32; ++cb) {
              uint32_t orr[32];
              tc::ld32(t_lane + C::kOCol + cb * 32, orr);
              tc::wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * f);
              tc::st32(t_lane + C::kOCol + cb * 32, orr);
            }
            tc::wait_st();
          }
        }
        l += ts;
        tc::st32(t_lane, pw);
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + hf));
      }
      // ---- epilogue: O / l -> bf16, lse
      if (ok && mbar_wait(bar(kBarPvDone + hf), 0)) {
        tc::fence_after();
        // a sink joins the denominator as one term with no value: the same
        // sum as starting the softmax from (max = sink, sum = 1), taken here
        // so that P stays scaled to the scores' own max (no fp16 underflow
        // when the sink dominates)
        float o_mul = 1.0f;
        if (a.sinks) {
          const float sk = sink_log2(a, hh);
          const float mn = fmaxf(m_used, sk);
          if (mn > -INFINITY) {
            o_mul = fast_exp2(m_used - mn);
            l = l * o_mul + fast_exp2(sk - mn);
            m_used = mn;
          }
        }
        const float inv = o_mul / l;
        uint16_t *dst = a.out + (static_cast<int64_t>(q_start + tok0 + tq) * a.hq + hh) * D;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t orr[32];
          tc::ld32(t_lane + C::kOCol + cb * 32, orr);
          tc::wait_ld();
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 w;
              w.x = pack_bf162(__uint_as_float(orr[i]) * inv, __uint_as_float(orr[i + 1]) * inv);
              w.y = pack_bf162(__uint_as_float(orr[i + 2]) * inv, __uint_as_float(orr[i + 3]) * inv);
              w.z = pack_bf162(__uint_as_float(orr[i + 4]) * inv, __uint_as_float(orr[i + 5]) * inv);
              w.w = pack_bf162(__uint_as_float(orr[i + 6]) * inv, __uint_as_float(orr[i + 7]) * inv);
              *reinterpret_cast<uint4 *>(dst + cb * 32 + i) = w;
            }
          }
        }
        if (valid && a.lse)
          a.lse[static_cast<int64_t>(q_start + tok0 + tq) * a.hq + hh] = (m_used + log2f(l)) * kLn2;
      } else {
        ok = false;
      }
    }
  }
  if (!ok && lane == 0) flag_status(a.status, PA_DEV_TIMEOUT);

  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int BS, bool F8>
static cudaError_t launch_prefill_tc_t(const AttnArgs &a, const CUtensorMap &tk,
                                       const CUtensorMap &tv, cudaStream_t stream) {
  using C = TcCfg<D, BS, F8>;
  static DeviceOnce configured;
  cudaError_t e = configured.get(nullptr, [](int, int *) {
    return cudaFuncSetAttribute(prefill_tc_kernel<D, BS, F8>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.n_qblocks), static_cast<unsigned>(a.hk), 1);
  prefill_tc_kernel<D, BS, F8><<<grid, C::kWarps * 32, C::kSmem, stream>>>(a, tk, tv);
  return cudaGetLastError();
}

bool prefill_tc_supported(int d) { return d == 64 || d == 128; }

// rows of one q-block of the tcgen05 prefill kernel
int prefill_tc_rows() { return 256; }

cudaError_t launch_prefill_tc(const AttnArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                              int d, int bs, bool f8v4, cudaStream_t stream) {
#define PAQ8_TC_CASE(DD, BB)                                               \
  if (d == DD && bs == BB)                                                 \
    return f8v4 ? launch_prefill_tc_t<DD, BB, true>(a, tk, tv, stream)     \
                : launch_prefill_tc_t<DD, BB, false>(a, tk, tv, stream);
  PAQ8_TC_CASE(64, 16)
  PAQ8_TC_CASE(64, 32)
  PAQ8_TC_CASE(128, 16)
  PAQ8_TC_CASE(128, 32)
#undef PAQ8_TC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace paq8
