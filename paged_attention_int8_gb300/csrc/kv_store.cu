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
// formed as x * (1/s) (fused, unrounded) and rounded to an integer there
// unless it lies within 2^-15 of a rounding tie, where the IEEE quotient
// decides (the two round alike elsewhere: they differ by less than 1.6e-5
// for |x / s| <= 127.00002).
// Its roofline is HBM: per (token, kv head) it reads 4*D bytes and writes
// 2*(D + D/16) bytes.  The V side is bound instead by memory-instruction
// issue: each channel-major V page takes one byte per (token, channel).
#include "common.cuh"
#include "launch.h"
#include "q8_quant.cuh"

namespace paq8 {

// Lane-wise unsigned max of two pairs of 16-bit values.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

constexpr int kStoreWarps = 8;
constexpr int kStoreStages = 3;
constexpr int kStoreStageBytes = 32 * 64 + 32 * 8;  // 32 rows of 32 bf16, then 32 slots
constexpr int kStoreSmem = kStoreWarps * kStoreStages * kStoreStageBytes;

// 16-byte chunk j of lane `lane`'s 64-byte row within a stage: rotated by
// lane / 2 so that the 8 lanes of each quarter-warp read 8 distinct bank
// groups
__device__ __forceinline__ uint32_t row_chunk(int lane, int j) {
  return static_cast<uint32_t>(lane * 64 + ((j + (lane >> 1)) & 3) * 16);
}

// grid: (token-block slots, ceil(2 * hk * D/32 / kStoreWarps)); block: 32 x
// kStoreWarps; dynamic shared memory kStoreSmem.  Warp (blockIdx.y *
// kStoreWarps + w) takes one (kv head, group) of K (even) or of V (odd) and
// walks the blocks of 32 consecutive tokens blockIdx.x, blockIdx.x +
// gridDim.x, ...  Each lane copies its own row slice and slot two token
// blocks ahead into the warp's 3-stage ring (cp.async) and reads back only
// what it copied, so loads stay in flight without holding registers and no
// barrier is needed.
template <int D, int BS>
__global__ void __launch_bounds__(32 * kStoreWarps, 4) kv_store_kernel(
    const uint16_t *__restrict__ key, int64_t key_stride, const uint16_t *__restrict__ value,
    int64_t value_stride, const int64_t *__restrict__ slot_mapping, int32_t num_tokens,
    int32_t hk, int8_t *__restrict__ k_cache, uint16_t *__restrict__ k_scale,
    int8_t *__restrict__ v_cache, uint16_t *__restrict__ v_scale, int64_t num_slots,
    uint32_t *status, int32_t values_only, const int64_t *__restrict__ positions,
    int32_t max_position) {
  constexpr int G = D / 32;
  constexpr int block_size = BS;
  extern __shared__ __align__(16) uint8_t store_smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int combo = blockIdx.y * kStoreWarps + warp;
  // (kv head, group) of K (even combos) or V (odd); values_only: V only
  if (combo >= (values_only ? 1 : 2) * hk * G) return;
  const bool is_v = values_only || (combo & 1);
  const int hg = values_only ? combo : combo >> 1;
  const int h = hg / G, g = hg % G;
  const uint16_t *src = (is_v ? value : key) + h * D + g * 32;
  const int64_t stride = is_v ? value_stride : key_stride;
  const int n_tblocks = (num_tokens + 31) / 32;
  const uint32_t ring = smem_u32(store_smem) + warp * (kStoreStages * kStoreStageBytes);
  // copies of token block tb into a stage (one commit group per call, empty
  // past the end).  Each token's 64-byte slice is two 32-byte sectors; in
  // copy j the lanes 2i and 2i+1 fetch the two halves of sector j / 2 of
  // token 2i + (j & 1), so every request covers whole sectors.
  auto issue = [&](int tb, int stage) {
    if (tb < n_tblocks) {
      const uint32_t dst = ring + stage * kStoreStageBytes;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tl = (lane & ~1) | (j & 1);           // token (lane) served
        const int chunk = 2 * (j >> 1) + (lane & 1);    // its 16-byte chunk
        const int64_t n = static_cast<int64_t>(tb) * 32 + tl;
        if (n < num_tokens)
          cp_async_16(dst + row_chunk(tl, chunk), src + n * stride + 8 * chunk);
      }
      const int64_t n = static_cast<int64_t>(tb) * 32 + lane;
      if (n < num_tokens) cp_async_8(dst + 32 * 64 + lane * 8, slot_mapping + n);
    }
    cp_async_commit();
  };
  int tb = blockIdx.x;
  issue(tb, 0);
  issue(tb + gridDim.x, 1);
#pragma unroll 1
  for (int i = 0; tb < n_tblocks; ++i, tb += gridDim.x) {
    const int stage = i % kStoreStages;
    issue(tb + 2 * gridDim.x, (i + 2) % kStoreStages);
    cp_async_wait<2>();  // this lane's copies of `stage` have landed
    __syncwarp();        // ... and those of its partner lane (half of its row)
    const int64_t n = static_cast<int64_t>(tb) * 32 + lane;
    const uint32_t sbase = ring + stage * kStoreStageBytes;
    // Every lane runs the whole body (the V stores below are warp-wide);
    // lanes without a token, padding rows and bad slots store nothing.
    int64_t slot = -1;
    if (n < num_tokens)
      asm volatile("ld.shared.s64 %0, [%1];" : "=l"(slot) : "r"(sbase + 32 * 64 + lane * 8));
    if (slot >= num_slots) {
      if (combo == 0 && !values_only) flag_status(status, PA_DEV_BAD_SLOT);
      slot = -1;
    }
    // the fused store skips a token whose rotation position is outside the
    // table (its keys are skipped and flagged by the key kernel)
    if (positions && slot >= 0) {
      const int64_t pos = positions[n];
      if (pos < 0 || pos >= max_position) slot = -1;
    }
    const bool active = slot >= 0;

    // ---- group scale from the group max
    uint32_t xw[16];  // the lane's 32 bf16 values, two per word
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = lds128(sbase + row_chunk(lane, j));
      xw[4 * j] = v.x;
      xw[4 * j + 1] = v.y;
      xw[4 * j + 2] = v.z;
      xw[4 * j + 3] = v.w;
    }
    // group max |x| on the bf16 bit patterns, two at a time: with the sign
    // cleared, their unsigned order is that of |x| (finite values)
    uint32_t m2 = 0u;
#pragma unroll
    for (int k = 0; k < 16; ++k) m2 = max_u16x2(m2, xw[k] & 0x7fff7fffu);
    const float amax = __uint_as_float(max(m2 & 0xffffu, m2 >> 16) << 16);
    const float sc = group_scale(amax);
    const float rs = __frcp_rn(sc);

    // ---- codes.  c = the integer nearest to q = x * (1/s), taken exactly
    // from one fused multiply-add of 1.5 * 2^23 (its low byte is then the
    // code); d = q - c from a second one.  q and the IEEE quotient x / s
    // differ by under 7.6e-6 (|x / s| <= 127.00002, one rounding of 1/s),
    // and RN(x / s) by under 1.6e-5, so where |d| < 1/2 - 2^-15 all three
    // round to c and nearest even is also half away from zero; no clamp is
    // needed.  Values closer to a tie are marked and decided exactly.
    constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
    constexpr float kFar = 0.5f - 0x1p-15f;
    const uint64_t rs2 = f32x2_pack(rs, rs);
    const uint64_t shift2 = f32x2_pack(kShift, kShift);
    const uint64_t minus1 = f32x2_pack(-1.0f, -1.0f);
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t tb2[4];
      float d[4], nc[4];
      bool near = false;  // a value of this word within 2^-15 of a tie
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t xx = xw[2 * k + u];
        const uint64_t x2 = f32x2_pack(bf16_lo(xx), bf16_hi(xx));
        const uint64_t t2 = f32x2_fma(x2, rs2, shift2);       // 1.5 * 2^23 + c
        const uint64_t nc2 = f32x2_fma(t2, minus1, shift2);   // -c, exact
        const uint64_t d2 = f32x2_fma(x2, rs2, nc2);          // x * rs - c
        float t0, t1;
        f32x2_unpack(t2, t0, t1);
        f32x2_unpack(d2, d[2 * u], d[2 * u + 1]);
        f32x2_unpack(nc2, nc[2 * u], nc[2 * u + 1]);
        tb2[2 * u] = __float_as_uint(t0);
        tb2[2 * u + 1] = __float_as_uint(t1);
        near = near || fabsf(d[2 * u]) >= kFar || fabsf(d[2 * u + 1]) >= kFar;
      }
      // Values within 2^-15 of a tie (with bf16 inputs, e.g. every x = max/2
      // exactly) take the code of the IEEE quotient, decided without a
      // divide from the half-integer h = c + sign(d) / 2 they lie next to.
      // Patched here so that the words stay in registers.
      if (near && active) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (fabsf(d[e]) >= kFar) {
            const uint32_t xx = xw[2 * k + (e >> 1)];
            const float h = __fsub_rn(copysignf(0.5f, d[e]), nc[e]);
            tb2[e] = tie_code_bits((e & 1) ? bf16_hi(xx) : bf16_lo(xx), sc, h);
          }
      }
      w[k] = __byte_perm(__byte_perm(tb2[0], tb2[1], 0x0040), __byte_perm(tb2[2], tb2[3], 0x0040),
                         0x5410);
    }
    const uint16_t sbits = __half_as_ushort(__float2half_rn(sc));
    const int64_t blk = active ? slot / block_size : 0;
    const int64_t off = active ? slot % block_size : 0;
    const int64_t page = blk * hk + h;
    if (!is_v) {
      // K: token-major page row, 32 codes (one sector) of group g; scale
      // [page][bs][G].  Lanes 2i and 2i+1 write the two halves of token
      // 2i's sector in one store and of token 2i+1's in the next, so each
      // store covers whole sectors: they swap the half the other one writes.
      const int64_t row = page * block_size + off;
      uint8_t *mine = reinterpret_cast<uint8_t *>(k_cache + row * D + g * 32);
      const bool odd = lane & 1;
      uint32_t send[4], recv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        send[k] = odd ? w[k] : w[4 + k];
        recv[k] = __shfl_xor_sync(0xffffffffu, send[k], 1);
      }
      uint8_t *other = reinterpret_cast<uint8_t *>(
          __shfl_xor_sync(0xffffffffu, reinterpret_cast<uintptr_t>(mine), 1));
      const bool other_active = __shfl_xor_sync(0xffffffffu, active ? 1 : 0, 1) != 0;
      // store 1: the even lane's token (even lane: bytes 0-15, odd: 16-31)
      if (odd ? other_active : active)
        *reinterpret_cast<uint4 *>((odd ? other : mine) + (odd ? 16 : 0)) =
            odd ? make_uint4(recv[0], recv[1], recv[2], recv[3])
                : make_uint4(w[0], w[1], w[2], w[3]);
      // store 2: the odd lane's token
      if (odd ? active : other_active)
        *reinterpret_cast<uint4 *>((odd ? mine : other) + (odd ? 16 : 0)) =
            odd ? make_uint4(w[4], w[5], w[6], w[7])
                : make_uint4(recv[0], recv[1], recv[2], recv[3]);
      if (active) k_scale[row * G + g] = sbits;
    } else {
      // V: channel-major pages, channel c of this token at (page * D + c) * bs + off;
      // scale [page][G][bs]
      if (active) v_scale[(page * G + g) * block_size + off] = sbits;
      // A run of lanes that fills one whole page in slot order (BS lanes with
      // offsets 0 .. BS-1 of one page: prefill chunks, cache population) is
      // written as 16-byte rows: the codes are transposed through shared
      // memory (the stage, no longer needed) so that lane c gathers channel
      // c's bytes of the run.  Other lanes store their 32 bytes one by one.
      constexpr int kRun = BS;  // lanes per page
      const int64_t base = slot - (lane % kRun);
      const int64_t lead = __shfl_sync(0xffffffffu, base, lane & ~(kRun - 1));
      const bool fits = active && off == lane % kRun && base == lead;
      const uint32_t ball = __ballot_sync(0xffffffffu, fits);
      const uint32_t run_mask = kRun == 32 ? 0xffffffffu : (0xffffu << (lane & 16));
      const bool whole = (ball & run_mask) == run_mask;
      if (ball == 0xffffffffu || (kRun == 16 && (ball & 0xffffu) == 0xffffu) ||
          (kRun == 16 && (ball >> 16) == 0xffffu)) {
        // T[k][lane]: word k (codes of channels 4k .. 4k+3) of token `lane`;
        // a row stride of 36 words keeps the gathers below free of conflicts
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(sbase + (k * 36 + lane) * 4), "r"(w[k])
                       : "memory");
        __syncwarp();
        const int c = lane;  // channel within the group
        const uint32_t sel = (c & 3) | (((c & 3) + 4) << 4);
#pragma unroll
        for (int p = 0; p < 2; ++p) {  // BS 16: page half p; BS 32: bytes 16p .. 16p+15
          const uint32_t rbase = sbase + ((c >> 2) * 36 + 16 * p) * 4;
          const uint4 a0 = lds128(rbase), a1 = lds128(rbase + 16);
          const uint4 a2 = lds128(rbase + 32), a3 = lds128(rbase + 48);
          uint4 o;
          o.x = __byte_perm(__byte_perm(a0.x, a0.y, sel), __byte_perm(a0.z, a0.w, sel), 0x5410);
          o.y = __byte_perm(__byte_perm(a1.x, a1.y, sel), __byte_perm(a1.z, a1.w, sel), 0x5410);
          o.z = __byte_perm(__byte_perm(a2.x, a2.y, sel), __byte_perm(a2.z, a2.w, sel), 0x5410);
          o.w = __byte_perm(__byte_perm(a3.x, a3.y, sel), __byte_perm(a3.z, a3.w, sel), 0x5410);
          // the run holding tokens 16p .. 16p+15
          const int src_lane = kRun == 16 ? 16 * p : 0;
          const uint32_t run_ok = kRun == 16 ? (ball >> (16 * p)) & 0xffffu : ball;
          const int64_t run_page = __shfl_sync(0xffffffffu, page, src_lane);
          if (run_ok == (kRun == 16 ? 0xffffu : 0xffffffffu)) {
            int8_t *dst = v_cache + (run_page * D + g * 32 + c) * block_size +
                          (kRun == 16 ? 0 : 16 * p);
            *reinterpret_cast<uint4 *>(dst) = o;
          }
        }
      }
      if (active && !whole) {
        int8_t *vdst = v_cache + (page * D + g * 32) * block_size + off;
#pragma unroll
        for (int k = 0; k < 32; ++k)
          vdst[static_cast<int64_t>(k) * block_size] =
              static_cast<int8_t>((w[k >> 2] >> (8 * (k & 3))) & 0xffu);
      }
    }
    __syncwarp();  // the stage (and its transpose) is refilled next iteration
  }
  cp_async_wait<0>();
}

// token-block slots of the grid
template <int D, int BS>
static cudaError_t store_grid_x(int n_tblocks, unsigned grid_y, int32_t blocks_per_sm,
                                unsigned *grid_x) {
  // blocks of the kernel resident at once on the current device
  static DeviceOnce resident_blocks;
  int res = 0;
  cudaError_t e = resident_blocks.get(&res, [](int dev, int *v) {
    cudaError_t err = cudaFuncSetAttribute(
        kv_store_kernel<D, BS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStoreSmem);
    if (err != cudaSuccess) return err;
    int sms = 0, per_sm = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kv_store_kernel<D, BS>,
                                                        32 * kStoreWarps, kStoreSmem);
    if (err != cudaSuccess) return err;
    *v = (sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  static DeviceOnce sm_count;
  int sms = 0;
  e = sm_count.get(&sms, [](int dev, int *v) {
    return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
  });
  if (e != cudaSuccess) return e;
  if (blocks_per_sm > 0 && sms > 0 && static_cast<int64_t>(sms) * blocks_per_sm < res)
    res = sms * blocks_per_sm;
  const unsigned resident = static_cast<unsigned>(res);
  // up to 16 waves: one block per token block (every block starts at once
  // with its own loads); beyond that, one resident set of blocks that walks
  // the token blocks with its loads two steps ahead
  const unsigned want = (resident + grid_y - 1) / grid_y;
  const unsigned n = static_cast<unsigned>(n_tblocks);
  // (a capped grid stays persistent: it shares the SMs with other work)
  *grid_x = blocks_per_sm == 0 && n <= 16 * want ? n : (n < want ? n : want);
  return cudaSuccess;
}

static cudaError_t launch_store(const uint16_t *key, int64_t key_stride, const uint16_t *value,
                                int64_t value_stride, const int64_t *slot_mapping,
                                int32_t num_tokens, int32_t hk, int32_t d, int8_t *k_cache,
                                uint16_t *k_scale, int8_t *v_cache, uint16_t *v_scale,
                                int32_t num_blocks, int32_t block_size, uint32_t *status,
                                int32_t values_only, const int64_t *positions,
                                int32_t max_position, cudaStream_t stream,
                                int32_t blocks_per_sm) {
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
  const dim3 block(32 * kStoreWarps);
  const int n_tblocks = (num_tokens + 31) / 32;
  const int combos = (values_only ? 1 : 2) * hk * (d / 32);
  const unsigned grid_y = static_cast<unsigned>((combos + kStoreWarps - 1) / kStoreWarps);
  unsigned grid_x = 0;
#define PAQ8_STORE_CASE(DD, BB)                                                               \
  if (d == DD && block_size == BB) {                                                          \
    if (cudaError_t e = store_grid_x<DD, BB>(n_tblocks, grid_y, blocks_per_sm, &grid_x); e != cudaSuccess)  \
      return e;                                                                               \
    kv_store_kernel<DD, BB><<<dim3(grid_x, grid_y), block, kStoreSmem, stream>>>(              \
        key, key_stride, value, value_stride, slot_mapping, num_tokens, hk, k_cache, k_scale, \
        v_cache, v_scale, num_slots, status, values_only, positions, max_position);           \
    return cudaGetLastError();                                                                \
  }
  PAQ8_STORE_CASE(64, 16)
  PAQ8_STORE_CASE(64, 32)
  PAQ8_STORE_CASE(128, 16)
  PAQ8_STORE_CASE(128, 32)
  PAQ8_STORE_CASE(256, 16)
  PAQ8_STORE_CASE(256, 32)
#undef PAQ8_STORE_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_kv_store(const uint16_t *key, int64_t key_stride, const uint16_t *value,
                            int64_t value_stride, const int64_t *slot_mapping,
                            int32_t num_tokens, int32_t hk, int32_t d, int8_t *k_cache,
                            uint16_t *k_scale, int8_t *v_cache, uint16_t *v_scale,
                            int32_t num_blocks, int32_t block_size, uint32_t *status,
                            cudaStream_t stream) {
  return launch_store(key, key_stride, value, value_stride, slot_mapping, num_tokens, hk, d,
                      k_cache, k_scale, v_cache, v_scale, num_blocks, block_size, status, 0,
                      nullptr, 0, stream, 0);
}

// The values of the fused norm and rotation store (launch.h).
cudaError_t launch_kv_store_values(const uint16_t *value, int64_t value_stride,
                                   const int64_t *slot_mapping, int32_t num_tokens, int32_t hk,
                                   int32_t d, int8_t *v_cache, uint16_t *v_scale,
                                   int32_t num_blocks, int32_t block_size, uint32_t *status,
                                   const int64_t *positions, int32_t max_position,
                                   cudaStream_t stream, int32_t blocks_per_sm) {
  return launch_store(value, value_stride, value, value_stride, slot_mapping, num_tokens, hk, d,
                      nullptr, nullptr, v_cache, v_scale, num_blocks, block_size, status, 1,
                      positions, max_position, stream, blocks_per_sm);
}

}  // namespace paq8
