// merge_attn_states: the attention of queries over the union of two disjoint
// key sets, from their attention over each set -- the log-sum-exp merge
// `_merge_lse_(out, lse, other, other_lse)` of "shared/attention_kit.py"
// (the page keeps base-2 LSEs; this library's LSE is natural-log), the same
// identity the split-KV reduce applies to its segments.
//
// Per row (one query token and q head): M = max(lse_a, lse_b),
// e_x = exp(lse_x - M), out = (e_a out_a + e_b out_b) / (e_a + e_b) in fp32,
// rounded to bf16; lse = M + ln(e_a + e_b).  A row whose two LSEs are both
// -inf (no key on either side) gets out = 0 and lse = -inf.
//
// HBM bound: per row it reads 2 * D * 2 + 8 bytes and writes D * 2 + 4.  One
// thread per 16-byte chunk (8 channels) of a row, grid-stride; a row's D / 8
// chunks (8, 16 or 32) lie inside one warp, so the row's LSE is read by all
// its threads before one of them writes the merged LSE (which may overwrite
// lse_a or lse_b in place).
#include "common.cuh"
#include "launch.h"
#include "merge.h"

namespace paq8 {

template <int D>
__global__ void __launch_bounds__(256) merge_states_kernel(
    const uint16_t *__restrict__ out_a, const float *__restrict__ lse_a,
    const uint16_t *__restrict__ out_b, const float *__restrict__ lse_b, uint16_t *out,
    float *lse, int64_t num_rows) {
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  static_assert(32 % kChunks == 0, "a row must not straddle two warps");
  const int64_t total = num_rows * kChunks;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // warp-uniform trip count: every lane reaches the __syncwarp below
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < total; base += stride) {
    const int64_t c = base + threadIdx.x;
    const bool active = c < total;
    const int64_t row = c / kChunks;
    float la = -INFINITY, lb = -INFINITY;
    uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
    if (active) {
      la = lse_a[row];
      lb = lse_b[row];
      va = *reinterpret_cast<const uint4 *>(out_a + c * 8);
      vb = *reinterpret_cast<const uint4 *>(out_b + c * 8);
    }
    __syncwarp();  // every lane of this row has read both LSEs and both chunks
    if (!active) continue;
    const float m = fmaxf(la, lb);
    float wa = 0.0f, wb = 0.0f, merged = -INFINITY;
    if (m > -INFINITY) {
      const float ea = expf(la - m), eb = expf(lb - m);
      const float sum = ea + eb;
      wa = ea / sum;
      wb = eb / sum;
      merged = m + logf(sum);
    }
    const uint32_t a[4] = {va.x, va.y, va.z, va.w};
    const uint32_t b[4] = {vb.x, vb.y, vb.z, vb.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = bf16_lo(a[i]) * wa + bf16_lo(b[i]) * wb;
      const float hi = bf16_hi(a[i]) * wa + bf16_hi(b[i]) * wb;
      o[i] = pack_bf162(lo, hi);
    }
    *reinterpret_cast<uint4 *>(out + c * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    if (lse && c % kChunks == 0) lse[row] = merged;
  }
}

cudaError_t launch_merge_states(const uint16_t *out_a, const float *lse_a, const uint16_t *out_b,
                                const float *lse_b, uint16_t *out, float *lse, int64_t num_rows,
                                int32_t d, cudaStream_t stream) {
  static DeviceOnce sm_count;
  int sms = 0;
  cudaError_t e = sm_count.get(&sms, [](int dev, int *v) {
    return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
  });
  if (e != cudaSuccess) return e;
  const int64_t chunks = num_rows * (d / 8);
  const int64_t blocks_needed = (chunks + 255) / 256;
  // at most 8 blocks of 256 per SM resident at once; beyond that, grid-stride
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 8;
  const unsigned grid = static_cast<unsigned>(blocks_needed < cap ? blocks_needed : cap);
  switch (d) {
    case 64:
      merge_states_kernel<64><<<grid, 256, 0, stream>>>(out_a, lse_a, out_b, lse_b, out, lse, num_rows);
      break;
    case 128:
      merge_states_kernel<128><<<grid, 256, 0, stream>>>(out_a, lse_a, out_b, lse_b, out, lse, num_rows);
      break;
    case 256:
      merge_states_kernel<256><<<grid, 256, 0, stream>>>(out_a, lse_a, out_b, lse_b, out, lse, num_rows);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace paq8
