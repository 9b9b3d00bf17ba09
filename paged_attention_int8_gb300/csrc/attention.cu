// paged_attention dispatch: tensor maps, kernel choice, and the merge of the
// split-KV segments.
//
// One call may launch up to three kernels on the caller's stream:
//  * decode_kernel  -- single-token sequences when Hq/Hk <= 8 (swap-AB form),
//                      split into KV segments (the pages' 3D kernel);
//  * prefill_tc_kernel -- multi-token sequences on tcgen05/TMEM, q-blocks of
//                      256/qpk tokens (D = 64, 128 with Hq/Hk <= 8);
//  * prefill_kernel -- otherwise every other sequence on mma.sync, in
//                      q-blocks of 64/qpk tokens (the pages' unified 2D
//                      kernel); it also takes the single-token rows when
//                      Hq/Hk > 8;
//  * reduce_kernel  -- merges the segment triples of split rows by
//                      log-sum-exp (the pages' reduce_segments step).
// Over the fp8-key / 4-bit-value format the same dispatch runs the kernels'
// instantiations for that format (decode_f8v4_kernel for the decode rows).
// A batch that holds only decode rows (max_query_len == 1) launches no
// prefill kernel; both kernels exit at once for rows that are not theirs.
#include <algorithm>
#include <mutex>

#include "attn_common.cuh"
#include "launch.h"

namespace paq8 {

cudaError_t launch_decode(const AttnArgs &a, const CUtensorMap &tk, const CUtensorMap &tv, int d,
                          int bs, cudaStream_t stream);
cudaError_t launch_prefill(const AttnArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                           int d, int bs, bool f8v4, cudaStream_t stream);
cudaError_t launch_prefill_tc(const AttnArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                              int d, int bs, bool f8v4, cudaStream_t stream);
cudaError_t launch_decode_f8v4(const AttnArgs &a, int d, int bs, cudaStream_t stream);
bool prefill_tc_supported(int d);
int prefill_tc_rows();
int decode_tile(int d);
constexpr int kPrefillTile = 64;

// Merge of the segment triples of single-token sequences, written from the
// online-softmax merge rule (the pages' reduce_segments is not shown):
//   M = max m_k;  w_k = 2^(m_k - M);  out = sum w_k acc_k / sum w_k l_k;
//   lse = (M + log2 sum w_k l_k) * ln 2.
// One warp per (sequence, q head); the segments that exist are those the
// kernel that wrote them counts (segments_of over the visible keys).
template <int D>
__global__ void __launch_bounds__(128) reduce_kernel(const float *__restrict__ part_acc,
                                                     const float *__restrict__ part_ml,
                                                     const int32_t *__restrict__ cu,
                                                     const int32_t *__restrict__ seq_lens,
                                                     int32_t num_seqs, int32_t num_tokens,
                                                     int32_t hq, int32_t num_splits,
                                                     int32_t seg_tile, int32_t seg_tiles,
                                                     int32_t window, uint16_t *__restrict__ out,
                                                     float *__restrict__ lse) {
  constexpr int V = D / 32;  // channels per lane
  // launched as a programmatic dependent of the decode / prefill kernel:
  // wait for that grid's partials before reading anything
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (gw >= static_cast<int64_t>(num_seqs) * hq) return;
  const int seq = static_cast<int>(gw / hq);
  const int hh = static_cast<int>(gw % hq);
  const int q0 = cu[seq];
  if (cu[seq + 1] - q0 != 1 || q0 < 0 || q0 >= num_tokens) return;
  const int L = seq_lens[seq];
  if (L < 1) return;
  const int kv_begin = window > 0 ? max(0, L - window) : 0;
  const int nseg = segments_of(kv_begin, L, seg_tile, seg_tiles, num_splits);
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
  // all segments' rows are independent loads: issue them together
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) {
    if (k < nseg) {
      const float wk = __shfl_sync(0xffffffffu, w, k);
      const float *src = part_acc + (prow + k) * D + lane * V;
#pragma unroll
      for (int v = 0; v < V; v += 2) {
        const float2 x = *reinterpret_cast<const float2 *>(src + v);
        acc[v] = fmaf(wk, x.x, acc[v]);
        acc[v + 1] = fmaf(wk, x.y, acc[v + 1]);
      }
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

// 2-D byte map: `rows` rows of `row_bytes`, boxes of box_x bytes x box_y rows.
static bool encode_map(CUtensorMap *map, const void *base, int64_t rows, int row_bytes, int box_x,
                       int box_y, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_x), static_cast<cuuint32_t>(box_y)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int32_t auto_num_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t max_query_len,
                        int32_t max_seq_len) {
  (void)max_query_len;
  // ~1024 keys per segment (measured best on the decode batch with four
  // decode CTAs per SM), at most 16 segments (the pages' default count), and
  // no more than ~8192 CTAs in all: past that, more segments only add
  // partials to merge (measured on the mixed batch)
  int32_t ns = (max_seq_len + 1023) / 1024;
  const int64_t units = static_cast<int64_t>(num_seqs > 0 ? num_seqs : 1) *
                        (num_kv_heads > 0 ? num_kv_heads : 1);
  const int64_t cap = (8192 + units - 1) / units;
  if (ns > cap) ns = static_cast<int32_t>(cap);
  return ns < 1 ? 1 : (ns > kMaxSplits ? kMaxSplits : ns);
}

// The side stream (launch.h) on which the tcgen05 prefill kernel runs beside
// the decode kernel of a mixed batch (one is bound by the tensor cores, the
// other by HBM), and the fused store's values beside its keys.
static std::mutex g_side_mu;
static SideStream g_side[64];

cudaError_t side_stream(SideStream **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream &ss = g_side[dev];
  if (!ss.s) {
    int lo = 0, hi = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithPriority(&ss.s, cudaStreamNonBlocking, hi)) != cudaSuccess)
      return e;
    if ((e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &ss;
  return cudaSuccess;
}

cudaError_t launch_paged_attention(const AttnLaunch &L, cudaStream_t stream) {
  AttnArgs a{};
  a.q = static_cast<const uint16_t *>(L.q);
  a.cu_seqlens_q = L.cu;
  a.seq_lens = L.seq_lens;
  a.block_table = L.block_table;
  a.k_cache = static_cast<const int8_t *>(L.k_cache);
  a.v_cache = static_cast<const int8_t *>(L.v_cache);
  a.k_scale = static_cast<const uint16_t *>(L.k_scale);
  a.v_scale = static_cast<const uint16_t *>(L.v_scale);
  a.v_zero = static_cast<const uint16_t *>(L.v_zero);
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
  a.num_splits = L.num_splits;
  a.scale_log2 = L.softmax_scale * kLog2e;
  a.causal = L.causal ? 1 : 0;
  a.window = L.window;
  a.sinks = L.sinks;
  a.test_timeout = L.test_timeout ? 1 : 0;
  a.wait_limit_ns = L.test_timeout ? kTestWaitLimitNs : kWaitLimitNs;
  a.part_acc = reinterpret_cast<float *>(L.workspace + 256);
  a.part_ml = a.part_acc + static_cast<int64_t>(L.num_seqs) * L.hq * L.num_splits * L.d;

  const bool use_decode = a.qpk <= 8;
  const bool use_prefill = !use_decode || L.max_query_len > 1;
  const int64_t pages = static_cast<int64_t>(L.num_blocks) * L.hk;
  CUtensorMap tk = {}, tv = {};
  const int krow = L.d >= 128 ? 128 : L.d;
  // K pages have one [bs][D] byte shape in both formats; the fp8 / 4-bit
  // format's V pages are copied whole (bulk copies or cp.async), with no map
  if (!encode_map(&tk, L.k_cache, pages * L.bs, L.d, krow, L.bs,
                  krow == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B) ||
      (!L.f8v4 && !encode_map(&tv, L.v_cache, pages * L.d, L.bs, L.bs, L.d,
                              L.bs == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE)))
    return cudaErrorInvalidValue;

  // keys a single-token row sees at most: the hint, or the window plus the
  // tile that a window start may fall into
  auto hint_tiles = [&](int tile) {
    int tiles = (L.max_seq_len + tile - 1) / tile;
    if (L.window > 0) tiles = std::min(tiles, (L.window + tile - 1) / tile + 1);
    return tiles;
  };
  int seg_tile = kPrefillTile;
  if (use_decode) {
    seg_tile = decode_tile(L.d);
    const int tiles = hint_tiles(seg_tile);
    a.seg_tiles = (tiles + L.num_splits - 1) / L.num_splits;
    if (a.seg_tiles < 1) a.seg_tiles = 1;
    a.block_q = 1;
    a.n_qblocks = 0;
    a.skip_single = 0;
    a.multi_token_ok = use_prefill ? 1 : 0;
  }
  // tcgen05 prefill for multi-token sequences when the decode kernel takes the
  // single-token ones; the mma.sync kernel otherwise (D = 256, Hq/Hk > 8)
  const bool use_tc = use_decode && prefill_tc_supported(L.d);
  auto decode = [&](cudaStream_t s) {
    return L.f8v4 ? launch_decode_f8v4(a, L.d, L.bs, s) : launch_decode(a, tk, tv, L.d, L.bs, s);
  };
  const bool fork = L.side_stream_ok && use_decode && use_prefill && use_tc;
  if (fork) {
    // mixed batch: the prefill kernel on the side stream, forked from and
    // joined back to the caller's stream around the decode kernel
    SideStream *ss = nullptr;
    cudaError_t e = side_stream(&ss);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(ss->mu);  // fork record .. join wait
    if ((e = cudaEventRecord(ss->fork, stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss->s, ss->fork, 0)) != cudaSuccess) return e;
    AttnArgs p = a;
    p.block_q = prefill_tc_rows() / a.qpk;
    p.n_qblocks = L.num_tokens / p.block_q + L.num_seqs;
    p.skip_single = 1;
    if ((e = launch_prefill_tc(p, tk, tv, L.d, L.bs, L.f8v4, ss->s)) != cudaSuccess) return e;
    if ((e = decode(stream)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(ss->join, ss->s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(stream, ss->join, 0)) != cudaSuccess) return e;
  } else if (use_decode) {
    cudaError_t e = decode(stream);
    if (e != cudaSuccess) return e;
  }
  if (use_prefill && use_tc) {
    if (!fork) {
      AttnArgs p = a;
      p.block_q = prefill_tc_rows() / a.qpk;
      p.n_qblocks = L.num_tokens / p.block_q + L.num_seqs;
      p.skip_single = 1;
      cudaError_t e = launch_prefill_tc(p, tk, tv, L.d, L.bs, L.f8v4, stream);
      if (e != cudaSuccess) return e;
    }
  } else if (use_prefill) {
    AttnArgs p = a;
    p.block_q = L.max_query_len <= 1 ? 1 : (64 / a.qpk > 0 ? 64 / a.qpk : 1);
    p.n_qblocks = p.block_q == 1 ? L.num_tokens : L.num_tokens / p.block_q + L.num_seqs;
    p.skip_single = use_decode ? 1 : 0;
    if (!use_decode) {
      const int tiles = hint_tiles(kPrefillTile);
      p.seg_tiles = (tiles + L.num_splits - 1) / L.num_splits;
      if (p.seg_tiles < 1) p.seg_tiles = 1;
      a.seg_tiles = p.seg_tiles;
    }
    cudaError_t e = launch_prefill(p, tk, tv, L.d, L.bs, L.f8v4, stream);
    if (e != cudaSuccess) return e;
  }
  if (L.num_splits <= 1) return cudaSuccess;

  const int64_t warps = static_cast<int64_t>(L.num_seqs) * L.hq;
  const unsigned blocks = static_cast<unsigned>((warps + 3) / 4);
  // programmatic dependent launch: the reduce's blocks are scheduled while
  // the previous kernel drains, and wait for it inside (griddepcontrol.wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
#define PAQ8_REDUCE_CASE(DD)                                                                     \
  case DD: {                                                                                     \
    cudaError_t e = cudaLaunchKernelEx(&cfg, reduce_kernel<DD>,                                  \
                                       static_cast<const float *>(a.part_acc),                   \
                                       static_cast<const float *>(a.part_ml), L.cu, L.seq_lens,  \
                                       L.num_seqs, L.num_tokens, L.hq, L.num_splits, seg_tile,   \
                                       a.seg_tiles, L.window, a.out, L.lse);                     \
    if (e != cudaSuccess) return e;                                                              \
    break;                                                                                       \
  }
  switch (L.d) {
    PAQ8_REDUCE_CASE(64)
    PAQ8_REDUCE_CASE(128)
    PAQ8_REDUCE_CASE(256)
  }
#undef PAQ8_REDUCE_CASE
  return cudaGetLastError();
}

}  // namespace paq8
