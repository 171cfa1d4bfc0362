// bi_roles.cuh -- the parts of the persistent tile pipeline that the GEMM and
// the implicit-im2col convolution share: tile decoding, the UMMA issue loop
// and the TMEM -> registers -> global epilogue.
//
// Fixed-order contract ("Unmasking the True Culprit: Why Temperature=0
// Doesn't Mean Deterministic LLM Inference", section "Why This Achieves Batch
// Invariance": fixed block sizes, one core owns a tile's whole reduction, the
// K tiles always in the same order, no split-K):
//   * every output tile has one fixed shape per kernel (GEMM: 256 x 256 on a
//     CTA pair; convolutions: 128 x 256 on one CTA) and is reduced by
//     exactly one CTA (pair);
//   * its K reduction is K blocks of 64 in ascending order, each issued as
//     four tcgen05.mma steps of K = 16 in ascending order into one fp32 TMEM
//     accumulator, the first step overwriting (accumulator starts from the
//     first product), out-of-range K read as zeros;
//   * the epilogue computes round(acc * alpha + bias) with separately
//     rounded fp32 multiply and add, then one conversion to the output type.
// Which CTA takes which tile (the persistent stride and the raster order)
// changes nothing in that sequence.  `stride` is the number of tile owners
// (CTAs, or CTA pairs): owner c takes tiles c, c + stride, c + 2*stride, ...
//
// PAIR: the GEMM runs on CTA pairs (cta_group::2).  A tile is then 256 x BN:
// each CTA of the pair stages its own 128 rows of A and half of the tile's BN
// columns of B, the even CTA issues 128 x 2 = 256-row MMAs that read both
// CTAs' stages, and each CTA's TMEM receives its own 128 rows x BN columns.
// Per output element this is the same reduction (same K blocks, same K = 16
// steps, same order) as above.  BN: the tile's columns (kBN by default); ACC:
// accumulators in TMEM (the epilogue of one overlaps the main loop of the
// next ACC - 1 tiles).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bi_common.h"
#include "bi_ptx.cuh"

namespace bi {

struct TileCoord {
  int l, mb, nb;
};

// tile -> (batch, m block, n block).  Within a batch, tiles run in groups of
// kGroupM m-blocks so that CTAs working at the same time share A and B panels
// in L2.  Purely a work assignment: it has no effect on any result.
__device__ __forceinline__ TileCoord decode_tile(int tile, int m_tiles, int n_tiles) {
  const int per_batch = m_tiles * n_tiles;
  const int l = tile / per_batch;
  const int t = tile - l * per_batch;
  const int span = kGroupM * n_tiles;
  const int g = t / span;
  const int first_m = g * kGroupM;
  const int gsize = min(m_tiles - first_m, kGroupM);
  const int r = t - g * span;
  return {l, first_m + r % gsize, r / gsize};
}

// Mbarrier addresses of one CTA's pipeline (8 bytes each; tfull / tempty:
// one per accumulator).
struct PipeBars {
  uint32_t full0, empty0, tfull0, tempty0, drain;
  __device__ __forceinline__ uint32_t full(uint32_t s) const { return full0 + 8u * s; }
  __device__ __forceinline__ uint32_t empty(uint32_t s) const { return empty0 + 8u * s; }
  __device__ __forceinline__ uint32_t tfull(uint32_t b) const { return tfull0 + 8u * b; }
  __device__ __forceinline__ uint32_t tempty(uint32_t b) const { return tempty0 + 8u * b; }
};

struct WaitCtl {
  volatile int* abort;
  unsigned int* status_word;
  uint64_t limit_ns;
};

// Single thread: issues every UMMA of this CTA's tiles.  Stage s holds
// A (128 x 64, K-major) at sA + s*A_BYTES and B (BN x 64, with PAIR BN/2 x 64
// per CTA) at sB + s*B_BYTES, B either K-major (rows of 128 bytes) or MN-major
// (64-column chunks of 64 K-rows x 128 bytes, 8 KB apart).
// With PAIR (even CTA only): the same loop with 256-row pair MMAs; stage and
// accumulator barriers are signalled in both CTAs, and the full / free
// barriers waited on here also count the peer's arrivals.
template <int STAGES, int A_BYTES, int B_BYTES, bool B_MN, bool PAIR = false, int BN = kBN,
          int ACC = 2>
__device__ __forceinline__ void mma_role(uint32_t sA, uint32_t sB, const PipeBars& bars,
                                         uint32_t tmem_base, int first_tile, int num_tiles,
                                         int k_blocks, int stride, const WaitCtl& w,
                                         bool in_f16 = false) {
  // A and B are both bf16 or both fp16 (one format for both, as kind::f16
  // requires): fp16 is format code 0 in the A and B fields.
  const uint32_t kIdesc = idesc_bf16_f32(PAIR ? 2 * kBM : kBM, BN, B_MN) &
                          ~(in_f16 ? ((7u << 7) | (7u << 10)) : 0u);
  constexpr uint16_t kBoth = 3;
  uint32_t it = 0;
  int local = 0;
  bool ok = true;
  for (int tile = first_tile; ok && tile < num_tiles; tile += stride, ++local) {
    const uint32_t buf = local % ACC;
    const uint32_t use = local / ACC;
    if (use > 0 &&
        !mbar_wait_bounded<PAIR>(bars.tempty(buf), (use - 1) & 1, w.abort, w.status_word, w.limit_ns,
                                 status_code(6, kSiteMmaTmemEmpty))) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    const uint32_t d = tmem_base + buf * BN;
    for (int kb = 0; kb < k_blocks; ++kb, ++it) {
      const uint32_t s = it % STAGES;
      const uint32_t r = it / STAGES;
      if (!mbar_wait_bounded<PAIR>(bars.full(s), r & 1, w.abort, w.status_word, w.limit_ns,
                                   status_code(6, kSiteMmaFull))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t a = sA + s * A_BYTES;
      const uint32_t b = sB + s * B_BYTES;
#pragma unroll
      for (int k = 0; k < kBK / kUmmaK; ++k) {
        const uint64_t ad = smem_desc_sw128(a + k * 32, 16, 1024);
        const uint64_t bd = B_MN ? smem_desc_sw128(b + k * 2048, 64 * 128, 1024)
                                 : smem_desc_sw128(b + k * 32, 16, 1024);
        if (PAIR)
          umma_bf16_pair(d, ad, bd, kIdesc, (kb | k) != 0 ? 1u : 0u);
        else
          umma_bf16(d, ad, bd, kIdesc, (kb | k) != 0 ? 1u : 0u);
      }
      // stage s may be refilled once these MMAs finish
      if (PAIR)
        umma_commit_pair(bars.empty(s), kBoth);
      else
        umma_commit(bars.empty(s));
    }
    if (!ok) break;
    // accumulator buf is complete
    if (PAIR)
      umma_commit_pair(bars.tfull(buf), kBoth);
    else
      umma_commit(bars.tfull(buf));
  }
  // Every MMA issued above has finished before TMEM can be released.
  if (PAIR)
    umma_commit_pair(bars.drain, 1);
  else
    umma_commit(bars.drain);
  mbar_wait_bounded(bars.drain, 0, nullptr, w.status_word, w.limit_ns,
                    status_code(6, kSiteDrain));
}

// Output addressing shared by the GEMM and the convolutions:
//   out[l][m][n] at c + l*c_batch_stride + m*ldc + n, or with `trans` at
//   c + l*c_batch_stride + n*ldc + m (the patch convolution, whose tile rows
//   are output positions and columns output channels),
//   value = round(acc * alpha (+ bias)), bias either per column n or per
//   row m (the convolution's output channel, offset by (l % bias_groups)*M).
// With tma_c set, each warp whose 32 rows all lie below M stages its 32 x 32
// chunk in shared memory (swizzled, bank-conflict free) and writes it with a
// TMA tile store that clips columns >= N; otherwise threads store directly.
struct OutDesc {
  void* c;
  const void* bias;
  const CUtensorMap* tma_c;  // tensor map of c as [L][M][N] with 32 x 32 boxes, or null
  int64_t ldc, c_batch_stride, bias_stride;
  float alpha;
  int32_t M, N;
  int32_t out_f32, bias_kind, vec_store;  // bias_kind: 0 none, 1 bf16, 2 fp32, 3 fp16
  int32_t out_f16;                        // 16-bit output as fp16 instead of bf16
  int32_t bias_per_row, bias_groups;
  int32_t trans;
  // Tile row r of m block mb is output row mb*tile_rows + r, and only rows
  // r < tile_rows are outputs (kBM except for the patch convolution).
  int32_t tile_rows;
};

// Epilogue staging: per epilogue warp, two 4 KB buffers (double-buffered
// against the TMA stores in flight), 1 KB aligned.
constexpr int kStageOutBytes = 4096;
constexpr int kEpilogueStagingBytes = 4 * 2 * kStageOutBytes;

__device__ __forceinline__ float load_bias(const OutDesc& o, int64_t idx) {
  if (o.bias_kind == 1) {
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(o.bias);
    return __bfloat162float(b[idx * o.bias_stride]);
  }
  if (o.bias_kind == 3) {
    const __half* b = reinterpret_cast<const __half*>(o.bias);
    return __half2float(b[idx * o.bias_stride]);
  }
  return reinterpret_cast<const float*>(o.bias)[idx * o.bias_stride];
}

// Bias values a warp needs for one tile, loaded before the accumulator is
// ready so their latency hides behind the tile's main loop: per row, this
// thread's row; per column, lane t holds the bias of column t of each
// 32-column chunk j (broadcast to the warp with shuffles when used).
template <int BN>
struct TileBias {
  float row;
  float col[BN / 32];
};

template <int BN>
__device__ __forceinline__ void load_tile_bias(const OutDesc& o, int l, int m, int n_base, int lane,
                                               TileBias<BN>& tb) {
  if (!o.bias_kind) return;
  if (o.bias_per_row) {
    tb.row = (m < o.M) ? load_bias(o, (int64_t)(l % o.bias_groups) * o.M + m) : 0.0f;
  } else {
#pragma unroll
    for (int j = 0; j < BN / 32; ++j) {
      const int n = n_base + j * 32 + lane;
      tb.col[j] = (n < o.N) ? load_bias(o, n) : 0.0f;
    }
  }
}

// f = acc * alpha (+ bias), each a separately rounded fp32 operation.
template <int BN>
__device__ __forceinline__ void epilogue_math(const OutDesc& o, int j, const TileBias<BN>& tb,
                                              const uint32_t (&v)[32], float (&f)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __fmul_rn(__uint_as_float(v[i]), o.alpha);
  if (o.bias_kind) {
    if (o.bias_per_row) {
#pragma unroll
      for (int i = 0; i < 32; ++i) f[i] = __fadd_rn(f[i], tb.row);
    } else {
      float bj = 0.0f;
#pragma unroll
      for (int jj = 0; jj < BN / 32; ++jj)
        if (jj == j) bj = tb.col[jj];
#pragma unroll
      for (int i = 0; i < 32; ++i) f[i] = __fadd_rn(f[i], __shfl_sync(0xffffffffu, bj, i));
    }
  }
}

// One rounding (RNE) of fp32 values to the 16-bit output type.
__device__ __forceinline__ uint16_t cvt_out1(const OutDesc& o, float v) {
  if (o.out_f16) {
    const __half h = __float2half_rn(v);
    return *reinterpret_cast<const uint16_t*>(&h);
  }
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_out2(const OutDesc& o, float lo, float hi) {
  if (o.out_f16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Thread owns output row m and 32 consecutive columns starting at n0 (row_ok:
// the thread's tile row is an output row).
__device__ __forceinline__ void store_32_direct(const OutDesc& o, int l, int m, int n0, bool row_ok,
                                                const float (&f)[32]) {
  if (!row_ok || m >= o.M || n0 >= o.N) return;
  if (o.trans) {
    // Column n of the tile is output row n: a warp's 32 threads (consecutive
    // m) write 32 consecutive elements of it per column.
    const int64_t base = (int64_t)l * o.c_batch_stride + m;
    if (o.out_f32) {
      float* dst = reinterpret_cast<float*>(o.c) + base;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < o.N) dst[(int64_t)(n0 + i) * o.ldc] = f[i];
    } else {
      uint16_t* dst = reinterpret_cast<uint16_t*>(o.c) + base;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < o.N) dst[(int64_t)(n0 + i) * o.ldc] = cvt_out1(o, f[i]);
    }
    return;
  }
  const int64_t off = (int64_t)l * o.c_batch_stride + (int64_t)m * o.ldc + n0;
  const bool full = o.vec_store && (n0 + 32 <= o.N);
  if (o.out_f32) {
    float* dst = reinterpret_cast<float*>(o.c) + off;
    if (full) {
      float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
      for (int i = 0; i < 8; ++i) d4[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < o.N) dst[i] = f[i];
    }
  } else {
    uint16_t* dst = reinterpret_cast<uint16_t*>(o.c) + off;
    if (full) {
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        d4[i] = make_uint4(pack_out2(o, f[8 * i], f[8 * i + 1]), pack_out2(o, f[8 * i + 2], f[8 * i + 3]),
                           pack_out2(o, f[8 * i + 4], f[8 * i + 5]), pack_out2(o, f[8 * i + 6], f[8 * i + 7]));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < o.N) dst[i] = cvt_out1(o, f[i]);
    }
  }
}

// Lane `lane` writes its row of the warp's 32 x 32 chunk into the staging
// buffer in the layout of the store's tensor map: fp32 rows of 128 bytes with
// the 128-byte swizzle, bf16 rows of 64 bytes with the 64-byte swizzle.
__device__ __forceinline__ void stage_32(const OutDesc& o, uint32_t sbuf, int lane,
                                         const float (&f)[32]) {
  if (o.out_f32) {
#pragma unroll
    for (int cc = 0; cc < 8; ++cc)
      st_shared_v4(sbuf + lane * 128 + ((cc ^ (lane & 7)) << 4), __float_as_uint(f[4 * cc]),
                   __float_as_uint(f[4 * cc + 1]), __float_as_uint(f[4 * cc + 2]),
                   __float_as_uint(f[4 * cc + 3]));
  } else {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
      st_shared_v4(sbuf + lane * 64 + ((cc ^ ((lane >> 1) & 3)) << 4),
                   pack_out2(o, f[8 * cc], f[8 * cc + 1]), pack_out2(o, f[8 * cc + 2], f[8 * cc + 3]),
                   pack_out2(o, f[8 * cc + 4], f[8 * cc + 5]), pack_out2(o, f[8 * cc + 6], f[8 * cc + 7]));
  }
}

// Converts and stores chunk j (32 columns) of this warp's 32 rows.
template <int BN>
__device__ __forceinline__ void epilogue_chunk(const OutDesc& o, int j, const TileBias<BN>& tb,
                                               const uint32_t (&v)[32], const TileCoord& tc, int m0,
                                               int lane, bool row_ok, uint32_t stage_base,
                                               uint32_t& chunk) {
  const int n0 = tc.nb * BN + j * 32;
  float f[32];
  epilogue_math<BN>(o, j, tb, v, f);
  // A quadrant with rows past M (a decode-sized M, or the last rows of a
  // problem) stores directly: its few rows do not pay for staging and for
  // waiting on the staging buffers.  Same values either way.
  if (o.tma_c && m0 + 32 <= o.M) {
    const uint32_t sbuf = stage_base + (chunk & 1) * kStageOutBytes;
    if (chunk >= 2) {  // the store issued two chunks ago must have read this buffer
      if (lane == 0) bulk_wait_read_1();
      __syncwarp();
    }
    stage_32(o, sbuf, lane, f);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(o.tma_c, sbuf, n0, m0, tc.l);
      bulk_commit();
    }
    ++chunk;
  } else {
    store_32_direct(o, tc.l, m0 + lane, n0, row_ok, f);
  }
}

// One warp of the epilogue group: drains TMEM lane quadrant q (rows
// 32q .. 32q+31 of each tile) for every tile of this CTA.  stage_base: this
// warp's two staging buffers (used when o.tma_c is set).
// With PAIR, m_tiles counts 256-row tiles and this CTA (rank `crank` of the
// pair) drains rows crank*128 .. crank*128+127 of each; the accumulator is
// released to the even CTA, whose MMA issuer waits for both CTAs.
template <bool PAIR = false, int BN = kBN, int ACC = 2>
__device__ __forceinline__ void epilogue_role(int q, int lane, uint32_t tmem_base,
                                              const PipeBars& bars, int first_tile, int num_tiles,
                                              int m_tiles, int n_tiles, int stride, const OutDesc& o,
                                              uint32_t stage_base, const WaitCtl& w,
                                              uint32_t crank = 0) {
  int local = 0;
  uint32_t chunk = 0;  // staged chunks issued by this warp (selects the buffer)
  for (int tile = first_tile; tile < num_tiles; tile += stride, ++local) {
    const uint32_t buf = local % ACC;
    const uint32_t use = local / ACC;
    TileCoord tc = decode_tile(tile, m_tiles, n_tiles);
    if (PAIR) tc.mb = 2 * tc.mb + (int)crank;
    const int r0 = q * 32;
    const int m0 = tc.mb * o.tile_rows + r0;
    const bool row_ok = r0 + lane < o.tile_rows;
    TileBias<BN> tb;
    load_tile_bias<BN>(o, tc.l, m0 + lane, tc.nb * BN, lane, tb);
    const bool ok = mbar_wait_bounded(bars.tfull(buf), use & 1, w.abort, w.status_word,
                                      w.limit_ns, status_code(6, kSiteEpilogueTmemFull));
    if (!__all_sync(0xffffffffu, ok)) break;
    tc_fence_after_sync();
    const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN;
    // Chunks holding any output: none when all 32 rows of this quadrant are
    // past M, and none past N.
    const int n_left = o.N - tc.nb * BN;
    const int n_chunks = (r0 < o.tile_rows && m0 < o.M) ? min(BN / 32, (n_left + 31) / 32) : 0;
    // Two register sets: the next chunk's TMEM load is in flight while the
    // current chunk is converted and stored.
    uint32_t va[32], vb[32];
    if (n_chunks > 0) tmem_load_32cols(lane_addr, va);
#pragma unroll 1
    for (int j = 0; j < n_chunks; j += 2) {
      tmem_load_wait(va);
      if (j + 1 < n_chunks) tmem_load_32cols(lane_addr + (j + 1) * 32, vb);
      epilogue_chunk<BN>(o, j, tb, va, tc, m0, lane, row_ok, stage_base, chunk);
      if (j + 1 < n_chunks) {
        tmem_load_wait(vb);
        if (j + 2 < n_chunks) tmem_load_32cols(lane_addr + (j + 2) * 32, va);
        epilogue_chunk<BN>(o, j + 1, tb, vb, tc, m0, lane, row_ok, stage_base, chunk);
      }
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) {
      if (PAIR && crank != 0)
        mbar_arrive_remote(bars.tempty(buf), 0);
      else
        mbar_arrive(bars.tempty(buf));
    }
  }
  // Shared memory must outlive the reads of the stores still in flight (the
  // writes themselves complete before the kernel does).
  if (o.tma_c && lane == 0) bulk_wait_read_all();
  __syncwarp();
}

}  // namespace bi
