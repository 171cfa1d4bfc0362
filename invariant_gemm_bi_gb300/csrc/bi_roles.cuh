// bi_roles.cuh -- the parts of the persistent tile pipeline that the GEMM and
// the implicit-im2col convolution share: tile decoding, the UMMA issue loop
// and the TMEM -> registers -> global epilogue.
//
// Fixed-order contract ("Unmasking the True Culprit: Why Temperature=0
// Doesn't Mean Deterministic LLM Inference", section "Why This Achieves Batch
// Invariance": fixed block sizes, one core owns a tile's whole reduction, the
// K tiles always in the same order, no split-K):
//   * every output tile is 128 x kBN and is reduced by exactly one CTA;
//   * its K reduction is K blocks of 64 in ascending order, each issued as
//     four tcgen05.mma steps of K = 16 in ascending order into one fp32 TMEM
//     accumulator, the first step overwriting (accumulator starts from the
//     first product), out-of-range K read as zeros;
//   * the epilogue computes round(acc * alpha + bias) with separately
//     rounded fp32 multiply and add, then one conversion to the output type.
// Which CTA takes which tile (the persistent stride and the raster order)
// changes nothing in that sequence.
#pragma once

#include <cuda_bf16.h>

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

// Mbarrier addresses of one CTA's pipeline (8 bytes each).
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
// A (128 x 64, K-major) at sA + s*A_BYTES and B (kBN x 64) at sB + s*B_BYTES,
// B either K-major (kBN rows of 128 bytes) or MN-major (kBN/64 chunks of
// 64 K-rows x 128 bytes, 8 KB apart).
template <int STAGES, int A_BYTES, int B_BYTES, bool B_MN>
__device__ __forceinline__ void mma_role(uint32_t sA, uint32_t sB, const PipeBars& bars,
                                         uint32_t tmem_base, int num_tiles, int k_blocks,
                                         const WaitCtl& w) {
  constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, B_MN);
  uint32_t it = 0;
  int local = 0;
  bool ok = true;
  for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
    const uint32_t buf = local & 1;
    const uint32_t use = local >> 1;
    if (use > 0 &&
        !mbar_wait_bounded(bars.tempty(buf), (use - 1) & 1, w.abort, w.status_word, w.limit_ns,
                           status_code(6, kSiteMmaTmemEmpty))) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    const uint32_t d = tmem_base + buf * kBN;
    for (int kb = 0; kb < k_blocks; ++kb, ++it) {
      const uint32_t s = it % STAGES;
      const uint32_t r = it / STAGES;
      if (!mbar_wait_bounded(bars.full(s), r & 1, w.abort, w.status_word, w.limit_ns,
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
        umma_bf16(d, ad, bd, kIdesc, (kb | k) != 0 ? 1u : 0u);
      }
      umma_commit(bars.empty(s));  // stage s may be refilled once these MMAs finish
    }
    if (!ok) break;
    umma_commit(bars.tfull(buf));  // accumulator buf is complete
  }
  // Every MMA issued above has finished before TMEM can be released.
  umma_commit(bars.drain);
  mbar_wait_bounded(bars.drain, 0, nullptr, w.status_word, w.limit_ns,
                    status_code(6, kSiteDrain));
}

// Output addressing shared by the GEMM and the convolution:
//   out[l][m][n] at c + l*c_batch_stride + m*ldc + n,
//   value = round(acc * alpha (+ bias)), bias either per column n or per
//   row m (the convolution's output channel, offset by (l % bias_groups)*M).
struct OutDesc {
  void* c;
  const void* bias;
  int64_t ldc, c_batch_stride, bias_stride;
  float alpha;
  int32_t M, N;
  int32_t out_f32, bias_kind, vec_store;
  int32_t bias_per_row, bias_groups;
};

__device__ __forceinline__ float load_bias(const OutDesc& o, int64_t idx) {
  if (o.bias_kind == 1) {
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(o.bias);
    return __bfloat162float(b[idx * o.bias_stride]);
  }
  return reinterpret_cast<const float*>(o.bias)[idx * o.bias_stride];
}

// Thread owns output row m and 32 consecutive columns starting at n0.
__device__ __forceinline__ void store_32(const OutDesc& o, int l, int m, int n0,
                                         const uint32_t (&v)[32]) {
  if (m >= o.M || n0 >= o.N) return;
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __fmul_rn(__uint_as_float(v[i]), o.alpha);
  if (o.bias_kind) {
    if (o.bias_per_row) {
      const float bv = load_bias(o, (int64_t)(l % o.bias_groups) * o.M + m);
#pragma unroll
      for (int i = 0; i < 32; ++i) f[i] = __fadd_rn(f[i], bv);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < o.N) f[i] = __fadd_rn(f[i], load_bias(o, n0 + i));
    }
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
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(o.c) + off;
    if (full) {
      uint32_t packed[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        packed[i] = *reinterpret_cast<uint32_t*>(&h);
      }
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < o.N) dst[i] = __float2bfloat16_rn(f[i]);
    }
  }
}

// One warp of the epilogue group: drains TMEM lane quadrant q (rows
// 32q .. 32q+31 of each tile) for every tile of this CTA.
__device__ __forceinline__ void epilogue_role(int q, int lane, uint32_t tmem_base,
                                              const PipeBars& bars, int num_tiles, int m_tiles,
                                              int n_tiles, const OutDesc& o, const WaitCtl& w) {
  int local = 0;
  for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
    const uint32_t buf = local & 1;
    const uint32_t use = local >> 1;
    const bool ok = mbar_wait_bounded(bars.tfull(buf), use & 1, w.abort, w.status_word,
                                      w.limit_ns, status_code(6, kSiteEpilogueTmemFull));
    if (!__all_sync(0xffffffffu, ok)) break;
    tc_fence_after_sync();
    const TileCoord tc = decode_tile(tile, m_tiles, n_tiles);
    const int m = tc.mb * kBM + q * 32 + lane;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * kBN;
#pragma unroll 1
    for (int j = 0; j < kBN / 32; ++j) {
      uint32_t v[32];
      tmem_load_32cols(lane_addr + j * 32, v);
      tmem_load_wait();
      store_32(o, tc.l, m, tc.nb * kBN + j * 32, v);
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.tempty(buf));
  }
}

}  // namespace bi
