// bi_conv.cu -- 2-D convolution as a per-sample implicit-im2col tcgen05 GEMM.
//
// For sample b and group g the convolution is the product
//   Y[b, g] (Cog x P) = W_g (Cog x Kg) . Patches[b, g]^T (Kg x P)  + bias
// with P = Ho*Wo output positions and Kg = Cig*KH*KW, the reduction index
// k = (ci*KH + kh)*KW + kw -- the unfold order of "Batch-Invariant VLAs",
// section "Replacing nn.Conv2d", and "Batch-Invariant Kernel Design: Conv2d
// and Attention BMM", section "Kernel 1: Conv2d" (stride, padding, dilation,
// groups).  No unfolded matrix is materialised: producer warps gather the
// weight rows and the patch elements for one K block straight into the
// 128-byte-swizzled K-major shared-memory layout the tensor core reads, then
// the same UMMA issue loop and epilogue as the GEMM run.  (sample, group) is
// the batch coordinate of the tile space, so a tile never mixes samples and
// one sample's arithmetic is the same for every batch size.
#include <cuda.h>
#include <cuda_runtime.h>

#include "bi_common.h"
#include "bi_launch.h"
#include "bi_ptx.cuh"
#include "bi_roles.cuh"

namespace bi {

struct ConvLayout {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = kBN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int MAX_DYN = 232448;
  static constexpr int FIT = (MAX_DYN - 1024 - BAR_BYTES - kEpilogueStagingBytes) / STAGE_BYTES;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr int DYN_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES + kEpilogueStagingBytes;
  static constexpr uint32_t TMEM_COLS = 2 * kBN;
  static_assert(DYN_BYTES > 116 * 1024, "one CTA per SM: TMEM is allocated whole");
};

constexpr int kConvProducerThreads = 128;
constexpr int kConvThreads = 288;  // 4 producer warps, 1 MMA warp, 4 epilogue warps

// Byte offset of element (row, k) of a 128-byte-swizzled K-major tile whose
// rows hold 64 bf16 of K: 16-byte chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
// Byte offset of bf16 element (row, c) in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_elem(int row, int c) {
  return (uint32_t)(row * 128 + ((((c >> 3) ^ (row & 7)) << 4) | ((c & 7) << 1)));
}

// A operand (weights of group g, rows = output channels, K contiguous):
// general gather, 8 elements per 16-byte chunk.
__device__ __forceinline__ void fill_a_general(const ConvParams& p, uint32_t a_dst, const uint16_t* wrow0,
                                               int mb, int kb, int tid) {
#pragma unroll 1
  for (int q = tid; q < kBM * 8; q += kConvProducerThreads) {
    const int row = q >> 3, ch = q & 7;
    const int m = mb * kBM + row;
    const int k0 = kb * kBK + ch * 8;
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    if (m < p.Cog) {
      const uint16_t* src = wrow0 + (int64_t)m * p.Kg;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int k = k0 + e;
        const uint32_t h = (k < p.Kg) ? (uint32_t)__ldg(src + k) : 0u;
        v[e >> 1] |= h << ((e & 1) * 16);
      }
    }
    st_shared_v4(a_dst + sw128_offset(row, ch), v[0], v[1], v[2], v[3]);
  }
}

// Same result when rows are 8-byte aligned (Kg % 4 == 0): one 8-byte load per
// 4 elements, 16 consecutive threads per weight row; all 16 loads of a thread
// are issued before any store so their latencies overlap.
__device__ __forceinline__ void fill_a_vec8(const ConvParams& p, uint32_t a_dst, const uint16_t* wrow0,
                                            int mb, int kb, int tid) {
  constexpr int kPer = kBM * 16 / kConvProducerThreads;
  uint2 v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int q = tid + i * kConvProducerThreads;
    const int row = q >> 4, pc = q & 15;
    const int m = mb * kBM + row;
    const int k0 = kb * kBK + pc * 4;
    v[i] = make_uint2(0u, 0u);
    if (m < p.Cog) {
      const uint16_t* src = wrow0 + (int64_t)m * p.Kg + k0;
      if (k0 + 4 <= p.Kg) {
        v[i] = __ldg(reinterpret_cast<const uint2*>(src));
      } else {
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = (k0 + e < p.Kg) ? (uint32_t)__ldg(src + e) : 0u;
        v[i] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int q = tid + i * kConvProducerThreads;
    const int row = q >> 4, pc = q & 15;
    st_shared_v2(a_dst + (uint32_t)(row * 128 + ((((pc >> 1) ^ (row & 7)) << 4) | ((pc & 1) << 3))),
                 v[i].x, v[i].y);
  }
}

// B operand (patches of sample b, rows = output positions, K contiguous):
// general gather for any stride / padding / dilation.
__device__ __forceinline__ void fill_b_general(const ConvParams& p, uint32_t b_dst, const uint16_t* ximg,
                                               int nb, int kb, int tid) {
  const int KHW = p.KH * p.KW;
#pragma unroll 1
  for (int q = tid; q < kBN * 8; q += kConvProducerThreads) {
    const int row = q >> 3, ch = q & 7;
    const int pos = nb * kBN + row;
    const int k0 = kb * kBK + ch * 8;
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    if (pos < p.P) {
      const int oh = pos / p.Wo;
      const int ow = pos - oh * p.Wo;
      const int ih0 = oh * p.sh - p.ph;
      const int iw0 = ow * p.sw - p.pw;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int k = k0 + e;
        uint32_t h = 0u;
        if (k < p.Kg) {
          const int ci = k / KHW;
          const int rr = k - ci * KHW;
          const int kh = rr / p.KW;
          const int kw = rr - kh * p.KW;
          const int ih = ih0 + kh * p.dh;
          const int iw = iw0 + kw * p.dw;
          if (ih >= 0 && ih < p.H && iw >= 0 && iw < p.W)
            h = (uint32_t)__ldg(ximg + ((int64_t)ci * p.H + ih) * p.W + iw);
        }
        v[e >> 1] |= h << ((e & 1) * 16);
      }
    }
    st_shared_v4(b_dst + sw128_offset(row, ch), v[0], v[1], v[2], v[3]);
  }
}

// B operand for non-overlapping patches (stride = kernel size, no padding,
// unit dilation): each image row (ci, ih) holds, side by side, the kw runs of
// every patch of one output row oh.  A warp reads whole image rows with
// coalesced (16-byte when aligned) loads and scatters each element to its
// (patch, k) place in the swizzled tile: the same bytes fill_b_general writes.
__device__ __forceinline__ void fill_b_patch(const ConvParams& p, uint32_t b_dst, const uint16_t* ximg,
                                             int nb, int kb, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const int k_lo = kb * kBK, k_hi = min(k_lo + kBK, p.Kg);
  const int p_lo = nb * kBN, p_hi = min(p_lo + kBN, p.P);
  const int ck_lo = k_lo / p.KW, ck_hi = (k_hi - 1) / p.KW;  // kernel rows (ci*KH + kh)
  const int oh_lo = p_lo / p.Wo, oh_hi = (p_hi - 1) / p.Wo;
  const int n_oh = oh_hi - oh_lo + 1;
  const int items = (ck_hi - ck_lo + 1) * n_oh;
  const int width = p.Wo * p.KW;  // image columns that belong to a patch
  // Zero what no image element lands on: k >= Kg columns, rows past P.
  const int valid_rows = p_hi - p_lo, valid_cols = k_hi - k_lo;
  if (valid_rows < kBN || valid_cols < kBK) {
    for (int q = tid; q < kBN * 8; q += kConvProducerThreads) {
      const int row = q >> 3, ch = q & 7;
      if (row >= valid_rows || ch * 8 >= valid_cols) {
        st_shared_v4(b_dst + sw128_offset(row, ch), 0u, 0u, 0u, 0u);
      } else if (ch * 8 + 8 > valid_cols) {
        for (int c = valid_cols; c < ch * 8 + 8; ++c) st_shared_u16(b_dst + sw128_elem(row, c), 0);
      }
    }
  }
  // Rows are taken kBatch at a time per warp: all loads of a batch are issued
  // before any element is scattered, so their latencies overlap.
  constexpr int kBatch = 8;
  constexpr int kWarps = kConvProducerThreads / 32;
  if (p.x_vec16 && (p.KW & 1) == 0 && width <= 256) {
    // Pair path: a lane's 8 elements are 4 (kw, kw+1) pairs at fixed patch
    // columns for every image row (KW even: a pair never straddles a patch and
    // starts at an even k, so it is one aligned 32-bit shared-memory word).
    const int e0 = lane * 8;
    int ow_i[4], kw_i[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = e0 + 2 * i;
      ow_i[i] = e / p.KW;
      kw_i[i] = e - ow_i[i] * p.KW;
    }
    if (e0 >= width) return;
    for (int base = warp; base < items; base += kWarps * kBatch) {
      uint4 raw[kBatch];
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const int it = base + r * kWarps;
        raw[r] = make_uint4(0u, 0u, 0u, 0u);
        if (it < items) {
          const int ck = ck_lo + it / n_oh;
          const int oh = oh_lo + it - (it / n_oh) * n_oh;
          const int ci = ck / p.KH, kh = ck - ci * p.KH;
          raw[r] = __ldg(reinterpret_cast<const uint4*>(
              ximg + ((int64_t)ci * p.H + (int64_t)oh * p.KH + kh) * p.W + e0));
        }
      }
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const int it = base + r * kWarps;
        if (it >= items) break;
        const int ck = ck_lo + it / n_oh;
        const int oh = oh_lo + it - (it / n_oh) * n_oh;
        const int c0 = ck * p.KW - k_lo;      // column of kw = 0 in this k block
        const int row0 = oh * p.Wo - p_lo;    // tile row of ow = 0
        const uint32_t w4[4] = {raw[r].x, raw[r].y, raw[r].z, raw[r].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = c0 + kw_i[i];
          const int row = row0 + ow_i[i];
          // ow_i < Wo: columns past the last whole patch belong to no patch
          if (ow_i[i] < p.Wo && c >= 0 && c < valid_cols && row >= 0 && row < valid_rows)
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(b_dst + sw128_elem(row, c)), "r"(w4[i])
                         : "memory");
        }
      }
    }
    return;
  }
  for (int base = warp; base < items; base += kWarps * kBatch) {
    for (int e0 = lane * 8; e0 < width; e0 += 256) {
      uint4 raw[kBatch];
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const int it = base + r * kWarps;
        raw[r] = make_uint4(0u, 0u, 0u, 0u);
        if (it < items) {
          const int ck = ck_lo + it / n_oh;
          const int oh = oh_lo + it - (it / n_oh) * n_oh;
          const int ci = ck / p.KH, kh = ck - ci * p.KH;
          const uint16_t* row_ptr = ximg + ((int64_t)ci * p.H + (int64_t)oh * p.KH + kh) * p.W;
          if (p.x_vec16) {
            raw[r] = __ldg(reinterpret_cast<const uint4*>(row_ptr + e0));
          } else {
            uint32_t h[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) h[j] = (e0 + j < width) ? (uint32_t)__ldg(row_ptr + e0 + j) : 0u;
            raw[r] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                                h[6] | (h[7] << 16));
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const int it = base + r * kWarps;
        if (it >= items) break;
        const int ck = ck_lo + it / n_oh;
        const int oh = oh_lo + it - (it / n_oh) * n_oh;
        const uint32_t w4[4] = {raw[r].x, raw[r].y, raw[r].z, raw[r].w};
        int ow = e0 / p.KW;
        int kw = e0 - ow * p.KW;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int k = ck * p.KW + kw;
          const int pp = oh * p.Wo + ow;
          if (e0 + j < width && k >= k_lo && k < k_hi && pp >= p_lo && pp < p_hi)
            st_shared_u16(b_dst + sw128_elem(pp - p_lo, k - k_lo),
                          (uint16_t)(w4[j >> 1] >> ((j & 1) * 16)));
          if (++kw == p.KW) {
            kw = 0;
            ++ow;
          }
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kConvThreads, 1) conv_kernel(const __grid_constant__ ConvParams p) {
  using Lay = ConvLayout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + Lay::STAGES * Lay::A_BYTES;
  const uint32_t bar0 = sB + Lay::STAGES * Lay::B_BYTES;
  PipeBars bars;
  bars.full0 = bar0;
  bars.empty0 = bar0 + 8 * Lay::STAGES;
  bars.tfull0 = bars.empty0 + 8 * Lay::STAGES;
  bars.tempty0 = bars.tfull0 + 16;
  bars.drain = bars.tempty0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + (bars.drain + 8 - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Lay::STAGES; ++s) {
      mbar_init(bars.full(s), kConvProducerThreads);
      mbar_init(bars.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.tfull(b), 1);
      mbar_init(bars.tempty(b), 4);
    }
    mbar_init(bars.drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), Lay::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status_word, p.wait_limit_ns};

  if (warp < 4) {
    // ---- producers: gather W rows and patch elements for each K block ----
    const int tid = threadIdx.x;
    const uint16_t* __restrict__ xg = p.x;
    const uint16_t* __restrict__ wg = p.w;
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const TileCoord tc = decode_tile(tile, p.m_tiles, p.n_tiles);
      const int b = tc.l / p.groups;
      const int g = tc.l - b * p.groups;
      const uint16_t* wrow0 = wg + (int64_t)g * p.Cog * p.Kg;
      const uint16_t* ximg = xg + ((int64_t)b * p.C + (int64_t)g * p.Cig) * p.H * p.W;
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        const uint32_t s = it % Lay::STAGES;
        const uint32_t r = it / Lay::STAGES;
        if (r > 0 && !mbar_wait_bounded(bars.empty(s), (r - 1) & 1, wc.abort, wc.status_word,
                                        wc.limit_ns, status_code(6, kSiteConvProducer))) {
          ok = false;
          break;
        }
        const uint32_t a_dst = sA + s * Lay::A_BYTES;
        const uint32_t b_dst = sB + s * Lay::B_BYTES;
        if (p.w_vec8)
          fill_a_vec8(p, a_dst, wrow0, tc.mb, kb, tid);
        else
          fill_a_general(p, a_dst, wrow0, tc.mb, kb, tid);
        if (p.patch_fast)
          fill_b_patch(p, b_dst, ximg, tc.nb, kb, tid);
        else
          fill_b_general(p, b_dst, ximg, tc.nb, kb, tid);
        fence_proxy_async_smem();
        mbar_arrive(bars.full(s));
        ++it;
      }
    }
  } else if (warp == 4) {
    if (lane == 0)
      mma_role<Lay::STAGES, Lay::A_BYTES, Lay::B_BYTES, false>(
          sA, sB, bars, tmem_base, blockIdx.x, p.num_tiles, p.k_blocks, gridDim.x, wc);
  } else {
    OutDesc o;
    o.c = p.y;
    o.bias = p.bias;
    o.ldc = p.P;
    o.c_batch_stride = (int64_t)p.Cog * p.P;
    o.bias_stride = 1;
    o.alpha = 1.0f;
    o.M = p.Cog;
    o.N = p.P;
    o.out_f32 = p.out_f32;
    o.bias_kind = p.bias_kind;
    o.vec_store = p.vec_store;
    o.bias_per_row = 1;
    o.bias_groups = p.groups;
    o.trans = 0;
    o.tile_rows = kBM;
    o.out_f16 = 0;
    o.tma_c = p.use_tma_store ? &p.tma_y : nullptr;
    const uint32_t staging = bar0 + Lay::BAR_BYTES + (warp - 5) * 2 * kStageOutBytes;
    epilogue_role(warp & 3, lane, tmem_base, bars, blockIdx.x, p.num_tiles, p.m_tiles, p.n_tiles,
                  gridDim.x, o, staging, wc);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Lay::TMEM_COLS);
  }
}

bi_status launch_conv(const ConvProblem& cp, cudaStream_t stream, std::string* why) {
  DeviceInfo dev;
  bi_status st = current_device_info(&dev, why);
  if (st != BI_OK) return st;
  ConvParams p;
  memset(&p, 0, sizeof(p));
  p.x = reinterpret_cast<const uint16_t*>(cp.x);
  p.w = reinterpret_cast<const uint16_t*>(cp.w);
  p.bias = cp.bias;
  p.y = cp.y;
  p.B = (int32_t)cp.B;
  p.C = (int32_t)cp.C;
  p.H = (int32_t)cp.H;
  p.W = (int32_t)cp.W;
  p.Co = (int32_t)cp.Co;
  p.KH = (int32_t)cp.KH;
  p.KW = (int32_t)cp.KW;
  p.Ho = (int32_t)cp.Ho;
  p.Wo = (int32_t)cp.Wo;
  p.sh = cp.sh;
  p.sw = cp.sw;
  p.ph = cp.ph;
  p.pw = cp.pw;
  p.dh = cp.dh;
  p.dw = cp.dw;
  p.groups = cp.groups;
  p.Cig = (int32_t)(cp.C / cp.groups);
  p.Cog = (int32_t)(cp.Co / cp.groups);
  p.Kg = p.Cig * p.KH * p.KW;
  p.P = p.Ho * p.Wo;
  p.m_tiles = (p.Cog + kBM - 1) / kBM;
  p.n_tiles = (p.P + kBN - 1) / kBN;
  p.k_blocks = (p.Kg + kBK - 1) / kBK;
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles * cp.B * cp.groups;
  if (tiles > INT32_MAX) {
    *why = "tile count exceeds 2^31";
    return BI_ERR_INVALID_ARG;
  }
  p.num_tiles = (int32_t)tiles;
  p.out_f32 = cp.out_f32;
  p.bias_kind = cp.bias_kind;
  const int esz = cp.out_f32 ? 4 : 2;
  p.vec_store = ((reinterpret_cast<uintptr_t>(cp.y) % 16) == 0 && ((int64_t)p.P * esz) % 16 == 0) ? 1 : 0;
  p.patch_fast = (cp.sh == cp.KH && cp.sw == cp.KW && cp.ph == 0 && cp.pw == 0 && cp.dh == 1 &&
                  cp.dw == 1)
                     ? 1
                     : 0;
  p.x_vec16 = ((reinterpret_cast<uintptr_t>(cp.x) % 16) == 0 && cp.W % 8 == 0) ? 1 : 0;
  p.w_vec8 = ((reinterpret_cast<uintptr_t>(cp.w) % 8) == 0 && p.Kg % 4 == 0) ? 1 : 0;
  p.use_tma_store = encode_output_map(&p.tma_y, cp.y, cp.out_f32 != 0, false, cp.B * cp.groups, p.Cog, p.P,
                                      p.P, (int64_t)p.Cog * p.P)
                        ? 1
                        : 0;
  p.status_word = dev.status_word;
  p.wait_limit_ns = kWaitLimitNs;
  const int grid = (int)std::min<int64_t>(tiles, dev.num_sms);
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&conv_kernel), ConvLayout::DYN_BYTES, 4);
  if (e == cudaSuccess) conv_kernel<<<grid, kConvThreads, ConvLayout::DYN_BYTES, stream>>>(p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("conv launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

}  // namespace bi
