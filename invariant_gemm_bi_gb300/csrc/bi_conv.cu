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
    const int KHW = p.KH * p.KW;
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
        // A: 128 rows (output channels of the group) x 8 chunks of 8 k.
#pragma unroll 1
        for (int q = tid; q < kBM * 8; q += kConvProducerThreads) {
          const int row = q >> 3, ch = q & 7;
          const int m = tc.mb * kBM + row;
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
        // B: kBN rows (output positions) x 8 chunks of 8 k.
#pragma unroll 1
        for (int q = tid; q < kBN * 8; q += kConvProducerThreads) {
          const int row = q >> 3, ch = q & 7;
          const int pos = tc.nb * kBN + row;
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
        fence_proxy_async_smem();
        mbar_arrive(bars.full(s));
        ++it;
      }
    }
  } else if (warp == 4) {
    if (lane == 0)
      mma_role<Lay::STAGES, Lay::A_BYTES, Lay::B_BYTES, false>(sA, sB, bars, tmem_base,
                                                               p.num_tiles, p.k_blocks, gridDim.x, wc);
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
    o.tma_c = p.use_tma_store ? &p.tma_y : nullptr;
    const uint32_t staging = bar0 + Lay::BAR_BYTES + (warp - 5) * 2 * kStageOutBytes;
    epilogue_role(warp & 3, lane, tmem_base, bars, p.num_tiles, p.m_tiles, p.n_tiles, gridDim.x, o,
                  staging, wc);
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
  p.use_tma_store = encode_output_map(&p.tma_y, cp.y, cp.out_f32 != 0, cp.B * cp.groups, p.Cog, p.P,
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
