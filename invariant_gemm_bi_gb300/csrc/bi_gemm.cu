// bi_gemm.cu -- persistent, warp-specialised tcgen05 GEMM for mm / addmm / bmm.
//
//   warp 0      TMA producer: A (128 x 64) and B (kBN x 64) tiles of each K
//               block into a ring of shared-memory stages (128-byte swizzle,
//               out-of-range elements zero-filled by the copy engine)
//   warp 1      TMEM allocator + single-thread UMMA issuer (fp32 accumulator
//               in TMEM, double-buffered so the epilogue of tile i overlaps
//               the main loop of tile i+1)
//   warps 2..5  epilogue: tcgen05.ld -> alpha / bias -> rounding -> global
//
// Batch elements of bmm are a third tile coordinate, so tiles never straddle
// batch elements ("Batch-Invariant Kernel Design: Conv2d and Attention BMM",
// section "Kernel 2: Attention BMM": each batch element gets its own base
// pointers and the same ordered reduction over K).
#include <cuda.h>
#include <cuda_runtime.h>

#include "bi_common.h"
#include "bi_launch.h"
#include "bi_ptx.cuh"
#include "bi_roles.cuh"

namespace bi {

struct GemmLayout {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = kBN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int MAX_DYN = 232448;  // 227 KB, the opt-in per-block maximum
  static constexpr int FIT = (MAX_DYN - 1024 - BAR_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr int DYN_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * kBN;
  static_assert(STAGES >= 2, "pipeline needs at least two stages");
  static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation must be a power of two");
  static_assert(DYN_BYTES > 116 * 1024, "one CTA per SM: TMEM is allocated whole");
};

constexpr int kGemmThreads = 192;

template <bool B_MN>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  using Lay = GemmLayout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1 KB alignment
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
      mbar_init(bars.full(s), 1);
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
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Lay::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status_word, p.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.tma_a);
      tma_prefetch_desc(&p.tma_b);
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const TileCoord tc = decode_tile(tile, p.m_tiles, p.n_tiles);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          const uint32_t s = it % Lay::STAGES;
          const uint32_t r = it / Lay::STAGES;
          if (r > 0 && !mbar_wait_bounded(bars.empty(s), (r - 1) & 1, wc.abort, wc.status_word,
                                          wc.limit_ns, status_code(6, kSiteProducerEmpty))) {
            ok = false;
            break;
          }
          const uint32_t fb = bars.full(s);
          mbar_arrive_expect_tx(fb, Lay::STAGE_BYTES);
          tma_load_3d(sA + s * Lay::A_BYTES, &p.tma_a, fb, kb * kBK, tc.mb * kBM, tc.l);
          const uint32_t b_dst = sB + s * Lay::B_BYTES;
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j)
              tma_load_3d(b_dst + j * 8192, &p.tma_b, fb, tc.nb * kBN + j * 64, kb * kBK, tc.l);
          } else {
            tma_load_3d(b_dst, &p.tma_b, fb, kb * kBK, tc.nb * kBN, tc.l);
          }
          if (kPrefetchKBlocks > 0 && kb + kPrefetchKBlocks < p.k_blocks) {
            const int kp = (kb + kPrefetchKBlocks) * kBK;
            tma_prefetch_l2_3d(&p.tma_a, kp, tc.mb * kBM, tc.l);
            if (B_MN) {
#pragma unroll
              for (int j = 0; j < kBN / 64; ++j)
                tma_prefetch_l2_3d(&p.tma_b, tc.nb * kBN + j * 64, kp, tc.l);
            } else {
              tma_prefetch_l2_3d(&p.tma_b, kp, tc.nb * kBN, tc.l);
            }
          }
          ++it;
        }
      }
      // No copy may still be landing in shared memory when the CTA exits:
      // wait (bounded) for the last fill of every stage.
      const uint32_t first = it > (uint32_t)Lay::STAGES ? it - Lay::STAGES : 0u;
      for (uint32_t j = first; j < it; ++j)
        mbar_wait_bounded(bars.full(j % Lay::STAGES), (j / Lay::STAGES) & 1, nullptr,
                          wc.status_word, wc.limit_ns, status_code(6, kSiteDrain));
    }
  } else if (warp == 1) {
    if (lane == 0)
      mma_role<Lay::STAGES, Lay::A_BYTES, Lay::B_BYTES, B_MN>(sA, sB, bars, tmem_base, p.num_tiles,
                                                              p.k_blocks, wc);
  } else {
    OutDesc o;
    o.c = p.c;
    o.bias = p.bias;
    o.ldc = p.ldc;
    o.c_batch_stride = p.c_batch_stride;
    o.bias_stride = p.bias_stride;
    o.alpha = p.alpha;
    o.M = p.M;
    o.N = p.N;
    o.out_f32 = p.out_f32;
    o.bias_kind = p.bias_kind;
    o.vec_store = p.vec_store;
    o.bias_per_row = 0;
    o.bias_groups = 1;
    epilogue_role(warp & 3, lane, tmem_base, bars, p.num_tiles, p.m_tiles, p.n_tiles, o, wc);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Lay::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

static bool encode_3d(CUtensorMap* map, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1,
                      std::string* why) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_tiled_bf16(map, const_cast<void*>(ptr), 3, dims, strides, box, estr, why);
}

bi_status launch_gemm(const GemmProblem& g, cudaStream_t stream, std::string* why) {
  DeviceInfo dev;
  bi_status st = current_device_info(&dev, why);
  if (st != BI_OK) return st;

  GemmParams p;
  memset(&p, 0, sizeof(p));
  const int64_t L = g.L, M = g.M, N = g.N, K = g.K;
  // A: [L][M][K]; the batch stride of a single batch element is never used,
  // but must still be a legal (16-byte multiple) stride.
  const uint64_t a_row = (uint64_t)g.lda * 2;
  const uint64_t a_bat = L > 1 ? (uint64_t)g.a_batch * 2 : round_up_u64(a_row * (uint64_t)M, 16);
  if (!encode_3d(&p.tma_a, g.a, K, M, L, a_row, a_bat, kBK, kBM, why)) return BI_ERR_CUDA;
  if (g.b_mn_major) {
    const uint64_t b_row = (uint64_t)g.ldb * 2;  // stride between k rows
    const uint64_t b_bat = L > 1 ? (uint64_t)g.b_batch * 2 : round_up_u64(b_row * (uint64_t)K, 16);
    if (!encode_3d(&p.tma_b, g.b, N, K, L, b_row, b_bat, 64, kBK, why)) return BI_ERR_CUDA;
  } else {
    const uint64_t b_row = (uint64_t)g.ldb * 2;  // stride between n rows
    const uint64_t b_bat = L > 1 ? (uint64_t)g.b_batch * 2 : round_up_u64(b_row * (uint64_t)N, 16);
    if (!encode_3d(&p.tma_b, g.b, K, N, L, b_row, b_bat, kBK, kBN, why)) return BI_ERR_CUDA;
  }
  p.c = g.c;
  p.bias = g.bias;
  p.ldc = g.ldc;
  p.c_batch_stride = g.c_batch;
  p.bias_stride = g.bias_stride;
  p.alpha = g.alpha;
  p.M = (int32_t)M;
  p.N = (int32_t)N;
  p.K = (int32_t)K;
  p.L = (int32_t)L;
  p.m_tiles = (int32_t)((M + kBM - 1) / kBM);
  p.n_tiles = (int32_t)((N + kBN - 1) / kBN);
  p.k_blocks = (int32_t)((K + kBK - 1) / kBK);
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles * L;
  if (tiles > INT32_MAX) {
    *why = "tile count exceeds 2^31";
    return BI_ERR_INVALID_ARG;
  }
  p.num_tiles = (int32_t)tiles;
  p.out_f32 = g.out_f32;
  p.bias_kind = g.bias_kind;
  p.vec_store = g.vec_store;
  p.status_word = dev.status_word;
  p.wait_limit_ns = kWaitLimitNs;

  const int grid = (int)std::min<int64_t>(tiles, dev.num_sms);
  cudaError_t e;
  if (g.b_mn_major) {
    e = set_smem_once(reinterpret_cast<const void*>(&gemm_kernel<true>), GemmLayout::DYN_BYTES, 0);
    if (e == cudaSuccess)
      gemm_kernel<true><<<grid, kGemmThreads, GemmLayout::DYN_BYTES, stream>>>(p);
  } else {
    e = set_smem_once(reinterpret_cast<const void*>(&gemm_kernel<false>), GemmLayout::DYN_BYTES, 1);
    if (e == cudaSuccess)
      gemm_kernel<false><<<grid, kGemmThreads, GemmLayout::DYN_BYTES, stream>>>(p);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("gemm launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

}  // namespace bi
