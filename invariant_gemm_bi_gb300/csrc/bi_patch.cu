// bi_patch.cu -- non-overlapping patch convolution (patch embedding) as an
// implicit-im2col tcgen05 GEMM with a packed filter.
//
// For stride = kernel size, no padding, no dilation and one group (the
// patch-embedding layer of "Batch-Invariant VLAs", section "Replacing
// nn.Conv2d", and "Batch-Invariant Kernel Design: Conv2d and Attention BMM",
// section "Kernel 1: Conv2d"), output position (oh, ow) of sample b reads the
// disjoint KH x KW window of every channel at (oh*KH, ow*KW).  Per sample
//   Y[b]^T (P x Co) = Patches[b] (P x Kp) . Wp^T (Kp x Co)  + bias
// with P = Ho*Wo positions as the rows of the product.  The reduction runs
// over kp = (ci*KHp + kh)*16 + kw, KHp = KH rounded up to a multiple of 4:
// every kernel row (ci, kh) occupies 16 slots, slots kh >= KH or kw >= KW
// are zero on both sides.  One tensor-core K = 16 step is thus one kernel row,
// and a 64-wide K block is four rows (ci, kh0 .. kh0+3) of one channel.
//
// No unfolded matrix exists anywhere.  Per K block the producers TMA-load,
// for the tile's t_oh output rows, the four image rows (ci, oh*KH + kh0 ..
// +3) of the sample -- whole rows, 16-byte aligned, rows past KH zero-filled
// by the copy engine -- and the [192 x 64] block of the packed filter.  Four
// builder warps then turn the staged rows into the patch tile (one row per
// output position, zeros for kw >= KW) and write it straight into tensor
// memory, where the MMA takes its A operand: the tile never passes through
// shared memory (writing and reading it there was the largest share of the
// shared-memory traffic).  A tile is (sample, block of t_oh output rows,
// 192 channels): it never mixes samples, so one sample's arithmetic is the
// same for every batch size.
//
//   warp 0      filter producer (TMA, a ring of 4 stages); with the filter
//               as given (not packed), warps 0 and 11-13 build each filter
//               stage instead (below)
//   warp 1      TMEM allocator + UMMA issuer (128 x 192 x 16, cta_group::1,
//               A from TMEM, B = the filter block from shared memory)
//   warps 2..5  epilogue: tcgen05.ld -> + bias -> rounding -> y (NCHW: the
//               32 threads of a warp write 32 consecutive positions of a
//               channel per store)
//   warps 6..9  patch-tile builders (warp w writes TMEM lanes 32 (w % 4) ..)
//   warp 10     image-row producer (TMA, a ring of up to 8 staged blocks: a
//               copy from L2 takes about a microsecond, several K blocks'
//               worth, so the rows are fetched well ahead of the filter)
//
// TMEM: accumulators at columns 0 and 192 (the epilogue of one tile overlaps
// the next tile's MMAs), patch-tile stages of 32 columns (64 bf16 k per
// position) from column 384.
#include <cuda.h>
#include <cuda_runtime.h>

#include "bi_common.h"
#include "bi_launch.h"
#include "bi_ptx.cuh"
#include "bi_ptx_ext.cuh"
#include "bi_roles.cuh"

namespace bi {

constexpr int kPatchBN = 192;  // output channels per tile

struct PatchLayout {
  static constexpr int B_BYTES = kPatchBN * kBK * 2;  // 192 channels x 64 k
  static constexpr int STAGES = 4;                    // K blocks in flight (filter + TMEM patch tile)
  static constexpr int STG_BUFS = 8;                  // staged image-row blocks, at most
  static constexpr int STG_REGION = 128 * 1024;       // holds min(8, region / block) blocks (>= 4)
  static constexpr int BAR_BYTES = 1024;
  static constexpr int DYN_BYTES = 1024 + STAGES * B_BYTES + STG_REGION + BAR_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t A_COL = 2 * kPatchBN;     // first patch-tile stage column
  static_assert(A_COL + STAGES * (kBK / 2) <= TMEM_COLS, "accumulators and patch stages fit TMEM");
  static_assert(DYN_BYTES <= 232448, "fits the opt-in shared memory of one CTA");
  static_assert(DYN_BYTES > 116 * 1024, "one CTA per SM: TMEM is allocated whole");
  static_assert(8 * (2 * STAGES + 2 * STG_BUFS + 5) + 8 <= BAR_BYTES, "barriers fit their block");
  static_assert(STG_REGION / kPatchStageMax >= 4, "at least four staged blocks of the largest size");
};

// Staged image blocks ([oh_l][g][x], x over the image width): each at a 1 KB
// boundary, as many as the region holds (up to 8).
struct StgRing {
  uint32_t stride;
  int n;
  __device__ __forceinline__ explicit StgRing(uint32_t bytes)
      : stride((bytes + 1023u) & ~1023u), n(min(PatchLayout::STG_BUFS, (int)(PatchLayout::STG_REGION / stride))) {}
};

constexpr int kPatchThreads = 352;
constexpr int kPatchThreadsPlain = 448;  // + warps 11..13: filter builders with warp 0
constexpr int kPatchBuilders = 128;      // warps 6..9
constexpr int kPatchFilterBuilders = 128;

// Filter builders (the filter as given, KW = 14 or 16): a K block's [192
// channels x 64 k] filter block laid out exactly as the TMA copy of the
// packed filter lays it out -- row r (channel nb*192 + r) of 128 bytes, its
// 16-byte unit u at u ^ (r % 8) (the 128-byte swizzle), words 8g .. 8g + 7 of
// the row holding kw = 0 .. 15 of kernel row kh0 + g as bf16 pairs -- with
// zeros for kw >= KW, kh >= KH and channels past Co.  A channel's kernel rows
// kh0 .. kh0 + 3 are one contiguous run of the filter (4 KW bf16), so thread
// t (0..127) reads half rows t, t + 128 and t + 256 (two kernel rows of a
// channel each) with 8-byte (KW = 14) or 16-byte (KW = 16) loads and writes
// each with four 16-byte stores, the pad words in place.  The pieces of the
// next two K blocks are in flight while a stage is waited for and written.
template <int KW>
struct FilterRun {
  static constexpr int kWords = KW;  // 2 kernel rows of KW bf16, as 32-bit words
  uint32_t w[3][kWords];             // half rows t, t + 128, t + 256
};

// Half row hr = 2 r + h2 of the block: kernel rows kh0 + 2 h2, kh0 + 2 h2 + 1
// of channel nb*192 + r.
template <int KW>
__device__ __forceinline__ void filter_load(const PatchParams& p, int t, int nb, int kb, FilterRun<KW>& f) {
  const int ci = kb / p.khq;
  const int kh0 = (kb - ci * p.khq) * 4;
  const int rows = min(4, p.KH - kh0);  // kernel rows of this block inside the filter
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int hr = t + 128 * j, r = hr >> 1, h2 = hr & 1;
    const int co = nb * kPatchBN + r;
    const bool live = co < p.Co && 2 * h2 < rows;  // KW = 14: rows is even, a half row is whole or absent
    const uint32_t* src = p.w_plain + (((int64_t)co * p.C + ci) * p.KH + kh0 + 2 * h2) * (KW / 2);
    if (KW == 16) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 16-byte pieces, two per kernel row
        const bool in = co < p.Co && 2 * h2 + c / 2 < rows;
        const uint4 v = in ? __ldg(reinterpret_cast<const uint4*>(src) + c) : make_uint4(0u, 0u, 0u, 0u);
        f.w[j][4 * c] = v.x;
        f.w[j][(4 * c + 1) % KW] = v.y;
        f.w[j][(4 * c + 2) % KW] = v.z;
        f.w[j][(4 * c + 3) % KW] = v.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < KW / 2; ++c) {  // 8-byte pieces
        const uint2 v = live ? __ldg(reinterpret_cast<const uint2*>(src) + c) : make_uint2(0u, 0u);
        f.w[j][2 * c] = v.x;
        f.w[j][2 * c + 1] = v.y;
      }
    }
  }
}

template <int KW>
__device__ __forceinline__ void filter_store(uint32_t dst, int t, const FilterRun<KW>& f) {
  constexpr int kw2 = KW / 2;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int hr = t + 128 * j, r = hr >> 1, h2 = hr & 1;
    const uint32_t row = dst + r * 128;
#pragma unroll
    for (int uu = 0; uu < 4; ++uu) {  // unit u = 4 h2 + uu: kernel row 2 h2 + uu / 2, pairs 4 (uu % 2) ..
      uint32_t q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int g = uu / 2, e = 4 * (uu % 2) + i;
        q[i] = e < kw2 ? f.w[j][g * kw2 + e] : 0u;
      }
      const int u = 4 * h2 + uu;
      st_shared_v4(row + ((uint32_t)(u ^ (r & 7)) << 4), q[0], q[1], q[2], q[3]);
    }
  }
}

template <int KW>
__device__ __forceinline__ void patch_filter_builder(const PatchParams& p, uint32_t sB, const PipeBars& bars, int t,
                                                     const WaitCtl& wc) {
  using Lay = PatchLayout;
  const int lane = t & 31;
  FilterRun<KW> f0, f1;
  int tile_ld = blockIdx.x, kb_ld = 0;  // the next block to load
  auto load_next = [&](FilterRun<KW>& dst) {
    if (tile_ld >= p.num_tiles) return;
    filter_load<KW>(p, t, decode_tile(tile_ld, p.m_tiles, p.n_tiles).nb, kb_ld, dst);
    if (++kb_ld == p.k_blocks) {
      kb_ld = 0;
      tile_ld += gridDim.x;
    }
  };
  load_next(f0);
  load_next(f1);
  const uint32_t total = (uint32_t)max(0, (p.num_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x) *
                         (uint32_t)p.k_blocks;
  // Block it from cur, then cur takes block it + 2.
  auto step = [&](uint32_t it, FilterRun<KW>& cur) -> bool {
    const uint32_t s = it % Lay::STAGES, r = it / Lay::STAGES;
    const bool got = r == 0 || mbar_wait_bounded(bars.empty(s), (r - 1) & 1, wc.abort, wc.status_word,
                                                  wc.limit_ns, status_code(6, kSiteProducerEmpty));
    if (!__all_sync(0xffffffffu, got)) return false;
    filter_store<KW>(sB + s * Lay::B_BYTES, t, cur);
    fence_proxy_async_smem();  // the tensor core reads the stage through the async proxy
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.full(s));
    load_next(cur);
    return true;
  };
  for (uint32_t it = 0; it < total; it += 2) {
    if (!step(it, f0)) break;
    if (it + 1 < total && !step(it + 1, f1)) break;
  }
}

// Patch-tile row r (one output position; zeros past the tile's positions) of
// one K block from the staged image rows, as the 32 TMEM columns of the
// position's lane: column 8g + e holds kw = 2e (low half) and 2e + 1 (high
// half) of kernel row kh0 + g.
__device__ __forceinline__ void build_patch_words(const PatchParams& p, uint32_t stg, int r, uint32_t (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 32; ++c) v[c] = 0u;
  if (r >= p.tile_rows) return;
  const int oh_l = r / p.Wo;
  const int ow = r - oh_l * p.Wo;
  if ((p.KW & 1) == 0) {
    // Even KW: every staged pair (kw, kw+1) with kw < KW is 4-byte aligned
    // and lies inside its image row; pairs past KW are not read.
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t row = stg + (uint32_t)(((oh_l * 4 + g) * p.W + ow * p.KW) * 2);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (2 * e < p.KW) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[8 * g + e]) : "r"(row + 4 * e));
    }
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t row = stg + (uint32_t)(((oh_l * 4 + g) * p.W + ow * p.KW) * 2);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (e < p.KW) {
          uint16_t h;
          asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(row + 2 * e));
          v[8 * g + (e >> 1)] |= (uint32_t)h << (16 * (e & 1));
        }
    }
  }
}

// Single thread: the tiles' UMMAs, A (the patch tile) from TMEM stage s, B
// (the filter block) from shared-memory stage s; accumulators alternate.
__device__ __forceinline__ void patch_mma(uint32_t sB, const PipeBars& bars, uint32_t tmem_base, int first_tile,
                                          int num_tiles, int k_blocks, int stride, const WaitCtl& w) {
  using Lay = PatchLayout;
  const uint32_t kIdesc = idesc_bf16_f32(kBM, kPatchBN, false);
  uint32_t it = 0;
  int local = 0;
  bool ok = true;
  for (int tile = first_tile; ok && tile < num_tiles; tile += stride, ++local) {
    const uint32_t buf = local & 1, use = local >> 1;
    if (use > 0 && !mbar_wait_bounded(bars.tempty(buf), (use - 1) & 1, w.abort, w.status_word, w.limit_ns,
                                      status_code(6, kSiteMmaTmemEmpty))) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    const uint32_t d = tmem_base + buf * kPatchBN;
    for (int kb = 0; kb < k_blocks; ++kb, ++it) {
      const uint32_t s = it % Lay::STAGES, r = it / Lay::STAGES;
      if (!mbar_wait_bounded(bars.full(s), r & 1, w.abort, w.status_word, w.limit_ns,
                             status_code(6, kSiteMmaFull))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t a = tmem_base + Lay::A_COL + s * (kBK / 2);
      const uint32_t b = sB + s * Lay::B_BYTES;
#pragma unroll
      for (int k = 0; k < kBK / kUmmaK; ++k)  // one kernel row per step, ascending
        umma_bf16_ts(d, a + k * (kUmmaK / 2), smem_desc_sw128(b + k * 32, 16, 1024), kIdesc,
                     (kb | k) != 0 ? 1u : 0u);
      umma_commit(bars.empty(s));  // filter stage and patch-tile stage s are free once these finish
    }
    if (!ok) break;
    umma_commit(bars.tfull(buf));
  }
  // Every MMA issued above has finished before TMEM can be released.
  umma_commit(bars.drain);
  mbar_wait_bounded(bars.drain, 0, nullptr, w.status_word, w.limit_ns, status_code(6, kSiteDrain));
}

template <bool PLAIN>
__global__ void __launch_bounds__(PLAIN ? kPatchThreadsPlain : kPatchThreads, 1)
    patch_kernel(const __grid_constant__ PatchParams p) {
  using Lay = PatchLayout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sB = base;
  const uint32_t sStg = sB + Lay::STAGES * Lay::B_BYTES;
  const uint32_t bar0 = sStg + Lay::STG_REGION;
  const StgRing ring(p.stg_bytes);
  PipeBars bars;
  bars.full0 = bar0;
  bars.empty0 = bar0 + 8 * Lay::STAGES;
  bars.tfull0 = bars.empty0 + 8 * Lay::STAGES;
  bars.tempty0 = bars.tfull0 + 16;
  bars.drain = bars.tempty0 + 16;
  const uint32_t stg_full0 = bars.drain + 8;
  const uint32_t stg_empty0 = stg_full0 + 8 * Lay::STG_BUFS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + (stg_empty0 + 8 * Lay::STG_BUFS - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // A stage is full when its filter block has landed (or the four filter
    // builder warps have written it) and the four patch builder warps have
    // written its patch tile into TMEM.
    for (int s = 0; s < Lay::STAGES; ++s) {
      mbar_init(bars.full(s), (PLAIN ? kPatchFilterBuilders / 32 : 1) + kPatchBuilders / 32);
      mbar_init(bars.empty(s), 1);
    }
    for (int q = 0; q < ring.n; ++q) {
      mbar_init(stg_full0 + 8 * q, 1);
      mbar_init(stg_empty0 + 8 * q, kPatchBuilders / 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.tfull(b), 1);
      mbar_init(bars.tempty(b), 4);
    }
    mbar_init(bars.drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&p.tma_x);
    if (!PLAIN) tma_prefetch_desc(&p.tma_w);
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

  if (PLAIN && (warp == 0 || warp >= 11)) {
    const int t = (warp == 0 ? 0 : warp - 10) * 32 + lane;
    if (p.KW == 16)
      patch_filter_builder<16>(p, sB, bars, t, wc);
    else
      patch_filter_builder<14>(p, sB, bars, t, wc);
  } else if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const TileCoord tc = decode_tile(tile, p.m_tiles, p.n_tiles);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const uint32_t s = it % Lay::STAGES, r = it / Lay::STAGES;
          if (r > 0 && !mbar_wait_bounded(bars.empty(s), (r - 1) & 1, wc.abort, wc.status_word,
                                          wc.limit_ns, status_code(6, kSiteProducerEmpty))) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bars.full(s), Lay::B_BYTES);
          tma_load_3d(sB + s * Lay::B_BYTES, &p.tma_w, bars.full(s), kb * kBK, tc.nb * kPatchBN, 0);
        }
      }
      // No copy may still be landing in shared memory when the CTA exits.
      const uint32_t first = it > (uint32_t)Lay::STAGES ? it - Lay::STAGES : 0u;
      for (uint32_t j = first; j < it; ++j)
        if (!mbar_wait_bounded(bars.full(j % Lay::STAGES), (j / Lay::STAGES) & 1, nullptr,
                               wc.status_word, wc.limit_ns, status_code(6, kSiteDrain)))
          break;
    }
  } else if (warp == 10) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const TileCoord tc = decode_tile(tile, p.m_tiles, p.n_tiles);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const uint32_t q = it % ring.n, rq = it / ring.n;
          if (rq > 0 && !mbar_wait_bounded(stg_empty0 + 8 * q, (rq - 1) & 1, wc.abort, wc.status_word,
                                           wc.limit_ns, status_code(6, kSiteProducerEmpty))) {
            ok = false;
            break;
          }
          const int ci = kb / p.khq;
          const int kh0 = (kb - ci * p.khq) * 4;
          mbar_arrive_expect_tx(stg_full0 + 8 * q, p.stg_bytes);
          tma_load_4d(sStg + q * ring.stride, &p.tma_x, stg_full0 + 8 * q, 0, kh0, tc.mb * p.t_oh,
                      tc.l * p.C + ci);
        }
      }
      const uint32_t first_q = it > (uint32_t)ring.n ? it - ring.n : 0u;
      for (uint32_t j = first_q; j < it; ++j)
        if (!mbar_wait_bounded(stg_full0 + 8 * (j % ring.n), (j / ring.n) & 1, nullptr, wc.status_word,
                               wc.limit_ns, status_code(6, kSiteDrain)))
          break;
    }
  } else if (warp == 1) {
    if (lane == 0) patch_mma(sB, bars, tmem_base, blockIdx.x, p.num_tiles, p.k_blocks, gridDim.x, wc);
  } else if (warp < 6) {
    OutDesc o;
    o.c = p.y;
    o.bias = p.bias;
    o.tma_c = nullptr;
    o.ldc = p.P;  // between output channels (the tile's columns)
    o.c_batch_stride = (int64_t)p.Co * p.P;
    o.bias_stride = 1;
    o.alpha = 1.0f;
    o.M = p.P;
    o.N = p.Co;
    o.out_f32 = p.out_f32;
    o.bias_kind = p.bias_kind;
    o.vec_store = 0;
    o.bias_per_row = 0;
    o.bias_groups = 1;
    o.trans = 1;
    o.tile_rows = p.tile_rows;
    o.out_f16 = 0;
    epilogue_role<false, kPatchBN, 2>(warp & 3, lane, tmem_base, bars, blockIdx.x, p.num_tiles, p.m_tiles,
                                      p.n_tiles, gridDim.x, o, 0u, wc);
  } else if (warp < 10) {
    // Patch-tile builders: a warp may reach only its TMEM lane quadrant, so
    // thread `lane` of warp w writes tile row 32 (w % 4) + lane.
    const int t = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + Lay::A_COL;
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const uint32_t s = it % Lay::STAGES, r = it / Lay::STAGES;
        const uint32_t q = it % ring.n, rq = it / ring.n;
        bool got = mbar_wait_bounded(stg_full0 + 8 * q, rq & 1, wc.abort, wc.status_word, wc.limit_ns,
                                     status_code(6, kSiteConvProducer));
        if (got && r > 0)
          got = mbar_wait_bounded(bars.empty(s), (r - 1) & 1, wc.abort, wc.status_word, wc.limit_ns,
                                  status_code(6, kSiteConvProducer));
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();  // the MMAs that read patch stage s have finished
        uint32_t v[32];
        build_patch_words(p, sStg + q * ring.stride, t, v);
        tmem_store_32cols(lane_base + s * (kBK / 2), v);
        tmem_store_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bars.full(s));
          mbar_arrive(stg_empty0 + 8 * q);
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Lay::TMEM_COLS);
  }
}

// Packed filter: wp[co][kp], kp = (ci*KHp + kh)*16 + kw, zero where kh >= KH
// or kw >= KW.  One thread per 8 consecutive kp (16-byte stores).
__global__ void conv_pack_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ wp, int Co, int C,
                                 int KH, int KW, int KHp, int Kp) {
  const int64_t groups = (int64_t)Co * (Kp / 8);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < groups;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int co = (int)(i / (Kp / 8));
    const int kp0 = (int)(i - (int64_t)co * (Kp / 8)) * 8;
    uint32_t v[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int kp = kp0 + e;
      const int kw = kp & 15;
      const int kh = (kp >> 4) % KHp;
      const int ci = (kp >> 4) / KHp;
      if (kh < KH && kw < KW)
        v[e >> 1] |= (uint32_t)w[(((int64_t)co * C + ci) * KH + kh) * KW + kw] << (16 * (e & 1));
    }
    *reinterpret_cast<uint4*>(wp + (int64_t)co * Kp + kp0) = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

int64_t patch_padded_k(int64_t C, int64_t KH) { return C * ((KH + 3) / 4 * 4) * 16; }

// The filter builders read a channel's kernel-row runs with 16-byte (KW = 16)
// or 8-byte (KW = 14: a run starts at ((co C + ci) KH + kh0) 28 bytes, a
// multiple of 8 when KH is even) loads.
bool patch_plain_filter_ok(int64_t KH, int64_t KW, const void* w) {
  return (KW == 16 || (KW == 14 && KH % 2 == 0)) && reinterpret_cast<uintptr_t>(w) % 16 == 0;
}

int64_t patch_stage_bytes(int64_t W, int64_t t_oh) { return W * 4 * t_oh * 2; }

int64_t patch_tile_rows(int64_t Ho, int64_t Wo, int64_t W) {
  int64_t t = std::min<int64_t>(Ho, kBM / std::max<int64_t>(Wo, 1));
  while (t > 1 && patch_stage_bytes(W, t) > kPatchStageMax) --t;
  return std::max<int64_t>(t, 1);
}

bi_status launch_conv_pack(const void* w, void* dst, int64_t Co, int64_t C, int64_t KH, int64_t KW,
                           cudaStream_t stream, std::string* why) {
  DeviceInfo dev;
  bi_status st = current_device_info(&dev, why);
  if (st != BI_OK) return st;
  const int64_t Kp = patch_padded_k(C, KH);
  const int64_t groups = Co * (Kp / 8);
  const int grid = (int)std::min<int64_t>((groups + 255) / 256, (int64_t)dev.num_sms * 8);
  conv_pack_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint16_t*>(w),
                                             reinterpret_cast<uint16_t*>(dst), (int)Co, (int)C, (int)KH,
                                             (int)KW, (int)((KH + 3) / 4 * 4), (int)Kp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("conv pack launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

bi_status launch_patch(const PatchProblem& pp, cudaStream_t stream, std::string* why) {
  DeviceInfo dev;
  bi_status st = current_device_info(&dev, why);
  if (st != BI_OK) return st;
  PatchParams p;
  memset(&p, 0, sizeof(p));
  const int64_t Kp = patch_padded_k(pp.C, pp.KH);
  const int64_t t_oh = patch_tile_rows(pp.Ho, pp.Wo, pp.W);
  // x as {W, KH, Ho, B*C}: element (x, kh, oh, b*C + ci) is x[b][ci][oh*KH + kh][x].
  {
    const cuuint64_t dims[4] = {(cuuint64_t)pp.W, (cuuint64_t)pp.KH, (cuuint64_t)pp.Ho,
                                (cuuint64_t)(pp.B * pp.C)};
    const cuuint64_t strides[3] = {(cuuint64_t)pp.W * 2, (cuuint64_t)(pp.KH * pp.W * 2),
                                   (cuuint64_t)(pp.H * pp.W * 2)};
    const cuuint32_t box[4] = {(cuuint32_t)pp.W, 4, (cuuint32_t)t_oh, 1};
    if (!encode_tiled(&p.tma_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_NONE,
                      const_cast<void*>(pp.x), 4, dims, strides, box, why))
      return BI_ERR_CUDA;
  }
  const bool plain = pp.wp == nullptr;
  if (plain) {
    if (!patch_plain_filter_ok(pp.KH, pp.KW, pp.w)) {
      *why = "the filter as given needs KW = 14 (with KH even) or 16, 16-byte aligned";
      return BI_ERR_UNSUPPORTED_LAYOUT;
    }
    p.w_plain = static_cast<const uint32_t*>(pp.w);
  } else {
    const cuuint64_t dims[3] = {(cuuint64_t)Kp, (cuuint64_t)pp.Co, 1};
    const cuuint64_t strides[2] = {(cuuint64_t)Kp * 2, (cuuint64_t)(Kp * 2 * pp.Co)};
    const cuuint32_t box[3] = {kBK, kPatchBN, 1};
    if (!encode_tiled_bf16(&p.tma_w, const_cast<void*>(pp.wp), 3, dims, strides, box, why))
      return BI_ERR_CUDA;
  }
  p.bias = pp.bias;
  p.y = pp.y;
  p.C = (int32_t)pp.C;
  p.W = (int32_t)pp.W;
  p.KW = (int32_t)pp.KW;
  p.KH = (int32_t)pp.KH;
  p.Wo = (int32_t)pp.Wo;
  p.khq = (int32_t)((pp.KH + 3) / 4);
  p.t_oh = (int32_t)t_oh;
  p.tile_rows = (int32_t)(t_oh * pp.Wo);
  p.P = (int32_t)(pp.Ho * pp.Wo);
  p.Co = (int32_t)pp.Co;
  p.m_tiles = (int32_t)((pp.Ho + t_oh - 1) / t_oh);
  p.n_tiles = (int32_t)((pp.Co + kPatchBN - 1) / kPatchBN);
  p.k_blocks = (int32_t)(Kp / kBK);
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles * pp.B;
  if (tiles > INT32_MAX) {
    *why = "tile count exceeds 2^31";
    return BI_ERR_INVALID_ARG;
  }
  p.num_tiles = (int32_t)tiles;
  p.stg_bytes = (uint32_t)(pp.W * 4 * t_oh * 2);
  p.out_f32 = pp.out_f32;
  p.bias_kind = pp.bias_kind;
  p.status_word = dev.status_word;
  p.wait_limit_ns = kWaitLimitNs;
  const void* fn = plain ? reinterpret_cast<const void*>(&patch_kernel<true>)
                         : reinterpret_cast<const void*>(&patch_kernel<false>);
  cudaError_t e = set_smem_once(fn, PatchLayout::DYN_BYTES, plain ? 15 : 6);
  if (e == cudaSuccess) {
    const int grid = (int)std::min<int64_t>(tiles, dev.num_sms);
    if (plain)
      patch_kernel<true><<<grid, kPatchThreadsPlain, PatchLayout::DYN_BYTES, stream>>>(p);
    else
      patch_kernel<false><<<grid, kPatchThreads, PatchLayout::DYN_BYTES, stream>>>(p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    *why = std::string("patch conv launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

}  // namespace bi
