// bi_gemm.cu -- persistent, warp-specialised tcgen05 GEMM for mm / addmm / bmm
// on CTA pairs, and the weight packer.
//
// The kernel runs as clusters of two CTAs on the two SMs of a TPC.  A tile is
// 256 rows x 256 columns; each CTA of the pair stages its own 128 rows of A
// and half of the tile's columns of B, and the even CTA issues 256-row
// tcgen05.mma (cta_group::2) instructions that read both CTAs' stages and
// leave rows 0..127 in its own TMEM, rows 128..255 in the odd CTA's.  Every SM
// thus ingests only half of the weight columns it multiplies -- for
// decode-sized M, where the weight stream is the whole cost, twice as many SMs
// stream it as with one CTA per tile.
//
//   warp 0      producer (each CTA): A (128 x 64) and its half of B (128 x 64)
//               of each K block into a ring of shared-memory stages (128-byte
//               swizzle), by TMA; the copies of both CTAs complete on the even
//               CTA's barrier of the stage.  Out-of-range rows / K are
//               zero-filled by the copy engine; an odd CTA whose 128 rows all
//               lie past M loads no A (its accumulator rows are never stored).
//               B comes from its strided layout or, for a packed weight, as
//               128-byte rows of the image already in shared-memory order.
//   warp 1      TMEM allocation (both CTAs, together); in the even CTA the
//               single-thread UMMA issuer (fp32 accumulators double-buffered
//               so the epilogue of tile i overlaps the main loop of tile i+1)
//   warps 2..5  epilogue (each CTA, its own 128 rows): tcgen05.ld -> alpha /
//               bias -> rounding -> global
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

// Shared-memory plan of one CTA of the pair.  A_ROWS = 128 is the general
// layout: A stages hold the CTA's whole 128-row A block, and the epilogue
// stages its output for TMA stores.  A_ROWS = 32 is the short-A layout for
// problems with at most 32 rows (decode-sized M), where the weight stream is
// the whole cost: A stages hold 32 rows, which frees room for more B stages
// in flight.  The tensor core still runs the same 256 x kGemmBN x 16 pair
// instructions in the same K order; its A rows 32..127 read whatever lies
// beyond the 32-row stage and only produce accumulator rows that are never
// stored (no output row reads another row's A data), so every stored element
// is computed exactly as in the general layout.
// Pair tile: 256 rows x kGemmBN columns; kGemmAcc accumulators of kGemmBN
// fp32 columns each in TMEM.
constexpr int kGemmBN = 256;
constexpr int kGemmAcc = 2;

template <int A_ROWS>
struct GemmLayout {
  static constexpr int A_BYTES = A_ROWS * kBK * 2;
  static constexpr int B_BYTES = (kGemmBN / 2) * kBK * 2;  // this CTA's half of the tile's columns
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int STAGING_BYTES = A_ROWS == kBM ? kEpilogueStagingBytes : 0;
  // The UMMA reads up to 128 A rows from each stage's A base: keep that span
  // inside the allocation for the last A stage.
  static constexpr int A_OVERREAD = (kBM - A_ROWS) * kBK * 2;
  static constexpr int MAX_DYN = 232448;  // 227 KB, the opt-in per-block maximum
  static constexpr int FIT = (MAX_DYN - 1024 - BAR_BYTES - STAGING_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = FIT > 16 ? 16 : FIT;
  static constexpr int DYN_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES + STAGING_BYTES;
  static constexpr uint32_t TMEM_COLS = kGemmAcc * kGemmBN;
  static_assert(STAGES >= 2, "pipeline needs at least two stages");
  static_assert(8 * (2 * STAGES + 2 * kGemmAcc + 1) + 8 <= BAR_BYTES, "barriers fit their block");
  static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation must be a power of two");
  static_assert(DYN_BYTES > 116 * 1024, "one CTA per SM: TMEM is allocated whole");
  static_assert(B_BYTES % kPackChunkBytes == 0, "packed half stage = whole chunks");
  static_assert(kBN % kGemmBN == 0, "packed tiles hold whole pair tiles");
  static_assert(A_OVERREAD <= STAGES * B_BYTES, "A over-read stays inside the B stages");
};

constexpr int kGemmThreads = 192;

// Producer cursor over this pair's (tile, k block) sequence.
struct ProdCursor {
  int tile, kb;
  uint32_t it;
  TileCoord tc;  // coordinates of `tile` for this CTA (mb: its 128-row block)
};

__device__ __forceinline__ TileCoord pair_tile(int tile, const GemmParams& p, uint32_t crank) {
  TileCoord tc = decode_tile(tile, p.m_tiles, p.n_tiles);
  tc.mb = 2 * tc.mb + (int)crank;
  return tc;
}

// One stage of this CTA: its A block (unless every one of its rows lies past
// M) and its half of the tile's B columns, into its own shared memory.  Every
// copy of both CTAs completes on the even CTA's full barrier of the stage,
// which the even CTA arms with the bytes of both.
template <bool B_MN, bool B_PACKED, int A_ROWS, bool STREAM_B>
__device__ __forceinline__ void issue_stage(const GemmParams& p, uint32_t sA, uint32_t sB,
                                            const PipeBars& bars, const ProdCursor& c,
                                            uint32_t crank) {
  using Lay = GemmLayout<A_ROWS>;
  const uint32_t s = c.it % Lay::STAGES;
  const TileCoord& tc = c.tc;
  const bool a_live = tc.mb * kBM < p.M;
  if (crank == 0) {
    const bool peer_live = (tc.mb + 1) * kBM < p.M;
    mbar_arrive_expect_tx(bars.full(s), 2 * Lay::B_BYTES + Lay::A_BYTES * (peer_live ? 2 : 1));
  }
  const uint32_t fb = cluster_map_shared(bars.full(s), 0);
  const uint32_t b_dst = sB + s * Lay::B_BYTES;
  const int n0 = tc.nb * kGemmBN + (int)crank * (kGemmBN / 2);
  // STREAM_B (at most two 256-row tiles): each block of B is used by one or
  // two CTA pairs and never again, so it is loaded with the evict-first L2
  // priority and the A rows, which every column tile reads again, with
  // evict-last.  Otherwise both take the default priority.  Data movement
  // only: the arithmetic is the same either way.
  auto load = [&](uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2, bool is_b) {
    if (STREAM_B)
      tma_load_3d_pair_hint(dst, map, fb, c0, c1, c2,
                            is_b ? l2_policy_evict_first() : l2_policy_evict_last());
    else
      tma_load_3d_pair(dst, map, fb, c0, c1, c2);
  };
  if (B_PACKED) {
    // The packed weight as rows of 128 bytes: this CTA's columns n0 .. are
    // whole 64-column chunks, B_BYTES / 128 consecutive rows of the image.
    const int64_t byte0 = (int64_t)c.kb * p.packed_kb_stride + (int64_t)(n0 / kPackChunk) * kPackChunkBytes;
    load(b_dst, &p.tma_b, 0, (int32_t)(byte0 / 128), 0, true);
  } else if (B_MN) {
#pragma unroll
    for (int j = 0; j < kGemmBN / 2 / 64; ++j) load(b_dst + j * 8192, &p.tma_b, n0 + j * 64, c.kb * kBK, tc.l, true);
  } else {
    load(b_dst, &p.tma_b, c.kb * kBK, n0, tc.l, true);
  }
  if (a_live) load(sA + s * Lay::A_BYTES, &p.tma_a, c.kb * kBK, tc.mb * kBM, tc.l, false);
}

__device__ __forceinline__ void advance(ProdCursor& c, const GemmParams& p, int stride,
                                        uint32_t crank) {
  ++c.it;
  if (++c.kb == p.k_blocks) {
    c.kb = 0;
    c.tile += stride;
    if (c.tile < p.num_tiles) c.tc = pair_tile(c.tile, p, crank);
  }
}

template <bool B_MN, bool B_PACKED, int A_ROWS, bool STREAM_B>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ GemmParams p) {
  using Lay = GemmLayout<A_ROWS>;
  const uint32_t crank = cluster_ctarank();  // 0: the pair's MMA issuer
  const int stride = gridDim.x >> 1;         // pairs; every pair owns tiles
  const int first_tile = blockIdx.x >> 1;
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
  bars.tempty0 = bars.tfull0 + 8 * kGemmAcc;
  bars.drain = bars.tempty0 + 8 * kGemmAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + (bars.drain + 8 - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  ProdCursor cur{first_tile, 0, 0u, {0, 0, 0}};

  if (threadIdx.x == 0) {
    // Even CTA: a stage is full when the copies of both CTAs have landed; an
    // accumulator is free when the four epilogue warps of both CTAs have
    // drained it.  (The odd CTA's full and tempty barriers stay unused.)
    for (int s = 0; s < Lay::STAGES; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    for (int b = 0; b < kGemmAcc; ++b) {
      mbar_init(bars.tfull(b), 1);
      mbar_init(bars.tempty(b), 8);
    }
    mbar_init(bars.drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&p.tma_a);
    tma_prefetch_desc(&p.tma_b);
    cur.tc = pair_tile(cur.tile, p, crank);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Lay::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // Both CTAs' barriers are initialised before any copy or signal crosses
  // between them.  Meanwhile the even CTA starts its first ring of loads,
  // which needs no free-stage wait and signals only its own barriers.
  cluster_arrive_relaxed();
  if (threadIdx.x == 0) {
    while (crank == 0 && cur.it < (uint32_t)Lay::STAGES && cur.tile < p.num_tiles) {
      issue_stage<B_MN, B_PACKED, A_ROWS, STREAM_B>(p, sA, sB, bars, cur, crank);
      advance(cur, p, stride, crank);
    }
  }
  __syncwarp();
  cluster_wait();
  const WaitCtl wc{abort_flag, p.status_word, p.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      while (cur.tile < p.num_tiles) {
        const uint32_t s = cur.it % Lay::STAGES;
        const uint32_t r = cur.it / Lay::STAGES;
        if (r > 0 && !mbar_wait_bounded(bars.empty(s), (r - 1) & 1, wc.abort, wc.status_word,
                                        wc.limit_ns, status_code(6, kSiteProducerEmpty)))
          break;
        issue_stage<B_MN, B_PACKED, A_ROWS, STREAM_B>(p, sA, sB, bars, cur, crank);
        advance(cur, p, stride, crank);
      }
      // No copy may still be landing in shared memory, and no MMA-completion
      // signal may still be on its way to this CTA, when it exits: wait
      // (bounded) until the last fill of every stage has been consumed.
      const uint32_t it = cur.it;
      const uint32_t first = it > (uint32_t)Lay::STAGES ? it - Lay::STAGES : 0u;
      for (uint32_t j = first; j < it; ++j)
        if (!mbar_wait_bounded(bars.empty(j % Lay::STAGES), (j / Lay::STAGES) & 1, nullptr,
                               wc.status_word, wc.limit_ns, status_code(6, kSiteDrain)))
          break;
    }
  } else if (warp == 1) {
    if (lane == 0 && crank == 0)
      mma_role<Lay::STAGES, Lay::A_BYTES, Lay::B_BYTES, B_MN, true, kGemmBN, kGemmAcc>(
          sA, sB, bars, tmem_base, first_tile, p.num_tiles, p.k_blocks, stride, wc, p.in_f16 != 0);
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
    o.trans = 0;
    o.tile_rows = kBM;
    o.out_f16 = p.out_f16;
    o.tma_c = (Lay::STAGING_BYTES > 0 && p.use_tma_store) ? &p.tma_c : nullptr;
    const uint32_t staging = bar0 + Lay::BAR_BYTES + (warp - 2) * 2 * kStageOutBytes;
    epilogue_role<true, kGemmBN, kGemmAcc>(warp & 3, lane, tmem_base, bars, first_tile, p.num_tiles, p.m_tiles,
                        p.n_tiles, stride, o, staging, wc, crank);
  }

  // Neither CTA leaves while the other may still signal it or use its TMEM.
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, Lay::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Weight packer: chunk c = (k block kb, 64-column chunk nc) of the packed
// buffer receives, byte for byte, the 64 x 64 shared-memory image that the
// GEMM's TMA path would load for it (same tensor map geometry, same swizzle,
// zeros outside the matrix).  One warp per CTA: TMA load -> smem -> bulk store.
// ---------------------------------------------------------------------------
constexpr int kPackThreads = 32;
constexpr int kPackDynBytes = 1024 + kPackChunkBytes + 64;

__global__ void __launch_bounds__(kPackThreads) pack_kernel(const __grid_constant__ CUtensorMap tmap,
                                                            uint8_t* dst, int k_blocks, int nc_pad,
                                                            int b_mn, unsigned int* status_word,
                                                            uint64_t limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t buf = (raw + 1023u) & ~1023u;
  const uint32_t bar = buf + kPackChunkBytes;
  int* abort_flag = reinterpret_cast<int*>(smem_raw + (bar + 8 - raw));
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmap);
    uint32_t phase = 0;
    const int64_t total = (int64_t)k_blocks * nc_pad;
    for (int64_t c = blockIdx.x; c < total; c += gridDim.x) {
      const int kb = (int)(c / nc_pad);
      const int nc = (int)(c - (int64_t)kb * nc_pad);
      mbar_arrive_expect_tx(bar, kPackChunkBytes);
      if (b_mn)
        tma_load_3d(buf, &tmap, bar, nc * kPackChunk, kb * kBK, 0);
      else
        tma_load_3d(buf, &tmap, bar, kb * kBK, nc * kPackChunk, 0);
      if (!mbar_wait_bounded(bar, phase, abort_flag, status_word, limit_ns,
                             status_code(6, kSitePack)))
        break;
      phase ^= 1u;
      bulk_store(dst + c * kPackChunkBytes, buf, kPackChunkBytes);
      bulk_commit();
      bulk_wait_read_all();  // the buffer is refilled next iteration
    }
    bulk_wait_all();
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// A 16-bit operand (bf16, or fp16 with f16) as a 3-D tensor map, 128-byte swizzle.
static bool encode_3d(CUtensorMap* map, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, bool f16,
                      std::string* why) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  const cuuint32_t box[3] = {b0, b1, 1};
  return encode_tiled(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      CU_TENSOR_MAP_SWIZZLE_128B, const_cast<void*>(ptr), 3, dims, strides, box, why);
}

// B's tensor map: MN-major as [L][K][N] with 64 x 64 boxes, K-major as
// [L][N][K] with 64 x rows boxes.
static bool encode_b(CUtensorMap* map, const GemmProblem& g, uint32_t k_major_rows, std::string* why) {
  const uint64_t b_row = (uint64_t)g.ldb * 2;
  if (g.b_mn_major) {
    const uint64_t b_bat = g.L > 1 ? (uint64_t)g.b_batch * 2 : round_up_u64(b_row * (uint64_t)g.K, 16);
    return encode_3d(map, g.b, g.N, g.K, g.L, b_row, b_bat, 64, kBK, g.in_f16 != 0, why);
  }
  const uint64_t b_bat = g.L > 1 ? (uint64_t)g.b_batch * 2 : round_up_u64(b_row * (uint64_t)g.N, 16);
  return encode_3d(map, g.b, g.K, g.N, g.L, b_row, b_bat, kBK, k_major_rows, g.in_f16 != 0, why);
}

int64_t packed_bytes(int64_t K, int64_t N) {
  if (K <= 0 || N <= 0) return 0;
  const int64_t k_blocks = (K + kBK - 1) / kBK;
  const int64_t n_tiles = (N + kBN - 1) / kBN;
  return k_blocks * n_tiles * (kBN / kPackChunk) * (int64_t)kPackChunkBytes;
}

bi_status launch_pack(const GemmProblem& g, void* dst, cudaStream_t stream, std::string* why) {
  DeviceInfo dev;
  bi_status st = current_device_info(&dev, why);
  if (st != BI_OK) return st;
  CUtensorMap map;
  if (!encode_b(&map, g, kPackChunk, why)) return BI_ERR_CUDA;
  const int k_blocks = (int)((g.K + kBK - 1) / kBK);
  const int nc_pad = (int)(((g.N + kBN - 1) / kBN) * (kBN / kPackChunk));
  const int64_t total = (int64_t)k_blocks * nc_pad;
  const int grid = (int)std::min<int64_t>(total, (int64_t)dev.num_sms * 8);
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&pack_kernel), kPackDynBytes, 5);
  if (e == cudaSuccess)
    pack_kernel<<<grid, kPackThreads, kPackDynBytes, stream>>>(map, reinterpret_cast<uint8_t*>(dst),
                                                               k_blocks, nc_pad, g.b_mn_major,
                                                               dev.status_word, kWaitLimitNs);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("pack launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

// Grid: two CTAs per pair, min(#tiles, #pairs that fit at once) pairs.
template <bool B_MN, bool B_PACKED, int A_ROWS, bool STREAM_B>
static cudaError_t launch_variant(const GemmParams& p, int64_t tiles, cudaStream_t stream, int slot) {
  using Lay = GemmLayout<A_ROWS>;
  const void* fn = reinterpret_cast<const void*>(&gemm_kernel<B_MN, B_PACKED, A_ROWS, STREAM_B>);
  cudaError_t e = set_smem_once(fn, Lay::DYN_BYTES, slot);
  if (e != cudaSuccess) return e;
  int pairs = 0;
  e = pair_capacity(fn, kGemmThreads, Lay::DYN_BYTES, slot, &pairs);
  if (e != cudaSuccess) return e;
  const int grid = 2 * (int)std::min<int64_t>(tiles, pairs);
  gemm_kernel<B_MN, B_PACKED, A_ROWS, STREAM_B><<<grid, kGemmThreads, Lay::DYN_BYTES, stream>>>(p);
  return cudaSuccess;
}

template <int A_ROWS, bool STREAM_B>
static cudaError_t launch_rows(const GemmProblem& g, const GemmParams& p, int64_t tiles,
                               cudaStream_t stream, int slot0) {
  if (g.b_packed)
    return g.b_mn_major ? launch_variant<true, true, A_ROWS, STREAM_B>(p, tiles, stream, slot0 + 2)
                        : launch_variant<false, true, A_ROWS, STREAM_B>(p, tiles, stream, slot0 + 3);
  return g.b_mn_major ? launch_variant<true, false, A_ROWS, STREAM_B>(p, tiles, stream, slot0)
                      : launch_variant<false, false, A_ROWS, STREAM_B>(p, tiles, stream, slot0 + 1);
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
  // Short-A layout when every tile has at most 32 rows (see GemmLayout).
  const bool short_a = M <= kShortARows;
  const uint64_t a_row = (uint64_t)g.lda * 2;
  const uint64_t a_bat = L > 1 ? (uint64_t)g.a_batch * 2 : round_up_u64(a_row * (uint64_t)M, 16);
  if (!encode_3d(&p.tma_a, g.a, K, M, L, a_row, a_bat, kBK, short_a ? kShortARows : kBM, g.in_f16 != 0,
                 why))
    return BI_ERR_CUDA;
  if (g.b_packed) {
    // The packed image as [rows][64] bf16 (128-byte rows, no swizzle: the
    // image is already in shared-memory order), boxes of 128 rows.
    p.packed_kb_stride = ((N + kBN - 1) / kBN) * (int64_t)(kBN * kBK * 2);
    const uint64_t rows = (uint64_t)((K + kBK - 1) / kBK) * (uint64_t)p.packed_kb_stride / 128;
    const cuuint64_t dims[3] = {64, rows, 1};
    const cuuint64_t strides[2] = {128, rows * 128};
    const cuuint32_t box[3] = {64, kGemmBN / 2 * kBK * 2 / 128, 1};
    if (rows > INT32_MAX || !encode_tiled(&p.tma_b,
                                          g.in_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                          CU_TENSOR_MAP_SWIZZLE_NONE,
                                          const_cast<void*>(g.b_packed), 3, dims, strides, box, why))
      return rows > INT32_MAX ? BI_ERR_INVALID_ARG : BI_ERR_CUDA;
  } else if (!encode_b(&p.tma_b, g, kGemmBN / 2, why)) {  // K-major: each CTA's columns
    return BI_ERR_CUDA;
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
  p.m_tiles = (int32_t)((M + 2 * kBM - 1) / (2 * kBM));  // 256-row pair tiles
  p.n_tiles = (int32_t)((N + kGemmBN - 1) / kGemmBN);
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
  p.use_tma_store =
      encode_output_map(&p.tma_c, g.c, g.out_f32 != 0, g.out_f16 != 0, L, M, N, g.ldc, g.c_batch) ? 1 : 0;
  p.out_f16 = g.out_f16;
  p.in_f16 = g.in_f16;
  p.status_word = dev.status_word;
  p.wait_limit_ns = kWaitLimitNs;

  // Kernel slots: 0-3 general layout, 16-19 the same with the weight
  // streamed (at most two row tiles), 8-11 short A (always one row tile).
  cudaError_t e = short_a         ? launch_rows<kShortARows, true>(g, p, tiles, stream, 8)
                  : p.m_tiles <= 2 ? launch_rows<kBM, true>(g, p, tiles, stream, 16)
                                   : launch_rows<kBM, false>(g, p, tiles, stream, 0);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("gemm launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

}  // namespace bi
