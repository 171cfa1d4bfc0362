// bi_common.h -- definitions shared by the host launchers and the kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace bi {

// ---------------------------------------------------------------------------
// The one fixed bf16 tile.  Never chosen from M, the batch count or the SM
// count: every output element of every call sees the same instruction
// sequence (128 x BN x 16 UMMA steps, K blocks of 64 in ascending order).
// ---------------------------------------------------------------------------
#ifndef BI_TILE_N
#define BI_TILE_N 256
#endif
constexpr int kBM = 128;        // UMMA M: rows of A / output rows per tile
constexpr int kBN = BI_TILE_N;  // UMMA N: output columns per tile
constexpr int kBK = 64;         // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kUmmaK = 16;      // K per tcgen05.mma (kind::f16)
constexpr int kGroupM = 16;     // raster group height (L2 reuse only; no numerical effect)
constexpr int kShortARows = 32; // A rows staged per k block when M <= 32 (same instructions)
// Packed weights: B is stored as the sequence of 64 x 64 shared-memory tile
// images the TMA path would produce (8 KB each, 128-byte swizzled), ordered
// [k block][64-column chunk], the chunk count padded to whole kBN tiles.  One
// pipeline stage of B is then one contiguous kBN/64 * 8 KB range.
constexpr int kPackChunk = 64;
constexpr int kPackChunkBytes = kPackChunk * kBK * 2;

// Device status codes (the status word holds the first failure of a device).
// Low byte: a bi_status value; next byte: where it happened.
enum : unsigned int {
  kSiteProducerEmpty = 1,
  kSiteMmaFull = 2,
  kSiteMmaTmemEmpty = 3,
  kSiteEpilogueTmemFull = 4,
  kSiteDrain = 5,
  kSiteDebugWait = 6,
  kSiteConvProducer = 7,
  kSitePack = 8,
  kSiteAttnSoftmax = 9,
};
__host__ __device__ constexpr unsigned int status_code(unsigned int bi_err, unsigned int site) {
  return bi_err | (site << 8);
}

struct GemmParams {
  CUtensorMap tma_a;  // A as [L][M][K] bf16, box {64, 128 (32 for M <= 32), 1}, 128B swizzle
  // B: K-major as [L][N][K], box {64, BN/2, 1}; MN-major as [L][K][N], box
  // {64, 64, 1} (both 128B swizzle); packed as [rows][64] (128-byte rows of
  // the packed image), box {64, BN/2*64*2/128, 1}, no swizzle
  CUtensorMap tma_b;
  CUtensorMap tma_c;  // C as [L][M][N], box {32, 32, 1} (fp32: 128B swizzle, bf16: 64B), if use_tma_store
  int64_t packed_kb_stride;  // bytes between consecutive k blocks of the packed B
  void* c;
  const void* bias;
  int64_t ldc;             // elements
  int64_t c_batch_stride;  // elements
  int64_t bias_stride;     // elements
  float alpha;
  int32_t M, N, K, L;
  int32_t m_tiles, n_tiles, k_blocks, num_tiles;
  int32_t out_f32;    // 1: fp32 output, 0: 16-bit output
  int32_t out_f16;    // 16-bit output is fp16 (else bf16)
  int32_t in_f16;     // A and B are fp16 (else bf16)
  int32_t bias_kind;  // 0: none, 1: bf16, 2: fp32, 3: fp16
  int32_t vec_store;  // 1: every output row start is 16-byte aligned
  int32_t use_tma_store;
  unsigned int* status_word;
  uint64_t wait_limit_ns;
};

struct ConvParams {
  CUtensorMap tma_y;   // y as [B*groups][Cog][P], box {32, 32, 1}, if use_tma_store
  const uint16_t* x;   // [B][C][H][W] bf16 contiguous
  const uint16_t* w;   // [Co][C/groups][KH][KW] bf16 contiguous
  const void* bias;    // [Co] or null
  void* y;             // [B][Co][Ho][Wo] contiguous
  int32_t B, C, H, W, Co, KH, KW, Ho, Wo;
  int32_t sh, sw, ph, pw, dh, dw, groups;
  int32_t Cig, Cog, Kg;       // channels per group in/out, reduction length per group
  int32_t P;                  // Ho*Wo output positions per sample
  int32_t m_tiles, n_tiles, k_blocks, num_tiles;  // per (sample, group) tile space
  int32_t out_f32, bias_kind, vec_store, use_tma_store;
  int32_t patch_fast;  // stride == kernel, no padding, unit dilation: row-wise patch loader
  int32_t x_vec16;     // image rows 16-byte aligned (16-byte loads in the patch loader)
  int32_t w_vec8;      // weight rows 8-byte aligned (8-byte loads for A)
  unsigned int* status_word;
  uint64_t wait_limit_ns;
};

// Largest staged K block of image rows of the patch convolution (4 kernel
// rows x t_oh output rows x the image width, bf16).
constexpr int kPatchStageMax = 32768;

// Non-overlapping patch convolution with a packed filter (see bi_patch.cu).
struct PatchParams {
  CUtensorMap tma_x;  // x as {W, KH, Ho, B*C}, box {W, 4, t_oh, 1}, no swizzle
  CUtensorMap tma_w;  // packed filter [Co][Kp], box {64, BN, 1}, 128B swizzle (packed filter only)
  const uint32_t* w_plain;  // or the filter as given, [Co][C][KH][KW] bf16 (KW 14 or 16), as bf16 pairs
  int32_t KH;
  const void* bias;   // [Co] or null
  void* y;            // [B][Co][Ho][Wo] contiguous
  int32_t C, W, KW, Wo, khq;    // khq: K blocks per input channel (KH rounded up to 4, / 4)
  int32_t t_oh, tile_rows, P, Co;  // output rows per tile, positions per tile, Ho*Wo
  int32_t m_tiles, n_tiles, k_blocks, num_tiles;
  uint32_t stg_bytes;  // bytes of one staged K block of image rows (W * 4 * t_oh * 2)
  int32_t out_f32, bias_kind;
  unsigned int* status_word;
  uint64_t wait_limit_ns;
};

struct SoftmaxParams {
  const float* s;
  void* p;
  int64_t R, N;
  int64_t ld_s, ld_p;  // elements
  int32_t out_f32;
};

}  // namespace bi
