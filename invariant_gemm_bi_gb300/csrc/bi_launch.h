// bi_launch.h -- host-side interfaces between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>
#include <string>

#include "../../include/bi.h"
#include "bi_common.h"

namespace bi {

// Fused attention (bi_attn.cu): o[l] = softmax(scale * q[l] k[l]^T) v[l].
struct AttnParams {
  CUtensorMap tma_q;  // q as {D, Tq, L}, box {64, 128, 1}, 128B swizzle
  CUtensorMap tma_k;  // k as {D, Tk, L}, box {64, 128, 1}
  CUtensorMap tma_v;  // v as {D, Tk, L}, box {64, 32, 1}
  void* o;            // o[l][t][d] at o + l*o_l + t*o_t + d (fp32 or bf16)
  int64_t o_t, o_l;
  float* ws_o;        // split key range: partial O [ns][L][Tq][256]
  float* ws_ml;       // and (m, l) [ns][L][Tq][2]
  int32_t ns;         // key-range splits (1: not split)
  int32_t L, Tq, Tk, q_tiles, num_tiles;
  int32_t pair_units, units;  // two-tile kernel: units holding two query tiles, all units
  float score_log2;  // scale * log2(e), rounded once to fp32
  int32_t out_f32;
  unsigned int* status_word;
  uint64_t wait_limit_ns;
};

// Row reductions over the last dimension (see bi_rows.cu).
enum : int { kRowRmsNorm = 0, kRowLogSoftmax = 1, kRowMean = 2 };
struct RowParams {
  const void* x;  // [R][N], row stride ld_x elements, unit column stride
  void* y;        // [R][N] (row stride ld_y), or for the mean [R] (stride ld_y)
  const void* w;  // RMSNorm weight [N] (stride w_stride), or null
  int64_t R, N, ld_x, ld_y, w_stride;
  int32_t x_kind, y_kind, w_kind;  // 0 bf16, 1 fp16, 2 fp32
  int32_t x_esz, y_esz;            // element sizes in bytes
  int32_t cl;                      // CTAs per row (a cluster) for 1024-thread teams, else 1
  float eps;
};


// Bound on every device-side wait: far above any legitimate wait (a tile's
// whole K loop takes well under a millisecond), short enough that a broken
// pipeline returns an error instead of holding the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

inline uint64_t round_up_u64(uint64_t v, uint64_t m) { return (v + m - 1) / m * m; }

struct DeviceInfo {
  int device;
  int num_sms;
  unsigned int* status_word;  // device address of this device's status word
};

// Fills `info` for the current device (cached per device).  Fails with
// BI_ERR_NO_DEVICE unless the device is compute capability 10.3 (sm_103).
bi_status current_device_info(DeviceInfo* info, std::string* why);

// cuTensorMapEncodeTiled with zero fill out of bounds (driver entry point
// resolved once through the runtime).
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle,
                  void* ptr, uint32_t rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                  const cuuint32_t* box, std::string* why);
// bf16 operand tiles with the 128-byte swizzle.
inline bool encode_tiled_bf16(CUtensorMap* map, void* ptr, uint32_t rank, const cuuint64_t* dims,
                              const cuuint64_t* strides_bytes, const cuuint32_t* box,
                              std::string* why) {
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, ptr, rank,
                      dims, strides_bytes, box, why);
}
// Tensor map of an output [L][M][N] (row stride ldc, batch stride c_batch,
// elements) for the epilogue's 32 x 32 tile stores; false when the layout is
// not TMA-legal (the epilogue then stores directly).
bool encode_output_map(CUtensorMap* map, void* c, bool f32, bool f16, int64_t L, int64_t M, int64_t N,
                       int64_t ldc, int64_t c_batch);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (device, slot).
cudaError_t set_smem_once(const void* func, int bytes, int slot);

// How many 2-CTA clusters of a kernel compiled with __cluster_dims__(2,1,1)
// can be resident at once (cudaOccupancyMaxActiveClusters), once per
// (device, slot); at least 1.
cudaError_t pair_capacity(const void* func, int threads, int dyn_bytes, int slot, int* pairs);

// A normalised matrix-product problem: c[l] = alpha * a[l] @ b[l] (+ bias).
struct GemmProblem {
  const void* a;  // bf16, [L][M][K], unit stride on K
  int64_t lda, a_batch;
  const void* b;  // bf16; b_mn_major: b[l][k][n] at k*ldb + n; else at n*ldb + k
  int64_t ldb, b_batch;
  int b_mn_major;
  const void* b_packed;  // packed weight (L == 1), or null; b_mn_major gives its image layout
  void* c;  // [L][M][N], unit stride on N
  int64_t ldc, c_batch;
  int out_f32;
  int out_f16;       // 16-bit output is fp16 (else bf16)
  int in_f16;        // a and b are fp16 (else bf16)
  const void* bias;  // per column n, or null
  int64_t bias_stride;
  int bias_kind;  // 0 none, 1 bf16, 2 fp32, 3 fp16
  float alpha;
  int64_t L, M, N, K;
  int vec_store;
};

bi_status launch_gemm(const GemmProblem& g, cudaStream_t stream, std::string* why);

// Bytes of the packed form of a [K, N] weight; packs g's B (L == 1) into dst.
int64_t packed_bytes(int64_t K, int64_t N);
bi_status launch_pack(const GemmProblem& g, void* dst, cudaStream_t stream, std::string* why);

struct ConvProblem {
  const void* x;
  const void* w;
  const void* bias;
  int bias_kind;
  void* y;
  int out_f32;
  int64_t B, C, H, W, Co, KH, KW, Ho, Wo;
  int sh, sw, ph, pw, dh, dw, groups;
};

bi_status launch_conv(const ConvProblem& cp, cudaStream_t stream, std::string* why);

// Non-overlapping patch convolution with a packed filter (bi_patch.cu).
struct PatchProblem {
  const void* x;   // [B][C][H][W] bf16 contiguous, 16-byte aligned, W*2 % 16 == 0
  const void* wp;  // packed filter [Co][patch_padded_k(C, KH)], or null:
  const void* w;   // the filter as given, [Co][C][KH][KW] bf16 contiguous (patch_plain_filter_ok)
  const void* bias;
  int bias_kind;
  void* y;  // [B][Co][Ho][Wo] contiguous
  int out_f32;
  int64_t B, C, H, W, Co, KH, KW, Ho, Wo;
};
// Row length of the packed filter: C * (KH rounded up to 4) * 16.
int64_t patch_padded_k(int64_t C, int64_t KH);
// Whether the patch kernel can build its filter stages from the filter as
// given: KW = 16, or KW = 14 with KH even; w 16-byte aligned.
bool patch_plain_filter_ok(int64_t KH, int64_t KW, const void* w);
// Shared memory of one staged K block of image rows (t_oh output rows of an
// image W pixels wide); at most kPatchStageMax.
int64_t patch_stage_bytes(int64_t W, int64_t t_oh);
// Output rows per tile: whole rows, at most 128 positions, one staged block
// within kPatchStageMax.  A function of the image shape only.
int64_t patch_tile_rows(int64_t Ho, int64_t Wo, int64_t W);
bi_status launch_conv_pack(const void* w, void* dst, int64_t Co, int64_t C, int64_t KH, int64_t KW,
                           cudaStream_t stream, std::string* why);
bi_status launch_patch(const PatchProblem& pp, cudaStream_t stream, std::string* why);

bi_status launch_softmax(const SoftmaxParams& sp, cudaStream_t stream, std::string* why);

// Fused attention: q [L][Tq][256], k and v [L][Tk][256] bf16 (unit stride on
// D, 16-byte row and batch strides), o [L][Tq][256] fp32 or bf16.
struct AttnProblem {
  const void *q, *k, *v;
  int64_t q_t, q_l, k_t, k_l, v_t, v_l;  // element strides over T and L
  void* o;
  int64_t o_t, o_l;
  int out_f32;
  float scale;
  int64_t L, Tq, Tk, D;
  void* ws;  // workspace for a split key range (Tk > 2048), or null
  int64_t ws_bytes;
};
bi_status launch_attention(const AttnProblem& ap, cudaStream_t stream, std::string* why);
// Key-range splits (2048 keys each) and the workspace they need (0 if one).
int64_t attention_splits(int64_t Tk);
int64_t attention_workspace_bytes(int64_t L, int64_t Tq, int64_t Tk, int64_t D);
// The head dimensions the fused attention kernel is built for: 64, 128, 256.
bool attention_head_dim_ok(int64_t D);

// op: kRowRmsNorm, kRowLogSoftmax or kRowMean.
bi_status launch_row_reduction(int op, const RowParams& rp, cudaStream_t stream, std::string* why);

bi_status launch_fill_bias(const GemmProblem& g, cudaStream_t stream, std::string* why);

bi_status launch_debug_wait(uint64_t limit_ns, cudaStream_t stream, std::string* why);

}  // namespace bi
