// bi_rows.cu -- invariant row reductions over the last dimension: RMSNorm,
// log-softmax and the row mean ("Unmasking the True Culprit: Why
// Temperature=0 Doesn't Mean Deterministic LLM Inference", section "Beyond
// Matrix Multiplication: Other Critical Operations"; aten::mean.dim in
// "Batch-Invariant VLAs"; "ai-infra handbook: deterministic inference", on
// normalisation, softmax and means: one block reduces one row in a fixed
// order, never splitting a row because there are few rows).
//
// A row of N elements is reduced by a team of T threads, T fixed by N alone:
// the smallest power of two from 32 to 1024 with N <= 32 T (so a thread holds
// at most 8 groups of 4 elements; rows longer than 32768 elements use 1024
// threads and more groups each).  Teams smaller than 256 threads share a
// 256-thread block.  The row is cut into groups of 4 consecutive elements;
// thread t owns groups t, t+T, t+2T, ... and accumulates their elements in
// ascending index order in fp32; each warp combines its 32 partials by a fixed
// xor butterfly, and a team of several warps adds the warp partials in warp
// order.  The order depends only on N and the element index -- not on the
// number of rows, on the row's address (aligned rows are loaded 4 elements at
// a time, others one at a time, with the same arithmetic) or on which SM runs
// it.  A thread loads its groups 8 at a time, all 8 before using any, and
// keeps them in registers: a row of up to 32768 elements is read from memory
// once, longer rows once per pass.
//
//   RMSNorm      ss = sum x_j^2;  ms = RN(ss / N);  r = RN(1 / RN(sqrt(ms + eps)))
//                y_j = RN(RN(x_j * r) * w_j)           (w absent: y_j = RN(x_j * r))
//   log-softmax  m = max x_j;  se = sum expf(x_j - m);  lse = logf(se)
//                y_j = RN(RN(x_j - m) - lse)
//   mean         y = RN(sum x_j / N)
// with every add / multiply / divide / square root a separately rounded fp32
// operation, then one rounding to the output type.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "bi_common.h"
#include "bi_launch.h"

namespace bi {

constexpr int kRowGroups = 8;          // groups a thread loads together (one chunk)
constexpr int kRowMinBlock = 256;      // teams smaller than this share a block
constexpr int kRowMaxTeam = 1024;

__device__ __forceinline__ float rows_warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float rows_warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// The team's total of the per-thread partials v, the same bits in every
// thread of the team.  For T > 32 every thread of the block must call it (it
// holds block barriers); the team's warps are contiguous in the block.
template <int T>
__device__ __forceinline__ float team_sum(float v, float* red) {
  v = rows_warp_sum(v);
  if constexpr (T == 32) {
    return v;
  } else {
    __syncthreads();  // red is free: every thread has read its previous contents
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    const float* r = red + (threadIdx.x / T) * (T / 32);
    float s = r[0];
#pragma unroll
    for (int i = 1; i < T / 32; ++i) s = __fadd_rn(s, r[i]);
    return s;
  }
}
template <int T>
__device__ __forceinline__ float team_max(float v, float* red) {
  v = rows_warp_max(v);
  if constexpr (T == 32) {
    return v;
  } else {
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    const float* r = red + (threadIdx.x / T) * (T / 32);
    float s = r[0];
#pragma unroll
    for (int i = 1; i < T / 32; ++i) s = fmaxf(s, r[i]);
    return s;
  }
}

// Element j of a row of type `kind` (0 bf16, 1 fp16, 2 fp32) as fp32 (exact).
__device__ __forceinline__ float row_load(const void* base, int kind, int64_t j) {
  if (kind == 2) return __ldg(reinterpret_cast<const float*>(base) + j);
  const uint16_t h = __ldg(reinterpret_cast<const unsigned short*>(base) + j);
  if (kind == 1) return __half2float(__ushort_as_half(h));
  return __bfloat162float(__ushort_as_bfloat16(h));
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h, int kind) {
  return kind == 1 ? __half2float(__ushort_as_half((unsigned short)h))
                   : __bfloat162float(__ushort_as_bfloat16((unsigned short)h));
}

// Group g (elements 4g .. 4g+3) of a row whose base is aligned to 4 elements.
__device__ __forceinline__ void load_group_vec(const void* base, int kind, int64_t g, float (&v)[4]) {
  if (kind == 2) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(base) + g);
    v[0] = q.x, v[1] = q.y, v[2] = q.z, v[3] = q.w;
  } else {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(base) + g);
    v[0] = half_bits_to_float(q.x & 0xffffu, kind), v[1] = half_bits_to_float(q.x >> 16, kind);
    v[2] = half_bits_to_float(q.y & 0xffffu, kind), v[3] = half_bits_to_float(q.y >> 16, kind);
  }
}

__device__ __forceinline__ void row_store(void* base, int kind, int64_t j, float v) {
  if (kind == 2)
    reinterpret_cast<float*>(base)[j] = v;
  else if (kind == 1)
    reinterpret_cast<__half*>(base)[j] = __float2half_rn(v);
  else
    reinterpret_cast<__nv_bfloat16*>(base)[j] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi, int kind) {
  if (kind == 1)
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// Stores the n (<= 4) values of the group starting at element j; vec: the row
// base is aligned to 4 elements (then a whole group is one store).
__device__ __forceinline__ void store_group(void* base, int kind, bool vec, int64_t j, int n,
                                            const float (&v)[4]) {
  if (vec && n == 4) {
    if (kind == 2)
      reinterpret_cast<float4*>(base)[j >> 2] = make_float4(v[0], v[1], v[2], v[3]);
    else
      reinterpret_cast<uint2*>(base)[j >> 2] =
          make_uint2(pack_half2(v[0], v[1], kind), pack_half2(v[2], v[3], kind));
    return;
  }
  for (int i = 0; i < n; ++i) row_store(base, kind, j + i, v[i]);
}

__device__ __forceinline__ bool aligned4(const void* p, int esz) {
  return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)(4 * esz)) == 0;
}

// One chunk of a thread's groups: chunk c holds its groups t + (8c + k) T,
// k = 0..7, as the raw words of the row (XK 2: fp32, a group is 4 words;
// XK 0: a 2-byte type, bf16 or fp16 as `kind` says, a group is 2 words), zeros
// past the end of the row.  All loads are issued before any value is used.
template <int XK>
struct RowChunk {
  static constexpr int kWords = XK == 2 ? 4 : 2;
  int kind;    // element type (0 bf16, 1 fp16, 2 fp32)
  uint32_t w[kRowGroups][kWords];
  int64_t g0;  // group index of k = 0
  int64_t nfull;
  int tail;    // elements in group nfull (N mod 4)
  // elements of group k that exist (0 past the end of the row)
  __device__ __forceinline__ int n(int k, int T) const {
    const int64_t g = g0 + (int64_t)k * T;
    return g < nfull ? 4 : (g == nfull ? tail : 0);
  }
  __device__ __forceinline__ float v(int k, int i) const {
    if constexpr (XK == 2) return __uint_as_float(w[k][i]);
    const uint32_t h = (w[k][i >> 1] >> (16 * (i & 1))) & 0xffffu;
    return half_bits_to_float(h, kind);
  }
};

template <int T, int XK>
__device__ __forceinline__ void load_chunk(const void* x, int kind, bool vec, int64_t N, int t, int c,
                                           RowChunk<XK>& ch) {
  ch.kind = kind;
  ch.nfull = N >> 2;
  ch.tail = (int)(N & 3);
  ch.g0 = (int64_t)c * kRowGroups * T + t;
#pragma unroll
  for (int k = 0; k < kRowGroups; ++k) {
    const int64_t g = ch.g0 + (int64_t)k * T;
    if (g < ch.nfull && vec) {
      if constexpr (XK == 2) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(x) + g);
        ch.w[k][0] = q.x, ch.w[k][1] = q.y, ch.w[k][2] = q.z, ch.w[k][3] = q.w;
      } else {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(x) + g);
        ch.w[k][0] = q.x, ch.w[k][1] = q.y;
      }
    } else {
      const int n = g < ch.nfull ? 4 : (g == ch.nfull ? ch.tail : 0);
      if constexpr (XK == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          ch.w[k][i] = i < n ? __float_as_uint(__ldg(reinterpret_cast<const float*>(x) + 4 * g + i)) : 0u;
      } else {
        const unsigned short* h = reinterpret_cast<const unsigned short*>(x) + 4 * g;
        uint32_t e[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) e[i] = i < n ? (uint32_t)__ldg(h + i) : 0u;
        ch.w[k][0] = e[0] | (e[1] << 16), ch.w[k][1] = e[2] | (e[3] << 16);
      }
    }
  }
}

// Number of chunks a thread of a T-team walks for a row of N elements.
template <int T>
__device__ __forceinline__ int row_chunks(int64_t N) {
  const int64_t groups = (N + 3) >> 2;
  return (int)((groups + (int64_t)T * kRowGroups - 1) / ((int64_t)T * kRowGroups));
}

// f(value) over the chunk's existing elements, groups then elements ascending.
template <int T, int XK, typename F>
__device__ __forceinline__ void chunk_visit(const RowChunk<XK>& ch, F&& f) {
#pragma unroll
  for (int k = 0; k < kRowGroups; ++k) {
    const int n = ch.n(k, T);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i < n) f(ch.v(k, i));
  }
}

// Which row a thread's team reduces and the thread's index in the team.
template <int T>
struct RowSlot {
  static constexpr int kBlock = T < kRowMinBlock ? kRowMinBlock : T;
  int64_t row;
  int t;
  __device__ __forceinline__ RowSlot()
      : row((int64_t)blockIdx.x * (kBlock / T) + threadIdx.x / T), t((int)(threadIdx.x % T)) {}
};

template <int T, int XK>
__device__ __forceinline__ void rms_store_chunk(const RowParams& p, void* y, bool yvec, bool wvec, float r,
                                                const RowChunk<XK>& ch) {
#pragma unroll
  for (int k = 0; k < kRowGroups; ++k) {
    const int n = ch.n(k, T);
    if (n == 0) continue;
    const int64_t j = 4 * (ch.g0 + (int64_t)k * T);
    float o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = __fmul_rn(ch.v(k, i), r);
    if (p.w) {
      float w[4];
      if (wvec && n == 4) {
        load_group_vec(p.w, p.w_kind, j >> 2, w);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = i < n ? row_load(p.w, p.w_kind, (j + i) * p.w_stride) : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = __fmul_rn(o[i], w[i]);
    }
    store_group(y, p.y_kind, yvec, j, n, o);
  }
}

template <int T, int XK>
__global__ void __launch_bounds__(RowSlot<T>::kBlock, 1024 / RowSlot<T>::kBlock) rmsnorm_kernel(const RowParams p) {
  __shared__ float red[RowSlot<T>::kBlock / 32];
  const RowSlot<T> rs;
  const bool live = rs.row < p.R;
  if (T == 32 && !live) return;  // warp teams hold no block barrier
  const int64_t row = live ? rs.row : 0;
  const void* x = static_cast<const char*>(p.x) + row * p.ld_x * p.x_esz;
  void* y = static_cast<char*>(p.y) + row * p.ld_y * p.y_esz;
  const bool xvec = aligned4(x, p.x_esz);
  const int nch = live ? row_chunks<T>(p.N) : 0;
  RowChunk<XK> ch;
  float acc = 0.0f;
  for (int c = 0; c < nch; ++c) {
    load_chunk<T, XK>(x, p.x_kind, xvec, p.N, rs.t, c, ch);
    chunk_visit<T>(ch, [&](float v) { acc = __fadd_rn(acc, __fmul_rn(v, v)); });
  }
  const float ss = team_sum<T>(acc, red);
  if (!live) return;  // past the team's last barrier
  const float ms = __fdiv_rn(ss, (float)p.N);
  const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, p.eps)));
  const bool yvec = aligned4(y, p.y_esz);
  const bool wvec = p.w && p.w_stride == 1 && aligned4(p.w, p.w_kind == 2 ? 4 : 2);
  for (int c = 0; c < nch; ++c) {
    if (nch > 1) load_chunk<T, XK>(x, p.x_kind, xvec, p.N, rs.t, c, ch);  // one chunk: still in registers
    rms_store_chunk<T>(p, y, yvec, wvec, r, ch);
  }
}

template <int T, int XK>
__global__ void __launch_bounds__(RowSlot<T>::kBlock, 1024 / RowSlot<T>::kBlock) log_softmax_kernel(const RowParams p) {
  __shared__ float red[RowSlot<T>::kBlock / 32];
  const RowSlot<T> rs;
  const bool live = rs.row < p.R;
  if (T == 32 && !live) return;
  const int64_t row = live ? rs.row : 0;
  const void* x = static_cast<const char*>(p.x) + row * p.ld_x * p.x_esz;
  void* y = static_cast<char*>(p.y) + row * p.ld_y * p.y_esz;
  const bool xvec = aligned4(x, p.x_esz);
  const int nch = live ? row_chunks<T>(p.N) : 0;
  RowChunk<XK> ch;
  float m = -INFINITY;
  for (int c = 0; c < nch; ++c) {
    load_chunk<T, XK>(x, p.x_kind, xvec, p.N, rs.t, c, ch);
    chunk_visit<T>(ch, [&](float v) { m = fmaxf(m, v); });
  }
  m = team_max<T>(m, red);
  float acc = 0.0f;
  for (int c = 0; c < nch; ++c) {
    if (nch > 1) load_chunk<T, XK>(x, p.x_kind, xvec, p.N, rs.t, c, ch);
    chunk_visit<T>(ch, [&](float v) { acc = __fadd_rn(acc, expf(__fsub_rn(v, m))); });
  }
  const float lse = logf(team_sum<T>(acc, red));
  if (!live) return;
  const bool yvec = aligned4(y, p.y_esz);
  for (int c = 0; c < nch; ++c) {
    if (nch > 1) load_chunk<T, XK>(x, p.x_kind, xvec, p.N, rs.t, c, ch);
#pragma unroll
    for (int k = 0; k < kRowGroups; ++k) {
      const int n = ch.n(k, T);
      if (n == 0) continue;
      float o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = __fsub_rn(__fsub_rn(ch.v(k, i), m), lse);
      store_group(y, p.y_kind, yvec, 4 * (ch.g0 + (int64_t)k * T), n, o);
    }
  }
}

template <int T, int XK>
__global__ void __launch_bounds__(RowSlot<T>::kBlock, 1024 / RowSlot<T>::kBlock) mean_kernel(const RowParams p) {
  __shared__ float red[RowSlot<T>::kBlock / 32];
  const RowSlot<T> rs;
  const bool live = rs.row < p.R;
  if (T == 32 && !live) return;
  const int64_t row = live ? rs.row : 0;
  const void* x = static_cast<const char*>(p.x) + row * p.ld_x * p.x_esz;
  const bool xvec = aligned4(x, p.x_esz);
  const int nch = live ? row_chunks<T>(p.N) : 0;
  RowChunk<XK> ch;
  float acc = 0.0f;
  for (int c = 0; c < nch; ++c) {
    load_chunk<T, XK>(x, p.x_kind, xvec, p.N, rs.t, c, ch);
    chunk_visit<T>(ch, [&](float v) { acc = __fadd_rn(acc, v); });
  }
  const float s = team_sum<T>(acc, red);
  if (live && rs.t == 0) row_store(p.y, p.y_kind, rs.row * p.ld_y, __fdiv_rn(s, (float)p.N));
}

template <int T, int XK>
static void launch_team_kind(int op, const RowParams& rp, cudaStream_t stream, std::string* why, bi_status* st) {
  constexpr int kBlock = RowSlot<T>::kBlock;
  const int64_t rows_per_block = kBlock / T;
  const int64_t blocks = (rp.R + rows_per_block - 1) / rows_per_block;
  if (blocks > INT32_MAX) {
    *why = "too many rows";
    *st = BI_ERR_INVALID_ARG;
    return;
  }
  const dim3 grid((unsigned)blocks), block(kBlock);
  if (op == kRowRmsNorm)
    rmsnorm_kernel<T, XK><<<grid, block, 0, stream>>>(rp);
  else if (op == kRowLogSoftmax)
    log_softmax_kernel<T, XK><<<grid, block, 0, stream>>>(rp);
  else
    mean_kernel<T, XK><<<grid, block, 0, stream>>>(rp);
  *st = BI_OK;
}

template <int T>
static void launch_team(int op, const RowParams& rp, cudaStream_t stream, std::string* why, bi_status* st) {
  if (rp.x_kind == 2)
    launch_team_kind<T, 2>(op, rp, stream, why, st);
  else
    launch_team_kind<T, 0>(op, rp, stream, why, st);
}

// The team size for rows of N elements: the smallest power of two from 32 to
// 1024 with N <= 32 T.  A function of N only.
int row_team_size(int64_t N) {
  int T = 32;
  while (T < kRowMaxTeam && N > (int64_t)4 * kRowGroups * T) T *= 2;
  return T;
}

bi_status launch_row_reduction(int op, const RowParams& rp, cudaStream_t stream, std::string* why) {
  bi_status st = BI_ERR_INVALID_ARG;
  switch (row_team_size(rp.N)) {
    case 32: launch_team<32>(op, rp, stream, why, &st); break;
    case 64: launch_team<64>(op, rp, stream, why, &st); break;
    case 128: launch_team<128>(op, rp, stream, why, &st); break;
    case 256: launch_team<256>(op, rp, stream, why, &st); break;
    case 512: launch_team<512>(op, rp, stream, why, &st); break;
    default: launch_team<1024>(op, rp, stream, why, &st); break;
  }
  if (st != BI_OK) return st;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("row reduction launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

}  // namespace bi
