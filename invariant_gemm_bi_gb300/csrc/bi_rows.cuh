// bi_rows.cuh -- invariant row reductions over the last dimension: RMSNorm,
// log-softmax and the row mean ("Unmasking the True Culprit: Why
// Temperature=0 Doesn't Mean Deterministic LLM Inference", section "Beyond
// Matrix Multiplication: Other Critical Operations"; aten::mean.dim in
// "Batch-Invariant VLAs"; "ai-infra handbook: deterministic inference", on
// normalisation, softmax and means: one block reduces one row in a fixed
// order, never splitting a row because there are few rows).
//
// A row of N elements is reduced by a team of T threads, T fixed by N and the
// input type alone: the first of 32, 64, 256, 1024 threads with N <= 4 G T,
// G = 16 groups for 16-bit inputs and 8 for fp32, so a thread holds at most G
// groups of 4 elements (32 registers of data) unless the row is longer than
// 4096 G elements -- then each of the 1024 threads walks several chunks of G
// groups.  Teams smaller than 256 threads share a 256-thread block.  Rows
// longer than 4096 G elements are split, by N alone, over a cluster of
// cl = ceil(N / 4096 G) <= 8 CTAs of 1024 threads: CTA r takes the r-th of
// cl equal contiguous slices of the row's groups.  The row (or each CTA's
// slice) is cut into groups of 4 consecutive elements; thread t owns groups
// t, t+T, t+2T, ... of it and accumulates their elements in
// ascending index order in fp32; each warp combines its 32 partials by a fixed
// xor butterfly, a team of several warps adds the warp partials in warp
// order, and a cluster adds its CTAs' totals in rank order (read by every
// CTA through distributed shared memory).  The order depends only on N, the input type and the element index
// -- not on the number of rows, on the row's address (aligned rows are loaded
// 4 elements at a time, others one at a time, with the same arithmetic) or on
// which SM runs it.  A thread loads a chunk of G groups, all before using any,
// and keeps them in registers: a row of up to 4096 G elements is read from
// memory once, longer rows once per pass.
//
//   RMSNorm      ss = sum x_j^2;  ms = RN(ss / N);  r = RN(1 / RN(sqrt(ms + eps)))
//                y_j = RN(RN(x_j * r) * w_j)           (w absent: y_j = RN(x_j * r))
//   log-softmax  m = max x_j;  se = sum expf(x_j - m);  lse = logf(se)
//                y_j = RN(RN(x_j - m) - lse)
//   mean         y = RN(sum x_j / N)
// with every add / multiply / divide / square root a separately rounded fp32
// operation, then one rounding to the output type.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "bi_common.h"
#include "bi_launch.h"
#include "bi_ptx_ext.cuh"

namespace bi {

// Team sizes (threads reducing one row) and the team for a row of N elements
// of type x_kind -- a function of N and the type only: the first of 32, 64,
// 256, 1024 threads with N <= 4 G T (G groups per thread).
int row_team_size(int64_t N, int x_kind);

// Groups of 4 a thread loads together (one chunk): 32 registers of data.
template <int X>
constexpr int chunk_groups() { return X == 2 ? 8 : 16; }

template <int T>
struct Team {
  static constexpr int kBlock = T < 256 ? 256 : T;  // threads per block
  static constexpr int kRows = kBlock / T;          // rows per block
};

// Element types: 0 bf16, 1 fp16, 2 fp32.
template <int K>
struct Elem {
  static constexpr int kBytes = K == 2 ? 4 : 2;
  static constexpr int kWords = K == 2 ? 4 : 2;  // 32-bit words per group of 4
};

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
// holds block barriers); a team's warps are contiguous in the block.
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

__device__ __forceinline__ float half_bits_to_float(uint32_t h, int kind) {
  return kind == 1 ? __half2float(__ushort_as_half((unsigned short)h))
                   : __uint_as_float(h << 16);  // bf16 -> fp32 is exact: the bits move up
}

// Element i (0..3) of a group held as raw words.
template <int K>
__device__ __forceinline__ float word_val(const uint32_t (&w)[Elem<K>::kWords], int i) {
  if constexpr (K == 2) {
    return __uint_as_float(w[i]);
  } else {
    const uint32_t h = (w[i >> 1] >> (16 * (i & 1))) & 0xffffu;
    return half_bits_to_float(h, K);
  }
}

// Element j of a row of runtime type `kind` as fp32 (exact).
__device__ __forceinline__ float row_load(const void* base, int kind, int64_t j) {
  if (kind == 2) return __ldg(reinterpret_cast<const float*>(base) + j);
  return half_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(base) + j), kind);
}

__device__ __forceinline__ bool aligned4(const void* p, int esz) {
  return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)(4 * esz)) == 0;
}

// The groups [gbeg, gend) of a row that one CTA reduces: the whole row, or
// for a cluster of cl CTAs the rank-th of cl equal contiguous slices.
struct RowSpan {
  int gbeg, gend;
};
__device__ __forceinline__ RowSpan row_span(int N, int cl, int rank) {
  const int ng = (N + 3) >> 2;
  const int per = (ng + cl - 1) / cl;
  const int b = min(ng, rank * per);
  return {b, min(ng, b + per)};
}

// One chunk of a thread's groups: chunk c holds its groups g0 + k T,
// k = 0..G-1, g0 = gbeg + GcT + t, as raw words (zeros past the end of the
// span).  All loads are issued before any value is used.  `full`: all G
// groups lie inside the span and the row and were loaded as vectors (no
// per-element checks needed).  A piece (GN < G) holds GN consecutive groups
// k0 .. k0 + GN - 1 of a chunk, with g0 its first.
template <int X, int GN = chunk_groups<X>()>
struct RowChunk {
  static constexpr int G = GN;
  uint32_t w[G][Elem<X>::kWords];
  int g0, gend;
  bool full;
};

// Elements of group g of the row that the span holds (0 outside it).
__device__ __forceinline__ int group_n(int g, int gend, int N) {
  const int nfull = N >> 2;
  return g >= gend ? 0 : (g < nfull ? 4 : (g == nfull ? (N & 3) : 0));
}

template <int T, int X, int GN>
__device__ __forceinline__ void load_chunk(const void* x, bool vec, int N, const RowSpan& sp, int t, int c,
                                           RowChunk<X, GN>& ch, int k0 = 0) {
  constexpr int W = Elem<X>::kWords;
  constexpr int G = GN;
  ch.g0 = sp.gbeg + (c * chunk_groups<X>() + k0) * T + t;
  ch.gend = sp.gend;
  ch.full = vec && ch.g0 + (G - 1) * T < min(N >> 2, sp.gend);
  if (ch.full) {
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const int g = ch.g0 + k * T;
      if constexpr (W == 4) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(x) + g);
        ch.w[k][0] = q.x, ch.w[k][1] = q.y, ch.w[k][2] = q.z, ch.w[k][3] = q.w;
      } else {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(x) + g);
        ch.w[k][0] = q.x, ch.w[k][1] = q.y;
      }
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int g = ch.g0 + k * T;
    const int n = group_n(g, sp.gend, N);
    if (n == 4 && vec) {
      if constexpr (W == 4) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(x) + g);
        ch.w[k][0] = q.x, ch.w[k][1] = q.y, ch.w[k][2] = q.z, ch.w[k][3] = q.w;
      } else {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(x) + g);
        ch.w[k][0] = q.x, ch.w[k][1] = q.y;
      }
    } else if constexpr (W == 4) {
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

// Elements of group k of the chunk that lie inside the span (0 past its end).
template <int T, int X, int GN>
__device__ __forceinline__ int chunk_n(const RowChunk<X, GN>& ch, int k, int N) {
  return ch.full ? 4 : group_n(ch.g0 + k * T, ch.gend, N);
}

// f(value) over the chunk's elements, groups then elements ascending.
template <int T, int X, int GN, typename F>
__device__ __forceinline__ void chunk_visit(const RowChunk<X, GN>& ch, int N, F&& f) {
  if (ch.full) {
#pragma unroll
    for (int k = 0; k < GN; ++k)
#pragma unroll
      for (int i = 0; i < 4; ++i) f(word_val<X>(ch.w[k], i));
  } else {
#pragma unroll
    for (int k = 0; k < GN; ++k) {
      const int n = chunk_n<T, X>(ch, k, N);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (i < n) f(word_val<X>(ch.w[k], i));
    }
  }
}

// Chunks a thread of a T-team walks over a span.
template <int T, int X>
__device__ __forceinline__ int row_chunks(const RowSpan& sp) {
  constexpr int G = RowChunk<X>::G;
  const int groups = sp.gend - sp.gbeg;
  return groups <= 0 ? 0 : (groups + T * G - 1) / (T * G);
}

// Where a thread's team works: its row, its index in the team and the span of
// the row its CTA reduces (T == 1024 with p.cl > 1: one row per cluster).
template <int T>
struct RowSlot {
  int64_t row;
  int t;
  int cl;
  RowSpan span;
};
template <int T>
__device__ __forceinline__ RowSlot<T> row_slot(const RowParams& p) {
  RowSlot<T> s;
  if constexpr (T == 1024) {
    s.cl = p.cl;
    s.row = blockIdx.x / s.cl;
    s.t = threadIdx.x;
    s.span = row_span((int)p.N, s.cl, (int)(blockIdx.x % s.cl));
  } else {
    s.cl = 1;
    s.row = (int64_t)blockIdx.x * Team<T>::kRows + threadIdx.x / T;
    s.t = threadIdx.x % T;
    s.span = row_span((int)p.N, 1, 0);
  }
  return s;
}

// The CTA's total v (the same in every thread) combined over the row's
// cluster of cl CTAs: each CTA publishes it, the cluster meets at a barrier,
// and every thread reads the totals of CTAs 0 .. cl-1 in rank order.  cx: two
// slots, used alternately (a slot is rewritten only after the next barrier,
// which every reader of it has passed).
template <bool MAX>
__device__ __forceinline__ float cluster_combine(float v, float* cx, int cl, int& slot) {
  if (threadIdx.x == 0) cx[slot] = v;
  cluster_sync_all();
  const uint32_t a = smem_u32(cx + slot);
  float s = ld_shared_cluster_f32(cluster_map_shared(a, 0));
  for (int r = 1; r < cl; ++r) {
    const float o = ld_shared_cluster_f32(cluster_map_shared(a, (uint32_t)r));
    s = MAX ? fmaxf(s, o) : __fadd_rn(s, o);
  }
  slot ^= 1;
  return s;
}

// Stores the n (<= 4) values of the group starting at element j of a row of
// type Y (0 bf16, 1 fp16, 2 fp32); vec: the row starts on a 4-element boundary.
__device__ __forceinline__ void store4_kind(void* y, int Y, int j, bool vec, int n, const float (&o)[4]) {
  if (vec && n == 4) {
    if (Y == 2) {
      reinterpret_cast<float4*>(y)[j >> 2] = make_float4(o[0], o[1], o[2], o[3]);
    } else if (Y == 1) {
      const __half2 a = __floats2half2_rn(o[0], o[1]), b = __floats2half2_rn(o[2], o[3]);
      reinterpret_cast<uint2*>(y)[j >> 2] =
          make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    } else {
      const __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]), b = __floats2bfloat162_rn(o[2], o[3]);
      reinterpret_cast<uint2*>(y)[j >> 2] =
          make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    }
    return;
  }
  for (int i = 0; i < n; ++i) {
    if (Y == 2)
      reinterpret_cast<float*>(y)[j + i] = o[i];
    else if (Y == 1)
      reinterpret_cast<__half*>(y)[j + i] = __float2half_rn(o[i]);
    else
      reinterpret_cast<__nv_bfloat16*>(y)[j + i] = __float2bfloat16_rn(o[i]);
  }
}

// The RMSNorm weight values w[j .. j+3] (type wk, n of them, zeros after).
__device__ __forceinline__ void load_w4_kind(const RowParams& p, int wk, int j, int n, bool wvec, float (&w)[4]) {
  if (wvec && n == 4) {
    if (wk == 2) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(p.w) + (j >> 2));
      w[0] = q.x, w[1] = q.y, w[2] = q.z, w[3] = q.w;
    } else {
      const uint2 q = __ldg(reinterpret_cast<const uint2*>(p.w) + (j >> 2));
      w[0] = half_bits_to_float(q.x & 0xffffu, wk), w[1] = half_bits_to_float(q.x >> 16, wk);
      w[2] = half_bits_to_float(q.y & 0xffffu, wk), w[3] = half_bits_to_float(q.y >> 16, wk);
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = i < n ? row_load(p.w, wk, (int64_t)(j + i) * p.w_stride) : 0.0f;
}

// Type parameters of the kernels: a kind code (0 bf16, 1 fp16, 2 fp32) fixed
// at compile time, or read from the parameters at run time, or no weight.
constexpr int kKindRuntime = -1;
constexpr int kNoWeight = -2;

template <int Y>
__device__ __forceinline__ void store4(const RowParams& p, void* y, int j, bool vec, int n, const float (&o)[4]) {
  store4_kind(y, Y == kKindRuntime ? p.y_kind : Y, j, vec, n, o);
}
template <int W>
__device__ __forceinline__ void load_w4(const RowParams& p, int j, int n, bool wvec, float (&w)[4]) {
  load_w4_kind(p, W == kKindRuntime ? p.w_kind : W, j, n, wvec, w);
}

// Launches a row kernel, as clusters of rp.cl CTAs when rp.cl > 1 (a launch
// error is left for the caller's cudaGetLastError).
template <typename K>
inline void launch_row_kernel(K kernel, const RowParams& rp, dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream) {
  if (rp.cl > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)rp.cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, rp);
  } else {
    kernel<<<grid, block, smem, stream>>>(rp);
  }
}

// CTAs per row: 1, or for rows longer than 4096 G elements ceil(N / 4096 G),
// at most 8 -- a function of N and the input type only.
int row_cluster_size(int64_t N, int x_kind);

// Launchers of the three operations for team size T (bi_rows_rms.cu,
// bi_rows_lsm.cu, bi_rows.cu); grid: one block per Team<T>::kRows rows.
// dense: the RMSNorm kernels' register-capped form (teams under 1024 threads,
// the common type combinations; the same bits).
void launch_rmsnorm_rows(int T, const RowParams& rp, dim3 grid, bool dense, cudaStream_t stream);
// CTAs of the register-resident 1024-thread log-softmax kernel (for rp's
// types and cluster size) that run at once on the current device; 0 if the
// occupancy query fails.
int log_softmax_register_capacity(const RowParams& rp);
// stream_form: the log-softmax's streaming form (1024-thread teams only; the
// same bits as the register-resident form).
void launch_log_softmax_rows(int T, const RowParams& rp, dim3 grid, bool stream_form, cudaStream_t stream);

}  // namespace bi
