// bi_softmax.cu -- row softmax over the last dimension, plus two small helper
// kernels (the empty-reduction fill and the bounded-wait test hook).
//
// Softmax: one warp owns one row ("ai-infra handbook: deterministic
// inference", section on normalisation and softmax: each row is reduced by
// one block in a fixed order, never split across blocks because there are few
// rows).  The row is cut into groups of 4 consecutive elements; lane t owns
// groups t, t+32, t+64, ... and sums its elements in ascending index order;
// the 32 lane partials are combined by a fixed xor-butterfly, which gives
// every lane the same bits (fp32 addition is commutative).  The order depends
// only on the element index, never on the number of rows or on alignment.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "bi_common.h"
#include "bi_launch.h"
#include "bi_ptx.cuh"

namespace bi {

constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxRegGroups = 8;  // rows up to 32*8*4 = 1024 columns stay in registers

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Group g of a row: elements 4g .. 4g+3 (those below N); absent ones read -inf.
template <bool VEC>
__device__ __forceinline__ float4 load_group(const float* s, int64_t g, int64_t N) {
  const int64_t j = 4 * g;
  if (VEC && j + 4 <= N) return __ldg(reinterpret_cast<const float4*>(s + j));
  float4 v;
  v.x = j + 0 < N ? __ldg(s + j + 0) : -INFINITY;
  v.y = j + 1 < N ? __ldg(s + j + 1) : -INFINITY;
  v.z = j + 2 < N ? __ldg(s + j + 2) : -INFINITY;
  v.w = j + 3 < N ? __ldg(s + j + 3) : -INFINITY;
  return v;
}

template <bool VEC>
__device__ __forceinline__ void store_group(const SoftmaxParams& p, int64_t row, int64_t g, float4 v) {
  const int64_t j = 4 * g;
  if (p.out_f32) {
    float* dst = reinterpret_cast<float*>(p.p) + row * p.ld_p + j;
    if (VEC && j + 4 <= p.N) {
      *reinterpret_cast<float4*>(dst) = v;
    } else {
      const float f[4] = {v.x, v.y, v.z, v.w};
      for (int i = 0; i < 4 && j + i < p.N; ++i) dst[i] = f[i];
    }
  } else {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.p) + row * p.ld_p + j;
    if (VEC && j + 4 <= p.N) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    } else {
      const float f[4] = {v.x, v.y, v.z, v.w};
      for (int i = 0; i < 4 && j + i < p.N; ++i) dst[i] = __float2bfloat16_rn(f[i]);
    }
  }
}

__device__ __forceinline__ float group_max(float4 v) { return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)); }

// e = exp(v - mx) for the present elements (absent -inf -> 0 and not added);
// partial sum += e in ascending element order.
__device__ __forceinline__ float4 group_exp_sum(float4 v, float mx, int64_t j, int64_t N, float& sum) {
  float4 e;
  if (j + 4 <= N) {  // whole group: same operations without the bounds tests
    e.x = expf(__fsub_rn(v.x, mx));
    e.y = expf(__fsub_rn(v.y, mx));
    e.z = expf(__fsub_rn(v.z, mx));
    e.w = expf(__fsub_rn(v.w, mx));
    sum = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(sum, e.x), e.y), e.z), e.w);
    return e;
  }
  e.x = j + 0 < N ? expf(__fsub_rn(v.x, mx)) : 0.0f;
  e.y = j + 1 < N ? expf(__fsub_rn(v.y, mx)) : 0.0f;
  e.z = j + 2 < N ? expf(__fsub_rn(v.z, mx)) : 0.0f;
  e.w = j + 3 < N ? expf(__fsub_rn(v.w, mx)) : 0.0f;
  if (j + 0 < N) sum = __fadd_rn(sum, e.x);
  if (j + 1 < N) sum = __fadd_rn(sum, e.y);
  if (j + 2 < N) sum = __fadd_rn(sum, e.z);
  if (j + 3 < N) sum = __fadd_rn(sum, e.w);
  return e;
}

// p = e * RN(1 / sum): one correctly rounded reciprocal per row, one
// multiply per element.
__device__ __forceinline__ float4 group_scale(float4 e, float rinv) {
  return make_float4(__fmul_rn(e.x, rinv), __fmul_rn(e.y, rinv), __fmul_rn(e.z, rinv),
                     __fmul_rn(e.w, rinv));
}

// N <= 32 * 4 * kSoftmaxRegGroups: the row is read once and kept in registers.
template <bool VEC>
__global__ void __launch_bounds__(kSoftmaxWarps * 32) softmax_reg_kernel(const SoftmaxParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kSoftmaxWarps + (threadIdx.x >> 5);
  if (row >= p.R) return;
  const float* s = p.s + row * p.ld_s;
  const int64_t groups = (p.N + 3) / 4;
  float4 v[kSoftmaxRegGroups];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kSoftmaxRegGroups; ++i) {
    const int64_t g = lane + 32 * i;
    v[i] = g < groups ? load_group<VEC>(s, g, p.N) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
#pragma unroll
  for (int i = 0; i < kSoftmaxRegGroups; ++i) mx = fmaxf(mx, group_max(v[i]));
  mx = warp_max(mx);
  float sum = 0.0f;
#pragma unroll
  for (int i = 0; i < kSoftmaxRegGroups; ++i) {
    const int64_t g = lane + 32 * i;
    if (g < groups) v[i] = group_exp_sum(v[i], mx, 4 * g, p.N, sum);
  }
  sum = warp_sum(sum);
  const float rinv = __frcp_rn(sum);
#pragma unroll
  for (int i = 0; i < kSoftmaxRegGroups; ++i) {
    const int64_t g = lane + 32 * i;
    if (g < groups) store_group<VEC>(p, row, g, group_scale(v[i], rinv));
  }
}

// Any N: the same arithmetic in the same order, re-reading the row.
template <bool VEC>
__global__ void __launch_bounds__(kSoftmaxWarps * 32) softmax_loop_kernel(const SoftmaxParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kSoftmaxWarps + (threadIdx.x >> 5);
  if (row >= p.R) return;
  const float* s = p.s + row * p.ld_s;
  const int64_t groups = (p.N + 3) / 4;
  float mx = -INFINITY;
  for (int64_t g = lane; g < groups; g += 32) mx = fmaxf(mx, group_max(load_group<VEC>(s, g, p.N)));
  mx = warp_max(mx);
  float sum = 0.0f;
  for (int64_t g = lane; g < groups; g += 32) group_exp_sum(load_group<VEC>(s, g, p.N), mx, 4 * g, p.N, sum);
  sum = warp_sum(sum);
  const float rinv = __frcp_rn(sum);
  for (int64_t g = lane; g < groups; g += 32) {
    float dummy = 0.0f;
    const float4 e = group_exp_sum(load_group<VEC>(s, g, p.N), mx, 4 * g, p.N, dummy);
    store_group<VEC>(p, row, g, group_scale(e, rinv));
  }
}

bi_status launch_softmax(const SoftmaxParams& sp, cudaStream_t stream, std::string* why) {
  const int64_t blocks = (sp.R + kSoftmaxWarps - 1) / kSoftmaxWarps;
  if (blocks > INT32_MAX) {
    *why = "too many rows";
    return BI_ERR_INVALID_ARG;
  }
  // 16-byte loads / 8- or 16-byte stores when every row start is aligned.
  const int esz = sp.out_f32 ? 4 : 2;
  const bool vec = reinterpret_cast<uintptr_t>(sp.s) % 16 == 0 && (sp.ld_s * 4) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(sp.p) % (4 * esz) == 0 && (sp.ld_p * esz) % (4 * esz) == 0;
  const dim3 grid((unsigned)blocks), block(kSoftmaxWarps * 32);
  if (sp.N <= 32 * 4 * kSoftmaxRegGroups) {
    if (vec)
      softmax_reg_kernel<true><<<grid, block, 0, stream>>>(sp);
    else
      softmax_reg_kernel<false><<<grid, block, 0, stream>>>(sp);
  } else {
    if (vec)
      softmax_loop_kernel<true><<<grid, block, 0, stream>>>(sp);
    else
      softmax_loop_kernel<false><<<grid, block, 0, stream>>>(sp);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("softmax launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

// ---------------------------------------------------------------------------
// K == 0: the reduction is empty, so c = round(alpha * 0 + bias).
// ---------------------------------------------------------------------------
__global__ void fill_bias_kernel(const GemmProblem g) {
  const int64_t total = g.L * g.M * g.N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i % g.N;
    const int64_t m = (i / g.N) % g.M;
    const int64_t l = i / (g.N * g.M);
    float v = __fmul_rn(0.0f, g.alpha);
    if (g.bias_kind == 1)
      v = __fadd_rn(v, __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(g.bias)[n * g.bias_stride]));
    else if (g.bias_kind == 2)
      v = __fadd_rn(v, reinterpret_cast<const float*>(g.bias)[n * g.bias_stride]);
    else if (g.bias_kind == 3)
      v = __fadd_rn(v, __half2float(reinterpret_cast<const __half*>(g.bias)[n * g.bias_stride]));
    const int64_t off = l * g.c_batch + m * g.ldc + n;
    if (g.out_f32)
      reinterpret_cast<float*>(g.c)[off] = v;
    else if (g.out_f16)
      reinterpret_cast<__half*>(g.c)[off] = __float2half_rn(v);
    else
      reinterpret_cast<__nv_bfloat16*>(g.c)[off] = __float2bfloat16_rn(v);
  }
}

bi_status launch_fill_bias(const GemmProblem& g, cudaStream_t stream, std::string* why) {
  const int64_t total = g.L * g.M * g.N;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 65536);
  fill_bias_kernel<<<(unsigned)blocks, 256, 0, stream>>>(g);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("fill launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

// ---------------------------------------------------------------------------
// Test hook: a bounded wait on an mbarrier that nothing signals.
// ---------------------------------------------------------------------------
__global__ void debug_wait_kernel(unsigned int* status_word, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, status_word, limit_ns,
                      status_code(6, kSiteDebugWait));
  __syncthreads();
}

bi_status launch_debug_wait(uint64_t limit_ns, cudaStream_t stream, std::string* why) {
  DeviceInfo dev;
  bi_status st = current_device_info(&dev, why);
  if (st != BI_OK) return st;
  debug_wait_kernel<<<1, 32, 0, stream>>>(dev.status_word, limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("debug wait launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

}  // namespace bi
