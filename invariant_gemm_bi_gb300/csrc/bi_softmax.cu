// bi_softmax.cu -- row softmax over the last dimension, plus two small helper
// kernels (the empty-reduction fill and the bounded-wait test hook).
//
// Softmax: one warp owns one row ("ai-infra handbook: deterministic
// inference", section on normalisation and softmax: each row is reduced by
// one block in a fixed order, never split across blocks because there are few
// rows).  Lane t takes elements t, t+32, t+64, ... in ascending order; the 32
// lane partials are combined by a fixed xor-butterfly, which gives every lane
// the same bits (fp32 addition is commutative).  The order depends only on the
// element index, never on the number of rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "bi_common.h"
#include "bi_launch.h"
#include "bi_ptx.cuh"

namespace bi {

constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxRegCols = 32;  // rows up to 32*32 = 1024 columns stay in registers

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

__device__ __forceinline__ void store_prob(const SoftmaxParams& p, int64_t row, int64_t j, float v) {
  if (p.out_f32)
    reinterpret_cast<float*>(p.p)[row * p.ld_p + j] = v;
  else
    reinterpret_cast<__nv_bfloat16*>(p.p)[row * p.ld_p + j] = __float2bfloat16_rn(v);
}

// N <= 32 * kSoftmaxRegCols: the row is read once and kept in registers.
__global__ void __launch_bounds__(kSoftmaxWarps * 32) softmax_reg_kernel(const SoftmaxParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kSoftmaxWarps + (threadIdx.x >> 5);
  if (row >= p.R) return;
  const float* s = p.s + row * p.ld_s;
  const int N = (int)p.N;
  float v[kSoftmaxRegCols];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kSoftmaxRegCols; ++i) {
    const int j = lane + 32 * i;
    v[i] = j < N ? __ldg(s + j) : -INFINITY;
    mx = fmaxf(mx, v[i]);
  }
  mx = warp_max(mx);
  float sum = 0.0f;
#pragma unroll
  for (int i = 0; i < kSoftmaxRegCols; ++i) {
    const int j = lane + 32 * i;
    if (j < N) {
      v[i] = expf(__fsub_rn(v[i], mx));
      sum = __fadd_rn(sum, v[i]);
    }
  }
  sum = warp_sum(sum);
#pragma unroll
  for (int i = 0; i < kSoftmaxRegCols; ++i) {
    const int j = lane + 32 * i;
    if (j < N) store_prob(p, row, j, __fdiv_rn(v[i], sum));
  }
}

// Any N: the same arithmetic in the same order, re-reading the row.
__global__ void __launch_bounds__(kSoftmaxWarps * 32) softmax_loop_kernel(const SoftmaxParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kSoftmaxWarps + (threadIdx.x >> 5);
  if (row >= p.R) return;
  const float* s = p.s + row * p.ld_s;
  float mx = -INFINITY;
  for (int64_t j = lane; j < p.N; j += 32) mx = fmaxf(mx, __ldg(s + j));
  mx = warp_max(mx);
  float sum = 0.0f;
  for (int64_t j = lane; j < p.N; j += 32) sum = __fadd_rn(sum, expf(__fsub_rn(__ldg(s + j), mx)));
  sum = warp_sum(sum);
  for (int64_t j = lane; j < p.N; j += 32)
    store_prob(p, row, j, __fdiv_rn(expf(__fsub_rn(__ldg(s + j), mx)), sum));
}

bi_status launch_softmax(const SoftmaxParams& sp, cudaStream_t stream, std::string* why) {
  const int64_t blocks = (sp.R + kSoftmaxWarps - 1) / kSoftmaxWarps;
  if (blocks > INT32_MAX) {
    *why = "too many rows";
    return BI_ERR_INVALID_ARG;
  }
  if (sp.N <= 32 * kSoftmaxRegCols)
    softmax_reg_kernel<<<(unsigned)blocks, kSoftmaxWarps * 32, 0, stream>>>(sp);
  else
    softmax_loop_kernel<<<(unsigned)blocks, kSoftmaxWarps * 32, 0, stream>>>(sp);
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
    const int64_t off = l * g.c_batch + m * g.ldc + n;
    if (g.out_f32)
      reinterpret_cast<float*>(g.c)[off] = v;
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
