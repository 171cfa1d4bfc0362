// bi_rows_rms.cu -- the RMSNorm kernels of the invariant row reductions
// (order and arithmetic: bi_rows.cuh).  Instantiated per team size and input
// type, with the output and weight types fixed at compile time when they
// match the input's (the common case) and read at run time otherwise.
#include "bi_rows.cuh"

namespace bi {

// Teams of fewer than 1024 threads (rows of at most 4096 G elements) stage the
// weight in shared memory as fp32, once per block, while their first chunk of
// x is in flight; longer rows read it from global memory next to the stores.
template <int T, int W>
constexpr bool rms_stages_weight() { return W != kNoWeight && T < 1024; }

// DENSE (teams under 1024 threads, many blocks): registers capped for four
// 256-thread blocks per SM instead of two or three -- more rows in flight and
// a shorter tail when the grid is several waves deep, a slightly longer chain
// per row when it is not.  The arithmetic is the same.
template <int T, int X, int Y, int W, bool DENSE = false>
__global__ void __launch_bounds__(Team<T>::kBlock,
                                  Team<T>::kBlock >= 512 ? 1 : (DENSE ? 1024 : 512) / Team<T>::kBlock)
    rmsnorm_kernel(const RowParams p) {
  constexpr bool kStage = rms_stages_weight<T, W>();
  constexpr int kBlock = Team<T>::kBlock;
  __shared__ float red[kBlock / 32];
  __shared__ float cx[2];
  extern __shared__ float wsm[];  // the weight as fp32 (kStage)
  const RowSlot<T> rs = row_slot<T>(p);
  const int t = rs.t;
  const int64_t row = rs.row;
  const bool live = row < p.R;
  const int64_t r0 = live ? row : 0;
  const void* x = static_cast<const char*>(p.x) + r0 * p.ld_x * Elem<X>::kBytes;
  void* y = static_cast<char*>(p.y) + r0 * p.ld_y * p.y_esz;
  const int N = (int)p.N;
  const bool xvec = aligned4(x, Elem<X>::kBytes);
  const int nch = live ? row_chunks<T, X>(rs.span) : 0;
  int slot = 0;
  const int wk = W == kKindRuntime ? p.w_kind : (W < 0 ? 0 : W);
  const bool wvec = W != kNoWeight && p.w_stride == 1 && aligned4(p.w, wk == 2 ? 4 : 2);
  RowChunk<X> ch;
  if (nch > 0) load_chunk<T, X>(x, xvec, N, rs.span, t, 0, ch);
  if constexpr (kStage) {
    if (wvec) {
#pragma unroll 4
      for (int g = threadIdx.x; g < (N >> 2); g += kBlock) {
        float w4[4];
        load_w4_kind(p, wk, 4 * g, 4, true, w4);
        *reinterpret_cast<float4*>(wsm + 4 * g) = make_float4(w4[0], w4[1], w4[2], w4[3]);
      }
      for (int j = (N & ~3) + threadIdx.x; j < N; j += kBlock) wsm[j] = row_load(p.w, wk, j);
    } else {
#pragma unroll 4
      for (int j = threadIdx.x; j < N; j += kBlock) wsm[j] = row_load(p.w, wk, (int64_t)j * p.w_stride);
    }
    __syncthreads();
  }
  if (T == 32 && !live) return;  // warp teams hold no later block barrier
  float acc = 0.0f;
  for (int c = 0; c < nch; ++c) {
    if (c > 0) load_chunk<T, X>(x, xvec, N, rs.span, t, c, ch);
    chunk_visit<T, X>(ch, N, [&](float v) { acc = __fadd_rn(acc, __fmul_rn(v, v)); });
  }
  float ss = team_sum<T>(acc, red);
  if (T == 1024 && rs.cl > 1) ss = cluster_combine<false>(ss, cx, rs.cl, slot);
  if (!live) return;  // past the team's last barrier
  const float ms = __fdiv_rn(ss, (float)N);
  const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, p.eps)));
  const bool yvec = aligned4(y, p.y_esz);
  constexpr int kWB = 2;  // weight groups loaded together (unstaged weight)
  for (int c = 0; c < nch; ++c) {
    if (nch > 1) load_chunk<T, X>(x, xvec, N, rs.span, t, c, ch);  // one chunk: still in registers
#pragma unroll
    for (int k0 = 0; k0 < RowChunk<X>::G; k0 += kWB) {
      float w[kWB][4];
      if constexpr (W != kNoWeight && !kStage) {
#pragma unroll
        for (int b = 0; b < kWB; ++b) {
          const int n = chunk_n<T, X>(ch, k0 + b, N);
          if (n > 0) load_w4<W>(p, 4 * (ch.g0 + (k0 + b) * T), n, wvec, w[b]);
        }
      }
#pragma unroll
      for (int b = 0; b < kWB; ++b) {
        const int k = k0 + b;
        const int n = chunk_n<T, X>(ch, k, N);
        if (n == 0) continue;
        const int j = 4 * (ch.g0 + k * T);
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = __fmul_rn(word_val<X>(ch.w[k], i), r);
        if constexpr (kStage) {
          if (n == 4) {
            const float4 wv = *reinterpret_cast<const float4*>(wsm + j);
            o[0] = __fmul_rn(o[0], wv.x), o[1] = __fmul_rn(o[1], wv.y);
            o[2] = __fmul_rn(o[2], wv.z), o[3] = __fmul_rn(o[3], wv.w);
          } else {
            for (int i = 0; i < n; ++i) o[i] = __fmul_rn(o[i], wsm[j + i]);
          }
        } else if constexpr (W != kNoWeight) {
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = __fmul_rn(o[i], w[b][i]);
        }
        store4<Y>(p, y, j, yvec, n, o);
      }
    }
  }
  if (T == 1024 && rs.cl > 1) cluster_sync_all();  // no CTA leaves while a peer may read its total
}

template <int T, int X, int Y, int W, bool DENSE = false>
static void launch_rms(const RowParams& rp, dim3 grid, cudaStream_t stream) {
  const size_t smem = rms_stages_weight<T, W>() ? (size_t)rp.N * sizeof(float) : 0;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(reinterpret_cast<const void*>(&rmsnorm_kernel<T, X, Y, W, DENSE>),
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_row_kernel(rmsnorm_kernel<T, X, Y, W, DENSE>, rp, grid, dim3(Team<T>::kBlock), smem, stream);
}

// The dense form exists for the common type combinations: output (and weight,
// if any) of the input's type.
template <int T, int X>
static void launch_rms_x(const RowParams& rp, dim3 grid, bool dense, cudaStream_t stream) {
  constexpr bool kDenseOk = T < 1024;
  if (!rp.w) {
    if (rp.y_kind == X) {
      if (kDenseOk && dense)
        launch_rms<T, X, X, kNoWeight, kDenseOk>(rp, grid, stream);
      else
        launch_rms<T, X, X, kNoWeight>(rp, grid, stream);
    } else {
      launch_rms<T, X, kKindRuntime, kNoWeight>(rp, grid, stream);
    }
  } else if (rp.y_kind == X && rp.w_kind == X) {
    if (kDenseOk && dense)
      launch_rms<T, X, X, X, kDenseOk>(rp, grid, stream);
    else
      launch_rms<T, X, X, X>(rp, grid, stream);
  } else {
    launch_rms<T, X, kKindRuntime, kKindRuntime>(rp, grid, stream);
  }
}

template <int T>
static void launch_rms_t(const RowParams& rp, dim3 grid, bool dense, cudaStream_t stream) {
  if (rp.x_kind == 2)
    launch_rms_x<T, 2>(rp, grid, dense, stream);
  else if (rp.x_kind == 1)
    launch_rms_x<T, 1>(rp, grid, dense, stream);
  else
    launch_rms_x<T, 0>(rp, grid, dense, stream);
}

void launch_rmsnorm_rows(int T, const RowParams& rp, dim3 grid, bool dense, cudaStream_t stream) {
  switch (T) {
    case 32: launch_rms_t<32>(rp, grid, dense, stream); break;
    case 64: launch_rms_t<64>(rp, grid, dense, stream); break;
    case 256: launch_rms_t<256>(rp, grid, dense, stream); break;
    default: launch_rms_t<1024>(rp, grid, false, stream); break;
  }
}

}  // namespace bi
