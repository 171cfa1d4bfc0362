// bi_rows_lsm.cu -- the log-softmax kernels of the invariant row reductions
// (order and arithmetic: bi_rows.cuh).  Instantiated per team size and input
// type, the output type fixed at compile time when it matches the input's.
#include "bi_rows.cuh"

namespace bi {

template <int T, int X, int Y>
__global__ void __launch_bounds__(Team<T>::kBlock, 1024 / Team<T>::kBlock) log_softmax_kernel(const RowParams p) {
  __shared__ float red[Team<T>::kBlock / 32];
  __shared__ float cx[2];
  const RowSlot<T> rs = row_slot<T>(p);
  const int t = rs.t;
  const int64_t row = rs.row;
  const bool live = row < p.R;
  if (T == 32 && !live) return;
  const int64_t r0 = live ? row : 0;
  const void* x = static_cast<const char*>(p.x) + r0 * p.ld_x * Elem<X>::kBytes;
  void* y = static_cast<char*>(p.y) + r0 * p.ld_y * p.y_esz;
  const int N = (int)p.N;
  const bool xvec = aligned4(x, Elem<X>::kBytes);
  const int nch = live ? row_chunks<T, X>(rs.span) : 0;
  int slot = 0;
  RowChunk<X> ch;
  float m = -INFINITY;
  for (int c = 0; c < nch; ++c) {
    load_chunk<T, X>(x, xvec, N, rs.span, t, c, ch);
    chunk_visit<T, X>(ch, N, [&](float v) { m = fmaxf(m, v); });
  }
  m = team_max<T>(m, red);
  if (T == 1024 && rs.cl > 1) m = cluster_combine<true>(m, cx, rs.cl, slot);
  float acc = 0.0f;
  for (int c = 0; c < nch; ++c) {
    if (nch > 1) load_chunk<T, X>(x, xvec, N, rs.span, t, c, ch);
    chunk_visit<T, X>(ch, N, [&](float v) { acc = __fadd_rn(acc, expf(__fsub_rn(v, m))); });
  }
  float se = team_sum<T>(acc, red);
  if (T == 1024 && rs.cl > 1) se = cluster_combine<false>(se, cx, rs.cl, slot);
  const float lse = logf(se);
  if (!live) return;
  const bool yvec = aligned4(y, p.y_esz);
  for (int c = 0; c < nch; ++c) {
    if (nch > 1) load_chunk<T, X>(x, xvec, N, rs.span, t, c, ch);
#pragma unroll
    for (int k = 0; k < RowChunk<X>::G; ++k) {
      const int n = chunk_n<T, X>(ch, k, N);
      if (n == 0) continue;
      float o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = __fsub_rn(__fsub_rn(word_val<X>(ch.w[k], i), m), lse);
      store4<Y>(p, y, 4 * (ch.g0 + k * T), yvec, n, o);
    }
  }
  if (T == 1024 && rs.cl > 1) cluster_sync_all();  // no CTA leaves while a peer may read its totals
}

template <int T, int X>
static void launch_lsm_x(const RowParams& rp, dim3 grid, cudaStream_t stream) {
  const dim3 block(Team<T>::kBlock);
  if (rp.y_kind == X)
    launch_row_kernel(log_softmax_kernel<T, X, X>, rp, grid, block, 0, stream);
  else
    launch_row_kernel(log_softmax_kernel<T, X, kKindRuntime>, rp, grid, block, 0, stream);
}

template <int T>
static void launch_lsm_t(const RowParams& rp, dim3 grid, cudaStream_t stream) {
  if (rp.x_kind == 2)
    launch_lsm_x<T, 2>(rp, grid, stream);
  else if (rp.x_kind == 1)
    launch_lsm_x<T, 1>(rp, grid, stream);
  else
    launch_lsm_x<T, 0>(rp, grid, stream);
}

void launch_log_softmax_rows(int T, const RowParams& rp, dim3 grid, cudaStream_t stream) {
  switch (T) {
    case 32: launch_lsm_t<32>(rp, grid, stream); break;
    case 64: launch_lsm_t<64>(rp, grid, stream); break;
    case 256: launch_lsm_t<256>(rp, grid, stream); break;
    default: launch_lsm_t<1024>(rp, grid, stream); break;
  }
}

}  // namespace bi
