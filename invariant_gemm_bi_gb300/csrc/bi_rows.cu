// bi_rows.cu -- the row-mean kernels and the dispatcher of the invariant row
// reductions (RMSNorm: bi_rows_rms.cu, log-softmax: bi_rows_lsm.cu; order
// and arithmetic: bi_rows.cuh).
#include "bi_rows.cuh"

namespace bi {

int row_team_size(int64_t N, int x_kind) {
  const int64_t g = x_kind == 2 ? 8 : 16;
  for (int T : {32, 64, 256}) if (N <= 4 * g * T) return T;
  return 1024;
}

int row_cluster_size(int64_t N, int x_kind) {
  const int64_t per = (x_kind == 2 ? 8 : 16) * 4 * 1024;  // elements one 1024-thread CTA holds
  return (int)std::min<int64_t>(8, std::max<int64_t>(1, (N + per - 1) / per));
}

template <int T, int X>
__global__ void __launch_bounds__(Team<T>::kBlock, 1024 / Team<T>::kBlock) mean_kernel(const RowParams p) {
  __shared__ float red[Team<T>::kBlock / 32];
  __shared__ float cx[2];
  const RowSlot<T> rs = row_slot<T>(p);
  const int t = rs.t;
  const int64_t row = rs.row;
  const bool live = row < p.R;
  if (T == 32 && !live) return;
  const int64_t r0 = live ? row : 0;
  const void* x = static_cast<const char*>(p.x) + r0 * p.ld_x * Elem<X>::kBytes;
  const int N = (int)p.N;
  const bool xvec = aligned4(x, Elem<X>::kBytes);
  const int nch = live ? row_chunks<T, X>(rs.span) : 0;
  int slot = 0;
  RowChunk<X> ch;
  float acc = 0.0f;
  for (int c = 0; c < nch; ++c) {
    load_chunk<T, X>(x, xvec, N, rs.span, t, c, ch);
    chunk_visit<T, X>(ch, N, [&](float v) { acc = __fadd_rn(acc, v); });
  }
  float s = team_sum<T>(acc, red);
  if (T == 1024 && rs.cl > 1) {
    s = cluster_combine<false>(s, cx, rs.cl, slot);
    cluster_sync_all();  // no CTA leaves while a peer may read its total
  }
  if (live && t == 0 && (T < 1024 || blockIdx.x % rs.cl == 0)) {
    const float v = __fdiv_rn(s, (float)N);
    if (p.y_kind == 2)
      reinterpret_cast<float*>(p.y)[row * p.ld_y] = v;
    else if (p.y_kind == 1)
      reinterpret_cast<__half*>(p.y)[row * p.ld_y] = __float2half_rn(v);
    else
      reinterpret_cast<__nv_bfloat16*>(p.y)[row * p.ld_y] = __float2bfloat16_rn(v);
  }
}

template <int T>
static void launch_mean_t(const RowParams& rp, dim3 grid, cudaStream_t stream) {
  const dim3 block(Team<T>::kBlock);
  if (rp.x_kind == 2)
    launch_row_kernel(mean_kernel<T, 2>, rp, grid, block, 0, stream);
  else if (rp.x_kind == 1)
    launch_row_kernel(mean_kernel<T, 1>, rp, grid, block, 0, stream);
  else
    launch_row_kernel(mean_kernel<T, 0>, rp, grid, block, 0, stream);
}

template <int T>
static dim3 row_grid(const RowParams& rp, bool* ok) {
  const int64_t blocks = (rp.R + Team<T>::kRows - 1) / Team<T>::kRows * rp.cl;
  *ok = blocks <= INT32_MAX;
  return dim3((unsigned)(*ok ? blocks : 1));
}

bi_status launch_row_reduction(int op, const RowParams& rp_in, cudaStream_t stream, std::string* why) {
  RowParams rp = rp_in;
  const int T = row_team_size(rp.N, rp.x_kind);
  rp.cl = T == 1024 ? row_cluster_size(rp.N, rp.x_kind) : 1;
  bool ok = true;
  const dim3 grid = T == 32 ? row_grid<32>(rp, &ok)
                  : T == 64 ? row_grid<64>(rp, &ok)
                  : T == 256 ? row_grid<256>(rp, &ok)
                             : row_grid<1024>(rp, &ok);
  if (!ok) {
    *why = "too many rows";
    return BI_ERR_INVALID_ARG;
  }
  if (op == kRowRmsNorm) {
    // More than four blocks per SM: the register-capped form (four resident
    // blocks per SM instead of two or three; the same bits).
    bool dense = false;
    if (T < 1024) {
      DeviceInfo dev;
      const bi_status st = current_device_info(&dev, why);
      if (st != BI_OK) return st;
      dense = (int64_t)grid.x > 4 * (int64_t)dev.num_sms;
    }
    launch_rmsnorm_rows(T, rp, grid, dense, stream);
  } else if (op == kRowLogSoftmax) {
    // 1024-thread teams hold a chunk in registers, one CTA per SM (and a
    // cluster's CTAs within one GPC): when the rows' clusters need more than
    // one wave of that kernel, the streaming form (two CTAs per SM, the same
    // bits) runs them instead.
    const bool stream_form = T == 1024 && (int64_t)grid.x > log_softmax_register_capacity(rp);
    launch_log_softmax_rows(T, rp, grid, stream_form, stream);
  } else {
    switch (T) {
      case 32: launch_mean_t<32>(rp, grid, stream); break;
      case 64: launch_mean_t<64>(rp, grid, stream); break;
      case 256: launch_mean_t<256>(rp, grid, stream); break;
      default: launch_mean_t<1024>(rp, grid, stream); break;
    }
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("row reduction launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

}  // namespace bi
