// bi_rows_lsm.cu -- the log-softmax kernels of the invariant row reductions
// (order and arithmetic: bi_rows.cuh).  Instantiated per team size and input
// type, the output type fixed at compile time when it matches the input's.
#include <map>
#include <mutex>
#include <tuple>

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

// The streaming form of the 1024-thread kernel: each pass loads the thread's
// groups again, kStreamGroups at a time, instead of holding a chunk in
// registers; the CTA's slice of the row (contiguous) is first asked into L2
// by bulk prefetches, so every pass reads it mostly from L2.  The values
// visited and their order are the register-resident kernel's, so the bits are
// the same; holding 4 kStreamGroups values instead of 4 G, a thread fits in 32
// registers and two CTAs share an SM, so twice as many rows' clusters run at
// once.
constexpr int kStreamGroups = 2;
constexpr uint32_t kStreamPrefetchBytes = 16384;  // per prefetch instruction

template <int X, int Y>
__global__ void __launch_bounds__(1024, 2) log_softmax_stream_kernel(const RowParams p) {
  constexpr int T = 1024, G = chunk_groups<X>(), NB = kStreamGroups;
  static_assert(G % NB == 0, "a chunk is a whole number of pieces");
  __shared__ float red[T / 32];
  __shared__ float cx[2];
  const RowSlot<T> rs = row_slot<T>(p);
  const int t = rs.t;
  const int64_t row = rs.row;
  const bool live = row < p.R;
  const int64_t r0 = live ? row : 0;
  const void* x = static_cast<const char*>(p.x) + r0 * p.ld_x * Elem<X>::kBytes;
  const int N = (int)p.N;
  const bool xvec = aligned4(x, Elem<X>::kBytes);
  const int nch = live ? row_chunks<T, X>(rs.span) : 0;
  if (live && t < 32) {
    // The slice's whole 16-byte units, one prefetch of up to 16 KB per lane
    // and round (a hint: no value depends on it).
    const uintptr_t b = reinterpret_cast<uintptr_t>(x) + (uintptr_t)rs.span.gbeg * 4 * Elem<X>::kBytes;
    const uintptr_t e = reinterpret_cast<uintptr_t>(x) +
                        (uintptr_t)min(4 * rs.span.gend, N) * Elem<X>::kBytes;
    const uintptr_t b16 = (b + 15) & ~(uintptr_t)15, e16 = e & ~(uintptr_t)15;
    for (uintptr_t a = b16 + (uintptr_t)t * kStreamPrefetchBytes; a < e16; a += 32 * (uintptr_t)kStreamPrefetchBytes)
      prefetch_l2_bulk(reinterpret_cast<const void*>(a), (uint32_t)min((uintptr_t)kStreamPrefetchBytes, e16 - a));
  }
  int slot = 0;
  // f(piece) over the thread's pieces, chunks then groups ascending.
  auto pieces = [&](auto&& f) {
    for (int c = 0; c < nch; ++c)
#pragma unroll 1
      for (int k0 = 0; k0 < G; k0 += NB) {
        RowChunk<X, NB> pc;
        load_chunk<T, X>(x, xvec, N, rs.span, t, c, pc, k0);
        f(pc);
      }
  };
  float m = -INFINITY;
  pieces([&](const RowChunk<X, NB>& pc) { chunk_visit<T, X>(pc, N, [&](float v) { m = fmaxf(m, v); }); });
  m = team_max<T>(m, red);
  if (rs.cl > 1) m = cluster_combine<true>(m, cx, rs.cl, slot);
  float acc = 0.0f;
  pieces([&](const RowChunk<X, NB>& pc) {
    chunk_visit<T, X>(pc, N, [&](float v) { acc = __fadd_rn(acc, expf(__fsub_rn(v, m))); });
  });
  float se = team_sum<T>(acc, red);
  if (rs.cl > 1) se = cluster_combine<false>(se, cx, rs.cl, slot);
  const float lse = logf(se);
  if (live) {
    void* y = static_cast<char*>(p.y) + r0 * p.ld_y * p.y_esz;
    const bool yvec = aligned4(y, p.y_esz);
    pieces([&](const RowChunk<X, NB>& pc) {
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        const int n = chunk_n<T, X>(pc, k, N);
        if (n == 0) continue;
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = __fsub_rn(__fsub_rn(word_val<X>(pc.w[k], i), m), lse);
        store4<Y>(p, y, 4 * (pc.g0 + k * T), yvec, n, o);
      }
    });
  }
  if (rs.cl > 1) cluster_sync_all();  // no CTA leaves while a peer may read its totals
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

template <int X>
static void launch_lsm_stream_x(const RowParams& rp, dim3 grid, cudaStream_t stream) {
  const dim3 block(1024);
  if (rp.y_kind == X)
    launch_row_kernel(log_softmax_stream_kernel<X, X>, rp, grid, block, 0, stream);
  else
    launch_row_kernel(log_softmax_stream_kernel<X, kKindRuntime>, rp, grid, block, 0, stream);
}

int log_softmax_register_capacity(const RowParams& rp) {
  const void* fn = rp.x_kind == 2   ? (rp.y_kind == 2 ? reinterpret_cast<const void*>(&log_softmax_kernel<1024, 2, 2>)
                                                       : reinterpret_cast<const void*>(&log_softmax_kernel<1024, 2, kKindRuntime>))
                   : rp.x_kind == 1 ? (rp.y_kind == 1 ? reinterpret_cast<const void*>(&log_softmax_kernel<1024, 1, 1>)
                                                       : reinterpret_cast<const void*>(&log_softmax_kernel<1024, 1, kKindRuntime>))
                                    : (rp.y_kind == 0 ? reinterpret_cast<const void*>(&log_softmax_kernel<1024, 0, 0>)
                                                       : reinterpret_cast<const void*>(&log_softmax_kernel<1024, 0, kKindRuntime>));
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  // cached per device, input type, output-type form and cluster size
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int>, int> cache;
  const auto key = std::make_tuple(dev, fn, rp.cl);
  {
    std::lock_guard<std::mutex> lk(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int ctas = 0;
  if (rp.cl > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rp.cl);
    cfg.blockDim = dim3(1024);
    cudaLaunchAttribute attr[1] = {};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)rp.cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) return 0;
    ctas = n * rp.cl;
  } else {
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 1024, 0) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    ctas = per_sm * sms;
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = ctas;
  return ctas;
}

void launch_log_softmax_rows(int T, const RowParams& rp, dim3 grid, bool stream_form, cudaStream_t stream) {
  if (T == 1024 && stream_form) {
    if (rp.x_kind == 2)
      launch_lsm_stream_x<2>(rp, grid, stream);
    else if (rp.x_kind == 1)
      launch_lsm_stream_x<1>(rp, grid, stream);
    else
      launch_lsm_stream_x<0>(rp, grid, stream);
    return;
  }
  switch (T) {
    case 32: launch_lsm_t<32>(rp, grid, stream); break;
    case 64: launch_lsm_t<64>(rp, grid, stream); break;
    case 256: launch_lsm_t<256>(rp, grid, stream); break;
    default: launch_lsm_t<1024>(rp, grid, stream); break;
  }
}

}  // namespace bi
