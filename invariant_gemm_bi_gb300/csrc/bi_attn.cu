// bi_attn.cu -- fused attention o = softmax(scale * q k^T) v per head, in one
// kernel, with a reduction order that no batch shape can change ("ai-infra
// handbook: deterministic inference", section on fixed splitting, attention:
// the key/value range is never split by load -- here it is not split at all,
// one CTA walks every key of its query rows -- and a query row's result must
// not depend on how the queries are chunked; "Batch-Invariant Kernel Design:
// Conv2d and Attention BMM", section "Kernel 2: Attention BMM": every
// flattened batch*head element is computed alone).
//
// Work unit: one head l and 128 consecutive query rows (a tile); a persistent
// CTA takes tiles c, c + grid, ...  Per tile, for key blocks j = 0, 1, ... of
// 128 keys in ascending order:
//   S_j  = q k_j^T                    tcgen05.mma 128 x 128 x 16, D / 16 steps
//                                      over D ascending, fp32 in TMEM (two S buffers)
//   t    = RN(S_j * c),  c = RN(scale * log2 e);  keys >= Tk -> -inf
//   m    = running row maximum of t, kept unless a block raises it by more
//          than 8 (then O and the running sum are rescaled by 2^(m_old - m_new))
//   p    = 2^(t - m) (SFU ex2)
//   l_h  = RN(l_h * alpha) + ((a0 + a1) + (a2 + a3)) for each half h of the
//          block (keys 0-63, 64-127), a_r the sum of the half's p with key
//          index = r mod 4, ascending;  l = l_0 + l_1 at the end
//   O   += bf16(p) v_j                tcgen05.mma 128 x D x 16, keys ascending,
//                                      P read from TMEM, fp32 O in TMEM
// and finally o = RN(O * RN(1 / l)), rounded once to the output type.  Every
// step is a function of the query row, the head's keys and values, Tk and
// scale only: not of L, Tq, the tile a row falls in or the SM that runs it.
//
// Warps: 0 TMA producer (q tile once per tile, then K and V blocks through a
// ring of 128 KB of stages), 1 MMA issuer (one thread), 2-9 softmax and
// epilogue: warps w and w + 4 share the 32 query rows of TMEM lane quadrant
// w % 4, one row per thread; warps 2-5 take keys 0-63 of each block and O
// columns 0-127, warps 6-9 keys 64-127 and O columns 128-255 (for D = 256;
// O columns D/2 h.. in general).  The two warps of a quadrant exchange their
// block maxima through shared memory, write their halves of the bf16 P row
// back into the S buffer they have consumed (keys 64h.. at columns
// 64h..64h+31), and decide every wait
// together (a barrier that ANDs their outcomes), so they always take the same
// path.  The tensor core runs one thread's MMAs in issue order, so S_{j+2}
// (issued after PV_j) never overwrites P_j before PV_j has read it, and the
// softmax waits for PV_{j-1} only when it must rescale O.
// Every wait is bounded; on expiry the kernel records the site, stops all
// roles, drains what it issued and frees TMEM.
#include <cuda_bf16.h>

#include "bi_common.h"
#include "bi_launch.h"
#include "bi_ptx_ext.cuh"
#include "bi_roles.cuh"

namespace bi {

constexpr int kAttnBM = 128;  // query rows per tile
constexpr int kAttnBN = 128;  // keys per block
constexpr int kAttnThreads = 320;
constexpr int kAttnSoftmaxWarps = 8;
constexpr uint32_t kAttnTmemCols = 512;  // S buffers at columns 0 and 128, O from 256
constexpr uint32_t kAttnOCol = 256;
constexpr float kAttnRescaleLog2 = 8.0f;  // keep a stale maximum while p <= 2^8
constexpr int kAttnSplitKeys = 2048;       // key range of one split (a multiple of kAttnBN)
constexpr int kAttnSmemMax = 232448;       // dynamic shared memory a CTA may use

// The shapes that follow the head dimension D (64, 128 or 256).  A ring stage
// holds kKC 16 KB pieces: of a K block, 64 columns of D for all 128 keys; of
// a V block, kVKeys keys with all D columns.  The ring takes what shared
// memory is left beside q and the output staging.
template <int D>
struct AttnCfg {
  static constexpr int kChunks = D / 64;  // 64-column chunks of D (TMA boxes, swizzle atoms)
  static constexpr int kKC = D >= 128 ? 2 : 1;
  static constexpr int kStageBytes = kKC * 16384;
  static constexpr int kKStages = kChunks / kKC;  // ring stages per K block
  static constexpr int kVKeys = kStageBytes / (D * 2) < kAttnBN ? kStageBytes / (D * 2) : kAttnBN;
  static constexpr int Q = 0;                        // kChunks x [128 rows x 64 D]
  static constexpr int OUT = Q + kAttnBM * D * 2;    // epilogue staging, 4 KB per warp
  static constexpr int STG = OUT + kAttnSoftmaxWarps * 4096;
  static constexpr int kStages = (kAttnSmemMax - 3072 - STG) / kStageBytes;
  static constexpr int BARS = STG + kStages * kStageBytes;  // mbarriers
  static constexpr int NBARS = 11 + 2 * kStages;
  static constexpr int XCH = BARS + 8 * NBARS;         // running-sum exchange, 2 x 128 floats
  static constexpr int SLOT = XCH + 2 * kAttnBM * 4;   // TMEM address, abort flag
  static constexpr int DYN = SLOT + 16 + 1024;         // + alignment slack
  static_assert(D == 64 || D == 128 || D == 256, "head dimension 64, 128 or 256");
  static_assert(DYN <= kAttnSmemMax, "attention shared memory exceeds 227 KB");
  static_assert(kStages >= 4, "at least four ring stages");
};

struct AttnBars {
  uint32_t b;
  int st;  // ring stages
  __device__ __forceinline__ uint32_t q_full() const { return b; }
  __device__ __forceinline__ uint32_t q_empty() const { return b + 8; }
  __device__ __forceinline__ uint32_t full(uint32_t s) const { return b + 16 + 8 * s; }
  __device__ __forceinline__ uint32_t empty(uint32_t s) const { return b + 16 + 8 * st + 8 * s; }
  __device__ __forceinline__ uint32_t s_full(uint32_t i) const { return b + 16 + 16 * st + 8 * i; }
  __device__ __forceinline__ uint32_t p_full() const { return b + 48 + 16 * st; }
  __device__ __forceinline__ uint32_t pv_done() const { return b + 56 + 16 * st; }
  __device__ __forceinline__ uint32_t o_full() const { return b + 64 + 16 * st; }
  __device__ __forceinline__ uint32_t o_free() const { return b + 72 + 16 * st; }
  __device__ __forceinline__ uint32_t drain() const { return b + 80 + 16 * st; }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<const uint32_t*>(&h);
}

// V stages (kVKeys keys each) of key block j that hold at least one key
// < Tk; a stage's worth of keys wholly past Tk is neither loaded nor
// multiplied.
template <int D>
__device__ __forceinline__ int attn_v_stages(int j, int Tk) {
  constexpr int V = AttnCfg<D>::kVKeys;
  const int left = Tk - j * kAttnBN;
  return left >= kAttnBN ? kAttnBN / V : (left + V - 1) / V;
}

// A work unit: head l, query rows q0 .. q0+127, and keys k0 .. k0+tk-1 (split
// sp of the key range; the whole range when it is not split) in nkb blocks.
// Units of one head and split are adjacent so that the CTAs working on them at
// the same time share its K and V in L2.
struct AttnTile {
  int l, q0, sp, k0, tk, nkb;
};
__device__ __forceinline__ AttnTile attn_tile(const AttnParams& p, int tile) {
  AttnTile t;
  const int per_head = p.ns * p.q_tiles;
  t.l = tile / per_head;
  const int r = tile - t.l * per_head;
  t.sp = r / p.q_tiles;
  t.q0 = (r - t.sp * p.q_tiles) * kAttnBM;
  t.k0 = t.sp * kAttnSplitKeys;
  t.tk = min(p.Tk - t.k0, kAttnSplitKeys);
  t.nkb = (t.tk + kAttnBN - 1) / kAttnBN;
  return t;
}

// ---------------------------------------------------------------------------
// Producer (one thread): per tile the q tile, then K_0, and for each block j
// K_{j+1} (if any) followed by V_j -- the order the MMA issuer consumes them.
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void attn_producer(const AttnParams& p, const AttnBars& bars, uint32_t sQ,
                                              uint32_t sS, const WaitCtl& wc) {
  using C = AttnCfg<D>;
  uint32_t it = 0;
  int q_loads = 0;
  bool ok = true;
  auto next_stage = [&](uint32_t& dst, uint32_t& bar) -> bool {
    const uint32_t s = it % C::kStages, r = it / C::kStages;
    if (r > 0 && !mbar_wait_bounded(bars.empty(s), (r - 1) & 1, wc.abort, wc.status_word, wc.limit_ns,
                                    status_code(6, kSiteProducerEmpty)))
      return false;
    dst = sS + s * C::kStageBytes;
    bar = bars.full(s);
    mbar_arrive_expect_tx(bar, C::kStageBytes);
    ++it;
    return true;
  };
  auto load_k = [&](int j, const AttnTile& t) -> bool {  // all keys of block j, D columns 64c.. per piece
    for (int cs = 0; cs < C::kKStages; ++cs) {
      uint32_t dst, bar;
      if (!next_stage(dst, bar)) return false;
      for (int b = 0; b < C::kKC; ++b)
        tma_load_3d(dst + b * 16384, &p.tma_k, bar, (cs * C::kKC + b) * 64, t.k0 + j * kAttnBN, t.l);
    }
    return true;
  };
  auto load_v = [&](int j, const AttnTile& t) -> bool {  // kVKeys keys of block j per stage, all D
    const int nst = attn_v_stages<D>(j, t.tk);
    for (int vs = 0; vs < nst; ++vs) {
      uint32_t dst, bar;
      if (!next_stage(dst, bar)) return false;
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_3d(dst + c * (C::kVKeys * 128), &p.tma_v, bar, c * 64, t.k0 + j * kAttnBN + vs * C::kVKeys,
                    t.l);
    }
    return true;
  };
  for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
    const AttnTile t = attn_tile(p, tile);
    const int l = t.l;
    const int q0 = t.q0;
    if (q_loads > 0 && !mbar_wait_bounded(bars.q_empty(), (q_loads - 1) & 1, wc.abort, wc.status_word,
                                          wc.limit_ns, status_code(6, kSiteProducerEmpty))) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(bars.q_full(), kAttnBM * D * 2);
    for (int c = 0; c < C::kChunks; ++c) tma_load_3d(sQ + c * 16384, &p.tma_q, bars.q_full(), c * 64, q0, l);
    ++q_loads;
    ok = load_k(0, t);
    for (int j = 0; ok && j < t.nkb; ++j) {
      if (j + 1 < t.nkb) ok = load_k(j + 1, t);
      if (ok) ok = load_v(j, t);
    }
  }
  // No copy may still be landing in shared memory when the CTA exits.
  if (q_loads > 0)
    mbar_wait_bounded(bars.q_full(), (q_loads - 1) & 1, nullptr, wc.status_word, wc.limit_ns,
                      status_code(6, kSiteDrain));
  const uint32_t first = it > (uint32_t)C::kStages ? it - C::kStages : 0u;
  for (uint32_t j = first; j < it; ++j)
    if (!mbar_wait_bounded(bars.full(j % C::kStages), (j / C::kStages) & 1, nullptr, wc.status_word,
                           wc.limit_ns, status_code(6, kSiteDrain)))
      break;
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread): S_0; then per block j: S_{j+1} (other S buffer),
// PV_j once the softmax warps have written P_j.
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void attn_mma(const AttnParams& p, const AttnBars& bars, uint32_t sQ, uint32_t sS,
                                         uint32_t tmem, const WaitCtl& wc) {
  using C = AttnCfg<D>;
  const uint32_t kIdS = idesc_bf16_f32(kAttnBM, kAttnBN, false);
  const uint32_t kIdO = idesc_bf16_f32(kAttnBM, D, true);
  uint32_t it = 0, sc = 0, pc = 0;
  int local = 0;
  bool ok = true;
  auto wait = [&](uint32_t bar, uint32_t par) {
    return mbar_wait_bounded(bar, par, wc.abort, wc.status_word, wc.limit_ns, status_code(6, kSiteMmaFull));
  };
  // S_j goes to TMEM buffer (block count) % 2; it is free: the softmax warps
  // consumed S_{j-2} before signalling P_{j-2}, and PV_{j-2} -- the last
  // reader of the buffer -- was issued before this S_j.
  int nkb = 0, tk = 0;  // the current tile's key blocks and keys
  auto issue_s = [&](int j) -> bool {
    const uint32_t buf = sc & 1;
    const uint32_t d = tmem + buf * kAttnBN;
    for (int cs = 0; cs < C::kKStages; ++cs) {
      const uint32_t s = it % C::kStages, r = it / C::kStages;
      if (!wait(bars.full(s), r & 1)) return false;
      tc_fence_after_sync();
      const uint32_t kb = sS + s * C::kStageBytes;
#pragma unroll
      for (int b = 0; b < C::kKC; ++b) {
        const int c = cs * C::kKC + b;  // D columns 64c..
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // K = 16 steps over D, ascending
          const uint64_t ad = smem_desc_sw128(sQ + c * 16384 + kk * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(kb + b * 16384 + kk * 32, 16, 1024);
          umma_bf16(d, ad, bd, kIdS, (c | kk) != 0 ? 1u : 0u);
        }
      }
      umma_commit(bars.empty(s));
      ++it;
    }
    umma_commit(bars.s_full(buf));
    ++sc;
    if (j == nkb - 1) umma_commit(bars.q_empty());  // the tile's last read of q
    return true;
  };
  auto issue_pv = [&](int j) -> bool {
    const uint32_t pbuf = tmem + (pc & 1) * kAttnBN;  // P_j: in the TMEM buffer of S_j
    const int nst = attn_v_stages<D>(j, tk);
    for (int vs = 0; vs < nst; ++vs) {  // keys vs * kVKeys.. of the block
      const uint32_t s = it % C::kStages, r = it / C::kStages;
      if (!wait(bars.full(s), r & 1)) return false;
      tc_fence_after_sync();
      const uint32_t vb = sS + s * C::kStageBytes;
#pragma unroll
      for (int k = 0; k < C::kVKeys / 16; ++k) {  // K = 16 steps over keys, ascending
        const int key = vs * C::kVKeys + 16 * k;  // first key of the step within the block
        const uint32_t acol = pbuf + (key >> 6) * 64 + ((key & 63) >> 4) * 8;
        const uint64_t bd = smem_desc_sw128(vb + k * 2048, C::kVKeys * 128, 1024);
        umma_bf16_ts(tmem + kAttnOCol, acol, bd, kIdO, (j | vs | k) != 0 ? 1u : 0u);
      }
      umma_commit(bars.empty(s));
      ++it;
    }
    umma_commit(bars.pv_done());
    ++pc;
    return true;
  };
  for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++local) {
    const AttnTile t = attn_tile(p, tile);
    nkb = t.nkb;
    tk = t.tk;
    if (!wait(bars.q_full(), local & 1)) break;
    tc_fence_after_sync();
    ok = issue_s(0);
    for (int j = 0; ok && j < nkb; ++j) {
      if (j + 1 < nkb) ok = issue_s(j + 1);
      if (ok) ok = wait(bars.p_full(), pc & 1);
      if (ok && j == 0 && local > 0) ok = wait(bars.o_free(), (local - 1) & 1);  // O is overwritten
      if (ok) {
        tc_fence_after_sync();
        ok = issue_pv(j);
      }
    }
    if (ok) umma_commit(bars.o_full());
  }
  // Every MMA issued above has finished before TMEM can be released.
  umma_commit(bars.drain());
  mbar_wait_bounded(bars.drain(), 0, nullptr, wc.status_word, wc.limit_ns, status_code(6, kSiteDrain));
}

// ---------------------------------------------------------------------------
// Softmax and epilogue (warps 2-9): one query row and one half of the keys /
// of O's columns per thread.
// ---------------------------------------------------------------------------
// A warp's share of the output: its 32 query rows (one per lane) x W columns
// of O starting at TMEM address tcol (this warp's lane quadrant) and at
// output column col0, scaled by rinv and rounded once to the output type,
// stored to rows 0 .. rows-1 of `out` (row stride ld elements).  The rows are
// turned around through the warp's 4 KB staging region one piece of PB bytes
// per row at a time (16-byte unit u of row r at unit u ^ swz(r),
// conflict-free both ways), so that each store instruction writes whole row
// segments of PB bytes.
template <int W, bool F32, typename T>
__device__ __forceinline__ void attn_store_rows(T* out, int64_t ld, int64_t rows, uint32_t tcol, int col0,
                                                int lane, uint32_t region, float rinv) {
  constexpr int esz = F32 ? 4 : 2;
  constexpr int PB = W * esz < 128 ? W * esz : 128;  // bytes of a row per piece
  constexpr int U = PB / 16;                         // 16-byte units per piece row
  constexpr int cols = PB / esz;                     // columns per piece
  auto swz = [](int r) { return U == 8 ? (r & 7) : ((r >> 1) & 3); };
#pragma unroll 1
  for (int c = 0; c < W / cols; ++c) {
    uint32_t w[PB / 4];
#pragma unroll
    for (int h = 0; h < cols / 32; ++h) {
      uint32_t r[32];
      tmem_load_32cols(tcol + c * cols + h * 32, r);
      tmem_load_wait(r);
      if constexpr (F32) {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), rinv));
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[h * 16 + i] =
              pack_bf16x2(__fmul_rn(__uint_as_float(r[2 * i]), rinv), __fmul_rn(__uint_as_float(r[2 * i + 1]), rinv));
      }
    }
    __syncwarp();  // the previous piece has been read back
#pragma unroll
    for (int u = 0; u < U; ++u)
      st_shared_v4(region + lane * PB + ((u ^ swz(lane)) << 4), w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
    __syncwarp();
    // read back: lane L takes unit L % U of rows (32 / U) i + L / U
    const int u = lane % U;
    const int col = col0 + c * cols + u * (16 / esz);
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int rr = (32 / U) * i + lane / U;
      const uint4 v = ld_shared_v4(region + rr * PB + ((u ^ swz(rr)) << 4));
      if (rr < rows) *reinterpret_cast<uint4*>(out + rr * ld + col) = v;
    }
  }
}

template <int D>
__device__ __forceinline__ void attn_softmax(const AttnParams& p, const AttnBars& bars, uint32_t sOut,
                                             float* xch, uint32_t tmem, int warp, int lane, const WaitCtl& wc) {
  constexpr int kHalf = D / 2;     // O columns per warp
  const int qd = warp & 3;         // TMEM lane quadrant this warp may access
  const int hc = (warp - 2) >> 2;  // half: keys 64hc.. of a block, O columns kHalf hc..
  const int row = qd * 32 + lane;
  const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
  const uint32_t pair_bar = 1 + qd;  // named barrier of the quadrant's two warps
  const float c2 = p.score_log2;
  uint32_t sc = 0, pc = 0;
  int local = 0;
  // Both warps of the quadrant wait, then agree: true only if both got it.
  auto wait_pair = [&](uint32_t bar, uint32_t par) -> bool {
    const bool got = mbar_wait_bounded(bar, par, wc.abort, wc.status_word, wc.limit_ns,
                                       status_code(6, kSiteAttnSoftmax));
    return named_barrier_and(pair_bar, 64, got);
  };
  bool ok = true;
  for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++local) {
    const AttnTile tl = attn_tile(p, tile);
    const int l = tl.l;
    const int q0 = tl.q0;
    float m = -INFINITY, lsum = 0.0f;
    for (int j = 0; j < tl.nkb; ++j) {
      const uint32_t buf = sc & 1, use = sc >> 1;
      if (!wait_pair(bars.s_full(buf), use & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t scol = trow + buf * kAttnBN + hc * 64;
      float t[64];
      {
        uint32_t r0[32], r1[32];
        tmem_load_32cols(scol, r0);
        tmem_load_32cols(scol + 32, r1);
        tmem_load_wait(r0);
        tmem_load_wait(r1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          t[i] = __fmul_rn(__uint_as_float(r0[i]), c2);
          t[32 + i] = __fmul_rn(__uint_as_float(r1[i]), c2);
        }
      }
      const int kvalid = tl.tk - j * kAttnBN - hc * 64;  // keys of this half inside the range
      if (kvalid < 64) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i >= kvalid) t[i] = -INFINITY;
      }
      float mx;
      {
        float mp[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) mp[r] = t[r];
#pragma unroll
        for (int i = 8; i < 64; ++i) mp[i & 7] = fmaxf(mp[i & 7], t[i]);
        mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])), fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      }
      // Exchange the halves' maxima through shared memory (the running-sum
      // exchange area, slot hc of the row).  A slot is written again only
      // after a later barrier of the pair: the P signal wait of this block,
      // or the one below for the first block.
      xch[hc * kAttnBM + row] = mx;
      named_barrier(pair_bar, 64);
      const float mo = xch[(1 - hc) * kAttnBM + row];
      ++sc;
      const float m_blk = hc == 0 ? fmaxf(mx, mo) : fmaxf(mo, mx);  // the same operands in both warps
      const float m_new = fmaxf(m, m_blk);
      float m_use = m, alpha = 1.0f;
      bool resc = false;
      if (j == 0) {
        m_use = m_new;
      } else if (m_new > __fadd_rn(m, kAttnRescaleLog2)) {
        alpha = ex2_approx(__fsub_rn(m, m_new));
        m_use = m_new;
        resc = true;
      }
      uint32_t pk[32];
      float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float p0 = ex2_approx(__fsub_rn(t[i], m_use));
        const float p1 = ex2_approx(__fsub_rn(t[i + 1], m_use));
        a4[i & 3] = __fadd_rn(a4[i & 3], p0);
        a4[(i + 1) & 3] = __fadd_rn(a4[(i + 1) & 3], p1);
        pk[i / 2] = pack_bf16x2(p0, p1);
      }
      const float ps = __fadd_rn(__fadd_rn(a4[0], a4[1]), __fadd_rn(a4[2], a4[3]));
      lsum = __fadd_rn(resc ? __fmul_rn(lsum, alpha) : lsum, ps);
      m = m_use;
      // Rescaling O needs PV_{j-1} finished (O stable).  At most that one PV
      // can be pending: S_j, whose completion was waited for above, was
      // issued after PV_{j-2}.
      if (__any_sync(0xffffffffu, resc)) {
        if (!wait_pair(bars.pv_done(), (pc - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const float f = resc ? alpha : 1.0f;
#pragma unroll 1
        for (int c = 0; c < kHalf / 32; ++c) {
          const uint32_t oc = trow + kAttnOCol + hc * kHalf + c * 32;
          uint32_t r[32];
          tmem_load_32cols(oc, r);
          tmem_load_wait(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), f));
          tmem_store_32cols(oc, r);
        }
        tmem_store_wait();
      }
      // This half's P row (64 keys, bf16 pairs) into columns 64 hc .. 64 hc + 31
      // of the S buffer: the A operand of PV_j.  (The buffer's previous P was
      // read by PV_{j-2}, complete since S_j, issued after it, is.)
      tmem_store_32cols(scol, pk);
      tmem_store_wait();
      tc_fence_before_sync();
      // Signal P_j only once every warp has signalled P_{j-1}: a warp that ran
      // ahead (quadrants with no output rows skip the epilogue) must not
      // arrive twice on one phase.
      if (pc > 0 && !wait_pair(bars.p_full(), (pc - 1) & 1)) {
        ok = false;
        break;
      }
      if (pc == 0) named_barrier(pair_bar, 64);  // the partner has read this block's maximum
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.p_full());
      ++pc;
    }
    if (!ok) break;

    // Epilogue: o = RN(O * RN(1 / (l_0 + l_1))).  Each warp turns its 32 rows
    // x 128 columns around through its own 4 KB of the staging buffer, 128
    // bytes of each row at a time, so that each global store instruction
    // writes four whole 128-byte row segments.
    if (!wait_pair(bars.o_full(), local & 1)) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    xch[hc * kAttnBM + row] = lsum;
    named_barrier(pair_bar, 64);
    const float lo = xch[(1 - hc) * kAttnBM + row];
    named_barrier(pair_bar, 64);  // both read before the next tile writes again
    const float lrow = hc == 0 ? __fadd_rn(lsum, lo) : __fadd_rn(lo, lsum);
    // Unsplit key range: the output o = RN(O * RN(1 / l)).  A split writes its
    // partial O (unnormalised, relative to its running maximum m) and (m, l)
    // to the workspace for the merge.
    const bool split = p.ns > 1;
    const float rinv = split ? 1.0f : __frcp_rn(lrow);
    if (split && hc == 0 && q0 + row < p.Tq) {
      float* ml = p.ws_ml + (((int64_t)tl.sp * p.L + l) * p.Tq + q0 + row) * 2;
      ml[0] = m;
      ml[1] = lrow;
    }
    if (q0 + qd * 32 < p.Tq) {  // warp-uniform: some of its rows are outputs
      const uint32_t region = sOut + (hc * 4 + qd) * 4096;
      const int64_t qrow = q0 + qd * 32;
      const uint32_t tcol = trow + kAttnOCol + hc * kHalf;
      if (split)
        attn_store_rows<kHalf, true>(p.ws_o + (((int64_t)tl.sp * p.L + l) * p.Tq + qrow) * D, D, p.Tq - qrow,
                                     tcol, hc * kHalf, lane, region, rinv);
      else if (p.out_f32)
        attn_store_rows<kHalf, true>(static_cast<float*>(p.o) + (int64_t)l * p.o_l + qrow * p.o_t, p.o_t,
                                     p.Tq - qrow, tcol, hc * kHalf, lane, region, rinv);
      else
        attn_store_rows<kHalf, false>(static_cast<__nv_bfloat16*>(p.o) + (int64_t)l * p.o_l + qrow * p.o_t,
                                      p.o_t, p.Tq - qrow, tcol, hc * kHalf, lane, region, rinv);
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.o_free());
  }
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using C = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + C::Q;
  const uint32_t sOut = base + C::OUT;
  const uint32_t sS = base + C::STG;
  const AttnBars bars{base + C::BARS, C::kStages};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bars.q_full(), 1);
    mbar_init(bars.q_empty(), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(bars.s_full(i), 1);
    mbar_init(bars.p_full(), kAttnSoftmaxWarps);
    mbar_init(bars.pv_done(), 1);
    mbar_init(bars.o_full(), 1);
    mbar_init(bars.o_free(), kAttnSoftmaxWarps);
    mbar_init(bars.drain(), 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&p.tma_q);
    tma_prefetch_desc(&p.tma_k);
    tma_prefetch_desc(&p.tma_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kAttnTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status_word, p.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) attn_producer<D>(p, bars, sQ, sS, wc);
  } else if (warp == 1) {
    if (lane == 0) attn_mma<D>(p, bars, sQ, sS, tmem, wc);
  } else {
    attn_softmax<D>(p, bars, sOut, reinterpret_cast<float*>(smem + C::XCH), tmem, warp, lane, wc);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kAttnTmemCols);
  }
}

// ===========================================================================
// Two query tiles per CTA, head dimension 64.
//
// A work unit holds query tiles A and B (rows qa.. and qa + 128..) of one
// head and one split of its key range; both read every K and V block, which
// is loaded once for the pair.  Warps 4-7 run the softmax and epilogue of
// tile A, warps 8-11 those of tile B, one query row per thread over all 128
// keys of a block, so each SM sub-partition holds one warp of each tile.
// Warp 1 issues tile A's MMAs and warp 2 tile B's.
// TMEM: tile X (0 = A, 1 = B) keeps S at columns 256X .. 256X + 127, P
// (bf16 pairs, key 2i and 2i + 1 in column i) at 256X + 128 .. 256X + 191
// and O at 256X + 192 .. 256X + 255.  With S, P and O apart, S_X(j + 1) is
// computed while the softmax of block j is still running: the softmax
// signals that it has read S_X(j) (s_free) before it computes and writes
// P_X(j), and the issuer then runs S_X(j + 1) ahead of PV_X(j).  Before it
// writes P_X(j) or rescales O the softmax waits for PV_X(j - 1) (pv_done).
// A query row's arithmetic is exactly the one-tile kernel's above: the same
// MMAs on the same operands (P's columns are arranged differently, its
// values and the K = 16 steps over keys are the same), the block maximum
// over both halves of the block, the halves' running sums l_0 and l_1 kept
// apart and added at the end, the same rescale rule -- so either kernel
// gives the same bits for a row, and which one runs depends on the head
// dimension and the query count only.
// Units with two tiles come first (head by head), then the units of heads
// with an odd number of query tiles that hold their last tile alone.
// ===========================================================================
// 12 warps: 0 producer, 1 and 2 the MMA issuers of tiles A and B, 3 idle
// (warpgroup 0, 64 registers a thread), 4-7 tile A's softmax, 8-11 tile B's
// (warpgroups 1 and 2, 216 registers): 128 x 64 + 256 x 216 <= 384 x 168,
// the registers the CTA is launched with.
constexpr int kAttn2Threads = 384;
constexpr uint32_t kAttn2RegsLow = 64, kAttn2RegsHigh = 216;
static_assert(128 * kAttn2RegsLow + 256 * kAttn2RegsHigh <= kAttn2Threads * 168, "register split exceeds the launch");
constexpr int kAttn2D = 64;
constexpr uint32_t kAttn2P = 128, kAttn2O = 192;  // column offsets within a tile's 256

struct Attn2Cfg {
  static constexpr int D = kAttn2D;
  static constexpr int kStageBytes = AttnCfg<D>::kStageBytes;  // one K block or one V block
  static constexpr int kQBytes = kAttnBM * D * 2;              // one query tile
  static constexpr int Q = 0;                                  // tiles A and B
  static constexpr int OUT = Q + 2 * kQBytes;                  // epilogue staging, 4 KB per warp
  static constexpr int STG = OUT + kAttnSoftmaxWarps * 4096;
  static constexpr int kStages = (kAttnSmemMax - 3072 - STG) / kStageBytes;
  static constexpr int BARS = STG + kStages * kStageBytes;
  static constexpr int NBARS = 2 + 2 * kStages + 2 * 7;
  static constexpr int SLOT = BARS + 8 * NBARS;  // TMEM address, abort flag
  static constexpr int DYN = SLOT + 16 + 1024;
  static_assert(AttnCfg<D>::kKStages == 1 && AttnCfg<D>::kVKeys == kAttnBN && AttnCfg<D>::kChunks == 1,
                "one 64-column piece per K or V block");
  static_assert(DYN <= kAttnSmemMax, "attention shared memory exceeds 227 KB");
  static_assert(kStages >= 4, "at least four ring stages");
};

struct Attn2Bars {
  uint32_t b;
  int st;
  __device__ __forceinline__ uint32_t q_full() const { return b; }
  __device__ __forceinline__ uint32_t q_empty() const { return b + 8; }
  __device__ __forceinline__ uint32_t full(uint32_t s) const { return b + 16 + 8 * s; }
  __device__ __forceinline__ uint32_t empty(uint32_t s) const { return b + 16 + 8 * st + 8 * s; }
  __device__ __forceinline__ uint32_t tile(int x, int i) const { return b + 16 + 16 * st + 56 * x + 8 * i; }
  __device__ __forceinline__ uint32_t s_full(int x) const { return tile(x, 0); }
  __device__ __forceinline__ uint32_t s_free(int x) const { return tile(x, 1); }
  __device__ __forceinline__ uint32_t p_full(int x) const { return tile(x, 2); }
  __device__ __forceinline__ uint32_t pv_done(int x) const { return tile(x, 3); }
  __device__ __forceinline__ uint32_t o_full(int x) const { return tile(x, 4); }
  __device__ __forceinline__ uint32_t o_free(int x) const { return tile(x, 5); }
  __device__ __forceinline__ uint32_t drain(int x) const { return tile(x, 6); }
};

struct Attn2Unit {
  int l, sp, k0, tk, nkb;
  int nt;  // query tiles in the unit (1 or 2): rows qa .. qa + 128 nt - 1
  int qa;
};
__device__ __forceinline__ Attn2Unit attn2_unit(const AttnParams& p, int u) {
  Attn2Unit t;
  const int pairs = p.q_tiles >> 1;  // two-tile units per head and split
  int hs, qt;
  if (u < p.pair_units) {
    hs = u / pairs;
    qt = 2 * (u - hs * pairs);
    t.nt = 2;
  } else {
    hs = u - p.pair_units;
    qt = p.q_tiles - 1;
    t.nt = 1;
  }
  t.l = hs / p.ns;
  t.sp = hs - t.l * p.ns;
  t.qa = qt * kAttnBM;
  t.k0 = t.sp * kAttnSplitKeys;
  t.tk = min(p.Tk - t.k0, kAttnSplitKeys);
  t.nkb = (t.tk + kAttnBN - 1) / kAttnBN;
  return t;
}

// Producer (one thread): per unit its query tiles, then K_0, V_0, K_1, V_1, ...
__device__ __forceinline__ void attn2_producer(const AttnParams& p, const Attn2Bars& bars, uint32_t sQ,
                                               uint32_t sS, const WaitCtl& wc) {
  using C = Attn2Cfg;
  uint32_t it = 0;
  int q_loads = 0;
  bool ok = true;
  auto load = [&](const CUtensorMap* map, int key, int l) -> bool {  // one K or V block: 128 keys x 64
    const uint32_t s = it % C::kStages, r = it / C::kStages;
    if (r > 0 && !mbar_wait_bounded(bars.empty(s), (r - 1) & 1, wc.abort, wc.status_word, wc.limit_ns,
                                    status_code(6, kSiteProducerEmpty)))
      return false;
    mbar_arrive_expect_tx(bars.full(s), C::kStageBytes);
    tma_load_3d(sS + s * C::kStageBytes, map, bars.full(s), 0, key, l);
    ++it;
    return true;
  };
  for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
    const Attn2Unit t = attn2_unit(p, u);
    if (q_loads > 0 && !mbar_wait_bounded(bars.q_empty(), (q_loads - 1) & 1, wc.abort, wc.status_word,
                                          wc.limit_ns, status_code(6, kSiteProducerEmpty))) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(bars.q_full(), t.nt * C::kQBytes);
    for (int x = 0; x < t.nt; ++x)
      tma_load_3d(sQ + x * C::kQBytes, &p.tma_q, bars.q_full(), 0, t.qa + x * kAttnBM, t.l);
    ++q_loads;
    ok = load(&p.tma_k, t.k0, t.l);
    for (int j = 0; ok && j < t.nkb; ++j) {
      ok = load(&p.tma_v, t.k0 + j * kAttnBN, t.l);
      if (ok && j + 1 < t.nkb) ok = load(&p.tma_k, t.k0 + (j + 1) * kAttnBN, t.l);
    }
  }
  if (q_loads > 0)
    mbar_wait_bounded(bars.q_full(), (q_loads - 1) & 1, nullptr, wc.status_word, wc.limit_ns,
                      status_code(6, kSiteDrain));
  const uint32_t first = it > (uint32_t)C::kStages ? it - C::kStages : 0u;
  for (uint32_t j = first; j < it; ++j)
    if (!mbar_wait_bounded(bars.full(j % C::kStages), (j / C::kStages) & 1, nullptr, wc.status_word,
                           wc.limit_ns, status_code(6, kSiteDrain)))
      break;
}

// MMA issuer of tile x (one thread of warp 1 for A, of warp 2 for B).  An
// mbarrier wait stalls the waiting warp until the MMAs it issued so far have
// completed, so each tile has its own issuer: while one waits, the tensor
// core runs the other's MMAs.  Per unit: S_x(0); then per key block j:
// S_x(j + 1) once the softmax has read S_x(j), and PV_x(j) once it has
// written P_x(j).  Every K or V stage is released by two commits (one per
// tile; a unit with tile A alone commits twice), and so is the q buffer.
// Units with both tiles come first in every CTA's sequence, so tile B's
// issuer stops at the first unit without one.  The ring holds, per unit,
// K_0, V_0, K_1, V_1, ...
__device__ __forceinline__ void attn2_mma(const AttnParams& p, const Attn2Bars& bars, uint32_t sQ, uint32_t sS,
                                          uint32_t tmem, int x, const WaitCtl& wc) {
  using C = Attn2Cfg;
  const uint32_t kIdS = idesc_bf16_f32(kAttnBM, kAttnBN, false);
  const uint32_t kIdO = idesc_bf16_f32(kAttnBM, C::D, true);
  const uint32_t tS = tmem + x * 256, tP = tS + kAttn2P, tO = tS + kAttn2O, qx = sQ + x * C::kQBytes;
  uint32_t it = 0, pc = 0, sf = 0;  // ring stages, PVs issued, S reads awaited
  int ul = 0, uq = 0;
  bool ok = true;
  auto wait = [&](uint32_t bar, uint32_t par) {
    return mbar_wait_bounded(bar, par, wc.abort, wc.status_word, wc.limit_ns, status_code(6, kSiteMmaFull));
  };
  auto stage_ready = [&](uint32_t i) { return wait(bars.full(i % C::kStages), (i / C::kStages) & 1); };
  // S_x = q_x k^T for the K block in ring stage i: 4 steps of 16 over D, ascending.
  auto issue_s = [&](uint32_t i) {
    const uint32_t kb = sS + (i % C::kStages) * C::kStageBytes;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      umma_bf16(tS, smem_desc_sw128(qx + kk * 32, 16, 1024), smem_desc_sw128(kb + kk * 32, 16, 1024), kIdS,
                kk != 0 ? 1u : 0u);
    umma_commit(bars.s_full(x));
  };
  // O_x (+)= P_x v for the V block in ring stage i: 8 steps of 16 keys, ascending.
  auto issue_pv = [&](uint32_t i, int j) {
    const uint32_t vb = sS + (i % C::kStages) * C::kStageBytes;
#pragma unroll
    for (int k = 0; k < kAttnBN / 16; ++k)
      umma_bf16_ts(tO, tP + 8 * k, smem_desc_sw128(vb + k * 2048, kAttnBN * 128, 1024), kIdO,
                   (j | k) != 0 ? 1u : 0u);
  };
  for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x, ++uq) {
    const Attn2Unit t = attn2_unit(p, u);
    if (x >= t.nt) break;  // tile B: no unit with two tiles follows
    const bool twice = t.nt == 1;
    auto release = [&](uint32_t bar) {
      umma_commit(bar);
      if (twice) umma_commit(bar);
    };
    const uint32_t k_first = it++;
    // S_x(0) overwrites the S buffer: the softmax has read the last S.
    if (ul > 0 && !wait(bars.s_free(x), sf++ & 1)) break;
    if (!wait(bars.q_full(), uq & 1) || !stage_ready(k_first)) break;
    tc_fence_after_sync();
    issue_s(k_first);
    release(bars.empty(k_first % C::kStages));
    if (t.nkb == 1) release(bars.q_empty());
    for (int j = 0; ok && j < t.nkb; ++j) {
      const bool more = j + 1 < t.nkb;
      const uint32_t vi = it++;  // the ring holds V_j, then K_(j+1)
      const uint32_t ki = more ? it++ : 0u;
      if (more) {
        ok = wait(bars.s_free(x), sf++ & 1) && stage_ready(ki);
        if (!ok) break;
        tc_fence_after_sync();
        issue_s(ki);
        release(bars.empty(ki % C::kStages));
        if (j + 2 == t.nkb) release(bars.q_empty());  // the unit's last read of q
      }
      ok = wait(bars.p_full(x), pc & 1);
      if (ok && j == 0 && ul > 0) ok = wait(bars.o_free(x), (ul - 1) & 1);  // O is overwritten
      if (ok) ok = stage_ready(vi);
      if (!ok) break;
      tc_fence_after_sync();
      issue_pv(vi, j);
      umma_commit(bars.pv_done(x));
      ++pc;
      if (!more) umma_commit(bars.o_full(x));
      release(bars.empty(vi % C::kStages));
    }
    ++ul;
  }
  umma_commit(bars.drain(x));
  mbar_wait_bounded(bars.drain(x), 0, nullptr, wc.status_word, wc.limit_ns, status_code(6, kSiteDrain));
}

// Running maxima mp[r] over keys 32 g .. 32 g + 31 of the thread's row: of the
// raw scores S (RAW: c finite and > 0), else of t = RN(S c); keys past the
// range (kvalid keys of the block are inside it) are left out.
template <bool RAW>
__device__ __forceinline__ void attn2_max32(const uint32_t (&r)[32], float (&mp)[8], float c2, int g, int kvalid) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = RAW ? __uint_as_float(r[i]) : __fmul_rn(__uint_as_float(r[i]), c2);
  if (kvalid < 32 * (g + 1)) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (32 * g + i >= kvalid) v[i] = -INFINITY;
  }
#pragma unroll
  for (int i = 0; i < 32; i += 2) mp[(i >> 1) & 7] = fmax3(mp[(i >> 1) & 7], v[i], v[i + 1]);
}

// Keys 32 g .. 32 g + 31: t = RN(S c) (-inf past the range), p = 2^(t - m)
// (SFU ex2), packed to bf16 pairs in pk[0..15], each p added to the partial
// sum a_r of its key index r mod 4 (keys ascending).
__device__ __forceinline__ void attn2_exp32(const uint32_t (&r)[32], float c2, float m, int g, int kvalid,
                                            uint32_t (&pk)[16], float (&a4)[4]) {
  float t[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) t[i] = __fmul_rn(__uint_as_float(r[i]), c2);
  if (kvalid < 32 * (g + 1)) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (32 * g + i >= kvalid) t[i] = -INFINITY;
  }
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float p0 = ex2_approx(__fsub_rn(t[i], m));
    const float p1 = ex2_approx(__fsub_rn(t[i + 1], m));
    a4[i & 3] = __fadd_rn(a4[i & 3], p0);
    a4[(i + 1) & 3] = __fadd_rn(a4[(i + 1) & 3], p1);
    pk[i / 2] = pack_bf16x2(p0, p1);
  }
}

// The block maximum of t = RN(S c) over one row of S (the block's four
// groups of 32 keys).
template <bool RAW>
__device__ __forceinline__ float attn2_block_max(const uint32_t (&r0)[32], const uint32_t (&r1)[32],
                                                 const uint32_t (&r2)[32], const uint32_t (&r3)[32], float c2,
                                                 int kvalid) {
  float mp[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) mp[r] = -INFINITY;
  attn2_max32<RAW>(r0, mp, c2, 0, kvalid);
  attn2_max32<RAW>(r1, mp, c2, 1, kvalid);
  attn2_max32<RAW>(r2, mp, c2, 2, kvalid);
  attn2_max32<RAW>(r3, mp, c2, 3, kvalid);
  const float mx = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
  // For a finite c > 0, RN(x c) rises with x: the maximum of t is RN(max S * c).
  return RAW ? __fmul_rn(mx, c2) : mx;
}

__device__ __forceinline__ void attn2_softmax(const AttnParams& p, const Attn2Bars& bars, uint32_t sOut,
                                              uint32_t tmem, int warp, int lane, const WaitCtl& wc) {
  constexpr int D = kAttn2D;
  const int x = (warp - 4) >> 2;  // tile: A for warps 4-7, B for 8-11
  const int qd = warp & 3;        // TMEM lane quadrant this warp may access
  const int row = qd * 32 + lane;
  const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16) + x * 256;  // S; P and O follow
  const float c2 = p.score_log2;
  const bool raw_max = c2 > 0.0f && c2 < INFINITY;
  uint32_t sc = 0, pcn = 0;  // S blocks received, P blocks handed over
  int ul = 0;
  auto wait = [&](uint32_t bar, uint32_t par) {
    return mbar_wait_bounded(bar, par, wc.abort, wc.status_word, wc.limit_ns, status_code(6, kSiteAttnSoftmax));
  };
  auto signal = [&](uint32_t bar) {  // after this warp's TMEM accesses
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  };
  bool ok = true;
  for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
    const Attn2Unit tl = attn2_unit(p, u);
    if (x >= tl.nt) break;  // tile B: no unit with two tiles follows
    const int q0 = tl.qa + x * kAttnBM;
    float m = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    for (int j = 0; j < tl.nkb; ++j) {
      if (!wait(bars.s_full(x), sc & 1)) {
        ok = false;
        break;
      }
      ++sc;
      tc_fence_after_sync();
      const int kvalid = tl.tk - j * kAttnBN;  // keys of the block inside the range
      // The row of S is read once; the S buffer is released at once for S_X(j + 1).
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_load_32cols(trow, r0);
      tmem_load_32cols(trow + 32, r1);
      tmem_load_32cols(trow + 64, r2);
      tmem_load_32cols(trow + 96, r3);
      tmem_load_wait(r0);
      tmem_load_wait(r1);
      tmem_load_wait(r2);
      tmem_load_wait(r3);
      signal(bars.s_free(x));
      const float mx = raw_max ? attn2_block_max<true>(r0, r1, r2, r3, c2, kvalid)
                               : attn2_block_max<false>(r0, r1, r2, r3, c2, kvalid);
      const float m_new = fmaxf(m, mx);
      float m_use = m, alpha = 1.0f;
      bool resc = false;
      if (j == 0) {
        m_use = m_new;
      } else if (m_new > __fadd_rn(m, kAttnRescaleLog2)) {
        alpha = ex2_approx(__fsub_rn(m, m_new));
        m_use = m_new;
        resc = true;
      }
      // P_X(j - 1) and O are free once PV_X(j - 1) has completed (for j = 0
      // the previous unit's epilogue waited for its last PV).
      if (j > 0) {
        if (!wait(bars.pv_done(x), (pcn - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
      // P, 32 keys at a time, into columns 16 g .. 16 g + 15 of the P buffer;
      // each half's sum is ((a0 + a1) + (a2 + a3)).
      float ps[2];
      {
        float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        uint32_t pk[16];
        attn2_exp32(r0, c2, m_use, 0, kvalid, pk, a4);
        tmem_store_16cols(trow + kAttn2P, pk);
        attn2_exp32(r1, c2, m_use, 1, kvalid, pk, a4);
        tmem_store_16cols(trow + kAttn2P + 16, pk);
        ps[0] = __fadd_rn(__fadd_rn(a4[0], a4[1]), __fadd_rn(a4[2], a4[3]));
      }
      {
        float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        uint32_t pk[16];
        attn2_exp32(r2, c2, m_use, 2, kvalid, pk, a4);
        tmem_store_16cols(trow + kAttn2P + 32, pk);
        attn2_exp32(r3, c2, m_use, 3, kvalid, pk, a4);
        tmem_store_16cols(trow + kAttn2P + 48, pk);
        ps[1] = __fadd_rn(__fadd_rn(a4[0], a4[1]), __fadd_rn(a4[2], a4[3]));
      }
      if (__any_sync(0xffffffffu, resc)) {  // O *= alpha before PV_X(j) adds to it
        const float f = resc ? alpha : 1.0f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          const uint32_t oc = trow + kAttn2O + c * 32;
          uint32_t r[32];
          tmem_load_32cols(oc, r);
          tmem_load_wait(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), f));
          tmem_store_32cols(oc, r);
        }
      }
      l0 = __fadd_rn(resc ? __fmul_rn(l0, alpha) : l0, ps[0]);
      l1 = __fadd_rn(resc ? __fmul_rn(l1, alpha) : l1, ps[1]);
      m = m_use;
      tmem_store_wait();
      signal(bars.p_full(x));
      ++pcn;
    }
    if (!ok) break;

    // Epilogue: o = RN(O * RN(1 / (l_0 + l_1))), or the split's partial O
    // and (m, l) for the merge.
    if (!wait(bars.o_full(x), ul & 1)) {
      ok = false;
      break;
    }
    ++ul;
    tc_fence_after_sync();
    const float lrow = __fadd_rn(l0, l1);
    const bool split = p.ns > 1;
    const float rinv = split ? 1.0f : __frcp_rn(lrow);
    if (split && q0 + row < p.Tq) {
      float* ml = p.ws_ml + (((int64_t)tl.sp * p.L + tl.l) * p.Tq + q0 + row) * 2;
      ml[0] = m;
      ml[1] = lrow;
    }
    if (q0 + qd * 32 < p.Tq) {
      const uint32_t region = sOut + (x * 4 + qd) * 4096;
      const int64_t qrow = q0 + qd * 32;
      const uint32_t tcol = trow + kAttn2O;
      if (split)
        attn_store_rows<D, true>(p.ws_o + (((int64_t)tl.sp * p.L + tl.l) * p.Tq + qrow) * D, D, p.Tq - qrow,
                                 tcol, 0, lane, region, rinv);
      else if (p.out_f32)
        attn_store_rows<D, true>(static_cast<float*>(p.o) + (int64_t)tl.l * p.o_l + qrow * p.o_t, p.o_t,
                                 p.Tq - qrow, tcol, 0, lane, region, rinv);
      else
        attn_store_rows<D, false>(static_cast<__nv_bfloat16*>(p.o) + (int64_t)tl.l * p.o_l + qrow * p.o_t,
                                  p.o_t, p.Tq - qrow, tcol, 0, lane, region, rinv);
    }
    signal(bars.o_free(x));
  }
}

__global__ void __launch_bounds__(kAttn2Threads, 1) attn2_kernel(const __grid_constant__ AttnParams p) {
  using C = Attn2Cfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + C::Q;
  const uint32_t sOut = base + C::OUT;
  const uint32_t sS = base + C::STG;
  const Attn2Bars bars{base + C::BARS, C::kStages};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bars.q_full(), 1);
    mbar_init(bars.q_empty(), 2);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bars.s_full(x), 1);
      mbar_init(bars.s_free(x), kAttnSoftmaxWarps / 2);
      mbar_init(bars.p_full(x), kAttnSoftmaxWarps / 2);
      mbar_init(bars.pv_done(x), 1);
      mbar_init(bars.o_full(x), 1);
      mbar_init(bars.o_free(x), kAttnSoftmaxWarps / 2);
      mbar_init(bars.drain(x), 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&p.tma_q);
    tma_prefetch_desc(&p.tma_k);
    tma_prefetch_desc(&p.tma_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kAttnTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status_word, p.wait_limit_ns};

  if (warp < 4) {
    setmaxnreg_dec<kAttn2RegsLow>();
    if (warp == 0 && lane == 0) attn2_producer(p, bars, sQ, sS, wc);
    if ((warp == 1 || warp == 2) && lane == 0) attn2_mma(p, bars, sQ, sS, tmem, warp - 1, wc);
  } else {
    setmaxnreg_inc<kAttn2RegsHigh>();
    attn2_softmax(p, bars, sOut, tmem, warp, lane, wc);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kAttnTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Merge of a split key range, one D-thread block per (head, query row),
// thread d for output column d: M = max over splits of m_s (log2 units);
// w_s = 2^(m_s - M); l = sum_s RN(w_s l_s), O_d = sum_s RN(w_s O_s,d), both in
// ascending split order; o_d = RN(O_d * RN(1 / l)), rounded once to o's type.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(D) attn_merge_kernel(const AttnParams p) {
  const int64_t rowi = blockIdx.x;  // l * Tq + q
  const int l = (int)(rowi / p.Tq);
  const int q = (int)(rowi - (int64_t)l * p.Tq);
  const int d = threadIdx.x;
  const int64_t per_split = (int64_t)p.L * p.Tq;
  float M = -INFINITY;
  for (int s = 0; s < p.ns; ++s) M = fmaxf(M, p.ws_ml[(s * per_split + rowi) * 2]);
  float lsum = 0.0f, o = 0.0f;
  for (int s = 0; s < p.ns; ++s) {
    const float w = ex2_approx(__fsub_rn(p.ws_ml[(s * per_split + rowi) * 2], M));
    const float ls = __fmul_rn(w, p.ws_ml[(s * per_split + rowi) * 2 + 1]);
    const float os = __fmul_rn(w, p.ws_o[(s * per_split + rowi) * D + d]);
    lsum = s == 0 ? ls : __fadd_rn(lsum, ls);
    o = s == 0 ? os : __fadd_rn(o, os);
  }
  const float v = __fmul_rn(o, __frcp_rn(lsum));
  char* dst = static_cast<char*>(p.o) + ((int64_t)l * p.o_l + (int64_t)q * p.o_t + d) * (p.out_f32 ? 4 : 2);
  if (p.out_f32)
    *reinterpret_cast<float*>(dst) = v;
  else
    *reinterpret_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(v);
}

int64_t attention_splits(int64_t Tk) { return Tk <= kAttnSplitKeys ? 1 : (Tk + kAttnSplitKeys - 1) / kAttnSplitKeys; }

int64_t attention_workspace_bytes(int64_t L, int64_t Tq, int64_t Tk, int64_t D) {
  const int64_t ns = attention_splits(Tk);
  return ns == 1 ? 0 : ns * L * Tq * (D + 2) * (int64_t)sizeof(float);
}

bool attention_head_dim_ok(int64_t D) { return D == 64 || D == 128 || D == 256; }

template <int D>
static cudaError_t attn_launch_d(const AttnParams& p, int64_t tiles, int num_sms, cudaStream_t stream) {
  using C = AttnCfg<D>;
  const int slot = D == 256 ? 7 : D == 128 ? 12 : 13;  // the GEMMs hold 0-3, 8-11 and 16-19
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&attn_kernel<D>), C::DYN, slot);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<int64_t>(tiles, num_sms);
  attn_kernel<D><<<grid, kAttnThreads, C::DYN, stream>>>(p);
  e = cudaGetLastError();
  if (e == cudaSuccess && p.ns > 1) {
    attn_merge_kernel<D><<<(unsigned)((int64_t)p.L * p.Tq), D, 0, stream>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

// The register split of attn2_kernel needs the registers it is launched with
// to cover both budgets; setmaxnreg.inc would wait for ever otherwise.
static bool attn2_registers_fit() {
  static int regs = -1;  // the same image serves every device
  if (regs < 0) {
    cudaFuncAttributes a;
    regs = cudaFuncGetAttributes(&a, reinterpret_cast<const void*>(&attn2_kernel)) == cudaSuccess ? a.numRegs : 0;
    cudaGetLastError();
  }
  return (uint32_t)regs * kAttn2Threads >= 128 * kAttn2RegsLow + 256 * kAttn2RegsHigh;
}

static cudaError_t attn2_launch(const AttnParams& p, int num_sms, cudaStream_t stream) {
  using C = Attn2Cfg;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&attn2_kernel), C::DYN, 14);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.units, num_sms);
  attn2_kernel<<<grid, kAttn2Threads, C::DYN, stream>>>(p);
  e = cudaGetLastError();
  if (e == cudaSuccess && p.ns > 1) {
    attn_merge_kernel<kAttn2D><<<(unsigned)((int64_t)p.L * p.Tq), kAttn2D, 0, stream>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

bi_status launch_attention(const AttnProblem& ap, cudaStream_t stream, std::string* why) {
  DeviceInfo dev;
  bi_status st = current_device_info(&dev, why);
  if (st != BI_OK) return st;
  if (!attention_head_dim_ok(ap.D)) {
    *why = "head dimension must be 64, 128 or 256";
    return BI_ERR_INVALID_ARG;
  }
  const int D = (int)ap.D;
  AttnParams p;
  memset(&p, 0, sizeof(p));
  auto map_in = [&](CUtensorMap* map, const void* ptr, int64_t T, int64_t st_t, int64_t st_l,
                    uint32_t box_rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)ap.L};
    const cuuint64_t strides[2] = {(cuuint64_t)st_t * 2, (cuuint64_t)st_l * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    return encode_tiled_bf16(map, const_cast<void*>(ptr), 3, dims, strides, box, why);
  };
  if (!map_in(&p.tma_q, ap.q, ap.Tq, ap.q_t, ap.q_l, kAttnBM) ||
      !map_in(&p.tma_k, ap.k, ap.Tk, ap.k_t, ap.k_l, kAttnBN) ||
      !map_in(&p.tma_v, ap.v, ap.Tk, ap.v_t, ap.v_l,
              D == 256 ? AttnCfg<256>::kVKeys : D == 128 ? AttnCfg<128>::kVKeys : AttnCfg<64>::kVKeys))
    return BI_ERR_CUDA;
  p.o = ap.o;
  p.o_t = ap.o_t;
  p.o_l = ap.o_l;
  p.L = (int32_t)ap.L;
  p.Tq = (int32_t)ap.Tq;
  p.Tk = (int32_t)ap.Tk;
  p.q_tiles = (int32_t)((ap.Tq + kAttnBM - 1) / kAttnBM);
  p.ns = (int32_t)attention_splits(ap.Tk);
  if (p.ns > 1) {
    const int64_t need = attention_workspace_bytes(ap.L, ap.Tq, ap.Tk, D);
    if (!ap.ws || ap.ws_bytes < need) {
      *why = "a key range longer than " + std::to_string(kAttnSplitKeys) + " needs a workspace of " +
             std::to_string(need) + " bytes";
      return BI_ERR_INVALID_ARG;
    }
    p.ws_o = static_cast<float*>(ap.ws);
    p.ws_ml = p.ws_o + p.ns * ap.L * ap.Tq * D;
  }
  const int64_t tiles = ap.L * (int64_t)p.q_tiles * p.ns;
  if (tiles > INT32_MAX) {
    *why = "tile count exceeds 2^31";
    return BI_ERR_INVALID_ARG;
  }
  p.num_tiles = (int32_t)tiles;
  p.score_log2 = (float)((double)ap.scale * 1.4426950408889634);  // scale * log2(e)
  p.out_f32 = ap.out_f32;
  p.status_word = dev.status_word;
  p.wait_limit_ns = kWaitLimitNs;
  if (p.ns > 1 && ap.L * ap.Tq > INT32_MAX) {
    *why = "too many query rows for the split merge";
    return BI_ERR_INVALID_ARG;
  }
  // Heads of 64 with at least two query tiles run two tiles per CTA; a
  // row's bits are the same in either kernel.
  const int64_t pair_units = ap.L * (int64_t)p.ns * (p.q_tiles / 2);
  const int64_t units = pair_units + (p.q_tiles % 2 ? ap.L * (int64_t)p.ns : 0);
  p.pair_units = (int32_t)pair_units;  // <= tiles
  p.units = (int32_t)units;
  const bool two = D == kAttn2D && p.q_tiles >= 2 && attn2_registers_fit();
  const cudaError_t e = D == 256   ? attn_launch_d<256>(p, tiles, dev.num_sms, stream)
                        : D == 128 ? attn_launch_d<128>(p, tiles, dev.num_sms, stream)
                        : two      ? attn2_launch(p, dev.num_sms, stream)
                                   : attn_launch_d<64>(p, tiles, dev.num_sms, stream);
  if (e != cudaSuccess) {
    *why = std::string("attention launch: ") + cudaGetErrorString(e);
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

}  // namespace bi
