/*
 * bi.h -- C ABI of the batch-invariant bf16 contraction library (GB300, sm_103a).
 *
 * Every output element's reduction over K runs in one fixed order: K blocks
 * of 64 in ascending order, each block as four 16-wide tensor-core steps, an
 * fp32 accumulator that starts from zero, then one epilogue.  The tile shape,
 * the K order and the epilogue never depend on M, on the batch count, on the
 * number of SMs or on which SM computes a tile; there is no split-K and no
 * atomic accumulation.  Consequently:
 *
 *   INVARIANCE CONTRACT.  For fixed operation, dtypes, K, N (and, for bmm /
 *   conv, the per-element shapes) and fixed operand layouts, output row m of
 *   mm/addmm depends only on row m of A (and on B, bias): its bits are the
 *   same for every M >= 1 and on every run.  The same holds per batch element
 *   for bmm, per sample for conv2d_patch and per row for softmax_lastdim.
 *
 * Sources of the operations (page title, section):
 *   mm, addmm  "Unmasking the True Culprit: Why Temperature=0 Doesn't Mean
 *              Deterministic LLM Inference", sections "The Data-Parallel
 *              Strategy" and "Implementation Analysis: The matmul_persistent
 *              Function" (fixed tiles per dtype, one CTA owns the whole K
 *              reduction of a tile, K tiles in fixed order, optional bias);
 *              "Batch-Invariant VLAs", section "Thinky's Ops were not enough"
 *              (aten::mm / aten::addmm replacements).
 *   bmm        "Batch-Invariant Kernel Design: Conv2d and Attention BMM",
 *              section "Kernel 2: Attention BMM" (rank-3 [B*H, T, D]
 *              operands, each batch element its own base pointers and the
 *              same ordered reduction over K).
 *   conv2d_patch  same page, section "Kernel 1: Conv2d", and "Batch-Invariant
 *              VLAs", section "Replacing nn.Conv2d" (per-sample unfold times
 *              the flattened filter, plus bias).
 *   softmax_lastdim  "ai-infra handbook: deterministic inference", section on
 *              making normalisation and softmax batch-independent (each row
 *              reduced by one block in a fixed order).
 *
 * General conventions (all entry points):
 *   - All tensor pointers are DEVICE pointers on the current CUDA device.
 *     The caller allocates and owns every buffer, outputs included; the
 *     library allocates no device memory.
 *   - Calls are asynchronous: they validate, enqueue kernels on `stream`
 *     (a cudaStream_t; NULL = legacy default stream) and return.
 *   - Argument, shape, dtype and layout errors are returned BEFORE any
 *     launch; outputs are then untouched.  bi_last_error_message() gives
 *     a one-line reason (thread-local).
 *   - Strides are in ELEMENTS.  Operands are read through TMA, so a matrix
 *     operand needs a unit stride on one of its two matrix dimensions, a
 *     16-byte-aligned base and 16-byte-multiple other strides; anything else
 *     returns BI_ERR_UNSUPPORTED_LAYOUT (there is no fallback path).
 *   - Device-side failures (a bounded wait that ran out) do not hang or trap:
 *     the kernel records a code and exits; bi_device_status() reports it.
 */
#ifndef BI_H_
#define BI_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* bi_stream;

typedef enum { BI_BF16 = 0, BI_F16 = 1, BI_F32 = 2 } bi_dtype;

typedef enum {
  BI_OK = 0,
  BI_ERR_INVALID_ARG = 1,        /* null pointer, bad rank, negative size ... */
  BI_ERR_SHAPE_MISMATCH = 2,     /* operand extents do not agree */
  BI_ERR_UNSUPPORTED_DTYPE = 3,  /* a dtype this operation does not take */
  BI_ERR_UNSUPPORTED_LAYOUT = 4, /* strides / alignment TMA cannot read */
  BI_ERR_CUDA = 5,               /* a CUDA runtime or driver call failed */
  BI_ERR_TIMEOUT = 6,            /* a device-side bounded wait ran out */
  BI_ERR_NO_DEVICE = 7           /* no usable sm_100-family device */
} bi_status;

/* A strided view of device memory.  shape/stride entries past ndim are ignored. */
typedef struct {
  void* ptr;          /* device address of element [0,...,0]; NULL = absent */
  int32_t ndim;       /* 1..4 */
  int32_t dtype;      /* a bi_dtype value */
  int64_t shape[4];
  int64_t stride[4];  /* in elements */
} bi_tensor;

/*
 * c[m,n] = sum_k a[m,k] * b[k,n]
 *   a: [M,K] bf16 or fp16, unit stride on K (row-major activations).
 *   b: [K,N] of the same type as a, unit stride on N (row-major weight) or on
 *      K (a transposed view of an [N,K] weight, as torch.nn.functional.linear
 *      stores it).  Mixed bf16 / fp16 operands return BI_ERR_UNSUPPORTED_DTYPE.
 *   c: [M,N] fp32, bf16 or fp16, unit stride on N; written, never read.
 *   M, N, K >= 1.  The fp32 accumulator is rounded once to c's dtype (RNE).
 *   fp16 inputs run the same tile and K order as bf16 inputs (the tensor
 *   core's f16 kind, one format for both operands).
 */
bi_status bi_mm(const bi_tensor* a, const bi_tensor* b, const bi_tensor* c, bi_stream stream);

/*
 * c[m,n] = (sum_k a[m,k] * b[k,n]) + bias[n]   (alpha = beta = 1)
 *   bias: [N] bf16, fp16 or fp32, any stride; added to the fp32 accumulator
 *   after the full K reduction, then one rounding to c's dtype.  Operand
 *   types and layouts as bi_mm.
 */
bi_status bi_addmm(const bi_tensor* bias, const bi_tensor* a, const bi_tensor* b,
                   const bi_tensor* c, bi_stream stream);

/*
 * c[l,m,n] = alpha * sum_k a[l,m,k] * b[l,k,n]   for l in [0, L)
 *   a: [L,M,K] bf16 or fp16, unit stride on K;  b: [L,K,N] of the same type,
 *   unit stride on N or on K (so Q @ K^T passes K^T as a stride view);
 *   c: [L,M,N] fp32, bf16 or fp16, unit stride on N.  The fp32 accumulator is
 *   multiplied by alpha (fp32), then rounded once.  Each l is an independent
 *   product.
 */
bi_status bi_bmm(const bi_tensor* a, const bi_tensor* b, const bi_tensor* c, float alpha,
                 bi_stream stream);

/*
 * y = conv2d(x, w, bias), non-transposed, cross-correlation (as nn.Conv2d):
 *   y[b,co,oh,ow] = bias[co] + sum_{ci,kh,kw} x[b, g*Cig+ci, oh*sh-ph+kh*dh, ow*sw-pw+kw*dw]
 *                                             * w[co, ci, kh, kw]
 *   with g = co / (Co/groups), out-of-image positions reading zero, and the
 *   reduction index k = (ci*KH + kh)*KW + kw (the unfold order) ascending.
 *   x: [B,C,H,W] bf16 contiguous;  w: [Co,C/groups,KH,KW] bf16 contiguous;
 *   bias: [Co] bf16 or fp32, or NULL / ptr == NULL for none;
 *   y: [B,Co,Ho,Wo] bf16 or fp32 contiguous, Ho = (H+2ph-dh(KH-1)-1)/sh+1.
 *   stride, padding, dilation: {h, w}.  Each sample is computed as its own
 *   implicit-im2col product (the patch gather happens in shared memory).
 *   Non-overlapping patches -- stride = (KH, KW), padding 0, dilation 1, one
 *   group, KW even and <= 16, W a multiple of 8 and <= 256, W/KW <= 128, x
 *   16-byte and w 4-byte aligned -- run the patch kernel of
 *   bi_conv2d_patch_packed straight from w (its filter stages are built from
 *   w in shared memory; nothing is allocated) and give its bits: each
 *   tensor-core K = 16 step is one kernel row (ci, kh), kw padded with exact
 *   zeros.  Every other geometry sums k in steps of 16 of the unfold order.
 *   Which of the two runs is a function of the geometry and of the two
 *   pointers' alignment, never of B (a batch slice of an aligned x stays
 *   aligned); the two groupings agree within rounding, not bit for bit.
 */
bi_status bi_conv2d_patch(const bi_tensor* x, const bi_tensor* w, const bi_tensor* bias,
                          const bi_tensor* y, const int32_t stride[2], const int32_t padding[2],
                          const int32_t dilation[2], int32_t groups, bi_stream stream);

/*
 * Packed patch-embedding filter, for bi_conv2d_patch_packed.  The filter
 * w[Co][C][KH][KW] of a non-overlapping patch convolution stored as a
 * row-major [Co][Kp] bf16 matrix with reduction index
 *   kp = (ci*KHp + kh)*16 + kw,   KHp = KH rounded up to a multiple of 4,
 * i.e. every kernel row (ci, kh) padded to 16 slots and every channel to a
 * multiple of 4 kernel rows; slots with kh >= KH or kw >= KW hold zero.
 * Packing is a data-layout service for the same convolution, not one of the
 * pages' operations.
 */
typedef struct {
  void* ptr;              /* device buffer holding the packed filter (caller-owned) */
  int64_t bytes;          /* its size in bytes */
  int64_t Co, C, KH, KW;  /* shape of the filter it was packed from */
  int64_t Kp;             /* row length C * KHp * 16 */
} bi_conv_packed_weight;

/* Bytes of the packed form of a [Co,C,KH,KW] filter (0 if KW > 16 or empty). */
int64_t bi_conv_packed_weight_bytes(int64_t Co, int64_t C, int64_t KH, int64_t KW);

/*
 * Packs w ([Co,C,KH,KW] bf16 contiguous, KW <= 16) into dst (device, 16-byte
 * aligned, dst_bytes >= bi_conv_packed_weight_bytes(...)); fills *out.
 * Asynchronous on `stream`.
 */
bi_status bi_conv_pack_weight(const bi_tensor* w, void* dst, int64_t dst_bytes,
                              bi_conv_packed_weight* out, bi_stream stream);

/*
 * y = conv2d(x, w, bias, stride = (KH, KW), padding 0, dilation 1, groups 1)
 * -- the patch embedding of "Batch-Invariant VLAs", section "Replacing
 * nn.Conv2d" -- with w given packed:
 *   y[b,co,oh,ow] = bias[co] + sum_{ci,kh,kw} x[b, ci, oh*KH+kh, ow*KW+kw] * w[co,ci,kh,kw]
 * The reduction runs over the packed index kp in ascending order; each
 * tensor-core K = 16 step is one kernel row (ci, kh) (its zero slots add
 * exact zeros; image pixels outside a position's own window are never read
 * into it).  Per output element this is a fixed order, the same for every
 * batch size, and the same as bi_conv2d_patch's for the geometries that
 * bi_conv2d_patch runs on the patch kernel (bit for bit).
 *   x: [B,C,H,W] bf16 contiguous, 16-byte aligned, W a multiple of 8 and
 *      <= 256;  y: [B,Co,H/KH,W/KW] bf16 or fp32 contiguous, W/KW <= 128;
 *   bias: [Co] bf16 or fp32, or NULL / ptr == NULL.  Image rows or columns
 *   past the last whole patch are ignored (as the size formula does).
 */
bi_status bi_conv2d_patch_packed(const bi_tensor* x, const bi_conv_packed_weight* w,
                                 const bi_tensor* bias, const bi_tensor* y, bi_stream stream);

/*
 * p[r,:] = softmax(s[r,:]) over the last dimension, per row r:
 *   mx = max_j s[r,j];  e_j = expf(s[r,j] - mx);  p[r,j] = e_j * RN(1 / sum_j e_j),
 *   sums in fp32 in a fixed order set by the element index only (4-element
 *   groups g, lane g mod 32 of one warp, then a fixed butterfly).
 *   s: [R,N] fp32, unit stride on N;  p: [R,N] bf16 or fp32, unit stride on N.
 */
bi_status bi_softmax_lastdim(const bi_tensor* s, const bi_tensor* p, bi_stream stream);

/*
 * Fused attention, per head l and query row i:
 *   o[l,i,:] = sum_j softmax_j(scale * q[l,i,:] . k[l,j,:]) v[l,j,:]
 * in one kernel, the scores and probabilities never written to memory
 * ("ai-infra handbook: deterministic inference", section on fixed splitting:
 * attention's key range is not split by load -- here not split at all -- and
 * a query row's result does not depend on how queries are chunked).  Per
 * query row: key blocks of 128 in ascending order; scores from a fixed
 * sequence of tensor-core steps over the head dimension (fp32); t = RN(s * c)
 * with c = RN(scale * log2 e); a running maximum m, replaced only when a block
 * raises it by more than 8; p = 2^(t - m) (the SFU's approximation);
 * l = RN(l * 2^(m_old - m_new)) + sum p (keys ascending); O accumulated in
 * fp32 from bf16(p) v in key order (rescaled with m); o = RN(O * RN(1/l)),
 * rounded once to o's type.  None of it depends on L, Tq, the tile a row
 * falls in or the SM count: a head alone gives the bits it gives in any
 * batch, and a query row the bits it gives among any other query rows.
 *   q: [L,Tq,D], k and v: [L,Tk,D], bf16, unit stride on the head
 *   dimension, 16-byte aligned bases, row and batch strides multiples of 16
 *   bytes;  o: [L,Tq,D] fp32 or bf16 (same layout rules);  scale finite.
 *   Head dimension D = 64, 128 or 256 (BI_ERR_INVALID_ARG otherwise); Tk >= 1
 *   (BI_ERR_INVALID_ARG otherwise); L == 0 or Tq == 0 launches nothing.
 *   Non-causal, no mask.
 */
bi_status bi_attention(const bi_tensor* q, const bi_tensor* k, const bi_tensor* v, float scale,
                       const bi_tensor* o, bi_stream stream);

/*
 * Long key ranges.  When Tk > 2048 the key range is split into fixed
 * 2048-key pieces ("ai-infra handbook: deterministic inference", section on
 * fixed splitting: a split by a fixed length, never by load, keeps attention
 * batch-invariant -- the split depends on Tk only).  Each (head, 128 query
 * rows, split) is one work unit of the kernel above, which writes its partial
 * O (relative to its own running maximum m_s) and (m_s, l_s) to a workspace;
 * a merge kernel then forms, per row, M = max_s m_s, w_s = 2^(m_s - M),
 * l = sum_s RN(w_s l_s), O = sum_s RN(w_s O_s) (splits in ascending order)
 * and o = RN(O * RN(1 / l)).  Tk <= 2048 is not split and needs no
 * workspace; bi_attention refuses a longer key range (BI_ERR_INVALID_ARG).
 *
 * Bytes of workspace bi_attention_ws needs for [L, Tq] queries against Tk
 * keys of head dimension D: 0 when Tk <= 2048 (or any argument is out of
 * range), else ceil(Tk / 2048) * L * Tq * (D + 2) * 4.
 */
int64_t bi_attention_workspace_bytes(int64_t L, int64_t Tq, int64_t Tk, int64_t D);

/*
 * bi_attention with a caller-owned device workspace (16-byte aligned, at
 * least bi_attention_workspace_bytes(L, Tq, Tk, D) bytes; may be NULL when that
 * is 0).  The workspace is scratch: its contents on entry do not matter and
 * on return are unspecified; it must not be used by other work on the device
 * while the call's kernels run (stream order).  Results for Tk <= 2048 are
 * those of bi_attention, bit for bit.
 */
bi_status bi_attention_ws(const bi_tensor* q, const bi_tensor* k, const bi_tensor* v, float scale,
                          const bi_tensor* o, void* workspace, int64_t workspace_bytes, bi_stream stream);

/*
 * bi_attention_ws without a caller workspace: a split key range uses a
 * scratch area the library keeps in static device memory (64 MiB per device,
 * 256-byte aligned, allocated when the library's module is loaded on the
 * device).  A problem whose workspace would not fit returns
 * BI_ERR_INVALID_ARG before any launch (use bi_attention_ws).  The scratch is
 * shared by every call on the device, so calls must not overlap: issue them
 * on one stream or order them.  Results are those of bi_attention_ws, bit
 * for bit.  The scratch's device address is looked up (cudaGetSymbolAddress)
 * on the first call on each device and again whenever that device's CUDA
 * context has been replaced (after cudaDeviceReset); that first call should
 * come before any stream capture.  No call allocates or frees device memory.
 * The pages have no counterpart of this entry point: it packages the same
 * operation for callers that cannot allocate device memory -- a serving
 * engine whose allocator reserves all device memory up front and gives no
 * library a way around it, or code that may not call cudaMalloc / cudaFree
 * because those synchronise the device.
 */
bi_status bi_attention_noalloc(const bi_tensor* q, const bi_tensor* k, const bi_tensor* v, float scale,
                               const bi_tensor* o, bi_stream stream);

/*
 * Row reductions over the last dimension -- the normalisation, log-softmax
 * and mean operations that "Unmasking the True Culprit: Why Temperature=0
 * Doesn't Mean Deterministic LLM Inference" (section "Beyond Matrix
 * Multiplication: Other Critical Operations") and "Batch-Invariant VLAs"
 * (aten::mean.dim) say must reduce each row in one fixed order.  A row of N
 * elements is reduced by a team of T threads, T chosen from N and the input
 * type alone: the first of 32, 64, 256, 1024 with N <= 4*G*T, G = 16 for
 * 16-bit inputs and 8 for fp32.  The row is cut into groups of 4 consecutive
 * elements; thread t adds the elements of groups t, t+T, t+2T, ... in
 * ascending index order in fp32, each warp combines its 32 partials by a
 * fixed xor butterfly, and the warp partials are added in warp order.  Rows
 * longer than 4096*G elements are split, by N alone, over a cluster of
 * cl = ceil(N / (4096*G)) <= 8 CTAs of 1024 threads: CTA r reduces the r-th
 * of cl equal contiguous slices of the row's groups as above, and the cl
 * slice totals are added in rank order.  The order therefore depends on N,
 * the input type and the element index only -- not on how many rows are
 * reduced together, on where the row sits in memory (aligned rows are loaded
 * 4 elements at a time, others one at a time, with the same arithmetic) or
 * on the launch.  Each add, multiply, divide and square root is one
 * separately rounded fp32 operation; the output is rounded once to its type.
 *
 * All three: x (or s): [R,N] bf16, fp16 or fp32 with a unit stride on N,
 * aligned to its element size, N <= 2^24; outputs of any of the three types.
 * Asynchronous on `stream`; R == 0 (or N == 0 for the first two) launches
 * nothing.  Shape, layout or type errors are returned before any launch.
 */

/*
 * y[r,j] = RN(RN(x[r,j] * inv) * weight[j]),
 *   inv = RN(1 / RN(sqrt(RN(RN(sum_j x[r,j]^2) / N) + eps))),
 * the multiply by weight left out when weight is NULL (or weight->ptr is
 * NULL).  weight: [N] of any of the three types, any stride; y: [R,N], unit
 * stride on N; eps finite and >= 0 (BI_ERR_INVALID_ARG otherwise).
 */
bi_status bi_rmsnorm_lastdim(const bi_tensor* x, const bi_tensor* weight, float eps,
                             const bi_tensor* y, bi_stream stream);

/*
 * y[r,j] = RN(RN(s[r,j] - mx) - lse),  mx = max_j s[r,j],
 *   lse = logf(sum_j expf(RN(s[r,j] - mx))).
 * y: [R,N], unit stride on N.  For 1024-thread teams, when the rows' clusters
 * are more than the GPU runs at once with each thread holding its groups in
 * registers, each pass reloads them instead (two CTAs per SM); the order
 * above, and so every bit, is the same either way.
 */
bi_status bi_log_softmax_lastdim(const bi_tensor* s, const bi_tensor* y, bi_stream stream);

/*
 * y[r] = RN(RN(sum_j x[r,j]) / N).  y: [R], any stride.  N == 0 with R > 0
 * is BI_ERR_INVALID_ARG (the mean of an empty row).
 */
bi_status bi_mean_lastdim(const bi_tensor* x, const bi_tensor* y, bi_stream stream);

/*
 * Packed weights -- for products whose B operand is a fixed weight streamed
 * from HBM many times (decode-sized M).  Packing stores B as the exact
 * sequence of 128-byte-swizzled 64 x 64 shared-memory tile images the kernel
 * would otherwise assemble with strided TMA loads, ordered [k block][64-column
 * chunk] and zero-padded to whole output tiles, so one pipeline stage of B is
 * one contiguous range moved by a single bulk copy.  The tensor core reads the
 * same shared-memory bytes either way: results with a packed weight are bit
 * identical to results with the plain weight.  Packing is not one of the
 * pages' operations; it is a data-layout service for the same product.
 */
typedef struct {
  void* ptr;        /* device buffer holding the packed form (caller-owned) */
  int64_t bytes;    /* its size in bytes */
  int64_t K, N;     /* logical shape of the packed [K, N] weight */
  int32_t layout;   /* 1: images of a row-major [K,N] weight, 2: of a [N,K] (transposed view) */
  int32_t tile_n;   /* output-tile width the packing was made for (must match the library) */
  int32_t dtype;    /* element type of the weight: BI_BF16 or BI_F16 */
} bi_packed_weight;

/* Bytes needed to pack a [K, N] bf16 weight (0 for an empty one). */
int64_t bi_packed_weight_bytes(int64_t K, int64_t N);

/*
 * Packs b ([K,N] bf16 or fp16 on the device, unit stride on N or on K, 16-byte aligned
 * base and 16-byte multiple other stride) into dst (device, 16-byte aligned,
 * dst_bytes >= bi_packed_weight_bytes(K, N)); fills *out.  Asynchronous on
 * `stream`; dst must not be used before the packing has run.
 */
bi_status bi_pack_weight(const bi_tensor* b, void* dst, int64_t dst_bytes, bi_packed_weight* out,
                         bi_stream stream);

/*
 * c[m,n] = sum_k a[m,k] * B[k,n] (+ bias[n] when bias is non-NULL with a
 * non-NULL ptr), B given in packed form.  a: [M,K] of the packed weight's
 * type, as in bi_mm; c: [M,N] fp32, bf16 or fp16; bias: [N] bf16, fp16 or
 * fp32.  Same arithmetic, same bits as bi_mm / bi_addmm on the unpacked weight.
 */
bi_status bi_addmm_packed(const bi_tensor* bias, const bi_tensor* a, const bi_packed_weight* b,
                          const bi_tensor* c, bi_stream stream);

/*
 * Synchronises `stream`, then returns and clears the device-side status word
 * of the current device: BI_OK, or BI_ERR_TIMEOUT when a kernel's bounded
 * wait ran out since the last call (detail in bi_last_error_message()).
 */
bi_status bi_device_status(bi_stream stream);

/*
 * Test hook for the failure path: launches one block that waits, with a
 * limit of `limit_ns` nanoseconds (1 ms .. 2 s), on a barrier that nothing
 * ever signals.  The wait runs out, the kernel records BI_ERR_TIMEOUT and
 * exits normally; the next bi_device_status() returns it.
 */
bi_status bi_debug_expire_wait(uint64_t limit_ns, bi_stream stream);

/* Static, human-readable name of a status code. */
const char* bi_status_string(bi_status status);

/* Reason for the last non-OK status returned on this thread ("" if none). */
const char* bi_last_error_message(void);

/* ABI version of this header (incremented on any signature change). */
int32_t bi_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BI_H_ */
