// bi_abi.cu -- the C ABI declared in include/bi.h: argument validation (all of
// it before any launch), operand-layout normalisation, per-device state (SM
// count, the device status word), TMA descriptor encoding and error reporting.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>
#include <string>

#include "../../include/bi.h"
#include "bi_common.h"
#include "bi_launch.h"

// First device-side failure since the last bi_device_status() (0 = none).
__device__ unsigned int g_bi_status_word;

// Static device scratch of bi_attention_noalloc (each device's context holds
// its own copy).  Uninitialised: it costs device memory at module load, not
// space in the library file.
constexpr int64_t kNoAllocScratchBytes = 64ll << 20;
__device__ __align__(256) unsigned char g_bi_noalloc_scratch[kNoAllocScratchBytes];

namespace bi {

namespace {

thread_local std::string t_last_error;
std::mutex g_mu;

constexpr int kMaxDevices = 64;
// What the library caches per device belongs to one CUDA context (the device
// addresses of its __device__ variables, kernel attributes): it is dropped and
// resolved again when the device's current context is another one, as after
// cudaDeviceReset and the primary context's re-creation.
struct DevState {
  bool ready = false;
  unsigned long long ctx_id = 0;  // the context the entries below were resolved in
  bi_status status = BI_OK;
  std::string why;
  int num_sms = 0;
  unsigned int* status_word = nullptr;
  bool smem_set[24] = {};
  int pairs[24] = {};  // resident 2-CTA clusters per kernel slot (0: not yet asked)
  void* scratch = nullptr;  // device address of g_bi_noalloc_scratch (0: not yet asked)
};
DevState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
bool g_ctx_tried = false;

// Unique id of the calling thread's current CUDA context; 0 when none is
// current (or the driver cannot say).  Caller holds g_mu.
unsigned long long current_context_id() {
  if (!g_ctx_tried) {
    g_ctx_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    cudaGetLastError();
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!g_ctx_current || !g_ctx_id || g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx ||
      g_ctx_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

bi_status finish(bi_status st, const std::string& why) {
  t_last_error = (st == BI_OK) ? std::string() : why;
  return st;
}

}  // namespace

bi_status current_device_info(DeviceInfo* info, std::string* why) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0) {
    *why = std::string("no CUDA device: ") + cudaGetErrorString(e);
    cudaGetLastError();
    return BI_ERR_NO_DEVICE;
  }
  if (dev >= kMaxDevices) {
    *why = "device ordinal out of range";
    return BI_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& d = g_dev[dev];
  unsigned long long ctx = current_context_id();
  if (ctx == 0) {
    // No context is current on this thread yet: the runtime binds the
    // device's primary context on first use, which this lookup is.
    void* addr = nullptr;
    cudaGetSymbolAddress(&addr, g_bi_status_word);
    cudaGetLastError();
    ctx = current_context_id();
  }
  if (d.ready && ctx != 0 && ctx != d.ctx_id) d = DevState();
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) {
      d.status = BI_ERR_NO_DEVICE;
      d.why = "device " + std::to_string(dev) + " has compute capability " + std::to_string(major) +
              "." + std::to_string(minor) + "; this library is built for sm_103a only";
    } else {
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_bi_status_word);
      if (e != cudaSuccess) {
        d.status = BI_ERR_CUDA;
        d.why = std::string("status word: ") + cudaGetErrorString(e);
      } else {
        d.status = BI_OK;
        d.num_sms = sms;
        d.status_word = reinterpret_cast<unsigned int*>(addr);
        d.ctx_id = current_context_id();
      }
    }
    d.ready = true;
  }
  if (d.status != BI_OK) {
    *why = d.why;
    return d.status;
  }
  info->device = dev;
  info->num_sms = d.num_sms;
  info->status_word = d.status_word;
  return BI_OK;
}

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle,
                  void* ptr, uint32_t rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                  const cuuint32_t* box, std::string* why) {
  const cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode_tried) {
      g_encode_tried = true;
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) == cudaSuccess &&
          q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      cudaGetLastError();
    }
  }
  if (!g_encode) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  CUresult r = g_encode(map, dtype, rank, ptr, dims, strides_bytes, box, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

bool encode_output_map(CUtensorMap* map, void* c, bool f32, bool f16, int64_t L, int64_t M, int64_t N,
                       int64_t ldc, int64_t c_batch) {
  const uint64_t esz = f32 ? 4 : 2;
  const uint64_t row = (uint64_t)ldc * esz;
  const uint64_t bat = L > 1 ? (uint64_t)c_batch * esz : round_up_u64(row * (uint64_t)M, 16);
  if (reinterpret_cast<uintptr_t>(c) % 16 != 0 || row % 16 != 0 || bat % 16 != 0 || row == 0 ||
      bat == 0 || M > INT32_MAX || N > INT32_MAX || L > INT32_MAX)
    return false;
  const cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)L};
  const cuuint64_t strides[2] = {row, bat};
  const cuuint32_t box[3] = {32, 32, 1};
  std::string why;
  return encode_tiled(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                             : (f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16),
                      f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, c, 3, dims,
                      strides, box, &why);
}

cudaError_t set_smem_once(const void* func, int bytes, int slot) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& d = g_dev[dev];
  if (d.smem_set[slot]) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) d.smem_set[slot] = true;
  return e;
}

cudaError_t pair_capacity(const void* func, int threads, int dyn_bytes, int slot, int* pairs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev[dev].pairs[slot] > 0) {
      *pairs = g_dev[dev].pairs[slot];
      return cudaSuccess;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = dyn_bytes;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, func, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) n = 1;
  std::lock_guard<std::mutex> lk(g_mu);
  g_dev[dev].pairs[slot] = n;
  *pairs = n;
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// Validation helpers
// ---------------------------------------------------------------------------
namespace {

int elem_size(int dtype) { return dtype == BI_F32 ? 4 : 2; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bi_status check_tensor(const bi_tensor* t, const char* name, int ndim, std::string* why) {
  if (!t) {
    *why = std::string(name) + ": null tensor descriptor";
    return BI_ERR_INVALID_ARG;
  }
  if (t->ndim != ndim) {
    *why = std::string(name) + ": expected rank " + std::to_string(ndim) + ", got " +
           std::to_string(t->ndim);
    return BI_ERR_INVALID_ARG;
  }
  if (t->dtype != BI_BF16 && t->dtype != BI_F16 && t->dtype != BI_F32) {
    *why = std::string(name) + ": unknown dtype code " + std::to_string(t->dtype);
    return BI_ERR_UNSUPPORTED_DTYPE;
  }
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0 || t->shape[i] > INT32_MAX) {
      *why = std::string(name) + ": dimension " + std::to_string(i) + " out of range";
      return BI_ERR_INVALID_ARG;
    }
    if (t->stride[i] < 0) {
      *why = std::string(name) + ": negative strides are not supported";
      return BI_ERR_UNSUPPORTED_LAYOUT;
    }
  }
  return BI_OK;
}

bi_status need_ptr(const bi_tensor* t, const char* name, std::string* why) {
  if (!t->ptr) {
    *why = std::string(name) + ": null data pointer";
    return BI_ERR_INVALID_ARG;
  }
  return BI_OK;
}

bool is_contiguous(const bi_tensor* t) {
  int64_t expect = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] != 1 && t->stride[i] != expect) return false;
    expect *= t->shape[i];
  }
  return true;
}

// B: unit stride on N (MN-major) or on K (K-major, a transposed view);
// 16-byte aligned base, 16-byte multiple non-unit strides.
bi_status normalize_b(const bi_tensor* b, int o, int64_t L, int64_t K, int64_t N, bool batched,
                      GemmProblem* g, std::string* why) {
  const bool mn_ok = (N == 1) || b->stride[o + 1] == 1;
  const bool k_ok = (K == 1) || b->stride[o] == 1;
  g->b = b->ptr;
  g->b_batch = batched ? b->stride[0] : 0;
  if (mn_ok && (N > 1 || !k_ok)) {
    g->b_mn_major = 1;
    g->ldb = (K == 1) ? (int64_t)round_up_u64((uint64_t)N, 8) : b->stride[o];
  } else if (k_ok) {
    g->b_mn_major = 0;
    g->ldb = (N == 1) ? (int64_t)round_up_u64((uint64_t)K, 8) : b->stride[o + 1];
  } else {
    *why = "b needs a unit stride on N or on K";
    return BI_ERR_UNSUPPORTED_LAYOUT;
  }
  if (!aligned(b->ptr, 16) || (g->ldb * 2) % 16 != 0 || g->ldb == 0 ||
      (L > 1 && ((g->b_batch * 2) % 16 != 0 || g->b_batch == 0))) {
    *why = "b: base must be 16-byte aligned and its non-unit strides multiples of 8 elements";
    return BI_ERR_UNSUPPORTED_LAYOUT;
  }
  return BI_OK;
}

// Shared by mm / addmm (batched = false) and bmm (batched = true); with
// `packed`, B comes from a packed weight instead of the tensor b.
bi_status matmul_impl(const bi_tensor* bias, const bi_tensor* a, const bi_tensor* b,
                      const bi_tensor* c, float alpha, bool batched, cudaStream_t stream,
                      std::string* why, const bi_packed_weight* packed = nullptr) {
  const int nd = batched ? 3 : 2;
  bi_status st;
  // A packed weight stands in for b as a [K, N] operand of its element type.
  bi_tensor pb;
  if (packed) {
    memset(&pb, 0, sizeof(pb));
    pb.ptr = packed->ptr;
    pb.ndim = 2;
    pb.dtype = packed->dtype;
    if (packed->dtype != BI_BF16 && packed->dtype != BI_F16) {
      *why = "packed weight: unknown element type";
      return BI_ERR_INVALID_ARG;
    }
    pb.shape[0] = packed->K;
    pb.shape[1] = packed->N;
    pb.stride[0] = packed->N;
    pb.stride[1] = 1;
    b = &pb;
  }
  if ((st = check_tensor(a, "a", nd, why)) != BI_OK) return st;
  if ((st = check_tensor(b, "b", nd, why)) != BI_OK) return st;
  if ((st = check_tensor(c, "c", nd, why)) != BI_OK) return st;
  // One input type for both operands: the tensor core's kind::f16 product
  // takes A and B of the same format (mixing them is refused here, before
  // anything reaches the GPU).
  if (!((a->dtype == BI_BF16 && b->dtype == BI_BF16) || (a->dtype == BI_F16 && b->dtype == BI_F16))) {
    *why = "a and b must both be bf16 or both be fp16";
    return BI_ERR_UNSUPPORTED_DTYPE;
  }
  if (c->dtype != BI_BF16 && c->dtype != BI_F32 && c->dtype != BI_F16) {
    *why = "c must be bf16, fp16 or fp32";
    return BI_ERR_UNSUPPORTED_DTYPE;
  }
  const int o = batched ? 1 : 0;  // offset of the matrix dims
  const int64_t L = batched ? a->shape[0] : 1;
  const int64_t M = a->shape[o], K = a->shape[o + 1];
  const int64_t N = b->shape[o + 1];
  if (b->shape[o] != K) {
    *why = "inner dimensions differ: a has K=" + std::to_string(K) + ", b has K=" +
           std::to_string(b->shape[o]);
    return BI_ERR_SHAPE_MISMATCH;
  }
  if (c->shape[o] != M || c->shape[o + 1] != N ||
      (batched && (b->shape[0] != L || c->shape[0] != L))) {
    *why = "output / batch extents do not match the operands";
    return BI_ERR_SHAPE_MISMATCH;
  }
  int bias_kind = 0;
  int64_t bias_stride = 0;
  if (bias && bias->ptr) {
    if ((st = check_tensor(bias, "bias", 1, why)) != BI_OK) return st;
    if (bias->shape[0] != N) {
      *why = "bias must have N elements";
      return BI_ERR_SHAPE_MISMATCH;
    }
    if (bias->dtype == BI_BF16)
      bias_kind = 1;
    else if (bias->dtype == BI_F32)
      bias_kind = 2;
    else
      bias_kind = 3;  // fp16 (check_tensor admits no other code)
    bias_stride = bias->stride[0];
    if (!aligned(bias->ptr, elem_size(bias->dtype))) {
      *why = "bias pointer is not aligned to its element size";
      return BI_ERR_UNSUPPORTED_LAYOUT;
    }
  }
  if (L == 0 || M == 0 || N == 0) return BI_OK;  // nothing to compute
  if ((st = need_ptr(c, "c", why)) != BI_OK) return st;

  GemmProblem g;
  memset(&g, 0, sizeof(g));
  g.L = L;
  g.M = M;
  g.N = N;
  g.K = K;
  g.alpha = alpha;
  g.bias = bias_kind ? bias->ptr : nullptr;
  g.bias_kind = bias_kind;
  g.bias_stride = bias_stride;
  g.c = c->ptr;
  g.out_f32 = c->dtype == BI_F32;
  g.out_f16 = c->dtype == BI_F16;
  g.in_f16 = a->dtype == BI_F16;
  const int cesz = elem_size(c->dtype);
  if (!(N == 1 || c->stride[o + 1] == 1)) {
    *why = "c needs a unit stride on N";
    return BI_ERR_UNSUPPORTED_LAYOUT;
  }
  g.ldc = (M == 1) ? N : c->stride[o];
  g.c_batch = batched ? c->stride[0] : 0;
  if (!aligned(c->ptr, cesz)) {
    *why = "c pointer is not aligned to its element size";
    return BI_ERR_UNSUPPORTED_LAYOUT;
  }
  g.vec_store = aligned(c->ptr, 16) && (g.ldc * cesz) % 16 == 0 &&
                (L <= 1 || (g.c_batch * cesz) % 16 == 0);

  if (K == 0) return launch_fill_bias(g, stream, why);

  if ((st = need_ptr(a, "a", why)) != BI_OK) return st;
  if ((st = need_ptr(b, "b", why)) != BI_OK) return st;

  // A: unit stride on K; row stride a 16-byte multiple; 16-byte aligned base.
  if (!(K == 1 || a->stride[o + 1] == 1)) {
    *why = "a needs a unit stride on K (row-major activations)";
    return BI_ERR_UNSUPPORTED_LAYOUT;
  }
  g.a = a->ptr;
  g.lda = (M == 1) ? (int64_t)round_up_u64((uint64_t)K, 8) : a->stride[o];
  g.a_batch = batched ? a->stride[0] : 0;
  if (!aligned(a->ptr, 16) || (g.lda * 2) % 16 != 0 || g.lda == 0 ||
      (L > 1 && ((g.a_batch * 2) % 16 != 0 || g.a_batch == 0))) {
    *why = "a: base must be 16-byte aligned and its row / batch strides multiples of 8 elements";
    return BI_ERR_UNSUPPORTED_LAYOUT;
  }
  if (packed) {
    if (packed->layout != 1 && packed->layout != 2) {
      *why = "packed weight: unknown layout";
      return BI_ERR_INVALID_ARG;
    }
    if (packed->tile_n != kBN) {
      *why = "packed weight was made for another tile width";
      return BI_ERR_INVALID_ARG;
    }
    if (!aligned(packed->ptr, 16) || packed->bytes < packed_bytes(K, N)) {
      *why = "packed weight: buffer not 16-byte aligned or too small";
      return BI_ERR_INVALID_ARG;
    }
    g.b_packed = packed->ptr;
    g.b_mn_major = packed->layout == 1;
    return launch_gemm(g, stream, why);
  }
  if ((st = normalize_b(b, o, L, K, N, batched, &g, why)) != BI_OK) return st;
  return launch_gemm(g, stream, why);
}

}  // namespace
}  // namespace bi

// ---------------------------------------------------------------------------
// C entry points
// ---------------------------------------------------------------------------
using namespace bi;

extern "C" bi_status bi_mm(const bi_tensor* a, const bi_tensor* b, const bi_tensor* c,
                           bi_stream stream) {
  std::string why;
  bi_status st = matmul_impl(nullptr, a, b, c, 1.0f, false, (cudaStream_t)stream, &why);
  return finish(st, why);
}

extern "C" bi_status bi_addmm(const bi_tensor* bias, const bi_tensor* a, const bi_tensor* b,
                              const bi_tensor* c, bi_stream stream) {
  std::string why;
  bi_status st;
  if (!bias || !bias->ptr) {
    why = "bias: null (use bi_mm for a product without bias)";
    st = BI_ERR_INVALID_ARG;
  } else {
    st = matmul_impl(bias, a, b, c, 1.0f, false, (cudaStream_t)stream, &why);
  }
  return finish(st, why);
}

extern "C" bi_status bi_bmm(const bi_tensor* a, const bi_tensor* b, const bi_tensor* c,
                            float alpha, bi_stream stream) {
  std::string why;
  bi_status st = matmul_impl(nullptr, a, b, c, alpha, true, (cudaStream_t)stream, &why);
  return finish(st, why);
}

extern "C" int64_t bi_packed_weight_bytes(int64_t K, int64_t N) { return packed_bytes(K, N); }

extern "C" bi_status bi_pack_weight(const bi_tensor* b, void* dst, int64_t dst_bytes,
                                    bi_packed_weight* out, bi_stream stream) {
  std::string why;
  bi_status st;
  if ((st = check_tensor(b, "b", 2, &why)) != BI_OK) return finish(st, why);
  if (b->dtype != BI_BF16 && b->dtype != BI_F16) return finish(BI_ERR_UNSUPPORTED_DTYPE, "b must be bf16 or fp16");
  if (!out) return finish(BI_ERR_INVALID_ARG, "out: null");
  const int64_t K = b->shape[0], N = b->shape[1];
  if (K == 0 || N == 0) return finish(BI_ERR_INVALID_ARG, "empty weight");
  const int64_t need = packed_bytes(K, N);
  if (!dst || !aligned(dst, 16) || dst_bytes < need)
    return finish(BI_ERR_INVALID_ARG, "dst must be 16-byte aligned with at least " +
                                          std::to_string(need) + " bytes");
  if (!b->ptr) return finish(BI_ERR_INVALID_ARG, "b: null data pointer");
  GemmProblem g;
  memset(&g, 0, sizeof(g));
  g.L = 1;
  g.K = K;
  g.N = N;
  g.in_f16 = b->dtype == BI_F16;
  if ((st = normalize_b(b, 0, 1, K, N, false, &g, &why)) != BI_OK) return finish(st, why);
  st = launch_pack(g, dst, (cudaStream_t)stream, &why);
  if (st == BI_OK) {
    out->ptr = dst;
    out->bytes = dst_bytes;
    out->K = K;
    out->N = N;
    out->layout = g.b_mn_major ? 1 : 2;
    out->tile_n = kBN;
    out->dtype = b->dtype;
  }
  return finish(st, why);
}

extern "C" bi_status bi_addmm_packed(const bi_tensor* bias, const bi_tensor* a,
                                     const bi_packed_weight* b, const bi_tensor* c,
                                     bi_stream stream) {
  std::string why;
  if (!b || !b->ptr) return finish(BI_ERR_INVALID_ARG, "packed weight: null");
  const bi_status st = matmul_impl(bias, a, nullptr, c, 1.0f, false, (cudaStream_t)stream, &why, b);
  return finish(st, why);
}

extern "C" bi_status bi_conv2d_patch(const bi_tensor* x, const bi_tensor* w, const bi_tensor* bias,
                                     const bi_tensor* y, const int32_t stride[2],
                                     const int32_t padding[2], const int32_t dilation[2],
                                     int32_t groups, bi_stream stream) {
  std::string why;
  bi_status st = BI_OK;
  auto fail = [&](bi_status s, const std::string& m) {
    why = m;
    return finish(s, why);
  };
  if ((st = check_tensor(x, "x", 4, &why)) != BI_OK) return finish(st, why);
  if ((st = check_tensor(w, "w", 4, &why)) != BI_OK) return finish(st, why);
  if ((st = check_tensor(y, "y", 4, &why)) != BI_OK) return finish(st, why);
  if (!stride || !padding || !dilation) return fail(BI_ERR_INVALID_ARG, "stride/padding/dilation: null");
  if (x->dtype != BI_BF16 || w->dtype != BI_BF16)
    return fail(BI_ERR_UNSUPPORTED_DTYPE, "x and w must be bf16");
  if (y->dtype != BI_BF16 && y->dtype != BI_F32)
    return fail(BI_ERR_UNSUPPORTED_DTYPE, "y must be bf16 or fp32");
  if (groups < 1) return fail(BI_ERR_INVALID_ARG, "groups must be >= 1");
  if (stride[0] < 1 || stride[1] < 1 || dilation[0] < 1 || dilation[1] < 1 || padding[0] < 0 ||
      padding[1] < 0)
    return fail(BI_ERR_INVALID_ARG, "stride and dilation must be >= 1, padding >= 0");
  const int64_t B = x->shape[0], C = x->shape[1], H = x->shape[2], W = x->shape[3];
  const int64_t Co = w->shape[0], Cig = w->shape[1], KH = w->shape[2], KW = w->shape[3];
  if (C % groups != 0 || Co % groups != 0 || Cig * groups != C)
    return fail(BI_ERR_SHAPE_MISMATCH, "channels do not divide into groups as w expects");
  if (KH < 1 || KW < 1) return fail(BI_ERR_INVALID_ARG, "kernel extents must be >= 1");
  const int64_t Ho = (H + 2 * padding[0] - (int64_t)dilation[0] * (KH - 1) - 1) / stride[0] + 1;
  const int64_t Wo = (W + 2 * padding[1] - (int64_t)dilation[1] * (KW - 1) - 1) / stride[1] + 1;
  if (H + 2 * padding[0] - (int64_t)dilation[0] * (KH - 1) - 1 < 0 ||
      W + 2 * padding[1] - (int64_t)dilation[1] * (KW - 1) - 1 < 0)
    return fail(BI_ERR_SHAPE_MISMATCH, "kernel window larger than the padded image");
  if (y->shape[0] != B || y->shape[1] != Co || y->shape[2] != Ho || y->shape[3] != Wo)
    return fail(BI_ERR_SHAPE_MISMATCH, "y must be [B, Co, Ho, Wo] = [" + std::to_string(B) + ", " +
                                           std::to_string(Co) + ", " + std::to_string(Ho) + ", " +
                                           std::to_string(Wo) + "]");
  if (!is_contiguous(x) || !is_contiguous(w) || !is_contiguous(y))
    return fail(BI_ERR_UNSUPPORTED_LAYOUT, "x, w and y must be contiguous (NCHW)");
  if (Ho * Wo > INT32_MAX || Cig * KH * KW > INT32_MAX)
    return fail(BI_ERR_INVALID_ARG, "per-sample problem too large");
  int bias_kind = 0;
  if (bias && bias->ptr) {
    if ((st = check_tensor(bias, "bias", 1, &why)) != BI_OK) return finish(st, why);
    if (bias->shape[0] != Co) return fail(BI_ERR_SHAPE_MISMATCH, "bias must have Co elements");
    if (bias->stride[0] != 1 && Co > 1) return fail(BI_ERR_UNSUPPORTED_LAYOUT, "bias must be contiguous");
    if (bias->dtype == BI_BF16)
      bias_kind = 1;
    else if (bias->dtype == BI_F32)
      bias_kind = 2;
    else
      return fail(BI_ERR_UNSUPPORTED_DTYPE, "bias must be bf16 or fp32");
  }
  if (B == 0 || Co == 0) return finish(BI_OK, why);
  if (!x->ptr || !w->ptr || !y->ptr) return fail(BI_ERR_INVALID_ARG, "null data pointer");
  if (!aligned(x->ptr, 2) || !aligned(w->ptr, 2) || !aligned(y->ptr, y->dtype == BI_F32 ? 4 : 2))
    return fail(BI_ERR_UNSUPPORTED_LAYOUT, "pointers must be aligned to their element size");
  if (C == 0 || KH * KW == 0) return fail(BI_ERR_INVALID_ARG, "empty reduction (C == 0)");
  // Non-overlapping patches (stride = kernel, no padding, unit dilation, one
  // group) run the patch kernel straight from this filter when the image rows
  // suit its copies; which kernel runs depends on the geometry and on the
  // alignment of x and w only, never on the batch size (a batch slice of an
  // aligned x is aligned: a sample spans whole 16-byte rows).
  const bool patch = stride[0] == KH && stride[1] == KW && padding[0] == 0 && padding[1] == 0 &&
                     dilation[0] == 1 && dilation[1] == 1 && groups == 1 &&
                     patch_plain_filter_ok(KH, KW, w->ptr) && (W * 2) % 16 == 0 && W <= 256 && Wo <= 128 &&
                     patch_stage_bytes(W, patch_tile_rows(Ho, Wo, W)) <= kPatchStageMax &&
                     aligned(x->ptr, 16) && C * KH * 16 <= INT32_MAX;
  if (patch) {
    if (B * C > INT32_MAX) return fail(BI_ERR_INVALID_ARG, "problem too large");
    PatchProblem pp;
    memset(&pp, 0, sizeof(pp));
    pp.x = x->ptr;
    pp.w = w->ptr;
    pp.bias = bias_kind ? bias->ptr : nullptr;
    pp.bias_kind = bias_kind;
    pp.y = y->ptr;
    pp.out_f32 = y->dtype == BI_F32;
    pp.B = B;
    pp.C = C;
    pp.H = H;
    pp.W = W;
    pp.Co = Co;
    pp.KH = KH;
    pp.KW = KW;
    pp.Ho = Ho;
    pp.Wo = Wo;
    st = launch_patch(pp, (cudaStream_t)stream, &why);
    return finish(st, why);
  }
  ConvProblem cp;
  memset(&cp, 0, sizeof(cp));
  cp.x = x->ptr;
  cp.w = w->ptr;
  cp.bias = bias_kind ? bias->ptr : nullptr;
  cp.bias_kind = bias_kind;
  cp.y = y->ptr;
  cp.out_f32 = y->dtype == BI_F32;
  cp.B = B;
  cp.C = C;
  cp.H = H;
  cp.W = W;
  cp.Co = Co;
  cp.KH = KH;
  cp.KW = KW;
  cp.Ho = Ho;
  cp.Wo = Wo;
  cp.sh = stride[0];
  cp.sw = stride[1];
  cp.ph = padding[0];
  cp.pw = padding[1];
  cp.dh = dilation[0];
  cp.dw = dilation[1];
  cp.groups = groups;
  st = launch_conv(cp, (cudaStream_t)stream, &why);
  return finish(st, why);
}

// ---------------------------------------------------------------------------
// Patch convolution with a packed filter
// ---------------------------------------------------------------------------

extern "C" int64_t bi_conv_packed_weight_bytes(int64_t Co, int64_t C, int64_t KH, int64_t KW) {
  if (Co <= 0 || C <= 0 || KH <= 0 || KW <= 0 || KW > 16) return 0;
  return Co * patch_padded_k(C, KH) * 2;
}

extern "C" bi_status bi_conv_pack_weight(const bi_tensor* w, void* dst, int64_t dst_bytes,
                                         bi_conv_packed_weight* out, bi_stream stream) {
  std::string why;
  bi_status st;
  if ((st = check_tensor(w, "w", 4, &why)) != BI_OK) return finish(st, why);
  if (w->dtype != BI_BF16) return finish(BI_ERR_UNSUPPORTED_DTYPE, "w must be bf16");
  if (!out) return finish(BI_ERR_INVALID_ARG, "out: null");
  const int64_t Co = w->shape[0], C = w->shape[1], KH = w->shape[2], KW = w->shape[3];
  if (Co < 1 || C < 1 || KH < 1 || KW < 1) return finish(BI_ERR_INVALID_ARG, "empty filter");
  if (KW > 16) return finish(BI_ERR_UNSUPPORTED_LAYOUT, "packed filters take KW <= 16");
  if (Co > INT32_MAX || patch_padded_k(C, KH) > INT32_MAX)
    return finish(BI_ERR_INVALID_ARG, "filter too large");
  if (!is_contiguous(w)) return finish(BI_ERR_UNSUPPORTED_LAYOUT, "w must be contiguous");
  const int64_t need = bi_conv_packed_weight_bytes(Co, C, KH, KW);
  if (!dst || !aligned(dst, 16) || dst_bytes < need)
    return finish(BI_ERR_INVALID_ARG, "dst must be 16-byte aligned with at least " +
                                          std::to_string(need) + " bytes");
  if (!w->ptr || !aligned(w->ptr, 2)) return finish(BI_ERR_INVALID_ARG, "w: null or misaligned data pointer");
  st = launch_conv_pack(w->ptr, dst, Co, C, KH, KW, (cudaStream_t)stream, &why);
  if (st == BI_OK) {
    out->ptr = dst;
    out->bytes = dst_bytes;
    out->Co = Co;
    out->C = C;
    out->KH = KH;
    out->KW = KW;
    out->Kp = patch_padded_k(C, KH);
  }
  return finish(st, why);
}

extern "C" bi_status bi_conv2d_patch_packed(const bi_tensor* x, const bi_conv_packed_weight* w,
                                            const bi_tensor* bias, const bi_tensor* y,
                                            bi_stream stream) {
  std::string why;
  bi_status st;
  auto fail = [&](bi_status s, const std::string& m) {
    why = m;
    return finish(s, why);
  };
  if ((st = check_tensor(x, "x", 4, &why)) != BI_OK) return finish(st, why);
  if ((st = check_tensor(y, "y", 4, &why)) != BI_OK) return finish(st, why);
  if (!w || !w->ptr) return fail(BI_ERR_INVALID_ARG, "packed filter: null");
  if (x->dtype != BI_BF16) return fail(BI_ERR_UNSUPPORTED_DTYPE, "x must be bf16");
  if (y->dtype != BI_BF16 && y->dtype != BI_F32) return fail(BI_ERR_UNSUPPORTED_DTYPE, "y must be bf16 or fp32");
  const int64_t Co = w->Co, C = w->C, KH = w->KH, KW = w->KW;
  if (Co < 1 || C < 1 || KH < 1 || KW < 1 || KW > 16 || w->Kp != patch_padded_k(C, KH) ||
      w->bytes < bi_conv_packed_weight_bytes(Co, C, KH, KW) || !aligned(w->ptr, 16))
    return fail(BI_ERR_INVALID_ARG, "packed filter descriptor is inconsistent");
  const int64_t B = x->shape[0], H = x->shape[2], W = x->shape[3];
  if (x->shape[1] != C) return fail(BI_ERR_SHAPE_MISMATCH, "x has " + std::to_string(x->shape[1]) +
                                                               " channels, the filter " + std::to_string(C));
  const int64_t Ho = H / KH, Wo = W / KW;
  if (y->shape[0] != B || y->shape[1] != Co || y->shape[2] != Ho || y->shape[3] != Wo)
    return fail(BI_ERR_SHAPE_MISMATCH, "y must be [B, Co, H/KH, W/KW] = [" + std::to_string(B) + ", " +
                                           std::to_string(Co) + ", " + std::to_string(Ho) + ", " +
                                           std::to_string(Wo) + "]");
  if (!is_contiguous(x) || !is_contiguous(y))
    return fail(BI_ERR_UNSUPPORTED_LAYOUT, "x and y must be contiguous (NCHW)");
  int bias_kind = 0;
  if (bias && bias->ptr) {
    if ((st = check_tensor(bias, "bias", 1, &why)) != BI_OK) return finish(st, why);
    if (bias->shape[0] != Co) return fail(BI_ERR_SHAPE_MISMATCH, "bias must have Co elements");
    if (bias->stride[0] != 1 && Co > 1) return fail(BI_ERR_UNSUPPORTED_LAYOUT, "bias must be contiguous");
    if (bias->dtype == BI_BF16)
      bias_kind = 1;
    else if (bias->dtype == BI_F32)
      bias_kind = 2;
    else
      return fail(BI_ERR_UNSUPPORTED_DTYPE, "bias must be bf16 or fp32");
  }
  if (B == 0 || Ho == 0 || Wo == 0) return finish(BI_OK, why);
  // The image is read as whole rows by TMA: 16-byte rows, at most 256 wide,
  // and one K block's rows (4 kernel rows of each output row of a tile) must
  // fit one staging buffer.
  const int64_t t_oh = patch_tile_rows(Ho, Wo, W);
  if ((W * 2) % 16 != 0 || W > 256 || Wo > 128 || patch_stage_bytes(W, t_oh) > kPatchStageMax)
    return fail(BI_ERR_UNSUPPORTED_LAYOUT,
                "image rows must be a multiple of 8 and at most 256 elements, with W/KW <= 128");
  if (!x->ptr || !y->ptr) return fail(BI_ERR_INVALID_ARG, "null data pointer");
  if (!aligned(x->ptr, 16) || !aligned(y->ptr, y->dtype == BI_F32 ? 4 : 2))
    return fail(BI_ERR_UNSUPPORTED_LAYOUT, "x must be 16-byte aligned, y aligned to its element size");
  if (B * C > INT32_MAX || Ho * Wo > INT32_MAX) return fail(BI_ERR_INVALID_ARG, "problem too large");
  PatchProblem pp;
  memset(&pp, 0, sizeof(pp));
  pp.x = x->ptr;
  pp.wp = w->ptr;
  pp.bias = bias_kind ? bias->ptr : nullptr;
  pp.bias_kind = bias_kind;
  pp.y = y->ptr;
  pp.out_f32 = y->dtype == BI_F32;
  pp.B = B;
  pp.C = C;
  pp.H = H;
  pp.W = W;
  pp.Co = Co;
  pp.KH = KH;
  pp.KW = KW;
  pp.Ho = Ho;
  pp.Wo = Wo;
  st = launch_patch(pp, (cudaStream_t)stream, &why);
  return finish(st, why);
}

// ---------------------------------------------------------------------------
// Row reductions: RMSNorm, log-softmax, mean
// ---------------------------------------------------------------------------
namespace {

int kind_of(int dtype) { return dtype == BI_F32 ? 2 : (dtype == BI_F16 ? 1 : 0); }

// x: [R, N] of any floating type with a unit stride on N; y: [R, N] (or [R]
// for the mean) of any floating type.  Fills the shared fields of rp.
bi_status check_rows(const bi_tensor* x, const bi_tensor* y, bool y_is_row_vector, RowParams* rp,
                     std::string* why) {
  bi_status st;
  if ((st = check_tensor(x, "x", 2, why)) != BI_OK) return st;
  if ((st = check_tensor(y, "y", y_is_row_vector ? 1 : 2, why)) != BI_OK) return st;
  const int64_t R = x->shape[0], N = x->shape[1];
  if (y_is_row_vector ? (y->shape[0] != R) : (y->shape[0] != R || y->shape[1] != N)) {
    *why = y_is_row_vector ? "y must be [R]" : "y must have x's shape";
    return BI_ERR_SHAPE_MISMATCH;
  }
  if (N > 1 && x->stride[1] != 1) {
    *why = "x needs a unit stride on its last dimension";
    return BI_ERR_UNSUPPORTED_LAYOUT;
  }
  if (!y_is_row_vector && N > 1 && y->stride[1] != 1) {
    *why = "y needs a unit stride on its last dimension";
    return BI_ERR_UNSUPPORTED_LAYOUT;
  }
  if (N > (1 << 24)) {
    *why = "rows longer than 2^24 elements are not supported (N must be exact in fp32)";
    return BI_ERR_INVALID_ARG;
  }
  rp->x = x->ptr;
  rp->y = y->ptr;
  rp->R = R;
  rp->N = N;
  rp->ld_x = R > 1 ? x->stride[0] : N;
  rp->ld_y = y_is_row_vector ? y->stride[0] : (R > 1 ? y->stride[0] : N);
  rp->x_kind = kind_of(x->dtype);
  rp->y_kind = kind_of(y->dtype);
  rp->x_esz = elem_size(x->dtype);
  rp->y_esz = elem_size(y->dtype);
  if (R > 0 && N > 0) {
    if (!x->ptr || !y->ptr) {
      *why = "null data pointer";
      return BI_ERR_INVALID_ARG;
    }
    if (!aligned(x->ptr, rp->x_esz) || !aligned(y->ptr, rp->y_esz)) {
      *why = "pointers must be aligned to their element size";
      return BI_ERR_UNSUPPORTED_LAYOUT;
    }
  }
  return BI_OK;
}

bi_status run_rows(int op, const RowParams& rp, bi_stream stream) {
  std::string why;
  DeviceInfo dev;
  bi_status st = current_device_info(&dev, &why);
  if (st == BI_OK) st = launch_row_reduction(op, rp, (cudaStream_t)stream, &why);
  return finish(st, why);
}

}  // namespace

extern "C" bi_status bi_rmsnorm_lastdim(const bi_tensor* x, const bi_tensor* weight, float eps,
                                        const bi_tensor* y, bi_stream stream) {
  std::string why;
  RowParams rp;
  memset(&rp, 0, sizeof(rp));
  bi_status st = check_rows(x, y, false, &rp, &why);
  if (st != BI_OK) return finish(st, why);
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return finish(BI_ERR_INVALID_ARG, "eps must be finite and >= 0");
  rp.eps = eps;
  if (weight && weight->ptr) {
    if ((st = check_tensor(weight, "weight", 1, &why)) != BI_OK) return finish(st, why);
    if (weight->shape[0] != rp.N) return finish(BI_ERR_SHAPE_MISMATCH, "weight must have N elements");
    if (!aligned(weight->ptr, elem_size(weight->dtype)))
      return finish(BI_ERR_UNSUPPORTED_LAYOUT, "weight pointer is not aligned to its element size");
    rp.w = weight->ptr;
    rp.w_kind = kind_of(weight->dtype);
    rp.w_stride = weight->stride[0];
  }
  if (rp.R == 0 || rp.N == 0) return finish(BI_OK, why);
  return run_rows(kRowRmsNorm, rp, stream);
}

extern "C" bi_status bi_log_softmax_lastdim(const bi_tensor* s, const bi_tensor* p, bi_stream stream) {
  std::string why;
  RowParams rp;
  memset(&rp, 0, sizeof(rp));
  bi_status st = check_rows(s, p, false, &rp, &why);
  if (st != BI_OK) return finish(st, why);
  if (rp.R == 0 || rp.N == 0) return finish(BI_OK, why);
  return run_rows(kRowLogSoftmax, rp, stream);
}

extern "C" bi_status bi_mean_lastdim(const bi_tensor* x, const bi_tensor* y, bi_stream stream) {
  std::string why;
  RowParams rp;
  memset(&rp, 0, sizeof(rp));
  bi_status st = check_rows(x, y, true, &rp, &why);
  if (st != BI_OK) return finish(st, why);
  if (rp.R == 0) return finish(BI_OK, why);
  if (rp.N == 0) return finish(BI_ERR_INVALID_ARG, "the mean of an empty row is undefined");
  return run_rows(kRowMean, rp, stream);
}

// ---------------------------------------------------------------------------
// Fused attention
// ---------------------------------------------------------------------------
namespace {

bi_status attention_impl(const bi_tensor* q, const bi_tensor* k, const bi_tensor* v, float scale,
                         const bi_tensor* o, void* ws, int64_t ws_bytes, bi_stream stream) {
  std::string why;
  bi_status st;
  if ((st = check_tensor(q, "q", 3, &why)) != BI_OK) return finish(st, why);
  if ((st = check_tensor(k, "k", 3, &why)) != BI_OK) return finish(st, why);
  if ((st = check_tensor(v, "v", 3, &why)) != BI_OK) return finish(st, why);
  if ((st = check_tensor(o, "o", 3, &why)) != BI_OK) return finish(st, why);
  const int64_t L = q->shape[0], Tq = q->shape[1], D = q->shape[2], Tk = k->shape[1];
  if (k->shape[0] != L || k->shape[2] != D || v->shape[0] != L || v->shape[1] != Tk || v->shape[2] != D)
    return finish(BI_ERR_SHAPE_MISMATCH, "k and v must be [L, Tk, D] with q's L and D");
  if (o->shape[0] != L || o->shape[1] != Tq || o->shape[2] != D)
    return finish(BI_ERR_SHAPE_MISMATCH, "o must be [L, Tq, D]");
  if (q->dtype != BI_BF16 || k->dtype != BI_BF16 || v->dtype != BI_BF16)
    return finish(BI_ERR_UNSUPPORTED_DTYPE, "q, k and v must be bf16");
  if (o->dtype != BI_F32 && o->dtype != BI_BF16) return finish(BI_ERR_UNSUPPORTED_DTYPE, "o must be fp32 or bf16");
  if (!attention_head_dim_ok(D)) return finish(BI_ERR_INVALID_ARG, "head dimension must be 64, 128 or 256");
  if (!std::isfinite(scale)) return finish(BI_ERR_INVALID_ARG, "scale must be finite");
  if (L == 0 || Tq == 0) return finish(BI_OK, why);
  if (Tk == 0) return finish(BI_ERR_INVALID_ARG, "softmax over an empty key range is undefined");
  const bi_tensor* ts[4] = {q, k, v, o};
  for (int i = 0; i < 4; ++i) {
    const bi_tensor* t = ts[i];
    const int esz = elem_size(t->dtype);
    if (t->stride[2] != 1) return finish(BI_ERR_UNSUPPORTED_LAYOUT, "unit stride on the head dimension required");
    if (!t->ptr) return finish(BI_ERR_INVALID_ARG, "null data pointer");
    if (!aligned(t->ptr, 16)) return finish(BI_ERR_UNSUPPORTED_LAYOUT, "base pointers must be 16-byte aligned");
    if ((t->shape[1] > 1 && (t->stride[1] * esz) % 16 != 0) || (t->shape[0] > 1 && (t->stride[0] * esz) % 16 != 0))
      return finish(BI_ERR_UNSUPPORTED_LAYOUT, "row and batch strides must be multiples of 16 bytes");
  }
  if ((L * ((Tq + 127) / 128)) > INT32_MAX) return finish(BI_ERR_INVALID_ARG, "too many query tiles");
  // Strides of size-1 dimensions do not matter; give the tensor maps
  // consistent ones.
  auto st_t = [&](const bi_tensor* t) { return t->shape[1] > 1 ? t->stride[1] : D; };
  auto st_l = [&](const bi_tensor* t) { return t->shape[0] > 1 ? t->stride[0] : t->shape[1] * st_t(t); };
  AttnProblem ap;
  ap.q = q->ptr;
  ap.k = k->ptr;
  ap.v = v->ptr;
  ap.o = o->ptr;
  ap.q_t = st_t(q), ap.q_l = st_l(q);
  ap.k_t = st_t(k), ap.k_l = st_l(k);
  ap.v_t = st_t(v), ap.v_l = st_l(v);
  ap.o_t = st_t(o), ap.o_l = st_l(o);
  ap.out_f32 = o->dtype == BI_F32;
  ap.scale = scale;
  ap.L = L, ap.Tq = Tq, ap.Tk = Tk, ap.D = D;
  ap.ws = ws;
  ap.ws_bytes = ws_bytes;
  if (ws && !aligned(ws, 16)) return finish(BI_ERR_UNSUPPORTED_LAYOUT, "the workspace must be 16-byte aligned");
  if (attention_splits(Tk) > 1 && (!ws || ws_bytes < attention_workspace_bytes(L, Tq, Tk, D)))
    return finish(BI_ERR_INVALID_ARG, "a key range longer than 2048 needs a workspace of " +
                                          std::to_string(attention_workspace_bytes(L, Tq, Tk, D)) +
                                          " bytes (bi_attention_workspace_bytes)");
  st = launch_attention(ap, (cudaStream_t)stream, &why);
  return finish(st, why);
}

}  // namespace

extern "C" int64_t bi_attention_workspace_bytes(int64_t L, int64_t Tq, int64_t Tk, int64_t D) {
  if (L <= 0 || Tq <= 0 || Tk <= 0 || !attention_head_dim_ok(D)) return 0;
  return attention_workspace_bytes(L, Tq, Tk, D);
}

extern "C" bi_status bi_attention(const bi_tensor* q, const bi_tensor* k, const bi_tensor* v, float scale,
                                  const bi_tensor* o, bi_stream stream) {
  return attention_impl(q, k, v, scale, o, nullptr, 0, stream);
}

// The device address of this device's static scratch (resolved once per device).
static bi_status noalloc_scratch(void** out, std::string* why) {
  DeviceInfo dev;
  bi_status st = current_device_info(&dev, why);
  if (st != BI_OK) return st;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& d = g_dev[dev.device];
  if (!d.scratch) {
    void* addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_bi_noalloc_scratch);
    if (e != cudaSuccess) {
      *why = std::string("scratch address: ") + cudaGetErrorString(e);
      cudaGetLastError();
      return BI_ERR_CUDA;
    }
    d.scratch = addr;
  }
  *out = d.scratch;
  return BI_OK;
}

extern "C" bi_status bi_attention_noalloc(const bi_tensor* q, const bi_tensor* k, const bi_tensor* v, float scale,
                                          const bi_tensor* o, bi_stream stream) {
  std::string why;
  bi_status st;
  if ((st = check_tensor(q, "q", 3, &why)) != BI_OK) return finish(st, why);
  if ((st = check_tensor(k, "k", 3, &why)) != BI_OK) return finish(st, why);
  const int64_t need = attention_head_dim_ok(q->shape[2])
                           ? attention_workspace_bytes(q->shape[0], q->shape[1], k->shape[1], q->shape[2])
                           : 0;  // attention_impl reports the head dimension
  if (q->shape[0] == 0 || q->shape[1] == 0 || k->shape[1] == 0 || need == 0)
    return attention_impl(q, k, v, scale, o, nullptr, 0, stream);
  if (need > kNoAllocScratchBytes)
    return finish(BI_ERR_INVALID_ARG, "the split key range needs " + std::to_string(need) +
                                          " bytes of scratch, more than the library's static " +
                                          std::to_string(kNoAllocScratchBytes) + " (use bi_attention_ws)");
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch, &why)) != BI_OK) return finish(st, why);
  return attention_impl(q, k, v, scale, o, scratch, kNoAllocScratchBytes, stream);
}

extern "C" bi_status bi_attention_ws(const bi_tensor* q, const bi_tensor* k, const bi_tensor* v, float scale,
                                     const bi_tensor* o, void* workspace, int64_t workspace_bytes,
                                     bi_stream stream) {
  if (workspace_bytes < 0) return finish(BI_ERR_INVALID_ARG, "negative workspace size");
  return attention_impl(q, k, v, scale, o, workspace, workspace_bytes, stream);
}

extern "C" bi_status bi_softmax_lastdim(const bi_tensor* s, const bi_tensor* p, bi_stream stream) {
  std::string why;
  bi_status st;
  if ((st = check_tensor(s, "s", 2, &why)) != BI_OK) return finish(st, why);
  if ((st = check_tensor(p, "p", 2, &why)) != BI_OK) return finish(st, why);
  if (s->dtype != BI_F32) return finish(BI_ERR_UNSUPPORTED_DTYPE, "s must be fp32");
  if (p->dtype != BI_BF16 && p->dtype != BI_F32)
    return finish(BI_ERR_UNSUPPORTED_DTYPE, "p must be bf16 or fp32");
  if (s->shape[0] != p->shape[0] || s->shape[1] != p->shape[1])
    return finish(BI_ERR_SHAPE_MISMATCH, "s and p must have the same shape");
  const int64_t R = s->shape[0], N = s->shape[1];
  if (R == 0 || N == 0) return finish(BI_OK, why);
  if (!s->ptr || !p->ptr) return finish(BI_ERR_INVALID_ARG, "null data pointer");
  if ((N > 1 && (s->stride[1] != 1 || p->stride[1] != 1)))
    return finish(BI_ERR_UNSUPPORTED_LAYOUT, "s and p need a unit stride on the last dimension");
  if (!aligned(s->ptr, 4) || !aligned(p->ptr, p->dtype == BI_F32 ? 4 : 2))
    return finish(BI_ERR_UNSUPPORTED_LAYOUT, "pointers must be aligned to their element size");
  SoftmaxParams sp;
  sp.s = reinterpret_cast<const float*>(s->ptr);
  sp.p = p->ptr;
  sp.R = R;
  sp.N = N;
  sp.ld_s = (R == 1) ? N : s->stride[0];
  sp.ld_p = (R == 1) ? N : p->stride[0];
  sp.out_f32 = p->dtype == BI_F32;
  st = launch_softmax(sp, (cudaStream_t)stream, &why);
  return finish(st, why);
}

extern "C" bi_status bi_device_status(bi_stream stream) {
  std::string why;
  DeviceInfo dev;
  bi_status st = current_device_info(&dev, &why);
  if (st != BI_OK) return finish(st, why);
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return finish(BI_ERR_CUDA, std::string("stream sync: ") + cudaGetErrorString(e));
  unsigned int v = 0;
  e = cudaMemcpy(&v, dev.status_word, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return finish(BI_ERR_CUDA, std::string("status read: ") + cudaGetErrorString(e));
  if (v == 0) return finish(BI_OK, why);
  e = cudaMemset(dev.status_word, 0, sizeof(v));
  if (e != cudaSuccess) return finish(BI_ERR_CUDA, std::string("status clear: ") + cudaGetErrorString(e));
  static const char* kSites[] = {"?", "producer waiting for a free stage", "MMA waiting for a full stage",
                                 "MMA waiting for a free accumulator", "epilogue waiting for an accumulator",
                                 "draining in-flight work", "debug wait", "conv producer waiting for a free stage",
                                 "weight packer waiting for its tile", "attention softmax waiting"};
  const unsigned site = (v >> 8) & 0xFF;
  why = std::string("device wait ran out: ") +
        (site < sizeof(kSites) / sizeof(kSites[0]) ? kSites[site] : "?");
  return finish((bi_status)(v & 0xFF), why);
}

extern "C" bi_status bi_debug_expire_wait(uint64_t limit_ns, bi_stream stream) {
  std::string why;
  if (limit_ns < 1000000ull || limit_ns > 2000000000ull)
    return finish(BI_ERR_INVALID_ARG, "limit_ns must be within [1 ms, 2 s]");
  bi_status st = launch_debug_wait(limit_ns, (cudaStream_t)stream, &why);
  return finish(st, why);
}

extern "C" const char* bi_status_string(bi_status s) {
  switch (s) {
    case BI_OK: return "BI_OK";
    case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG";
    case BI_ERR_SHAPE_MISMATCH: return "BI_ERR_SHAPE_MISMATCH";
    case BI_ERR_UNSUPPORTED_DTYPE: return "BI_ERR_UNSUPPORTED_DTYPE";
    case BI_ERR_UNSUPPORTED_LAYOUT: return "BI_ERR_UNSUPPORTED_LAYOUT";
    case BI_ERR_CUDA: return "BI_ERR_CUDA";
    case BI_ERR_TIMEOUT: return "BI_ERR_TIMEOUT";
    case BI_ERR_NO_DEVICE: return "BI_ERR_NO_DEVICE";
  }
  return "BI_ERR_UNKNOWN";
}

extern "C" const char* bi_last_error_message(void) { return t_last_error.c_str(); }

extern "C" int32_t bi_abi_version(void) { return 8; }
