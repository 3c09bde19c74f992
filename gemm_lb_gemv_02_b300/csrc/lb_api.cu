// liblb C ABI: argument validation, error reporting and dispatch to the kernel launchers.
#include <atomic>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "lb_common.cuh"

namespace {

thread_local char g_last_error[512] = "";
std::mutex g_pack_mutex;

// Sticky device error bits (one instance per device context; see lb_device_error).
__device__ uint32_t g_device_error;

constexpr int kMaxDevices = 64;
uint32_t* g_error_ptr[kMaxDevices] = {};
unsigned long long g_error_ctx[kMaxDevices] = {};
std::mutex g_error_ptr_mutex;

}  // namespace

namespace lb {

lb_status fail(lb_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

lb_status cuda_fail(cudaError_t e, const char* where) {
  return fail(LB_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
}

int sm_count() {
  static int cached[kMaxDevices] = {};
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  if (cached[dev] > 0) return cached[dev];
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  cached[dev] = n;
  return n;
}

// Unique id of the calling thread's current CUDA context (cuCtxGetId ids are never reused within a
// process, unlike context handles), or 0 if the driver cannot report one.  A cached device address of
// a module-scope __device__ variable is valid only for the context it was taken in: after
// cudaDeviceReset the module is loaded again, possibly elsewhere.
unsigned long long context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

uint32_t* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long ctx = context_id();
  std::lock_guard<std::mutex> lk(g_error_ptr_mutex);
  if (!g_error_ptr[dev] || ctx == 0 || ctx != g_error_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_error_ptr[dev] = static_cast<uint32_t*>(p);
    g_error_ctx[dev] = ctx;
  }
  return g_error_ptr[dev];
}

std::atomic<int> g_test_fault{0};

bool take_test_fault(int kernel) {
  int expected = kernel;
  return g_test_fault.load(std::memory_order_relaxed) == kernel &&
         g_test_fault.compare_exchange_strong(expected, 0);
}

}  // namespace lb

using lb::fail;

namespace {

lb_status check_shape(int64_t n, int64_t k) {
  if (n < 1) return fail(LB_ERR_SHAPE, "n must be >= 1 (got %lld)", (long long)n);
  if (k < lb::kGroup || k % lb::kGroup)
    return fail(LB_ERR_SHAPE, "k must be a positive multiple of 128 (got %lld)", (long long)k);
  if (n > (int64_t(1) << 31) || k > (int64_t(1) << 24))
    return fail(LB_ERR_SHAPE, "n = %lld or k = %lld beyond the supported range", (long long)n, (long long)k);
  return LB_OK;
}

lb_status check_weight(const lb_weight* W) {
  if (!W) return fail(LB_ERR_NULL, "W is NULL");
  if (W->fmt != LB_FMT_1BIT_G128 && W->fmt != LB_FMT_TERNARY_G128 && W->fmt != LB_FMT_TERNARY5_G128)
    return fail(LB_ERR_DTYPE, "unknown weight format %d", (int)W->fmt);
  lb_status s = check_shape(W->n, W->k);
  if (s != LB_OK) return s;
  if (!W->codes || !W->scales) return fail(LB_ERR_NULL, "W->codes or W->scales is NULL");
  if (!lb::aligned16(W->codes) || !lb::aligned16(W->scales))
    return fail(LB_ERR_ALIGN, "W->codes and W->scales must be 16-byte aligned");
  return LB_OK;
}

bool valid_dtype(int d) { return d == LB_F16 || d == LB_BF16; }

// Launch-shape limit of the GEMM: 65535 token tiles of 256 along grid y.
constexpr int64_t kGemmMaxM = int64_t(65535) * 256;

}  // namespace

extern "C" {

const char* lb_status_string(lb_status s) {
  switch (s) {
    case LB_OK: return "LB_OK";
    case LB_ERR_NULL: return "LB_ERR_NULL: a required pointer is NULL";
    case LB_ERR_SHAPE: return "LB_ERR_SHAPE: invalid matrix shape or batch";
    case LB_ERR_ALIGN: return "LB_ERR_ALIGN: a device pointer is not 16-byte aligned";
    case LB_ERR_DTYPE: return "LB_ERR_DTYPE: unknown data type or weight format";
    case LB_ERR_CODE: return "LB_ERR_CODE: ternary code outside {-1, 0, +1}";
    case LB_ERR_NONFINITE: return "LB_ERR_NONFINITE: NaN or Inf among the weights";
    case LB_ERR_RANGE: return "LB_ERR_RANGE: value outside the binary16 range";
    case LB_ERR_CUDA: return "LB_ERR_CUDA: CUDA call failed";
    case LB_ERR_UNSUPPORTED: return "LB_ERR_UNSUPPORTED: not implemented";
    case LB_ERR_WORKSPACE: return "LB_ERR_WORKSPACE: workspace missing or too small";
  }
  return "unknown lb_status";
}

const char* lb_last_error(void) { return g_last_error; }

int lb_version(void) { return 100; }

lb_status lb_packed_bytes(int fmt, int64_t n, int64_t k, size_t* codes_bytes, size_t* scales_bytes) {
  if (!codes_bytes || !scales_bytes) return fail(LB_ERR_NULL, "output pointer is NULL");
  if (fmt != LB_FMT_1BIT_G128 && fmt != LB_FMT_TERNARY_G128 && fmt != LB_FMT_TERNARY5_G128)
    return fail(LB_ERR_DTYPE, "unknown format %d", fmt);
  lb_status s = check_shape(n, k);
  if (s != LB_OK) return s;
  if (fmt == LB_FMT_TERNARY5_G128)
    *codes_bytes = static_cast<size_t>(n) * static_cast<size_t>(k / lb::kGroup) * 26;
  else
    *codes_bytes = static_cast<size_t>(n) * static_cast<size_t>(k) / (fmt == LB_FMT_1BIT_G128 ? 8 : 4);
  *scales_bytes = static_cast<size_t>(n) * static_cast<size_t>(k / lb::kGroup) * 2;
  return LB_OK;
}

lb_status lb_pack_1bit(const float* w, int64_t n, int64_t k, uint8_t* codes, uint16_t* scales,
                       lb_stream stream) {
  lb_status s = check_shape(n, k);
  if (s != LB_OK) return s;
  if (!w || !codes || !scales) return fail(LB_ERR_NULL, "w, codes and scales must be non-NULL");
  if (!lb::aligned16(w) || !lb::aligned16(codes) || !lb::aligned16(scales))
    return fail(LB_ERR_ALIGN, "w, codes and scales must be 16-byte aligned");
  std::lock_guard<std::mutex> lk(g_pack_mutex);
  uint32_t flags = 0;
  s = lb::launch_pack_1bit(w, n, k, codes, scales, reinterpret_cast<cudaStream_t>(stream), &flags);
  if (s != LB_OK) return s;
  if (flags & lb::kPackNonFinite) return fail(LB_ERR_NONFINITE, "weights contain NaN or Inf");
  if (flags & lb::kPackRange) return fail(LB_ERR_RANGE, "a group max |w| rounds to binary16 infinity");
  return LB_OK;
}

lb_status lb_pack_ternary(const int8_t* t, const uint16_t* s_in, int64_t n, int64_t k, uint8_t* codes,
                          uint16_t* scales, lb_stream stream) {
  lb_status s = check_shape(n, k);
  if (s != LB_OK) return s;
  if (!t || !s_in || !codes || !scales) return fail(LB_ERR_NULL, "t, s_in, codes and scales must be non-NULL");
  if (!lb::aligned16(t) || !lb::aligned16(s_in) || !lb::aligned16(codes) || !lb::aligned16(scales))
    return fail(LB_ERR_ALIGN, "t, s_in, codes and scales must be 16-byte aligned");
  std::lock_guard<std::mutex> lk(g_pack_mutex);
  uint32_t flags = 0;
  s = lb::launch_pack_ternary(t, s_in, n, k, codes, scales, reinterpret_cast<cudaStream_t>(stream), &flags);
  if (s != LB_OK) return s;
  if (flags & lb::kPackCode) return fail(LB_ERR_CODE, "a ternary code is outside {-1, 0, +1}");
  return LB_OK;
}

lb_status lb_pack_ternary5(const int8_t* t, const uint16_t* s_in, int64_t n, int64_t k, uint8_t* codes,
                           uint16_t* scales, lb_stream stream) {
  lb_status s = check_shape(n, k);
  if (s != LB_OK) return s;
  if (!t || !s_in || !codes || !scales) return fail(LB_ERR_NULL, "t, s_in, codes and scales must be non-NULL");
  if (!lb::aligned16(t) || !lb::aligned16(s_in) || !lb::aligned16(codes) || !lb::aligned16(scales))
    return fail(LB_ERR_ALIGN, "t, s_in, codes and scales must be 16-byte aligned");
  std::lock_guard<std::mutex> lk(g_pack_mutex);
  uint32_t flags = 0;
  s = lb::launch_pack_ternary5(t, s_in, n, k, codes, scales, reinterpret_cast<cudaStream_t>(stream), &flags);
  if (s != LB_OK) return s;
  if (flags & lb::kPackCode) return fail(LB_ERR_CODE, "a ternary code is outside {-1, 0, +1}");
  return LB_OK;
}

lb_status lb_gemv(const lb_weight* W, const void* x, int xdt, int batch, void* y, lb_stream stream) {
  lb_status s = check_weight(W);
  if (s != LB_OK) return s;
  if (!x || !y) return fail(LB_ERR_NULL, "x and y must be non-NULL");
  if (!valid_dtype(xdt)) return fail(LB_ERR_DTYPE, "unknown activation dtype %d", xdt);
  if (batch < 1 || batch > 8) return fail(LB_ERR_SHAPE, "batch must be in [1, 8] (got %d)", batch);
  if (!lb::aligned16(x) || !lb::aligned16(y)) return fail(LB_ERR_ALIGN, "x and y must be 16-byte aligned");
  if (W->fmt == LB_FMT_TERNARY5_G128 && !lb::gemv_t5_lut_ok(*W, batch))
    return lb::launch_gemv_t5(*W, x, xdt, batch, y, reinterpret_cast<cudaStream_t>(stream));
  return lb::launch_gemv(*W, x, xdt, batch, y, reinterpret_cast<cudaStream_t>(stream));
}

lb_status lb_gemv_batched(const lb_gemv_problem* problems, int count, int xdt, int batch, lb_stream stream) {
  if (!problems) return fail(LB_ERR_NULL, "problems is NULL");
  if (count < 1 || count > LB_GEMV_BATCH_MAX)
    return fail(LB_ERR_SHAPE, "count must be in [1, %d] (got %d)", LB_GEMV_BATCH_MAX, count);
  if (!valid_dtype(xdt)) return fail(LB_ERR_DTYPE, "unknown activation dtype %d", xdt);
  if (batch < 1 || batch > 8) return fail(LB_ERR_SHAPE, "batch must be in [1, 8] (got %d)", batch);
  for (int i = 0; i < count; ++i) {
    const lb_gemv_problem& pb = problems[i];
    lb_status s = check_weight(&pb.W);
    if (s != LB_OK) return s;
    if (pb.W.fmt != problems[0].W.fmt)
      return fail(LB_ERR_UNSUPPORTED, "problem %d: every problem of one call must have the same format", i);
    if (!pb.x || !pb.y) return fail(LB_ERR_NULL, "problem %d: x and y must be non-NULL", i);
    if (!lb::aligned16(pb.x) || !lb::aligned16(pb.y)) return fail(LB_ERR_ALIGN, "problem %d: x and y must be 16-byte aligned", i);
  }
  return lb::launch_gemv_batched(problems, count, xdt, batch, reinterpret_cast<cudaStream_t>(stream));
}

lb_status lb_gemv_swiglu(const lb_weight* Wg, const lb_weight* Wu, const void* x, int xdt, int batch, void* h,
                         lb_stream stream) {
  lb_status s = check_weight(Wg);
  if (s != LB_OK) return s;
  s = check_weight(Wu);
  if (s != LB_OK) return s;
  if (Wg->fmt != Wu->fmt) return fail(LB_ERR_UNSUPPORTED, "gate and up must have the same format");
  if (Wg->n != Wu->n || Wg->k != Wu->k)
    return fail(LB_ERR_SHAPE, "gate (%lld x %lld) and up (%lld x %lld) must have the same shape", (long long)Wg->n,
                (long long)Wg->k, (long long)Wu->n, (long long)Wu->k);
  if (!x || !h) return fail(LB_ERR_NULL, "x and h must be non-NULL");
  if (!valid_dtype(xdt)) return fail(LB_ERR_DTYPE, "unknown activation dtype %d", xdt);
  if (batch < 1 || batch > 8) return fail(LB_ERR_SHAPE, "batch must be in [1, 8] (got %d)", batch);
  if (Wg->fmt == LB_FMT_TERNARY5_G128 && !lb::gemv_t5_lut_ok(*Wg, batch))
    return fail(LB_ERR_UNSUPPORTED,
                "lb_gemv_swiglu on five-per-byte weights runs at batch 1 with k a multiple of 1024 (k <= 40960)");
  if (!lb::aligned16(x) || !lb::aligned16(h)) return fail(LB_ERR_ALIGN, "x and h must be 16-byte aligned");
  return lb::launch_gemv_swiglu(*Wg, *Wu, x, xdt, batch, h, reinterpret_cast<cudaStream_t>(stream));
}

lb_status lb_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int xdt, size_t* bytes) {
  if (!bytes) return fail(LB_ERR_NULL, "bytes is NULL");
  if (!valid_dtype(xdt)) return fail(LB_ERR_DTYPE, "unknown activation dtype %d", xdt);
  if (m < 1) return fail(LB_ERR_SHAPE, "m must be >= 1");
  lb_status s = check_shape(n, k);
  if (s != LB_OK) return s;
  *bytes = lb::gemm_workspace_bytes(m, k);
  return LB_OK;
}

lb_status lb_gemm(const lb_weight* W, const void* x, int xdt, int64_t m, void* y, int ydt, void* workspace,
                  size_t workspace_bytes, lb_stream stream) {
  lb_status s = check_weight(W);
  if (s != LB_OK) return s;
  if (W->fmt == LB_FMT_TERNARY5_G128) return fail(LB_ERR_UNSUPPORTED, "lb_gemm takes the 1-bit and 2-bit ternary formats");
  if (!x || !y) return fail(LB_ERR_NULL, "x and y must be non-NULL");
  if (!valid_dtype(xdt) || !valid_dtype(ydt)) return fail(LB_ERR_DTYPE, "unknown dtype (x %d, y %d)", xdt, ydt);
  if (m < 1 || m > kGemmMaxM) return fail(LB_ERR_SHAPE, "m must be in [1, %lld] (got %lld)", (long long)kGemmMaxM, (long long)m);
  if (W->n % 16) return fail(LB_ERR_SHAPE, "lb_gemm needs n %% 16 == 0 (got %lld)", (long long)W->n);
  if (!lb::aligned16(x) || !lb::aligned16(y)) return fail(LB_ERR_ALIGN, "x and y must be 16-byte aligned");
  const size_t need = lb::gemm_workspace_bytes(m, W->k);
  if (need && (!workspace || workspace_bytes < need))
    return fail(LB_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need, workspace_bytes);
  if (need && (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(LB_ERR_ALIGN, "workspace must be 256-byte aligned");
  return lb::launch_gemm(*W, x, xdt, m, y, ydt, workspace, reinterpret_cast<cudaStream_t>(stream));
}

lb_status lb_gemm_noalloc(const lb_weight* W, const void* x, int xdt, int64_t m, void* y, int ydt,
                          lb_stream stream) {
  lb_status s = check_weight(W);
  if (s != LB_OK) return s;
  if (W->fmt == LB_FMT_TERNARY5_G128)
    return fail(LB_ERR_UNSUPPORTED, "lb_gemm_noalloc takes the 1-bit and 2-bit ternary formats");
  if (!x || !y) return fail(LB_ERR_NULL, "x and y must be non-NULL");
  if (!valid_dtype(xdt) || !valid_dtype(ydt)) return fail(LB_ERR_DTYPE, "unknown dtype (x %d, y %d)", xdt, ydt);
  if (m < 1 || m > kGemmMaxM) return fail(LB_ERR_SHAPE, "m must be in [1, %lld] (got %lld)", (long long)kGemmMaxM, (long long)m);
  if (W->n % 16) return fail(LB_ERR_SHAPE, "lb_gemm_noalloc needs n %% 16 == 0 (got %lld)", (long long)W->n);
  if (!lb::aligned16(x) || !lb::aligned16(y)) return fail(LB_ERR_ALIGN, "x and y must be 16-byte aligned");
  return lb::launch_gemm_noalloc(*W, x, xdt, m, y, ydt, reinterpret_cast<cudaStream_t>(stream));
}

lb_status lb_embed(const lb_weight* W, const int32_t* ids, int64_t count, void* out, int out_dtype,
                   lb_stream stream) {
  lb_status s = check_weight(W);
  if (s != LB_OK) return s;
  if (W->fmt == LB_FMT_TERNARY5_G128) return fail(LB_ERR_UNSUPPORTED, "lb_embed takes the 1-bit and 2-bit ternary formats");
  if (count < 0 || count > INT32_MAX) return fail(LB_ERR_SHAPE, "count must be in [0, 2^31) (got %lld)", (long long)count);
  if (count * ((W->k + 1023) / 1024) > (int64_t(1) << 34) - 8)
    return fail(LB_ERR_SHAPE, "count x K too large for one launch (count %lld, k %lld)", (long long)count,
                (long long)W->k);
  if (!valid_dtype(out_dtype)) return fail(LB_ERR_DTYPE, "unknown output dtype %d", out_dtype);
  if (count == 0) return LB_OK;
  if (!ids || !out) return fail(LB_ERR_NULL, "ids and out must be non-NULL");
  if (!lb::aligned16(out) || (reinterpret_cast<uintptr_t>(ids) & 3u))
    return fail(LB_ERR_ALIGN, "out must be 16-byte aligned and ids 4-byte aligned");
  return lb::launch_embed(*W, ids, count, out, out_dtype, reinterpret_cast<cudaStream_t>(stream));
}

lb_status lb_read_probe(const void* data, size_t bytes, uint32_t* sink, lb_stream stream) {
  if (bytes == 0) return LB_OK;
  if (!data || !sink) return fail(LB_ERR_NULL, "data and sink must be non-NULL");
  if (!lb::aligned16(data) || (reinterpret_cast<uintptr_t>(sink) & 3u))
    return fail(LB_ERR_ALIGN, "data must be 16-byte and sink 4-byte aligned");
  if (bytes % 16) return fail(LB_ERR_SHAPE, "bytes must be a multiple of 16 (got %zu)", bytes);
  return lb::launch_read_probe(data, bytes, sink, reinterpret_cast<cudaStream_t>(stream));
}

// Test-only (not declared in lb.h): make the next GEMV (kernel 1) or GEMM (kernel 2) launch of this
// process give up its pipeline waits after a short bound; 0 clears the setting.
lb_status lb_testing_fault_next_launch(int kernel) {
  if (kernel != 0 && kernel != lb::kTestFaultGemv && kernel != lb::kTestFaultGemm)
    return fail(LB_ERR_UNSUPPORTED, "unknown kernel %d", kernel);
  lb::g_test_fault.store(kernel);
  return LB_OK;
}

lb_status lb_device_error(uint32_t* word, int clear) {
  if (!word) return fail(LB_ERR_NULL, "word is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return lb::cuda_fail(e, "lb_device_error: cudaDeviceSynchronize");
  e = cudaMemcpyFromSymbol(word, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return lb::cuda_fail(e, "lb_device_error: read");
  if (clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
    if (e != cudaSuccess) return lb::cuda_fail(e, "lb_device_error: clear");
  }
  return LB_OK;
}

}  // extern "C"
