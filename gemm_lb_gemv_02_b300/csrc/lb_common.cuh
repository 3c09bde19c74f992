// Internal helpers of liblb: host-side status plumbing and thin inline-PTX wrappers for the
// sm_103a features the kernels use (mbarrier, bulk async copies, tcgen05 / TMEM).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cstddef>

#include "../../include/lb.h"

namespace lb {

constexpr int kGroup = 128;

// ----------------------------------------------------------------------------------- host side
lb_status fail(lb_status s, const char* fmt, ...);           // records the thread-local text
lb_status cuda_fail(cudaError_t e, const char* where);       // LB_ERR_CUDA with the CUDA text
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int sm_count();                                              // SMs of the current device

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry point (nullptr if the
// driver does not provide it).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// Device word with sticky error bits (see lb_device_error); one per device, owned by lb_api.cu.
uint32_t* device_error_word();
// Unique id of the current CUDA context (0 if unknown); device addresses of module-scope variables
// are cached per context id.
unsigned long long context_id();
constexpr uint32_t kErrGemmTimeout = 1u;        // a GEMM pipeline wait gave up
constexpr uint32_t kErrEmbedId = 4u;            // an embedding row id outside [0, n)

// Bound of every mbarrier wait in a kernel, and the short bound of a launch that tests the give-up
// path (see take_test_fault).
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kTestWaitNs = 1000000ull;
// Test-only switch, off unless a test sets it through lb_testing_fault_next_launch (exported for the
// test suite, not declared in lb.h): the next launch of the named kernel issues none of its
// asynchronous copies and waits with the short bound, so that every pipeline wait runs out and the
// kernel's give-up path (error bit, no compute, cluster barriers joined, TMEM released) executes.
// take_test_fault returns true once per setting.
constexpr int kTestFaultGemv = 1;
constexpr int kTestFaultGemm = 2;
bool take_test_fault(int kernel);

// Launchers implemented by the kernel translation units.  They assume validated arguments.
lb_status launch_pack_1bit(const float* w, int64_t n, int64_t k, uint8_t* codes, uint16_t* scales,
                           cudaStream_t st, uint32_t* flags_out);
lb_status launch_pack_ternary(const int8_t* t, const uint16_t* s_in, int64_t n, int64_t k,
                              uint8_t* codes, uint16_t* scales, cudaStream_t st, uint32_t* flags_out);
lb_status launch_gemv(const lb_weight& W, const void* x, int xdt, int batch, void* y, cudaStream_t st);
// Whether launch_gemv takes a five-per-byte weight (batch 1, lookup tables); otherwise
// launch_gemv_t5 (CUDA cores) does.
bool gemv_t5_lut_ok(const lb_weight& W, int batch);
// The GEMM of 1 .. 32 token rows on the GEMV's mma.sync engine (lb_gemm_ms.cu); lb_gemm dispatches
// to it.  The tensor maps are lb_gemm's (codes: 128 x 128-row boxes, 128-byte swizzle; scales:
// 8 x 128-row boxes).
constexpr int64_t kGemmSmallM = 32;
size_t gemm_ms_workspace_bytes(int64_t m, int64_t k);
lb_status launch_gemm_ms(const lb_weight& W, const void* x, int xdt, int64_t m, void* y, int ydt, void* ws,
                         const CUtensorMap& tm_codes, const CUtensorMap& tm_scales, int scales_tma, bool fault,
                         cudaStream_t st);
lb_status launch_pack_ternary5(const int8_t* t, const uint16_t* s_in, int64_t n, int64_t k, uint8_t* codes,
                               uint16_t* scales, cudaStream_t st, uint32_t* flags_out);
lb_status launch_gemv_t5(const lb_weight& W, const void* x, int xdt, int batch, void* y, cudaStream_t st);
lb_status launch_gemv_swiglu(const lb_weight& Wg, const lb_weight& Wu, const void* x, int xdt, int batch, void* h,
                             cudaStream_t st);
lb_status launch_gemv_batched(const lb_gemv_problem* probs, int count, int xdt, int batch, cudaStream_t st);
size_t gemm_workspace_bytes(int64_t m, int64_t k);
lb_status launch_gemm(const lb_weight& W, const void* x, int xdt, int64_t m, void* y, int ydt,
                      void* ws, cudaStream_t st);
lb_status launch_embed(const lb_weight& W, const int32_t* ids, int64_t count, void* out, int out_dtype,
                       cudaStream_t st);
lb_status launch_gemm_noalloc(const lb_weight& W, const void* x, int xdt, int64_t m, void* y, int ydt,
                              cudaStream_t st);
lb_status launch_read_probe(const void* data, size_t bytes, uint32_t* sink, cudaStream_t st);

// Pack validation bits reported by the pack kernels.
constexpr uint32_t kPackNonFinite = 1u;
constexpr uint32_t kPackRange = 2u;
constexpr uint32_t kPackCode = 4u;

}  // namespace lb

// ----------------------------------------------------------------------------------- device side
namespace lbdev {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// mbarrier ------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: returns false (and the caller reports an error) if the phase has not completed
// after about `limit_ns` nanoseconds of global time.  Each try_wait carries a suspend-time hint, so
// a waiting thread sleeps in the barrier unit until the phase completes instead of spinning and
// taking issue slots from the threads that do the work.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
  const uint64_t t0 = globaltimer_ns();
  do {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
  } while (globaltimer_ns() - t0 < limit_ns);
  return false;
}
// Bounded wait for a thread that is usually far ahead of the phase it waits for (a producer
// waiting for a free ring slot): between polls it sleeps on the SM's nanosleep timer, so that its
// warp issues almost nothing while it waits and leaves the issue slots of its sub-partition to the
// warps that do the work.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  do {
    __nanosleep(128);
    if (mbar_try_wait(bar, parity)) return true;
  } while (globaltimer_ns() - t0 < limit_ns);
  return false;
}

// async proxy / bulk copies -------------------------------------------------------------------
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 1-D bulk copy global -> shared, completion counted on `bar` (transaction bytes).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled TMA load of the box at coordinates (c0 = innermost, c1) of `tmap` into shared memory,
// completion counted on `bar`.  c0 * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// tcgen05 / TMEM ------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D(tmem) (+)= A(smem desc) * B(smem desc), kind::f16, issued by one thread.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once all previously issued tcgen05.mma of this thread have completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns; thread i receives lane (base_lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format) for a K-major operand stored with the 128-byte
// swizzle: rows of 128 bytes, 8-row atoms of 1024 bytes (stride between atoms = 1024 bytes).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);          // start address
  d |= static_cast<uint64_t>(1u) << 16;                         // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;                 // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;                         // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                         // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16: FP16 A and B (K-major), FP32 accumulator, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t m, uint32_t n) {
  return (1u << 4)                  // D format: F32
         | (0u << 7) | (0u << 10)   // A, B format: F16
         | ((n >> 3) << 17) | ((m >> 4) << 24);
}

}  // namespace lbdev
