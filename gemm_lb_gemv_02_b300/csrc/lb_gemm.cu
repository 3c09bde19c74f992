// Prefill GEMM against packed ternary weights on the 5th-generation tensor cores (tcgen05 + TMEM).
//
//   Y[r][n] = sum_g s[n][g] * sum_{i<128} t[n][128g+i] * X[r][128g+i]
//
// (7minutos.es, "PrismML lanza Bonsai 27B", section "Rendimiento y decodificación especulativa
// DSpark": prefill is compute bound; section "Cómo funciona la compresión": w = s_g t_i.)
//
// Exactness: with FP16 operands every decoded weight s*t (s binary16, t in {-1,0,+1}) is exact and
// every product is exact in the FP32 accumulator, so the group scale costs nothing inside the
// k-loop.  BF16 activations are converted to binary16 once (exact for normal-range values).
//
// Structure (one 128 x 256 output tile per CTA, K in steps of 64):
//   * prologue kernel: X -> binary16, K permuted inside each 16-block to match the decoder's
//     register order, written as ready-made 128-byte-swizzled shared-memory images of the
//     128 x 64 A tiles (one 16 KB contiguous block per tile), so that one bulk copy moves a tile;
//   * warp 8 (one lane): bulk-copies A tiles into a STAGES-deep ring (mbarrier complete_tx);
//   * warps 0-7: thread i owns weight row n0 + i, loads its 2-bit codes and scale, decodes them
//     with one LOP3 + two half2 ops per two weights into the swizzled B tile, and arrives;
//   * warp 9: allocates TMEM (256 columns), one lane issues tcgen05.mma kind::f16 (M128 N256 K16)
//     and commits each stage back to the producers;
//   * epilogue: warps 0-7 read the FP32 accumulator with tcgen05.ld and store BF16/FP16 rows.
// Every mbarrier wait is bounded; a timeout sets a bit in the device error word and the CTA
// finishes (TMEM is always released).
#include <mutex>

#include "lb_common.cuh"

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int kDecodeWarps = 8;
constexpr int kThreads = (kDecodeWarps + 2) * 32;
constexpr uint32_t kTmemCols = 256;
constexpr size_t kSmemBytes = 1024 + STAGES * (A_BYTES + B_BYTES) + 256;

// ------------------------------------------------------------------------------- prologue
// One thread per (row, 16-wide K block): 16 activations -> binary16, positions 2p / 2p+1 of the
// block take elements p / p+8, and the two 16-byte chunks go to their swizzled slots.
template <bool BF>
__global__ void __launch_bounds__(256) xprep_kernel(const uint16_t* __restrict__ x, int64_t m, int k,
                                                    int64_t total, uint8_t* __restrict__ ws,
                                                    uint32_t* __restrict__ err) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= total) return;
  const int kb = k / 16;
  const int64_t row = gid / kb;
  const int blk = static_cast<int>(gid - row * kb);
  const int64_t mt = row / BM;
  const int r = static_cast<int>(row - mt * BM);
  const int kt = blk / 4, b = blk & 3;
  const int KT = k / BK;
  uint32_t X[8];
  if (row < m) {
    const uint4* src = reinterpret_cast<const uint4*>(x + row * k + 16 * blk);
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    X[0] = v0.x; X[1] = v0.y; X[2] = v0.z; X[3] = v0.w; X[4] = v1.x; X[5] = v1.y; X[6] = v1.z; X[7] = v1.w;
    if (BF) {
      bool inf = false;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float lo = __uint_as_float(X[i] << 16), hi = __uint_as_float(X[i] & 0xffff0000u);
        const __half2 h = __floats2half2_rn(lo, hi);
        inf |= __hisinf(__low2half(h)) || __hisinf(__high2half(h));
        X[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      if (inf) atomicOr(err, lb::kErrGemmInputRange);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) X[i] = 0u;
  }
  uint4 c0, c1;
  c0.x = __byte_perm(X[0], X[4], 0x5410); c0.y = __byte_perm(X[0], X[4], 0x7632);
  c0.z = __byte_perm(X[1], X[5], 0x5410); c0.w = __byte_perm(X[1], X[5], 0x7632);
  c1.x = __byte_perm(X[2], X[6], 0x5410); c1.y = __byte_perm(X[2], X[6], 0x7632);
  c1.z = __byte_perm(X[3], X[7], 0x5410); c1.w = __byte_perm(X[3], X[7], 0x7632);
  uint8_t* tile = ws + (static_cast<size_t>(mt) * KT + kt) * A_BYTES + r * 128;
  const int sw = r & 7;
  *reinterpret_cast<uint4*>(tile + (((2 * b) ^ sw) << 4)) = c0;
  *reinterpret_cast<uint4*>(tile + (((2 * b + 1) ^ sw) << 4)) = c1;
}

// ------------------------------------------------------------------------------- B decode
__device__ __forceinline__ uint32_t h2sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t h2mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ constexpr uint32_t e16(int m) {
  return (static_cast<uint32_t>(25 - m) << 10) * 0x00010001u;   // 2^(10-m) in both halves
}

// One 32-bit word = 16 ternary fields -> 8 half2 registers holding s*t for (k = p, k = p + 8).
// Field p sits at mantissa bits (m, m+1) of a half with exponent 2^(10-m): value o + f exactly;
// subtracting o + 1 gives t, multiplying by s gives the exact binary16 weight.
__device__ __forceinline__ void decode_word_st(uint32_t w, uint32_t s2, uint32_t (&o)[8]) {
  const uint32_t w6 = w >> 6;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int m = p <= 4 ? 2 * p : 2 * p - 6;
    const uint32_t src = p <= 4 ? w : w6;
    const uint32_t a = (src & (0x00030003u << m)) | e16(m);
    const uint32_t t = h2sub(a, e16(m) | (0x00010001u << m));
    o[p] = h2mul(t, s2);
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// ------------------------------------------------------------------------------- main kernel
__global__ void __launch_bounds__(kThreads, 1)
    gemm_ternary_kernel(const uint8_t* __restrict__ ws_a, const uint8_t* __restrict__ codes,
                        const uint16_t* __restrict__ scales, uint16_t* __restrict__ y, int m, int n, int k,
                        int y_bf16, uint32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* full_a = bars;
  uint64_t* full_b = bars + STAGES;
  uint64_t* empty = bars + 2 * STAGES;
  uint64_t* tmem_full = bars + 3 * STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int mt = blockIdx.y;
  const int m0 = mt * BM;
  const int KT = k / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      lbdev::mbar_init(&full_a[s], 1);
      lbdev::mbar_init(&full_b[s], kDecodeWarps * 32);
      lbdev::mbar_init(&empty[s], 1);
    }
    lbdev::mbar_init(tmem_full, 1);
    lbdev::fence_mbar_init();
  }
  if (warp == kDecodeWarps + 1) {
    lbdev::tmem_alloc(tmem_slot, kTmemCols);
    lbdev::tmem_relinquish();
  }
  lbdev::tc_fence_before();
  __syncthreads();
  lbdev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == kDecodeWarps) {
    // ---------------- A producer
    if (lane == 0) {
      for (int it = 0; it < KT; ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!lbdev::mbar_wait(&empty[s], ph ^ 1)) { ok = false; break; }
        lbdev::mbar_arrive_expect_tx(&full_a[s], A_BYTES);
        lbdev::bulk_g2s(sA + s * A_BYTES, ws_a + (static_cast<size_t>(mt) * KT + it) * A_BYTES, A_BYTES, &full_a[s]);
      }
    }
  } else if (warp == kDecodeWarps + 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = lbdev::idesc_f16_f32(BM, BN);
      for (int it = 0; it < KT; ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!lbdev::mbar_wait(&full_a[s], ph) || !lbdev::mbar_wait(&full_b[s], ph)) { ok = false; break; }
        lbdev::tc_fence_after();
        const uint32_t a_base = lbdev::smem_u32(sA + s * A_BYTES);
        const uint32_t b_base = lbdev::smem_u32(sB + s * B_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          lbdev::tc_mma_f16(tmem, lbdev::smem_desc_sw128(a_base + 32 * kk), lbdev::smem_desc_sw128(b_base + 32 * kk),
                            idesc, (it | kk) != 0 ? 1u : 0u);
        }
        lbdev::tc_commit(&empty[s]);
      }
      lbdev::tc_commit(tmem_full);
    }
  } else {
    // ---------------- B decoders: thread i <-> weight row n0 + i
    const int i = threadIdx.x;
    const int row = n0 + i;
    const bool valid = row < n;
    const int G = k / lb::kGroup;
    const uint4* crow = reinterpret_cast<const uint4*>(codes + static_cast<int64_t>(valid ? row : 0) * (k / 4));
    const uint16_t* srow = scales + static_cast<int64_t>(valid ? row : 0) * G;
    const uint32_t sw = static_cast<uint32_t>(i & 7);
    uint4 nc0 = make_uint4(0, 0, 0, 0), nc1 = nc0;
    uint32_t ns = 0;
    if (valid) { nc0 = __ldg(crow); nc1 = __ldg(crow + 1); ns = __ldg(srow); }
    for (int g = 0; g < G && ok; ++g) {
      const uint4 c0 = nc0, c1 = nc1;
      const uint32_t s2 = ns * 0x00010001u;
      if (valid && g + 1 < G) { nc0 = __ldg(crow + 2 * (g + 1)); nc1 = __ldg(crow + 2 * (g + 1) + 1); ns = __ldg(srow + g + 1); }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int it = 2 * g + h;
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!lbdev::mbar_wait(&empty[s], ph ^ 1)) { ok = false; break; }
        const uint4 c = h ? c1 : c0;
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
        const uint32_t dst = lbdev::smem_u32(sB + s * B_BYTES + i * 128);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t o[8];
          decode_word_st(words[u], s2, o);
          st_shared_v4(dst + (((2u * u) ^ sw) << 4), o[0], o[1], o[2], o[3]);
          st_shared_v4(dst + (((2u * u + 1u) ^ sw) << 4), o[4], o[5], o[6], o[7]);
        }
        lbdev::fence_proxy_async_smem();
        lbdev::mbar_arrive(&full_b[s]);
      }
    }
    // ---------------- epilogue
    if (!lbdev::mbar_wait(tmem_full, 0)) ok = false;
    lbdev::tc_fence_after();
    const int quad = warp & 3, half = warp >> 2;
    const int token = m0 + 32 * quad + lane;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int col = 128 * half + 32 * c;
      uint32_t v[32];
      lbdev::tmem_ld32(tmem + (static_cast<uint32_t>(32 * quad) << 16) + static_cast<uint32_t>(col), v);
      lbdev::tmem_ld_wait();
      if (token < m) {
        uint16_t* dst = y + static_cast<int64_t>(token) * n + n0 + col;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (n0 + col + 8 * j + 8 <= n) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a = __uint_as_float(v[8 * j + 2 * e]), b = __uint_as_float(v[8 * j + 2 * e + 1]);
              if (y_bf16) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
                pk[e] = *reinterpret_cast<const uint32_t*>(&h);
              } else {
                const __half2 h = __floats2half2_rn(a, b);
                pk[e] = *reinterpret_cast<const uint32_t*>(&h);
              }
            }
            *reinterpret_cast<uint4*>(dst + 8 * j) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
    }
  }
  if (!ok) atomicOr(err, lb::kErrGemmTimeout);
  lbdev::tc_fence_before();
  __syncthreads();
  if (warp == kDecodeWarps + 1) {
    lbdev::tc_fence_after();
    lbdev::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

// Library-owned staging for lb_gemm_noalloc: callers that cannot allocate get the activation tiles
// staged here instead of in a workspace of their own.  Every call rewrites every byte it later
// reads (the prologue writes whole padded tiles), so the array never needs clearing; concurrent
// calls would share it and must be serialised by the caller.
static __device__ __align__(256) uint8_t g_noalloc_scratch[LB_GEMM_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {};
}  // namespace

namespace lb {

lb_status launch_gemm_noalloc(const lb_weight& W, const void* x, int xdt, int64_t m, void* y, int ydt,
                              cudaStream_t st) {
  const size_t need = gemm_workspace_bytes(m, W.k);
  if (need > LB_GEMM_NOALLOC_SCRATCH_BYTES)
    return fail(LB_ERR_WORKSPACE, "lb_gemm_noalloc: m = %lld, k = %lld needs %zu bytes of staging, more than the "
                "%zu-byte library scratch", (long long)m, (long long)W.k, need,
                static_cast<size_t>(LB_GEMM_NOALLOC_SCRATCH_BYTES));
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "lb_gemm_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(LB_ERR_UNSUPPORTED, "lb_gemm_noalloc: device index %d", dev);
  void* ptr = nullptr;
  {
    // first call on this device (with it current): the host-side symbol is only a stand-in, the
    // kernels need the array's device address
    std::lock_guard<std::mutex> lk(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return cuda_fail(e, "lb_gemm_noalloc: cudaGetSymbolAddress");
      g_noalloc_ptr[dev] = p;
    }
    ptr = g_noalloc_ptr[dev];
  }
  return launch_gemm(W, x, xdt, m, y, ydt, ptr, st);
}

size_t gemm_workspace_bytes(int64_t m, int64_t k) {
  const int64_t mpad = (m + BM - 1) / BM * BM;
  return static_cast<size_t>(mpad) * static_cast<size_t>(k) * 2;
}

lb_status launch_gemm(const lb_weight& W, const void* x, int xdt, int64_t m, void* y, int ydt, void* ws,
                      cudaStream_t st) {
  uint32_t* err = device_error_word();
  if (!err) return fail(LB_ERR_CUDA, "lb_gemm: device error word unavailable");
  const int k = static_cast<int>(W.k), n = static_cast<int>(W.n);
  const int64_t mpad = (m + BM - 1) / BM * BM;
  const int64_t total = mpad * (k / 16);
  const int64_t blocks = (total + 255) / 256;
  if (xdt == LB_BF16)
    xprep_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const uint16_t*>(x), m, k, total,
                                                                        static_cast<uint8_t*>(ws), err);
  else
    xprep_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const uint16_t*>(x), m, k, total,
                                                                         static_cast<uint8_t*>(ws), err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "lb_gemm: prologue launch");
  {
    // once per device: raise the dynamic shared-memory limit of the GEMM kernel
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "lb_gemm: cudaGetDevice");
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64 || !done[dev]) {
      e = cudaFuncSetAttribute(gemm_ternary_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemBytes));
      if (e != cudaSuccess) return cuda_fail(e, "lb_gemm: set shared memory size");
      if (dev >= 0 && dev < 64) done[dev] = true;
    }
  }
  const dim3 grid((n + BN - 1) / BN, static_cast<unsigned>(mpad / BM));
  gemm_ternary_kernel<<<grid, kThreads, kSmemBytes, st>>>(static_cast<const uint8_t*>(ws), W.codes, W.scales,
                                                          static_cast<uint16_t*>(y), static_cast<int>(m), n, k,
                                                          ydt == LB_BF16 ? 1 : 0, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "lb_gemm: launch");
  return LB_OK;
}

}  // namespace lb
