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
// Structure (one tile of 128 weight rows x 256 tokens per CTA, K in steps of 64): the decoded
// weights are the MMA's A operand and live in tensor memory; the activations are the B operand in
// shared memory.  Decoder threads own weight rows, i.e. TMEM lanes, so their decoded registers go to
// TMEM with tcgen05.st and never pass through shared memory, which then carries only the
// activation tiles (one bulk-copy write and one tensor-core read per byte).
//   * prologue kernel: X -> binary16, K permuted inside each 16-block to match the decoder's
//     register order, written as ready-made 128-byte-swizzled shared-memory images of 128-token
//     x 64 tiles (one 16 KB contiguous block per tile), so that one bulk copy moves a tile;
//   * warp 8 (one lane): after griddepcontrol.wait, bulk-copies two such tiles (256 tokens) per
//     stage into a STAGES-deep ring (mbarrier complete_tx);
//   * warps 0-7: warp w owns TMEM lanes 32(w % 4) .. +31 (weight rows n0 + lane) and half of each
//     stage's K; it loads 2-bit codes and the group scale, decodes them with one LOP3 + two half2
//     ops per two weights and stores the stage's A columns with tcgen05.st;
//   * warp 9: allocates TMEM (4 A stages x 32 columns + a 256-column FP32 accumulator), one lane
//     issues tcgen05.mma kind::f16 (M128 N256 K16, A from TMEM) and commits each stage back;
//   * epilogue: warps 0-7 read the accumulator with tcgen05.ld (lane = weight row, column =
//     token) and store BF16/FP16 Y[token][row].
// The GEMM is launched with programmatic dependent launch, so the weight decode of the first
// stages overlaps the activation prologue.  Every mbarrier wait is bounded; a timeout sets a bit in
// the device error word and the CTA finishes (TMEM is always released).
#include <mutex>

#include "lb_common.cuh"

namespace {

constexpr int BM = 128, BK = 64, STAGES = 4;     // BM: tokens per activation tile
constexpr int WM = 128, TN = 256;                 // weight rows and tokens per CTA (MMA M and N)
constexpr int A_BYTES = BM * BK * 2;              // one activation tile: 16 KB
constexpr int X_BYTES = 2 * A_BYTES;              // activation stage: 256 tokens x 64
constexpr int kDecodeWarps = 8;
constexpr int kThreads = (kDecodeWarps + 2) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcc = 256;                    // first accumulator column
constexpr size_t kSmemBytes = 1024 + STAGES * X_BYTES + 256;

// ------------------------------------------------------------------------------- prologue
// One thread per (row, 16-wide K block): 16 activations -> binary16, positions 2p / 2p+1 of the
// block take elements p / p+8, and the two 16-byte chunks go to their swizzled slots.
template <bool BF>
__global__ void __launch_bounds__(256) xprep_kernel(const uint16_t* __restrict__ x, int64_t m, int k,
                                                    int64_t total, uint8_t* __restrict__ ws,
                                                    uint32_t* __restrict__ err) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the GEMM may start decoding weights
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
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 32 lanes x 16 consecutive columns; thread i writes lane (base lane + i), register j -> column j.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_ternary_kernel(const uint8_t* __restrict__ ws_x, const uint8_t* __restrict__ codes,
                        const uint16_t* __restrict__ scales, uint16_t* __restrict__ y, int m, int mpad, int n,
                        int k, int y_bf16, uint32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sX = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sX + STAGES * X_BYTES);
  uint64_t* full_x = bars;
  uint64_t* a_full = bars + STAGES;
  uint64_t* empty = bars + 2 * STAGES;
  uint64_t* tmem_full = bars + 3 * STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * WM;
  const int t0 = blockIdx.y * TN;                                  // first token of the tile
  const int ntiles = min(2, (mpad - t0) / BM);                     // 128-token activation tiles (1 or 2)
  const int KT = k / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      lbdev::mbar_init(&full_x[s], 1);
      lbdev::mbar_init(&a_full[s], kDecodeWarps);
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
    // ---------------- activation producer (the prologue kernel wrote the tiles)
    griddep_wait();
    if (lane == 0) {
      const uint32_t bytes = static_cast<uint32_t>(ntiles * A_BYTES);
      const size_t mt0 = static_cast<size_t>(t0 / BM);
      for (int it = 0; it < KT; ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!lbdev::mbar_wait(&empty[s], ph ^ 1)) { ok = false; break; }
        lbdev::mbar_arrive_expect_tx(&full_x[s], bytes);
        for (int tt = 0; tt < ntiles; ++tt)
          lbdev::bulk_g2s(sX + s * X_BYTES + tt * A_BYTES, ws_x + ((mt0 + tt) * KT + it) * A_BYTES, A_BYTES,
                          &full_x[s]);
      }
    }
  } else if (warp == kDecodeWarps + 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = lbdev::idesc_f16_f32(WM, static_cast<uint32_t>(ntiles * BM));
      for (int it = 0; it < KT; ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!lbdev::mbar_wait(&full_x[s], ph) || !lbdev::mbar_wait(&a_full[s], ph)) { ok = false; break; }
        lbdev::tc_fence_after();
        const uint32_t x_base = lbdev::smem_u32(sX + s * X_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_f16_ts(tmem + kAcc, tmem + static_cast<uint32_t>(32 * s + 8 * kk),
                        lbdev::smem_desc_sw128(x_base + 32 * kk), idesc, (it | kk) != 0 ? 1u : 0u);
        lbdev::tc_commit(&empty[s]);                               // frees the A columns and the X slot
      }
      lbdev::tc_commit(tmem_full);
    }
  } else {
    // ---------------- weight decoders: warp w -> TMEM lanes 32q.. (rows n0 + 32q + lane), K half h
    const int q = warp & 3, h = warp >> 2;
    const int row = 32 * q + lane;
    const int wrow = n0 + row;
    const bool valid = wrow < n;
    const int G = k / lb::kGroup;
    const uint8_t* crow = codes + static_cast<int64_t>(valid ? wrow : 0) * (k / 4) + 8 * h;
    const uint16_t* srow = scales + static_cast<int64_t>(valid ? wrow : 0) * G;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    uint2 nc = make_uint2(0u, 0u);
    uint32_t ns = 0;
    if (valid) { nc = __ldg(reinterpret_cast<const uint2*>(crow)); ns = __ldg(srow); }
    for (int it = 0; it < KT && ok; ++it) {
      const int s = it % STAGES;
      const uint32_t ph = (it / STAGES) & 1;
      const uint2 c = nc;
      const uint32_t s2 = ns * 0x00010001u;
      if (valid && it + 1 < KT) {                                  // next stage: 16 bytes of codes per row
        nc = __ldg(reinterpret_cast<const uint2*>(crow + 16 * (it + 1)));
        ns = __ldg(srow + (it + 1) / 2);
      }
      uint32_t o[16];
      {
        uint32_t a8[8], b8[8];
        decode_word_st(c.x, s2, a8);
        decode_word_st(c.y, s2, b8);
#pragma unroll
        for (int i = 0; i < 8; ++i) { o[i] = a8[i]; o[8 + i] = b8[i]; }
      }
      if (!lbdev::mbar_wait(&empty[s], ph ^ 1)) { ok = false; break; }   // the stage's MMAs retired
      lbdev::tc_fence_after();
      tmem_st16(lane_base + static_cast<uint32_t>(32 * s + 16 * h), o);
      tmem_st_wait();
      lbdev::tc_fence_before();
      __syncwarp();
      if (lane == 0) lbdev::mbar_arrive(&a_full[s]);
    }
    // ---------------- epilogue: lane = weight row, columns = tokens
    if (!lbdev::mbar_wait(tmem_full, 0)) ok = false;
    lbdev::tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int col = 128 * h + 32 * c;                            // token offset in the tile
      uint32_t v[32];
      lbdev::tmem_ld32(lane_base + kAcc + static_cast<uint32_t>(col), v);
      lbdev::tmem_ld_wait();
      if (valid) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int tok = t0 + col + j;
          if (tok < m) {
            const float f = __uint_as_float(v[j]);
            y[static_cast<int64_t>(tok) * n + wrow] =
                y_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(f)) : __half_as_ushort(__float2half_rn(f));
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n + WM - 1) / WM, static_cast<unsigned>((mpad + TN - 1) / TN), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the prologue kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemm_ternary_kernel, static_cast<const uint8_t*>(ws), W.codes, W.scales,
                         static_cast<uint16_t*>(y), static_cast<int>(m), static_cast<int>(mpad), n, k,
                         ydt == LB_BF16 ? 1 : 0, err);
  if (e != cudaSuccess) return cuda_fail(e, "lb_gemm: launch");
  return LB_OK;
}

}  // namespace lb
