// Prefill GEMM against packed 1-bit or ternary weights on the 5th-generation tensor cores
// (tcgen05 + TMEM).
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
// Structure (one tile of 128 weight rows x up to 256 tokens per CTA, K in steps of 64): the decoded
// weights are the MMA's A operand and live in tensor memory; the activations are the B operand in
// shared memory.  Decoder threads own weight rows, i.e. TMEM lanes, so their decoded registers go to
// TMEM with tcgen05.st and never pass through shared memory.
//   * prologue kernel: X -> binary16, K permuted inside each 16- (ternary) or 32-block (1-bit) to
//     match the decoder's register order, written as ready-made 128-byte-swizzled shared-memory
//     images of 128-token x 64 tiles (one 16 KB contiguous block per tile), so that one bulk copy
//     moves a tile;
//   * warp 16 (one lane): after griddepcontrol.wait, bulk-copies the token rows of one or two such
//     tiles per stage into the stage ring (mbarrier complete_tx);
//   * warp 18 (one lane): TMA-loads the CTA's packed codes, 128 rows x 128 bytes per chunk (512 K of
//     ternary, 1024 K of 1-bit), into a CR-deep ring, so the decoders read their codes from shared
//     memory long after the HBM latency was paid;
//   * warp 19: the group scales, 128 rows x 8 groups per chunk, into an SR-deep ring: one TMA per
//     chunk when a scale row is a multiple of 16 bytes, otherwise 32 lanes load and store them;
//   * warps 0-15: two groups of 8 take alternate stages; in a group, warp w owns TMEM lanes
//     32(w % 4) .. +31 (weight rows n0 + lane) and half of the stage's K; it decodes its codes with
//     the group scale (a LOP3 and two half2 operations per two ternary weights, one LOP3 per two
//     1-bit weights), stores the stage's A columns with tcgen05.st and publishes the store after it
//     has decoded its next stage;
//   * warp 17: allocates TMEM (an 8-stage ring of 32 A columns + a 256-column FP32 accumulator); one
//     lane issues tcgen05.mma kind::f16 (M128, N = the tile's tokens rounded up to 16, K16, A from
//     TMEM): one wait and four MMAs per stage;
//   * one stage ring (8 stages with one activation tile, 5 with two) carries both operands: its full
//     barrier counts the 8 decoder warps of the stage plus the activation bytes, and one commit
//     per stage frees the TMEM columns and the activation slot together;
//   * epilogue: warps 0-15 read the accumulator with tcgen05.ld (lane = weight row, 64 tokens per
//     warp) and store BF16/FP16 Y[token][row].
// The GEMM is launched with programmatic dependent launch, so the weight decode of the first
// stages overlaps the activation prologue.  Every mbarrier wait is bounded; a timeout sets a bit in
// the device error word and the CTA finishes (TMEM is always released).
#include <cstring>
#include <mutex>

#include "lb_common.cuh"

namespace {

constexpr int BM = 128, BK = 64;                 // BM: tokens per activation tile
constexpr int WM = 128, TN = 256;                 // weight rows and tokens per CTA (MMA M and N)
constexpr int A_BYTES = BM * BK * 2;              // one activation tile: 16 KB
constexpr int XR_BYTES = 10 * A_BYTES;            // activation ring: up to 8 one-tile or 5 two-tile stages
constexpr int DMAX = 8;                           // stage ring depth (decoded A stages in TMEM: 32 columns each)
constexpr int kDecodeWarps = 16;                  // two groups of 8, alternate stages
constexpr int kWarpX = kDecodeWarps, kWarpMma = kDecodeWarps + 1;
constexpr int kWarpCodes = kDecodeWarps + 2, kWarpScales = kDecodeWarps + 3;
constexpr int kThreads = (kDecodeWarps + 4) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcc = 256;                    // first accumulator column
constexpr int CR = 3, C_BYTES = WM * 128;         // code ring: chunks of 128 rows x 128 bytes
constexpr int SR = 4, S_BYTES = WM * 16;          // scale ring: chunks of 128 rows x 8 groups
constexpr int kBars = 2 * DMAX + 1 + 2 * CR + 2 * SR;
constexpr size_t kSmemBytes = 1024 + XR_BYTES + CR * C_BYTES + SR * S_BYTES + kBars * 8 + 16 + TN * 4;
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(DMAX * 32 <= 256, "A ring and accumulator share 512 TMEM columns");

// ------------------------------------------------------------------------------- prologue
// One CTA per token row (rows m .. mpad - 1 are the zero padding of the last tile).  bfloat16 rows
// are scaled by an exact power of two 2^p chosen so that the row's largest magnitude lies in
// [2^15, 2^16) (|p| <= 126), then converted to binary16: every element within 2^32 of the row
// maximum is then exact (a bfloat16 value has 8 significant bits, and binary16 holds 8 bits down
// to 2^-17), smaller ones round to the binary16 subnormal grid (an error of at most 2^-25 in the
// scaled units), and nothing overflows.  The row's factor 2^-p goes to fac[row] for the epilogue;
// binary16 rows are copied unchanged (factor 1).  The K order inside each 16- (ternary) or 32-block
// (1-bit) matches the decoder's registers: ternary (SPAN 16) puts elements p / p + 8 at positions
// 2p / 2p + 1; 1-bit (SPAN 32) puts elements r / r + 16 at positions 2r / 2r + 1.  The 16-byte
// chunks go to their 128-byte-swizzled slots of the 128-token x 64 tile image.
template <bool BF, int FMT>
__global__ void __launch_bounds__(256) xprep_kernel(const uint16_t* __restrict__ x, int64_t m, int k,
                                                    uint8_t* __restrict__ ws, float* __restrict__ fac) {
  constexpr int SPAN = FMT == 1 ? 32 : 16;
  constexpr int NW = SPAN / 2;                                   // 32-bit words per block
  constexpr int CACHE = FMT == 1 ? 1 : 2;                        // blocks a thread keeps in registers
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the GEMM may start decoding weights
  __shared__ uint32_t warp_max[8];
  const int64_t row = blockIdx.x;
  const bool live = row < m;
  const int kb = k / SPAN;
  const int64_t mt = row / BM;
  const int r = static_cast<int>(row - mt * BM);
  const int KT = k / BK;
  const uint4* src_row = reinterpret_cast<const uint4*>(x + row * k);
  auto load = [&](int blk, uint32_t (&X)[NW]) {
    if (live && blk < kb) {
#pragma unroll
      for (int i = 0; i < NW / 4; ++i) {
        const uint4 v = __ldg(src_row + (SPAN / 8) * blk + i);
        X[4 * i] = v.x; X[4 * i + 1] = v.y; X[4 * i + 2] = v.z; X[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < NW; ++i) X[i] = 0u;
    }
  };
  uint32_t C[CACHE][NW];                                         // blocks threadIdx.x + 256 c
#pragma unroll
  for (int c = 0; c < CACHE; ++c) load(threadIdx.x + 256 * c, C[c]);
  float sc = 1.f;
  if (BF && live) {
    uint32_t mx = 0;
    auto fold = [&](const uint32_t (&X)[NW]) {
#pragma unroll
      for (int i = 0; i < NW; ++i) mx = max(mx, max((X[i] << 16) & 0x7f800000u, X[i] & 0x7f800000u));
    };
#pragma unroll
    for (int c = 0; c < CACHE; ++c) fold(C[c]);
    for (int blk = threadIdx.x + 256 * CACHE; blk < kb; blk += 256) {   // rows longer than the cache
      uint32_t X[NW];
      load(blk, X);
      fold(X);
    }
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) mx = max(mx, warp_max[w]);      // exponent fields order like magnitudes
    const int e = static_cast<int>(mx >> 23) - 127;              // -127: zero or subnormal maximum
    const int p = min(126, max(-126, 15 - e));
    sc = __uint_as_float(static_cast<uint32_t>(127 + p) << 23);
    if (threadIdx.x == 0) fac[row] = __uint_as_float(static_cast<uint32_t>(127 - p) << 23);
  } else if (threadIdx.x == 0) {
    fac[row] = 1.f;
  }
  auto emit = [&](int blk, uint32_t (&X)[NW]) {
    if (blk >= kb) return;
    const int kt = blk / (BK / SPAN), b = blk % (BK / SPAN);
    if (BF && live) {
#pragma unroll
      for (int i = 0; i < NW; ++i) {
        const float lo = __uint_as_float(X[i] << 16) * sc, hi = __uint_as_float(X[i] & 0xffff0000u) * sc;
        const __half2 h = __floats2half2_rn(lo, hi);
        X[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
    // output word j = (element j, element j + SPAN/2)
    uint32_t P[NW];
#pragma unroll
    for (int j = 0; j < NW; ++j) P[j] = __byte_perm(X[j >> 1], X[(j >> 1) + NW / 2], (j & 1) ? 0x7632 : 0x5410);
    uint8_t* tile = ws + (static_cast<size_t>(mt) * KT + kt) * A_BYTES + r * 128;
    const int sw = r & 7;
#pragma unroll
    for (int c = 0; c < NW / 4; ++c)
      *reinterpret_cast<uint4*>(tile + ((((NW / 4) * b + c) ^ sw) << 4)) =
          make_uint4(P[4 * c], P[4 * c + 1], P[4 * c + 2], P[4 * c + 3]);
  };
#pragma unroll
  for (int c = 0; c < CACHE; ++c) emit(threadIdx.x + 256 * c, C[c]);
  for (int blk = threadIdx.x + 256 * CACHE; blk < kb; blk += 256) {
    uint32_t X[NW];
    load(blk, X);
    emit(blk, X);
  }
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

// One 1-bit word (32 codes, bit i = weight i) -> 16 half2 registers holding s*t for (k = r,
// k = r + 16): shifting left by 15 - r puts bits r and r + 16 into the two sign positions, and
// t = +1 for bit 1, so s*t = s with the sign bit set where the code bit is 0 (exact).
__device__ __forceinline__ void decode_word_1bit(uint32_t w, uint32_t s2, uint32_t (&o)[16]) {
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const uint32_t sh = w << (15 - r);
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0xA6;" : "=r"(v) : "r"(sh), "r"(0x80008000u), "r"(s2));    // (~a & b) ^ c
    o[r] = v;
  }
}

// ------------------------------------------------------------------------------- main kernel
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
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

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_lowbit_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                       const uint8_t* __restrict__ ws_x, const float* __restrict__ fac,
                       const uint16_t* __restrict__ scales, uint16_t* __restrict__ y, int m, int mpad, int n, int k,
                       int scales_tma, int y_bf16, uint32_t* __restrict__ err, uint64_t wait_ns, int test_fault) {
  constexpr int RB = FMT == 1 ? 8 : 16;                            // code bytes per row per 64-K stage
  constexpr int SPC = 128 / RB;                                    // stages per code chunk (even)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sX = smem;
  uint8_t* sC = sX + XR_BYTES;
  uint8_t* sS = sC + CR * C_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sS + SR * S_BYTES);
  uint64_t* full = bars;                        // stage ready: its activations landed + its A stored
  uint64_t* empty = bars + DMAX;                // the stage's MMAs retired (frees both slots)
  uint64_t* tmem_full = bars + 2 * DMAX;
  uint64_t* c_full = tmem_full + 1;             // code chunk landed
  uint64_t* c_empty = c_full + CR;              // code chunk read by every decoder warp
  uint64_t* s_full = c_empty + CR;
  uint64_t* s_empty = s_full + SR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_empty + SR);
  float* sfac = reinterpret_cast<float*>(tmem_slot + 4);        // the tile's token factors (TN)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * WM;
  const int t0 = blockIdx.y * TN;                                  // first token of the tile
  // MMA N: the tile's tokens rounded up to 16 (mid-M products do not pay for 256 columns)
  const int nmma = min(TN, (min(m - t0, TN) + 15) / 16 * 16);
  const int ntiles = nmma > BM ? 2 : 1;                            // 128-token activation tiles
  const int D = ntiles == 1 ? DMAX : 5;                            // stage ring depth
  const int x_slot = ntiles * A_BYTES;
  const int KT = k / BK;
  const int G = k / lb::kGroup;
  const int NC = (KT + SPC - 1) / SPC;                             // code chunks
  const int NS = (G + 7) / 8;                                      // scale chunks (16 stages each)

  if (threadIdx.x == 0) {
    for (int s = 0; s < DMAX; ++s) {
      lbdev::mbar_init(&full[s], 8 + 1);                           // 8 decoder warps + the activation copy
      lbdev::mbar_init(&empty[s], 1);
    }
    lbdev::mbar_init(tmem_full, 1);
    for (int c = 0; c < CR; ++c) {
      lbdev::mbar_init(&c_full[c], 1);
      lbdev::mbar_init(&c_empty[c], kDecodeWarps);
    }
    for (int c = 0; c < SR; ++c) {
      lbdev::mbar_init(&s_full[c], scales_tma ? 1 : 32);
      lbdev::mbar_init(&s_empty[c], kDecodeWarps);
    }
    lbdev::fence_mbar_init();
  }
  if (warp == kWarpMma) {
    lbdev::tmem_alloc(tmem_slot, kTmemCols);
    lbdev::tmem_relinquish();
  }
  lbdev::tc_fence_before();
  __syncthreads();
  lbdev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == kWarpX) {
    // ---------------- activation producer (the prologue kernel wrote the tiles)
    griddep_wait();
    // the tile's per-token factors for the epilogue; the stage barriers, the last commit and the
    // epilogue's wait order these stores before the epilogue's loads
    for (int i = lane; i < TN; i += 32) sfac[i] = t0 + i < mpad ? fac[t0 + i] : 0.f;
    __syncwarp();                                  // the whole warp's stores precede lane 0's arrivals
    if (lane == 0) {
      // only the token rows the MMA reads (nmma rows of 128 bytes; the second tile's rows follow
      // the first tile's 128)
      const uint32_t bytes = static_cast<uint32_t>(nmma * 128);
      const uint32_t tile_bytes[2] = {static_cast<uint32_t>(min(nmma, BM) * 128),
                                      static_cast<uint32_t>(max(nmma - BM, 0) * 128)};
      const size_t mt0 = static_cast<size_t>(t0 / BM);
      int it = 0, s = 0;
      uint32_t ph = 0;
      for (; it < KT && !test_fault; ++it) {          // test_fault: issue nothing, so every wait gives up
        if (!lbdev::mbar_wait(&empty[s], ph ^ 1, wait_ns)) { ok = false; break; }
        lbdev::mbar_arrive_expect_tx(&full[s], bytes);
        for (int tt = 0; tt < ntiles; ++tt)
          lbdev::bulk_g2s(sX + s * x_slot + tt * A_BYTES, ws_x + ((mt0 + tt) * KT + it) * A_BYTES, tile_bytes[tt],
                          &full[s]);
        if (++s == D) { s = 0; ph ^= 1u; }
      }
      for (int j = max(0, it - D); j < it; ++j)                  // copies in flight land before exit
        if (!lbdev::mbar_wait(&full[j % D], (j / D) & 1, wait_ns)) ok = false;
    }
  } else if (warp == kWarpCodes) {
    // ---------------- code producer: 128 rows x 128 bytes per chunk, 128-byte swizzle
    if (lane == 0) {
      lbdev::prefetch_tmap(&tm_codes);
      int cc = 0;
      for (; cc < NC && !test_fault; ++cc) {
        const int c = cc % CR;
        if (!lbdev::mbar_wait(&c_empty[c], ((cc / CR) & 1) ^ 1, wait_ns)) { ok = false; break; }
        lbdev::mbar_arrive_expect_tx(&c_full[c], C_BYTES);
        lbdev::tma_load_2d(sC + c * C_BYTES, &tm_codes, 128 * cc, n0, &c_full[c]);
      }
      for (int j = max(0, cc - CR); j < cc; ++j)
        if (!lbdev::mbar_wait(&c_full[j % CR], (j / CR) & 1, wait_ns)) ok = false;
    }
  } else if (warp == kWarpScales) {
    // ---------------- scale producer: 128 rows x 8 groups per chunk, [row][group] in shared memory
    if (scales_tma) {
      if (lane == 0) {
        lbdev::prefetch_tmap(&tm_scales);
        int sc = 0;
        for (; sc < NS; ++sc) {
          const int c = sc % SR;
          if (!lbdev::mbar_wait(&s_empty[c], ((sc / SR) & 1) ^ 1, wait_ns)) { ok = false; break; }
          lbdev::mbar_arrive_expect_tx(&s_full[c], S_BYTES);
          lbdev::tma_load_2d(sS + c * S_BYTES, &tm_scales, 8 * sc, n0, &s_full[c]);
        }
        for (int j = max(0, sc - SR); j < sc; ++j)
          if (!lbdev::mbar_wait(&s_full[j % SR], (j / SR) & 1, wait_ns)) ok = false;
      }
    } else {
      // a scale row is not a multiple of 16 bytes: lane l loads rows l, l + 32, l + 64, l + 96 of
      // the next chunk while the decoders use the previous ones
      uint32_t v[16];
      auto load = [&](int sc) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = n0 + lane + 32 * i;
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            const int g = 8 * sc + j;
            const uint16_t* p = scales + static_cast<int64_t>(row) * G + g;
            const uint32_t lo = (row < n && g < G) ? __ldg(p) : 0u;
            const uint32_t hi = (row < n && g + 1 < G) ? __ldg(p + 1) : 0u;
            v[4 * i + j / 2] = lo | (hi << 16);
          }
        }
      };
      load(0);
      for (int sc = 0; sc < NS; ++sc) {
        const int c = sc % SR;
        if (!lbdev::mbar_wait(&s_empty[c], ((sc / SR) & 1) ^ 1, wait_ns)) { ok = false; break; }
        uint8_t* dst = sS + c * S_BYTES;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(dst + (lane + 32 * i) * 16) = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2],
                                                                              v[4 * i + 3]);
        lbdev::mbar_arrive(&s_full[c]);
        if (sc + 1 < NS) load(sc + 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer.  One thread issues every MMA, so its loop is kept short: one wait
    // and one commit per stage, ring positions advance by counters, operand addresses by additions
    // (a descriptor's start-address field counts 16-byte units), and only the first MMA of the tile
    // clears the accumulator.
    if (lane == 0) {
      const uint32_t idesc = lbdev::idesc_f16_f32(WM, static_cast<uint32_t>(nmma));
      const uint64_t bdesc0 = lbdev::smem_desc_sw128(lbdev::smem_u32(sX));
      const uint32_t slot16 = static_cast<uint32_t>(x_slot >> 4);
      int s = 0;
      uint32_t ph = 0;
      uint64_t bd = bdesc0;
      uint32_t acc_in = 0;
      for (int it = 0; it < KT; ++it) {
        if (!lbdev::mbar_wait(&full[s], ph, wait_ns)) { ok = false; break; }
        lbdev::tc_fence_after();
        const uint32_t ad = tmem + static_cast<uint32_t>(32 * s);
        tc_mma_f16_ts(tmem + kAcc, ad, bd, idesc, acc_in);
        tc_mma_f16_ts(tmem + kAcc, ad + 8, bd + 2, idesc, 1u);
        tc_mma_f16_ts(tmem + kAcc, ad + 16, bd + 4, idesc, 1u);
        tc_mma_f16_ts(tmem + kAcc, ad + 24, bd + 6, idesc, 1u);
        acc_in = 1u;
        lbdev::tc_commit(&empty[s]);                               // frees the activation slot and the A columns
        bd += slot16;
        if (++s == D) { s = 0; ph ^= 1u; bd = bdesc0; }
      }
      lbdev::tc_commit(tmem_full);
    }
  } else {
    // ---------------- weight decoders: warp w -> TMEM lanes 32q.. (rows n0 + 32q + lane), K half h
    // of every stage of parity par
    const int q = warp & 3, h = (warp >> 2) & 1, par = warp >> 3;
    const int row = 32 * q + lane;                                 // row inside the chunk images
    const int wrow = n0 + row;
    const bool valid = wrow < n;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const uint8_t* crow = sC + row * 128;                          // this row's 128 bytes of a code chunk
    const uint8_t* srow = sS + row * 16;
    // ring positions of this warp's stages (it = par, par + 2, ...), advanced by counters:
    // stage slot s / phase ph, code chunk slot c / phase cph / stage j inside it, scale chunk
    // slot cs / phase sph / group sj inside it
    int s = par, j = par, c = 0, cs = 0, sj = 0;
    uint32_t ph = 0, cph = 0, sph = 0;
    int prev_s = -1;
    for (int it = par; it < KT && ok; it += 2) {
      if (j < 2 && !lbdev::mbar_wait(&c_full[c], cph, wait_ns)) { ok = false; break; }
      if (sj == 0 && !lbdev::mbar_wait(&s_full[cs], sph, wait_ns)) { ok = false; break; }
      // the chunk's 16-byte units are stored at unit ^ (row % 8) (128-byte swizzle)
      uint2 w;
      if (FMT == 1) {
        const int byte = 8 * j + 4 * h;
        w.x = *reinterpret_cast<const uint32_t*>(crow + c * C_BYTES + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15)));
        w.y = 0u;
      } else {
        w = *reinterpret_cast<const uint2*>(crow + c * C_BYTES + (((j ^ (row & 7)) << 4) | (8 * h)));
      }
      const uint32_t s2 = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(srow + cs * S_BYTES + 2 * sj)) *
                          0x00010001u;
      __syncwarp();
      if (lane == 0) {
        if (j >= SPC - 2) lbdev::mbar_arrive(&c_empty[c]);         // this warp's last stage of the chunk
        if (sj == 7) lbdev::mbar_arrive(&s_empty[cs]);
      }
      uint32_t o[16];
      if (FMT == 1) {
        decode_word_1bit(w.x, s2, o);                              // word h: k = 32h .. 32h + 31
      } else {
        uint32_t a8[8], b8[8];                                     // words 2h, 2h + 1
        decode_word_st(w.x, s2, a8);
        decode_word_st(w.y, s2, b8);
#pragma unroll
        for (int i = 0; i < 8; ++i) { o[i] = a8[i]; o[8 + i] = b8[i]; }
      }
      // this warp's previous TMEM store ran while this stage was decoded: publish it now
      if (prev_s >= 0) {
        tmem_st_wait();
        lbdev::tc_fence_before();
        __syncwarp();
        if (lane == 0) lbdev::mbar_arrive(&full[prev_s]);
      }
      if (!lbdev::mbar_wait(&empty[s], ph ^ 1, wait_ns)) { ok = false; break; }   // the slot's MMAs retired
      lbdev::tc_fence_after();
      tmem_st16(lane_base + static_cast<uint32_t>(32 * s + 16 * h), o);
      prev_s = s;
      if ((s += 2) >= D) { s -= D; ph ^= 1u; }
      if ((j += 2) >= SPC) {
        j -= SPC;
        if (++c == CR) { c = 0; cph ^= 1u; }
      }
      if (++sj == 8) {
        sj = 0;
        if (++cs == SR) { cs = 0; sph ^= 1u; }
      }
    }
    if (prev_s >= 0 && ok) {
      tmem_st_wait();
      lbdev::tc_fence_before();
      __syncwarp();
      if (lane == 0) lbdev::mbar_arrive(&full[prev_s]);
    }
    // ---------------- epilogue: lane = weight row, columns = tokens; warp (h, par) takes 64 of them
    if (!lbdev::mbar_wait(tmem_full, 0, wait_ns)) ok = false;
    lbdev::tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      const int col = 64 * (2 * par + h) + 32 * c;                 // token offset in the tile
      if (t0 + col >= m) break;                                    // warp-uniform: no tokens left
      uint32_t v[32];
      lbdev::tmem_ld32(lane_base + kAcc + static_cast<uint32_t>(col), v);
      lbdev::tmem_ld_wait();
      if (valid) {
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int tok = t0 + col + jj;
          const float f = __uint_as_float(v[jj]) * sfac[col + jj];   // undo the prologue's 2^p
          if (tok < m)
            y[static_cast<int64_t>(tok) * n + wrow] =
                y_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(f)) : __half_as_ushort(__float2half_rn(f));
        }
      }
    }
  }
  if (!ok) atomicOr(err, lb::kErrGemmTimeout);
  lbdev::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
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
unsigned long long g_noalloc_ctx[64] = {};
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
    // set-up, once per device and context (with the device current): the host-side symbol is only
    // a stand-in, the kernels need the array's device address; a new context (after a device
    // reset) loads the module again, so the address is looked up again
    const unsigned long long ctx = context_id();
    std::lock_guard<std::mutex> lk(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return cuda_fail(e, "lb_gemm_noalloc: cudaGetSymbolAddress");
      g_noalloc_ptr[dev] = p;
      g_noalloc_ctx[dev] = ctx;
    }
    ptr = g_noalloc_ptr[dev];
  }
  return launch_gemm(W, x, xdt, m, y, ydt, ptr, st);
}

namespace {

// Tensor maps of a weight for this kernel (codes: 128-byte x 128-row boxes, 128-byte swizzle;
// scales: 8-group x 128-row boxes) depend only on its planes' addresses, shape and format; they are
// kept in a small direct-mapped host cache keyed by all of those.
struct GemmMaps {
  const uint8_t* codes;
  const uint16_t* scales;
  int64_t n, k;
  int fmt, valid;
  CUtensorMap tm_codes, tm_scales;
};
constexpr int kGemmMapCache = 256;
GemmMaps g_gemm_maps[kGemmMapCache];
std::mutex g_gemm_maps_mu;

lb_status gemm_maps(const lb_weight& W, int scales_tma, CUtensorMap& tm_codes, CUtensorMap& tm_scales) {
  const uintptr_t key = (reinterpret_cast<uintptr_t>(W.codes) >> 8) ^ (reinterpret_cast<uintptr_t>(W.codes) >> 20);
  std::lock_guard<std::mutex> lk(g_gemm_maps_mu);
  GemmMaps& e = g_gemm_maps[key % kGemmMapCache];
  if (!(e.valid && e.codes == W.codes && e.scales == W.scales && e.n == W.n && e.k == W.k && e.fmt == W.fmt)) {
    e.valid = 0;
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return fail(LB_ERR_CUDA, "lb_gemm: cuTensorMapEncodeTiled unavailable");
    const int G = static_cast<int>(W.k / kGroup);
    memset(&e.tm_codes, 0, sizeof(CUtensorMap));
    memset(&e.tm_scales, 0, sizeof(CUtensorMap));
    {
      const cuuint64_t row_bytes = static_cast<cuuint64_t>(W.k) / (W.fmt == LB_FMT_1BIT_G128 ? 8 : 4);
      const cuuint64_t dims[2] = {row_bytes, static_cast<cuuint64_t>(W.n)};
      const cuuint64_t strides[1] = {row_bytes};
      const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(WM)};
      const cuuint32_t estr[2] = {1, 1};
      CUresult r = enc(&e.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(W.codes), dims, strides,
                       box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(LB_ERR_CUDA, "lb_gemm: codes tensor map (CUresult %d)", static_cast<int>(r));
    }
    if (scales_tma) {
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(W.n)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(G) * 2};
      const cuuint32_t box[2] = {8, static_cast<cuuint32_t>(WM)};
      const cuuint32_t estr[2] = {1, 1};
      CUresult r = enc(&e.tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(W.scales), dims,
                       strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS)
        return fail(LB_ERR_CUDA, "lb_gemm: scales tensor map (CUresult %d)", static_cast<int>(r));
    }
    e.codes = W.codes;
    e.scales = W.scales;
    e.n = W.n;
    e.k = W.k;
    e.fmt = W.fmt;
    e.valid = 1;
  }
  tm_codes = e.tm_codes;
  tm_scales = e.tm_scales;
  return LB_OK;
}

}  // namespace

// Workspace: the binary16 activation tile images (mpad x k x 2 bytes), then one FP32 factor per
// padded token row.
size_t gemm_workspace_bytes(int64_t m, int64_t k) {
  const int64_t mpad = (m + BM - 1) / BM * BM;
  const size_t tiles = static_cast<size_t>(mpad) * (static_cast<size_t>(k) * 2 + 4);
  if (m > kGemmSmallM) return tiles;
  const size_t small = gemm_ms_workspace_bytes(m, k);              // the small-M path's staging
  return small > tiles ? small : tiles;
}

lb_status launch_gemm(const lb_weight& W, const void* x, int xdt, int64_t m, void* y, int ydt, void* ws,
                      cudaStream_t st) {
  const bool fault = take_test_fault(kTestFaultGemm);
  uint32_t* err = device_error_word();
  if (!err) return fail(LB_ERR_CUDA, "lb_gemm: device error word unavailable");
  const int k = static_cast<int>(W.k), n = static_cast<int>(W.n);
  const int64_t mpad = (m + BM - 1) / BM * BM;
  const bool one = W.fmt == LB_FMT_1BIT_G128;
  const int scales_tma = (k / kGroup) % 8 == 0 ? 1 : 0;            // scale row: a multiple of 16 bytes
  CUtensorMap tm_codes, tm_scales;
  lb_status ms = gemm_maps(W, scales_tma, tm_codes, tm_scales);
  if (ms != LB_OK) return ms;
  if (m <= kGemmSmallM)                                            // few tokens: the decode dominates
    return launch_gemm_ms(W, x, xdt, m, y, ydt, ws, tm_codes, tm_scales, scales_tma, fault, st);
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* fac = reinterpret_cast<float*>(wsb + static_cast<size_t>(mpad) * static_cast<size_t>(k) * 2);
  const unsigned rows = static_cast<unsigned>(mpad);                // one CTA per (padded) token row
  if (xdt == LB_BF16) {
    if (one) xprep_kernel<true, 1><<<rows, 256, 0, st>>>(xs, m, k, wsb, fac);
    else xprep_kernel<true, 2><<<rows, 256, 0, st>>>(xs, m, k, wsb, fac);
  } else {
    if (one) xprep_kernel<false, 1><<<rows, 256, 0, st>>>(xs, m, k, wsb, fac);
    else xprep_kernel<false, 2><<<rows, 256, 0, st>>>(xs, m, k, wsb, fac);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "lb_gemm: prologue launch");
  {
    // once per device: raise the dynamic shared-memory limit of the GEMM kernel
    static std::mutex mu;
    static bool done[2][64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "lb_gemm: cudaGetDevice");
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64 || !done[one][dev]) {
      e = cudaFuncSetAttribute(one ? gemm_lowbit_kernel<1> : gemm_lowbit_kernel<2>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
      if (e != cudaSuccess) return cuda_fail(e, "lb_gemm: set shared memory size");
      if (dev >= 0 && dev < 64) done[one][dev] = true;
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
  e = cudaLaunchKernelEx(&cfg, one ? gemm_lowbit_kernel<1> : gemm_lowbit_kernel<2>, tm_codes, tm_scales,
                         static_cast<const uint8_t*>(ws), static_cast<const float*>(fac), W.scales,
                         static_cast<uint16_t*>(y), static_cast<int>(m),
                         static_cast<int>(mpad), n, k, scales_tma, ydt == LB_BF16 ? 1 : 0, err,
                         fault ? kTestWaitNs : kWaitNs, fault ? 1 : 0);
  if (e != cudaSuccess) return cuda_fail(e, "lb_gemm: launch");
  return LB_OK;
}

}  // namespace lb
