// Decode GEMV / small-batch GEMV against packed 1-bit or ternary weights (batch 1..8).
//
//   y[b][n] = sum_g s[n][g] * sum_{i<128} t[n][128g+i] * x[b][128g+i]
//
// (7minutos.es, "PrismML lanza Bonsai 27B", sections "Cómo funciona la compresión" for w = s_g t_i
// and "Rendimiento y decodificación especulativa DSpark" for the bandwidth-bound decode and the
// width-5 speculative verification.)
//
// Design.  A 1-bit GEMV must retire ~37 T weights/s to stream at 80% of B300 HBM bandwidth, about
// one lane-operation per weight over the whole GPU; integer LOP3 issues at half rate on sm_103a,
// so the per-weight multiply cannot stay on the CUDA cores.  The packed codes are therefore
// decoded straight into FP16/BF16 tensor-core A fragments with one LOP3 per two weights and the
// dot products run on mma.sync m16n8k16 (batch <= 8 fills its n = 8 columns):
//
//   * "offset exponent" decode: a half whose exponent encodes 2^(10-m) (fp16; 2^(7-m) for bf16)
//     and whose mantissa bit m (ternary: bits m, m+1) is copied from the code word has the exact
//     value o + b (o = 2^(10-m)), b the code bit (or 2-bit field).  One LOP3 builds two of them.
//   * the tensor core returns D_g = sum (o_k + b_k) x_k for one 128-group; the per-column constant
//     C_g = sum (o_k + c) x_k (c = 1/2 for 1-bit, 1 for ternary) comes from the same MMA with A
//     set to the constants, so sum t x = 2 (D_g - C_g) for 1-bit (t = 2b - 1) and D_g - C_g for
//     ternary (t = f - 1).  All A values are exact, products are exact in FP32, and the group scale
//     is applied once per group in FP32: y += s * (D_g - C_g).
//   * the MMA reduction order along K is free, so code bit j of a word lands in whichever k slot
//     its register occupies and x is gathered into B fragments in the matching order.
#include "lb_common.cuh"

namespace {

// ----------------------------------------------------------------------------- decode constants
// fp16 half with exponent for 2^(10-m), replicated in both halves; bf16: 2^(7-m).
template <bool BF>
__device__ __forceinline__ constexpr uint32_t expo(int m) {
  return BF ? (static_cast<uint32_t>(134 - m) << 7) * 0x00010001u
            : (static_cast<uint32_t>(25 - m) << 10) * 0x00010001u;
}

// 1-bit: register j (0..15) of a 32-bit code word holds bits j (low half) and j+16 (high half),
// i.e. weights k = j and k = j + 16 of the word's 32.  Mantissa positions m >= 1 keep o + 1/2
// exact (fp16: m in 1..9, bf16: m in 1..6).
template <bool BF>
__device__ __forceinline__ void decode_1bit(uint32_t w, uint32_t (&a)[16]) {
  const uint32_t w1 = w << 1;
  if (!BF) {
    const uint32_t w6 = w >> 6;
    a[0] = (w1 & (0x00010001u << 1)) | expo<false>(1);
#pragma unroll
    for (int j = 1; j <= 9; ++j) a[j] = (w & (0x00010001u << j)) | expo<false>(j);
#pragma unroll
    for (int j = 10; j <= 15; ++j) a[j] = (w6 & (0x00010001u << (j - 6))) | expo<false>(j - 6);
  } else {
    const uint32_t w6 = w >> 6, w12 = w >> 12;
    a[0] = (w1 & (0x00010001u << 1)) | expo<true>(1);
#pragma unroll
    for (int j = 1; j <= 6; ++j) a[j] = (w & (0x00010001u << j)) | expo<true>(j);
#pragma unroll
    for (int j = 7; j <= 12; ++j) a[j] = (w6 & (0x00010001u << (j - 6))) | expo<true>(j - 6);
#pragma unroll
    for (int j = 13; j <= 15; ++j) a[j] = (w12 & (0x00010001u << (j - 12))) | expo<true>(j - 12);
  }
}

template <bool BF>
__device__ __forceinline__ int pos_1bit(int j) {
  return BF ? (j == 0 ? 1 : j <= 6 ? j : j <= 12 ? j - 6 : j - 12) : (j == 0 ? 1 : j <= 9 ? j : j - 6);
}

// Constant A register for the 1-bit baseline: value o + 1/2 (mantissa bit m-1 set).
template <bool BF>
__device__ __forceinline__ uint32_t const_1bit(int j) {
  const int m = pos_1bit<BF>(j);
  return expo<BF>(m) | (0x00010001u << (m - 1));
}

// Ternary: register p (0..7) of a 32-bit code word (16 fields) holds field p (low half) and field
// p + 8 (high half), i.e. weights k = p and k = p + 8 of the word's 16.  Field at mantissa bits
// (m, m+1): fp16 m in {0,2,4,6,8}; bf16 m in {0,2,4}.
template <bool BF>
__device__ __forceinline__ int pos_tern(int p) {
  return BF ? (p <= 2 ? 2 * p : p <= 5 ? 2 * p - 6 : 2 * p - 12) : (p <= 4 ? 2 * p : 2 * p - 6);
}

template <bool BF>
__device__ __forceinline__ void decode_tern(uint32_t w, uint32_t* a) {
  const uint32_t w6 = w >> 6;
  if (!BF) {
#pragma unroll
    for (int p = 0; p <= 4; ++p) a[p] = (w & (0x00030003u << (2 * p))) | expo<false>(2 * p);
#pragma unroll
    for (int p = 5; p <= 7; ++p) a[p] = (w6 & (0x00030003u << (2 * p - 6))) | expo<false>(2 * p - 6);
  } else {
    const uint32_t w12 = w >> 12;
#pragma unroll
    for (int p = 0; p <= 2; ++p) a[p] = (w & (0x00030003u << (2 * p))) | expo<true>(2 * p);
#pragma unroll
    for (int p = 3; p <= 5; ++p) a[p] = (w6 & (0x00030003u << (2 * p - 6))) | expo<true>(2 * p - 6);
#pragma unroll
    for (int p = 6; p <= 7; ++p) a[p] = (w12 & (0x00030003u << (2 * p - 12))) | expo<true>(2 * p - 12);
  }
}

// Constant A register for the ternary baseline: value o + 1 (mantissa bit m set).
template <bool BF>
__device__ __forceinline__ uint32_t const_tern(int p) {
  const int m = pos_tern<BF>(p);
  return expo<BF>(m) | (0x00010001u << m);
}

template <bool BF>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if (BF) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }

template <bool BF>
__device__ __forceinline__ float to_f32(uint16_t h) {
  return BF ? __uint_as_float(static_cast<uint32_t>(h) << 16) : __half2float(__ushort_as_half(h));
}

template <bool BF>
__device__ __forceinline__ uint16_t from_f32(float v) {
  return BF ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
}

// ----------------------------------------------------------------------------- the kernel
// CTA = 4 warps over the same 16*T rows; warp w takes groups w, w+4, ...  Lane = (r, q) with
// r = lane / 4 (rows r and r + 8 of each 16-row tile, and batch column r for the B fragment) and
// q = lane % 4 (the quarter of the group this lane's code words cover).
template <int FMT, bool BF, int T>
__global__ void __launch_bounds__(128) gemv_mma_kernel(const uint8_t* __restrict__ codes,
                                                       const uint16_t* __restrict__ scales,
                                                       const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
                                                       int n_rows, int k, int batch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, q = lane & 3;
  const int G = k / lb::kGroup;
  const int row0 = blockIdx.x * (16 * T);
  const int64_t crow = FMT == 1 ? k / 8 : k / 4;   // code bytes per row

  float acc[T][4];
#pragma unroll
  for (int t = 0; t < T; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  uint32_t cst[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) cst[j] = FMT == 1 ? const_1bit<BF>(j) : const_tern<BF>(j & 7);

  for (int g = warp; g < G; g += 4) {
    // ---- B fragments: x[r][128g + 32q + perm], gathered to match the decode order
    uint32_t bx[16];
    if (r < batch) {
      const uint4* xp = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(r) * k + g * lb::kGroup + 32 * q);
      uint32_t X[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(xp + i);
        X[4 * i] = v.x; X[4 * i + 1] = v.y; X[4 * i + 2] = v.z; X[4 * i + 3] = v.w;
      }
      if (FMT == 1) {
#pragma unroll
        for (int j = 0; j < 16; ++j) bx[j] = prmt(X[j >> 1], X[(j >> 1) + 8], (j & 1) ? 0x7632 : 0x5410);
      } else {
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          const int uu = rr >> 3, p = rr & 7;
          bx[rr] = prmt(X[8 * uu + (p >> 1)], X[8 * uu + (p >> 1) + 4], (p & 1) ? 0x7632 : 0x5410);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) bx[j] = 0u;
    }
    // ---- per-column baseline C_g (identical for every row)
    float cc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) mma16816<BF>(cc, cst[2 * i], cst[2 * i], cst[2 * i + 1], cst[2 * i + 1], bx[2 * i], bx[2 * i + 1]);

#pragma unroll
    for (int t = 0; t < T; ++t) {
      const int ra = row0 + 16 * t + r, rb = ra + 8;
      uint32_t A[16], B8[16];
      float sa = 0.f, sb = 0.f;
      if (FMT == 1) {
        uint32_t wa = 0, wb = 0;
        if (ra < n_rows) {
          wa = __ldg(reinterpret_cast<const uint32_t*>(codes + ra * crow + 16 * g) + q);
          sa = __half2float(__ushort_as_half(__ldg(scales + static_cast<int64_t>(ra) * G + g)));
        }
        if (rb < n_rows) {
          wb = __ldg(reinterpret_cast<const uint32_t*>(codes + rb * crow + 16 * g) + q);
          sb = __half2float(__ushort_as_half(__ldg(scales + static_cast<int64_t>(rb) * G + g)));
        }
        decode_1bit<BF>(wa, A);
        decode_1bit<BF>(wb, B8);
      } else {
        uint2 wa = make_uint2(0u, 0u), wb = make_uint2(0u, 0u);
        if (ra < n_rows) {
          wa = __ldg(reinterpret_cast<const uint2*>(codes + ra * crow + 32 * g) + q);
          sa = __half2float(__ushort_as_half(__ldg(scales + static_cast<int64_t>(ra) * G + g)));
        }
        if (rb < n_rows) {
          wb = __ldg(reinterpret_cast<const uint2*>(codes + rb * crow + 32 * g) + q);
          sb = __half2float(__ushort_as_half(__ldg(scales + static_cast<int64_t>(rb) * G + g)));
        }
        decode_tern<BF>(wa.x, A);
        decode_tern<BF>(wa.y, A + 8);
        decode_tern<BF>(wb.x, B8);
        decode_tern<BF>(wb.y, B8 + 8);
      }
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 8; ++i) mma16816<BF>(d, A[2 * i], B8[2 * i], A[2 * i + 1], B8[2 * i + 1], bx[2 * i], bx[2 * i + 1]);
      acc[t][0] = fmaf(sa, d[0] - cc[0], acc[t][0]);
      acc[t][1] = fmaf(sa, d[1] - cc[1], acc[t][1]);
      acc[t][2] = fmaf(sb, d[2] - cc[2], acc[t][2]);
      acc[t][3] = fmaf(sb, d[3] - cc[3], acc[t][3]);
    }
  }

  // ---- reduce the four warps' K slices and store y (column c = 2q + {0,1}, rows ra / rb)
  __shared__ float red[4][T][4][32];
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) red[warp][t][e][lane] = acc[t][e];
  __syncthreads();
  const float mul = FMT == 1 ? 2.f : 1.f;
  for (int idx = threadIdx.x; idx < T * 4 * 32; idx += blockDim.x) {
    const int t = idx / 128, e = (idx / 32) & 3, l = idx & 31;
    const float v = (red[0][t][e][l] + red[1][t][e][l] + red[2][t][e][l] + red[3][t][e][l]) * mul;
    const int rr = l >> 2, qq = l & 3;
    const int row = row0 + 16 * t + rr + ((e & 2) ? 8 : 0);
    const int col = 2 * qq + (e & 1);
    if (row < n_rows && col < batch) y[static_cast<int64_t>(col) * n_rows + row] = from_f32<BF>(v);
  }
}

template <int FMT, bool BF>
lb_status launch_t(const lb_weight& W, const uint16_t* x, int batch, uint16_t* y, cudaStream_t st) {
  const int n = static_cast<int>(W.n), k = static_cast<int>(W.k);
  const int sms = lb::sm_count();
  int T = 1;
  if ((n + 63) / 64 >= 2 * sms) T = 4;
  else if ((n + 31) / 32 >= 2 * sms) T = 2;
  const int rows = 16 * T;
  const dim3 grid((n + rows - 1) / rows);
  if (T == 4) gemv_mma_kernel<FMT, BF, 4><<<grid, 128, 0, st>>>(W.codes, W.scales, x, y, n, k, batch);
  else if (T == 2) gemv_mma_kernel<FMT, BF, 2><<<grid, 128, 0, st>>>(W.codes, W.scales, x, y, n, k, batch);
  else gemv_mma_kernel<FMT, BF, 1><<<grid, 128, 0, st>>>(W.codes, W.scales, x, y, n, k, batch);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return lb::cuda_fail(e, "lb_gemv: launch");
  return LB_OK;
}

}  // namespace

namespace lb {

lb_status launch_gemv(const lb_weight& W, const void* x, int xdt, int batch, void* y, cudaStream_t st) {
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint16_t* ys = static_cast<uint16_t*>(y);
  const bool bf = xdt == LB_BF16;
  if (W.fmt == LB_FMT_1BIT_G128)
    return bf ? launch_t<1, true>(W, xs, batch, ys, st) : launch_t<1, false>(W, xs, batch, ys, st);
  return bf ? launch_t<2, true>(W, xs, batch, ys, st) : launch_t<2, false>(W, xs, batch, ys, st);
}

}  // namespace lb
