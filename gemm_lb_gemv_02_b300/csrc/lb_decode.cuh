// Register decode of packed 1-bit / ternary code words into binary16 mma.sync A fragments, the
// m16n8k16 MMA forms the decoders feed, and the shared-memory load forms they use.  Shared by the
// decode GEMV and the mid-size GEMM built on the same engine.
//
// (7minutos.es, "PrismML lanza Bonsai 27B", section "Cómo funciona la compresión": w = s_g t_i with
// t in {-1, +1} (1-bit) or {-1, 0, +1} (ternary); the decode below produces t, the scale s_g is
// applied per group in FP32 by the caller.)
#pragma once

#include <cstdint>

namespace lbdec {

// ----------------------------------------------------------------------------- decode
__host__ __device__ constexpr uint32_t expo16(int m) {   // 2^(10-m) in both halves
  return (static_cast<uint32_t>(25 - m) << 10) * 0x00010001u;
}
// 1-bit: register j of a 32-bit code word holds bits j (low half) and j+16 (high half) = weights
// k = j and k = j + 16 of the word, at mantissa position m_j in 4..9: j = 0..5 from w << 4, j = 6..11
// from w >> 2, j = 12..15 from w >> 8.  The offsets o = 2^(10-m) stay <= 64, so the baseline the
// MMA cancels is at most 64.5 times the activations it multiplies (m >= 1 keeps o + 1/2 exact).
__host__ __device__ constexpr int pos1(int j) { return j <= 5 ? j + 4 : (j <= 11 ? j - 2 : j - 8); }
// Ternary: register p of a 32-bit word (16 fields) holds field p (low) and p + 8 (high) = weights
// k = p and k = p + 8 of the word; the field sits at mantissa bits (m, m+1), m in {0,2,4,6,8}.
__host__ __device__ constexpr int pos2(int p) { return p <= 4 ? 2 * p : 2 * p - 6; }

template <int FMT>
__device__ __forceinline__ constexpr float reg_offset(int i) {
  return static_cast<float>(1 << (10 - (FMT == 1 ? pos1(i) : pos2(i & 7))));
}

template <uint32_t E>
__device__ __forceinline__ uint32_t lop_and_or(uint32_t src, uint32_t mask) {   // (src & mask) | E
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(src), "r"(mask), "n"(E));
  return r;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Decoder state for one 32-bit code word: its shifted copies.
struct Word1 {
  uint32_t w4, w2, w8;
};
__device__ __forceinline__ Word1 prep1(uint32_t w) { return Word1{w << 4, w >> 2, w >> 8}; }
template <int J>
__device__ __forceinline__ uint32_t dec1(const Word1& x, const uint32_t (&M)[10]) {
  constexpr int m = pos1(J);
  const uint32_t src = J <= 5 ? x.w4 : (J <= 11 ? x.w2 : x.w8);
  return lop_and_or<expo16(m)>(src, M[m]);
}
struct Word2 {
  uint32_t w, w6;
};
__device__ __forceinline__ Word2 prep2(uint32_t w) { return Word2{w, w >> 6}; }
template <int P>
__device__ __forceinline__ uint32_t dec2(const Word2& x, const uint32_t (&M)[10]) {
  constexpr int m = pos2(P);
  return lop_and_or<expo16(m)>(P <= 4 ? x.w : x.w6, M[m]);
}

// A-fragment register I (0..15) of the lane's 32-k block of one row.
//   1-bit: o + b; the MMA's C operand removes sum (o + 1/2) x, leaving sum t x / 2 (t = 2b - 1).
//   ternary: (o + f) - (o + 1) = t exactly (SC[m] holds o + 1 in both halves), with no baseline:
//   a zero code contributes exactly nothing, however large the activation it meets.
template <int FMT, int I>
__device__ __forceinline__ uint32_t areg(const Word1& a1, const Word2& a2lo, const Word2& a2hi,
                                         const uint32_t (&M)[10], const uint32_t (&SC)[10]) {
  if constexpr (FMT == 1) return dec1<I>(a1, M);
  else return hsub2(dec2<(I & 7)>(I < 8 ? a2lo : a2hi, M), SC[pos2(I & 7)]);
}

// D = A * B + C with C = {-C_g[2q], -C_g[2q+1], -C_g[2q], -C_g[2q+1]} (the baseline of my columns).
__device__ __forceinline__ void mma_c4(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                       uint32_t b0, uint32_t b1, const float4& c) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y), "f"(c.z), "f"(c.w));
}
// D = A * B (the accumulator starts from zero).
__device__ __forceinline__ void mma_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Shared-memory loads with 32-bit shared addresses.  Loads from a pipeline slot are volatile, so
// they stay between the barrier wait that makes the slot valid and the arrive that hands it back.
// Loads from the CTA-private x / baseline region are plain asm whose addresses carry a token made
// after the barrier that published the region, so they cannot be hoisted above it but otherwise
// schedule freely.
__device__ __forceinline__ uint32_t ldsv32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 ldsv64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 ldsv128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}

}  // namespace lbdec
