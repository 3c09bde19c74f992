// Embedding-row gather from a packed 1-bit or ternary table.
//
//   out[i][k] = s[id_i][k / 128] * t[id_i][k],   rounded to binary16 or bfloat16 (RNE)
//
// (7minutos.es, "PrismML lanza Bonsai 27B", section "Cómo funciona la compresión", and
// es.news.hada.io topic 31450, section "Configuración multimodal y de bajo bit de extremo a
// extremo": the low-bit representation covers the embedding table too, so the step before the
// first GEMV dequantises one table row per token.)
//
// The work is a streaming write: 2 bytes out per weight against 1/8 (1-bit) or 1/4 (ternary) byte
// in, so the kernel is HBM-bound on its stores.  One warp produces a 1024-weight piece of one row
// (the last piece of a row may be shorter): in step q (0..3) lane l decodes the 8 weights
// 256q + 8l .. +7 from one code byte (1-bit) or two (ternary) and writes them as one 16-byte store,
// so every warp store is one contiguous 512-byte run and every code load a contiguous 32- or
// 64-byte run.
//
// Exactness: s * t is +-s or a signed zero, so the products are formed on the bit patterns: the
// scale is rounded once to the output format (binary16 -> bfloat16 RNE; binary16 -> binary16 is
// the identity), t = -1 flips the sign bit, t = 0 keeps only the sign bit (IEEE: s * 0 carries the
// sign of s).
#include "lb_common.cuh"

namespace {

// 16-bit pattern of the group scale in the output format.
template <bool BF>
__device__ __forceinline__ uint32_t scale_bits(uint16_t s) {
  if (!BF) return s;
  const float f = __half2float(__ushort_as_half(s));
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

constexpr int kPiece = 1024;                                   // weights per warp

template <int FMT, bool BF>
__global__ void __launch_bounds__(256) embed_kernel(const uint8_t* __restrict__ codes,
                                                    const uint16_t* __restrict__ scales,
                                                    const int32_t* __restrict__ ids, int64_t total_warps,
                                                    int n, int k, uint16_t* __restrict__ out,
                                                    uint32_t* __restrict__ err) {
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= total_warps) return;
  const int pieces = (k + kPiece - 1) / kPiece;                // pieces per row
  const int64_t i = wid / pieces;
  const int k0 = static_cast<int>(wid - i * pieces) * kPiece;  // first weight of this piece
  const int id = __ldg(ids + i);
  uint16_t* row_out = out + i * k;
  const bool bad = id < 0 || id >= n;
  if (bad && k0 == 0 && lane == 0) atomicOr(err, lb::kErrEmbedId);   // not a table row: +0 row, flagged
  const int G = k / lb::kGroup;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int kk = k0 + 256 * q + 8 * lane;                     // first of this lane's 8 weights
    if (kk >= k) break;                                         // k % 128 == 0: whole 8-weight runs
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (!bad) {
      const uint32_t s = scale_bits<BF>(__ldg(scales + static_cast<int64_t>(id) * G + kk / lb::kGroup));
      const uint32_t s2 = s * 0x00010001u;
      uint32_t o[4];
      if (FMT == LB_FMT_1BIT_G128) {
        // bit j of the byte is weight kk + j; bit 0 -> -s (sign bit set), bit 1 -> +s
        const uint32_t nb = ~static_cast<uint32_t>(__ldg(codes + static_cast<int64_t>(id) * (k / 8) + kk / 8));
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = s2 ^ ((((nb >> (2 * j)) & 1u) << 15) | (((nb >> (2 * j + 1)) & 1u) << 31));
      } else {
        // 2-bit field f = t + 1 per weight: f = 0 -> -s, 1 -> zero with the sign of s, 2 -> +s
        const uint32_t w = __ldg(reinterpret_cast<const uint16_t*>(codes + static_cast<int64_t>(id) * (k / 4) + kk / 4));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r = 0;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint32_t f = (w >> (2 * (2 * j + hf))) & 3u;
            const uint32_t h = f == 2u ? s : (f == 0u ? (s ^ 0x8000u) : (s & 0x8000u));
            r |= h << (16 * hf);
          }
          o[j] = r;
        }
      }
      v = make_uint4(o[0], o[1], o[2], o[3]);
    }
    *reinterpret_cast<uint4*>(row_out + kk) = v;
  }
}

template <int FMT, bool BF>
lb_status launch_t(const lb_weight& W, const int32_t* ids, int64_t count, uint16_t* out, cudaStream_t st) {
  uint32_t* err = lb::device_error_word();
  if (!err) return lb::fail(LB_ERR_CUDA, "lb_embed: device error word unavailable");
  const int k = static_cast<int>(W.k);
  const int64_t warps = count * ((k + kPiece - 1) / kPiece);
  const int64_t blocks = (warps + 7) / 8;
  embed_kernel<FMT, BF><<<static_cast<unsigned>(blocks), 256, 0, st>>>(W.codes, W.scales, ids, warps,
                                                                       static_cast<int>(W.n), k, out, err);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return lb::cuda_fail(e, "lb_embed: launch");
  return LB_OK;
}

}  // namespace

namespace lb {

lb_status launch_embed(const lb_weight& W, const int32_t* ids, int64_t count, void* out, int out_dtype,
                       cudaStream_t st) {
  uint16_t* o = static_cast<uint16_t*>(out);
  const bool bf = out_dtype == LB_BF16;
  if (W.fmt == LB_FMT_1BIT_G128)
    return bf ? launch_t<LB_FMT_1BIT_G128, true>(W, ids, count, o, st)
              : launch_t<LB_FMT_1BIT_G128, false>(W, ids, count, o, st);
  return bf ? launch_t<LB_FMT_TERNARY_G128, true>(W, ids, count, o, st)
            : launch_t<LB_FMT_TERNARY_G128, false>(W, ids, count, o, st);
}

}  // namespace lb
