// Packers: the 1-bit sign / max-abs quantiser and the ternary code packer.
//
// 1-bit: 7minutos.es, "Un tutorial de codificacion para ejecutar PrismML Bonsai 1-bit LLM en CUDA
// con GGUF", section "7 · Q1_0_g128 Cuantización" — per group of 128: scale = max |w|, bit = w >= 0.
// Ternary: 7minutos.es, "PrismML lanza Bonsai 27B", section "Cómo funciona la compresión" —
// codes t in {-1, 0, +1} with a given FP16 group scale; stored as 2-bit fields t + 1.
//
// Both kernels stream their input once (HBM bound: 4 bytes per weight for the fp32 weights,
// 1 byte per weight for the int8 codes) and report validation problems through a device word
// that the synchronous host wrapper reads back.
#include <mutex>

#include "lb_common.cuh"

namespace {

__device__ uint32_t g_pack_flags;

// One warp per 128-weight group.  Lane i reads w[32j + i] for j = 0..3 (four fully coalesced
// 128-byte loads), so the ballot of j is exactly code word j of the group (bit i <-> weight 32j+i,
// LSB-first).  The group maximum of |w| is a warp max over the IEEE bit patterns of |w| (monotonic
// for non-negative floats; NaN patterns sort above +Inf and are reported).
__global__ void __launch_bounds__(256) pack1_kernel(const float* __restrict__ w, int64_t total_groups,
                                                    int64_t groups_per_row, int64_t k,
                                                    uint8_t* __restrict__ codes, uint16_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  uint32_t flags = 0;
  for (int64_t gi = warp; gi < total_groups; gi += nwarps) {
    const int64_t row = gi / groups_per_row;
    const int64_t g = gi - row * groups_per_row;
    const float* src = w + row * k + g * lb::kGroup;
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __ldcs(src + 32 * j + lane);
    uint32_t amax = 0;
    uint32_t word[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      word[j] = __ballot_sync(0xffffffffu, v[j] >= 0.0f);
      amax = max(amax, __float_as_uint(v[j]) & 0x7fffffffu);
    }
    amax = __reduce_max_sync(0xffffffffu, amax);
    if (amax >= 0x7f800000u) flags |= lb::kPackNonFinite;           // Inf or NaN in the group
    const __half s = __float2half_rn(__uint_as_float(amax));
    if (__hisinf(s)) flags |= lb::kPackRange;
    uint32_t* dst = reinterpret_cast<uint32_t*>(codes + row * (k / 8) + g * 16);
    if (lane < 4) {
      uint32_t wv = word[0];
      if (lane == 1) wv = word[1];
      if (lane == 2) wv = word[2];
      if (lane == 3) wv = word[3];
      dst[lane] = wv;
    }
    if (lane == 0) scales[gi] = __half_as_ushort(s);
  }
  if (flags) atomicOr(&g_pack_flags, flags);
}

// Each thread packs 16 consecutive codes (one 16-byte load) into 4 bytes (one 32-bit store).
// Per byte lane: f = t + 1 computed with a carry-free SIMD add; valid codes give f <= 2.
__device__ __forceinline__ uint32_t pack4_fields(uint32_t u, uint32_t& bad) {
  const uint32_t f = __vadd4(u, 0x01010101u);
  bad |= ~__vcmpleu4(f, 0x02020202u);
  return (f & 3u) | ((f >> 6) & 0xCu) | ((f >> 12) & 0x30u) | ((f >> 18) & 0xC0u);
}

__global__ void __launch_bounds__(256) pack_ternary_kernel(const int8_t* __restrict__ t, int64_t chunks,
                                                           uint8_t* __restrict__ codes) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  uint32_t bad = 0;
  for (int64_t c = tid; c < chunks; c += nthreads) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(t) + c);
    const uint32_t out = pack4_fields(v.x, bad) | (pack4_fields(v.y, bad) << 8) |
                         (pack4_fields(v.z, bad) << 16) | (pack4_fields(v.w, bad) << 24);
    reinterpret_cast<uint32_t*>(codes)[c] = out;
  }
  if (bad) atomicOr(&g_pack_flags, lb::kPackCode);
}

lb_status reset_flags(cudaStream_t st) {
  const uint32_t zero = 0;
  cudaError_t e = cudaMemcpyToSymbolAsync(g_pack_flags, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return lb::cuda_fail(e, "pack: reset flags");
  return LB_OK;
}

lb_status read_flags(cudaStream_t st, uint32_t* out) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_pack_flags, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return lb::cuda_fail(e, "pack: read flags");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return lb::cuda_fail(e, "pack: synchronize");
  return LB_OK;
}

int grid_for(int64_t work_items, int items_per_block) {
  const int64_t want = (work_items + items_per_block - 1) / items_per_block;
  const int64_t cap = static_cast<int64_t>(lb::sm_count()) * 16;
  return static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace

namespace lb {

lb_status launch_pack_1bit(const float* w, int64_t n, int64_t k, uint8_t* codes, uint16_t* scales,
                           cudaStream_t st, uint32_t* flags_out) {
  lb_status s = reset_flags(st);
  if (s != LB_OK) return s;
  const int64_t gpr = k / kGroup;
  const int64_t total = n * gpr;
  pack1_kernel<<<grid_for(total, 8), 256, 0, st>>>(w, total, gpr, k, codes, scales);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "lb_pack_1bit: launch");
  return read_flags(st, flags_out);
}

lb_status launch_pack_ternary(const int8_t* t, const uint16_t* s_in, int64_t n, int64_t k, uint8_t* codes,
                              uint16_t* scales, cudaStream_t st, uint32_t* flags_out) {
  lb_status s = reset_flags(st);
  if (s != LB_OK) return s;
  const int64_t chunks = n * k / 16;
  pack_ternary_kernel<<<grid_for(chunks, 256), 256, 0, st>>>(t, chunks, codes);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "lb_pack_ternary: launch");
  if (scales != s_in) {
    e = cudaMemcpyAsync(scales, s_in, static_cast<size_t>(n) * (k / kGroup) * 2, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "lb_pack_ternary: copy scales");
  }
  return read_flags(st, flags_out);
}

}  // namespace lb
