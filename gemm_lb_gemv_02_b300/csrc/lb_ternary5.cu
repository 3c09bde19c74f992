// Ternary codes stored five to a byte: packer and decode GEMV.
//
// Format (es.news.hada.io topic 31450, comments: five three-state values fit one byte, 1.6 bits
// each; kerneldigest.dev, "Compresión ternaria de modelos LLM: Bonsai 2 27B", section
// "Arquitectura del Sistema": 1.76 effective bits per weight): digit f = t + 1 in {0, 1, 2}; within
// each 128-weight group byte j holds weights 5j .. 5j+4 as sum_i f_(5j+i) 3^i, byte 25 holds weights
// 125..127; 26 bytes of codes per group, row-major [N][26 K/128], plus the binary16 scales
// [N][K/128].  1.625 + 0.125 = 1.75 bits per weight against 2.125 for the 2-bit fields.
//
// GEMV  y[b][n] = sum_g s[n][g] * sum_i t[n][128g+i] * x[b][128g+i]  (FP32 accumulation), for
// batches 2..8, and at batch 1 when K is not a multiple of 1024 or too long for the tables
// (otherwise batch 1 runs the GEMV kernel's lookup-table form): a CUDA-core kernel.  A 243-entry shared-memory table turns a code byte into its five digits, one
// per byte of a 64-bit entry; one byte permute then drops digit f into the low byte of the float
// 1.5 * 2^23 (whose low mantissa bits are zero), so that float minus (1.5 * 2^23 + 1) is t = f - 1
// exactly: a digit costs a PRMT and an FADD before its FFMA.  Lane l of a warp
// owns byte l of every group (weights 5l .. 5l+4; lanes 26..31 idle), so the warp reads a group's
// 26 code bytes as one 32-byte sector and the activations at a lane stride of five words, which
// touches 32 distinct banks.  A CTA owns 32 rows (8 warps x 4 rows); x is staged in shared memory
// as FP32 [batch][KC] in chunks of KC = 48 KB / (4 batch) activations (all of K at batch 1 for
// K <= 12288), and every warp runs its rows over each chunk.  The code bytes and scales of a
// group are loaded two groups ahead of the arithmetic.
#include <mutex>

#include "lb_common.cuh"

namespace {

constexpr int kT5Bytes = 26;          // code bytes per 128-weight group
constexpr int kXBytes = 48 * 1024;    // activation chunk in shared memory (FP32 [batch][KC])
constexpr int kRowsPerWarp = 4;
constexpr int kWarps = 8;
constexpr int kRowsPerCta = kRowsPerWarp * kWarps;

__device__ uint32_t g_t5_flags;       // validation bits of the packer

// ------------------------------------------------------------------------------------ packer
// One thread per code byte: (row, group, byte j) -> sum_i (t + 1) 3^i over the byte's weights.
__global__ void __launch_bounds__(256) pack_t5_kernel(const int8_t* __restrict__ t, int64_t n, int G,
                                                      uint8_t* __restrict__ codes) {
  const int64_t total = n * G * kT5Bytes;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int k = G * lb::kGroup;
  uint32_t bad = 0;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t row = idx / (static_cast<int64_t>(G) * kT5Bytes);
    const int rem = static_cast<int>(idx - row * G * kT5Bytes);
    const int g = rem / kT5Bytes, j = rem - g * kT5Bytes;
    const int8_t* src = t + row * k + g * lb::kGroup + 5 * j;
    const int nd = j == kT5Bytes - 1 ? 3 : 5;
    uint32_t v = 0, p = 1;
    for (int i = 0; i < nd; ++i) {
      const int f = static_cast<int>(src[i]) + 1;
      bad |= static_cast<uint32_t>(f < 0 || f > 2);
      v += static_cast<uint32_t>(f < 0 ? 0 : (f > 2 ? 2 : f)) * p;
      p *= 3;
    }
    codes[idx] = static_cast<uint8_t>(v);
  }
  if (bad) atomicOr(&g_t5_flags, lb::kPackCode);
}

// ------------------------------------------------------------------------------------ GEMV
template <bool XBF>
__device__ __forceinline__ float act(uint16_t v) {
  return XBF ? __uint_as_float(static_cast<uint32_t>(v) << 16) : __half2float(__ushort_as_half(v));
}

template <int BP>
__host__ __device__ constexpr int kc_of() { return kXBytes / (4 * BP) / lb::kGroup * lb::kGroup; }

template <bool XBF, int BP>
__global__ void __launch_bounds__(kWarps * 32) gemv_t5_kernel(const uint8_t* __restrict__ codes,
                                                               const uint16_t* __restrict__ scales,
                                                               const uint16_t* __restrict__ x,
                                                               uint16_t* __restrict__ y, int n, int k, int batch) {
  __shared__ uint2 lut[256];                                   // byte -> five digits, one per byte
  extern __shared__ float xs[];                                // [BP][KC]
  constexpr int kKC = kc_of<BP>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = k / lb::kGroup;
  const int row0 = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp;
  for (int v = threadIdx.x; v < 256; v += blockDim.x) {
    uint32_t d[5], r = static_cast<uint32_t>(v);
    for (int i = 0; i < 5; ++i) { d[i] = r % 3u; r /= 3u; }
    lut[v] = make_uint2(d[0] | (d[1] << 8) | (d[2] << 16) | (d[3] << 24), d[4]);
  }
  // lane l: byte l of each group; its digits i < nd are weights 5l + i
  const int nd = lane < 25 ? 5 : (lane == 25 ? 3 : 0);
  // this warp's rows (rows past n read row n - 1 and are not stored): code and scale row starts
  const uint8_t* crow[kRowsPerWarp];
  const uint16_t* srow[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int64_t row = min(row0 + r, n - 1);
    crow[r] = codes + row * G * kT5Bytes + lane;
    srow[r] = scales + row * G;
  }
  float acc[kRowsPerWarp][BP];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int b = 0; b < BP; ++b) acc[r][b] = 0.f;
  // bfloat16 x reaches 3.4e38, where FP32 partial sums overflow although the product is finite:
  // a column whose largest magnitude is 2^100 or more is scaled down by an exact power of two
  // (largest magnitude below 2^100) and its results scaled back.  One pass over x finds the
  // columns' largest exponents.
  __shared__ uint32_t cmax[8];
  float xsc[BP], ysc[BP];
#pragma unroll
  for (int b = 0; b < BP; ++b) xsc[b] = ysc[b] = 1.f;
  if (XBF) {
    if (threadIdx.x < 8) cmax[threadIdx.x] = 0u;
    __syncthreads();
    uint32_t mx[BP];
#pragma unroll
    for (int b = 0; b < BP; ++b) mx[b] = 0u;
    for (int w8 = threadIdx.x; w8 < k / 8; w8 += blockDim.x)
#pragma unroll
      for (int b = 0; b < BP; ++b)
        if (b < batch) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(b) * k) + w8);
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) mx[b] = max(mx[b], max((u[i] << 16) & 0x7f800000u, u[i] & 0x7f800000u));
        }
#pragma unroll
    for (int b = 0; b < BP; ++b) {
      for (int o = 16; o > 0; o >>= 1) mx[b] = max(mx[b], __shfl_xor_sync(0xffffffffu, mx[b], o));
      if (lane == 0 && b < batch) atomicMax(&cmax[b], mx[b]);
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < BP; ++b) {
      const int e = static_cast<int>(cmax[b] >> 23) - 127;
      if (e >= 100) {
        xsc[b] = __uint_as_float(static_cast<uint32_t>(127 + 99 - e) << 23);
        ysc[b] = __uint_as_float(static_cast<uint32_t>(127 - 99 + e) << 23);
      }
    }
  }

  for (int c0 = 0; c0 < k; c0 += kKC) {
    const int kc = min(kKC, k - c0);
    __syncthreads();                                           // the previous chunk is consumed
    for (int e = threadIdx.x; e < BP * (kc / 8); e += blockDim.x) {
      const int b = e / (kc / 8), w8 = e - b * (kc / 8);
      float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
      if (b < batch) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(b) * k + c0) + w8);
        float f = 1.f;                                         // the column's power-of-two scale
#pragma unroll
        for (int bb = 0; bb < BP; ++bb)
          if (bb == b) f = xsc[bb];
        lo = make_float4(act<XBF>(v.x & 0xffffu) * f, act<XBF>(v.x >> 16) * f, act<XBF>(v.y & 0xffffu) * f,
                         act<XBF>(v.y >> 16) * f);
        hi = make_float4(act<XBF>(v.z & 0xffffu) * f, act<XBF>(v.z >> 16) * f, act<XBF>(v.w & 0xffffu) * f,
                         act<XBF>(v.w >> 16) * f);
      }
      float4* d = reinterpret_cast<float4*>(xs + b * kKC + 8 * w8);
      d[0] = lo;
      d[1] = hi;
    }
    __syncthreads();
    if (nd == 0) continue;                                     // lanes 26..31 hold no byte
    const int g0 = c0 / lb::kGroup;
    const int ng = kc / lb::kGroup;
    // the rows' code bytes and scales of a group, loaded together (rows past n read row n - 1 and
    // are not stored), two groups ahead of the arithmetic through two named buffers
    uint32_t ca[kRowsPerWarp], sa[kRowsPerWarp], cbf[kRowsPerWarp], sbf[kRowsPerWarp];
    auto load = [&](int gl, uint32_t (&c)[kRowsPerWarp], uint32_t (&sv)[kRowsPerWarp]) {
      if (gl >= ng) return;
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        c[r] = __ldg(crow[r] + (g0 + gl) * kT5Bytes);
        sv[r] = __ldg(srow[r] + g0 + gl);
      }
    };
    auto group = [&](int gl, const uint32_t (&c)[kRowsPerWarp], const uint32_t (&sv)[kRowsPerWarp]) {
      if (gl >= ng) return;
      const float* xg = xs + gl * lb::kGroup + 5 * lane;
      float xv[BP][5];
#pragma unroll
      for (int b = 0; b < BP; ++b)
#pragma unroll
        for (int i = 0; i < 5; ++i) xv[b][i] = i < nd ? xg[b * kKC + i] : 0.f;
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const uint2 f = lut[c[r]];
        const float s = __half2float(__ushort_as_half(static_cast<uint16_t>(sv[r])));
        float p[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b) p[b] = 0.f;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
          // bytes {digit i, 0x00, 0x40, 0x4B} = 12582912 + f as a float
          const uint32_t bits = __byte_perm(i < 4 ? f.x : f.y, 0x4B400000u, i < 4 ? (0x7650u | i) : 0x7650u);
          const float tv = __uint_as_float(bits) - 12582913.0f;
#pragma unroll
          for (int b = 0; b < BP; ++b) p[b] = fmaf(tv, xv[b][i], p[b]);
        }
#pragma unroll
        for (int b = 0; b < BP; ++b) acc[r][b] = fmaf(s, p[b], acc[r][b]);
      }
    };
    load(0, ca, sa);
    load(1, cbf, sbf);
    for (int gl = 0; gl < ng; gl += 2) {
      group(gl, ca, sa);
      load(gl + 2, ca, sa);
      group(gl + 1, cbf, sbf);
      load(gl + 3, cbf, sbf);
    }
  }
  // lanes -> row sums; lane 0 stores
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int row = row0 + r;
#pragma unroll
    for (int b = 0; b < BP; ++b) {
      float v = acc[r][b];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      v *= ysc[b];
      if (lane == 0 && row < n && b < batch)
        y[static_cast<int64_t>(b) * n + row] =
            XBF ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
    }
  }
}

template <bool XBF, int BP>
lb_status launch_bp(const lb_weight& W, const uint16_t* x, int batch, uint16_t* y, cudaStream_t st) {
  const int n = static_cast<int>(W.n), k = static_cast<int>(W.k);
  const size_t smem = static_cast<size_t>(BP) * kc_of<BP>() * sizeof(float);
  if (smem + 4096 > 48 * 1024) {                                // with the static table: raise the limit once per device
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return lb::cuda_fail(e, "lb_gemv (5-per-byte ternary): cudaGetDevice");
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64 || !done[dev]) {
      e = cudaFuncSetAttribute(gemv_t5_kernel<XBF, BP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return lb::cuda_fail(e, "lb_gemv (5-per-byte ternary): shared memory attribute");
      if (dev >= 0 && dev < 64) done[dev] = true;
    }
  }
  const unsigned blocks = static_cast<unsigned>((n + kRowsPerCta - 1) / kRowsPerCta);
  gemv_t5_kernel<XBF, BP><<<blocks, kWarps * 32, smem, st>>>(W.codes, W.scales, x, y, n, k, batch);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return lb::cuda_fail(e, "lb_gemv (5-per-byte ternary): launch");
  return LB_OK;
}

// One instantiation per batch: every FMA of the digit loop then serves a live column (padding
// batch 5 to 8 spent 3 of every 8 FMAs and activation loads on zeros).
template <bool XBF>
lb_status launch_x(const lb_weight& W, const uint16_t* x, int batch, uint16_t* y, cudaStream_t st) {
  switch (batch) {
    case 1: return launch_bp<XBF, 1>(W, x, batch, y, st);
    case 2: return launch_bp<XBF, 2>(W, x, batch, y, st);
    case 3: return launch_bp<XBF, 3>(W, x, batch, y, st);
    case 4: return launch_bp<XBF, 4>(W, x, batch, y, st);
    case 5: return launch_bp<XBF, 5>(W, x, batch, y, st);
    case 6: return launch_bp<XBF, 6>(W, x, batch, y, st);
    case 7: return launch_bp<XBF, 7>(W, x, batch, y, st);
    default: return launch_bp<XBF, 8>(W, x, batch, y, st);
  }
}

}  // namespace

namespace lb {

lb_status launch_pack_ternary5(const int8_t* t, const uint16_t* s_in, int64_t n, int64_t k, uint8_t* codes,
                               uint16_t* scales, cudaStream_t st, uint32_t* flags_out) {
  const uint32_t zero = 0;
  cudaError_t e = cudaMemcpyToSymbolAsync(g_t5_flags, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "lb_pack_ternary5: reset flags");
  const int G = static_cast<int>(k / kGroup);
  const int64_t total = n * G * kT5Bytes;
  const int64_t want = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  pack_t5_kernel<<<static_cast<unsigned>(want < cap ? want : cap), 256, 0, st>>>(t, n, G, codes);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "lb_pack_ternary5: launch");
  if (scales != s_in) {
    e = cudaMemcpyAsync(scales, s_in, static_cast<size_t>(n) * G * 2, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "lb_pack_ternary5: copy scales");
  }
  e = cudaMemcpyFromSymbolAsync(flags_out, g_t5_flags, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "lb_pack_ternary5: read flags");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "lb_pack_ternary5: synchronize");
  return LB_OK;
}

lb_status launch_gemv_t5(const lb_weight& W, const void* x, int xdt, int batch, void* y, cudaStream_t st) {
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint16_t* ys = static_cast<uint16_t*>(y);
  return xdt == LB_BF16 ? launch_x<true>(W, xs, batch, ys, st) : launch_x<false>(W, xs, batch, ys, st);
}

}  // namespace lb
