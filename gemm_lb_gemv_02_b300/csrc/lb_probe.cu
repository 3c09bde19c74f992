// Read-bandwidth reference for the decode GEMVs: a launch that only reads a buffer, with the launch
// shape and programmatic-dependent-launch behaviour of the GEMV kernels (every CTA lets the next
// kernel on the stream launch at once, and back-to-back launches overlap their ramps).  It is no
// part of the method: the GEMV rows of the benchmark are read against it as the practical ceiling
// of one launch of the same byte count (7minutos.es, "PrismML lanza Bonsai 27B", section
// "Rendimiento y decodificación especulativa DSpark": decode is bound by memory bandwidth).
#include "lb_common.cuh"

namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeCtasPerSm = 4;
constexpr int kUnroll = 16;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// CTA c reads the c-th contiguous share of the buffer, kUnroll 16-byte loads per thread in flight,
// and folds everything it read into one XOR that goes to *sink (so that no load can be dropped).
__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4* __restrict__ p, size_t n16,
                                                                   uint32_t* __restrict__ sink) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const size_t per = (n16 + gridDim.x - 1) / gridDim.x;
  const size_t b = static_cast<size_t>(blockIdx.x) * per, e = min(n16, b + per);
  uint32_t acc = 0;
  size_t i = b + threadIdx.x;
  for (; i + static_cast<size_t>(kUnroll - 1) * kProbeThreads < e; i += static_cast<size_t>(kUnroll) * kProbeThreads) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(p + i + static_cast<size_t>(u) * kProbeThreads);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < e; i += kProbeThreads) {
    const uint4 v = ld_stream(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  asm volatile("griddepcontrol.wait;" ::: "memory");            // *sink is shared with earlier launches
  if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace

namespace lb {

lb_status launch_read_probe(const void* data, size_t bytes, uint32_t* sink, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sm_count() * kProbeCtasPerSm), 1, 1);
  cfg.blockDim = dim3(kProbeThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, read_probe_kernel, static_cast<const uint4*>(data), bytes / 16, sink);
  if (e != cudaSuccess) return cuda_fail(e, "lb_read_probe: launch");
  return LB_OK;
}

}  // namespace lb
