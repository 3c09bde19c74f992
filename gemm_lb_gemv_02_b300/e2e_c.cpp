// End-to-end timing of the C ABI from a plain C++ caller, with host buffers: the 27B-class ternary
// decode layer set (q, o 5120 x 5120; gate, up 17408 x 5120; down 5120 x 17408) at batch 1 with
// bfloat16 activations, issued as a decoder layer issues it ([q], [o], [gate, up] on one x,
// [down]) through `layers` distinct copies of the set.  One step: the four activation vectors are
// copied from pinned host memory, every layer's four calls are made, the five outputs of the last
// layer are copied back, and the stream is synchronised.  Host wall clock over `steps` steps after
// `warmup` steps and ~0.3 s of the same load (an idle GPU lowers its clocks).
//
// Prints one JSON line: GB/s of algorithmic bytes (codes + scales + x + y, a shared x counted
// once), microseconds per step, and the host time spent inside the lb_* calls per call (the
// library's own host cost: argument checks, tensor-map cache lookups, launch).
//
//   e2e_c [layers] [steps] [warmup]
#include <cuda_runtime.h>

#include <chrono>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "lb.h"

namespace {

struct Mat {
  int64_t n, k;
};
const Mat kMats[5] = {{5120, 5120}, {5120, 5120}, {17408, 5120}, {17408, 5120}, {5120, 17408}};

#define CK(x)                                                                        \
  do {                                                                               \
    cudaError_t e_ = (x);                                                            \
    if (e_ != cudaSuccess) {                                                         \
      std::fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
      std::exit(1);                                                                  \
    }                                                                                \
  } while (0)
#define LB(x)                                                                                   \
  do {                                                                                          \
    lb_status s_ = (x);                                                                         \
    if (s_ != LB_OK) {                                                                          \
      std::fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, lb_status_string(s_), lb_last_error()); \
      std::exit(1);                                                                             \
    }                                                                                           \
  } while (0)

uint64_t g_state = 0x9E3779B97F4A7C15ull;
uint64_t next_u64() {  // xorshift64*
  g_state ^= g_state >> 12;
  g_state ^= g_state << 25;
  g_state ^= g_state >> 27;
  return g_state * 0x2545F4914F6CDD1Dull;
}
uint16_t bf16_of(float f) {  // round to nearest even (finite inputs)
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}
uint16_t half_scale() {  // a binary16 scale in [2^-7, 2^-5): exponent 8..9, random mantissa
  return static_cast<uint16_t>(((8 + (next_u64() & 1)) << 10) | (next_u64() & 0x3FF));
}

}  // namespace

int main(int argc, char** argv) {
  const int layers = argc > 1 ? std::atoi(argv[1]) : 8;
  const int steps = argc > 2 ? std::atoi(argv[2]) : 20;
  const int warmup = argc > 3 ? std::atoi(argv[3]) : 3;
  cudaStream_t st;
  CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));

  // one packed copy of the set through the packer, then device copies of it for the other layers
  std::vector<lb_weight> W(5 * layers);
  size_t weight_bytes = 0;
  for (int m = 0; m < 5; ++m) {
    const int64_t n = kMats[m].n, k = kMats[m].k;
    std::vector<int8_t> t(static_cast<size_t>(n * k));
    for (auto& v : t) v = static_cast<int8_t>(static_cast<int>(next_u64() % 3) - 1);
    std::vector<uint16_t> s(static_cast<size_t>(n * (k / 128)));
    for (auto& v : s) v = half_scale();
    int8_t* dt;
    uint16_t* ds;
    CK(cudaMalloc(&dt, t.size()));
    CK(cudaMalloc(&ds, s.size() * 2));
    CK(cudaMemcpy(dt, t.data(), t.size(), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(ds, s.data(), s.size() * 2, cudaMemcpyHostToDevice));
    size_t cb, sb;
    LB(lb_packed_bytes(LB_FMT_TERNARY_G128, n, k, &cb, &sb));
    for (int l = 0; l < layers; ++l) {
      uint8_t* codes;
      uint16_t* scales;
      CK(cudaMalloc(&codes, cb));
      CK(cudaMalloc(&scales, sb));
      if (l == 0) {
        LB(lb_pack_ternary(dt, ds, n, k, codes, scales, st));
      } else {
        CK(cudaMemcpy(codes, W[m].codes, cb, cudaMemcpyDeviceToDevice));
        CK(cudaMemcpy(scales, W[m].scales, sb, cudaMemcpyDeviceToDevice));
      }
      W[5 * l + m] = lb_weight{LB_FMT_TERNARY_G128, 0, n, k, codes, scales};
      weight_bytes += cb + sb;
    }
    CK(cudaFree(dt));
    CK(cudaFree(ds));
  }

  // activations: [q], [o], [gate, up], [down] read 4 distinct vectors; 5 outputs
  const int64_t xk[4] = {5120, 5120, 5120, 17408};
  void* x[4];
  uint16_t* xh[4];
  size_t h2d = 0, d2h = 0;
  for (int i = 0; i < 4; ++i) {
    CK(cudaMalloc(&x[i], xk[i] * 2));
    CK(cudaMallocHost(&xh[i], xk[i] * 2));
    for (int64_t j = 0; j < xk[i]; ++j)
      xh[i][j] = bf16_of(static_cast<float>(static_cast<int64_t>(next_u64() % 2001) - 1000) / 500.f);
    h2d += xk[i] * 2;
  }
  void* y[5];
  uint16_t* yh[5];
  for (int m = 0; m < 5; ++m) {
    CK(cudaMalloc(&y[m], kMats[m].n * 2));
    CK(cudaMallocHost(&yh[m], kMats[m].n * 2));
    d2h += kMats[m].n * 2;
  }
  const size_t bytes_per_step = weight_bytes + static_cast<size_t>(layers) * (h2d + d2h);
  CK(cudaDeviceSynchronize());

  double call_s = 0.0;
  long calls = 0;
  auto step = [&](bool count) {
    for (int i = 0; i < 4; ++i) CK(cudaMemcpyAsync(x[i], xh[i], xk[i] * 2, cudaMemcpyHostToDevice, st));
    for (int l = 0; l < layers; ++l) {
      const lb_weight* w = &W[5 * l];
      const auto t0 = std::chrono::steady_clock::now();
      LB(lb_gemv(&w[0], x[0], LB_BF16, 1, y[0], st));
      LB(lb_gemv(&w[1], x[1], LB_BF16, 1, y[1], st));
      const lb_gemv_problem gu[2] = {{w[2], x[2], y[2]}, {w[3], x[2], y[3]}};
      LB(lb_gemv_batched(gu, 2, LB_BF16, 1, st));
      LB(lb_gemv(&w[4], x[3], LB_BF16, 1, y[4], st));
      if (count) {
        call_s += std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
        calls += 4;
      }
    }
    for (int m = 0; m < 5; ++m) CK(cudaMemcpyAsync(yh[m], y[m], kMats[m].n * 2, cudaMemcpyDeviceToHost, st));
    CK(cudaStreamSynchronize(st));
  };

  const auto b0 = std::chrono::steady_clock::now();
  while (std::chrono::duration<double>(std::chrono::steady_clock::now() - b0).count() < 0.3) step(false);
  for (int i = 0; i < warmup; ++i) step(false);
  const auto t0 = std::chrono::steady_clock::now();
  for (int i = 0; i < steps; ++i) step(true);
  const double dt = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  uint32_t err = 0;
  LB(lb_device_error(&err, 1));
  std::printf("{\"value\": %.1f, \"unit\": \"GB/s\", \"us_per_step\": %.2f, \"layers\": %d, \"steps\": %d, "
              "\"host_us_per_call\": %.2f, \"calls_per_step\": %d, \"h2d_bytes_per_step\": %zu, "
              "\"d2h_bytes_per_step\": %zu, \"device_error\": %u}\n",
              bytes_per_step / dt * steps / 1e9, dt / steps * 1e6, layers, steps, call_s / calls * 1e6,
              4 * layers, h2d, d2h, err);
  return err == 0 ? 0 : 2;
}
