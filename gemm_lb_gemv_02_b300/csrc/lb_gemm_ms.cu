// Small-M GEMM (1 .. 32 token rows) against packed 1-bit or ternary weights, on the decode GEMV's
// engine:
//
//   Y[r][n] = sum_g s[n][g] * sum_{i<128} t[n][128g+i] * X[r][128g+i]
//
// (7minutos.es, "PrismML lanza Bonsai 27B", section "Rendimiento y decodificación especulativa
// DSpark": verification of k drafted tokens runs the target at width k + 1, and short prefill
// chunks are the same shape; section "Cómo funciona la compresión": w = s_g t_i.)
//
// With few tokens the cost is the weight decode, not the multiply-adds, so each decoded A fragment
// (mma.sync m16n8k16, the GEMV's exact decode) feeds MT = ceil(M / 8) MMAs, one per 8-token
// column tile.  The activations do not fit in shared memory next to the weight ring at this width,
// so they are streamed with the weights:
//   * prologue kernel: X -> binary16 B fragments in the decoder's K order (one CTA per padded token
//     row; bfloat16 rows are scaled by an exact power of two that puts the row's largest magnitude
//     in [2^15, 2^16), undone per output column), laid out [group][column tile][k pair][lane] so
//     that one bulk copy moves a stage's fragments; for 1-bit also the per-group baselines
//     -sum (o + 1/2) x of every column (the MMA's C operand, as in the GEMV);
//   * producer warp: per stage, 2-D TMA of the codes (128 rows x 8 groups, 128-byte swizzle) and
//     scales, and after griddepcontrol.wait one bulk copy of the stage's fragments (and baselines);
//   * 16 consumer warps, two per 16-row tile, each half of a stage's groups: codes and scales to
//     registers, then per group and MMA step one decode of the A fragment and MT MMAs against the
//     fragments in the slot; the slot is released after the stage's MMAs; the two halves of a
//     tile add their sums in shared memory at the end of a row block.
// CTAs are persistent over 128-row blocks.  Every mbarrier wait is bounded; a timeout sets a bit
// in the device error word and the CTA finishes.
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "lb_common.cuh"
#include "lb_decode.cuh"

namespace {

using namespace lbdec;

constexpr int NT = 8;                     // 16-row tiles per row block
constexpr int NW = 2 * NT;                // consumer warps
constexpr int ROWS = 16 * NT;
constexpr int kThreads = (NW + 1) * 32;   // + one producer warp
constexpr int GS = 8, GH = GS / 2;        // groups per stage; per consumer warp
constexpr int kBox = 16384, kScaleBox = ROWS * 16;
constexpr int kFrag = 2048;               // B fragments of one group and one 8-column tile
constexpr int kSmemMax = 227 * 1024;

template <int FMT>
struct MsFmt;
template <>
struct MsFmt<1> {
  static constexpr int gbytes = 16, nb = 1;
};
template <>
struct MsFmt<2> {
  static constexpr int gbytes = 32, nb = 2;
};

template <int FMT, int MT>
struct MsLayout {
  static constexpr int xoff = MsFmt<FMT>::nb * kBox + kScaleBox;   // in a slot: codes, scales, fragments
  static constexpr int xbytes = GS * MT * kFrag;
  static constexpr int coff = xoff + xbytes;                          // 1-bit baselines
  static constexpr int cbytes = FMT == 1 ? GS * MT * 64 : 0;
  static constexpr int slot = (coff + cbytes + 1023) / 1024 * 1024;
  static constexpr int red_bytes = ROWS * 8 * MT * 4;
  static constexpr int stages0 = (kSmemMax - 1024 - 256 - red_bytes) / slot;
  static constexpr int stages = stages0 > 6 ? 6 : stages0;
  static constexpr int bars = stages * slot;
  static constexpr int red = bars + 256;
  static constexpr int total = red + red_bytes + 1024;
  static_assert(stages >= 2, "two stages at least");
  static_assert(total <= kSmemMax, "shared memory");
};

struct MsArgs {
  CUtensorMap tm_codes;
  CUtensorMap tm_scales;
  const uint16_t* scales;   // for the non-TMA scale path
  const uint8_t* xfr;       // [Gpad][MT][4][32][16 B] fragments
  const uint8_t* cfr;       // [Gpad][MT][16] float baselines (1-bit)
  const float* fac;         // [8 MT] per-token factors
  uint16_t* y;              // [m][n]
  int n, k, G, m, row_blocks, scales_tma, y_bf16, test_fault;
  uint32_t* err;
  uint64_t wait_ns;
};

__device__ __forceinline__ void tile_sync(int t) { asm volatile("bar.sync %0, 64;" ::"r"(1 + t) : "memory"); }

// ------------------------------------------------------------------------------- prologue
// One CTA per padded token row r (rows >= m write zeros).  Tuple (g, qq): the 32 activations
// X[r][128g + 32qq ..] of one fragment lane, arranged exactly as the GEMV's prologue arranges them.
template <bool BF, int FMT, int MT>
__global__ void __launch_bounds__(256) xprep_ms_kernel(const uint16_t* __restrict__ x, int m, int k, int gpad,
                                                       uint8_t* __restrict__ xfr, float* __restrict__ cfr,
                                                       float* __restrict__ fac) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the GEMM may start loading weights
  __shared__ uint32_t warp_max[8];
  const int row = blockIdx.x;
  const bool live = row < m;
  const int G = k / 128;
  const int nt = row >> 3, col = row & 7;
  float sc = 1.f;
  if (BF) {
    uint32_t mx = 0;
    if (live) {
      const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(row) * k);
      for (int i = threadIdx.x; i < k / 8; i += 256) {
        const uint4 v = __ldg(src + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) mx = max(mx, max((w[j] << 16) & 0x7f800000u, w[j] & 0x7f800000u));
      }
    }
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) mx = max(mx, warp_max[w]);     // exponent fields order like magnitudes
    const int e = static_cast<int>(mx >> 23) - 127;
    const int p = min(126, max(-126, 15 - e));
    sc = __uint_as_float(static_cast<uint32_t>(127 + p) << 23);
    if (threadIdx.x == 0) fac[row] = live ? __uint_as_float(static_cast<uint32_t>(127 - p) << 23) : 0.f;
  } else if (threadIdx.x == 0) {
    fac[row] = live ? 1.f : 0.f;
  }
  const int tuples = gpad * 4;
  for (int base = 0; base < tuples; base += 256) {                 // uniform: quads stay together
    const int t = base + static_cast<int>(threadIdx.x);
    const int g = t >> 2, qq = t & 3;
    uint32_t X[16];
    const bool act = live && t < tuples && g < G;
    if (act) {
      const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(row) * k + 128 * g + 32 * qq);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(src + i);
        X[4 * i] = v.x; X[4 * i + 1] = v.y; X[4 * i + 2] = v.z; X[4 * i + 3] = v.w;
      }
      if (BF) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float lo = __uint_as_float(X[i] << 16) * sc, hi = __uint_as_float(X[i] & 0xffff0000u) * sc;
          const __half2 h2 = __floats2half2_rn(lo, hi);
          X[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) X[i] = 0u;
    }
    uint32_t B[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint32_t lo_src, hi_src, sel;
      if (FMT == 1) {
        lo_src = X[i >> 1]; hi_src = X[(i >> 1) + 8]; sel = (i & 1) ? 0x7632 : 0x5410;
      } else {
        const int uu = i >> 3, pp = i & 7;
        lo_src = X[8 * uu + (pp >> 1)]; hi_src = X[8 * uu + (pp >> 1) + 4]; sel = (pp & 1) ? 0x7632 : 0x5410;
      }
      B[i] = __byte_perm(lo_src, hi_src, sel);
    }
    float c = 0.f;
    if (FMT == 1) {
      // baseline sum_k (o_k + 1/2) x_k of this column and group: offsets summed per position first
#pragma unroll
      for (int mm = 4; mm <= 9; ++mm) {
        float sx = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (pos1(i) == mm) {
            const float2 fv = __half22float2(*reinterpret_cast<const __half2*>(&B[i]));
            sx += fv.x + fv.y;
          }
        c = fmaf(static_cast<float>(1 << (10 - mm)) + 0.5f, sx, c);
      }
      c += __shfl_xor_sync(0xffffffffu, c, 1);
      c += __shfl_xor_sync(0xffffffffu, c, 2);
    }
    if (t < tuples) {
      uint8_t* dst = xfr + (static_cast<size_t>(g) * MT + nt) * kFrag + (col * 4 + qq) * 16;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4*>(dst + i * 512) = make_uint4(B[4 * i], B[4 * i + 1], B[4 * i + 2], B[4 * i + 3]);
      if (FMT == 1 && qq == 0) {
        float* cb = cfr + (static_cast<size_t>(g) * MT + nt) * 16 + (col >> 1) * 4 + (col & 1);
        cb[0] = act ? -c : 0.f;                                    // {-C[2q], -C[2q+1], -C[2q], -C[2q+1]}
        cb[2] = act ? -c : 0.f;
      }
    }
  }
}

// ------------------------------------------------------------------------------- main kernel
template <int FMT, int MT>
__global__ void __launch_bounds__(kThreads, 1) gemm_ms_kernel(const __grid_constant__ MsArgs a) {
  using FT = MsFmt<FMT>;
  using L = MsLayout<FMT, MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (lbdev::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::bars);
  uint64_t* empty = full + L::stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nst = (a.G + GS - 1) / GS;                           // stages per row block
  const int my_rbs = (a.row_blocks - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x;
  const int total_st = my_rbs * nst;
  bool ok = true;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::stages; ++s) {
      lbdev::mbar_init(&full[s], a.scales_tma ? 1 : 32);
      lbdev::mbar_init(&empty[s], NW);
    }
    lbdev::fence_mbar_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ---------------- producer: weights first; the fragments only after the prologue kernel
    const bool stma = a.scales_tma != 0;
    if (lane == 0) {
      lbdev::prefetch_tmap(&a.tm_codes);
      if (stma) lbdev::prefetch_tmap(&a.tm_scales);
    }
    const uint32_t bytes = static_cast<uint32_t>(FT::nb * kBox + (stma ? kScaleBox : 0) + L::xbytes + L::cbytes);
    bool xdep = false;
    if (stma ? lane == 0 : true) {
      for (int st = 0; st < total_st && !a.test_fault; ++st) {
        const int s = st % L::stages;
        if (!lbdev::mbar_wait_backoff(&empty[s], static_cast<uint32_t>(((st / L::stages) & 1) ^ 1), a.wait_ns)) {
          ok = false;
          break;
        }
        const int row0 = (static_cast<int>(blockIdx.x) + (st / nst) * static_cast<int>(gridDim.x)) * ROWS;
        const int g0 = (st % nst) * GS;
        uint8_t* slot = sm + s * L::slot;
        if (!stma) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = row0 + lane + 32 * i;
            uint32_t v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int g = g0 + 2 * j;
              const uint16_t* src = a.scales + static_cast<int64_t>(row) * a.G + g;
              const uint32_t lo = (row < a.n && g < a.G) ? __ldg(src) : 0u;
              const uint32_t hi = (row < a.n && g + 1 < a.G) ? __ldg(src + 1) : 0u;
              v[j] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4*>(slot + FT::nb * kBox + (lane + 32 * i) * 16) = make_uint4(v[0], v[1], v[2], v[3]);
          }
          if (lane != 0) lbdev::mbar_arrive(&full[s]);
        }
        if (lane == 0) {
          lbdev::mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
          for (int b = 0; b < FT::nb; ++b)
            lbdev::tma_load_2d(slot + b * kBox, &a.tm_codes, (g0 + b * (GS / FT::nb)) * FT::gbytes, row0, &full[s]);
          if (stma) lbdev::tma_load_2d(slot + FT::nb * kBox, &a.tm_scales, g0, row0, &full[s]);
          if (!xdep) {
            griddep_wait();                                        // the prologue kernel wrote the fragments
            xdep = true;
          }
          lbdev::bulk_g2s(slot + L::xoff, a.xfr + static_cast<size_t>(g0) * MT * kFrag, L::xbytes, &full[s]);
          if (FMT == 1)
            lbdev::bulk_g2s(slot + L::coff, a.cfr + static_cast<size_t>(g0) * MT * 64, L::cbytes, &full[s]);
        }
      }
    }
    __syncwarp();
    griddep_launch();
  } else {
    // ---------------- consumers (they read the prologue's token factors and write y: wait for it)
    griddep_wait();
    const int r = lane >> 2, q = lane & 3;
    const int tile = warp & (NT - 1), half = warp / NT;
    const int ia = tile * 16 + r;
    uint32_t M[10], SC[10];
    constexpr uint32_t kMask = FMT == 1 ? 0x00010001u : 0x00030003u;
#define LB_MASK(mm)                                                                                  \
  asm volatile("mov.b32 %0, %1;" : "=r"(M[mm]) : "n"(kMask << (mm)));                               \
  asm volatile("mov.b32 %0, %1;" : "=r"(SC[mm]) : "n"(expo16(mm) | (0x00010001u << (mm))))
    LB_MASK(0); LB_MASK(1); LB_MASK(2); LB_MASK(3); LB_MASK(4);
    LB_MASK(5); LB_MASK(6); LB_MASK(7); LB_MASK(8); LB_MASK(9);
#undef LB_MASK
    uint32_t pcode;
    if (FMT == 1) {
      pcode = static_cast<uint32_t>(ia * 128) | (4u * q) | (static_cast<uint32_t>(r) << 4);
      pcode ^= static_cast<uint32_t>(half * GH) << 4;
    } else {
      pcode = static_cast<uint32_t>(ia * 128) | (8u * (q & 1)) | (static_cast<uint32_t>((q >> 1) ^ r) << 4);
      pcode += static_cast<uint32_t>(half * kBox);
    }
    uint32_t pc[GH];
#pragma unroll
    for (int j = 0; j < GH; ++j) pc[j] = pcode ^ (static_cast<uint32_t>(j) << (FMT == 1 ? 4 : 5));
    const uint32_t sm32 = lbdev::smem_u32(sm);
    const uint32_t sc_off = static_cast<uint32_t>(FT::nb * kBox + ia * 16 + half * 8);
    const uint32_t x_off = static_cast<uint32_t>(L::xoff + half * GH * MT * kFrag + lane * 16);
    const uint32_t c_off = static_cast<uint32_t>(L::coff + half * GH * MT * 64 + 16 * q);
    float* red = reinterpret_cast<float*>(sm + L::red);
    float acc[MT][4];
#pragma unroll
    for (int nt = 0; nt < MT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    int s = 0;
    uint32_t ph = 0;
    for (int j_rb = 0; j_rb < my_rbs; ++j_rb) {
      for (int cst = 0; cst < nst; ++cst) {
        const uint32_t slot = sm32 + static_cast<uint32_t>(s * L::slot);
        if (ok && !lbdev::mbar_wait(&full[s], ph, a.wait_ns)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          uint2 ca[GH], cb[GH];
#pragma unroll
          for (int j = 0; j < GH; ++j) {
            const uint32_t o = slot + pc[j];
            if (FMT == 1) {
              ca[j] = make_uint2(ldsv32(o), 0u);
              cb[j] = make_uint2(ldsv32(o + 1024), 0u);
            } else {
              ca[j] = ldsv64(o);
              cb[j] = ldsv64(o + 1024);
            }
          }
          const uint2 va = ldsv64(slot + sc_off), vb = ldsv64(slot + sc_off + 128);
          float sa[GH], sb[GH];
          {
            const float2 a01 = __half22float2(*reinterpret_cast<const __half2*>(&va.x));
            const float2 a23 = __half22float2(*reinterpret_cast<const __half2*>(&va.y));
            const float2 b01 = __half22float2(*reinterpret_cast<const __half2*>(&vb.x));
            const float2 b23 = __half22float2(*reinterpret_cast<const __half2*>(&vb.y));
            sa[0] = a01.x; sa[1] = a01.y; sa[2] = a23.x; sa[3] = a23.y;
            sb[0] = b01.x; sb[1] = b01.y; sb[2] = b23.x; sb[3] = b23.y;
          }
#pragma unroll
          for (int j = 0; j < GH; ++j) {
            const Word1 w1a = prep1(ca[j].x), w1b = prep1(cb[j].x);
            const Word2 la = prep2(ca[j].x), ha = prep2(ca[j].y), lb = prep2(cb[j].x), hb = prep2(cb[j].y);
            const uint32_t xj = slot + x_off + static_cast<uint32_t>(j * MT * kFrag);
            float d[MT][4];
#pragma unroll
            for (int iq = 0; iq < 4; ++iq) {
              // the fragments of two MMA steps (all column tiles), or, with 4 tiles, of one step at
              // a time (registers)
              uint4 bx[MT];
              if (MT < 4) {
#pragma unroll
                for (int nt = 0; nt < MT; ++nt) bx[nt] = ldsv128(xj + nt * kFrag + iq * 512);
              }
#define LB_STEP(I)                                                                                   \
  {                                                                                                  \
    const uint32_t e0 = areg<FMT, 2 * (I)>(w1a, la, ha, M, SC), e1 = areg<FMT, 2 * (I)>(w1b, lb, hb, M, SC); \
    const uint32_t e2 = areg<FMT, 2 * (I) + 1>(w1a, la, ha, M, SC);                                   \
    const uint32_t e3 = areg<FMT, 2 * (I) + 1>(w1b, lb, hb, M, SC);                                   \
    _Pragma("unroll") for (int nt = 0; nt < MT; ++nt) {                                              \
      uint32_t b0, b1;                                                                               \
      if (MT < 4) {                                                                                  \
        b0 = (I) % 2 == 0 ? bx[nt].x : bx[nt].z;                                                     \
        b1 = (I) % 2 == 0 ? bx[nt].y : bx[nt].w;                                                     \
      } else {                                                                                       \
        const uint2 bb = ldsv64(xj + nt * kFrag + ((I) >> 1) * 512 + ((I) & 1) * 8);                \
        b0 = bb.x;                                                                                   \
        b1 = bb.y;                                                                                   \
      }                                                                                              \
      if ((I) == 0 && FMT == 1) {                                                                    \
        const uint32_t ca4 = slot + c_off + static_cast<uint32_t>((j * MT + nt) * 64);               \
        float4 cn;                                                                                   \
        asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"                                         \
                     : "=f"(cn.x), "=f"(cn.y), "=f"(cn.z), "=f"(cn.w) : "r"(ca4));                   \
        mma_c4(d[nt], e0, e1, e2, e3, b0, b1, cn);                                                   \
      } else if ((I) == 0) {                                                                         \
        mma_zero(d[nt], e0, e1, e2, e3, b0, b1);                                                     \
      } else {                                                                                       \
        mma_acc(d[nt], e0, e1, e2, e3, b0, b1);                                                      \
      }                                                                                              \
    }                                                                                                \
  }
              if (iq == 0) { LB_STEP(0) LB_STEP(1) }
              else if (iq == 1) { LB_STEP(2) LB_STEP(3) }
              else if (iq == 2) { LB_STEP(4) LB_STEP(5) }
              else { LB_STEP(6) LB_STEP(7) }
#undef LB_STEP
            }
#pragma unroll
            for (int nt = 0; nt < MT; ++nt) {
              acc[nt][0] = fmaf(sa[j], d[nt][0], acc[nt][0]);
              acc[nt][1] = fmaf(sa[j], d[nt][1], acc[nt][1]);
              acc[nt][2] = fmaf(sb[j], d[nt][2], acc[nt][2]);
              acc[nt][3] = fmaf(sb[j], d[nt][3], acc[nt][3]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) lbdev::mbar_arrive(&empty[s]);             // the stage's fragments are read
        if (++s == L::stages) { s = 0; ph ^= 1u; }
      }
      // ---- row block done: the two halves of each tile add up in shared memory
      const int rb = static_cast<int>(blockIdx.x) + j_rb * static_cast<int>(gridDim.x);
      constexpr int RW = 8 * MT;                                   // floats per row in `red`
      if (half == 1) {
#pragma unroll
        for (int nt = 0; nt < MT; ++nt) {
          red[ia * RW + 8 * nt + 2 * q] = acc[nt][0];
          red[ia * RW + 8 * nt + 2 * q + 1] = acc[nt][1];
          red[(ia + 8) * RW + 8 * nt + 2 * q] = acc[nt][2];
          red[(ia + 8) * RW + 8 * nt + 2 * q + 1] = acc[nt][3];
        }
      }
      if (j_rb == my_rbs - 1) griddep_launch();
      tile_sync(tile);
      if (half == 0) {
        const float mul = FMT == 1 ? 2.f : 1.f;                    // 1-bit: the MMA gives sum t x / 2
        const int row_a = rb * ROWS + ia, row_b = row_a + 8;
#pragma unroll
        for (int nt = 0; nt < MT; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int lrow = e < 2 ? ia : ia + 8, row = e < 2 ? row_a : row_b;
            const int col = 8 * nt + 2 * q + (e & 1);
            const float v = (acc[nt][e] + red[lrow * RW + col]) * (mul * a.fac[col]);
            if (row < a.n && col < a.m)
              a.y[static_cast<int64_t>(col) * a.n + row] =
                  a.y_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
          }
        }
      }
      tile_sync(tile);                                             // red is free for the next row block
#pragma unroll
      for (int nt = 0; nt < MT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    }
  }
  if (!ok) atomicOr(a.err, lb::kErrGemmTimeout);
}

template <int FMT, int MT>
lb_status launch_t(const MsArgs& args, cudaStream_t st) {
  using L = MsLayout<FMT, MT>;
  {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return lb::cuda_fail(e, "lb_gemm: cudaGetDevice");
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64 || !done[dev]) {
      e = cudaFuncSetAttribute(gemm_ms_kernel<FMT, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total);
      if (e != cudaSuccess) return lb::cuda_fail(e, "lb_gemm: set shared memory size");
      if (dev >= 0 && dev < 64) done[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(min(args.row_blocks, lb::sm_count())), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;    // overlap the prologue kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_ms_kernel<FMT, MT>, args);
  if (e != cudaSuccess) return lb::cuda_fail(e, "lb_gemm: launch");
  return LB_OK;
}

template <bool BF, int FMT, int MT>
void launch_prep(const uint16_t* x, int m, int k, int gpad, uint8_t* xfr, float* cfr, float* fac, cudaStream_t st) {
  xprep_ms_kernel<BF, FMT, MT><<<8 * MT, 256, 0, st>>>(x, m, k, gpad, xfr, cfr, fac);
}

template <int FMT, int MT>
lb_status launch_fm(const lb_weight& W, const void* x, int xdt, int64_t m, void* y, int ydt, void* ws,
                    const CUtensorMap& tm_codes, const CUtensorMap& tm_scales, int scales_tma, bool fault,
                    cudaStream_t st) {
  const int k = static_cast<int>(W.k), n = static_cast<int>(W.n), G = k / lb::kGroup;
  const int gpad = (G + GS - 1) / GS * GS;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  uint8_t* xfr = wsb;
  const size_t xfr_bytes = static_cast<size_t>(gpad) * MT * kFrag;
  float* cfr = reinterpret_cast<float*>(wsb + xfr_bytes);
  const size_t cfr_bytes = (static_cast<size_t>(gpad) * MT * 64 + 255) / 256 * 256;
  float* fac = reinterpret_cast<float*>(wsb + xfr_bytes + cfr_bytes);
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  if (xdt == LB_BF16) launch_prep<true, FMT, MT>(xs, static_cast<int>(m), k, gpad, xfr, cfr, fac, st);
  else launch_prep<false, FMT, MT>(xs, static_cast<int>(m), k, gpad, xfr, cfr, fac, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return lb::cuda_fail(e, "lb_gemm: prologue launch");
  uint32_t* err = lb::device_error_word();
  if (!err) return lb::fail(LB_ERR_CUDA, "lb_gemm: device error word unavailable");
  MsArgs args;
  memset(&args, 0, sizeof(args));
  args.tm_codes = tm_codes;
  args.tm_scales = tm_scales;
  args.scales = W.scales;
  args.xfr = xfr;
  args.cfr = reinterpret_cast<const uint8_t*>(cfr);
  args.fac = fac;
  args.y = static_cast<uint16_t*>(y);
  args.n = n;
  args.k = k;
  args.G = G;
  args.m = static_cast<int>(m);
  args.row_blocks = (n + ROWS - 1) / ROWS;
  args.scales_tma = scales_tma;
  args.y_bf16 = ydt == LB_BF16 ? 1 : 0;
  args.test_fault = fault ? 1 : 0;
  args.err = err;
  args.wait_ns = fault ? lb::kTestWaitNs : lb::kWaitNs;
  return launch_t<FMT, MT>(args, st);
}

}  // namespace

namespace lb {

// Workspace of the small-M path: fragments (Gpad x MT x 2 KB), baselines, per-token factors; it is
// never larger than the tcgen05 path's workspace for the same m and k.
size_t gemm_ms_workspace_bytes(int64_t m, int64_t k) {
  const int mt = m <= 8 ? 1 : m <= 16 ? 2 : 4;
  const int64_t gpad = (k / kGroup + GS - 1) / GS * GS;
  return static_cast<size_t>(gpad) * mt * kFrag + (static_cast<size_t>(gpad) * mt * 64 + 255) / 256 * 256 +
         static_cast<size_t>(8 * mt) * 4;
}

lb_status launch_gemm_ms(const lb_weight& W, const void* x, int xdt, int64_t m, void* y, int ydt, void* ws,
                         const CUtensorMap& tm_codes, const CUtensorMap& tm_scales, int scales_tma, bool fault,
                         cudaStream_t st) {
  const bool one = W.fmt == LB_FMT_1BIT_G128;
  if (m <= 8) return one ? launch_fm<1, 1>(W, x, xdt, m, y, ydt, ws, tm_codes, tm_scales, scales_tma, fault, st)
                         : launch_fm<2, 1>(W, x, xdt, m, y, ydt, ws, tm_codes, tm_scales, scales_tma, fault, st);
  if (m <= 16) return one ? launch_fm<1, 2>(W, x, xdt, m, y, ydt, ws, tm_codes, tm_scales, scales_tma, fault, st)
                          : launch_fm<2, 2>(W, x, xdt, m, y, ydt, ws, tm_codes, tm_scales, scales_tma, fault, st);
  return one ? launch_fm<1, 4>(W, x, xdt, m, y, ydt, ws, tm_codes, tm_scales, scales_tma, fault, st)
             : launch_fm<2, 4>(W, x, xdt, m, y, ydt, ws, tm_codes, tm_scales, scales_tma, fault, st);
}

}  // namespace lb
