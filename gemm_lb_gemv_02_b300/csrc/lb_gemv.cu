// Decode GEMV / small-batch GEMV against packed 1-bit or ternary weights (batch 1..8; ternary in
// 2-bit fields, or five per byte at batch 1).
//
//   y[b][n] = sum_g s[n][g] * sum_{i<128} t[n][128g+i] * x[b][128g+i]
//
// (7minutos.es, "PrismML lanza Bonsai 27B", sections "Cómo funciona la compresión" for w = s_g t_i
// and "Rendimiento y decodificación especulativa DSpark" for the bandwidth-bound decode and the
// width-5 speculative verification.)
//
// Why tensor cores in a GEMV.  A 1-bit GEMV must retire ~37 T weights/s to stream at 80% of B300
// HBM bandwidth, about one lane-operation per weight over the whole GPU, and integer LOP3 issues
// at half rate on sm_103a.  The per-weight multiply-add therefore runs on mma.sync m16n8k16
// (batch <= 8 fills its n = 8 columns), fed by a decode of one LOP3 per two weights:
//
//   * "offset exponent" decode: a binary16 whose exponent encodes 2^(10-m) and whose mantissa bit
//     m (ternary: bits m, m+1) is copied from the code word has the exact value o + b, o = 2^(10-m),
//     b the code bit (2-bit field).  One LOP3 (mask held in a register, exponent as immediate)
//     builds two such halves, i.e. one half2 A-fragment register.
//   * 1-bit: per group g and batch column c the constant C_g[c] = sum_k (o_k + 1/2) x[c][k] is
//     computed once per CTA in FP32 and fed as the MMA's C operand -C_g, so the tensor core
//     returns sum_k (b_k - 1/2) x_k = sum t x / 2.  The offsets are kept <= 64, and every element
//     of a 1-bit row counts in sum |s t x|, so the cancellation stays far inside the tolerance.
//   * ternary: one HSUB2 turns o + f into f - 1 = t exactly, and the MMA starts from zero.  A zero
//     code then contributes exactly nothing; a baseline would cancel o x against o x, and for a large
//     x met by zero codes that rounding alone could exceed the tolerance of the row.
//   * the group scale is applied once per group in FP32: acc += s * D_g; 1-bit doubles at the end.
//   * the reduction order along K is free, so code bit j of a word lands in whichever k slot its
//     register occupies; x is gathered once per CTA into B fragments in the matching order.
//   * bfloat16 x is converted to binary16 after an exact power-of-two rescaling per batch column
//     that puts the column's largest magnitude in [2^15, 2^16) (undone on the FP32 result), so both
//     activation types share the binary16 decode; every element within 2^32 of the column maximum
//     is converted exactly.
//
// Lookup-table form (batch 1, BP = 0): thread = weight row, and the activations become tables of
// signed sums in shared memory, built once per CTA for its K range.  1-bit: per chunk of four
// activations the 16 sums of +-x, so a code nibble costs one lookup and one FADD.  Five per byte:
// per byte slot of a group, the 9 sums over its first two weights and the 27 over its last three,
// so a code byte b costs two lookups (b mod 9, b / 9) and two FADDs.
//
// Memory pipeline: a producer warp streams the codes (and scales) of 128-row x 8-group tiles with
// 2-D TMA loads (128-byte swizzled, so the consumers' fragment reads hit 32 distinct banks) into a
// ring of shared-memory stages.  Sixteen consumer warps work on the eight 16-row tiles of a row
// block, two per tile, each taking half of a stage's groups; their partial sums meet in shared
// memory at the end of the row block.  CTAs are persistent over row blocks.  When a matrix has
// too few row blocks to fill the GPU, K is split across the CTAs of a thread-block cluster: each
// rank stores its partial sums into the row owner's shared memory with st.async, counted in bytes
// on the owner's exchange mbarrier, and each owner sums its rows.  The kernel is launched with programmatic
// dependent launch: weight loads start before griddepcontrol.wait, which guards every read of x
// and write of y.
//
// Launch modes (the problem table in the kernel's arguments): one GEMV with persistent CTAs; up to
// 8 GEMVs in one launch with one CTA (or cluster) per (problem, row block); and the SiLU-gated
// pair, in which one CTA (or cluster) runs a row block of the gate matrix and then the same row
// block of the up matrix on one x prologue and writes h = silu(g) * u (g and u stay in FP32).
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "lb_common.cuh"
#include "lb_decode.cuh"

namespace {

using namespace lbdec;

constexpr int NT = 8;                     // 16-row tiles per row block
constexpr int NW = 2 * NT;                // consumer warps: two per tile
constexpr int ROWS = 16 * NT;             // rows per row block
constexpr int kThreads = (NW + 1) * 32;   // + one TMA producer warp
constexpr int kMaxCluster = 8;
constexpr int GS = 8;                     // groups per pipeline stage
constexpr int GH = GS / 2;                // groups per consumer warp per stage
constexpr int kBox = 16384;               // one codes box: 128 rows x 128 bytes
constexpr int kScaleBox = ROWS * 16;      // 128 rows x 8 binary16 scales
constexpr int kSmemMax = 227 * 1024;

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<1> {                     // 1-bit: 16 B per group per row, 8 groups per box
  static constexpr int gbytes = 16, nb = 1, stages = 6;
  static constexpr int box = kBox;
};
template <>
struct FmtTraits<2> {                     // ternary: 32 B per group per row, 4 groups per box
  static constexpr int gbytes = 32, nb = 2, stages = 3;
  static constexpr int box = kBox;
};
template <>
struct FmtTraits<3> {                     // ternary five per byte: 26 B per group per row, one
  static constexpr int gbytes = 26, nb = 1, stages = 2;   // 128-row x 208-byte box (no swizzle)
  static constexpr int box = 8 * 26 * 128;
};

// SiLU gate, silu(g) = g * sigmoid(g) = g / (1 + e^-g), in FP32 (expf: CUDA's accurate
// exponential; e^-g = inf for very negative g gives a signed zero, as the limit does).
__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

// ----------------------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
// An arrival that releases nothing: for a thread whose only writes the cluster must see are
// mbarrier initialisations, which fence.mbarrier_init.release.cluster has already released.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// v into the shared memory of cluster CTA `rank`, at the image of `local_addr` there; the store
// counts its 4 bytes on that CTA's mbarrier at the image of `local_bar` (complete_tx), which makes
// the value visible to the threads that wait on that barrier.
__device__ __forceinline__ void st_async_f32(uint32_t local_addr, uint32_t local_bar, uint32_t rank, float v) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(local_bar), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(ra),
               "r"(__float_as_uint(v)), "r"(rb)
               : "memory");
}
// Phase trace (compiled in only with -DLB_GEMV_TRACE, for timing studies): per CTA, event e holds
// {%globaltimer, clock64} of the moment one fixed thread passed a point of the kernel.  Events:
// 0 CTA start, 1 producer's first copy issued, 2 producer's last copy issued, 3 consumers past
// griddepcontrol.wait, 4 x prologue done, 5 + i (i < 16) warp 0 got stage i, 21 + j (j < 8) warp
// 0 finished unit j, 29 consumers done, 30 CTA end; producer start-up: 31 barriers initialised
// and fenced, 32 past its start-up arrivals, 33 at the start of its copy loop, 34 first slot granted;
// the last slot holds {gridDim.x, gridDim.y}.
#ifdef LB_GEMV_TRACE
constexpr int kTraceCtas = 2048, kTraceEvents = 40;
__device__ unsigned long long g_gemv_trace[kTraceCtas][kTraceEvents][2];
__device__ __forceinline__ void trace_ev(int e) {
  const unsigned cta = blockIdx.y * gridDim.x + blockIdx.x;
  if (cta < kTraceCtas && e < kTraceEvents) {
    g_gemv_trace[cta][e][0] = lbdev::globaltimer_ns();
    g_gemv_trace[cta][e][1] = static_cast<unsigned long long>(clock64());
  }
}
#define LB_TRACE(cond, e) \
  do {                    \
    if (cond) trace_ev(e); \
  } while (0)
#else
#define LB_TRACE(cond, e) \
  do {                    \
  } while (0)
#endif

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory"); }
constexpr int kBarInit = 10;              // named barrier: the producer's barrier setup -> consumers
// the two consumer warps of 16-row tile t (named barriers 2 .. NT + 1)
__device__ __forceinline__ void tile_sync(int t) { asm volatile("bar.sync %0, 64;" ::"r"(2 + t) : "memory"); }

constexpr int kMaxProblems = 8;           // GEMVs of one grouped launch

// One GEMV of a launch.
struct Prob {
  CUtensorMap tm_codes;       // codes plane as a 2-D u8 tensor {code bytes per row, n}, box 128 x 128
  CUtensorMap tm_scales;      // scales plane as a 2-D u16 tensor {G, n}, box 8 x 128 (if scales_tma)
  const uint16_t* scales;
  const uint16_t* x;
  uint16_t* y;
  int n, k, G;
  int gpc;         // groups per K chunk (a multiple of GS when S > 1)
  int row_blocks;
  int scales_tma;  // scales arrive in the stage through tm_scales
  int unit0;       // first grid row (blockIdx.y) of this problem in a grouped launch
};
struct Args {
  Prob p[kMaxProblems];
  uint32_t* err;
  int count;       // problems; 1 = one GEMV with persistent CTAs, > 1 = one CTA per row block
  int batch;
  int S;           // CTAs per cluster along K (chunk = cluster rank); 1 when count > 1
  int fuse;        // 1: SiLU-gated pair, p[0] = gate, p[1] = up (same n, k, x); h -> p[0].y
  int shared;      // count > 1, S == 1, one x and one K for all: CTAs persistent over all units
  int units;       // units of a shared launch
  int test_fault;  // issue no weight copy, so that every pipeline wait gives up after wait_ns
  uint64_t wait_ns;
};

// BP = 0 selects the 1-bit lookup-table consumer at batch 1 (see the kernel): its x region is a
// table of 2 KB per group instead of mma.sync fragments, and it has no baselines.
template <int FMT, int BP>
struct Layout {
  static constexpr bool LU = BP == 0;
  static constexpr int stages = FmtTraits<FMT>::stages;
  static constexpr int slot = FmtTraits<FMT>::nb * FmtTraits<FMT>::box + kScaleBox;
  static constexpr int ring = stages * slot;                     // 1024-byte aligned base
  static constexpr int bars = ring;                              // full[stages], empty[stages], xbar at 15
  static_assert(2 * stages <= 15, "stage barriers and the exchange barrier share 128 bytes");
  static constexpr int red = bars + 128;                         // 2 x ROWS x 8 floats
  static constexpr int colf = red + 2 * ROWS * 8 * 4;            // 8 column factors + 8 column maxima
  // K split across a cluster: rank p's partial of row r (unit u) lands in the row's owner at
  // slot (u * S + p) * per + (r - owner's first row), per = ceil(ROWS / S) rows per owner
  static constexpr int xchg = colf + 64;                         // 2 units x (ROWS + kMaxCluster) x 8 floats
  static constexpr int cneg = xchg + 2 * (ROWS + kMaxCluster) * 8 * 4;   // gpc x 4 x float4 {-C[2q], -C[2q+1], same}
  static constexpr int xgroup = LU ? (FMT == 3 ? 26 * 36 * 4 : 32 * 16 * 4) : 4 * 4 * BP * 16;   // x fragments (table) of one group
  // the x fragments and baselines are padded to whole stages (zeros), so a stage is always full;
  // the table starts on a 256-byte boundary (its lookups replace an address's low byte)
  __host__ __device__ static int pad(int gpc) { return (gpc + GS - 1) / GS * GS; }
  __host__ __device__ static int xs(int gpc) { return LU ? (cneg + 255) / 256 * 256 : cneg + pad(gpc) * 64; }
  // + 512 bytes that lanes outside the batch may read past the last group, + 1024 alignment slack
  __host__ __device__ static int total(int gpc) { return xs(gpc) + pad(gpc) * xgroup + 512 + 1024; }
};

template <int FMT, bool XBF, int BP>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ Args a) {
  using FT = FmtTraits<FMT>;
  using L = Layout<FMT, BP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (lbdev::smem_u32(smem_raw) & 1023u)) & 1023u);   // 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::bars);
  uint64_t* empty = full + L::stages;
  uint64_t* xbar = full + 15;                                    // K split: this CTA's exchange has landed

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  LB_TRACE(threadIdx.x == 0, 0);
#ifdef LB_GEMV_TRACE
  if (threadIdx.x == 0 && blockIdx.y * gridDim.x + blockIdx.x < kTraceCtas) {   // which launch wrote the CTA's events
    g_gemv_trace[blockIdx.y * gridDim.x + blockIdx.x][kTraceEvents - 1][0] = gridDim.x;
    g_gemv_trace[blockIdx.y * gridDim.x + blockIdx.x][kTraceEvents - 1][1] = gridDim.y;
  }
#endif
  int pi = 0;                                                    // this CTA's problem
  for (int i = 1; i < a.count && !a.fuse; ++i)
    if (static_cast<int>(blockIdx.y) >= a.p[i].unit0) pi = i;
  const Prob& P = a.p[pi];
  const uint32_t rank = a.S > 1 ? cluster_rank() : 0u;
  const int gpc = P.gpc;
  const int g_begin = static_cast<int>(rank) * gpc;
  const int ng = min(gpc, P.G - g_begin);                        // groups of this CTA's chunk (<= 0: none)
  const int nst = (ng + GS - 1) / GS;                            // stages per row block
  // Units (row blocks) of this CTA, j = 0, 1, ...: one GEMV with persistent CTAs takes row blocks
  // rb0, rb0 + gridDim.y, ...; a grouped launch whose problems share x and K (a.shared) takes units
  // blockIdx.y, blockIdx.y + gridDim.y, ... of the whole unit list, whichever problem they belong
  // to; any other grouped launch takes exactly its one unit; a fused SiLU-gated pair runs row
  // block rb0 twice, unit 0 on the gate matrix and unit 1 on the up matrix.
  const int rb0 = static_cast<int>(blockIdx.y) - P.unit0;
  const int my_rbs = a.fuse ? 2
                     : a.shared ? (a.units - static_cast<int>(blockIdx.y) + gridDim.y - 1) / gridDim.y
                     : a.count > 1 ? 1
                     : (P.row_blocks - rb0 + gridDim.y - 1) / gridDim.y;
  auto unit_prob = [&](int j) -> int {
    if (a.fuse) return j;
    if (!a.shared) return pi;
    const int u = static_cast<int>(blockIdx.y) + j * static_cast<int>(gridDim.y);
    int q = 0;
    for (int i = 1; i < a.count; ++i)
      if (u >= a.p[i].unit0) q = i;
    return q;
  };
  auto unit_rb = [&](int j) -> int {
    if (a.fuse || (a.count > 1 && !a.shared)) return rb0;
    if (!a.shared) return rb0 + j * static_cast<int>(gridDim.y);
    const int u = static_cast<int>(blockIdx.y) + j * static_cast<int>(gridDim.y);
    return u - a.p[unit_prob(j)].unit0;
  };
  const int total_st = my_rbs * nst;
  bool ok = true;

  // Start-up without a block-wide barrier: the producer warp initialises the pipeline and exchange
  // barriers itself and starts copying at once, then publishes the barriers on named barrier
  // kBarInit; the consumers zero the column maxima among themselves and wait on kBarInit just
  // before griddepcontrol.wait, so that inside a launch chain the wait is hidden behind the
  // previous kernel.  (With a block barrier first, a traced small launch issued its first copy
  // ~2.9 kcyc after the start and its consumers then waited ~1.4 kcyc for it.)  K split: every
  // thread also arrives on the cluster barrier after this, and the consumers wait on it before
  // their first stage, so that no CTA's exchange barrier is used before it is initialised (by then
  // it has long completed).  The producer's tensor-map prefetches come first, so that the
  // descriptor fetches overlap the barrier set-up, and its cluster arrival is relaxed (the init
  // fence already released the barriers; a releasing arrival held the producer ~0.7-1.0 kcyc
  // before its first copy in traced 3-CTA-cluster launches).
  if (warp == NW) {
    if (lane == 0)
      for (int i = 0; i < a.count; ++i)
        if (i == pi || a.fuse || a.shared) {
          lbdev::prefetch_tmap(&a.p[i].tm_codes);
          if (P.scales_tma) lbdev::prefetch_tmap(&a.p[i].tm_scales);
        }
    if (lane == 0) {
      for (int s = 0; s < L::stages; ++s) {
        lbdev::mbar_init(&full[s], P.scales_tma ? 1 : 32);       // 32: the lanes store the scales
        lbdev::mbar_init(&empty[s], NW);
      }
      lbdev::mbar_init(xbar, 1);
      lbdev::fence_mbar_init();
      LB_TRACE(true, 31);
    }
    __syncwarp();
    asm volatile("bar.arrive %0, %1;" ::"n"(kBarInit), "n"((NW + 1) * 32) : "memory");
    if (a.S > 1) cluster_arrive_relaxed();
    LB_TRACE(lane == 0, 32);
  } else {
    if (threadIdx.x < 8) reinterpret_cast<uint32_t*>(sm + L::colf)[8 + threadIdx.x] = 0u;   // column maxima
    consumer_sync();
    if (a.S > 1) cluster_arrive();
  }

  if (warp == NW) {
    // ======================= producer: weights do not depend on earlier kernels, so no wait.
    // Codes (and scales, when a scale row is a multiple of 16 bytes) arrive by TMA; otherwise the
    // 32 lanes load the stage's scales from global memory, store them in the slot in the TMA
    // box's layout and arrive on the stage's barrier themselves.
    const bool stma = P.scales_tma != 0;
    LB_TRACE(lane == 0, 33);
    const uint32_t bytes = static_cast<uint32_t>(FT::nb * FT::box + (stma ? kScaleBox : 0));
    if (stma ? lane == 0 : true) {
      for (int st = 0; st < total_st && !a.test_fault; ++st) {
        const int s = st % L::stages;
        if (!lbdev::mbar_wait_backoff(&empty[s], static_cast<uint32_t>(((st / L::stages) & 1) ^ 1), a.wait_ns)) {
          ok = false;
          break;
        }
        LB_TRACE(lane == 0 && st == 0, 34);
        const int row0 = unit_rb(st / nst) * ROWS;
        const Prob& PU = a.p[unit_prob(st / nst)];                 // the matrix of this unit
        const int g0 = g_begin + (st % nst) * GS;
        uint8_t* slot = sm + s * L::slot;
        if (!stma) {
          // rows row0 + lane + 32i, groups g0 .. g0 + 7; zero outside the matrix, as TMA fills
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = row0 + lane + 32 * i;
            uint32_t v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int g = g0 + 2 * j;
              const uint16_t* src = PU.scales + static_cast<int64_t>(row) * PU.G + g;
              const uint32_t lo = (row < PU.n && g < PU.G) ? __ldg(src) : 0u;
              const uint32_t hi = (row < PU.n && g + 1 < PU.G) ? __ldg(src + 1) : 0u;
              v[j] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4*>(slot + FT::nb * FT::box + (lane + 32 * i) * 16) = make_uint4(v[0], v[1], v[2], v[3]);
          }
          if (lane != 0) lbdev::mbar_arrive(&full[s]);
        }
        if (lane == 0) {
          lbdev::mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
          for (int b = 0; b < FT::nb; ++b)
            lbdev::tma_load_2d(slot + b * FT::box, &PU.tm_codes, (g0 + b * (GS / FT::nb)) * FT::gbytes, row0, &full[s]);
          if (stma) lbdev::tma_load_2d(slot + FT::nb * FT::box, &PU.tm_scales, g0, row0, &full[s]);
          LB_TRACE(st == 0, 1);
          LB_TRACE(st == total_st - 1, 2);
        }
      }
    }
    __syncwarp();
    griddep_launch();
  } else if constexpr (L::LU) {
    // ======================= consumers, lookup-table form (batch 1; 1-bit, and ternary five per
    // byte, whose tables are described at the build below).  1-bit: per chunk of four
    // activations the table holds the 16 signed sums sum_i (b_i ? +x_i : -x_i) (FP32, in the
    // chunk's 64 bytes), so a code nibble b_0..b_3 costs one lookup and one add: thread = weight row,
    // warp = 32 rows x 2 of a stage's 8 groups; four warps share rows and add up at the row block's
    // end.  bfloat16 x is scaled by the same exact power of two as the fragment form (column max in
    // [2^15, 2^16)) and the result scaled back.
    float* colf = reinterpret_cast<float*>(sm + L::colf);
    float* tab = reinterpret_cast<float*>(sm + L::xs(gpc));
    asm volatile("bar.sync %0, %1;" ::"n"(kBarInit), "n"((NW + 1) * 32) : "memory");   // the producer's barriers
    griddep_wait();                                   // x is read and y written only after this
    LB_TRACE(threadIdx.x == 0, 3);
    const int chunks = ng > 0 ? ng * 32 : 0;
    const uint16_t* xrow = P.x + static_cast<int64_t>(g_begin) * 128;
    // item t = (chunk c, quarter h): the four entries 4h .. 4h + 3 of chunk c, so that a warp's
    // 16-byte stores are contiguous (no bank conflicts).  The entries are FP32 sums of the exact
    // activations, built in one pass; bfloat16 columns whose largest magnitude is 2^100 or more
    // (where sums of four could overflow) are built again scaled down by a power of two.
    const int items = L::pad(ng > 0 ? ng : 0) * 128;
    auto bf_exp = [](uint32_t u) { return u & 0x7f800000u; };     // a bfloat16 pattern's exponent field
    auto build = [&](float scale) -> uint32_t {
      uint32_t mx = 0;
      if constexpr (FMT == 3) {
        // five per byte: byte j of a group holds digits d0..d4 (weights 5j .. 5j+4); slot j of the
        // group's table (144 bytes, at (26 g + j) * 144) holds A[d0 + 3 d1] = (d0 - 1) x_5j +
        // (d1 - 1) x_5j+1 (9 floats) and then B[d2 + 3 d3 + 9 d4] = sum (d - 1) x over weights
        // 5j+2 .. 5j+4 (27 floats); weights past 127 (byte 25) count as x = 0.  A thread builds
        // whole slots: it loads the slot's five activations (the loads of all its slots issued
        // together), forms the 36 sums in registers and writes them as nine 16-byte stores
        // (slots 144 bytes apart: no bank conflicts).
        const int slots = L::pad(ng > 0 ? ng : 0) * 26;
        constexpr int kS = 3;                                      // 3 x 512 >= 26 x 40 slots
        for (int t0 = threadIdx.x; t0 < slots; t0 += kS * NW * 32) {
          uint32_t raw[kS][5];
#pragma unroll
          for (int u = 0; u < kS; ++u) {
            const int it = t0 + u * NW * 32;
            const int g = it / 26, j = it - g * 26;
#pragma unroll
            for (int q = 0; q < 5; ++q) {
              const int kk = 5 * j + q;
              raw[u][q] = (it < slots && kk < 128 && g < ng) ? static_cast<uint32_t>(__ldg(xrow + g * 128 + kk)) : 0u;
            }
          }
#pragma unroll
          for (int u = 0; u < kS; ++u) {
            const int it = t0 + u * NW * 32;
            if (it >= slots) break;
            float v[5];
#pragma unroll
            for (int q = 0; q < 5; ++q) {
              if (XBF) {
                mx = max(mx, bf_exp(raw[u][q] << 16));
                v[q] = __uint_as_float(raw[u][q] << 16) * scale;
              } else {
                v[q] = __half2float(__ushort_as_half(static_cast<unsigned short>(raw[u][q])));
              }
            }
            float e36[36];
#pragma unroll
            for (int e = 0; e < 9; ++e) {
              e36[e] = (e % 3 - 1) * v[0] + (e / 3 - 1) * v[1];
              const float p23 = (e % 3 - 1) * v[2] + (e / 3 - 1) * v[3];
#pragma unroll
              for (int d4 = 0; d4 < 3; ++d4) e36[9 + e + 9 * d4] = p23 + (d4 - 1) * v[4];
            }
            float4* dst = reinterpret_cast<float4*>(tab + 36 * it);
#pragma unroll
            for (int c = 0; c < 9; ++c)
              dst[c] = make_float4(e36[4 * c], e36[4 * c + 1], e36[4 * c + 2], e36[4 * c + 3]);
          }
        }
      } else {
#pragma unroll 4
      for (int t = threadIdx.x; t < items; t += NW * 32) {
        const int c = t >> 2, h = t & 3;
        float v[4] = {0.f, 0.f, 0.f, 0.f};                        // padding chunks: all-zero sums
        if (c < chunks) {
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(xrow) + c);
          if (XBF) {
            mx = max(mx, max(max((u.x << 16) & 0x7f800000u, u.x & 0x7f800000u),
                             max((u.y << 16) & 0x7f800000u, u.y & 0x7f800000u)));
            v[0] = __uint_as_float(u.x << 16) * scale; v[1] = __uint_as_float(u.x & 0xffff0000u) * scale;
            v[2] = __uint_as_float(u.y << 16) * scale; v[3] = __uint_as_float(u.y & 0xffff0000u) * scale;
          } else {
            const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
            const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
            v[0] = lo.x; v[1] = lo.y; v[2] = hi.x; v[3] = hi.y;
          }
        }
        const float lo4[4] = {-v[0] - v[1], v[0] - v[1], v[1] - v[0], v[0] + v[1]};   // bits 0, 1
        const float hi = ((h & 1) ? v[2] : -v[2]) + ((h & 2) ? v[3] : -v[3]);         // bits 2, 3 = h
        reinterpret_cast<float4*>(tab)[t] = make_float4(lo4[0] + hi, lo4[1] + hi, lo4[2] + hi, lo4[3] + hi);
      }
      }
      return mx;
    };
    uint32_t mx = build(1.f);
    if (XBF) {
      for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) atomicMax(reinterpret_cast<uint32_t*>(colf + 8), mx);
    }
    consumer_sync();
    const int e = XBF ? static_cast<int>(reinterpret_cast<uint32_t*>(colf + 8)[0] >> 23) - 127 : 0;
    if (e >= 100) {                                                 // block-uniform
      const int p = 99 - e;                                         // largest magnitude below 2^100
      build(__uint_as_float(static_cast<uint32_t>(127 + p) << 23));
      if (threadIdx.x == 0) colf[0] = __uint_as_float(static_cast<uint32_t>(127 - p) << 23);
      consumer_sync();
    } else if (threadIdx.x == 0) {
      colf[0] = 1.f;
    }
    consumer_sync();
    LB_TRACE(threadIdx.x == 0, 4);
    if (a.S > 1) cluster_wait();                                   // every exchange barrier is initialised

    const int rq = warp & 3, kq = warp >> 2;                      // rows 32 rq .., groups 2 kq, 2 kq + 1
    const int row_l = 32 * rq + lane;
    const uint32_t sm32 = lbdev::smem_u32(sm);
    const uint32_t tb = sm32 + static_cast<uint32_t>(L::xs(gpc));   // 256-byte aligned
    const uint32_t code0 = static_cast<uint32_t>(row_l * 128 + (((2 * kq) ^ (row_l & 7)) << 4));   // 1-bit
    const uint32_t code1 = static_cast<uint32_t>(row_l * 128 + (((2 * kq + 1) ^ (row_l & 7)) << 4));
    const uint32_t sc_off = static_cast<uint32_t>(FT::nb * FT::box + row_l * 16 + 4 * kq);
    float acc = 0.f;
    int s = 0, st = 0;
    uint32_t ph = 0;
    for (int i_rb = 0; i_rb < my_rbs; ++i_rb) {
      for (int cstage = 0; cstage < nst; ++cstage, ++st) {
        const uint32_t slot = sm32 + static_cast<uint32_t>(s * L::slot);
        if (ok && !lbdev::mbar_wait(&full[s], ph, a.wait_ns)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        LB_TRACE(threadIdx.x == 0 && st < 16, 5 + st);
        uint4 w[2];
        uint32_t c13[13];                                          // five per byte: my 52 code bytes
        uint32_t sc2 = 0;
        if (ok) {
          if constexpr (FMT == 3) {
            // the row's 208 bytes of the stage (13 x 16 bytes: a warp's 16-byte loads hit every
            // bank once per quarter), my two groups at byte 52 kq: four 16-byte loads from the
            // 16-byte boundary below, then a shift by 52 kq mod 16 = 4 kq bytes (warp-uniform)
            uint32_t w16[16];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 v = ldsv128(slot + static_cast<uint32_t>(row_l * 208 + ((52 * kq) & ~15) + 16 * c));
              w16[4 * c] = v.x; w16[4 * c + 1] = v.y; w16[4 * c + 2] = v.z; w16[4 * c + 3] = v.w;
            }
            uint32_t t15[15];
#pragma unroll
            for (int i = 0; i < 15; ++i) t15[i] = (kq & 1) ? w16[i + 1] : w16[i];
#pragma unroll
            for (int i = 0; i < 13; ++i) c13[i] = (kq & 2) ? t15[i + 2] : t15[i];
          } else {
            w[0] = ldsv128(slot + code0);
            w[1] = ldsv128(slot + code1);
          }
          sc2 = ldsv32(slot + sc_off);
        }
        __syncwarp();
        if (lane == 0) lbdev::mbar_arrive(&empty[s]);             // slot s released by this warp
        if (++s == L::stages) { s = 0; ph ^= 1u; }
        if (FMT == 3 && ok && cstage * GS + 2 * kq < ng) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // byte b = sum d_i 3^i: b mod 9 indexes A (two weights), b / 9 = (57 b) >> 9 (exact for
            // b <= 242) indexes B (three weights) of the byte's table slot (144 bytes)
            const uint32_t base = tb + static_cast<uint32_t>((cstage * GS + 2 * kq + h) * (26 * 36 * 4));
            float p4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 26; ++j) {
              const int kb = 26 * h + j;
              const uint32_t b = __byte_perm(c13[kb >> 2], 0u, 0x4440u | static_cast<uint32_t>(kb & 3));
              const uint32_t q = (b * 57u) >> 9;
              const uint32_t r = b - 9u * q;
              float ta, tbv;
              asm("ld.shared.f32 %0, [%1];" : "=f"(ta) : "r"(base + static_cast<uint32_t>(j * 144) + 4u * r));
              asm("ld.shared.f32 %0, [%1];" : "=f"(tbv) : "r"(base + static_cast<uint32_t>(j * 144 + 36) + 4u * q));
              p4[j & 3] += ta + tbv;
            }
            const float sg = __half2float(__ushort_as_half(static_cast<unsigned short>(sc2 >> (16 * h))));
            acc = fmaf(sg, (p4[0] + p4[1]) + (p4[2] + p4[3]), acc);
          }
        }
        if (FMT == 1 && ok && cstage * GS + 2 * kq < ng) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // the chunk of nibble j of word u is 8u + j of the group: low byte (j % 4) * 64 + 4 * idx,
            // (j / 4) * 256 and u * 512 as offsets from the group's 2 KB
            const uint32_t base = tb + static_cast<uint32_t>((cstage * GS + 2 * kq + h) * 2048);
            float p4[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t wd[4] = {w[h].x, w[h].y, w[h].z, w[h].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint32_t ev, od;
              asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(ev) : "r"(wd[u] << 2), "r"(0x3C3C3C3Cu), "r"(0x80008000u));
              asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(od) : "r"(wd[u] >> 2), "r"(0x3C3C3C3Cu), "r"(0xC040C040u));
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const uint32_t ad = __byte_perm((j & 1) ? od : ev, base, 0x7650 | (j >> 1));
                float t;
                asm("ld.shared.f32 %0, [%1];" : "=f"(t) : "r"(ad + u * 512 + (j >> 2) * 256));
                p4[j & 3] += t;
              }
            }
            const float sg = __half2float(__ushort_as_half(static_cast<unsigned short>(sc2 >> (16 * h))));
            acc = fmaf(sg, (p4[0] + p4[1]) + (p4[2] + p4[3]), acc);
          }
        }
      }
      // ---- row block done: the four K quarters of each row meet in shared memory
      const int rb = unit_rb(i_rb);
      const Prob& PU = a.p[unit_prob(i_rb)];
      float* red = reinterpret_cast<float*>(sm + L::red) + (i_rb & 1) * ROWS * 8;
      if (kq != 0) red[kq * ROWS + row_l] = acc;
      if (i_rb == my_rbs - 1) griddep_launch();
      asm volatile("bar.sync %0, 128;" ::"r"(2 + rq) : "memory");
      if (kq == 0) {
        const float v = (acc + red[ROWS + row_l] + red[2 * ROWS + row_l] + red[3 * ROWS + row_l]) * colf[0];
        float* gate = reinterpret_cast<float*>(sm + L::red);      // the gate unit's outputs (fused pair)
        if (a.S == 1 && a.fuse && i_rb == 0) {
          gate[row_l] = v;
        } else if (a.S == 1) {
          const int row = rb * ROWS + row_l;
          const float o = a.fuse ? v * silu(gate[row_l]) : v;
          if (row < PU.n)
            PU.y[row] = XBF ? __bfloat16_as_ushort(__float2bfloat16_rn(o)) : __half_as_ushort(__float2half_rn(o));
        } else {
          const int per = (ROWS + a.S - 1) / a.S;
          const int o = row_l / per;
          const int slot_i = ((i_rb * a.S + static_cast<int>(rank)) * per + (row_l - o * per)) * 8;
          st_async_f32(sm32 + static_cast<uint32_t>(L::xchg + slot_i * 4), lbdev::smem_u32(xbar), static_cast<uint32_t>(o), v);
        }
      }
      acc = 0.f;
      LB_TRACE(threadIdx.x == 0 && i_rb < 8, 21 + i_rb);
    }
    LB_TRACE(threadIdx.x == 0, 29);
  } else {
    // ======================= consumers
    const int r = lane >> 2, q = lane & 3;
    const int tile = warp & (NT - 1), half = warp / NT;
    float* colf = reinterpret_cast<float*>(sm + L::colf);            // [8] factors, then [8] maxima
    float* cneg = reinterpret_cast<float*>(sm + L::cneg);            // [gpc][4][4]
    uint8_t* xs = sm + L::xs(gpc);
    asm volatile("bar.sync %0, %1;" ::"n"(kBarInit), "n"((NW + 1) * 32) : "memory");   // the producer's barriers
    griddep_wait();                                   // x is read and y written only after this
    LB_TRACE(threadIdx.x == 0, 3);

    // ---- x prologue.  Tuple (g, n, qq): the 32 activations x[n][128(g_begin+g) + 32qq ..] of one
    // fragment lane.  bfloat16 columns are scaled by an exact power of two 2^p that puts the
    // column's largest magnitude in [2^15, 2^16) (|p| <= 126) and converted to binary16: every
    // element within 2^32 of the column maximum is then exact (8 significant bits fit binary16 down
    // to 2^-17), smaller ones round to the binary16 subnormal grid, nothing overflows, and the FP32
    // result is scaled back by 2^-p.  A thread's first tuple stays in registers between the two
    // passes, so the common case reads x from memory once.
    const int tuples = ng * BP * 4;
    auto load32 = [&](int t, uint32_t (&X)[16]) -> bool {
      const int qq = t & 3, n = (t >> 2) % BP, g = (t >> 2) / BP;
      if (t >= tuples || n >= a.batch) {
#pragma unroll
        for (int i = 0; i < 16; ++i) X[i] = 0u;
        return false;
      }
      const uint4* src = reinterpret_cast<const uint4*>(P.x + static_cast<int64_t>(n) * P.k +
                                                        static_cast<int64_t>(g_begin + g) * 128 + 32 * qq);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(src + i);
        X[4 * i] = v.x; X[4 * i + 1] = v.y; X[4 * i + 2] = v.z; X[4 * i + 3] = v.w;
      }
      return true;
    };
    uint32_t X0[16];
    const bool act0 = load32(static_cast<int>(threadIdx.x), X0);
    if (XBF) {
      uint32_t* cmax = reinterpret_cast<uint32_t*>(colf + 8);
      uint32_t mx = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) mx = max(mx, max((X0[i] << 16) & 0x7f800000u, X0[i] & 0x7f800000u));
      if (act0) atomicMax(&cmax[(threadIdx.x >> 2) % BP], mx);      // exponent fields order like magnitudes
      for (int base = NW * 32; base < tuples; base += NW * 32) {
        const int t = base + static_cast<int>(threadIdx.x);
        uint32_t X[16];
        if (load32(t, X)) {
          mx = 0;
#pragma unroll
          for (int i = 0; i < 16; ++i) mx = max(mx, max((X[i] << 16) & 0x7f800000u, X[i] & 0x7f800000u));
          atomicMax(&cmax[(t >> 2) % BP], mx);
        }
      }
      consumer_sync();
    }
    auto col_p = [&](int n) -> int {                               // the column's exponent p
      const int e = static_cast<int>(reinterpret_cast<uint32_t*>(colf + 8)[n] >> 23) - 127;   // -127: zero
      return max(-126, min(126, 15 - e));
    };
    if (threadIdx.x < 8)                                           // 2^-p (1 for binary16 columns)
      colf[threadIdx.x] = XBF ? __uint_as_float(static_cast<uint32_t>(127 - col_p(threadIdx.x)) << 23) : 1.f;
    for (int base = 0; base < tuples; base += NW * 32) {          // uniform: quads stay together
      const int t = base + static_cast<int>(threadIdx.x);
      const int qq = t & 3, n = (t >> 2) % BP, g = (t >> 2) / BP;
      uint32_t X[16];
      bool act;
      if (base == 0) {
        act = act0;
#pragma unroll
        for (int i = 0; i < 16; ++i) X[i] = X0[i];
      } else {
        act = load32(t, X);
      }
      if (XBF && act) {
        const float scale = __uint_as_float(static_cast<uint32_t>(127 + col_p(n)) << 23);   // 2^p (exact)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float lo = __uint_as_float(X[i] << 16) * scale, hi = __uint_as_float(X[i] & 0xffff0000u) * scale;
          const __half2 h2 = __floats2half2_rn(lo, hi);
          X[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
      uint32_t B[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        uint32_t lo_src, hi_src, sel;
        if (FMT == 1) {
          lo_src = X[i >> 1]; hi_src = X[(i >> 1) + 8]; sel = (i & 1) ? 0x7632 : 0x5410;
        } else {
          const int uu = i >> 3, p = i & 7;
          lo_src = X[8 * uu + (p >> 1)]; hi_src = X[8 * uu + (p >> 1) + 4]; sel = (p & 1) ? 0x7632 : 0x5410;
        }
        B[i] = __byte_perm(lo_src, hi_src, sel);
      }
      float c = 0.f;
      if (FMT == 1) {
        // 1-bit baseline sum_k (o_k + 1/2) x_k: the activations of each offset are summed first
        // (no large multiplier inside), then one product per offset
#pragma unroll
        for (int m = 4; m <= 9; ++m) {
          float sx = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (pos1(i) == m) {
              const float2 fv = __half22float2(*reinterpret_cast<const __half2*>(&B[i]));
              sx += fv.x + fv.y;
            }
          c = fmaf(static_cast<float>(1 << (10 - m)) + 0.5f, sx, c);
        }
        c += __shfl_xor_sync(0xffffffffu, c, 1);
        c += __shfl_xor_sync(0xffffffffu, c, 2);
      }
      if (t < tuples) {
        uint8_t* dst = xs + g * L::xgroup + (n * 4 + qq) * 16;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(dst + i * (L::xgroup / 4)) = make_uint4(B[4 * i], B[4 * i + 1], B[4 * i + 2], B[4 * i + 3]);
        if (FMT == 1 && qq == 0) {
          const float v = act ? -c : 0.f;
          cneg[g * 16 + (n >> 1) * 4 + (n & 1)] = v;
          cneg[g * 16 + (n >> 1) * 4 + 2 + (n & 1)] = v;
        }
      }
    }
    if (FMT == 1) {
      // columns beyond the padded batch, and every column of the groups that pad the last stage
      for (int i = threadIdx.x; i < L::pad(ng) * 16; i += NW * 32)
        if (i >= ng * 16 || ((i >> 2) & 3) * 2 + (i & 1) >= BP) cneg[i] = 0.f;
    }
    for (int i = ng * (L::xgroup / 16) + threadIdx.x; i < L::pad(ng) * (L::xgroup / 16); i += NW * 32)
      reinterpret_cast<uint4*>(xs)[i] = make_uint4(0u, 0u, 0u, 0u);  // x of the padding groups: zero
    consumer_sync();
    LB_TRACE(threadIdx.x == 0, 4);
    if (a.S > 1) cluster_wait();                                   // every exchange barrier is initialised

    uint32_t tok;                                      // orders the private-region loads after the barrier
    asm volatile("mov.u32 %0, 0;" : "=r"(tok)::"memory");

    // ---- per-thread constants
    uint32_t M[10];                                    // decode masks, kept in registers
    constexpr uint32_t kMask = FMT == 1 ? 0x00010001u : 0x00030003u;
    uint32_t SC[10];                                   // ternary: o + 1 in both halves, by position
#define LB_MASK(m)                                                                                   \
  asm volatile("mov.b32 %0, %1;" : "=r"(M[m]) : "n"(kMask << (m)));                                 \
  asm volatile("mov.b32 %0, %1;" : "=r"(SC[m]) : "n"(expo16(m) | (0x00010001u << (m))))
    LB_MASK(0); LB_MASK(1); LB_MASK(2); LB_MASK(3); LB_MASK(4);
    LB_MASK(5); LB_MASK(6); LB_MASK(7); LB_MASK(8); LB_MASK(9);
#undef LB_MASK
    const int ia = tile * 16 + r;                                  // rows ia and ia + 8 of the block
    uint32_t pcode;                                                // this lane's words, first group of my half
    if (FMT == 1) {
      pcode = static_cast<uint32_t>(ia * 128) | (4u * q) | (static_cast<uint32_t>(r) << 4);
      pcode ^= static_cast<uint32_t>(half * GH) << 4;
    } else {
      pcode = static_cast<uint32_t>(ia * 128) | (8u * (q & 1)) | (static_cast<uint32_t>((q >> 1) ^ r) << 4);
      pcode += static_cast<uint32_t>(half * kBox);                 // ternary: one box per half
    }
    uint32_t pc[GH];                                               // my words of group j of a stage
#pragma unroll
    for (int j = 0; j < GH; ++j) pc[j] = pcode ^ (static_cast<uint32_t>(j) << (FMT == 1 ? 4 : 5));
    const uint32_t sm32 = lbdev::smem_u32(sm);
    const uint32_t xs_lane = sm32 + static_cast<uint32_t>(L::xs(gpc)) + lane * 16 + tok;
    const uint32_t cn_q = sm32 + static_cast<uint32_t>(L::cneg) + 16 * q + tok;
    const uint32_t sc_off = static_cast<uint32_t>(FT::nb * FT::box + ia * 16 + half * 8);
    const float mul = FMT == 1 ? 2.f : 1.f;
    const int c0col = 2 * q, c1col = 2 * q + 1;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int s = 0, st = 0;
    uint32_t ph = 0;

    // units (row blocks) of this CTA; per unit nst stages of the ring, then the unit's epilogue
    for (int i_rb = 0; i_rb < my_rbs; ++i_rb) {
     for (int cstage = 0; cstage < nst; ++cstage, ++st) {
      const int g0 = cstage * GS + half * GH;                     // my first group, relative to g_begin
      const int cnt = min(GH, ng - g0);                           // my groups in this stage (may be <= 0)
      const uint32_t slot = sm32 + static_cast<uint32_t>(s * L::slot);
      float sa[GH], sb[GH];
      if (ok && !lbdev::mbar_wait(&full[s], ph, a.wait_ns)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      LB_TRACE(threadIdx.x == 0 && st < 16, 5 + st);
      // ---- the stage's codes and scales -> registers, then the slot goes back to the producer
      uint2 ca[GH], cb[GH];                                        // rows ia / ia + 8, my 4 groups
      if (ok) {
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
        {
          const uint2 va = ldsv64(slot + sc_off), vb = ldsv64(slot + sc_off + 128);
          const float2 a01 = __half22float2(*reinterpret_cast<const __half2*>(&va.x));
          const float2 a23 = __half22float2(*reinterpret_cast<const __half2*>(&va.y));
          const float2 b01 = __half22float2(*reinterpret_cast<const __half2*>(&vb.x));
          const float2 b23 = __half22float2(*reinterpret_cast<const __half2*>(&vb.y));
          sa[0] = a01.x; sa[1] = a01.y; sa[2] = a23.x; sa[3] = a23.y;
          sb[0] = b01.x; sb[1] = b01.y; sb[2] = b23.x; sb[3] = b23.y;
        }
      }
      __syncwarp();
      if (lane == 0) lbdev::mbar_arrive(&empty[s]);               // slot s released by this warp
      if (++s == L::stages) { s = 0; ph ^= 1u; }

      if (ok && cnt > 0) {                                        // cnt <= 0: a half with no groups
        const uint32_t xbase = xs_lane + static_cast<uint32_t>(g0 * L::xgroup);
        const uint32_t cbase = cn_q + static_cast<uint32_t>(g0 * 64);
        {
          // a stage is always full (codes and scales past the end of K arrive as zeros, and the x
          // of the padding groups is zero): two pairs of groups, two accumulator chains per pair
#pragma unroll
          for (int jp = 0; jp < GH; jp += 2) {
            Word1 w1a0 = prep1(ca[jp].x), w1b0 = prep1(cb[jp].x), w1a1 = prep1(ca[jp + 1].x), w1b1 = prep1(cb[jp + 1].x);
            Word2 la0 = prep2(ca[jp].x), ha0 = prep2(ca[jp].y), lb0 = prep2(cb[jp].x), hb0 = prep2(cb[jp].y);
            Word2 la1 = prep2(ca[jp + 1].x), ha1 = prep2(ca[jp + 1].y), lb1 = prep2(cb[jp + 1].x), hb1 = prep2(cb[jp + 1].y);
            float4 cn0, cn1;                                      // 1-bit baselines (ternary: unused)
            if (FMT == 1) {
              cn0 = lds128f(cbase + jp * 64);
              cn1 = lds128f(cbase + (jp + 1) * 64);
            }
            uint4 bx0[4], bx1[4];
#pragma unroll
            for (int iq = 0; iq < 4; ++iq) {
              bx0[iq] = lds128(xbase + jp * L::xgroup + iq * (L::xgroup / 4));
              bx1[iq] = lds128(xbase + (jp + 1) * L::xgroup + iq * (L::xgroup / 4));
            }
            float d0[4], d1[4];
#define LB_PAIR(I)                                                                                         \
  {                                                                                                        \
    const uint32_t b0lo = (I) % 2 == 0 ? bx0[(I) / 2].x : bx0[(I) / 2].z;                                   \
    const uint32_t b0hi = (I) % 2 == 0 ? bx0[(I) / 2].y : bx0[(I) / 2].w;                                   \
    const uint32_t b1lo = (I) % 2 == 0 ? bx1[(I) / 2].x : bx1[(I) / 2].z;                                   \
    const uint32_t b1hi = (I) % 2 == 0 ? bx1[(I) / 2].y : bx1[(I) / 2].w;                                   \
    const uint32_t e00 = areg<FMT, 2 * (I)>(w1a0, la0, ha0, M, SC), e01 = areg<FMT, 2 * (I)>(w1b0, lb0, hb0, M, SC);  \
    const uint32_t e02 = areg<FMT, 2 * (I) + 1>(w1a0, la0, ha0, M, SC);                                         \
    const uint32_t e03 = areg<FMT, 2 * (I) + 1>(w1b0, lb0, hb0, M, SC);                                         \
    const uint32_t e10 = areg<FMT, 2 * (I)>(w1a1, la1, ha1, M, SC), e11 = areg<FMT, 2 * (I)>(w1b1, lb1, hb1, M, SC);  \
    const uint32_t e12 = areg<FMT, 2 * (I) + 1>(w1a1, la1, ha1, M, SC);                                         \
    const uint32_t e13 = areg<FMT, 2 * (I) + 1>(w1b1, lb1, hb1, M, SC);                                         \
    if ((I) == 0 && FMT == 1) {                                                                            \
      mma_c4(d0, e00, e01, e02, e03, b0lo, b0hi, cn0);                                                     \
      mma_c4(d1, e10, e11, e12, e13, b1lo, b1hi, cn1);                                                     \
    } else if ((I) == 0) {                                                                                 \
      mma_zero(d0, e00, e01, e02, e03, b0lo, b0hi);                                                        \
      mma_zero(d1, e10, e11, e12, e13, b1lo, b1hi);                                                        \
    } else {                                                                                               \
      mma_acc(d0, e00, e01, e02, e03, b0lo, b0hi);                                                         \
      mma_acc(d1, e10, e11, e12, e13, b1lo, b1hi);                                                         \
    }                                                                                                      \
  }
            LB_PAIR(0) LB_PAIR(1) LB_PAIR(2) LB_PAIR(3) LB_PAIR(4) LB_PAIR(5) LB_PAIR(6) LB_PAIR(7)
#undef LB_PAIR
            acc[0] = fmaf(sa[jp], d0[0], acc[0]);
            acc[1] = fmaf(sa[jp], d0[1], acc[1]);
            acc[2] = fmaf(sb[jp], d0[2], acc[2]);
            acc[3] = fmaf(sb[jp], d0[3], acc[3]);
            acc[0] = fmaf(sa[jp + 1], d1[0], acc[0]);
            acc[1] = fmaf(sa[jp + 1], d1[1], acc[1]);
            acc[2] = fmaf(sb[jp + 1], d1[2], acc[2]);
            acc[3] = fmaf(sb[jp + 1], d1[3], acc[3]);
          }
        }
      }

     }
      {
        // ---- row block done: the two halves of each tile meet in shared memory (double-buffered
        // by row block); only the tile's two warps wait for each other
        const int rb = unit_rb(i_rb);
        const Prob& PU = a.p[unit_prob(i_rb)];                    // the matrix of this unit
        float* red = reinterpret_cast<float*>(sm + L::red) + (i_rb & 1) * ROWS * 8;
        if (half == 1) {
          red[ia * 8 + c0col] = acc[0];
          red[ia * 8 + c1col] = acc[1];
          red[(ia + 8) * 8 + c0col] = acc[2];
          red[(ia + 8) * 8 + c1col] = acc[3];
        }
        if (i_rb == my_rbs - 1) griddep_launch();
        tile_sync(tile);
        if (half == 0) {
          const float f0 = colf[c0col] * mul, f1 = colf[c1col] * mul;   // output factors of my columns
          const float v0 = (acc[0] + red[ia * 8 + c0col]) * f0;
          const float v1 = (acc[1] + red[ia * 8 + c1col]) * f1;
          const float v2 = (acc[2] + red[(ia + 8) * 8 + c0col]) * f0;
          const float v3 = (acc[3] + red[(ia + 8) * 8 + c1col]) * f1;
          if (a.S == 1 && a.fuse && i_rb == 0) {
            // the gate unit: its outputs wait in the first reduction buffer (which the up unit,
            // using the second, leaves alone) where this thread reads them back
            red[ia * 8 + c0col] = v0;
            red[ia * 8 + c1col] = v1;
            red[(ia + 8) * 8 + c0col] = v2;
            red[(ia + 8) * 8 + c1col] = v3;
          } else if (a.S == 1) {
            const int row_a = rb * ROWS + ia, row_b = row_a + 8;
            auto put = [&](int row, int col, float v) {
              if (row < PU.n && col < a.batch)
                PU.y[static_cast<int64_t>(col) * PU.n + row] =
                    XBF ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
            };
            float o0 = v0, o1 = v1, o2 = v2, o3 = v3;
            if (a.fuse) {                                          // the up unit: h = silu(g) * u
              const float* g = reinterpret_cast<const float*>(sm + L::red);
              o0 *= silu(g[ia * 8 + c0col]);
              o1 *= silu(g[ia * 8 + c1col]);
              o2 *= silu(g[(ia + 8) * 8 + c0col]);
              o3 *= silu(g[(ia + 8) * 8 + c1col]);
            }
            put(row_a, c0col, o0);
            put(row_a, c1col, o1);
            put(row_b, c0col, o2);
            put(row_b, c1col, o3);
          } else {
            // this CTA's partial, in output units, goes straight into the shared memory of the
            // cluster CTA that owns the row, counted on that CTA's exchange barrier
            const int per = (ROWS + a.S - 1) / a.S;
            const uint32_t xchg = sm32 + static_cast<uint32_t>(L::xchg);
            const uint32_t xb = lbdev::smem_u32(xbar);
            auto push = [&](int lrow, int col, float v) {
              if (col < a.batch) {
                const int o = lrow / per;
                const int slot_i = ((i_rb * a.S + static_cast<int>(rank)) * per + (lrow - o * per)) * 8 + col;
                st_async_f32(xchg + static_cast<uint32_t>(slot_i * 4), xb, static_cast<uint32_t>(o), v);
              }
            };
            push(ia, c0col, v0);
            push(ia, c1col, v1);
            push(ia + 8, c0col, v2);
            push(ia + 8, c1col, v3);
          }
        }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        LB_TRACE(threadIdx.x == 0 && i_rb < 8, 21 + i_rb);
      }
    }
    LB_TRACE(threadIdx.x == 0, 29);
  }

  if (a.S > 1 && warp < NW) {
    // one or two row blocks per cluster (or one fused pair): every rank pushed its partials of
    // each unit to the rows' owners with remote stores that count their bytes on the owner's
    // exchange barrier (every rank pushes every row it holds, also a rank without groups); each
    // owner expects S x units x its rows x batch x 4 bytes, waits, and sums its rows locally, in
    // rank order.  A CTA leaves only after its own exchange has landed, and no CTA stores into
    // another after that CTA's exchange is complete.  The kernel parameters the owners need are
    // read into registers before the wait.
    int S_r = a.S, batch_r = a.batch, fuse_r = a.fuse, n_r = P.n, nrank = min(a.S, (P.G + gpc - 1) / gpc);
    uint16_t* y_r = P.y;
    int rbs_r[2] = {a.fuse ? rb0 : unit_rb(0), (!a.fuse && my_rbs > 1) ? unit_rb(1) : 0};
    asm volatile("" : "+r"(S_r), "+r"(batch_r), "+r"(fuse_r), "+r"(n_r), "+r"(nrank), "+l"(y_r), "+r"(rbs_r[0]),
                 "+r"(rbs_r[1]));
    const int per = (ROWS + S_r - 1) / S_r;
    const int lo = static_cast<int>(rank) * per, hi = min(ROWS, lo + per);
    if (threadIdx.x == 0)
      lbdev::mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(S_r * (fuse_r ? 2 : my_rbs) * (hi - lo) * batch_r * 4));
    // twice the pipeline's limit: a rank that gave up on its own stages still pushes (zeros) within
    // one limit of its start, so an owner never leaves while a late push is still to come
    if (!lbdev::mbar_wait(xbar, 0, 2 * a.wait_ns)) ok = false;
    if (ok) {
      const float* xchg = reinterpret_cast<const float*>(sm + L::xchg);
      for (int u0 = 0; u0 < (fuse_r ? 1 : my_rbs); ++u0) {       // my_rbs <= 2 when S > 1
        const int rb = u0 == 0 ? rbs_r[0] : rbs_r[1];
        for (int e = threadIdx.x; e < (hi - lo) * batch_r; e += NW * 32) {
          const int lrow = lo + e / batch_r, col = e % batch_r;
          const int row = rb * ROWS + lrow;
          float v = 0.f;
          for (int p = 0; p < nrank; ++p) v += xchg[((u0 * S_r + p) * per + lrow - lo) * 8 + col];
          if (fuse_r) {                                            // v is the gate; the up partials follow
            float u = 0.f;
            for (int p = 0; p < nrank; ++p) u += xchg[((S_r + p) * per + lrow - lo) * 8 + col];
            v = silu(v) * u;
          }
          if (row < n_r)
            y_r[static_cast<int64_t>(col) * n_r + row] =
                XBF ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
        }
      }
    }
  }
  if (!ok) atomicOr(a.err, lb::kErrGemmTimeout);
  LB_TRACE(threadIdx.x == 0, 30);
}

// ----------------------------------------------------------------------------- host side
int pad_batch(int b) { return b <= 1 ? 1 : b <= 2 ? 2 : b <= 4 ? 4 : 8; }

// Weight of one 128-row x 128-column tile against the fixed costs in the split model below (ns):
// the packed bytes at ~40 B/ns (halved for the 1-bit tables), except for the five-per-byte
// tables, whose measured stage period (~3.0 kcyc per 8 groups on B300) is used instead.  (With
// the measured periods for every path, 2048-wide 1-bit GEMVs and the one-launch c2 set chose K
// splits that measured slower.)
template <int FMT, bool LU>
constexpr double group_ns() {
  return (LU && FMT == 3) ? 195.0 : (LU ? 0.5 : 1.0) * 16384.0 * (FmtTraits<FMT>::gbytes + 2) / 128.0 / 40.0;
}

// Split of K across a cluster (S CTAs, chunk of gpc groups) from a simple time model: every CTA
// pays a fixed cost (launch ramp, x prologue, first TMA latency; more with a cluster reduction),
// then runs its row blocks x groups at group_ns each.  A cluster takes one
// row block or two (rpc; the exchange buffer holds two units' partials), which matters when S x
// the row blocks would not fit on the SMs in one wave.
struct Plan {
  int S, gpc, rpc;
};
template <int FMT, int BP>
Plan plan_split(int G, int row_blocks, int sms) {
  using L = Layout<FMT, BP>;
  const double t_group = group_ns<FMT, L::LU>();
  Plan best{0, 0, 1};
  double best_t = 1e30;
  for (int s_try = 1; s_try <= kMaxCluster; ++s_try) {
    const int per = (G + s_try - 1) / s_try;
    const int g_try = s_try == 1 ? G : (per + GS - 1) / GS * GS;
    const int s_eff = (G + g_try - 1) / g_try;
    if (s_eff != s_try) continue;
    if (L::total(g_try) > kSmemMax) continue;
    if (s_eff == 1) {
      const int per_cta = (row_blocks + sms - 1) / sms;
      const double t = 2500.0 + per_cta * g_try * t_group;
      if (t < best_t * 0.999) { best_t = t; best = Plan{1, g_try, 1}; }
      continue;
    }
    const int clusters = max(1, sms / s_eff);
    for (int r = 1; r <= 2; ++r) {
      const int need = (row_blocks + r - 1) / r;
      const int waves = (need + clusters - 1) / clusters;
      const double t = waves * (3000.0 + r * g_try * t_group);
      if (t < best_t * 0.999) { best_t = t; best = Plan{s_eff, g_try, r}; }
    }
  }
  return best;
}

// Tensor maps of a weight depend only on its planes' addresses, its shape and its format, so they
// are encoded once and kept in a small direct-mapped host cache (a hit is checked field by field;
// a miss re-encodes and replaces the entry).
struct MapEntry {
  const uint8_t* codes;
  const uint16_t* scales;
  int64_t n, k;
  int fmt, valid;
  CUtensorMap tm_codes, tm_scales;
};
constexpr int kMapCache = 1024;
MapEntry g_maps[kMapCache];
std::mutex g_maps_mu;

template <int FMT>
lb_status encode_maps(const lb_weight& W, CUtensorMap& tm_codes, CUtensorMap& tm_scales, int scales_tma) {
  const int n = static_cast<int>(W.n), k = static_cast<int>(W.k), G = k / lb::kGroup;
  const int gbytes = FmtTraits<FMT>::gbytes;
  lb::EncodeTiledFn enc = lb::tensor_map_encoder();
  if (!enc) return lb::fail(LB_ERR_CUDA, "lb_gemv: cuTensorMapEncodeTiled unavailable");
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k) * gbytes / 128, static_cast<cuuint64_t>(n)};
    const cuuint64_t strides[1] = {dims[0]};
    // 2-bit / 1-bit: 128-byte boxes, 128-byte swizzle; five per byte: 8 groups = 208 bytes, no swizzle
    const cuuint32_t box[2] = {FMT == 3 ? 8u * 26u : 128u, static_cast<cuuint32_t>(ROWS)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(W.codes), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     FMT == 3 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return lb::fail(LB_ERR_CUDA, "lb_gemv: codes tensor map (CUresult %d)", static_cast<int>(r));
  }
  if (scales_tma) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(n)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(G) * 2};
    const cuuint32_t box[2] = {8, static_cast<cuuint32_t>(ROWS)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(W.scales), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return lb::fail(LB_ERR_CUDA, "lb_gemv: scales tensor map (CUresult %d)", static_cast<int>(r));
  }
  return LB_OK;
}

// Tensor maps and sizes of one problem (gpc: groups per K chunk of the launch's split).
template <int FMT>
lb_status fill_prob(const lb_weight& W, const void* x, void* y, int gpc, Prob& pr) {
  const int n = static_cast<int>(W.n), k = static_cast<int>(W.k), G = k / lb::kGroup;
  memset(&pr, 0, sizeof(pr));
  pr.scales_tma = (G % 8 == 0) ? 1 : 0;                            // scales row stride: 16-byte multiple
  {
    const uintptr_t h = (reinterpret_cast<uintptr_t>(W.codes) >> 8) ^ (reinterpret_cast<uintptr_t>(W.codes) >> 20);
    std::lock_guard<std::mutex> lk(g_maps_mu);
    MapEntry& e = g_maps[h % kMapCache];
    if (!(e.valid && e.codes == W.codes && e.scales == W.scales && e.n == W.n && e.k == W.k && e.fmt == W.fmt)) {
      e.valid = 0;
      lb_status s = encode_maps<FMT>(W, e.tm_codes, e.tm_scales, pr.scales_tma);
      if (s != LB_OK) return s;
      e.codes = W.codes;
      e.scales = W.scales;
      e.n = W.n;
      e.k = W.k;
      e.fmt = W.fmt;
      e.valid = 1;
    }
    pr.tm_codes = e.tm_codes;
    pr.tm_scales = e.tm_scales;
  }
  pr.scales = W.scales;
  pr.x = static_cast<const uint16_t*>(x);
  pr.y = static_cast<uint16_t*>(y);
  pr.n = n;
  pr.k = k;
  pr.G = G;
  pr.gpc = gpc;
  pr.row_blocks = (n + ROWS - 1) / ROWS;
  return LB_OK;
}

template <int FMT, bool XBF, int BP>
lb_status launch_args(Args& args, int grid_x, int grid_y, int smem, cudaStream_t st) {
  args.test_fault = lb::take_test_fault(lb::kTestFaultGemv) ? 1 : 0;
  args.wait_ns = args.test_fault ? lb::kTestWaitNs : lb::kWaitNs;
  args.err = lb::device_error_word();
  if (!args.err) return lb::fail(LB_ERR_CUDA, "lb_gemv: device error word unavailable");
  {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64 || !done[dev]) {
      cudaError_t e = cudaFuncSetAttribute(gemv_kernel<FMT, XBF, BP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemMax);
      if (e != cudaSuccess) return lb::cuda_fail(e, "lb_gemv: shared memory attribute");
      if (dev >= 0 && dev < 64) done[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_x, grid_y, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (args.S > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = args.S;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_kernel<FMT, XBF, BP>, args);
  if (e != cudaSuccess) return lb::cuda_fail(e, "lb_gemv: launch");
  return LB_OK;
}

// One GEMV: persistent CTAs over row blocks, K split across a cluster when that is faster.
template <int FMT, bool XBF, int BP>
lb_status launch_t(const lb_weight& W, const uint16_t* x, int batch, uint16_t* y, cudaStream_t st) {
  using L = Layout<FMT, BP>;
  const int k = static_cast<int>(W.k), G = k / lb::kGroup;
  const int sms = lb::sm_count();
  const int row_blocks = static_cast<int>((W.n + ROWS - 1) / ROWS);
  const Plan plan = plan_split<FMT, BP>(G, row_blocks, sms);
  if (plan.S == 0) return lb::fail(LB_ERR_UNSUPPORTED, "lb_gemv: K = %d too long for batch %d", k, batch);
  static_assert(sizeof(Args) <= 4096, "kernel parameters");
  Args args;
  memset(&args, 0, sizeof(args));
  lb_status s = fill_prob<FMT>(W, x, y, plan.gpc, args.p[0]);
  if (s != LB_OK) return s;
  args.count = 1;
  args.batch = batch;
  args.S = plan.S;
  return launch_args<FMT, XBF, BP>(args, plan.S,
                                   plan.S > 1 ? (row_blocks + plan.rpc - 1) / plan.rpc : min(row_blocks, sms),
                                   L::total(plan.gpc), st);
}

// Several GEMVs in one launch: one CTA (S > 1: one cluster of S CTAs, each a K chunk) per
// (problem, row block).  One split S serves every problem (cluster dimensions are per launch); it
// comes from the same time model as plan_split.  Problems with the longest K get the first grid
// rows, so that the slowest CTAs start first.
template <int FMT, bool XBF, int BP>
lb_status launch_many(const lb_gemv_problem* probs, int count, int batch, cudaStream_t st) {
  using L = Layout<FMT, BP>;
  int order[kMaxProblems];
  for (int i = 0; i < count; ++i) order[i] = i;
  for (int i = 1; i < count; ++i)                                  // stable insertion sort, K descending
    for (int j = i; j > 0 && probs[order[j]].W.k > probs[order[j - 1]].W.k; --j) {
      const int t = order[j];
      order[j] = order[j - 1];
      order[j - 1] = t;
    }
  const int sms = lb::sm_count();
  const double t_group = group_ns<FMT, L::LU>();
  int units = 0, gmax = 0;
  for (int i = 0; i < count; ++i) {
    units += static_cast<int>((probs[i].W.n + ROWS - 1) / ROWS);
    gmax = max(gmax, static_cast<int>(probs[i].W.k / lb::kGroup));
  }
  if (units > 65535)
    return lb::fail(LB_ERR_SHAPE, "lb_gemv_batched: %d row blocks of 128 exceed one launch (65535)", units);
  auto chunk = [](int G, int S) { return S == 1 ? G : ((G + S - 1) / S + GS - 1) / GS * GS; };
  int best_s = 0;
  double best_t = 1e30;
  for (int s_try = 1; s_try <= kMaxCluster; ++s_try) {
    const int g = chunk(gmax, s_try);
    if (s_try > 1 && (gmax + g - 1) / g != s_try) continue;        // the longest problem uses every rank
    if (L::total(g) > kSmemMax) continue;
    const int clusters = max(1, sms / s_try);
    const int waves = (units + clusters - 1) / clusters;
    const double t = waves * ((s_try == 1 ? 2500.0 : 3000.0) + g * t_group);
    if (t < best_t * 0.999) { best_t = t; best_s = s_try; }
  }
  if (best_s == 0)
    return lb::fail(LB_ERR_UNSUPPORTED, "lb_gemv_batched: K = %d too long at batch %d", gmax * lb::kGroup, batch);
  Args args;
  memset(&args, 0, sizeof(args));
  int smem = 0;
  units = 0;
  for (int i = 0; i < count; ++i) {
    const lb_gemv_problem& pb = probs[order[i]];
    const int gpc = chunk(static_cast<int>(pb.W.k / lb::kGroup), best_s);
    lb_status s = fill_prob<FMT>(pb.W, pb.x, pb.y, gpc, args.p[i]);
    if (s != LB_OK) return s;
    args.p[i].unit0 = units;
    units += args.p[i].row_blocks;
    smem = max(smem, L::total(gpc));
  }
  args.count = count;
  args.batch = batch;
  args.S = best_s;
  // one x and one K for every problem (q / k / v, gate / up): persistent CTAs over all the units,
  // one x prologue per CTA
  bool same = best_s == 1;
  for (int i = 1; i < count; ++i)
    same = same && probs[i].x == probs[0].x && probs[i].W.k == probs[0].W.k;
  if (same && count > 1) {
    args.shared = 1;
    args.units = units;
    return launch_args<FMT, XBF, BP>(args, 1, min(units, sms), smem, st);
  }
  return launch_args<FMT, XBF, BP>(args, best_s, units, smem, st);
}

// SiLU-gated pair h = silu(W_gate x) * (W_up x): one CTA (S > 1: one cluster of S CTAs) per
// 128-row block runs the block's gate rows, then its up rows, on one x prologue.  S comes from the
// same time model, with two units of work per CTA.
template <int FMT, bool XBF, int BP>
lb_status launch_pair(const lb_weight& Wg, const lb_weight& Wu, const uint16_t* x, int batch, uint16_t* h,
                      cudaStream_t st) {
  using L = Layout<FMT, BP>;
  const int sms = lb::sm_count();
  const double t_group = group_ns<FMT, L::LU>();
  const int G = static_cast<int>(Wg.k / lb::kGroup);
  const int units = static_cast<int>((Wg.n + ROWS - 1) / ROWS);
  auto chunk = [](int g, int S) { return S == 1 ? g : ((g + S - 1) / S + GS - 1) / GS * GS; };
  int best_s = 0;
  double best_t = 1e30;
  for (int s_try = 1; s_try <= kMaxCluster; ++s_try) {
    const int g = chunk(G, s_try);
    if (s_try > 1 && (G + g - 1) / g != s_try) continue;            // every rank has groups
    if (L::total(g) > kSmemMax) continue;
    const int clusters = max(1, sms / s_try);
    const int waves = (units + clusters - 1) / clusters;
    const double t = waves * ((s_try == 1 ? 2500.0 : 3000.0) + 2 * g * t_group);
    if (t < best_t * 0.999) { best_t = t; best_s = s_try; }
  }
  if (best_s == 0) return lb::fail(LB_ERR_UNSUPPORTED, "lb_gemv_swiglu: K = %d too long at batch %d", G * lb::kGroup, batch);
  if (units > 65535) return lb::fail(LB_ERR_SHAPE, "lb_gemv_swiglu: %d row blocks of 128 exceed one launch (65535)", units);
  Args args;
  memset(&args, 0, sizeof(args));
  const int gpc = chunk(G, best_s);
  lb_status s = fill_prob<FMT>(Wg, x, h, gpc, args.p[0]);
  if (s != LB_OK) return s;
  s = fill_prob<FMT>(Wu, x, h, gpc, args.p[1]);
  if (s != LB_OK) return s;
  args.count = 2;
  args.batch = batch;
  args.S = best_s;
  args.fuse = 1;
  return launch_args<FMT, XBF, BP>(args, best_s, units, L::total(gpc), st);
}

// 1-bit at batch 1 takes the lookup-table consumer (BP = 0) whenever its table fits.
template <int FMT>
bool lut_fits(int G, int row_blocks) {
  return FMT == 1 && plan_split<FMT, 0>(G, row_blocks, lb::sm_count()).S != 0;
}
template <int FMT, bool XBF>
lb_status launch_b(const lb_weight& W, const uint16_t* x, int batch, uint16_t* y, cudaStream_t st) {
  switch (pad_batch(batch)) {
    case 1:
      if constexpr (FMT == 1)
        if (lut_fits<FMT>(static_cast<int>(W.k / lb::kGroup), static_cast<int>((W.n + ROWS - 1) / ROWS)))
          return launch_t<FMT, XBF, 0>(W, x, batch, y, st);
      return launch_t<FMT, XBF, 1>(W, x, batch, y, st);
    case 2: return launch_t<FMT, XBF, 2>(W, x, batch, y, st);
    case 4: return launch_t<FMT, XBF, 4>(W, x, batch, y, st);
    default: return launch_t<FMT, XBF, 8>(W, x, batch, y, st);
  }
}
template <int FMT, bool XBF>
lb_status launch_pb(const lb_weight& Wg, const lb_weight& Wu, const uint16_t* x, int batch, uint16_t* h,
                    cudaStream_t st) {
  switch (pad_batch(batch)) {
    case 1:
      if constexpr (FMT == 1)
        if (lut_fits<FMT>(static_cast<int>(Wg.k / lb::kGroup), static_cast<int>((Wg.n + ROWS - 1) / ROWS)))
          return launch_pair<FMT, XBF, 0>(Wg, Wu, x, batch, h, st);
      return launch_pair<FMT, XBF, 1>(Wg, Wu, x, batch, h, st);
    case 2: return launch_pair<FMT, XBF, 2>(Wg, Wu, x, batch, h, st);
    case 4: return launch_pair<FMT, XBF, 4>(Wg, Wu, x, batch, h, st);
    default: return launch_pair<FMT, XBF, 8>(Wg, Wu, x, batch, h, st);
  }
}
template <int FMT, bool XBF>
lb_status launch_mb(const lb_gemv_problem* probs, int count, int batch, cudaStream_t st) {
  switch (pad_batch(batch)) {
    case 1:
      if constexpr (FMT == 1) {
        int gmax = 0, units = 0;
        for (int i = 0; i < count; ++i) {
          gmax = max(gmax, static_cast<int>(probs[i].W.k / lb::kGroup));
          units += static_cast<int>((probs[i].W.n + ROWS - 1) / ROWS);
        }
        if (lut_fits<FMT>(gmax, units)) return launch_many<FMT, XBF, 0>(probs, count, batch, st);
      }
      return launch_many<FMT, XBF, 1>(probs, count, batch, st);
    case 2: return launch_many<FMT, XBF, 2>(probs, count, batch, st);
    case 4: return launch_many<FMT, XBF, 4>(probs, count, batch, st);
    default: return launch_many<FMT, XBF, 8>(probs, count, batch, st);
  }
}

}  // namespace

namespace lb {

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Five per byte at batch 1 on the lookup-table consumer: needs TMA-able code rows (26 G bytes a
// multiple of 16, i.e. G % 8 == 0) and a table that fits some K split.
bool gemv_t5_lut_ok(const lb_weight& W, int batch) {
  const int G = static_cast<int>(W.k / kGroup);
  return batch == 1 && G % 8 == 0 &&
         plan_split<3, 0>(G, static_cast<int>((W.n + ROWS - 1) / ROWS), sm_count()).S != 0;
}

lb_status launch_gemv(const lb_weight& W, const void* x, int xdt, int batch, void* y, cudaStream_t st) {
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint16_t* ys = static_cast<uint16_t*>(y);
  const bool bf = xdt == LB_BF16;
  if (W.fmt == LB_FMT_TERNARY5_G128)                               // callers checked gemv_t5_lut_ok
    return bf ? launch_t<3, true, 0>(W, xs, batch, ys, st) : launch_t<3, false, 0>(W, xs, batch, ys, st);
  if (W.fmt == LB_FMT_1BIT_G128)
    return bf ? launch_b<1, true>(W, xs, batch, ys, st) : launch_b<1, false>(W, xs, batch, ys, st);
  return bf ? launch_b<2, true>(W, xs, batch, ys, st) : launch_b<2, false>(W, xs, batch, ys, st);
}

lb_status launch_gemv_swiglu(const lb_weight& Wg, const lb_weight& Wu, const void* x, int xdt, int batch, void* h,
                             cudaStream_t st) {
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint16_t* hs = static_cast<uint16_t*>(h);
  const bool bf = xdt == LB_BF16;
  if (Wg.fmt == LB_FMT_TERNARY5_G128)                              // callers checked gemv_t5_lut_ok
    return bf ? launch_pair<3, true, 0>(Wg, Wu, xs, batch, hs, st) : launch_pair<3, false, 0>(Wg, Wu, xs, batch, hs, st);
  if (Wg.fmt == LB_FMT_1BIT_G128)
    return bf ? launch_pb<1, true>(Wg, Wu, xs, batch, hs, st) : launch_pb<1, false>(Wg, Wu, xs, batch, hs, st);
  return bf ? launch_pb<2, true>(Wg, Wu, xs, batch, hs, st) : launch_pb<2, false>(Wg, Wu, xs, batch, hs, st);
}

lb_status launch_gemv_batched(const lb_gemv_problem* probs, int count, int xdt, int batch, cudaStream_t st) {
  if (count > kMaxProblems) return fail(LB_ERR_SHAPE, "lb_gemv_batched: count %d > %d", count, kMaxProblems);
  const bool bf = xdt == LB_BF16;
  if (probs[0].W.fmt == LB_FMT_TERNARY5_G128) {
    // five per byte: one lookup-table launch at batch 1 when every problem's tables fit,
    // otherwise one CUDA-core launch per problem
    bool lut = true;
    for (int i = 0; i < count; ++i) lut = lut && gemv_t5_lut_ok(probs[i].W, batch);
    if (lut) return bf ? launch_many<3, true, 0>(probs, count, batch, st) : launch_many<3, false, 0>(probs, count, batch, st);
    for (int i = 0; i < count; ++i) {
      const lb_status s = launch_gemv_t5(probs[i].W, probs[i].x, xdt, batch, probs[i].y, st);
      if (s != LB_OK) return s;
    }
    return LB_OK;
  }
  if (probs[0].W.fmt == LB_FMT_1BIT_G128)
    return bf ? launch_mb<1, true>(probs, count, batch, st) : launch_mb<1, false>(probs, count, batch, st);
  return bf ? launch_mb<2, true>(probs, count, batch, st) : launch_mb<2, false>(probs, count, batch, st);
}

}  // namespace lb

#ifdef LB_GEMV_TRACE
// Trace builds only: copy the phase trace (kTraceCtas x kTraceEvents x {globaltimer ns, clock64})
// to host memory and clear it.  Returns the bytes copied, or -1 on a CUDA error.
extern "C" long long lb_gemv_trace_read(void* host, long long bytes) {
  const long long n = static_cast<long long>(sizeof(g_gemv_trace));
  if (bytes < n) return -1;
  if (cudaMemcpyFromSymbol(host, g_gemv_trace, sizeof(g_gemv_trace)) != cudaSuccess) return -1;
  static unsigned long long zero[kTraceCtas][kTraceEvents][2];
  if (cudaMemcpyToSymbol(g_gemv_trace, zero, sizeof(zero)) != cudaSuccess) return -1;
  return n;
}
#endif
