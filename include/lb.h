/*
 * lb.h — C ABI of liblb: products against Bonsai-style low-bit weights on B300 (sm_103a).
 *
 * Weight formats (group size 128 along K; one IEEE binary16 scale per group; w = s_g * t_i):
 *   - 1-bit ("Q1_0_g128"): t in {-1,+1}; bit 0 -> -scale, bit 1 -> +scale; 16 B of bits + 2 B of
 *     scale per 128 weights = 1.125 bits per weight.  Defined by 7minutos.es, "Un tutorial de
 *     codificacion para ejecutar PrismML Bonsai 1-bit LLM en CUDA con GGUF", section
 *     "7 · Q1_0_g128 Cuantización" (representation box and Python demo).
 *   - ternary: t in {-1,0,+1} with the same FP16 group scale (7minutos.es, "PrismML lanza
 *     Bonsai 27B: compilaciones ternarias y de 1 bit", section "Cómo funciona la compresión"),
 *     stored as 2-bit fields f = t + 1 (0 -> -1, 1 -> 0, 2 -> +1; 3 is invalid): 32 B of codes
 *     + 2 B of scale per 128 weights = 2.125 bits per weight.
 *   - ternary, five per byte (LB_FMT_TERNARY5_G128; es.news.hada.io topic 31450, comments: five
 *     three-state values fit one byte; kerneldigest.dev, "Bonsai 2 27B", section "Arquitectura
 *     del Sistema": 1.76 effective bits per weight): the same codes as base-3 digits f = t + 1,
 *     26 B of codes + 2 B of scale per 128 weights = 1.75 bits per weight.  Taken by
 *     lb_pack_ternary5 and lb_gemv; the other products return LB_ERR_UNSUPPORTED for it.
 *
 * Packed layout of an N x K matrix (rows n = output features, K = reduction, K % 128 == 0),
 * two planes, both row-major and contiguous:
 *   codes : 1-bit   uint8 [N][K/8],  weight k of row n = bit (k % 8) of byte k/8 (LSB first)
 *           ternary uint8 [N][K/4],  weight k of row n = bits 2(k%4)..2(k%4)+1 of byte k/4
 *           ternary five per byte: uint8 [N][26 K/128]; group g of row n is bytes 26g .. 26g+25,
 *           byte j of a group holds its weights 5j .. 5j+4 as sum_i (t + 1) 3^i (first weight in
 *           the lowest digit); byte 25 holds weights 125..127
 *   scales: uint16  [N][K/128], the binary16 bit pattern of the scale of group k/128 of row n
 *
 * Activations and outputs are row-major [rows][K] / [rows][N] arrays of binary16 (LB_F16) or
 * bfloat16 (LB_BF16) values; all accumulation is FP32.
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller (allocated with cudaMalloc or a
 *     framework allocator); the library never frees them and keeps no reference after a call.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream); work is enqueued on it.
 *   - Errors are returned as lb_status and never abort the process; nothing traps on the GPU.
 *     lb_last_error() returns a thread-local text for the last failing call of this thread.
 *   - lb_gemv, lb_gemv_batched, lb_gemv_swiglu, lb_gemm, lb_gemm_noalloc and lb_embed validate
 *     their arguments on the host and then launch asynchronously: LB_OK means "enqueued".  The pack calls synchronise `stream` to read the device-side
 *     validation result, so their LB_OK means "done and valid".
 *   - Thread safety: every call may be made from any host thread; pack calls serialise on an
 *     internal mutex (they share one device-side validation word per device).
 *   - Launch order: lb_gemv, lb_gemv_batched and lb_gemv_swiglu are launched with programmatic
 *     dependent launch (the five-per-byte format only on its batch-1 lookup-table path).  Such a launch may start while the kernel
 *     enqueued just before it on `stream` is still running; it reads x and writes y only after
 *     that kernel has completed, but it starts streaming the packed weights (codes and scales)
 *     before.  The weights must therefore not be written by the kernel that immediately precedes
 *     the call on `stream`: write them at least one kernel earlier, or separate the two by a host
 *     synchronisation.  The pack calls synchronise, so packing and then multiplying is safe.
 *     Activations and outputs carry no such restriction (x may come from the preceding kernel, y
 *     may be read by the next one).  lb_gemm, lb_gemm_noalloc, lb_embed and the five-per-byte
 *     GEMV's CUDA-core path wait for the preceding kernel before reading anything.
 */
#ifndef LB_H_
#define LB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t; declared here so that this header needs no CUDA headers. */
typedef struct CUstream_st* lb_stream;

typedef enum lb_status {
  LB_OK = 0,
  LB_ERR_NULL = 1,        /* a required pointer is NULL                                        */
  LB_ERR_SHAPE = 2,       /* n < 1, k < 128 or k % 128 != 0, batch outside [1, 8], m < 1       */
  LB_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned                          */
  LB_ERR_DTYPE = 4,       /* unknown lb_dtype / lb_format                                      */
  LB_ERR_CODE = 5,        /* a ternary code outside {-1, 0, +1} (pack_ternary)                 */
  LB_ERR_NONFINITE = 6,   /* NaN or Inf among the fp32 weights (pack_1bit)                      */
  LB_ERR_RANGE = 7,       /* a group max |w| rounds to binary16 infinity (pack_1bit)            */
  LB_ERR_CUDA = 8,        /* a CUDA runtime/driver call failed; see lb_last_error()           */
  LB_ERR_UNSUPPORTED = 9, /* valid request this build does not implement                      */
  LB_ERR_WORKSPACE = 10   /* workspace pointer/size smaller than lb_gemm_workspace_bytes()    */
} lb_status;

typedef enum lb_format { LB_FMT_1BIT_G128 = 1, LB_FMT_TERNARY_G128 = 2, LB_FMT_TERNARY5_G128 = 3 } lb_format;

typedef enum lb_dtype { LB_F16 = 1, LB_BF16 = 2 } lb_dtype;

/* A packed weight matrix; all pointers are device pointers owned by the caller. */
typedef struct lb_weight {
  int32_t fmt;            /* lb_format                                                         */
  int32_t reserved;       /* must be 0                                                         */
  int64_t n;              /* rows (output features), >= 1                                      */
  int64_t k;              /* columns (reduction length), a positive multiple of 128            */
  const uint8_t* codes;   /* codes plane, 16-byte aligned                                      */
  const uint16_t* scales; /* scales plane, 16-byte aligned                                     */
} lb_weight;

/* Text for a status code (static storage). */
const char* lb_status_string(lb_status s);

/* Thread-local description of the last failing call on this thread ("" if none). */
const char* lb_last_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int lb_version(void);

/*
 * Byte sizes of the two planes of an n x k matrix in format `fmt` (pure host arithmetic):
 *   1-bit:   codes = n*k/8, scales = n*(k/128)*2   (18 bytes per group, 7minutos.es tutorial, §7 demo)
 *   ternary: codes = n*k/4, scales = n*(k/128)*2   (34 bytes per group)
 *   ternary five per byte: codes = n*(k/128)*26, scales = n*(k/128)*2   (28 bytes per group)
 * Errors: LB_ERR_NULL (an output pointer is NULL), LB_ERR_SHAPE, LB_ERR_DTYPE (unknown fmt).
 */
lb_status lb_packed_bytes(int fmt, int64_t n, int64_t k, size_t* codes_bytes, size_t* scales_bytes);

/*
 * 1-bit sign / max-abs quantiser (7minutos.es tutorial, section "7 · Q1_0_g128 Cuantización",
 * Python demo): for every row n and group g of 128 weights,
 *     scale[n][g] = binary16_RNE( max_i |w[n][128g+i]| )      (maximum taken exactly in fp32)
 *     bit i       = 1 if w[n][128g+i] >= 0 else 0              (+0.0 and -0.0 give 1)
 *
 * w      : device float32 [n][k], row-major, 16-byte aligned, read only.
 * codes  : device uint8 [n][k/8] (output), 16-byte aligned.
 * scales : device uint16 [n][k/128] (output), 16-byte aligned.
 * Synchronous: the call synchronises `stream` and then reports
 *   LB_ERR_NONFINITE if any weight is NaN/Inf, LB_ERR_RANGE if a group maximum rounds to
 *   binary16 infinity (|w| >= 65520).  On these errors the outputs are unspecified.
 */
lb_status lb_pack_1bit(const float* w, int64_t n, int64_t k, uint8_t* codes, uint16_t* scales,
                       lb_stream stream);

/*
 * Ternary packer (7minutos.es, "PrismML lanza Bonsai 27B", section "Cómo funciona la compresión";
 * kerneldigest.dev, "Bonsai 2 27B", section "Arquitectura del Sistema"): codes are given, not
 * quantised.  Writes field t + 1 for every weight and copies the scales bit for bit.
 *
 * t      : device int8 [n][k], values in {-1, 0, +1}, 16-byte aligned.
 * s_in   : device uint16 [n][k/128] binary16 scale patterns, 16-byte aligned.
 * codes  : device uint8 [n][k/4] (output); scales: device uint16 [n][k/128] (output; may equal s_in).
 * Synchronous; returns LB_ERR_CODE if any t is outside {-1, 0, +1} (outputs then unspecified).
 */
lb_status lb_pack_ternary(const int8_t* t, const uint16_t* s_in, int64_t n, int64_t k,
                          uint8_t* codes, uint16_t* scales, lb_stream stream);

/*
 * The same ternary packing, five codes per byte (LB_FMT_TERNARY5_G128 layout above): byte j of a
 * group is sum_i (t[5j+i] + 1) 3^i.  Arguments as lb_pack_ternary, with codes a device uint8
 * [n][26 k/128] output (16-byte aligned base).  Synchronous; LB_ERR_CODE if any t is outside
 * {-1, 0, +1}.
 */
lb_status lb_pack_ternary5(const int8_t* t, const uint16_t* s_in, int64_t n, int64_t k,
                           uint8_t* codes, uint16_t* scales, lb_stream stream);

/*
 * Decode GEMV and small-batch GEMV (7minutos.es, "PrismML lanza Bonsai 27B", section
 * "Rendimiento y decodificación especulativa DSpark": generation is memory-bandwidth bound;
 * speculative verification of k = 4 drafted tokens runs the target at width k + 1):
 *     y[b][n] = sum_g s[n][g] * sum_{i<128} t[n][128g+i] * x[b][128g+i],   0 <= b < batch,
 * with FP32 accumulation, rounded once to the dtype of x (round to nearest even).
 *
 * W     : packed matrix (n x k), any format.  The five-per-byte ternary format at batch 1 with
 *         k a multiple of 1024 runs the pipelined kernel of the other formats, adding per code
 *         byte two entries of shared-memory tables of signed activation sums (k <= 40960, where
 *         the tables of a K chunk fit one CTA of an 8-CTA cluster); otherwise it runs a CUDA-core kernel
 *         that decodes a code byte through a 243-entry table (no K limit).
 * x     : device [batch][k] of `xdt`, 16-byte aligned.     y : device [batch][n] of `xdt`.
 * batch : 1 .. 8.
 * Asynchronous on `stream`.  Errors (no launch): LB_ERR_NULL, LB_ERR_SHAPE, LB_ERR_ALIGN,
 * LB_ERR_DTYPE; LB_ERR_UNSUPPORTED if k is longer than 8 CTAs of a cluster hold in shared memory
 * (1-bit: k <= 327680 at batch 1, 180224 at batch 2, 90112 at batch 3-4, 49152 at batch 5-8;
 * ternary: k <= 344064, 188416, 98304, 49152); LB_ERR_CUDA if the launch fails.
 */
lb_status lb_gemv(const lb_weight* W, const void* x, int xdt, int batch, void* y, lb_stream stream);

/* One GEMV of a grouped call: y = W x with the layouts of lb_gemv (all pointers device, caller-owned). */
typedef struct lb_gemv_problem {
  lb_weight W;
  const void* x;          /* [batch][W.k] of the call's xdt, 16-byte aligned */
  void* y;                /* [batch][W.n] of the call's xdt, 16-byte aligned */
} lb_gemv_problem;

#define LB_GEMV_BATCH_MAX 8

/*
 * Several independent decode GEMVs in one launch (the matrices of one decoder layer that read the
 * same activations, e.g. q / k / v or gate / up; 7minutos.es, "PrismML lanza Bonsai 27B", section
 * "Rendimiento y decodificación especulativa DSpark": decode streams every weight once per token, so
 * at small matrix sizes the fixed cost of a launch dominates).  Each problem computes exactly what
 * lb_gemv computes for it; problems may differ in n, k, x and y (x buffers may be shared).
 *
 * problems : host array of `count` problems, 1 <= count <= LB_GEMV_BATCH_MAX, all of the same format.
 *            Five per byte: one launch when lb_gemv would take the lookup-table path for every
 *            problem, otherwise one CUDA-core launch per problem, in order.
 * xdt      : LB_F16 or LB_BF16 for every x and y;  batch : 1 .. 8 for every problem.
 * No y may overlap another problem's x or y.  Asynchronous on `stream`.  Errors (no launch):
 * LB_ERR_NULL, LB_ERR_SHAPE (count or batch out of range, a bad n / k), LB_ERR_ALIGN, LB_ERR_DTYPE,
 * LB_ERR_UNSUPPORTED (mixed formats, or a k above the lb_gemv limit), LB_ERR_SHAPE also when the
 * problems hold more than 65535 blocks of 128 rows in total, LB_ERR_CUDA if the launch fails.
 */
lb_status lb_gemv_batched(const lb_gemv_problem* problems, int count, int xdt, int batch, lb_stream stream);

/*
 * SiLU-gated pair of one decoder layer's feed-forward block in one launch:
 *     h[b][n] = silu(g[b][n]) * u[b][n],   g = W_gate x[b],  u = W_up x[b],  silu(z) = z / (1 + e^-z),
 * with g and u each computed exactly as lb_gemv computes them (FP32 accumulation), combined in FP32
 * and rounded once to `xdt` (RNE); g and u are never stored.  (openclawradar.com, "Bonsai 1.7B
 * Modelo Ternario Alcanza 442 T/s en M4 Max", section "Detalles técnicos": the fastest decode came
 * from kernels specialised at the matvec / FFN level; 7minutos.es, "PrismML lanza Bonsai 27B": the
 * models are builds of a Qwen3-family base, whose feed-forward block is SiLU-gated.)  One CTA
 * (or cluster) per 128-row block runs the block's gate rows and then its up rows on one prologue of
 * x, so the pair costs one launch and one x prologue.
 *
 * Wg, Wu   : packed matrices of the same format and shape (N x K).  Five per byte: batch 1 with K a
 *            multiple of 1024 (K <= 40960; the lookup-table form), LB_ERR_UNSUPPORTED otherwise.
 * x        : device [batch][K] of `xdt`, 16-byte aligned;  h : device [batch][N] of `xdt`, 16-byte
 *            aligned, caller-owned, not overlapping x.
 * batch    : 1 .. 8, with the K limits of lb_gemv;  N <= 65535 * 128.
 * Asynchronous on `stream`.  Errors (no launch): LB_ERR_NULL, LB_ERR_SHAPE (different shapes,
 * batch), LB_ERR_ALIGN, LB_ERR_DTYPE, LB_ERR_UNSUPPORTED (different formats, K above the limit),
 * LB_ERR_CUDA if the launch fails.
 */
lb_status lb_gemv_swiglu(const lb_weight* Wg, const lb_weight* Wu, const void* x, int xdt, int batch, void* h,
                         lb_stream stream);

/*
 * Workspace bytes that lb_gemm needs for an m x k activation matrix of dtype `xdt` against an
 * n x k weight (0 means none is needed).  Pure host arithmetic.
 */
lb_status lb_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int xdt, size_t* bytes);

/*
 * Prefill GEMM (same product as lb_gemv for m token rows; 7minutos.es, "PrismML lanza Bonsai
 * 27B", section "Rendimiento …": prefill is compute bound):
 *     Y[r][n] = sum_g s[n][g] * sum_{i<128} t[n][128g+i] * X[r][128g+i],   0 <= r < m,
 * FP32 accumulation on the tensor cores, output rounded to `ydt` (RNE).
 *
 * W                : packed matrix (n x k), 1-bit or ternary; n must be a multiple of 16.
 * x                : device [m][k] of `xdt`, 16-byte aligned, any finite values.  The product runs
 *                    on FP16 tensor-core operands, where s * t is exact.  binary16 rows are used as
 *                    they are; each bfloat16 row is first scaled by an exact power of two that puts
 *                    its largest magnitude in [2^15, 2^16), converted to binary16 (exact for every
 *                    element within 2^32 of the row maximum; smaller ones round to the binary16
 *                    subnormal grid), and the FP32 results are scaled back.
 * y                : device [m][n] of `ydt`, 16-byte aligned.
 * workspace        : device scratch of at least lb_gemm_workspace_bytes(...) bytes, 256-byte
 *                    aligned, used only during this call's kernels (may be reused afterwards).
 * Asynchronous on `stream`.  Errors (no launch): LB_ERR_NULL, LB_ERR_SHAPE, LB_ERR_ALIGN,
 * LB_ERR_DTYPE, LB_ERR_WORKSPACE; LB_ERR_CUDA.  Limit of one call: 1 <= m <= 65535 * 256
 * (LB_ERR_SHAPE beyond).  Any m is served by the
 * same kernels: a token tile holding fewer than 256 tokens runs its tensor-core products only as
 * wide as its token count (rounded up to 16), so mid-size m (16 .. 128) pays for the tokens it
 * has.
 */
lb_status lb_gemm(const lb_weight* W, const void* x, int xdt, int64_t m, void* y, int ydt,
                  void* workspace, size_t workspace_bytes, lb_stream stream);

/*
 * Embedding-row gather (7minutos.es, "PrismML lanza Bonsai 27B", section "Cómo funciona la
 * compresión", and es.news.hada.io topic 31450, section "Configuración multimodal y de bajo bit
 * de extremo a extremo": the low-bit representation covers the embedding table too):
 *     out[i][k] = s[ids[i]][k / 128] * t[ids[i]][k],   0 <= i < count, 0 <= k < K,
 * rounded to `out_dtype` (RNE; binary16 output is exact, bfloat16 output rounds the scale once).
 * t = 0 gives a zero carrying the sign of s, as IEEE multiplication does.
 *
 * W         : packed table (N rows x K), either format.
 * ids       : device int32 [count] row ids, 4-byte aligned.  An id outside [0, N) is not a
 *             table row: its output row is written as +0 and bit 2 of the device error word is
 *             set (lb_device_error); the call itself cannot see device data and returns LB_OK.
 * count     : 0 .. 2^31 - 1 rows with count * ceil(K / 1024) <= 2^34 - 8; 0 launches nothing (ids
 *             and out may then be NULL).
 * out       : device [count][K] of `out_dtype`, 16-byte aligned, caller-owned.
 * Asynchronous on `stream`.  Errors (no launch): LB_ERR_NULL, LB_ERR_SHAPE, LB_ERR_ALIGN,
 * LB_ERR_DTYPE (format or out_dtype), LB_ERR_CUDA if the launch fails.
 */
lb_status lb_embed(const lb_weight* W, const int32_t* ids, int64_t count, void* out, int out_dtype,
                   lb_stream stream);

/*
 * Sticky device-side error word of the current device (0 = none).  Kernels that wait on an
 * mbarrier give up after a bounded number of polls, set a bit here and return instead of
 * hanging.  lb_device_error() synchronises the device, reads the word and, if `clear` is
 * non-zero, resets it.  Bit 0: a GEMM or GEMV pipeline wait timed out.  Bit 1: unused.  Bit 2:
 * an lb_embed row id lay outside [0, n).
 */
lb_status lb_device_error(uint32_t* word, int clear);

/* Size of the library-owned scratch used by lb_gemm_noalloc: 8 MiB of activation tiles plus 64 KiB
 * of per-token factors, e.g. 512 tokens at k = 8192. */
#define LB_GEMM_NOALLOC_SCRATCH_BYTES (((size_t)8 << 20) + ((size_t)64 << 10))

/*
 * lb_gemm without a caller-provided workspace and without any allocation.  (The pages describe
 * no such call: it exists for callers of this library that cannot allocate device memory.)
 *
 * Some callers cannot hand lb_gemm a workspace: plug-in style hosts that pass a kernel only its
 * input and output buffers and give it no allocator, and serving loops that must not call
 * cudaMalloc because it can synchronise the device and stall every other stream.  This entry point
 * computes exactly what lb_gemm computes, with the same kernels, but keeps the activation staging
 * in a scratch array that the library itself defines at file scope in device memory
 * (LB_GEMM_NOALLOC_SCRATCH_BYTES; every GPU that loads the library holds it until the process
 * exits).  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments, layout, dtypes and error codes are those of lb_gemm, without the workspace pair.
 * Additionally returns LB_ERR_WORKSPACE, before launching anything, when the staging the call
 * needs (lb_gemm_workspace_bytes(m, n, k, xdt)) exceeds LB_GEMM_NOALLOC_SCRATCH_BYTES.
 *
 * The first call on a device looks up the device address of the scratch array with
 * cudaGetSymbolAddress (with that device current) and caches it; make that first call before any
 * stream capture.  All calls share the one array and it keeps the contents of the last call; each
 * call rewrites every byte of it that it later reads, so nothing needs clearing between calls.
 * Calls that overlap on the GPU (issued to different streams without ordering, or from several
 * host threads at once) race on the array and give undefined results: serialise them.
 */
lb_status lb_gemm_noalloc(const lb_weight* W, const void* x, int xdt, int64_t m, void* y, int ydt,
                          lb_stream stream);

/*
 * Read-bandwidth reference (no part of the method; the pages describe no such call): reads `bytes`
 * bytes of device memory with plain 16-byte loads in one launch shaped like the decode GEMV's (every
 * CTA lets the next kernel on the stream launch at once), and XORs all it read into *sink, so that
 * the benchmark can time the practical read ceiling of one launch of a GEMV's byte count.
 *
 * data  : device buffer, 16-byte aligned, read only.   bytes : a multiple of 16 (0 launches nothing).
 * sink  : device uint32, 4-byte aligned; its value is a checksum of no meaning.
 * Asynchronous on `stream`.  Errors (no launch): LB_ERR_NULL, LB_ERR_ALIGN, LB_ERR_SHAPE (bytes not
 * a multiple of 16); LB_ERR_CUDA if the launch fails.
 */
lb_status lb_read_probe(const void* data, size_t bytes, uint32_t* sink, lb_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* LB_H_ */
