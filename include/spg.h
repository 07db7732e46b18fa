/*
 * spg.h -- C ABI of the scaled-precision GEMM library for GB300 (sm_103a).
 *
 * The library computes the scaled low-precision linear-layer GEMM
 *     Y[T, N] = epilogue( dequant(A) . dequant(W)^T )
 * with fp32 accumulation in tensor memory and bf16 output, in two formats:
 *   - FP8 E4M3 with one fp32 scale per activation row and per weight row
 *     (ninfer PR #167, "The fp8 A8 GEMM stages its operands through TMA",
 *     opening paragraph and "What actually changes");
 *   - NVFP4: E2M1 codes, one E4M3 scale per 16 K-elements and one fp32
 *     global scale per tensor (ninfer PR #160, "The NVFP4 TMA route reads
 *     activation scales as one tile", body);
 * plus a per-tensor-scaled FP8 GEMM in NT / NN / TN / TT layouts with batch
 * strides (AstrAI commit log of csrc/kernels/fp8/gemm.cuh, first bullet).
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument is caller-owned DEVICE memory unless stated
 *     otherwise.  Nothing is allocated by the library on any call.  Scales
 *     (row, global, per-tensor) are device pointers, so no call reads a
 *     value back to the host.
 *   - Every call only enqueues work on `stream` (0 = the legacy default
 *     stream) and returns; results are ready when the stream reaches them.
 *   - Matrices are row-major with their natural leading dimension (no
 *     padding) unless stated otherwise.  bf16 values are passed as raw
 *     16-bit patterns (`void*`).
 *   - All base pointers must be 16-byte aligned (SPG_ERR_MISALIGNED).
 *   - Argument errors are detected on the host before any launch and leave
 *     outputs untouched.  A launch failure returns SPG_ERR_CUDA.  Every wait
 *     inside a kernel is bounded in time; a wait that runs out records a
 *     code in the library's device error word, the kernel returns without
 *     faulting, and spg_last_device_error() reports SPG_ERR_TIMEOUT.
 *   - Empty problems (T == 0, N == 0, rows == 0, batch == 0) return SPG_OK
 *     without launching anything.
 */
#ifndef SPG_H_
#define SPG_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPG_API __attribute__((visibility("default")))
#else
#define SPG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t. */
typedef struct CUstream_st* spg_stream_t;

typedef enum {
  SPG_EPI_LINEAR = 0, /* Y = s * acc                                   */
  SPG_EPI_ADD = 1,    /* Y = s * acc + residual   (linear_add)         */
  SPG_EPI_SWIGLU = 2  /* Y[:, j] = silu(y[:, 2j]) * y[:, 2j+1]         */
} spg_epilogue;

typedef enum {
  SPG_OK = 0,
  SPG_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum   */
  SPG_ERR_UNSUPPORTED_SHAPE = 2, /* a divisibility rule below is broken     */
  SPG_ERR_MISALIGNED = 3,        /* a base pointer is not 16-byte aligned   */
  SPG_ERR_CUDA = 4,              /* a CUDA launch / driver call failed      */
  SPG_ERR_TIMEOUT = 5            /* a bounded in-kernel wait ran out        */
} spg_status;

typedef enum {
  SPG_KIND_FP8_ROWSCALED = 0,
  SPG_KIND_NVFP4 = 1,
  SPG_KIND_FP8_TENSOR = 2
} spg_kind;

/* One launch configuration picked by the route selector. */
typedef struct {
  int32_t kind;         /* spg_kind                                           */
  int32_t block_m;      /* output rows per CTA tile (tcgen05 M)               */
  int32_t block_n;      /* accumulator columns per CTA tile (tcgen05 N total) */
  int32_t block_k;      /* K elements per pipeline stage                      */
  int32_t stages;       /* shared-memory ring depth                           */
  int32_t acc_buffers;  /* TMEM accumulator buffers (epilogue overlap)        */
  int32_t group_m;      /* m-blocks per rasterization group                   */
  int32_t grid;         /* persistent CTAs launched                           */
  int64_t tiles;        /* output tiles of the whole problem (all batches)    */
  int32_t smem_bytes;   /* dynamic shared memory per CTA                      */
  int32_t variant;      /* kernel variant index inside the library (FP8:      */
                        /* 0-3 pair tiles 256/192/160/128 wide, 4-5 one-CTA  */
                        /* 256/128, 6 swapped pair tile, 8 swapped pair tile */
                        /* whose K pieces run as the pairs of one cluster    */
                        /* (no workspace); NVFP4: 0 pair tile                */
                        /* with copied scales, 2 one-CTA, 3 pair tile with   */
                        /* warp-stored scales, 4 CUDA-core GEMV for T <= 4   */
                        /* (block_m 1, block_n 2 weight rows per warp), 5    */
                        /* cluster of two one-CTA tiles sharing B by TMA     */
                        /* multicast, 7 one-CTA tiles whose K is split over  */
                        /* the split_k CTAs of a cluster and reduced through */
                        /* distributed shared memory: no workspace)          */
  int32_t split_n;      /* last partial wave: tiles split along N this many ways */
  int32_t split_k;      /* last partial wave: tiles split along K this many ways */
                        /* (variant 7: every tile, one piece per cluster CTA) */
  int64_t workspace_bytes; /* workspace the K split needs (0 without one)     */
  int32_t swap_ab;      /* 1: operands exchanged (weights on the M side, the   */
                        /* T tokens on the N side; block_n covers tokens)     */
  int32_t reserved;     /* 0                                                  */
} spg_route;

/* Human-readable name of a status code (static string). */
SPG_API const char* spg_status_string(int status);

/* Library ABI version (major * 100 + minor).  2.00: spg_route grew the
 * swap_ab / reserved fields (its size changed). */
SPG_API int spg_version(void);

/* Bound, in nanoseconds, of every in-kernel wait of later launches
 * (default 2e9).  Host-side setting; not thread-safe against concurrent
 * launches. */
SPG_API void spg_set_wait_timeout_ns(uint64_t ns);

/* Test hook for failure detection: while enabled, every launch of the
 * tile GEMM kernels (one-CTA and two-SM) makes its epilogue wait on a
 * barrier that nothing arrives on, so that wait runs out after the bound set
 * above, the kernel records code 0x106 and every role drains and returns
 * without a fault (in a CTA pair the two producers first settle which of
 * their copies are still landing).  Host-side setting; not thread-safe
 * against concurrent launches. */
SPG_API void spg_debug_inject_stall(int enable);

/* Test hook: the route selector reads the environment variables
 * SPG_FORCE_VARIANT (pin a kernel variant), SPG_FORCE_TAIL (pin how the
 * last partial wave is split: none | n | k) and SPG_FORCE_GROUP_M (m-blocks
 * per rasterization group) once, on its first call; this makes the next
 * call read them again.  Host-side setting; not thread-safe
 * against concurrent launches. */
SPG_API void spg_debug_reload_env(void);

/* Counts of tensor-map (TMA descriptor) cache hits and misses since the
 * library was loaded.  Each GEMM call needs 3 to 6 descriptors; a descriptor
 * encoded for the same base pointer, shape, strides, box and swizzle is
 * reused.  Both pointers must be non-null (host memory). */
SPG_API void spg_debug_tmap_cache_stats(uint64_t* hits, uint64_t* misses);

/* Switch the tensor-map cache on (the default) or off; off also empties it.
 * For timing the host side of a call with and without the cache.  Host-side
 * setting; not thread-safe against concurrent launches. */
SPG_API void spg_debug_set_tmap_cache(int enable);

/* Synchronizes `stream`, then reads and clears the library's device error
 * word.  Returns SPG_OK, SPG_ERR_TIMEOUT (a bounded wait ran out in some
 * earlier launch) or SPG_ERR_CUDA (the stream reported an error). */
SPG_API spg_status spg_last_device_error(spg_stream_t stream);

/* Same as spg_last_device_error, and stores the raw code of the first wait
 * that ran out (0 if none) in *code: 0x101 ring slot free, 0x102 ring slot
 * full, 0x103 accumulator free, 0x104 accumulator full, 0x105 drain,
 * 0x106 injected stall (spg_debug_inject_stall), 0x107 a K-split arrival
 * counter could not be updated (bounded compare-and-swap loop). */
SPG_API spg_status spg_last_device_error_code(spg_stream_t stream, uint32_t* code);

/* ---------------------------------------------------------------------
 * Quantizers
 * ------------------------------------------------------------------- */

/* FP8 E4M3 row quantizer (activations at run time, weights once).
 * For each row r of x [rows, K] (bf16):
 *   amax = max_k |x[r,k]|;  s = amax / 448 (IEEE fp32; s = 1 when amax = 0);
 *   codes[r,k] = E4M3(x[r,k] / s), round-to-nearest-even, saturating to
 *   +-448, sign kept for values that round to zero;  scales[r] = s.
 * ninfer PR #167, opening paragraph (row-scaled A8 activations) and
 * "What actually changes".
 * x: bf16 [rows, K]; codes: u8 [rows, K]; scales: fp32 [rows].
 * Requires K % 8 == 0 and K > 0. */
SPG_API spg_status spg_quantize_fp8_rows(const void* x, int64_t rows, int64_t K, uint8_t* codes,
                                 float* scales, spg_stream_t stream);

/* FP8 E4M3 per-tensor quantizer: one scale s = amax(x)/448 for all numel
 * values (s = 1 when amax = 0), then the same code rule as above.
 * AstrAI commit log of csrc/kernels/fp8/gemm.cuh, quantize bullets (amax
 * scratch zeroed with a memset, codes plus a scale published on device).
 * x: bf16 [numel]; codes: u8 [numel]; scale: fp32 [1] (device);
 * amax_scratch: caller-owned device scratch of ONE fp32, overwritten.
 * Requires numel % 8 == 0. */
SPG_API spg_status spg_quantize_fp8_tensor(const void* x, int64_t numel, uint8_t* codes, float* scale,
                                   float* amax_scratch, spg_stream_t stream);

/* Allocation-free variant of spg_quantize_fp8_tensor (same codes and scale,
 * bit for bit).  No counterpart on the source pages: it exists for callers
 * that cannot allocate device memory for the amax scratch -- latency-critical
 * paths where an allocator call may block or fail, programs running under a
 * device-memory budget that forbids new allocations, and foreign-language
 * callers that reach this library through its C ABI with no device allocator
 * of their own.  The scratch is instead a file-scope device array of
 * 4096 + 64 floats (about 16 KB) that every GPU loading the library holds
 * until the process exits.  The caller still passes x, codes and scale.  The
 * first call on each device looks up the array's device address (once, with
 * that device current); make that first call before any stream capture.
 * All calls share the array: calls that overlap on the GPU (for example on
 * two streams) race and must be ordered by the caller.  Nothing in the array
 * needs clearing between calls.  Requires numel % 8 == 0 and
 * numel <= 4096 * 65536 = 268,435,456 elements (SPG_ERR_UNSUPPORTED_SHAPE
 * beyond).  Calls no allocating routine. */
SPG_API spg_status spg_quantize_fp8_tensor_noalloc(const void* x, int64_t numel, uint8_t* codes,
                                                   float* scale, spg_stream_t stream);

/* Delayed per-tensor scaling with an amax history ring, in one kernel.
 * Each call encodes x with the scale the previous call published,
 *   scale_used = ring.scale;  codes = E4M3(x / scale_used)  (RNE, satfinite)
 * then folds amax(x) into the ring and publishes the next scale:
 *   hist[idx] = amax(x);  idx = (idx + 1) % history;
 *   ring.scale = max(hist) / 448  (1 when the history is all zero).
 * The last block of the kernel (elected by an atomic counter after a
 * fence) does the fold, so no extra launch is needed.  AstrAI commit log of
 * csrc/kernels/fp8/gemm.cuh, scale-ring bullets.
 * ring: caller-owned device buffer of spg_fp8_scale_ring_bytes(history)
 * bytes, set up once with spg_fp8_scale_ring_init; layout (fp32 words):
 * [0, history) amax history, [history] scale, then three private words.
 * scale_used: fp32 [1], receives the scale the codes were made with (pass it
 * to the GEMM).  Calls on one ring must be ordered (one stream).
 * Requires numel % 8 == 0 and 1 <= history <= 65536. */
SPG_API size_t spg_fp8_scale_ring_bytes(int history);
SPG_API spg_status spg_fp8_scale_ring_init(void* ring, int history, float initial_scale,
                                           spg_stream_t stream);
SPG_API spg_status spg_quantize_fp8_tensor_delayed(const void* x, int64_t numel, uint8_t* codes,
                                                   float* scale_used, void* ring, int history,
                                                   spg_stream_t stream);

/* NVFP4 global scale g = amax(x) / (448 * 6) (g = 1 when amax = 0), written
 * to the device scalar g.  The largest 16-element block scale of the tensor
 * then encodes to the E4M3 maximum 448.  ninfer PR #160 body (an E4M3 scale
 * per 16 elements) with one fp32 global scale per tensor.
 * amax_scratch: caller-owned device scratch of ONE fp32, overwritten.
 * Requires numel % 8 == 0. */
SPG_API spg_status spg_nvfp4_global_scale(const void* x, int64_t numel, float* g, float* amax_scratch,
                                  spg_stream_t stream);

/* NVFP4 block quantizer.  For each 16-element block b of row r of x
 * [rows, K] (bf16), with the device scalar g:
 *   sf   = E4M3((amax_b / 6) / g)        (two IEEE fp32 divisions, RNE, satfinite)
 *   d    = dec(sf) * g                   (IEEE fp32 multiply)
 *   code = E2M1(x / d)  (RNE, satfinite, sign kept), or 0 when d == 0
 * codes: u8 [rows, K/2], element 2i in the low nibble of byte i.
 * sf: the blocked scale layout below, spg_nvfp4_sf_bytes(rows, K) bytes; the
 * padding rows are written as zero.  ninfer PR #160 body: the quantizer writes
 * the scale plane in the tile layout the GEMM loads as one TMA tile.
 * Requires K % 64 == 0. */
SPG_API spg_status spg_quantize_nvfp4(const void* x, int64_t rows, int64_t K, const float* g,
                              uint8_t* codes, uint8_t* sf, spg_stream_t stream);

/* The activations' NVFP4 quantization in one call: spg_nvfp4_global_scale
 * (x -> g) followed by spg_quantize_nvfp4 (x, g -> codes, sf), bit for bit.
 * Tensors of at most 73,728 elements (decode widths) take a single kernel
 * (one CTA finds the maximum and encodes every block) instead of the four
 * launches of the two calls (GB300: 10.8 against 21.0 us at 1 x 17408, 14.9
 * against 16.9 at 4 x 17408); up to 524,288 elements one cluster of CTAs
 * (16 where the device can hold such a cluster, else 8) shares its maxima
 * through distributed shared memory and encodes in the same launch (10.8
 * against 14.9 us at 16 x 17408).  Larger tensors take the maximum over all
 * SMs and then the block encoder, which forms g itself (three launches with
 * the scratch's memset, one fewer than the two calls).  Arguments, layouts
 * and errors as for the two calls (amax_scratch: one fp32 of caller-owned
 * scratch). */
SPG_API spg_status spg_quantize_nvfp4_act(const void* x, int64_t rows, int64_t K, float* g,
                                          float* amax_scratch, uint8_t* codes, uint8_t* sf,
                                          spg_stream_t stream);

/* Bytes of the blocked NVFP4 scale layout for a [rows, K] operand:
 * ceil(rows/128)*128 * ceil(K/64)*4.  Layout: the [rows, K/16] scale matrix
 * is cut into tiles of 128 rows x 4 scales (512 bytes), stored tile row by
 * tile row, K-tiles innermost; inside a tile the scale of (row r, column c)
 * sits at byte (r % 32) * 16 + (r / 32) * 4 + c.  (Host function.) */
SPG_API size_t spg_nvfp4_sf_bytes(int64_t rows, int64_t K);

/* Byte offset of the scale of (row, 16-element block kb) in that layout
 * (host function; -1 for out-of-range arguments). */
SPG_API int64_t spg_nvfp4_sf_offset(int64_t row, int64_t kb, int64_t K);

/* ---------------------------------------------------------------------
 * GEMMs
 * ------------------------------------------------------------------- */

/* FP8 E4M3 row-scaled GEMM with a fused epilogue.
 *   acc[t,n] = sum_k e4m3(A[t,k]) * e4m3(W[n,k])          (fp32, TMEM)
 *   y[t,n]   = acc[t,n] * sa[t] * sw[n]
 *   LINEAR: Y[t,n] = bf16(y);  ADD: Y[t,n] = bf16(y + residual[t,n]);
 *   SWIGLU: Y[t,j] = bf16(silu(y[t,2j]) * y[t,2j+1]),  Y is [T, N/2].
 * ninfer PR #167: opening paragraph (linear, linear_add, linear_swiglu call
 * sites; same accumulator, scale application and epilogue on every route),
 * review item "paired SwiGLU handling".
 * A: u8 [T,K]; sa: fp32 [T]; W: u8 [N,K]; sw: fp32 [N];
 * residual: bf16 [T,N] (ADD only, else may be NULL); Y: bf16 [T,N] or [T,N/2].
 * Requires K % 16 == 0, K > 0, N % 8 == 0 (N % 16 == 0 for SWIGLU). */
SPG_API spg_status fp8_rowscaled_gemm(const uint8_t* A, const float* sa, const uint8_t* W,
                              const float* sw, const void* residual, void* Y, int64_t T,
                              int64_t N, int64_t K, int epilogue, spg_stream_t stream);

/* NVFP4 block-scaled GEMM with the same epilogues.
 *   acc[t,n] = sum_k e2m1(A[t,k]) e4m3(sfA[t,k/16]) e2m1(W[n,k]) e4m3(sfW[n,k/16])
 *   y[t,n]   = acc[t,n] * gA * gW, then the epilogue as above.
 * ninfer PR #160 body (E2M1 codes, E4M3 scale per 16 elements, linear_add and
 * the fused SwiGLU route).
 * A: u8 [T, K/2] packed codes; sfA: blocked layout for (T, K); gA: fp32 [1];
 * W: u8 [N, K/2]; sfW: blocked layout for (N, K); gW: fp32 [1];
 * residual / Y as for the FP8 GEMM.
 * Requires K % 256 == 0, N % 8 == 0 (N % 16 == 0 for SWIGLU). */
SPG_API spg_status nvfp4_gemm(const uint8_t* A, const uint8_t* sfA, const float* gA, const uint8_t* W,
                      const uint8_t* sfW, const float* gW, const void* residual, void* Y,
                      int64_t T, int64_t N, int64_t K, int epilogue, spg_stream_t stream);

/* Per-tensor-scaled FP8 E4M3 GEMM, bf16 out, batched.
 *   C[b] = bf16( sA * sB * opA(A[b]) . opB(B[b]) ),  C[b] is [M, N]
 * layout_a = 'N': A[b] is [M, K];   'T': A[b] is [K, M]  (opA = transpose)
 * layout_b = 'T': B[b] is [N, K];   'N': B[b] is [K, N]
 * so "NT" is the forward A.B^T, "NN" the dX product and "TN" the dW product
 * of a linear layer (AstrAI commit log: layout tags, 3D operands).
 * Matrix b of A starts at A + b*strideA elements (likewise B, C); a stride
 * of 0 broadcasts one matrix over the batch (A and B only).
 * sA, sB: fp32 [1] device scalars.
 * Requires K % 16 == 0 for a K-major operand, M % 16 == 0 for a 'T' A,
 * N % 16 == 0 for an 'N' B, N % 8 == 0, strides that are multiples of 16
 * elements (C: of 8) and, for a non-zero stride, at least one matrix. */
SPG_API spg_status fp8_tensor_gemm(char layout_a, char layout_b, int64_t batch, const uint8_t* A,
                           int64_t strideA, const float* sA, const uint8_t* B, int64_t strideB,
                           const float* sB, void* C, int64_t strideC, int64_t M, int64_t N,
                           int64_t K, spg_stream_t stream);

/* The three GEMMs with a fused bias per output column, added after the
 * scales and before the epilogue:
 *   y[t,n] = acc[t,n] * scale + bias[n],  then LINEAR / ADD / SWIGLU as above
 *   (for SWIGLU the gate and up columns each get their own bias).
 * bias: bf16 [N] when bias_scale is NULL; otherwise E4M3 codes [N] (uint8)
 * dequantized as fp32(dec(code) * bias_scale[0]) with bias_scale an fp32 [1]
 * device scalar.  bias NULL means no bias (then bias_scale must be NULL).
 * AstrAI commit log of csrc/kernels/fp8/gemm.cuh, bias bullets (bias fused
 * into the epilogue for both dtypes; fp8 storage dequantized after the
 * operand scaling).  Other arguments and rules as for the plain entry points. */
SPG_API spg_status fp8_rowscaled_gemm_bias(const uint8_t* A, const float* sa, const uint8_t* W,
                                           const float* sw, const void* bias,
                                           const float* bias_scale, const void* residual, void* Y,
                                           int64_t T, int64_t N, int64_t K, int epilogue,
                                           spg_stream_t stream);
SPG_API spg_status nvfp4_gemm_bias(const uint8_t* A, const uint8_t* sfA, const float* gA,
                                   const uint8_t* W, const uint8_t* sfW, const float* gW,
                                   const void* bias, const float* bias_scale, const void* residual,
                                   void* Y, int64_t T, int64_t N, int64_t K, int epilogue,
                                   spg_stream_t stream);
SPG_API spg_status fp8_tensor_gemm_bias(char layout_a, char layout_b, int64_t batch,
                                        const uint8_t* A, int64_t strideA, const float* sA,
                                        const uint8_t* B, int64_t strideB, const float* sB,
                                        const void* bias, const float* bias_scale, void* C,
                                        int64_t strideC, int64_t M, int64_t N, int64_t K,
                                        spg_stream_t stream);

/* Workspace entry points: the GEMMs above, plus a caller-owned device
 * workspace that lets the last partial wave of two-SM tiles (every tile,
 * when the problem has fewer tiles than CTA pairs: narrow T such as decode
 * and small prefill chunks) be split along K into up to 4 pieces, when the
 * route's cost model says that pays.  Each piece writes its fp32 partial
 * sums to the workspace; for every 32-column chunk (64 for SwiGLU) of a
 * lane quarter, the piece that arrives last adds all pieces in split order
 * (so the result does not depend on the arrival order and repeats bit for
 * bit) and runs the fused epilogue on it.  The result is the same GEMM as
 * the plain entry points define, with fp32 sums taken in a different order.  The pages keep a separate
 * small-T route on sm_120 (ninfer PR #160, the paragraph on the quantizer's
 * plane layout); here the tcgen05 kernels cover narrow T by this split and,
 * for fp8_rowscaled_gemm(_ws) linear / linear_add at T <= 128 (and the
 * per-tensor NT GEMM at M <= 128), by a swapped pair tile (the weights on
 * the MMA's 256-row side, the tokens on its N side; spg_route.swap_ab).
 * With fewer tiles than the GPU has CTA pairs (swapped FP8 tile) or SMs
 * (NVFP4 one-CTA tiles), every tile's K pieces run as the CTAs of one
 * thread-block cluster and are summed in split order through distributed
 * shared memory (route variants 8 and 7): no workspace, so the plain entry
 * points take those splits too and spg_gemm_workspace_bytes is 0 for them.
 *
 * workspace: device memory, 16-byte aligned, at least
 *   spg_gemm_workspace_bytes(kind, T, N, K, epilogue, batch) bytes for the
 *   split to be used (for fp8_tensor_gemm_ws the size covers both B
 *   layouts); with less (or nullptr) the call runs the plain route.
 *   Needs no initialisation: its arrival counters are tagged with a per-call
 *   number and every completed call leaves them at zero.  One workspace
 *   serves one launch at a time (calls on one stream may share it).
 * Other arguments, rules and errors as for the _bias entry points. */
SPG_API int64_t spg_gemm_workspace_bytes(int kind, int64_t T, int64_t N, int64_t K, int epilogue,
                                         int64_t batch);
SPG_API spg_status fp8_rowscaled_gemm_ws(const uint8_t* A, const float* sa, const uint8_t* W,
                                         const float* sw, const void* bias,
                                         const float* bias_scale, const void* residual, void* Y,
                                         int64_t T, int64_t N, int64_t K, int epilogue,
                                         void* workspace, int64_t workspace_bytes,
                                         spg_stream_t stream);
SPG_API spg_status nvfp4_gemm_ws(const uint8_t* A, const uint8_t* sfA, const float* gA,
                                 const uint8_t* W, const uint8_t* sfW, const float* gW,
                                 const void* bias, const float* bias_scale, const void* residual,
                                 void* Y, int64_t T, int64_t N, int64_t K, int epilogue,
                                 void* workspace, int64_t workspace_bytes, spg_stream_t stream);
SPG_API spg_status fp8_tensor_gemm_ws(char layout_a, char layout_b, int64_t batch,
                                      const uint8_t* A, int64_t strideA, const float* sA,
                                      const uint8_t* B, int64_t strideB, const float* sB,
                                      const void* bias, const float* bias_scale, void* C,
                                      int64_t strideC, int64_t M, int64_t N, int64_t K,
                                      void* workspace, int64_t workspace_bytes,
                                      spg_stream_t stream);

/* Activation operators: the GEMMs above taking bf16 activations X [T, K]
 * (row-major, 16-byte aligned) and quantizing them inside the call, the
 * operator the pages time (ninfer PR #160 "The NVFP4 TMA route reads
 * activation scales as one tile", the operator table, which counts the
 * bf16 activation read; ninfer PR #167 "The fp8 A8 GEMM stages its operands
 * through TMA", the A8 call sites with per-row activation scales).
 *   fp8_rowscaled_linear_bf16 = spg_quantize_fp8_rows(X) -> (A, sa), then
 *     fp8_rowscaled_gemm_ws(A, sa, W, sw, ...);
 *   nvfp4_linear_bf16 = spg_nvfp4_global_scale(X) -> gA,
 *     spg_quantize_nvfp4(X, gA) -> (A, sfA) (as spg_quantize_nvfp4_act does
 *     them), then nvfp4_gemm_ws(A, sfA, gA, ...).
 * The codes, scales and result are exactly those of that sequence.  The
 * quantizer and the GEMM run back to back on `stream`, the codes and scales
 * held in the workspace.  With SPG_FORCE_VARIANT=gemv_fused the NVFP4
 * operator at T <= 4 is instead one kernel (each CTA cluster of the GEMV
 * quantizes X into its shared memory; nothing but Y is written and no
 * workspace is needed) -- measured slower than the two kernels.
 * workspace: device memory, 16-byte aligned, owned by the caller, at least
 *   spg_act_workspace_bytes(kind, T, N, K, epilogue) bytes for the full
 *   route (activation codes and scales, then the GEMM's K-split workspace);
 *   the activation part alone is required (SPG_ERR_INVALID_ARG with less),
 *   the K split is taken only when the rest is there too.  One workspace
 *   serves one call at a time.  spg_act_workspace_bytes returns 0 when the
 *   call needs none (the fused decode kernel) or the arguments are invalid.
 * Other arguments, requirements and errors as for the _ws GEMM entry points
 * (NVFP4: K % 256 == 0; FP8: K % 16 == 0). */
SPG_API int64_t spg_act_workspace_bytes(int kind, int64_t T, int64_t N, int64_t K, int epilogue);
SPG_API spg_status fp8_rowscaled_linear_bf16(const void* X, const uint8_t* W, const float* sw,
                                             const void* bias, const float* bias_scale,
                                             const void* residual, void* Y, int64_t T, int64_t N,
                                             int64_t K, int epilogue, void* workspace,
                                             int64_t workspace_bytes, spg_stream_t stream);
SPG_API spg_status nvfp4_linear_bf16(const void* X, const uint8_t* W, const uint8_t* sfW,
                                     const float* gW, const void* bias, const float* bias_scale,
                                     const void* residual, void* Y, int64_t T, int64_t N,
                                     int64_t K, int epilogue, void* workspace,
                                     int64_t workspace_bytes, spg_stream_t stream);

/* Per-shape tile / route selector (host only, no device query after the
 * first call).  kind: spg_kind; T: rows of the output (M for the tensor
 * GEMM).  Fills *out with the configuration the GEMM entry points would
 * launch for this shape.  ninfer PR #167 "Routing" (a waves-times-work cost
 * comparison) and the AstrAI dispatch-threshold bullets, re-derived for
 * 152 SMs. */
SPG_API spg_status spg_select_route(int kind, int64_t T, int64_t N, int64_t K, int epilogue,
                            int64_t batch, spg_route* out);
/* The route of the workspace entry points given a large enough workspace
 * (split_k > 1 and workspace_bytes > 0 when the K split through the
 * workspace is taken; variants 7 and 8 split inside clusters with
 * workspace_bytes 0). */
SPG_API spg_status spg_select_route_ws(int kind, int64_t T, int64_t N, int64_t K, int epilogue,
                                       int64_t batch, spg_route* out);

#ifdef __cplusplus
}
#endif

#endif /* SPG_H_ */
